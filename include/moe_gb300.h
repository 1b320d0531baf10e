/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) fused, grouped-routed MoE layer forward.
 *
 * Conventions shared by every call:
 *  - All array pointers are DEVICE pointers (cudaMalloc'd or equivalent) unless a
 *    comment says "host". Arrays are dense row-major; every base address must be
 *    16-byte aligned. The library never allocates, frees or copies to the host
 *    inside a compute call; the caller owns inputs, outputs and workspace.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Every compute call only enqueues work on that stream: it returns before the
 *    GPU has run it and performs no host synchronisation.
 *  - Arguments are validated on the host before anything is launched; a rejected
 *    call launches nothing and returns MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or
 *    MOE_ERR_WORKSPACE. A launch failure returns MOE_ERR_CUDA.
 *  - Data errors that only the GPU can see (an expert id outside [0, E), group
 *    metadata that does not add up) never trap: the kernel skips the bad element
 *    and ORs a code into the error word at the start of the workspace, which
 *    moe_check_device_error() reads back. Kernels that wait on on-chip barriers
 *    bound every wait (about two seconds) and report MOE_DEVERR_TIMEOUT instead
 *    of hanging.
 *  - Floating-point inputs must be finite (NaN / infinity are outside the contract).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, inconsistent or out-of-range argument */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement (alignment, sizes) */
  MOE_ERR_WORKSPACE = 3,    /* workspace pointer null or ws_bytes too small */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_DEVICE_DATA = 5   /* moe_check_device_error found a nonzero device error word */
} moe_status_t;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_t;

typedef enum { MOE_DT_BF16 = 0, MOE_DT_F32 = 1, MOE_DT_I8 = 2, MOE_DT_E4M3 = 3 } moe_dtype_t;

/* Bits of the device error word (first 4 bytes of every workspace). */
#define MOE_DEVERR_EXPERT_ID   0x1  /* an expert id outside [0, E) was skipped */
#define MOE_DEVERR_GROUP_META  0x2  /* expert_offsets / expert_sizes inconsistent; rows skipped */
#define MOE_DEVERR_TIMEOUT     0x4  /* an on-chip wait exceeded its bound; output incomplete */

/* Largest sizes the kernels accept. */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 32

/*
 * moe_grouped_topk -- grouped top-k routing.
 * Defined by "GroupedTopK 算子优化入门" (blog.freezetheflame.cc), section 三 steps
 * 3.1-3.6, with section 二's interface Model(topk, renormalize, num_expert_group,
 * topk_group, scoring_func, routed_scaling_factor); for num_expert_group = 1 it is
 * the mini-sglang MoE chapter's select_experts (softmax -> top-k -> renormalise).
 *
 *  gating        [T, E] fp32 router logits (the only input read; hidden_states of
 *                the blog's interface contributes its row count T only).
 *  T             tokens, >= 0 (T = 0 launches nothing).
 *  E             experts, 1..MOE_MAX_EXPERTS, divisible by num_expert_group.
 *  num_expert_group  G; group i holds experts [i*E/G, (i+1)*E/G).
 *  topk_group    groups kept per token, 1..G.
 *  topk          experts kept per token, 1..min(MOE_MAX_TOPK, topk_group*E/G).
 *  scoring       MOE_SCORE_SOFTMAX (per-token softmax) or MOE_SCORE_SIGMOID.
 *  renormalize   nonzero: selected weights are divided by their sum.
 *  routed_scaling_factor  multiplies the final weights (renormalised or not).
 *  topk_weights  [T, topk] fp32 out, descending; topk_ids [T, topk] int32 out.
 * Selection follows the exact scores, i.e. the logit order (both score functions
 * are strictly increasing); equal logits go to the lower index, equal group
 * maxima to the lower group index.
 */
MOE_API moe_status_t moe_grouped_topk(const float* gating, int T, int E, int num_expert_group,
                              int topk_group, int topk, int scoring, int renormalize,
                              float routed_scaling_factor, float* topk_weights,
                              int32_t* topk_ids, void* stream);

/*
 * moe_router_topk -- the router projection, then grouped top-k routing.
 * Defined by the mini-sglang MoE chapter, MoEMLP.forward (gate = a replicated linear
 * layer H -> E whose output, the router logits, feeds select_experts) and by
 * "GroupedTopK 算子优化入门" section 二, whose gating_output is that output; the
 * routing step is moe_grouped_topk's.
 *
 *  x              [T, H] bf16 hidden states.
 *  w_gate         [E, H] fp32 router weights (K-major, as a linear layer's weight).
 *  T, H, E        tokens (>= 0), hidden size (multiple of 32), experts (1..MOE_MAX_EXPERTS).
 *  num_expert_group, topk_group, topk, scoring, renormalize, routed_scaling_factor:
 *                 as for moe_grouped_topk.
 *  router_logits  [T, E] fp32 out: sum_k x[t,k] * w_gate[e,k], every product and sum an
 *                 fp32 operation in a fixed order (the same bits on every call); within
 *                 H * 2^-24 * sum_k |x[t,k] w_gate[e,k]| of the exact value.
 *  topk_weights   [T, topk] fp32 out, topk_ids [T, topk] int32 out: grouped top-k of
 *                 router_logits (selection on those fp32 logits).
 *  ws, ws_bytes   at least moe_router_topk_workspace_size(T, H, E) bytes, 256-byte
 *                 aligned (partial sums when few tokens split H across CTAs); may be
 *                 NULL when that size is 0. Nothing in it needs to start at zero.
 */
MOE_API size_t moe_router_topk_workspace_size(int T, int H, int E);
MOE_API moe_status_t moe_router_topk(const void* x, const float* w_gate, int T, int H, int E,
                                     int num_expert_group, int topk_group, int topk, int scoring,
                                     int renormalize, float routed_scaling_factor, float* router_logits,
                                     float* topk_weights, int32_t* topk_ids, void* ws, size_t ws_bytes,
                                     void* stream);

/*
 * moe_align_block_size -- sort the (token, expert) pairs by expert and pad.
 * Defined by the mini-sglang MoE chapter, "fused MoE", moe_align_block_size: a
 * stable sort of the flat pair indices p = token*topk + slot by expert id, every
 * expert's segment padded to a multiple of block_m with the sentinel num_pairs,
 * and the expert of every block of block_m entries.
 *
 *  topk_ids          [num_pairs] int32 expert ids (topk_ids[T, topk] flattened).
 *  num_pairs         >= 0 (0 launches only the padding fill).
 *  E                 experts, 1..MOE_MAX_EXPERTS.
 *  block_m           one of 1, 2, 4, 8, 16, 32, 64, 128, 256.
 *  sorted_token_ids  [moe_align_max_padded(num_pairs, E, block_m)] int32 out; entries
 *                    past num_tokens_post_padded hold the sentinel num_pairs too.
 *  expert_ids        [moe_align_max_padded(...) / block_m] int32 out; blocks past the
 *                    last padded segment hold -1.
 *  expert_offsets    [E + 1] int32 out: start of every expert's padded segment, then
 *                    the total.
 *  num_tokens_post_padded  [1] int32 out: the total padded length.
 *  ws, ws_bytes      workspace of at least moe_align_workspace_size(...) bytes,
 *                    256-byte aligned and zero-filled before its first use (the
 *                    call keeps a completion ticket there and leaves it at zero).
 *                    Its first 4 bytes are the device error word; ids outside
 *                    [0, E) are skipped and set MOE_DEVERR_EXPERT_ID.
 */
MOE_API size_t moe_align_max_padded(int num_pairs, int E, int block_m);
MOE_API size_t moe_align_workspace_size(int num_pairs, int E, int block_m);
MOE_API moe_status_t moe_align_block_size(const int32_t* topk_ids, int num_pairs, int E, int block_m,
                                  int32_t* sorted_token_ids, int32_t* expert_ids,
                                  int32_t* expert_offsets, int32_t* num_tokens_post_padded,
                                  void* ws, size_t ws_bytes, void* stream);

/*
 * moe_fused_forward -- the whole routed MoE layer, one stream, no host sync.
 * Defined by the mini-sglang MoE chapter, FusedMoeBackend.forward (routing, align,
 * gate_up grouped GEMM gathering rows token = pair / topk, silu(gate) * up, down
 * grouped GEMM scaled by the route weight, sum over the topk slots), with weights
 * packed as in its MoELayer, and by "Fused MoE Part 3" section 01 (no materialised
 * weight[topk_ids] and no permuted copy of x: rows are gathered inside the GEMM).
 *
 *  x            [T, H] bf16 hidden states.
 *  gating       [T, E] fp32 router logits.
 *  w_gate_up    [E, 2I, H] bf16: rows [0, I) gate, rows [I, 2I) up (K-major).
 *  w_down       [E, H, I] bf16 (K-major).
 *  T, H, I, E   tokens (>= 0), hidden (multiple of 256), intermediate (multiple of 128),
 *               experts (1..MOE_MAX_EXPERTS).
 *  num_expert_group, topk_group, topk, scoring, renormalize, routed_scaling_factor:
 *               as for moe_grouped_topk.
 *  y            [T, H] bf16 out: sum_j w[t,j] * W2[e] (silu(G_e x_t) * U_e x_t).
 *  topk_weights [T, topk] fp32 out, topk_ids [T, topk] int32 out (the routing).
 *  ws, ws_bytes workspace of at least moe_fused_forward_workspace_size(...) bytes,
 *               256-byte aligned and zero-filled before its first use (a ticket
 *               counter inside is left at zero by every call); holds the sorted pair
 *               layout, h = silu(gate)*up in sorted order and an fp32 accumulator for
 *               y. Its first 4 bytes are the device error word. The size is that of
 *               the kernels the problem size selects (16-row blocks when
 *               T * topk <= 32 * E, else 128-row blocks).
 */
MOE_API size_t moe_fused_forward_workspace_size(int T, int H, int I, int E, int topk);
MOE_API moe_status_t moe_fused_forward(const void* x, const float* gating, const void* w_gate_up,
                               const void* w_down, int T, int H, int I, int E,
                               int num_expert_group, int topk_group, int topk, int scoring,
                               int renormalize, float routed_scaling_factor, void* y,
                               float* topk_weights, int32_t* topk_ids, void* ws,
                               size_t ws_bytes, void* stream);

/*
 * moe_fused_forward_fp8 -- the same layer with FP8-e4m3 GEMM operands.
 * Defined by the low-precision GMM article (pwwt.cn): section 2.3 (weights with one
 * scale per output channel, activations with one scale per token computed from the
 * activation itself, fp32 accumulation, 8-bit values only as the matrix
 * instructions' operands), section 3.2 (symmetric scales, absmax / 448 for FP8) and
 * section 4.3 (gate and up share one epilogue whose output feeds the next GEMM);
 * the layer around it is that of moe_fused_forward. Steps, all on the device:
 * routing; align; x quantised per token to e4m3 (scale sx[t]); gate_up on the
 * gathered code rows with g = sx[t] * sw1[e, n] * acc, u likewise, h = silu(g) * u
 * held in bf16; h quantised per row to e4m3 (scale sh[row]); down with
 * y[t] += w[t, j] * sh[row] * sw2[e, n] * acc; cast of y to bf16.
 *
 *  x                [T, H] bf16 hidden states (quantised inside the call).
 *  gating           [T, E] fp32 router logits.
 *  w_gate_up        [E, 2I, H] e4m3 codes (one byte each, OCP E4M3), K-major; rows
 *                   [0, I) gate, [I, 2I) up.
 *  scales_gate_up   [E, 2I] fp32 per-output-channel scales (16-byte aligned).
 *  w_down           [E, H, I] e4m3 codes, K-major.
 *  scales_down      [E, H] fp32 per-output-channel scales (16-byte aligned).
 *  Other arguments, outputs and conditions as for moe_fused_forward (H a multiple of
 *  256, I a multiple of 128); ws of at least moe_fused_forward_fp8_workspace_size(...)
 *  bytes, 256-byte aligned and zero-filled before its first use. Kernels as for
 *  moe_fused_forward: decode-sized problems (T * topk <= 32 * E) take the swap-AB
 *  kernels (128 weight rows on the MMA's M side, an expert's tokens on N, 16-row
 *  blocks), streaming one byte per weight; larger ones the 128-row block layout.
 *  Streams: x is quantised on a second stream of the library's own (one per host
 *  thread and device, created at the first call and kept), forked from `stream` by an
 *  event at the start of the call and joined back into it before the gate_up GEMM,
 *  so that it overlaps routing and align; everything stays ordered on `stream` and the
 *  call can be captured into a CUDA graph. Make the first call outside a capture.
 */
MOE_API size_t moe_fused_forward_fp8_workspace_size(int T, int H, int I, int E, int topk);
MOE_API moe_status_t moe_fused_forward_fp8(const void* x, const float* gating, const void* w_gate_up,
                                           const float* scales_gate_up, const void* w_down,
                                           const float* scales_down, int T, int H, int I, int E,
                                           int num_expert_group, int topk_group, int topk, int scoring,
                                           int renormalize, float routed_scaling_factor, void* y,
                                           float* topk_weights, int32_t* topk_ids, void* ws,
                                           size_t ws_bytes, void* stream);

/*
 * moe_fused_forward_noalloc -- moe_fused_forward without a caller-provided workspace.
 * The pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory (a plug-in or backend inside a host framework that owns
 * all device memory and hands out no workspace; a latency-critical caller that
 * cannot afford cudaMalloc, which may synchronise the device).
 *
 * Arguments, outputs and results are those of moe_fused_forward; the scratch comes
 * from a fixed MOE_NOALLOC_SCRATCH_BYTES array inside the library, which every GPU
 * that loads the library's device code holds until the process exits. The call
 * allocates nothing.
 *  - Problems whose moe_fused_forward_workspace_size(T, H, I, E, topk) exceeds
 *    MOE_NOALLOC_SCRATCH_BYTES are rejected with MOE_ERR_WORKSPACE, before any launch.
 *    The size is that of the kernels the problem selects: decode-sized problems
 *    (T * topk <= 32 * E) use 16-row blocks, e.g. about 23 MiB at T = 128 for
 *    E = 256, H = 7168, I = 2048, topk = 8.
 *  - The first call made while a device is current looks up the array's device
 *    address on that device (cudaGetSymbolAddress) and caches it with the current
 *    CUDA context (a call under a new context, e.g. after cudaDeviceReset, looks
 *    it up again); make that first call before any stream capture on the device.
 *  - All calls share the array, which keeps the last call's contents (nothing in
 *    it needs to start at zero). Calls whose GPU work overlaps (different streams
 *    or host threads) race on it: serialise them.
 *  - The array's device error word collects MOE_DEVERR_* bits of every call on
 *    the device until moe_fused_forward_noalloc_check_error reads and clears it.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
MOE_API moe_status_t moe_fused_forward_noalloc(const void* x, const float* gating,
                                               const void* w_gate_up, const void* w_down, int T,
                                               int H, int I, int E, int num_expert_group,
                                               int topk_group, int topk, int scoring,
                                               int renormalize, float routed_scaling_factor,
                                               void* y, float* topk_weights, int32_t* topk_ids,
                                               void* stream);

/*
 * moe_fused_forward_noalloc_check_error -- moe_check_device_error for the scratch
 * array of moe_fused_forward_noalloc on the current device: synchronises `stream`,
 * writes the MOE_DEVERR_* bits collected since the last check to *code and clears
 * them. Allocates nothing. Returns MOE_OK if no bit was set, MOE_ERR_DEVICE_DATA
 * otherwise.
 */
MOE_API moe_status_t moe_fused_forward_noalloc_check_error(int* code, void* stream);

/*
 * moe_set_stage_events -- optional per-stage timing of moe_fused_forward (not in the
 * pages; instrumentation only). While set, every moe_fused_forward call made by
 * the calling host thread records events[0] on its stream before the routing
 * kernel and events[i] after its i-th step: 1 routing, 2 align, 3 gate_up GEMM,
 * 4 down GEMM, 5 cast to bf16 (n >= 6 records all). The fp32 accumulator of the
 * down pass is cleared inside step 3 (prefill kernels) or step 1 (decode
 * kernels). moe_fused_forward_fp8 records events[0] before routing and after
 * 1 routing, 2 align, 3 the join with the quantisation of x (which runs beside
 * steps 1-2 on a second stream: interval 3 is the part of it left exposed),
 * 4 gate_up GEMM, 5 quantisation of h, 6 down GEMM, 7 cast (n = 8 records all). The events are cudaEvent_t handles
 * owned by the caller. events = NULL or n = 0 switches the recording off.
 */
MOE_API void moe_set_stage_events(void* const* events, int n);

/*
 * moe_quant_per_token -- symmetric per-row quantisation.
 * Defined by the low-precision GMM article (pwwt.cn), section 3.2: per row,
 * scale = absmax / 127 and q = clamp(round_half_even(x / scale), -127, 127) for
 * INT8; scale = absmax / 448 and q = e4m3(x / scale) (nearest, ties to even,
 * saturating) for FP8-e4m3. Rows of activations give per-token scales; rows of a
 * weight matrix [E*N, K] give per-output-channel scales. An all-zero row gets
 * scale 1 and codes 0. Scale and quotient are IEEE fp32 operations.
 *
 *  x       [M, K] of x_dt (MOE_DT_BF16 or MOE_DT_F32).
 *  q       [M, K] out of q_dt (MOE_DT_I8 or MOE_DT_E4M3), one byte per element.
 *  scales  [M] fp32 out.
 *  K must be a multiple of 8.
 */
MOE_API moe_status_t moe_quant_per_token(const void* x, int x_dt, int M, int K, int q_dt, void* q,
                                 float* scales, void* stream);

/*
 * gmm_lowp -- low-precision grouped GEMM with scales fused in the epilogue.
 * Defined by the low-precision GMM article (pwwt.cn): section 2.1
 * Y_e = X[S_e] W_e^T with X pre-sorted so that S_e = [offsets[e], offsets[e]+sizes[e]),
 * section 3.1 interface gmm(input, weights, scales_x, scales_w, expert_offsets,
 * expert_sizes, output, M, K, N, E), section 2.3 fp32 accumulation:
 *   out[m, n] = scales_x[m] * scales_w[e, n] * sum_k q_x[m, k] * q_w[e, n, k].
 *
 *  input          [M, K] codes of in_dt (MOE_DT_I8 or MOE_DT_E4M3), rows sorted by expert.
 *  weights        [E, N, K] codes of the same dtype, K contiguous.
 *  scales_x       [M] fp32; scales_w [E, N] fp32.
 *  expert_offsets [E + 1] int32, nondecreasing, offsets[0] = 0, offsets[E] = M.
 *  expert_sizes   [E] int32, sizes[e] = offsets[e+1] - offsets[e].
 *  out            [M, N] of out_dt (MOE_DT_BF16 or MOE_DT_F32). Rows not covered by
 *                 any expert are left untouched.
 *  K multiple of 128, N multiple of 128. Inconsistent metadata: the offending
 *  expert is skipped and MOE_DEVERR_GROUP_META is set.
 *  ws, ws_bytes   at least gmm_lowp_workspace_size(...) bytes, 256-byte aligned,
 *                 zero-filled before its first use: bytes [4, 12) hold the task
 *                 counters, which every call leaves zero for the next one (one call at
 *                 a time per workspace); ws[0..4) is the error word.
 *  One launch for e4m3 (the GEMM, started as a programmatic dependent of the kernel
 *  before it in the stream), two for INT8 (the activation widening, then the GEMM).
 */
MOE_API size_t gmm_lowp_workspace_size(int M, int K, int N, int E);
MOE_API moe_status_t gmm_lowp(const void* input, const void* weights, const float* scales_x,
                      const float* scales_w, const int32_t* expert_offsets,
                      const int32_t* expert_sizes, void* out, int M, int K, int N, int E,
                      int in_dt, int out_dt, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_check_device_error -- read (and clear) the device error word at ws[0..4).
 * Synchronises `stream` (the only call that does). *code receives the MOE_DEVERR_*
 * bits. Returns MOE_OK if the word was zero, MOE_ERR_DEVICE_DATA otherwise.
 */
MOE_API moe_status_t moe_check_device_error(void* ws, int* code, void* stream);

/*
 * moe_read_probe -- instrumentation, not in the pages: reads `bytes` bytes (a multiple
 * of 16, 16-byte aligned) at `src` once with 16-byte loads over a grid of 8 CTAs per
 * SM, and nothing else (*sink, one float, is written only for a sum no finite input
 * of the benchmark produces). The benchmark times it beside the routing kernel on a
 * buffer of the logits' size, as the device's streaming-read floor for those bytes.
 */
MOE_API moe_status_t moe_read_probe(const void* src, size_t bytes, float* sink, void* stream);

/*
 * moe_wait_timeout_probe -- test of the device-side failure detection, not in the pages:
 * launches one CTA whose first warp waits on an on-chip barrier that nothing completes,
 * with the same bounded wait every GEMM kernel uses but a limit of limit_ns (1 ..
 * 2e9 ns), so that it runs out; the warp then raises the CTA's abort flag, a second
 * warp waiting with the full limit leaves through that flag, and MOE_DEVERR_TIMEOUT is
 * ORed into the error word at ws[0..4) (read it with moe_check_device_error). Nothing is
 * in flight when the kernel returns; the context stays usable.
 */
MOE_API moe_status_t moe_wait_timeout_probe(void* ws, unsigned long long limit_ns, void* stream);

/* Human-readable name of a status code (static string, never NULL). */
MOE_API const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
