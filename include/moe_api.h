/*
 * moe_api.h -- C ABI of the GB300 (sm_103a) forward pass of one top-k-routed
 * SwiGLU mixture-of-experts layer.
 *
 * The layer (page "Mixture of Experts in vLLM - From First Principles to
 * fused_moe", below [vLLM]):
 *   logits = x W_r^T (+ bias)                      "One token uses only 8 experts"
 *   p = softmax(logits); keep top_k; renormalize   "One token uses only 8 experts"
 *   group the M*top_k (token, expert) pairs by
 *   expert, padded to BLOCK_SIZE_M blocks          "The two index lists"
 *   a_p = SiLU(h_gate) * h_up, h = W13_e x_t       "An expert is a small SwiGLU MLP"
 *   y_t = sum_j w_j W2_{e_j} a_{t*top_k+j}         "Put the results back, and combine
 *                                                   them per token"
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the
 *     library never frees, keeps or reallocates it.  Tensors are dense and
 *     row-major.  bf16 tensors hold raw bfloat16 bit patterns (moe_bf16_t).
 *   - Every call is asynchronous on `stream`, allocates no memory and never
 *     synchronises with the host (except moe_get_device_status).
 *   - Pointers to bf16 matrices are 16-byte aligned; the workspace pointer is
 *     256-byte aligned (MOE_ERR_INVALID_ARG otherwise).
 *   - Weight layouts follow nn.Linear (the reduction dimension is
 *     contiguous): W13 [E, 2I, H] with gate rows [0, I) above up rows
 *     [I, 2I) ([vLLM] "An expert is a small SwiGLU MLP"); W2 [E, H, I];
 *     W_r [E, H].
 *   - Pair id p = t * top_k + j ([vLLM] "A batch: (token, expert) pairs").
 *   - Limits: 1 <= E <= 1024; 1 <= top_k <= min(E, 32); H, I multiples of 16
 *     with 16 <= H, I <= 65536; M >= 0 (M == 0 is a no-op returning MOE_OK);
 *     1 <= block_size_m <= 256, or 0 for the automatic choice where the
 *     entry point allows it.  M * top_k < 2^31 - 2^18.
 *   - Rounding: bf16 round-to-nearest-even of fp32 values at the logits, the
 *     GEMM-1 output h, the activation a and the output y; fp32 accumulation;
 *     the GEMM-2 output is not rounded before the weighted combine.
 *
 * Errors: shape, pointer and size problems are found on the host before any
 * launch and returned (nothing is launched).  A failed launch returns
 * MOE_ERR_CUDA.  Data-dependent problems (an expert id outside [0, E) in a
 * caller-given topk_ids) are written to a status word at the start of the
 * workspace and read back by moe_get_device_status; kernels never trap.
 */
#ifndef MOE_API_H
#define MOE_API_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16_t; /* raw bfloat16 bit pattern */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,          /* null pointer, negative size, bad flag */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,    /* outside the limits above */
    MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < moe_workspace_size(...) */
    MOE_ERR_CUDA = 4,                 /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE_BAD_EXPERT_ID = 5, /* device status: topk_ids entry outside [0, E) */
    MOE_ERR_DEVICE_TIMEOUT = 6        /* device status: a bounded wait ran out */
} moe_status_t;

/* Bytes of workspace that moe_forward, moe_align_block_size and
 * moe_grouped_gemm_w2_combine need for any M <= M_max with these shapes.
 * block_size_m = 0 sizes for every block size the automatic choice may
 * pick.  The workspace is the per-layer buffer set that the MoE execution
 * analysis page ("Memory allocation per step") proposes to allocate once and
 * reuse across layers: one buffer, reused by every layer and every call.
 * Returns 0 when the arguments are outside the limits. */
size_t moe_workspace_size(int M_max, int E, int top_k, int H, int I, int block_size_m);

/* Entries of sorted_token_ids for M tokens: M*top_k + E*(B-1), rounded up to
 * a multiple of B.  expert_ids has capacity / B entries.  [vLLM] "The two
 * index lists": each expert's group is padded up to a multiple of B.
 * Returns -1 when the arguments are outside the limits (B must be explicit). */
long moe_align_capacity(int M, int top_k, int E, int block_size_m);

/* The block size moe_forward uses when given block_size_m = 0. */
int moe_pick_block_size(int M, int E, int top_k, int H, int I);

/* S0. Router logits.  [vLLM] "One token uses only 8 experts": W_r [E, H]
 * gives one score per expert.
 *   logits[t, e] = bf16( sum_h x[t, h] * w_router[e, h] + router_bias[e] )
 * x [M, H] bf16; w_router [E, H] bf16; router_bias [E] fp32 or NULL;
 * logits [M, E] bf16 (output). */
moe_status_t moe_router_logits(const moe_bf16_t *x, const moe_bf16_t *w_router,
                               const float *router_bias, int M, int E, int H,
                               moe_bf16_t *logits, cudaStream_t stream);

/* S1. Softmax, top-k and renormalize.  [vLLM] "One token uses only 8
 * experts", steps 1-3.  Slot j of token t holds the j-th largest logit; equal
 * logits go to the lower expert id.  With renormalize != 0 the kept weights
 * are rescaled to sum to 1, otherwise they are the softmax probabilities.
 * logits [M, E] bf16; topk_ids [M, top_k] int32 (output); topk_weights
 * [M, top_k] fp32 (output).  Logits must be finite. */
moe_status_t moe_topk_softmax(const moe_bf16_t *logits, int M, int E, int top_k,
                              int renormalize, int32_t *topk_ids, float *topk_weights,
                              cudaStream_t stream);

/* S2. Group the pairs by expert.  [vLLM] "The two index lists" and
 * "Group by expert": sorted_token_ids lists the pair ids grouped by expert in
 * ascending expert id, ascending pair id inside a group (a stable counting
 * sort), each group padded with the id M*top_k up to a multiple of B;
 * experts with no pair get no block.  expert_ids[b] is the expert of block b;
 * expert_offsets[e] is where expert e's padded group starts
 * (expert_offsets[E] = n_post); *num_tokens_post_padded = n_post.
 * Entries of sorted_token_ids at and after n_post and of expert_ids at and
 * after n_post / B are left unspecified.
 * topk_ids [M*top_k] int32; sorted_token_ids [moe_align_capacity()] int32,
 * expert_ids [capacity / B] int32, expert_offsets [E + 1] int32,
 * num_tokens_post_padded [1] int32 (outputs).  block_size_m must be explicit.
 * ws/ws_bytes: the workspace (status word and scratch counters).  An id
 * outside [0, E) is left out of the grouping and reported as
 * MOE_ERR_DEVICE_BAD_EXPERT_ID through moe_get_device_status. */
moe_status_t moe_align_block_size(const int32_t *topk_ids, int M, int top_k, int E,
                                  int block_size_m, int32_t *sorted_token_ids,
                                  int32_t *expert_ids, int32_t *expert_offsets,
                                  int32_t *num_tokens_post_padded, void *ws, size_t ws_bytes,
                                  cudaStream_t stream);

/* S0 + S1 + S2 together: router logits (or the given logits), softmax /
 * top-k / renormalize and the block-padded grouping, with the results of
 * moe_router_logits, moe_topk_softmax and moe_align_block_size.  The SGLang
 * issue page describes a kernel that fuses the router with softmax and top-k,
 * and the MoE execution analysis page ("Per-decode-step kernel launches")
 * counts one launch per step per layer; for batches of up to 256 tokens (with
 * M * top_k <= 16384) this runs as one launch, otherwise as the router (its
 * K range split over up to four CTAs per tile, through the workspace, when
 * the tiles leave SMs idle), top-k and align kernels (count and scatter above
 * 2048 pairs).
 * Exactly one of w_router [E, H] and router_logits [M, E] is non-NULL
 * (router_bias only with w_router; H is ignored with router_logits).
 * Outputs as for moe_topk_softmax and moe_align_block_size (block_size_m
 * explicit).  router_logits_out [M, E] bf16 or NULL: with w_router, the
 * logits the routing was decided on are written there (they equal what
 * moe_router_logits gives up to the order of the fp32 sums); not written
 * when router_logits is given.  ws/ws_bytes: a workspace of at least moe_workspace_size(M, E,
 * top_k, 16, 16, block_size_m) bytes, initialised once with moe_workspace_init
 * (its control block holds counters that must start at zero; each call leaves
 * them at zero); calls sharing a workspace must not overlap on the GPU. */
moe_status_t moe_route(const moe_bf16_t *x, const moe_bf16_t *w_router,
                       const moe_bf16_t *router_logits, const float *router_bias, int M, int E,
                       int top_k, int H, int renormalize, int block_size_m, int32_t *topk_ids,
                       float *topk_weights, int32_t *sorted_token_ids, int32_t *expert_ids,
                       int32_t *expert_offsets, int32_t *num_tokens_post_padded,
                       moe_bf16_t *router_logits_out, void *ws, size_t ws_bytes,
                       cudaStream_t stream);

/* S3. Grouped GEMM 1 with SiLU-and-mul.  [vLLM] "One GEMM 1 program, step by
 * step" and "The rest of the layer stays in pair order": for every real pair
 * p in block b (p < M*top_k), with e = expert_ids[b] and t = p / top_k,
 *   h = bf16(W13_e x_t)  [2I];   a[p, i] = bf16( SiLU(h[i]) * h[I + i] )
 * Input rows are read in place through p / top_k (no permuted copy).
 * x [M, H]; w13 [E, 2I, H]; sorted_token_ids / expert_ids /
 * num_tokens_post_padded as produced by moe_align_block_size with the same
 * M, top_k, E and block_size_m (explicit); a [M*top_k, I] bf16 (output, pair
 * order).  Blocks whose expert id lies outside [0, E) are skipped. */
moe_status_t moe_grouped_gemm_w13_act(const moe_bf16_t *x, const moe_bf16_t *w13,
                                      const int32_t *sorted_token_ids, const int32_t *expert_ids,
                                      const int32_t *num_tokens_post_padded, int M, int top_k,
                                      int E, int H, int I, int block_size_m, moe_bf16_t *a,
                                      cudaStream_t stream);

/* S4. Grouped GEMM 2 with the router-weighted combine.  [vLLM] "The rest of
 * the layer stays in pair order" and "Put the results back, and combine them
 * per token":
 *   o_p = W2_e a_p (fp32, not rounded);
 *   y[t] = bf16( sum_j topk_weights[t, j] * o_{t*top_k + j} + residual[t] )
 * a [M*top_k, I]; w2 [E, H, I]; topk_weights [M, top_k] fp32; residual
 * [M, H] bf16 or NULL; y [M, H] bf16 (output).  Index lists as for S3.
 * ws/ws_bytes: the workspace (holds the fp32 accumulator). */
moe_status_t moe_grouped_gemm_w2_combine(const moe_bf16_t *a, const moe_bf16_t *w2,
                                         const int32_t *sorted_token_ids,
                                         const int32_t *expert_ids,
                                         const int32_t *num_tokens_post_padded,
                                         const float *topk_weights, const moe_bf16_t *residual,
                                         int M, int top_k, int E, int H, int I, int block_size_m,
                                         moe_bf16_t *y, void *ws, size_t ws_bytes,
                                         cudaStream_t stream);

/* moe_grouped_gemm_w2_combine for callers that cannot provide a workspace.
 * The pages this library follows have no counterpart of this entry point.
 * It serves callers that cannot allocate device memory: plugin code inside a
 * host application that owns every device allocation and offers the plugin no
 * allocator, and latency-critical code that may not call cudaMalloc (which can
 * synchronise the device and takes unbounded time).  Same arguments and result
 * as moe_grouped_gemm_w2_combine, without ws / ws_bytes.
 * The fp32 accumulator is a fixed array of 2,097,152 floats (8 MiB) compiled
 * into the library; every GPU that loads the library holds it until the
 * process exits.  M * H above 2,097,152 returns MOE_ERR_UNSUPPORTED_SHAPE
 * (nothing is launched).  No memory is allocated: the first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) and keeps it, so
 * make that first call on each device before capturing a stream.  All calls
 * share the one array, which keeps the last call's contents (each call clears
 * the part it uses first): calls that may overlap on the GPU (different
 * streams, or different host threads) race on it and give wrong results. */
moe_status_t moe_grouped_gemm_w2_combine_noalloc(const moe_bf16_t *a, const moe_bf16_t *w2,
                                                 const int32_t *sorted_token_ids,
                                                 const int32_t *expert_ids,
                                                 const int32_t *num_tokens_post_padded,
                                                 const float *topk_weights,
                                                 const moe_bf16_t *residual, int M, int top_k,
                                                 int E, int H, int I, int block_size_m,
                                                 moe_bf16_t *y, cudaStream_t stream);

/* The whole layer: S0 (skipped when router_logits is given) .. S4.
 * Exactly one of w_router [E, H] and router_logits [M, E] is non-NULL.
 * router_bias [E] fp32 or NULL (only with w_router); residual [M, H] or NULL.
 * y [M, H] bf16 (output); topk_ids_out [M, top_k] int32 and
 * topk_weights_out [M, top_k] fp32 are optional copies of the routing;
 * router_logits_out [M, E] bf16 (optional, with w_router only) receives the
 * logits the routing was decided on.
 * block_size_m = 0 picks moe_pick_block_size(M, E, top_k, H, I).
 * ws_bytes >= moe_workspace_size(M, E, top_k, H, I, block_size_m).
 * The workspace's intermediate lists are internal to this call: for
 * M * top_k * 4 <= E it gives each pair its own block instead of grouping by
 * expert (the vLLM blog, "Small batches skip the sort"); y is the same.
 * With the environment variable MOE_DECODE_LAYER=on, decode-sized calls
 * (M * top_k <= 512, I <= 1536, the shapes fitting one CTA's shared memory)
 * run the whole layer as one persistent cooperative kernel (router, top-k,
 * grouping, both GEMMs and the combine; the MoE execution analysis page,
 * "Per-decode-step kernel launches"); same arguments, same results within
 * the output tolerance.  It is off by default: on this GPU it measured no
 * faster than the kernel chain.   The
 * kernels of the layer are programmatic dependent launches, so a layer may
 * start while the previous kernel on `stream` is still finishing; it waits
 * for that kernel before it reads anything the kernel writes (x, residual,
 * router_logits). */
moe_status_t moe_forward(const moe_bf16_t *x, const moe_bf16_t *w_router,
                         const moe_bf16_t *router_logits, const float *router_bias,
                         const moe_bf16_t *w13, const moe_bf16_t *w2,
                         const moe_bf16_t *residual, int M, int E, int top_k, int H, int I,
                         int renormalize, int block_size_m, moe_bf16_t *y,
                         int32_t *topk_ids_out, float *topk_weights_out,
                         moe_bf16_t *router_logits_out, void *ws, size_t ws_bytes,
                         cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * FP8 (E4M3) expert weights, W8A8.  [vLLM] "fused_experts_impl": one kernel
 * serves bf16 and FP8 weights, and for an FP8 model the GEMM-1 input is the
 * quantized copy of x.  Format and scale granularity are not given there;
 * this library takes:
 *   - E4M3 codes (uint8: 1 sign, 4 exponent bits with bias 7, 3 mantissa
 *     bits, largest finite 448), each weight matrix with one fp32 scale per
 *     output row: w13_scales [E, 2I] for W13 codes [E, 2I, H], w2_scales
 *     [E, H] for W2 codes [E, H, I];
 *   - activations quantized per row at run time (moe_quantize_rows_fp8):
 *     x per token before GEMM 1, a per pair before GEMM 2;
 *   - scales applied after the fp32 sums: h = bf16(s_x s_w sum q_x q_w),
 *     a = bf16(SiLU(h_gate) * h_up) as in the bf16 layer, and the GEMM-2
 *     output s_a s_w2 sum q_a q_w2 combined without rounding.
 * Limits as above; every block size must be one of 16, 32, 64, 128, 256
 * (the tensor-core tiles; MOE_ERR_UNSUPPORTED_SHAPE otherwise).  Code
 * pointers are 16-byte aligned.  The router stays bf16.
 * ------------------------------------------------------------------------- */

/* Per-row dynamic quantization of src [R, K] bf16 (K a multiple of 16):
 * scales[r] = amax_k |src[r, k]| / 448 (1 for an all-zero row), q[r, k] =
 * E4M3(src[r, k] / scales[r]) rounded to nearest, ties to even, saturating
 * at +-448.  amax, the scale and each quotient are fp32 with correctly
 * rounded division, so the codes depend on the row alone.  q [R, K] uint8
 * and scales [R] fp32 are outputs.  R == 0 is a no-op. */
moe_status_t moe_quantize_rows_fp8(const moe_bf16_t *src, int R, int K, uint8_t *q,
                                   float *scales, cudaStream_t stream);

/* Workspace bytes for moe_forward_fp8: moe_workspace_size's regions plus the quantized x [M, H] / a [M*top_k, I]
 * codes and their per-row scales.  0 when the arguments are outside the
 * limits. */
size_t moe_workspace_size_fp8(int M_max, int E, int top_k, int H, int I, int block_size_m);

/* S3 on E4M3 operands: a [M*top_k, I] bf16 from qx [M, H] codes with
 * x_scales [M], W13 codes w13 [E, 2I, H] with w13_scales [E, 2I], and the
 * align lists (as moe_grouped_gemm_w13_act).  block_size_m explicit. */
moe_status_t moe_grouped_gemm_w13_act_fp8(const uint8_t *qx, const float *x_scales,
                                          const uint8_t *w13, const float *w13_scales,
                                          const int32_t *sorted_token_ids,
                                          const int32_t *expert_ids,
                                          const int32_t *num_tokens_post_padded, int M,
                                          int top_k, int E, int H, int I, int block_size_m,
                                          moe_bf16_t *a, cudaStream_t stream);

/* S4 on E4M3 operands: y [M, H] bf16 = bf16(sum_j w_j s_a s_w2 (q_a . q_w2)
 * + residual) from qa [M*top_k, I] codes with a_scales [M*top_k], W2 codes
 * w2 [E, H, I] with w2_scales [E, H], topk_weights [M, top_k] fp32 and the
 * align lists.  ws_bytes >= moe_workspace_size(M, E, top_k, H, I,
 * block_size_m) (the fp32 accumulator lives there). */
moe_status_t moe_grouped_gemm_w2_combine_fp8(const uint8_t *qa, const float *a_scales,
                                             const uint8_t *w2, const float *w2_scales,
                                             const int32_t *sorted_token_ids,
                                             const int32_t *expert_ids,
                                             const int32_t *num_tokens_post_padded,
                                             const float *topk_weights,
                                             const moe_bf16_t *residual, int M, int top_k,
                                             int E, int H, int I, int block_size_m,
                                             moe_bf16_t *y, void *ws, size_t ws_bytes,
                                             cudaStream_t stream);

/* The whole layer with E4M3 expert weights: routing as moe_forward (bf16
 * router or given logits), x quantized per token, GEMM 1 on codes, a
 * quantized per pair, GEMM 2 + combine on codes.  Arguments as moe_forward,
 * with the W13 / W2 codes and their row scales in place of the bf16 weights;
 * ws_bytes >= moe_workspace_size_fp8(M, E, top_k, H, I, block_size_m).
 * Runs the kernel chain (MOE_DECODE_LAYER does not apply). */
moe_status_t moe_forward_fp8(const moe_bf16_t *x, const moe_bf16_t *w_router,
                             const moe_bf16_t *router_logits, const float *router_bias,
                             const uint8_t *w13, const float *w13_scales, const uint8_t *w2,
                             const float *w2_scales, const moe_bf16_t *residual, int M, int E,
                             int top_k, int H, int I, int renormalize, int block_size_m,
                             moe_bf16_t *y, int32_t *topk_ids_out, float *topk_weights_out,
                             moe_bf16_t *router_logits_out, void *ws, size_t ws_bytes,
                             cudaStream_t stream);

/* Clears the whole workspace (asynchronously on `stream`).  Call it once on a
 * freshly allocated workspace before its first use: the status word at its
 * start must begin at zero.  ws must be 256-byte aligned. */
moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronises `stream`, returns the device status word kept at the start of
 * the workspace (MOE_OK if no kernel reported a problem) and clears it.  The
 * entry points that take no workspace (moe_router_logits,
 * moe_grouped_gemm_w13_act, moe_grouped_gemm_w2_combine_noalloc) report into
 * one library-wide word per device instead; it is read (and cleared) here as
 * well, and on its own when ws is NULL -- the way a caller without a
 * workspace learns that one of those calls gave up on a bounded wait.  With
 * ws NULL and no usable CUDA device the result is MOE_ERR_CUDA. */
moe_status_t moe_get_device_status(void *ws, cudaStream_t stream);

/* Self-test of the device failure path.  Launches one CTA that waits, with
 * the bounded wait every kernel of the library uses, on an mbarrier that
 * nothing completes; after about limit_ms milliseconds of SM clock (clamped to
 * [1, 2000]) the wait gives up, records MOE_ERR_DEVICE_TIMEOUT in the
 * workspace's status word and the kernel returns -- nothing traps, and the
 * context stays usable.  Read the result with moe_get_device_status.
 * Returns MOE_ERR_INVALID_ARG for a null or misaligned workspace or one
 * smaller than its status block. */
moe_status_t moe_selftest_device_timeout(void *ws, size_t ws_bytes, int limit_ms,
                                         cudaStream_t stream);

/* A static, human-readable name for a status code. */
const char *moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_API_H */
