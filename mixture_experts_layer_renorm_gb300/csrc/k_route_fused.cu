// k_route_fused.cu -- S0 + S1 + S2 in one launch for decode-sized batches.
//
// Page "Mixture of Experts in vLLM - From First Principles to fused_moe",
// sections "One token uses only 8 experts" (router, softmax, top-k,
// renormalize) and "The two index lists" (grouping the pairs by expert).  The
// SGLang issue page describes its topkGatingSoftmax kernel as fusing the
// router with softmax and top-k; the MoE execution analysis page counts the
// separate launches per decode step.  Here one launch does all three steps:
//
//   CTA (g, h) computes the router logits of token group g (TOK tokens, TOK
//   the smallest of 1, 2, 4, 8 that covers a decode batch) against expert
//   group h (8 experts, two warps per expert splitting K), writes them, and
//   counts itself done for group g; the last CTA of group g runs the top-k of
//   its tokens (one warp per token) and counts the group done; the last
//   group's CTA runs the whole align in one CTA.  "Last" is decided by an
//   atomic counter after a memory fence -- no CTA ever waits for another, so
//   nothing can hang.  The counters live in the workspace's control block;
//   the CTA that finishes a counter resets it for the next call.
//
// As a side task every CTA zeroes its share of the combine accumulator, which
// GEMM 2 adds into later in the same layer.
#include <algorithm>

#include "align_dev.cuh"
#include "route_dev.cuh"

namespace moe {

namespace {

constexpr int kFusedThreads = kAlignThreads;  // 16 warps: the align needs 512 threads
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kFusedExperts = kFusedWarps / 2;   // experts per CTA: two warps (K halves) each
constexpr int kFusedKChunk = 2048;             // x columns staged per chunk
constexpr int kFusedVec = kFusedKChunk / 8 / 32 / 2;  // 16-byte router loads per lane per chunk half

template <int VPL, int TOK>
__global__ void __launch_bounds__(kFusedThreads)
k_route_fused(const uint16_t *__restrict__ x, const uint16_t *__restrict__ w_router,
              const float *__restrict__ bias, const uint16_t *__restrict__ logits_in, int M,
              int E, int H, int top_k, int renormalize, int B, uint16_t *__restrict__ logits_ws,
              int32_t *__restrict__ topk_ids, float *__restrict__ topk_w,
              int32_t *__restrict__ sorted_ids, int32_t *__restrict__ expert_ids,
              int32_t *__restrict__ expert_offsets, int32_t *__restrict__ n_post,
              int *__restrict__ counters, int *status, float4 *__restrict__ zero_buf,
              long zero_n4, int skip_sort) {
  // the previous layer may still read the accumulator this kernel clears
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int last;
  __shared__ float half_sum[kFusedExperts][TOK];
  const int g = blockIdx.x, h = blockIdx.y;
  const int n_g = gridDim.x, n_h = gridDim.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // side task: zero the combine accumulator
  if (zero_buf != nullptr) {
    const long cta = (long)g * n_h + h, n_cta = (long)n_g * n_h;
    for (long i = cta * kFusedThreads + tid; i < zero_n4; i += n_cta * kFusedThreads)
      zero_buf[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const int t0 = g * TOK;
  const int nt = min(TOK, M - t0);
  const uint16_t *lg = logits_in;
  if (logits_in == nullptr) {
    // ---- router logits of tokens [t0, t0 + nt) x expert e; warp pair (2i, 2i+1)
    // takes expert h*8 + i, each warp one half of every K chunk
    uint4 *xs = reinterpret_cast<uint4 *>(smem);
    const int el = warp >> 1, kh = warp & 1;
    const int e = h * kFusedExperts + el;
    float acc[TOK];
#pragma unroll
    for (int j = 0; j < TOK; ++j) acc[j] = 0.f;
    for (int kc = 0; kc < H; kc += kFusedKChunk) {
      const int kw = min(kFusedKChunk, H - kc);
      const int vrow = kw / 8;                 // 16-byte columns in this chunk
      const int vh = (vrow + 1) / 2;           // columns of each half
      const int c0 = kh * vh;
      // the router row's loads go out first, so their latency overlaps the x staging
      uint4 wv[kFusedVec];
      if (e < E) {
        const uint16_t *wrow = w_router + (size_t)e * H + kc;
#pragma unroll
        for (int u = 0; u < kFusedVec; ++u) {
          const int c = c0 + lane + 32 * u;
          wv[u] = (lane + 32 * u < vh && c < vrow) ? ld_stream_16(wrow + c * 8) : make_uint4(0, 0, 0, 0);
        }
      }
      __syncthreads();
      // stage x[t0 .. t0+nt) of this chunk; every load is issued before any store
      constexpr int kStage = (TOK * (kFusedKChunk / 8) + kFusedThreads - 1) / kFusedThreads;
      uint4 xv[kStage];
#pragma unroll
      for (int it = 0; it < kStage; ++it) {
        const int v = tid + it * kFusedThreads;
        const int r = v / vrow, c = v - r * vrow;
        xv[it] = (r < nt) ? *reinterpret_cast<const uint4 *>(x + (size_t)(t0 + r) * H + kc + c * 8)
                          : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int it = 0; it < kStage; ++it) {
        const int v = tid + it * kFusedThreads;
        const int r = v / vrow, c = v - r * vrow;
        if (r < TOK) xs[r * (kFusedKChunk / 8) + c] = xv[it];
      }
      __syncthreads();
      if (e < E) {
#pragma unroll
        for (int u = 0; u < kFusedVec; ++u) {
          const int c = c0 + lane + 32 * u;
          if (lane + 32 * u < vh && c < vrow) {
            float wf[8];
            bf16x8_to_float(wv[u], wf);
#pragma unroll
            for (int j = 0; j < TOK; ++j) {
              float xf[8];
              bf16x8_to_float(xs[j * (kFusedKChunk / 8) + c], xf);
#pragma unroll
              for (int q = 0; q < 8; ++q) acc[j] = fmaf(xf[q], wf[q], acc[j]);
            }
          }
        }
      }
    }
    // reduce each token's sum over the lanes; the upper K half hands its sums
    // to the lower one through shared memory
    float mine = 0.f;
#pragma unroll
    for (int j = 0; j < TOK; ++j) {
      float v = acc[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == j) mine = v;
    }
    if (kh == 1 && lane < TOK) half_sum[el][lane] = mine;
    __syncthreads();
    if (kh == 0 && e < E && lane < nt) {
      float v = mine + half_sum[el][lane];
      if (bias != nullptr) v += bias[e];
      logits_ws[(size_t)(t0 + lane) * E + e] = float_to_bf16_bits(v);
    }
    lg = logits_ws;
    // ---- the last CTA of token group g goes on
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(&counters[g], 1) == n_h - 1;
    __syncthreads();
    if (!last) return;
    if (tid == 0) counters[g] = 0;
    __threadfence();
  }

  // ---- softmax / top-k / renormalize, one warp per token of the group
  if (warp < nt) {
    const int t = t0 + warp;
    topk_softmax_warp<VPL, true>(lg + (size_t)t * E, E, top_k, renormalize,
                                 topk_ids + (size_t)t * top_k, topk_w + (size_t)t * top_k, lane);
  }
  // with one token group this CTA holds every token's ids already (its own
  // warps wrote them); with several, the last group's CTA goes on
  if (n_g > 1) {
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(&counters[kRouteFusedMaxGroups], 1) == n_g - 1;
    __syncthreads();
    if (!last) return;
    if (tid == 0) counters[kRouteFusedMaxGroups] = 0;
    __threadfence();
  } else {
    __syncthreads();
  }

  if (skip_sort) {
    // ---- small batch (M * top_k * 4 <= E): no grouping; block p holds pair p
    // alone and its expert is topk_ids[p] (vLLM blog, "Small batches skip the
    // sort").  expert_offsets is not written: this layout has no groups.
    const int P = M * top_k;
    for (int i = tid; i < P * B; i += kFusedThreads) {
      const int p = i / B, r = i - p * B;
      sorted_ids[i] = r == 0 ? p : P;
      if (r == 0) {
        const int e = __ldcg(topk_ids + p);
        if (e < 0 || e >= E) report_status(status, kStatusBadExpertId);
        expert_ids[p] = e;
      }
    }
    if (tid == 0) *n_post = P * B;
    return;
  }
  // ---- the align over every pair, in this one CTA
  align_one_cta<true>(reinterpret_cast<int *>(smem), topk_ids, M * top_k, E, B, sorted_ids,
                      expert_ids, expert_offsets, n_post, status);
}

// Tokens per group: the smallest of 1, 2, 4, 8 covering M (decode), else 8.
int fused_tok(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

template <int VPL, int TOK>
cudaError_t launch_fused_vt(dim3 grid, size_t smem, const uint16_t *x, const uint16_t *w_router,
                            const float *bias, const uint16_t *logits_in, int M, int E, int H,
                            int top_k, int renormalize, int B, uint16_t *logits_ws,
                            int32_t *topk_ids, float *topk_w, int32_t *sorted_ids,
                            int32_t *expert_ids, int32_t *expert_offsets, int32_t *n_post,
                            int *counters, int *status, float4 *zb, long zn4, int skip_sort,
                            cudaStream_t s) {
  const void *fn = reinterpret_cast<const void *>(k_route_fused<VPL, TOK>);
  cudaError_t err = ensure_smem_limit(fn, smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_route_fused<VPL, TOK>, grid, dim3(kFusedThreads), smem, s, x, w_router, bias,
                    logits_in, M, E, H, top_k, renormalize, B, logits_ws, topk_ids, topk_w,
                    sorted_ids, expert_ids, expert_offsets, n_post, counters, status, zb, zn4,
                    skip_sort);
}

template <int VPL>
cudaError_t launch_fused_v(int tok, dim3 grid, size_t smem, const uint16_t *x,
                           const uint16_t *w_router, const float *bias, const uint16_t *logits_in,
                           int M, int E, int H, int top_k, int renormalize, int B,
                           uint16_t *logits_ws, int32_t *topk_ids, float *topk_w,
                           int32_t *sorted_ids, int32_t *expert_ids, int32_t *expert_offsets,
                           int32_t *n_post, int *counters, int *status, float4 *zb, long zn4,
                           int skip_sort, cudaStream_t s) {
#define MOE_FUSED_TOK(T)                                                                        \
  return launch_fused_vt<VPL, T>(grid, smem, x, w_router, bias, logits_in, M, E, H, top_k,      \
                                 renormalize, B, logits_ws, topk_ids, topk_w, sorted_ids,       \
                                 expert_ids, expert_offsets, n_post, counters, status, zb, zn4, \
                                 skip_sort, s)
  switch (tok) {
    case 1: MOE_FUSED_TOK(1);
    case 2: MOE_FUSED_TOK(2);
    case 4: MOE_FUSED_TOK(4);
    default: MOE_FUSED_TOK(8);
  }
#undef MOE_FUSED_TOK
}

}  // namespace

bool route_fused_supports(int M, int E, int top_k) {
  return M >= 1 && M <= 8 * kRouteFusedMaxGroups && (long)M * top_k <= 16384 && E <= kMaxExperts;
}

cudaError_t launch_route_fused(const uint16_t *x, const uint16_t *w_router, const float *bias,
                               const uint16_t *logits_in, int M, int E, int H, int top_k,
                               int renormalize, int B, uint16_t *logits_ws, int32_t *topk_ids,
                               float *topk_w, int32_t *sorted_ids, int32_t *expert_ids,
                               int32_t *expert_offsets, int32_t *n_post, int *counters,
                               int *status, float *zero_buf, long zero_n, bool skip_sort,
                               cudaStream_t s) {
  const int tok = fused_tok(M);
  const int n_g = (M + tok - 1) / tok;
  const int n_h = logits_in != nullptr ? 1 : (E + kFusedExperts - 1) / kFusedExperts;
  const size_t x_bytes = logits_in != nullptr ? 0 : sizeof(uint16_t) * tok * kFusedKChunk;
  const size_t smem = std::max(x_bytes, align_smem_bytes(E));
  const dim3 grid(n_g, n_h);
  float4 *zb = reinterpret_cast<float4 *>(zero_buf);
  const long zn4 = zero_buf != nullptr ? zero_n / 4 : 0;
#define MOE_FUSED_CASE(V)                                                                        \
  return launch_fused_v<V>(tok, grid, smem, x, w_router, bias, logits_in, M, E, H, top_k,        \
                           renormalize, B, logits_ws, topk_ids, topk_w, sorted_ids, expert_ids, \
                           expert_offsets, n_post, counters, status, zb, zn4, skip_sort ? 1 : 0, s)
  switch (topk_vpl(E)) {
    case 1: MOE_FUSED_CASE(1);
    case 2: MOE_FUSED_CASE(2);
    case 4: MOE_FUSED_CASE(4);
    case 8: MOE_FUSED_CASE(8);
    case 16: MOE_FUSED_CASE(16);
    default: MOE_FUSED_CASE(32);
  }
#undef MOE_FUSED_CASE
}

}  // namespace moe
