// k_route_fused.cu -- S0 + S1 + S2 in one launch for decode-sized batches.
//
// Page "Mixture of Experts in vLLM - From First Principles to fused_moe",
// sections "One token uses only 8 experts" (router, softmax, top-k,
// renormalize) and "The two index lists" (grouping the pairs by expert).  The
// SGLang issue page describes its topkGatingSoftmax kernel as fusing the
// router with softmax and top-k; the MoE execution analysis page counts the
// separate launches per decode step.  Here one launch does all three steps:
//
//   CTA (g, h) computes the router logits of token group g (8 tokens) against
//   expert group h (16 experts, one per warp), writes them, and counts itself
//   done for group g; the last CTA of group g runs the top-k of its tokens
//   (one warp per token) and counts the group done; the last group's CTA runs
//   the whole align in one CTA.  "Last" is decided by an atomic counter after
//   a memory fence -- no CTA ever waits for another, so nothing can hang.
//   The counters live in the workspace's control block; the CTA that finishes
//   a counter resets it for the next call.
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
constexpr int kFusedKChunk = 2048;             // x columns staged per chunk
constexpr int kFusedVec = kFusedKChunk / 8 / 32;  // 16-byte router loads per lane per chunk

template <int VPL>
__global__ void __launch_bounds__(kFusedThreads)
k_route_fused(const uint16_t *__restrict__ x, const uint16_t *__restrict__ w_router,
              const float *__restrict__ bias, const uint16_t *__restrict__ logits_in, int M,
              int E, int H, int top_k, int renormalize, int B, uint16_t *__restrict__ logits_ws,
              int32_t *__restrict__ topk_ids, float *__restrict__ topk_w,
              int32_t *__restrict__ sorted_ids, int32_t *__restrict__ expert_ids,
              int32_t *__restrict__ expert_offsets, int32_t *__restrict__ n_post,
              int *__restrict__ counters, int *status, float4 *__restrict__ zero_buf,
              long zero_n4) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int last;
  const int g = blockIdx.x, h = blockIdx.y;
  const int n_g = gridDim.x, n_h = gridDim.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // side task: zero the combine accumulator
  if (zero_buf != nullptr) {
    const long cta = (long)g * n_h + h, n_cta = (long)n_g * n_h;
    for (long i = cta * kFusedThreads + tid; i < zero_n4; i += n_cta * kFusedThreads)
      zero_buf[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const int t0 = g * kRouteFusedTok;
  const int nt = min(kRouteFusedTok, M - t0);
  const uint16_t *lg = logits_in;
  if (logits_in == nullptr) {
    // ---- router logits of tokens [t0, t0 + nt) x expert e (one warp each)
    uint4 *xs = reinterpret_cast<uint4 *>(smem);
    const int e = h * kFusedWarps + warp;
    float acc[kRouteFusedTok];
#pragma unroll
    for (int j = 0; j < kRouteFusedTok; ++j) acc[j] = 0.f;
    for (int kc = 0; kc < H; kc += kFusedKChunk) {
      const int kw = min(kFusedKChunk, H - kc);
      const int vrow = kw / 8;
      // the router row's loads go out first, so their latency overlaps the x staging
      uint4 wv[kFusedVec];
      if (e < E) {
        const uint16_t *wrow = w_router + (size_t)e * H + kc;
#pragma unroll
        for (int u = 0; u < kFusedVec; ++u) {
          const int c = lane + 32 * u;
          wv[u] = c < vrow ? ld_stream_16(wrow + c * 8) : make_uint4(0, 0, 0, 0);
        }
      }
      __syncthreads();
      for (int v = tid; v < kRouteFusedTok * vrow; v += kFusedThreads) {
        const int r = v / vrow, c = v - r * vrow;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r < nt) val = *reinterpret_cast<const uint4 *>(x + (size_t)(t0 + r) * H + kc + c * 8);
        xs[r * (kFusedKChunk / 8) + c] = val;
      }
      __syncthreads();
      if (e < E) {
#pragma unroll
        for (int u = 0; u < kFusedVec; ++u) {
          const int c = lane + 32 * u;
          if (c < vrow) {
            float wf[8];
            bf16x8_to_float(wv[u], wf);
#pragma unroll
            for (int j = 0; j < kRouteFusedTok; ++j) {
              float xf[8];
              bf16x8_to_float(xs[j * (kFusedKChunk / 8) + c], xf);
#pragma unroll
              for (int q = 0; q < 8; ++q) acc[j] = fmaf(xf[q], wf[q], acc[j]);
            }
          }
        }
      }
    }
    if (e < E) {
      float mine = 0.f;
#pragma unroll
      for (int j = 0; j < kRouteFusedTok; ++j) {
        float v = acc[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == j) mine = v;
      }
      if (lane < nt) {
        if (bias != nullptr) mine += bias[e];
        logits_ws[(size_t)(t0 + lane) * E + e] = float_to_bf16_bits(mine);
      }
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
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(&counters[kRouteFusedMaxGroups], 1) == n_g - 1;
  __syncthreads();
  if (!last) return;
  if (tid == 0) counters[kRouteFusedMaxGroups] = 0;
  __threadfence();

  // ---- the align over every pair, in this one CTA
  align_one_cta<true>(reinterpret_cast<int *>(smem), topk_ids, M * top_k, E, B, sorted_ids,
                      expert_ids, expert_offsets, n_post, status);
}

}  // namespace

bool route_fused_supports(int M, int E, int top_k) {
  return M >= 1 && M <= kRouteFusedTok * kRouteFusedMaxGroups && (long)M * top_k <= 16384 &&
         E <= kMaxExperts;
}

cudaError_t launch_route_fused(const uint16_t *x, const uint16_t *w_router, const float *bias,
                               const uint16_t *logits_in, int M, int E, int H, int top_k,
                               int renormalize, int B, uint16_t *logits_ws, int32_t *topk_ids,
                               float *topk_w, int32_t *sorted_ids, int32_t *expert_ids,
                               int32_t *expert_offsets, int32_t *n_post, int *counters,
                               int *status, float *zero_buf, long zero_n, cudaStream_t s) {
  const int n_g = (M + kRouteFusedTok - 1) / kRouteFusedTok;
  const int n_h = logits_in != nullptr ? 1 : (E + kFusedWarps - 1) / kFusedWarps;
  const size_t x_bytes = logits_in != nullptr ? 0 : sizeof(uint16_t) * kRouteFusedTok * kFusedKChunk;
  const size_t smem = std::max(x_bytes, align_smem_bytes(E));
  const dim3 grid(n_g, n_h);
  float4 *zb = reinterpret_cast<float4 *>(zero_buf);
  const long zn4 = zero_buf != nullptr ? zero_n / 4 : 0;
#define MOE_FUSED_CASE(V)                                                                          \
  do {                                                                                             \
    cudaError_t err = ensure_smem_limit(reinterpret_cast<const void *>(k_route_fused<V>), smem);   \
    if (err != cudaSuccess) return err;                                                            \
    k_route_fused<V><<<grid, kFusedThreads, smem, s>>>(                                            \
        x, w_router, bias, logits_in, M, E, H, top_k, renormalize, B, logits_ws, topk_ids, topk_w, \
        sorted_ids, expert_ids, expert_offsets, n_post, counters, status, zb, zn4);                \
  } while (0)
  switch (topk_vpl(E)) {
    case 1: MOE_FUSED_CASE(1); break;
    case 2: MOE_FUSED_CASE(2); break;
    case 4: MOE_FUSED_CASE(4); break;
    case 8: MOE_FUSED_CASE(8); break;
    case 16: MOE_FUSED_CASE(16); break;
    default: MOE_FUSED_CASE(32); break;
  }
#undef MOE_FUSED_CASE
  return cudaGetLastError();
}

}  // namespace moe
