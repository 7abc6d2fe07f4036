// k_route.cu -- S0 router logits (CUDA-core path) and S1 softmax / top-k /
// renormalize.
//
// Page "Mixture of Experts in vLLM - From First Principles to fused_moe",
// section "One token uses only 8 experts": the router is one linear layer
// W_r [E, H]; softmax over the E scores; keep the top_k largest; rescale the
// kept weights to sum to 1 (renormalize).
#include "route_dev.cuh"

namespace moe {

namespace {

constexpr int kRouterTok = 8;        // tokens per CTA
constexpr int kRouterWarps = 8;      // one expert per warp
constexpr int kRouterKChunk = 2048;  // x columns staged in shared memory at once
constexpr int kRouterVec = kRouterKChunk / 8 / 32;  // 16-byte router loads per lane per chunk

// CUDA-core router for small batches: one CTA covers kRouterTok tokens and
// kRouterWarps experts.  x rows are staged in shared memory chunk by chunk;
// each warp issues all of its router row's loads for the chunk at once
// (kRouterVec 16-byte loads per lane in flight), then accumulates every staged
// token against them in fp32.  Large batches use the tensor-core router.
__global__ void __launch_bounds__(kRouterWarps * 32)
k_router_logits(const uint16_t *__restrict__ x, const uint16_t *__restrict__ w_router,
                const float *__restrict__ bias, int M, int E, int H, uint16_t *__restrict__ logits) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ uint4 xs[kRouterTok * (kRouterKChunk / 8)];
  const int t0 = blockIdx.x * kRouterTok;
  const int nt = min(kRouterTok, M - t0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.y * kRouterWarps + warp;
  float acc[kRouterTok];
#pragma unroll
  for (int j = 0; j < kRouterTok; ++j) acc[j] = 0.f;

  for (int kc = 0; kc < H; kc += kRouterKChunk) {
    const int kw = min(kRouterKChunk, H - kc);
    const int vrow = kw / 8;
    __syncthreads();
    for (int v = threadIdx.x; v < kRouterTok * vrow; v += blockDim.x) {
      const int r = v / vrow, c = v - r * vrow;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (r < nt) val = *reinterpret_cast<const uint4 *>(x + (size_t)(t0 + r) * H + kc + c * 8);
      xs[r * (kRouterKChunk / 8) + c] = val;
    }
    __syncthreads();
    if (e < E) {
      const uint16_t *wrow = w_router + (size_t)e * H + kc;
      uint4 wv[kRouterVec];
#pragma unroll
      for (int u = 0; u < kRouterVec; ++u) {
        const int c = lane + 32 * u;
        wv[u] = c < vrow ? ld_stream_16(wrow + c * 8) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kRouterVec; ++u) {
        const int c = lane + 32 * u;
        if (c < vrow) {
          float wf[8];
          bf16x8_to_float(wv[u], wf);
#pragma unroll
          for (int j = 0; j < kRouterTok; ++j) {
            float xf[8];
            bf16x8_to_float(xs[j * (kRouterKChunk / 8) + c], xf);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[j] = fmaf(xf[q], wf[q], acc[j]);
          }
        }
      }
    }
  }
  if (e >= E) return;
  float mine = 0.f;
#pragma unroll
  for (int j = 0; j < kRouterTok; ++j) {
    float v = acc[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == j) mine = v;
  }
  if (lane < nt) {
    if (bias != nullptr) mine += bias[e];
    logits[(size_t)(t0 + lane) * E + e] = float_to_bf16_bits(mine);
  }
}

// One warp per token.
template <int VPL>
__global__ void __launch_bounds__(256)
k_topk_softmax(const uint16_t *__restrict__ logits, int M, int E, int top_k, int renormalize,
               int32_t *__restrict__ topk_ids, float *__restrict__ topk_weights) {
  griddep_wait();
  griddep_launch_dependents();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= M) return;
  topk_softmax_warp<VPL, false>(logits + (size_t)t * E, E, top_k, renormalize,
                                topk_ids + (size_t)t * top_k, topk_weights + (size_t)t * top_k,
                                threadIdx.x & 31);
}

}  // namespace

cudaError_t launch_router_logits(const uint16_t *x, const uint16_t *w_router, const float *bias,
                                 int M, int E, int H, uint16_t *logits, cudaStream_t s) {
  dim3 grid((M + kRouterTok - 1) / kRouterTok, (E + kRouterWarps - 1) / kRouterWarps);
  return launch_pdl(k_router_logits, grid, dim3(kRouterWarps * 32), 0, s, x, w_router, bias, M, E,
                    H, logits);
}

cudaError_t launch_topk_softmax(const uint16_t *logits, int M, int E, int top_k, int renormalize,
                                int32_t *topk_ids, float *topk_weights, cudaStream_t s) {
  const int threads = 256;
  const int blocks = (M * 32 + threads - 1) / threads;
#define MOE_TOPK_CASE(V)                                                                    \
  return launch_pdl(k_topk_softmax<V>, dim3(blocks), dim3(threads), 0, s, logits, M, E, top_k, \
                    renormalize, topk_ids, topk_weights)
  if (E <= 32) MOE_TOPK_CASE(1);
  if (E <= 64) MOE_TOPK_CASE(2);
  if (E <= 128) MOE_TOPK_CASE(4);
  if (E <= 256) MOE_TOPK_CASE(8);
  if (E <= 512) MOE_TOPK_CASE(16);
  MOE_TOPK_CASE(32);
#undef MOE_TOPK_CASE
}

}  // namespace moe
