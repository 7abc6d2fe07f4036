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
  __shared__ int32_t ids_s[TOK * kMaxTopK];  // one token group: the ids for the grouping
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
                                 topk_ids + (size_t)t * top_k, topk_w + (size_t)t * top_k, lane,
                                 n_g == 1 ? ids_s + warp * top_k : nullptr);
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
  // ---- the align over every pair, in this one CTA (one warp when the
  // batch is one token group: its ids are in shared memory)
  if (n_g == 1 && M * top_k <= 32 * kWarpAlignRounds) {
    if (warp == 0)
      align_one_warp(reinterpret_cast<int *>(smem), ids_s, M * top_k, E, B, sorted_ids,
                     expert_ids, expert_offsets, n_post, status);
    return;
  }
  align_one_cta<true>(reinterpret_cast<int *>(smem), topk_ids, M * top_k, E, B, sorted_ids,
                      expert_ids, expert_offsets, n_post, status);
}

// ---------------------------------------------------------------- one token group, one cluster
// Decode batches (M <= 8) with router weights: the CTAs of one thread-block
// cluster (up to 8) each compute the logits of E / n experts for every token
// and write them, besides the logits buffer, straight into the shared memory
// of the cluster's first CTA; one cluster barrier (release / acquire) then
// hands the complete logits over, with no global fence, counter or read-back
// between the router and top-k.  The first CTA runs top-k (its ids kept in
// shared memory for the grouping) and the grouping; the others clear the
// combine accumulator and leave.  The cluster barrier is a hardware barrier
// that every thread of every CTA reaches exactly once.
constexpr int kSmallMaxCluster = 8;
constexpr int kSmallMaxE = 256;        // experts per CTA <= 32: two per warp at most
constexpr int kSmallMaxTok = 8;

__device__ __forceinline__ void cluster_barrier_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// 16-bit store into the shared memory of CTA `rank` of the cluster, at the
// offset of `local` in this CTA.
__device__ __forceinline__ void st_cluster_u16(const void *local, uint32_t rank, uint16_t v) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(remote), "h"(v) : "memory");
}

template <int VPL, int TOK>
__global__ void __launch_bounds__(kFusedThreads)
k_route_small(const uint16_t *__restrict__ x, const uint16_t *__restrict__ w_router,
              const float *__restrict__ bias, int M, int E, int H, int top_k, int renormalize,
              int B, uint16_t *__restrict__ logits_ws, int32_t *__restrict__ topk_ids,
              float *__restrict__ topk_w, int32_t *__restrict__ sorted_ids,
              int32_t *__restrict__ expert_ids, int32_t *__restrict__ expert_offsets,
              int32_t *__restrict__ n_post, int *status, float4 *__restrict__ zero_buf,
              long zero_n4, int skip_sort) {
  // x is the previous kernel's output, and the previous layer may still read
  // the accumulator this kernel clears
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint16_t lg_s[TOK * kSmallMaxE];      // the first CTA's copy of every logit
  __shared__ int32_t ids_s[TOK * kMaxTopK];
  const int nc = gridDim.x, h = blockIdx.x;       // one cluster: the block index is its rank
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int epc = (E + nc - 1) / nc;
  const int e0 = h * epc, e1 = min(E, e0 + epc);
  uint4 *xs = reinterpret_cast<uint4 *>(smem);
  // ---- logits: warp w takes experts e0 + w and (E > 128: more than 16
  // experts per CTA) e0 + w + 16; lanes split each K chunk
  constexpr bool kTwo = VPL >= 8;  // E > 128
  const int ea = e0 + warp, eb = e0 + warp + kFusedWarps;
  const bool has_a = ea < e1, has_b = kTwo && eb < e1;
  float acc_a[TOK], acc_b[TOK];
#pragma unroll
  for (int j = 0; j < TOK; ++j) acc_a[j] = acc_b[j] = 0.f;
  constexpr int kChunkV = kFusedKChunk / 8;       // 16-byte columns per chunk
  constexpr int kPerLane = kChunkV / 32;
  for (int kc = 0; kc < H; kc += kFusedKChunk) {
    const int vrow = min(kFusedKChunk, H - kc) / 8;
    // the router rows' loads go out before x is staged
    uint4 wa[kPerLane], wb[kPerLane];
#pragma unroll
    for (int u = 0; u < kPerLane; ++u) {
      const int c = lane + 32 * u;
      wa[u] = (has_a && c < vrow) ? ld_stream_16(w_router + (size_t)ea * H + kc + c * 8) : make_uint4(0, 0, 0, 0);
      if (kTwo) wb[u] = (has_b && c < vrow) ? ld_stream_16(w_router + (size_t)eb * H + kc + c * 8) : make_uint4(0, 0, 0, 0);
    }
    // x of this chunk: every load is issued before any store
    constexpr int kStage = (TOK * kChunkV + kFusedThreads - 1) / kFusedThreads;
    uint4 xv[kStage];
#pragma unroll
    for (int it = 0; it < kStage; ++it) {
      const int v = tid + it * kFusedThreads;
      const int r = v / kChunkV, c = v - r * kChunkV;
      xv[it] = (r < M && c < vrow) ? *reinterpret_cast<const uint4 *>(x + (size_t)r * H + kc + c * 8)
                                   : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();  // the previous chunk's readers of xs are done
#pragma unroll
    for (int it = 0; it < kStage; ++it) {
      const int v = tid + it * kFusedThreads;
      if (v < TOK * kChunkV) xs[v] = xv[it];
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kPerLane; ++u) {
      const int c = lane + 32 * u;
      if (c < vrow) {
#pragma unroll
        for (int j = 0; j < TOK; ++j) {
          const uint4 xv = xs[j * kChunkV + c];
          acc_a[j] = dot8_bf16(wa[u], xv, acc_a[j]);
          if (kTwo) acc_b[j] = dot8_bf16(wb[u], xv, acc_b[j]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < TOK; ++j) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc_a[j] += __shfl_xor_sync(0xffffffffu, acc_a[j], o);
      if (kTwo) acc_b[j] += __shfl_xor_sync(0xffffffffu, acc_b[j], o);
    }
  }
  // lane j writes token j's logits (rounded to bf16) here and to the first CTA
#pragma unroll
  for (int j = 0; j < TOK; ++j) {
    if (lane == j && j < M) {
      if (has_a) {
        const uint16_t b = float_to_bf16_bits(acc_a[j] + (bias != nullptr ? bias[ea] : 0.f));
        logits_ws[(size_t)j * E + ea] = b;
        st_cluster_u16(&lg_s[j * kSmallMaxE + ea], 0, b);
      }
      if (has_b) {
        const uint16_t b = float_to_bf16_bits(acc_b[j] + (bias != nullptr ? bias[eb] : 0.f));
        logits_ws[(size_t)j * E + eb] = b;
        st_cluster_u16(&lg_s[j * kSmallMaxE + eb], 0, b);
      }
    }
  }
  cluster_barrier_sync();  // every logit is in the first CTA's shared memory
  // side task: the combine accumulator, cleared by the CTAs other than the first
  if (zero_buf != nullptr && (h > 0 || nc == 1)) {
    const int nz = nc > 1 ? nc - 1 : 1, iz = nc > 1 ? h - 1 : 0;
    for (long i = (long)iz * kFusedThreads + tid; i < zero_n4; i += (long)nz * kFusedThreads)
      zero_buf[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (h > 0) return;
  // ---- softmax / top-k / renormalize, one warp per token
  if (warp < M)
    topk_softmax_warp<VPL, false>(lg_s + warp * kSmallMaxE, E, top_k, renormalize,
                                  topk_ids + (size_t)warp * top_k, topk_w + (size_t)warp * top_k,
                                  lane, ids_s + warp * top_k);
  __syncthreads();
  const int P = M * top_k;
  if (skip_sort) {
    // small batch: block p holds pair p alone (vLLM blog, "Small batches skip the sort")
    for (int i = tid; i < P * B; i += kFusedThreads) {
      const int p = i / B, r = i - p * B;
      sorted_ids[i] = r == 0 ? p : P;
      if (r == 0) expert_ids[p] = ids_s[p];
    }
    if (tid == 0) *n_post = P * B;
    return;
  }
  if (warp == 0)
    align_one_warp(reinterpret_cast<int *>(smem), ids_s, P, E, B, sorted_ids, expert_ids,
                   expert_offsets, n_post, status);
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

bool route_small_supports(int M, int E, int H, const void *logits_in) {
  return logits_in == nullptr && M >= 1 && M <= kSmallMaxTok && E <= kSmallMaxE && H % 8 == 0;
}

template <int VPL, int TOK>
cudaError_t launch_small_vt(int nc, size_t smem, const uint16_t *x, const uint16_t *w_router,
                            const float *bias, int M, int E, int H, int top_k, int renormalize,
                            int B, uint16_t *logits_ws, int32_t *topk_ids, float *topk_w,
                            int32_t *sorted_ids, int32_t *expert_ids, int32_t *expert_offsets,
                            int32_t *n_post, int *status, float4 *zb, long zn4, int skip_sort,
                            cudaStream_t s) {
  const void *fn = reinterpret_cast<const void *>(k_route_small<VPL, TOK>);
  cudaError_t err = ensure_smem_limit(fn, smem);
  if (err != cudaSuccess) return err;
  return launch_pdl_cluster(k_route_small<VPL, TOK>, dim3(nc), dim3(kFusedThreads), smem, s,
                            static_cast<unsigned>(nc), x, w_router, bias, M, E, H, top_k,
                            renormalize, B, logits_ws, topk_ids, topk_w, sorted_ids, expert_ids,
                            expert_offsets, n_post, status, zb, zn4, skip_sort);
}

template <int VPL>
cudaError_t launch_small_v(int tok, int nc, size_t smem, const uint16_t *x,
                           const uint16_t *w_router, const float *bias, int M, int E, int H,
                           int top_k, int renormalize, int B, uint16_t *logits_ws,
                           int32_t *topk_ids, float *topk_w, int32_t *sorted_ids,
                           int32_t *expert_ids, int32_t *expert_offsets, int32_t *n_post,
                           int *status, float4 *zb, long zn4, int skip_sort, cudaStream_t s) {
#define MOE_SMALL_TOK(T)                                                                       \
  return launch_small_vt<VPL, T>(nc, smem, x, w_router, bias, M, E, H, top_k, renormalize, B,  \
                                 logits_ws, topk_ids, topk_w, sorted_ids, expert_ids,          \
                                 expert_offsets, n_post, status, zb, zn4, skip_sort, s)
  switch (tok) {
    case 1: MOE_SMALL_TOK(1);
    case 2: MOE_SMALL_TOK(2);
    case 4: MOE_SMALL_TOK(4);
    default: MOE_SMALL_TOK(8);
  }
#undef MOE_SMALL_TOK
}

cudaError_t launch_route_fused(const uint16_t *x, const uint16_t *w_router, const float *bias,
                               const uint16_t *logits_in, int M, int E, int H, int top_k,
                               int renormalize, int B, uint16_t *logits_ws, int32_t *topk_ids,
                               float *topk_w, int32_t *sorted_ids, int32_t *expert_ids,
                               int32_t *expert_offsets, int32_t *n_post, int *counters,
                               int *status, float *zero_buf, long zero_n, bool skip_sort,
                               cudaStream_t s) {
  const int tok = fused_tok(M);
  if (route_small_supports(M, E, H, logits_in)) {
    // one token group: the cluster kernel (up to 8 CTAs of at most 32 experts)
    const int nc = std::min(kSmallMaxCluster, (E + 15) / 16);
    const size_t smem = std::max(sizeof(uint16_t) * tok * kFusedKChunk, align_smem_bytes(E));
    float4 *zb = reinterpret_cast<float4 *>(zero_buf);
    const long zn4 = zero_buf != nullptr ? zero_n / 4 : 0;
#define MOE_SMALL_CASE(V)                                                                         \
  return launch_small_v<V>(tok, nc, smem, x, w_router, bias, M, E, H, top_k, renormalize, B,      \
                           logits_ws, topk_ids, topk_w, sorted_ids, expert_ids, expert_offsets,   \
                           n_post, status, zb, zn4, skip_sort ? 1 : 0, s)
    switch (topk_vpl(E)) {
      case 1: MOE_SMALL_CASE(1);
      case 2: MOE_SMALL_CASE(2);
      case 4: MOE_SMALL_CASE(4);
      default: MOE_SMALL_CASE(8);
    }
#undef MOE_SMALL_CASE
  }
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
