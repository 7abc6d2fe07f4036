// k_decode_layer.cu -- the whole layer (S0 .. S4) as ONE persistent kernel,
// for decode-sized batches.
//
// Page "MoE execution analysis" (vLLM port on ixformer), sections
// "Per-decode-step kernel launches" and "Memory allocation per step": a
// decode step of a 64-layer MoE model pays for six or more launches and
// three allocations per layer, while at decode sizes each routed expert sees
// about one token and the layer is bound by reading the chosen experts'
// weights from HBM.  Here one launch runs the layer; the steps are those of
// the page "Mixture of Experts in vLLM - From First Principles to
// fused_moe": the router ("One token uses only 8 experts"), softmax, top-k
// and renormalize (same section, steps 1-3), grouping the pairs by expert
// ("Group by expert"), GEMM 1 with SiLU(gate) * up ("An expert is a small
// SwiGLU MLP") and GEMM 2 with the router-weighted per-token sum ("Put the
// results back, and combine them per token").
//
// One CTA per SM, all resident at once (a cooperative launch).
//
//   router   each CTA computes the logits of its experts (E / G rows of W_r,
//            copied into shared memory before the kernel waits for the
//            previous one) for every token, from x staged in shared memory;
//            grid barrier (skipped when the logits are given).
//   routing  every CTA reads all M x E logits and runs softmax / top-k /
//            renormalize (one warp per token) and the grouping by expert on
//            its own, in shared memory: the same inputs and code give every
//            CTA the same experts and pair counts, so no barrier is needed.
//   weights  both GEMMs are laid out expert by expert: GEMM 1 as the D x I
//            (expert, channel) jobs -- gate row and up row, 2 x H bf16 --
//            and GEMM 2 as the D x H (expert, output channel) rows of W2,
//            I bf16 each; every CTA takes a contiguous range of each, so it
//            reads a few long contiguous stretches of weights.  Each warp
//            streams its rows with 16-byte loads, a whole job (or a batch of
//            W2 rows) in flight at once, and computes on CUDA cores (bf16
//            products, fp32 sums); a warp issues its first W2 rows before it
//            waits for the other CTAs' activations.
//   GEMM 1   a[p, i] = bf16(SiLU(bf16 gate) * bf16 up) to global memory; a
//            grid barrier once every CTA has written its part of a;
//   GEMM 2   each CTA stages the activations of the pairs its W2 rows need,
//            forms o = W2_e[n] . a_p and adds w_p * o into the fp32 combine
//            accumulator y_acc[t, n]; a grid barrier;
//   output   y = bf16(y_acc (+ residual)), each CTA a slice.
//
// The weights stream at decode sizes, where tensor cores would idle.  Every
// wait is bounded (about 1 s): a CTA that gives up records
// MOE_ERR_DEVICE_TIMEOUT and raises an abort flag, every CTA then skips to
// the exit (letting its own copies land first), and the last one out resets
// the grid-barrier counters for the next call (they live in the workspace's
// control block).
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "align_dev.cuh"
#include "route_dev.cuh"

namespace moe {

namespace {

constexpr int kDecThreads = kAlignThreads;  // 512: the block scan of align_dev.cuh
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kG1Cpl = 4;        // GEMM 1: 16-byte chunks per lane per piece (1024 bf16)
constexpr int kPairsPerPass = 4;  // pairs of one expert per pass over a row
constexpr uint32_t kMaxSmem = 227 * 1024;
// Cost model of the work split.  A CTA's streaming and its arithmetic
// overlap, so an item costs the larger of the two: a GEMM-1 job max(3, n)
// (its 4H bytes take about as long as three passes of the multiply-adds over
// them for one pair), a W2 row max(3, 2 n) in half units (its 2I bytes about
// one and a half passes); n = pairs of the item's expert.
constexpr int kJobFloor = 3, kRowFloor = 3, kRowPerPair = 2;
__host__ __device__ inline int job_cost(int n) { return n > kJobFloor ? n : kJobFloor; }
__host__ __device__ inline int row_cost(int n) { return kRowPerPair * n > kRowFloor ? kRowPerPair * n : kRowFloor; }

// control block ints in the workspace (after the fused routing counters)
constexpr int kDecBar = 0, kDecExit = 1, kDecAbort = 2;
// shared control ints
constexpr int kCtlJoin1 = 0, kCtlJoin2 = 1, kCtlAbort = 2, kCtlD = 3, kCtlInts = 8;
// A waiting thread looks at the global abort flag and the clock only this
// often: each look at the flag is a round trip to L2.
constexpr long long kCheckCycles = 8192;

__device__ __forceinline__ uint32_t dsmem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void dmbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void dmbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool dmbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Linear copy global -> this CTA's shared memory by the bulk-copy engine;
// completion counted on the barrier in bytes.  16-byte aligned, size a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_volatile(const int *p) { return *reinterpret_cast<const volatile int *>(p); }
__device__ __forceinline__ void st_volatile(int *p, int v) { *reinterpret_cast<volatile int *>(p) = v; }
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}


// a = bf16( SiLU(bf16(gate)) * bf16(up) ); the fast exponential and division
// stay far below the final bf16 rounding.
__device__ __forceinline__ uint16_t dec_silu_mul(float gate, float up) {
  const float gb = bf16_bits_to_float(float_to_bf16_bits(gate));
  const float ub = bf16_bits_to_float(float_to_bf16_bits(up));
  return float_to_bf16_bits(__fdividef(gb, 1.0f + __expf(-gb)) * ub);
}

struct DecodeArgs {
  const uint16_t *x, *w_router, *logits_in;
  const float *bias;
  const uint16_t *w13, *w2, *residual;
  int M, E, top_k, H, I, renormalize;
  uint16_t *y;
  int32_t *ids_out;
  float *wts_out;
  uint16_t *logits_buf;  // [M, E]: router output (unused with logits_in)
  uint16_t *a_buf;       // [M * top_k, I]: GEMM 1 -> GEMM 2
  float *y_acc;          // [M, H]: fp32 combine accumulator
  int *ctl;              // barrier counter, exit counter, abort flag (zero between calls)
  int *status;
  int wr_rows;           // W_r rows per CTA in shared memory (ceil(E / G))
  int a_rows;            // activation rows a CTA's GEMM-2 range may need
  long long wait_cycles; // bound of a wait
};

// Shared-memory layout, computed the same way on the host and the device.
struct DecLayout {
  uint32_t bars, ctl, region, wr, ids, wts, plist, pos, mask, cnt, dexp, doff, cost1, cost2, misc,
      total;
};

__host__ __device__ inline uint32_t dec_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline DecLayout dec_layout(int M, int E, int top_k, int H, int I, int wr_rows,
                                                int a_rows) {
  const uint32_t P = static_cast<uint32_t>(M) * top_k;
  DecLayout L;
  uint32_t o = 0;
  auto take = [&](uint32_t bytes, uint32_t align) {
    o = dec_up(o, align);
    const uint32_t at = o;
    o += bytes;
    return at;
  };
  L.bars = take(16, 16);                      // W_r copy, x copy
  L.ctl = take(4u * kCtlInts, 16);
  const uint32_t xb = static_cast<uint32_t>(M) * H * 2, ab = static_cast<uint32_t>(a_rows) * I * 2;
  L.region = take(xb > ab ? xb : ab, 128);    // x [M, H], then the GEMM-2 activations
  L.wr = take(static_cast<uint32_t>(wr_rows) * H * 2, 16);
  L.ids = take(4 * P, 16);
  L.wts = take(4 * P, 16);
  L.plist = take(4 * P, 16);                  // pairs grouped by expert
  L.pos = take(4 * P, 16);                    // a pair's rank inside its expert
  L.mask = take(4 * ((E + 31) / 32), 16);     // experts with at least one pair
  L.cnt = take(4 * static_cast<uint32_t>(E), 16);
  L.dexp = take(4 * (P + 1), 16);             // distinct expert d -> expert id
  L.doff = take(4 * (P + 1), 16);             // d -> first slot in plist
  L.cost1 = take(4 * (P + 1), 16);            // cost of GEMM-1 jobs of experts below d
  L.cost2 = take(4 * (P + 1), 16);            // cost of W2 rows of experts below d
  L.misc = take(4 * (kAlignWarps + 1 + 32), 16);  // scan scratch, per-word expert counts
  L.total = o;
  return L;
}

// Gives up a wait: true once another CTA raised the abort flag or the wait
// has lasted longer than the bound (then this thread raises it).
__device__ bool dec_give_up(long long t0, const DecodeArgs &A) {
  if (ld_volatile(A.ctl + kDecAbort) != 0) return true;
  if (clock64() - t0 > A.wait_cycles) {
    report_status(A.status, kStatusTimeout);
    atomicExch(A.ctl + kDecAbort, 1);
    return true;
  }
  return false;
}

// One thread: the `round`-th grid barrier of the call.  Adds this CTA to the
// counter and waits until every CTA has (round * G); false when a CTA gave up.
__device__ bool grid_arrive_wait(const DecodeArgs &A, int round) {
  __threadfence();  // (the CTA's writers fenced their own writes before this)
  atomicAdd(A.ctl + kDecBar, 1);
  const int target = round * static_cast<int>(gridDim.x);
  const long long t0 = clock64();
  long long next = t0 + kCheckCycles;
  while (ld_acquire_gpu(A.ctl + kDecBar) < target) {
    if (clock64() > next) {
      if (dec_give_up(t0, A)) return false;
      next = clock64() + kCheckCycles;
    }
  }
  return true;
}

// One thread, bounded wait for a barrier phase.
__device__ bool dec_wait_bar(uint32_t bar, uint32_t parity, const DecodeArgs &A) {
  if (dmbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  long long next = t0 + kCheckCycles;
  while (!dmbar_try_wait(bar, parity)) {
    if (clock64() > next) {
      if (dec_give_up(t0, A)) return false;
      next = clock64() + kCheckCycles;
    }
  }
  return true;
}

// One thread, bounded wait until a shared int reaches `want`.
__device__ bool dec_wait_smem(const int *p, int want, const DecodeArgs &A) {
  if (ld_volatile(p) >= want) return true;
  const long long t0 = clock64();
  long long next = t0 + kCheckCycles;
  while (ld_volatile(p) < want) {
    __nanosleep(16);
    if (clock64() > next) {
      if (dec_give_up(t0, A)) return false;
      next = clock64() + kCheckCycles;
    }
  }
  return true;
}

// C2: 16-byte chunks of a W2 row per lane (I <= 256 * C2); R2 W2 rows in
// flight per warp.
template <int VPL, int C2>
__global__ void __launch_bounds__(kDecThreads, 1) k_decode_layer(const __grid_constant__ DecodeArgs A) {
  constexpr int R2 = C2 <= 4 ? 4 : 3;
  extern __shared__ __align__(128) uint8_t dsm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int M = A.M, E = A.E, K = A.top_k, H = A.H, I = A.I;
  const int P = M * K;
  const DecLayout L = dec_layout(M, E, K, H, I, A.wr_rows, A.a_rows);
  const uint32_t bar_wr = dsmem_u32(dsm + L.bars), bar_x = bar_wr + 8;
  int *ctl = reinterpret_cast<int *>(dsm + L.ctl);
  uint16_t *region = reinterpret_cast<uint16_t *>(dsm + L.region);
  int *ids = reinterpret_cast<int *>(dsm + L.ids);
  float *wts = reinterpret_cast<float *>(dsm + L.wts);
  int *plist = reinterpret_cast<int *>(dsm + L.plist);
  int *pos = reinterpret_cast<int *>(dsm + L.pos);
  uint32_t *mask = reinterpret_cast<uint32_t *>(dsm + L.mask);
  int *cnt = reinterpret_cast<int *>(dsm + L.cnt);
  int *dexp = reinterpret_cast<int *>(dsm + L.dexp);
  int *doff = reinterpret_cast<int *>(dsm + L.doff);
  int *misc = reinterpret_cast<int *>(dsm + L.misc);
  int *cost1 = reinterpret_cast<int *>(dsm + L.cost1);
  int *cost2 = reinterpret_cast<int *>(dsm + L.cost2);
  int *wpre = misc + kAlignWarps + 1;  // [32] experts present below each mask word
  const bool router = A.logits_in == nullptr;
  const int n_wr = router ? max(0, min(A.wr_rows, (E - c + G - 1) / G)) : 0;  // experts c + G r
  const int hv = H / 8, iv = I / 8;  // 16-byte chunks of a row of W13 / of W2

  if (tid == 0) {
    dmbar_init(bar_wr, 1);
    dmbar_init(bar_x, 1);
    for (int i = 0; i < kCtlInts; ++i) ctl[i] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // the router rows do not depend on the previous kernel: copy them first
  if (tid == 0 && n_wr > 0) {
    dmbar_expect_tx(bar_wr, static_cast<uint32_t>(n_wr * H * 2));
    for (int r = 0; r < n_wr; ++r)
      bulk_g2s(dsmem_u32(dsm + L.wr + (size_t)r * H * 2), A.w_router + (size_t)(c + G * r) * H,
               H * 2, bar_wr);
  }
  griddep_wait();  // x, residual and the logits are the previous kernel's output
  griddep_launch_dependents();
  if (tid == 0) {
    dmbar_expect_tx(bar_x, static_cast<uint32_t>(M * H * 2));
    bulk_g2s(dsmem_u32(region), A.x, M * H * 2, bar_x);
  }
  const uint4 *xs = reinterpret_cast<const uint4 *>(region);

  // ------------------------------------------------------------ router
  if (tid == 0 && !((n_wr == 0 || dec_wait_bar(bar_wr, 0, A)) && dec_wait_bar(bar_x, 0, A)))
    ctl[kCtlAbort] = 1;
  __syncthreads();
  const int round = router ? 1 : 0;  // grid barriers before GEMM 1
  if (router) {
    if (ctl[kCtlAbort] == 0) {
      const uint4 *wrs = reinterpret_cast<const uint4 *>(dsm + L.wr);
      for (int job = warp; job < n_wr * M; job += kDecWarps) {
        const int r = job / M, t = job - r * M;
        float acc = 0.f;
        for (int ch = lane; ch < hv; ch += 32)
          acc = dot8_bf16(wrs[(size_t)r * hv + ch], xs[(size_t)t * hv + ch], acc);
        acc = warp_sum(acc);
        if (lane == 0) {
          const int e = c + G * r;
          if (A.bias != nullptr) acc += A.bias[e];
          A.logits_buf[(size_t)t * E + e] = float_to_bf16_bits(acc);
        }
      }
      __threadfence();
    }
    __syncthreads();
    if (tid == 0 && ctl[kCtlAbort] == 0 && !grid_arrive_wait(A, 1)) ctl[kCtlAbort] = 1;
    __syncthreads();
  }

  // ------------------------------------------------------------ routing
  if (ctl[kCtlAbort] == 0) {
    const uint16_t *lg = router ? A.logits_buf : A.logits_in;
    for (int t = warp; t < M; t += kDecWarps)
      topk_softmax_warp<VPL, true>(lg + (size_t)t * E, E, K, A.renormalize, ids + t * K,
                                   wts + t * K, lane);
    for (int e = tid; e < E; e += kDecThreads) cnt[e] = 0;
    for (int w = tid; w < (E + 31) / 32; w += kDecThreads) mask[w] = 0u;
    // this CTA's slice of the combine accumulator starts at zero
    const long mh = (long)M * H;
    // (each warp's fence before the GEMM-1 barrier makes the zeros visible)
    for (long v = (long)c * mh / G + tid; v < (long)(c + 1) * mh / G; v += kDecThreads) A.y_acc[v] = 0.f;
    __syncthreads();
    if (c == 0)
      for (int p = tid; p < P; p += kDecThreads) {
        A.ids_out[p] = ids[p];
        A.wts_out[p] = wts[p];
      }
    // grouping: experts present (a bit mask), pairs per expert, each pair's
    // rank inside its expert (the order inside an expert does not matter to y)
    for (int p = tid; p < P; p += kDecThreads) {
      const int e = ids[p];
      atomicOr(&mask[e >> 5], 1u << (e & 31));
      pos[p] = atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // distinct experts in ascending id: d(e) = experts present below e
    const int nw = (E + 31) / 32;
    if (warp == 0) {
      const int v = lane < nw ? __popc(mask[lane]) : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      wpre[lane] = incl - v;
      if (lane == 31) ctl[kCtlD] = incl;
    }
    __syncthreads();
    const int D = ctl[kCtlD];
    for (int e = tid; e < E; e += kDecThreads) {
      const uint32_t m = mask[e >> 5];
      if ((m >> (e & 31)) & 1u) {
        const int d = wpre[e >> 5] + __popc(m & ((1u << (e & 31)) - 1u));
        dexp[d] = e;
        doff[d] = cnt[e];
      }
    }
    __syncthreads();
    block_exclusive_scan(doff, D, misc);  // pair counts -> first slot of each expert
    if (tid == 0) doff[D] = P;
    __syncthreads();
    for (int p = tid; p < P; p += kDecThreads) {
      const int e = ids[p];
      const uint32_t m = mask[e >> 5];
      const int d = wpre[e >> 5] + __popc(m & ((1u << (e & 31)) - 1u));
      plist[doff[d] + pos[p]] = p;
    }
    __syncthreads();

    // this CTA's ranges, GEMM 1 jobs [j0, j1) of D * I and GEMM 2 rows [r0, r1)
    // of D * H, cut at equal cost: an expert's items cost more the more pairs
    // it has, so every CTA finishes at about the same time
    for (int d = tid; d < D; d += kDecThreads) {
      const int n = doff[d + 1] - doff[d];
      cost1[d] = I * job_cost(n);
      cost2[d] = H * row_cost(n);
    }
    __syncthreads();
    const int T1 = block_exclusive_scan(cost1, D, misc);
    const int T2 = block_exclusive_scan(cost2, D, misc);
    if (tid == 0) {
      cost1[D] = T1;
      cost2[D] = T2;
    }
    __syncthreads();
    // first item of CTA cc in a D x U list whose expert d costs cost[d + 1] - cost[d]
    auto cut = [&](const int *cost, int T, int U, bool rows, int cc) {
      const long x = (long)cc * T / G;
      int lo = 0, hi = D;  // the last d with cost[d] <= x
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cost[mid] <= x) lo = mid;
        else hi = mid - 1;
      }
      if (lo >= D) return D * U;
      const int n = doff[lo + 1] - doff[lo];
      const int per = rows ? row_cost(n) : job_cost(n);
      return lo * U + min(U, static_cast<int>((x - cost[lo]) / per));
    };
    const int j0 = cut(cost1, T1, I, false, c), j1 = cut(cost1, T1, I, false, c + 1);
    const int r0 = cut(cost2, T2, H, true, c), r1 = cut(cost2, T2, H, true, c + 1);
    // the pairs the GEMM-2 rows need: those of experts r0 / H .. (r1 - 1) / H
    const int w_base = r1 > r0 ? doff[r0 / H] : 0;
    const int n_win = r1 > r0 ? doff[(r1 - 1) / H + 1] - w_base : 0;

    // ---------------------------------------------------------- GEMM 1 + SiLU-and-mul
    // Warp w takes jobs j0 + w, j0 + w + 16, ...  A job is streamed in pieces
    // (kG1Cpl 16-byte chunks per lane of its gate row and of its up row,
    // 1024 bf16 of each) through two register buffers: the next piece's loads
    // are in flight while the current one is multiplied, so the warp always
    // has a piece on its way.  Experts with more than kPairsPerPass pairs take
    // one pass over the job per kPairsPerPass pairs.
    {
      const int nk = (hv + 32 * kG1Cpl - 1) / (32 * kG1Cpl);  // pieces per pass
      // the piece after (j, q0, k): the next K piece, the next pass, the next job
      auto advance = [&](int &j, int &q0, int &k) {
        if (++k < nk) return;
        k = 0;
        const int d = j / I;
        q0 += kPairsPerPass;
        if (q0 < doff[d + 1]) return;
        j += kDecWarps;
        q0 = j < j1 ? doff[j / I] : 0;
      };
      uint4 gb[2][kG1Cpl], ub[2][kG1Cpl];
      auto issue = [&](auto B, int j, int k) {
        constexpr int b = decltype(B)::value;
        if (j >= j1) return;
        const int d = j / I, i = j - d * I;
        const uint16_t *grow = A.w13 + ((size_t)dexp[d] * 2 * I + i) * H;
        const uint16_t *urow = grow + (size_t)I * H;
#pragma unroll
        for (int u = 0; u < kG1Cpl; ++u) {
          const int ch = k * 32 * kG1Cpl + u * 32 + lane;
          gb[b][u] = ch < hv ? ld_stream_16(grow + (size_t)ch * 8) : make_uint4(0, 0, 0, 0);
          ub[b][u] = ch < hv ? ld_stream_16(urow + (size_t)ch * 8) : make_uint4(0, 0, 0, 0);
        }
      };
      float ag[kPairsPerPass], au[kPairsPerPass];
#pragma unroll
      for (int q = 0; q < kPairsPerPass; ++q) ag[q] = au[q] = 0.f;
      // multiplies piece (j, q0, k) held in buffer B; after the last K piece
      // of a pass, forms a for the pass's pairs
      auto consume = [&](auto B, int j, int q0, int k) {
        constexpr int b = decltype(B)::value;
        const int d = j / I, i = j - d * I;
        const int nq = min(kPairsPerPass, doff[d + 1] - q0);
        int tok[kPairsPerPass];
#pragma unroll
        for (int q = 0; q < kPairsPerPass; ++q) tok[q] = q < nq ? plist[q0 + q] / K : 0;
#pragma unroll
        for (int u = 0; u < kG1Cpl; ++u) {
          const int ch = k * 32 * kG1Cpl + u * 32 + lane;
          if (ch < hv) {
#pragma unroll
            for (int q = 0; q < kPairsPerPass; ++q) {
              if (q < nq) {
                const uint4 xv = xs[(size_t)tok[q] * hv + ch];
                ag[q] = dot8_bf16(gb[b][u], xv, ag[q]);
                au[q] = dot8_bf16(ub[b][u], xv, au[q]);
              }
            }
          }
        }
        if (k == nk - 1) {
#pragma unroll
          for (int q = 0; q < kPairsPerPass; ++q) {
            if (q < nq) {  // (nq is the same in every lane)
              const float gs = warp_sum(ag[q]), us = warp_sum(au[q]);
              if (lane == q) A.a_buf[(size_t)plist[q0 + q] * I + i] = dec_silu_mul(gs, us);
            }
            ag[q] = au[q] = 0.f;
          }
        }
      };
      using B0 = std::integral_constant<int, 0>;
      using B1 = std::integral_constant<int, 1>;
      int cj = j0 + warp, cq = cj < j1 ? doff[cj / I] : 0, ck = 0;  // the piece in buffer 0
      issue(B0{}, cj, ck);
      while (cj < j1) {
        int nj = cj, nq0 = cq, nkk = ck;
        advance(nj, nq0, nkk);
        issue(B1{}, nj, nkk);
        consume(B0{}, cj, cq, ck);
        if (nj >= j1) break;
        cj = nj, cq = nq0, ck = nkk;
        advance(nj, nq0, nkk);
        issue(B0{}, nj, nkk);
        consume(B1{}, cj, cq, ck);
        cj = nj, cq = nq0, ck = nkk;
      }
    }

    // ---------------------------------------------------------- GEMM 2 + combine
    // The CTA's rows in groups of R2 consecutive rows (one expert, unless the
    // group crosses to the next); warp w takes groups w, w + 16, ...  For each
    // pair of the expert, the pair's activation is read once and dotted with
    // every row of the group (R2 independent sums).  A warp loads its first
    // group before it waits for the other CTAs' activations.
    uint4 wv[R2][C2];
    auto load_group = [&](int g) {
#pragma unroll
      for (int r = 0; r < R2; ++r) {
        const int row = r0 + g * R2 + r;
        const uint16_t *wrow = A.w2;
        if (row < r1) {
          const int d = row / H;
          wrow = A.w2 + ((size_t)dexp[d] * H + (row - d * H)) * I;
        }
#pragma unroll
        for (int u = 0; u < C2; ++u) {
          const int ch = u * 32 + lane;
          wv[r][u] = (row < r1 && ch < iv) ? ld_stream_16(wrow + (size_t)ch * 8) : make_uint4(0, 0, 0, 0);
        }
      }
    };
    const int n_groups = (r1 - r0 + R2 - 1) / R2;
    if (warp < n_groups) load_group(warp);
    // this warp's activations are visible GPU-wide before it counts itself in;
    // warp 0's first lane takes the CTA through the grid barrier
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(ctl + kCtlJoin1, 1);
    if (tid == 0) {
      const bool ok = ld_volatile(ctl + kCtlAbort) == 0 && dec_wait_smem(ctl + kCtlJoin1, kDecWarps, A) &&
                      grid_arrive_wait(A, round + 1);
      if (!ok) st_volatile(ctl + kCtlAbort, 1);
    }
    __syncthreads();
    if (ctl[kCtlAbort] == 0) {
      // the activations of the pairs this CTA's rows need (written by other CTAs)
      uint4 *aw = reinterpret_cast<uint4 *>(region);
      const uint4 *ag = reinterpret_cast<const uint4 *>(A.a_buf);
      for (int v = tid; v < n_win * iv; v += kDecThreads) {
        const int k = v / iv, ch = v - k * iv;
        aw[(size_t)k * iv + ch] = __ldcg(ag + (size_t)plist[w_base + k] * iv + ch);
      }
      __syncthreads();
      for (int g = warp; g < n_groups; g += kDecWarps) {
        if (g != warp) load_group(g);
        const int row0 = r0 + g * R2;
        const int d0 = row0 / H;
        const int dl = (min(row0 + R2, r1) - 1) / H;
        // the experts of the group's rows (one, or two at an expert boundary)
        for (int d = d0; d <= dl; ++d) {
          const int n0 = row0 - d * H;  // row r of the group is output channel n0 + r of expert d
          const int pb = doff[d], pe = doff[d + 1];
          for (int q = pb; q < pe; ++q) {
            uint4 av[C2];
#pragma unroll
            for (int u = 0; u < C2; ++u) {
              const int ch = u * 32 + lane;
              av[u] = ch < iv ? aw[(size_t)(q - w_base) * iv + ch] : make_uint4(0, 0, 0, 0);  // (smem)
            }
            float o[R2];
#pragma unroll
            for (int r = 0; r < R2; ++r) {
              o[r] = 0.f;
#pragma unroll
              for (int u = 0; u < C2; ++u) o[r] = dot8_bf16(wv[r][u], av[u], o[r]);
            }
#pragma unroll
            for (int r = 0; r < R2; ++r) o[r] = warp_sum(o[r]);
            const int p = plist[q];
            const float wp = wts[p];
#pragma unroll
            for (int r = 0; r < R2; ++r) {
              const int n = n0 + r;
              if (lane == r && row0 + r < r1 && n >= 0 && n < H)
                atomicAdd(A.y_acc + (size_t)(p / K) * H + n, wp * o[r]);
            }
          }
        }
      }
      // this warp's additions are visible GPU-wide before it counts itself
      // done; every CTA's GEMM 2 is in y_acc after the last grid barrier
      __threadfence();
      __syncwarp();
      if (lane == 0) atomicAdd(ctl + kCtlJoin2, 1);
      if (tid == 0) {
        const bool ok = dec_wait_smem(ctl + kCtlJoin2, kDecWarps, A) && grid_arrive_wait(A, round + 2);
        if (!ok) st_volatile(ctl + kCtlAbort, 1);
      }
    }
  }
  __syncthreads();

  // ------------------------------------------------------------ output
  if (ctl[kCtlAbort] == 0) {
    const long mh = (long)M * H;
    for (long v = (long)c * mh / G + tid; v < (long)(c + 1) * mh / G; v += kDecThreads) {
      float acc = __ldcg(A.y_acc + v);
      if (A.residual != nullptr) acc += bf16_bits_to_float(A.residual[v]);
      A.y[v] = float_to_bf16_bits(acc);
    }
  } else if (tid == 0) {
    atomicExch(A.ctl + kDecAbort, 1);
  }

  // ------------------------------------------------------------ exit
  // the last CTA out resets the grid-barrier counters for the next call
  // (every CTA gets here, also after a timeout)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(A.ctl + kDecExit, 1) == G - 1) {
      A.ctl[kDecBar] = 0;
      A.ctl[kDecAbort] = 0;
      __threadfence();
      A.ctl[kDecExit] = 0;
    }
  }
}

// SM clock of the current device in kHz, queried once per device (the query
// is far too slow for every launch); it converts the wait bound to cycles.
int sm_clock_khz() {
  static std::mutex m;
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(m);
  if (cached[dev] == 0) {
    int khz = 0;
    if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    cached[dev] = khz;
  }
  return cached[dev];
}

// Cooperative launch (all CTAs resident: the grid barriers need it) with
// programmatic dependent launch where the driver accepts the combination.
template <int VPL, int C2>
cudaError_t launch_decode_v(const DecodeArgs &args, int grid, size_t smem, cudaStream_t s) {
  const void *fn = reinterpret_cast<const void *>(k_decode_layer<VPL, C2>);
  cudaError_t err = ensure_smem_limit(fn, smem);
  if (err != cudaSuccess) return err;
  static int pdl_ok[64];  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  cudaGetDevice(&dev);
  const int slot = (dev >= 0 && dev < 64) ? dev : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  if (pdl_ok[slot] != 2) {
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, k_decode_layer<VPL, C2>, args);
    if (err == cudaSuccess) {
      pdl_ok[slot] = 1;
      return err;
    }
    if (pdl_ok[slot] == 1) return err;
    (void)cudaGetLastError();
    pdl_ok[slot] = 2;
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_layer<VPL, C2>, args);
}

// Whether one CTA of the decode kernel fits an SM with this shared memory
// (cached per device and size).
bool decode_fits(size_t smem) {
  static std::mutex m;
  static int cached[64];
  static size_t cached_smem[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(m);
  if (cached[dev] == 0 || cached_smem[dev] != smem) {
    // (every instantiation has the same resources; the limit must be raised
    // before the query)
    if (ensure_smem_limit(reinterpret_cast<const void *>(k_decode_layer<4, 4>), smem) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_layer<4, 4>, kDecThreads, smem) !=
        cudaSuccess) {
      (void)cudaGetLastError();
      per_sm = 0;
    }
    cached[dev] = per_sm >= 1 ? 1 : -1;
    cached_smem[dev] = smem;
  }
  return cached[dev] == 1;
}

struct DecPlan {
  int grid, wr_rows, a_rows;
  uint32_t smem;
};

// Sizes of one launch, or false where the kernel does not apply.
bool decode_plan(int M, int E, int top_k, int H, int I, DecPlan *plan) {
  if (M < 1 || E > kMaxExperts || top_k > kMaxTopK) return false;
  const long P = (long)M * top_k;
  if (P > 512) return false;
  if (I > 256 * 6) return false;  // a W2 row in one pass of a warp's registers
  DecPlan p;
  p.grid = num_sms();
  p.wr_rows = (E + p.grid - 1) / p.grid;
  // A CTA's GEMM-2 rows are consecutive rows of the D x H expert-major list,
  // cut at equal cost (total at most H (3 D + 2 P) <= 5 H P, D <= P) with a
  // row costing at least 3: at most 5 H P / (3 G) + 1 rows, touching at most
  // ceil(len / H) + 1 experts, each with at most M pairs.
  const long len = (5 * P * H + 3 * p.grid - 1) / (3 * p.grid) + 1;
  const long span = (len + H - 1) / H + 1;
  p.a_rows = static_cast<int>(std::min<long>(P, span * M));
  p.smem = dec_layout(M, E, top_k, H, I, p.wr_rows, p.a_rows).total;
  if (p.smem > kMaxSmem) return false;
  *plan = p;
  return true;
}

}  // namespace

bool decode_layer_supports(int M, int E, int top_k, int H, int I) {
  DecPlan p;
  return decode_plan(M, E, top_k, H, I, &p);
}

cudaError_t launch_decode_layer(const uint16_t *x, const uint16_t *w_router,
                                const uint16_t *logits_in, const float *bias,
                                const uint16_t *w13, const uint16_t *w2,
                                const uint16_t *residual, int M, int E, int top_k, int H, int I,
                                int renormalize, uint16_t *y, int32_t *ids_out, float *wts_out,
                                uint16_t *logits_buf, uint16_t *a_buf, float *y_acc, int *ctl,
                                int *status, cudaStream_t s) {
  DecPlan plan;
  if (!decode_plan(M, E, top_k, H, I, &plan)) return cudaErrorInvalidValue;
  if (!decode_fits(plan.smem)) return cudaErrorInvalidConfiguration;
  const int khz = sm_clock_khz();
  if (khz <= 0) return cudaErrorInvalidValue;
  DecodeArgs a{};
  a.x = x;
  a.w_router = w_router;
  a.logits_in = logits_in;
  a.bias = bias;
  a.w13 = w13;
  a.w2 = w2;
  a.residual = residual;
  a.M = M;
  a.E = E;
  a.top_k = top_k;
  a.H = H;
  a.I = I;
  a.renormalize = renormalize;
  a.y = y;
  a.ids_out = ids_out;
  a.wts_out = wts_out;
  a.logits_buf = logits_buf;
  a.a_buf = a_buf;
  a.y_acc = y_acc;
  a.ctl = ctl;
  a.status = status;
  a.wr_rows = plan.wr_rows;
  a.a_rows = plan.a_rows;
  a.wait_cycles = static_cast<long long>(khz) * 1000;  // about 1 s
  const bool wide = I > 256 * 4;
#define MOE_DEC_CASE(V)                                                              \
  return wide ? launch_decode_v<V, 6>(a, plan.grid, plan.smem, s)                    \
              : launch_decode_v<V, 4>(a, plan.grid, plan.smem, s)
  switch (topk_vpl(E)) {
    case 1: MOE_DEC_CASE(1);
    case 2: MOE_DEC_CASE(2);
    case 4: MOE_DEC_CASE(4);
    case 8: MOE_DEC_CASE(8);
    case 16: MOE_DEC_CASE(16);
    default: MOE_DEC_CASE(32);
  }
#undef MOE_DEC_CASE
}

}  // namespace moe
