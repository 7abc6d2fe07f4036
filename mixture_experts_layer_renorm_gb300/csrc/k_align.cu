// k_align.cu -- S2: group the (token, expert) pairs by expert, block-padded.
//
// Page "Mixture of Experts in vLLM - From First Principles to fused_moe",
// sections "Group by expert" and "The two index lists": sorted_token_ids holds
// the pair ids grouped by expert, each group padded with the id M*top_k to a
// multiple of BLOCK_SIZE_M; expert_ids holds one expert per block.
//
// Method: a counting sort.  Count pairs per expert (shared-memory atomics;
// a count does not depend on the order of the additions), pad the counts,
// exclusive-scan them into group offsets, then scatter every pair to
// offset + (number of earlier pairs with the same expert).  That rank is
// computed without atomics -- __match_any_sync within a warp and a per-warp
// count table across warps -- so the scatter is stable: ascending pair id
// inside each group, bit-reproducible from run to run.
//
// Small inputs run as one CTA.  Large inputs run as two kernels: per-chunk
// histograms, then a scan + scatter in which every CTA derives its own
// starting positions from the histogram table.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kAlignThreads = 512;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kAlignChunk = 2048;          // pairs per CTA in the multi-CTA path
constexpr int kAlignSingleMax = 16384;     // up to this many pairs: one CTA

// Exclusive scan of v[0..n) (n <= 2 * kAlignThreads) in place; returns the total.
__device__ int block_exclusive_scan(int *v, int n, int *warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = 2 * tid;
  const int a = i0 < n ? v[i0] : 0;
  const int b = i0 + 1 < n ? v[i0 + 1] : 0;
  int incl = a + b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kAlignWarps ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    if (lane < kAlignWarps) warp_tot[lane] = wi - w;  // exclusive warp base
    if (lane == kAlignWarps - 1) warp_tot[kAlignWarps] = wi;
  }
  __syncthreads();
  const int excl = warp_tot[warp] + incl - (a + b);
  if (i0 < n) v[i0] = excl;
  if (i0 + 1 < n) v[i0 + 1] = excl + a;
  const int total = warp_tot[kAlignWarps];
  __syncthreads();
  return total;
}

// Shared state of one align CTA.
struct AlignSmem {
  int *cnt;   // [E]  pairs per expert (this CTA's chunk, or the whole input)
  int *off;   // [E]  padded group start
  int *run;   // [E]  next free slot of each expert for this CTA
  int *wc;    // [kAlignWarps * E] per-warp counts of the current tile
  int *misc;  // [kAlignWarps + 1] scan scratch
};

__device__ AlignSmem carve(int *smem, int E) {
  AlignSmem s;
  s.cnt = smem;
  s.off = s.cnt + E;
  s.run = s.off + E;
  s.wc = s.run + E;
  s.misc = s.wc + kAlignWarps * E;
  return s;
}

// Writes expert_offsets, n_post, expert_ids of every real block and the pad
// entries of every group.  cnt/off hold whole-input counts and offsets.
__device__ void write_layout(const AlignSmem &s, int E, int B, int P, int total,
                             int32_t *sorted_ids, int32_t *expert_ids, int32_t *expert_offsets,
                             int32_t *n_post) {
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) expert_offsets[e] = s.off[e];
  if (tid == 0) {
    expert_offsets[E] = total;
    *n_post = total;
  }
  // expert of block blk: the last expert whose group starts at or before blk*B
  for (int blk = tid; blk < total / B; blk += blockDim.x) {
    const int pos = blk * B;
    int lo = 0, hi = E;  // first e with off[e] > pos, minus one
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s.off[mid] <= pos) lo = mid + 1;
      else hi = mid;
    }
    expert_ids[blk] = lo - 1;
  }
  const int warp = tid >> 5, lane = tid & 31;
  for (int e = warp; e < E; e += blockDim.x / 32) {
    const int c = s.cnt[e];
    const int padded = (c + B - 1) / B * B;
    for (int r = c + lane; r < padded; r += 32) sorted_ids[s.off[e] + r] = P;
  }
}

// Stable scatter of pairs [begin, end) using s.run as each expert's next slot.
__device__ void scatter_chunk(const AlignSmem &s, const int32_t *__restrict__ topk_ids, int begin,
                              int end, int E, int32_t *__restrict__ sorted_ids) {
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int base = begin; base < end; base += kAlignThreads) {
    const int p = base + tid;
    int e = -1;
    if (p < end) {
      e = topk_ids[p];
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lanemask_lt());
    const bool leader = rank == 0;
    if (e >= 0 && leader) s.wc[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int prefix = 0;
      for (int w = 0; w < warp; ++w) prefix += s.wc[w * E + e];
      sorted_ids[s.run[e] + prefix + rank] = p;
    }
    __syncthreads();
    if (e >= 0 && leader) {
      atomicAdd(&s.run[e], __popc(peers));
      s.wc[warp * E + e] = 0;
    }
    __syncthreads();
  }
}

// One CTA does the whole align.
__global__ void __launch_bounds__(kAlignThreads)
k_align_single(const int32_t *__restrict__ topk_ids, int P, int E, int B,
               int32_t *__restrict__ sorted_ids, int32_t *__restrict__ expert_ids,
               int32_t *__restrict__ expert_offsets, int32_t *__restrict__ n_post, int *status) {
  extern __shared__ int smem[];
  const AlignSmem s = carve(smem, E);
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) s.cnt[e] = 0;
  for (int i = tid; i < kAlignWarps * E; i += blockDim.x) s.wc[i] = 0;
  __syncthreads();
  bool bad = false;
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = topk_ids[p];
    if (e >= 0 && e < E) atomicAdd(&s.cnt[e], 1);
    else bad = true;
  }
  if (bad) report_status(status, kStatusBadExpertId);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) s.off[e] = (s.cnt[e] + B - 1) / B * B;
  __syncthreads();
  const int total = block_exclusive_scan(s.off, E, s.misc);
  for (int e = tid; e < E; e += blockDim.x) s.run[e] = s.off[e];
  write_layout(s, E, B, P, total, sorted_ids, expert_ids, expert_offsets, n_post);
  __syncthreads();
  scatter_chunk(s, topk_ids, 0, P, E, sorted_ids);
}

// Multi-CTA, pass 1: histogram of chunk c into hist[c * E + e].
__global__ void __launch_bounds__(kAlignThreads)
k_align_count(const int32_t *__restrict__ topk_ids, int P, int E, int32_t *__restrict__ hist,
              int *status) {
  extern __shared__ int smem[];
  int *cnt = smem;
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int begin = blockIdx.x * kAlignChunk;
  const int end = min(P, begin + kAlignChunk);
  bool bad = false;
  for (int p = begin + tid; p < end; p += blockDim.x) {
    const int e = topk_ids[p];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else bad = true;
  }
  if (bad) report_status(status, kStatusBadExpertId);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = cnt[e];
}

// Multi-CTA, pass 2: every CTA sums the histogram table (whole-input counts
// and the counts of the chunks before its own), scans the padded counts, and
// scatters its chunk.  CTA 0 also writes offsets, expert_ids and pads.
__global__ void __launch_bounds__(kAlignThreads)
k_align_scatter(const int32_t *__restrict__ topk_ids, int P, int E, int B,
                const int32_t *__restrict__ hist, int32_t *__restrict__ sorted_ids,
                int32_t *__restrict__ expert_ids, int32_t *__restrict__ expert_offsets,
                int32_t *__restrict__ n_post) {
  extern __shared__ int smem[];
  const AlignSmem s = carve(smem, E);
  const int tid = threadIdx.x;
  const int c = blockIdx.x, C = gridDim.x;
  for (int i = tid; i < kAlignWarps * E; i += blockDim.x) s.wc[i] = 0;
  for (int e = tid; e < E; e += blockDim.x) {
    int tot = 0, before = 0;
    for (int cc = 0; cc < C; ++cc) {
      const int v = hist[(size_t)cc * E + e];
      tot += v;
      if (cc < c) before += v;
    }
    s.cnt[e] = tot;
    s.run[e] = before;
    s.off[e] = (tot + B - 1) / B * B;
  }
  __syncthreads();
  const int total = block_exclusive_scan(s.off, E, s.misc);
  for (int e = tid; e < E; e += blockDim.x) s.run[e] += s.off[e];
  if (c == 0) write_layout(s, E, B, P, total, sorted_ids, expert_ids, expert_offsets, n_post);
  __syncthreads();
  const int begin = c * kAlignChunk;
  scatter_chunk(s, topk_ids, begin, min(P, begin + kAlignChunk), E, sorted_ids);
}

size_t align_smem_bytes(int E) { return sizeof(int) * (3 * (size_t)E + kAlignWarps * E + kAlignWarps + 1); }

}  // namespace

int align_num_ctas(long P) {
  if (P <= kAlignSingleMax) return 1;
  return static_cast<int>((P + kAlignChunk - 1) / kAlignChunk);
}

long align_hist_entries(long P, int E) {
  const int C = align_num_ctas(P);
  return C > 1 ? static_cast<long>(C) * E : 0;
}

cudaError_t launch_align(const int32_t *topk_ids, int P, int E, int B, int cap,
                         int32_t *sorted_ids, int32_t *expert_ids, int32_t *expert_offsets,
                         int32_t *n_post, int32_t *hist, int *status, cudaStream_t s) {
  (void)cap;
  const size_t smem = align_smem_bytes(E);
  static bool attr_done = false;
  if (!attr_done) {
    cudaFuncSetAttribute(k_align_single, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    cudaFuncSetAttribute(k_align_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    attr_done = true;
  }
  const int C = align_num_ctas(P);
  if (C == 1) {
    k_align_single<<<1, kAlignThreads, smem, s>>>(topk_ids, P, E, B, sorted_ids, expert_ids,
                                                  expert_offsets, n_post, status);
    return cudaGetLastError();
  }
  k_align_count<<<C, kAlignThreads, sizeof(int) * E, s>>>(topk_ids, P, E, hist, status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  k_align_scatter<<<C, kAlignThreads, smem, s>>>(topk_ids, P, E, B, hist, sorted_ids, expert_ids,
                                                 expert_offsets, n_post);
  return cudaGetLastError();
}

}  // namespace moe
