// align_dev.cuh -- device pieces of the align (S2) shared by the align
// kernels and the fused routing kernel: a block-wide exclusive scan, the
// group layout (offsets, expert_ids, pads) and the stable scatter.
// Page "Mixture of Experts in vLLM - From First Principles to fused_moe",
// sections "Group by expert" and "The two index lists".
#pragma once

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kAlignThreads = 512;
constexpr int kAlignWarps = kAlignThreads / 32;

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
// entries of every group.  cnt/off hold whole-input counts and offsets.  With
// several CTAs holding the same counts, CTA `part` of `parts` writes the
// expert ids of every parts-th block and the pads of every parts-th expert.
__device__ void write_layout(const AlignSmem &s, int E, int B, int P, int total,
                             int32_t *sorted_ids, int32_t *expert_ids, int32_t *expert_offsets,
                             int32_t *n_post, int part = 0, int parts = 1) {
  const int tid = threadIdx.x;
  if (part == 0) {
    for (int e = tid; e < E; e += blockDim.x) expert_offsets[e] = s.off[e];
    if (tid == 0) {
      expert_offsets[E] = total;
      *n_post = total;
    }
  }
  // expert of block blk: the last expert whose group starts at or before blk*B
  for (int blk = part + parts * tid; blk < total / B; blk += parts * blockDim.x) {
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
  for (int e = part + parts * warp; e < E; e += parts * (blockDim.x / 32)) {
    const int c = s.cnt[e];
    const int padded = (c + B - 1) / B * B;
    for (int r = c + lane; r < padded; r += 32) sorted_ids[s.off[e] + r] = P;
  }
}

// topk_ids written earlier in the same kernel by other CTAs are read around L1.
template <bool kFromOtherCtas>
__device__ __forceinline__ int load_id(const int32_t *p) {
  return kFromOtherCtas ? __ldcg(p) : *p;
}

// Stable scatter of pairs [begin, end) using s.run as each expert's next slot.
// The id of a thread's pair in the next round is loaded before this round's
// barriers, so no round waits on a global load.
template <bool kFromOtherCtas = false>
__device__ void scatter_chunk(const AlignSmem &s, const int32_t *__restrict__ topk_ids, int begin,
                              int end, int E, int32_t *__restrict__ sorted_ids) {
  const int tid = threadIdx.x, warp = tid >> 5;
  int e_next = begin + tid < end ? load_id<kFromOtherCtas>(topk_ids + begin + tid) : -1;
  for (int base = begin; base < end; base += kAlignThreads) {
    const int p = base + tid;
    int e = e_next;
    if (p + kAlignThreads < end) e_next = load_id<kFromOtherCtas>(topk_ids + p + kAlignThreads);
    if (p >= end || e < 0 || e >= E) e = -1;
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

// The whole align in one CTA of kAlignThreads threads (smem: align_smem_bytes(E)).
template <bool kFromOtherCtas>
__device__ void align_one_cta(int *smem, const int32_t *__restrict__ topk_ids, int P, int E, int B,
                              int32_t *__restrict__ sorted_ids, int32_t *__restrict__ expert_ids,
                              int32_t *__restrict__ expert_offsets, int32_t *__restrict__ n_post,
                              int *status) {
  const AlignSmem s = carve(smem, E);
  const int tid = threadIdx.x;
  // up to one pair per thread: its expert id is loaded once and kept for the scatter
  const bool one_pass = P <= kAlignThreads;
  const int my_e = (one_pass && tid < P) ? load_id<kFromOtherCtas>(topk_ids + tid) : -1;
  for (int e = tid; e < E; e += blockDim.x) s.cnt[e] = 0;
  for (int i = tid; i < kAlignWarps * E; i += blockDim.x) s.wc[i] = 0;
  __syncthreads();
  bool bad = false;
  if (one_pass) {
    if (tid < P) {
      if (my_e >= 0 && my_e < E) atomicAdd(&s.cnt[my_e], 1);
      else bad = true;
    }
  } else {
#pragma unroll 4
    for (int p = tid; p < P; p += blockDim.x) {
      const int e = load_id<kFromOtherCtas>(topk_ids + p);
      if (e >= 0 && e < E) atomicAdd(&s.cnt[e], 1);
      else bad = true;
    }
  }
  if (bad) report_status(status, kStatusBadExpertId);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) s.off[e] = (s.cnt[e] + B - 1) / B * B;
  __syncthreads();
  const int total = block_exclusive_scan(s.off, E, s.misc);
  for (int e = tid; e < E; e += blockDim.x) s.run[e] = s.off[e];
  write_layout(s, E, B, P, total, sorted_ids, expert_ids, expert_offsets, n_post);
  __syncthreads();
  if (one_pass) {
    // the single tile of scatter_chunk, with the id already in hand
    const int warp = tid >> 5;
    const int e = (tid < P && my_e >= 0 && my_e < E) ? my_e : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lanemask_lt());
    if (e >= 0 && rank == 0) s.wc[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int prefix = 0;
      for (int w = 0; w < warp; ++w) prefix += s.wc[w * E + e];
      sorted_ids[s.run[e] + prefix + rank] = tid;
    }
  } else {
    scatter_chunk<kFromOtherCtas>(s, topk_ids, 0, P, E, sorted_ids);
  }
}

// The same layout from ONE warp, for small inputs (P <= 32 * kWarpAlignRounds
// pairs, E <= 1024): no block-wide barrier, ids read from `ids` (shared
// memory of this CTA).  Pairs are ranked within their expert in pair order
// (__match_any_sync per round of 32, counts carried across rounds), padded
// group starts come from a warp scan over the experts (E / 32 contiguous
// experts per lane), pads are written over the whole used range before the
// pairs (ordered by __syncwarp).  smem: 2 * E + 1 ints.
constexpr int kWarpAlignRounds = 8;

__device__ void align_one_warp(int *smem, const int32_t *ids, int P, int E, int B,
                               int32_t *__restrict__ sorted_ids, int32_t *__restrict__ expert_ids,
                               int32_t *__restrict__ expert_offsets, int32_t *__restrict__ n_post,
                               int *status) {
  const int lane = threadIdx.x & 31;
  int *cnt = smem, *off = smem + E;  // off: E + 1 entries
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  int my_e[kWarpAlignRounds], my_r[kWarpAlignRounds];
  bool bad = false;
#pragma unroll
  for (int r = 0; r < kWarpAlignRounds; ++r) {
    const int p = lane + 32 * r;
    int e = p < P ? ids[p] : -1;
    if (p < P && (e < 0 || e >= E)) {
      bad = true;
      e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const uint32_t before = peers & lanemask_lt();
    my_e[r] = e;
    my_r[r] = (e >= 0 ? cnt[e] : 0) + __popc(before);
    __syncwarp();  // every lane has read cnt before the group leaders add to it
    if (e >= 0 && before == 0) cnt[e] += __popc(peers);
    __syncwarp();
    if (32 * (r + 1) >= P) break;
  }
  if (bad) report_status(status, kStatusBadExpertId);
  // padded group starts: lane l scans experts [l * per, (l + 1) * per)
  const int per = (E + 31) / 32;
  const int e_lo = min(E, lane * per), e_hi = min(E, e_lo + per);
  int sum = 0;
  for (int e = e_lo; e < e_hi; ++e) sum += (cnt[e] + B - 1) / B * B;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  int run = incl - sum;
  for (int e = e_lo; e < e_hi; ++e) {
    off[e] = run;
    expert_offsets[e] = run;
    const int padded = (cnt[e] + B - 1) / B * B;
    for (int b = run / B; b < (run + padded) / B; ++b) expert_ids[b] = e;
    run += padded;
  }
  if (lane == 0) {
    expert_offsets[E] = total;
    *n_post = total;
  }
  for (int i = lane; i < total; i += 32) sorted_ids[i] = P;  // pads; the pairs overwrite theirs
  __syncwarp();
#pragma unroll
  for (int r = 0; r < kWarpAlignRounds; ++r) {
    if (my_e[r] >= 0) sorted_ids[off[my_e[r]] + my_r[r]] = lane + 32 * r;
    if (32 * (r + 1) >= P) break;
  }
}

inline size_t align_smem_bytes(int E) {
  return sizeof(int) * (3 * (size_t)E + kAlignWarps * E + kAlignWarps + 1);
}

}  // namespace
}  // namespace moe
