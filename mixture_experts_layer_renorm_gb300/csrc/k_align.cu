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
#include "align_dev.cuh"

namespace moe {

namespace {

constexpr int kAlignChunk = 2048;          // pairs per CTA in the multi-CTA path
constexpr int kAlignSingleMax = 2048;      // up to this many pairs: one CTA

// One CTA does the whole align.
__global__ void __launch_bounds__(kAlignThreads)
k_align_single(const int32_t *__restrict__ topk_ids, int P, int E, int B,
               int32_t *__restrict__ sorted_ids, int32_t *__restrict__ expert_ids,
               int32_t *__restrict__ expert_offsets, int32_t *__restrict__ n_post, int *status) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ int smem[];
  align_one_cta<false>(smem, topk_ids, P, E, B, sorted_ids, expert_ids, expert_offsets, n_post,
                       status);
}

// Multi-CTA, pass 1: histogram of chunk c into hist[c * E + e].
__global__ void __launch_bounds__(kAlignThreads)
k_align_count(const int32_t *__restrict__ topk_ids, int P, int E, int32_t *__restrict__ hist,
              int *status) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ int smem[];
  int *cnt = smem;
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int begin = blockIdx.x * kAlignChunk;
  const int end = min(P, begin + kAlignChunk);
  bool bad = false;
#pragma unroll 4
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
// and the counts of the chunks before its own; all threads over the whole
// table, added up with shared-memory atomics), scans the padded counts, and
// scatters its chunk.  CTA 0 also writes offsets, expert_ids and pads.
__global__ void __launch_bounds__(kAlignThreads)
k_align_scatter(const int32_t *__restrict__ topk_ids, int P, int E, int B,
                const int32_t *__restrict__ hist, int32_t *__restrict__ sorted_ids,
                int32_t *__restrict__ expert_ids, int32_t *__restrict__ expert_offsets,
                int32_t *__restrict__ n_post) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ int smem[];
  const AlignSmem s = carve(smem, E);
  const int tid = threadIdx.x;
  const int c = blockIdx.x, C = gridDim.x;
  for (int i = tid; i < kAlignWarps * E; i += blockDim.x) s.wc[i] = 0;
  for (int e = tid; e < E; e += blockDim.x) {
    s.cnt[e] = 0;
    s.run[e] = 0;
  }
  __syncthreads();
  // sixteen table entries per thread in flight at once, then their sums
  const int n_hist = C * E;
  for (int i0 = tid; i0 < n_hist; i0 += 16 * kAlignThreads) {
    int v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = i0 + u * kAlignThreads;
      v[u] = i < n_hist ? hist[i] : 0;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = i0 + u * kAlignThreads;
      if (v[u] != 0) {
        atomicAdd(&s.cnt[i % E], v[u]);
        if (i < c * E) atomicAdd(&s.run[i % E], v[u]);  // a chunk before this CTA's
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) s.off[e] = (s.cnt[e] + B - 1) / B * B;
  __syncthreads();
  const int total = block_exclusive_scan(s.off, E, s.misc);
  for (int e = tid; e < E; e += blockDim.x) s.run[e] += s.off[e];
  write_layout(s, E, B, P, total, sorted_ids, expert_ids, expert_offsets, n_post, c, C);
  __syncthreads();
  const int begin = c * kAlignChunk;
  scatter_chunk(s, topk_ids, begin, min(P, begin + kAlignChunk), E, sorted_ids);
}

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
  cudaError_t attr = ensure_smem_limit(reinterpret_cast<const void *>(k_align_single), 96 * 1024);
  if (attr == cudaSuccess)
    attr = ensure_smem_limit(reinterpret_cast<const void *>(k_align_scatter), 96 * 1024);
  if (attr != cudaSuccess) return attr;
  const int C = align_num_ctas(P);
  if (C == 1) {
    return launch_pdl(k_align_single, dim3(1), dim3(kAlignThreads), smem, s, topk_ids, P, E, B,
                      sorted_ids, expert_ids, expert_offsets, n_post, status);
  }
  cudaError_t err = launch_pdl(k_align_count, dim3(C), dim3(kAlignThreads), sizeof(int) * E, s,
                               topk_ids, P, E, hist, status);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_align_scatter, dim3(C), dim3(kAlignThreads), smem, s, topk_ids, P, E, B,
                    static_cast<const int32_t *>(hist), sorted_ids, expert_ids, expert_offsets,
                    n_post);
}

}  // namespace moe
