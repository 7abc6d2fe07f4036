// k_gemv.cu -- S3 / S4 for decode-sized expert groups on the CUDA cores, and
// the final fp32 -> bf16 output pass.
//
// Page "Mixture of Experts in vLLM - From First Principles to fused_moe",
// section "Each expert is now an ordinary GEMM": with about one row per
// expert, every expert reads all of its weights to make about one output row,
// so the layer is bound by reading expert weights from HBM.  These kernels
// stream the weights once with 16-byte non-allocating loads, many in flight
// per thread, and multiply each weight against the block's few gathered rows
// kept in shared memory.
//
// Work unit of GEMM 1: (block b of sorted_token_ids, 8 output channels i):
// one warp per channel computes both the gate row i and the up row I+i, so
// SiLU(gate) * up is formed right after the warp reduction.  Input rows are
// read in place through pair id / top_k ("One GEMM 1 program, step by step").
// Work unit of GEMM 2: (block b, 8 rows n of W2): one warp per row; the
// router-weighted result is added into the fp32 accumulator row of the token
// ("The rest of the layer stays in pair order", "Put the results back").
//
// Grids are persistent (a multiple of the SM count); the number of real
// blocks is read on the device from num_tokens_post_padded, so no host
// synchronisation is needed and the launch can be captured in a CUDA graph.
#include <algorithm>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvMaxTok = 8;      // rows gathered per pass (a block is walked in passes)
constexpr int kGemvUnroll = 2;      // 16-byte loads per row kept in flight per lane
constexpr int kGemvSmemBudget = 192 * 1024;  // gathered rows staged per pass

// Rows gathered per pass: the largest power of two (at most 8) whose rows fit
// the shared-memory budget.  A power of two, so that the NT bucket a pass
// dispatches to (the next power of two >= its real rows) never exceeds it.
int gemv_pass_rows(int K) {
  int r = kGemvMaxTok;
  while (r > 1 && r * 2 * K > kGemvSmemBudget) r >>= 1;
  return r;
}

template <int NT>
__device__ __forceinline__ void dot_rows_2(const uint16_t *__restrict__ wa,
                                           const uint16_t *__restrict__ wb, const uint4 *xs,
                                           int xs_stride_vec, int K, int lane, float (&acc_a)[NT],
                                           float (&acc_b)[NT]) {
  const int nvec = K / 8;
  for (int c0 = lane; c0 < nvec; c0 += 32 * kGemvUnroll) {
    uint4 va[kGemvUnroll], vb[kGemvUnroll];
#pragma unroll
    for (int u = 0; u < kGemvUnroll; ++u) {
      const int c = c0 + u * 32;
      if (c < nvec) {
        va[u] = ld_stream_16(wa + (size_t)c * 8);
        vb[u] = ld_stream_16(wb + (size_t)c * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kGemvUnroll; ++u) {
      const int c = c0 + u * 32;
      if (c < nvec) {
        float fa[8], fb[8];
        bf16x8_to_float(va[u], fa);
        bf16x8_to_float(vb[u], fb);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          float xf[8];
          bf16x8_to_float(xs[j * xs_stride_vec + c], xf);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            acc_a[j] = fmaf(fa[q], xf[q], acc_a[j]);
            acc_b[j] = fmaf(fb[q], xf[q], acc_b[j]);
          }
        }
      }
    }
  }
}

template <int NT>
__device__ __forceinline__ void dot_rows_1(const uint16_t *__restrict__ wa, const uint4 *xs,
                                           int xs_stride_vec, int K, int lane, float (&acc)[NT]) {
  const int nvec = K / 8;
  for (int c0 = lane; c0 < nvec; c0 += 32 * kGemvUnroll * 2) {
    uint4 va[2 * kGemvUnroll];
#pragma unroll
    for (int u = 0; u < 2 * kGemvUnroll; ++u) {
      const int c = c0 + u * 32;
      if (c < nvec) va[u] = ld_stream_16(wa + (size_t)c * 8);
    }
#pragma unroll
    for (int u = 0; u < 2 * kGemvUnroll; ++u) {
      const int c = c0 + u * 32;
      if (c < nvec) {
        float fa[8];
        bf16x8_to_float(va[u], fa);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          float xf[8];
          bf16x8_to_float(xs[j * xs_stride_vec + c], xf);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[j] = fmaf(fa[q], xf[q], acc[j]);
        }
      }
    }
  }
}

template <int NT>
__device__ __forceinline__ void warp_sum(float (&v)[NT]) {
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[j] += __shfl_xor_sync(0xffffffffu, v[j], o);
}

// Loads up to kGemvMaxTok pair ids of block b starting at entry `first`; returns
// how many are real (pads sit at the end of a group, so reals come first).
__device__ __forceinline__ int load_pass_pairs(const int32_t *__restrict__ sorted_ids, int b, int B,
                                               int first, int pass_rows, int P, int *pairs) {
  __syncthreads();
  if (threadIdx.x < kGemvMaxTok) {
    int p = P;
    const int idx = first + threadIdx.x;
    if (threadIdx.x < pass_rows && idx < B) p = sorted_ids[(size_t)b * B + idx];
    pairs[threadIdx.x] = (p >= 0 && p < P) ? p : -1;
  }
  __syncthreads();
  int n = 0;
#pragma unroll
  for (int j = 0; j < kGemvMaxTok; ++j) n += pairs[j] >= 0 ? 1 : 0;
  return n;
}

// Stage rows src[row_of(pairs[j])] (K bf16 each) into xs; rows j >= n are zero.
__device__ __forceinline__ void stage_rows(const uint16_t *__restrict__ src, const int *pairs, int n,
                                           int pass_rows, int div, int K, uint4 *xs,
                                           int xs_stride_vec) {
  const int nvec = K / 8;
  for (int v = threadIdx.x; v < pass_rows * nvec; v += blockDim.x) {
    const int j = v / nvec, c = v - j * nvec;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (j < n) val = *reinterpret_cast<const uint4 *>(src + (size_t)(pairs[j] / div) * K + c * 8);
    xs[j * xs_stride_vec + c] = val;
  }
  __syncthreads();
}

template <int NT>
__device__ __forceinline__ void w13_channel(const uint16_t *__restrict__ W, int i, int I, int H,
                                            const uint4 *xs, int xs_stride_vec, const int *pairs,
                                            int n, int lane, uint16_t *__restrict__ a) {
  float g[NT], u[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) g[j] = u[j] = 0.f;
  dot_rows_2<NT>(W + (size_t)i * H, W + (size_t)(I + i) * H, xs, xs_stride_vec, H, lane, g, u);
  warp_sum<NT>(g);
  warp_sum<NT>(u);
  float hg = 0.f, hu = 0.f;
#pragma unroll
  for (int j = 0; j < NT; ++j)
    if (lane == j) {
      hg = g[j];
      hu = u[j];
    }
  if (lane < n) {
    const float gb = bf16_bits_to_float(float_to_bf16_bits(hg));
    const float ub = bf16_bits_to_float(float_to_bf16_bits(hu));
    const float silu = gb / (1.0f + expf(-gb));
    a[(size_t)pairs[lane] * I + i] = float_to_bf16_bits(silu * ub);
  }
}

__global__ void __launch_bounds__(kGemvThreads, 2)
k_gemv_w13_act(const uint16_t *__restrict__ x, const uint16_t *__restrict__ w13,
               const int32_t *__restrict__ sorted_ids, const int32_t *__restrict__ expert_ids,
               const int32_t *__restrict__ n_post_ptr, int P, int top_k, int E, int H, int I, int B,
               int cap, int pass_rows, uint16_t *__restrict__ a) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint4 xs[];
  __shared__ int pairs[kGemvMaxTok];
  const int n_post = min(max(*n_post_ptr, 0), cap);
  const int nblocks = n_post / B;
  const int groups = (I + kGemvWarps - 1) / kGemvWarps;
  const long units = (long)nblocks * groups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stride_vec = H / 8;
  for (long unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int b = static_cast<int>(unit / groups);
    const int g = static_cast<int>(unit - (long)b * groups);
    const int e = expert_ids[b];
    if (e < 0 || e >= E) continue;
    const uint16_t *W = w13 + (size_t)e * 2 * I * H;
    const int i = g * kGemvWarps + warp;
    for (int first = 0; first < B; first += pass_rows) {
      const int n = load_pass_pairs(sorted_ids, b, B, first, pass_rows, P, pairs);
      if (n == 0) break;
      stage_rows(x, pairs, n, pass_rows, top_k, H, xs, stride_vec);
      if (i < I) {
        if (n <= 1) w13_channel<1>(W, i, I, H, xs, stride_vec, pairs, n, lane, a);
        else if (n <= 2) w13_channel<2>(W, i, I, H, xs, stride_vec, pairs, n, lane, a);
        else if (n <= 4) w13_channel<4>(W, i, I, H, xs, stride_vec, pairs, n, lane, a);
        else w13_channel<8>(W, i, I, H, xs, stride_vec, pairs, n, lane, a);
      }
    }
  }
}

template <int NT>
__device__ __forceinline__ void w2_row(const uint16_t *__restrict__ W, int n_row, int H, int I,
                                       const uint4 *xs, int xs_stride_vec, const int *pairs, int n,
                                       int lane, int top_k, const float *__restrict__ topk_w,
                                       float *__restrict__ y_acc) {
  float o[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j] = 0.f;
  dot_rows_1<NT>(W + (size_t)n_row * I, xs, xs_stride_vec, I, lane, o);
  warp_sum<NT>(o);
  float mine = 0.f;
#pragma unroll
  for (int j = 0; j < NT; ++j)
    if (lane == j) mine = o[j];
  if (lane < n) {
    const int p = pairs[lane];
    atomicAdd(y_acc + (size_t)(p / top_k) * H + n_row, topk_w[p] * mine);
  }
}

__global__ void __launch_bounds__(kGemvThreads, 2)
k_gemv_w2_combine(const uint16_t *__restrict__ a, const uint16_t *__restrict__ w2,
                  const int32_t *__restrict__ sorted_ids, const int32_t *__restrict__ expert_ids,
                  const int32_t *__restrict__ n_post_ptr, const float *__restrict__ topk_w, int P,
                  int top_k, int E, int H, int I, int B, int cap, int pass_rows,
                  float *__restrict__ y_acc) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint4 xs[];
  __shared__ int pairs[kGemvMaxTok];
  const int n_post = min(max(*n_post_ptr, 0), cap);
  const int nblocks = n_post / B;
  const int groups = (H + kGemvWarps - 1) / kGemvWarps;
  const long units = (long)nblocks * groups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stride_vec = I / 8;
  for (long unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int b = static_cast<int>(unit / groups);
    const int g = static_cast<int>(unit - (long)b * groups);
    const int e = expert_ids[b];
    if (e < 0 || e >= E) continue;
    const uint16_t *W = w2 + (size_t)e * H * I;
    const int n_row = g * kGemvWarps + warp;
    for (int first = 0; first < B; first += pass_rows) {
      const int n = load_pass_pairs(sorted_ids, b, B, first, pass_rows, P, pairs);
      if (n == 0) break;
      stage_rows(a, pairs, n, pass_rows, 1, I, xs, stride_vec);
      if (n_row < H) {
        if (n <= 1) w2_row<1>(W, n_row, H, I, xs, stride_vec, pairs, n, lane, top_k, topk_w, y_acc);
        else if (n <= 2) w2_row<2>(W, n_row, H, I, xs, stride_vec, pairs, n, lane, top_k, topk_w, y_acc);
        else if (n <= 4) w2_row<4>(W, n_row, H, I, xs, stride_vec, pairs, n, lane, top_k, topk_w, y_acc);
        else w2_row<8>(W, n_row, H, I, xs, stride_vec, pairs, n, lane, top_k, topk_w, y_acc);
      }
    }
  }
}

// y = bf16(y_acc + residual), 4 elements per thread.
__global__ void k_finalize(const float4 *__restrict__ y_acc, const uint2 *__restrict__ residual,
                           long n4, uint2 *__restrict__ y) {
  griddep_wait();
  griddep_launch_dependents();
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4; i += (long)gridDim.x * blockDim.x) {
    float4 v = y_acc[i];
    if (residual != nullptr) {
      const uint2 r = residual[i];
      v.x += __uint_as_float(r.x << 16);
      v.y += __uint_as_float(r.x & 0xFFFF0000u);
      v.z += __uint_as_float(r.y << 16);
      v.w += __uint_as_float(r.y & 0xFFFF0000u);
    }
    uint2 o;
    o.x = static_cast<uint32_t>(float_to_bf16_bits(v.x)) | (static_cast<uint32_t>(float_to_bf16_bits(v.y)) << 16);
    o.y = static_cast<uint32_t>(float_to_bf16_bits(v.z)) | (static_cast<uint32_t>(float_to_bf16_bits(v.w)) << 16);
    y[i] = o;
  }
}

constexpr int kMaxDevices = 64;

}  // namespace

int num_sms() {
  static int cached[kMaxDevices] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 152;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 152;
  }
  return cached[dev];
}

namespace {
struct SmemLimit {
  const void *fn;
  int dev;
  size_t bytes;
};
std::mutex g_smem_mutex;
SmemLimit g_smem_limits[256];
int g_smem_count = 0;
}  // namespace

cudaError_t ensure_smem_limit(const void *fn, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_smem_mutex);
  for (int i = 0; i < g_smem_count; ++i)
    if (g_smem_limits[i].fn == fn && g_smem_limits[i].dev == dev && g_smem_limits[i].bytes >= bytes)
      return cudaSuccess;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (err != cudaSuccess) return err;
  for (int i = 0; i < g_smem_count; ++i)
    if (g_smem_limits[i].fn == fn && g_smem_limits[i].dev == dev) {
      g_smem_limits[i].bytes = bytes;
      return cudaSuccess;
    }
  if (g_smem_count < 256) g_smem_limits[g_smem_count++] = {fn, dev, bytes};
  return cudaSuccess;
}

static cudaError_t set_smem_attr(const void *fn, size_t bytes) { return ensure_smem_limit(fn, bytes); }

cudaError_t launch_gemv_w13_act(const uint16_t *x, const uint16_t *w13, const int32_t *sorted_ids,
                                const int32_t *expert_ids, const int32_t *n_post, int P, int top_k,
                                int E, int H, int I, int B, int cap, uint16_t *a, cudaStream_t s) {
  const int pass_rows = gemv_pass_rows(H);
  const size_t smem = sizeof(uint16_t) * (size_t)pass_rows * H;
  cudaError_t err = set_smem_attr(reinterpret_cast<const void *>(k_gemv_w13_act), smem);
  if (err != cudaSuccess) return err;
  const long units_max = (long)(cap / B) * ((I + kGemvWarps - 1) / kGemvWarps);
  const int grid = static_cast<int>(std::min<long>(units_max, (long)num_sms() * 8));
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(k_gemv_w13_act, dim3(grid), dim3(kGemvThreads), smem, s, x, w13, sorted_ids,
                    expert_ids, n_post, P, top_k, E, H, I, B, cap, pass_rows, a);
}

cudaError_t launch_gemv_w2_combine(const uint16_t *a, const uint16_t *w2, const int32_t *sorted_ids,
                                   const int32_t *expert_ids, const int32_t *n_post,
                                   const float *topk_weights, int P, int top_k, int E, int H, int I,
                                   int B, int cap, float *y_acc, cudaStream_t s) {
  const int pass_rows = gemv_pass_rows(I);
  const size_t smem = sizeof(uint16_t) * (size_t)pass_rows * I;
  cudaError_t err = set_smem_attr(reinterpret_cast<const void *>(k_gemv_w2_combine), smem);
  if (err != cudaSuccess) return err;
  const long units_max = (long)(cap / B) * ((H + kGemvWarps - 1) / kGemvWarps);
  const int grid = static_cast<int>(std::min<long>(units_max, (long)num_sms() * 8));
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(k_gemv_w2_combine, dim3(grid), dim3(kGemvThreads), smem, s, a, w2, sorted_ids,
                    expert_ids, n_post, topk_weights, P, top_k, E, H, I, B, cap, pass_rows, y_acc);
}

cudaError_t launch_finalize(const float *y_acc, const uint16_t *residual, int M, int H, uint16_t *y,
                            cudaStream_t s) {
  const long n4 = (long)M * H / 4;
  if (n4 == 0) return cudaSuccess;
  const int threads = 256;
  const int grid = static_cast<int>(std::min<long>((n4 + threads - 1) / threads, (long)num_sms() * 8));
  return launch_pdl(k_finalize, dim3(grid), dim3(threads), 0, s,
                    reinterpret_cast<const float4 *>(y_acc),
                    reinterpret_cast<const uint2 *>(residual), n4, reinterpret_cast<uint2 *>(y));
}

}  // namespace moe
