// k_quant.cu -- per-row dynamic E4M3 quantization of a bf16 matrix, the
// activation side of the FP8 layer.
//
// Page "Mixture of Experts in vLLM - From First Principles to fused_moe",
// section "fused_experts_impl": for an FP8 model the GEMM-1 input is the
// quantized copy of x (qhidden_states).  Here a row (a token of x, a pair of
// the GEMM-1 output a) gets the scale s = amax / 448 (1 for an all-zero row)
// and the codes e4m3(v / s), rounded to nearest, ties to even, saturating at
// +-448.  amax, s and v / s are fp32 with correctly rounded division, so the
// codes are a function of the row alone.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kQuantThreads = 256;

// Two fp32 values -> two E4M3 codes (lo in the low byte).
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// The 8 codes of e4m3(v / s) for one chunk (lo in the low byte).
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float s) {
  uint2 out;
  out.x = static_cast<uint32_t>(e4m3x2(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s))) |
          (static_cast<uint32_t>(e4m3x2(__fdiv_rn(f[2], s), __fdiv_rn(f[3], s))) << 16);
  out.y = static_cast<uint32_t>(e4m3x2(__fdiv_rn(f[4], s), __fdiv_rn(f[5], s))) |
          (static_cast<uint32_t>(e4m3x2(__fdiv_rn(f[6], s), __fdiv_rn(f[7], s))) << 16);
  return out;
}

// amax over the warp -> the row's scale.
__device__ __forceinline__ float row_scale(float amax) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

// From this many rows on, a row is read once (the register-resident kernel).
// Decode batches stay below it: there the rows are few and L2-resident, and
// the two-pass kernel measured a few percent faster per layer.
constexpr int kQuantRegMinRows = 4096;

// Register-resident kernel: 128-thread CTAs (4 rows at a time), small enough
// (128 x 80 registers for rows of 2048) to sit beside a 512-thread grouped
// GEMM CTA of up to 96 registers a thread, which programmatic dependent
// launch starts while the quantization is still running.
constexpr int kQuantRegThreads = 128;
template <int CH>
constexpr int kQuantRegBlocks = CH >= 8 ? 6 : CH >= 4 ? 8 : 12;  // resident CTAs per SM

// One warp per row, the whole row held in registers: up to CH chunks of 8
// bf16 per lane (rows of at most 256 CH elements).  Every chunk of the row is
// requested before the first is used, and the row is read from memory once.
template <int CH>
__global__ void __launch_bounds__(kQuantRegThreads, kQuantRegBlocks<CH>)
k_quant_rows_reg(const uint16_t *__restrict__ src, int R, int K, uint8_t *__restrict__ q,
                 float *__restrict__ s) {
  griddep_wait();  // the rows are the previous kernel's output
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x / 32);
  const int kv = K / 8;
  for (int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < R; r += nwarps) {
    const uint4 *row = reinterpret_cast<const uint4 *>(src + (size_t)r * K);
    uint4 v[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int c = lane + 32 * j;
      v[j] = c < kv ? row[c] : make_uint4(0u, 0u, 0u, 0u);  // zeros leave amax unchanged
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      float f[8];
      bf16x8_to_float(v[j], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    }
    const float sc = row_scale(amax);
    if (lane == 0) s[r] = sc;
    uint2 *qrow = reinterpret_cast<uint2 *>(q + (size_t)r * K);
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int c = lane + 32 * j;
      if (c < kv) {
        float f[8];
        bf16x8_to_float(v[j], f);
        qrow[c] = quant8(f, sc);
      }
    }
  }
}

// Fewer than kQuantRegMinRows rows, or rows longer than 2048: one warp per
// row, two passes over it (amax, then the codes), 16-byte chunks of 8 bf16
// strided over the lanes.
__global__ void __launch_bounds__(kQuantThreads)
k_quant_rows(const uint16_t *__restrict__ src, int R, int K, uint8_t *__restrict__ q,
             float *__restrict__ s) {
  griddep_wait();  // the rows are the previous kernel's output
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x / 32);
  const int kv = K / 8;
  for (int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < R; r += nwarps) {
    const uint4 *row = reinterpret_cast<const uint4 *>(src + (size_t)r * K);
    float amax = 0.f;
    for (int c = lane; c < kv; c += 32) {
      float f[8];
      bf16x8_to_float(row[c], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    }
    const float sc = row_scale(amax);
    if (lane == 0) s[r] = sc;
    uint2 *qrow = reinterpret_cast<uint2 *>(q + (size_t)r * K);
    for (int c = lane; c < kv; c += 32) {
      float f[8];
      bf16x8_to_float(row[c], f);
      qrow[c] = quant8(f, sc);
    }
  }
}

}  // namespace

cudaError_t launch_quant_rows(const uint16_t *src, int R, int K, uint8_t *q, float *s,
                              cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  // one resident wave, the rows strided over its warps (one warp per row)
  auto grid = [&](int threads, int per_sm) {
    const long ctas = (R + threads / 32 - 1) / (threads / 32);
    return dim3(static_cast<int>(std::min<long>(ctas, (long)num_sms() * per_sm)));
  };
  const dim3 b(kQuantRegThreads);
  const int chunks = R >= kQuantRegMinRows ? (K / 8 + 31) / 32 : 0;  // 16-byte chunks per lane
  if (chunks == 0 || chunks > 8)
    return launch_pdl(k_quant_rows, grid(kQuantThreads, 8), dim3(kQuantThreads), 0, st, src, R, K,
                      q, s);
  if (chunks <= 1)
    return launch_pdl(k_quant_rows_reg<1>, grid(kQuantRegThreads, kQuantRegBlocks<1>), b, 0, st,
                      src, R, K, q, s);
  if (chunks <= 2)
    return launch_pdl(k_quant_rows_reg<2>, grid(kQuantRegThreads, kQuantRegBlocks<2>), b, 0, st,
                      src, R, K, q, s);
  if (chunks <= 4)
    return launch_pdl(k_quant_rows_reg<4>, grid(kQuantRegThreads, kQuantRegBlocks<4>), b, 0, st,
                      src, R, K, q, s);
  return launch_pdl(k_quant_rows_reg<8>, grid(kQuantRegThreads, kQuantRegBlocks<8>), b, 0, st, src,
                    R, K, q, s);
}

}  // namespace moe
