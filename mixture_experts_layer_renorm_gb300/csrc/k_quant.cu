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

// One warp per row; 16-byte chunks of 8 bf16 strided over the lanes.
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    if (lane == 0) s[r] = sc;
    uint2 *qrow = reinterpret_cast<uint2 *>(q + (size_t)r * K);
    for (int c = lane; c < kv; c += 32) {
      float f[8];
      bf16x8_to_float(row[c], f);
      uint2 out;
      out.x = static_cast<uint32_t>(e4m3x2(__fdiv_rn(f[0], sc), __fdiv_rn(f[1], sc))) |
              (static_cast<uint32_t>(e4m3x2(__fdiv_rn(f[2], sc), __fdiv_rn(f[3], sc))) << 16);
      out.y = static_cast<uint32_t>(e4m3x2(__fdiv_rn(f[4], sc), __fdiv_rn(f[5], sc))) |
              (static_cast<uint32_t>(e4m3x2(__fdiv_rn(f[6], sc), __fdiv_rn(f[7], sc))) << 16);
      qrow[c] = out;
    }
  }
}

}  // namespace

cudaError_t launch_quant_rows(const uint16_t *src, int R, int K, uint8_t *q, float *s,
                              cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  const int per_cta = kQuantThreads / 32;
  const int grid = static_cast<int>(std::min<long>((R + per_cta - 1) / per_cta, (long)num_sms() * 8));
  return launch_pdl(k_quant_rows, dim3(grid), dim3(kQuantThreads), 0, st, src, R, K, q, s);
}

}  // namespace moe
