// route_dev.cuh -- the warp-level softmax / top-k / renormalize (S1) shared
// by the top-k kernel and the fused routing kernel.
// Page "Mixture of Experts in vLLM - From First Principles to fused_moe",
// section "One token uses only 8 experts", steps 1-3.
#pragma once

#include "moe_internal.cuh"

namespace moe {
namespace {

// Order-preserving map of a bf16 pattern to 16 unsigned bits: larger value ->
// larger key; -0 is folded onto +0 so that the two compare equal.
__device__ __forceinline__ uint32_t bf16_order_key(uint16_t b) {
  if (b == 0x8000u) b = 0;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
__device__ __forceinline__ uint16_t bf16_from_order_key(uint32_t k) {
  return (k & 0x8000u) ? static_cast<uint16_t>(k & 0x7FFFu) : static_cast<uint16_t>(~k & 0xFFFFu);
}

// One warp, one token.  Lane l holds logits l, l+32, ... as 32-bit keys
// (order key << 16 | (0xFFFF - e)), so the largest key is the largest logit
// and, among equal logits, the lowest expert id.  top_k rounds of a warp
// max-reduction pick the slots in order; the winner's key is cleared.
// Logits written earlier in the same kernel by other CTAs are read around L1.
// ids_copy (nullable, e.g. shared memory): a second copy of the chosen ids.
template <int VPL, bool kFromOtherCtas>
__device__ __forceinline__ void topk_softmax_warp(const uint16_t *__restrict__ row, int E,
                                                  int top_k, int renormalize,
                                                  int32_t *__restrict__ ids_out,
                                                  float *__restrict__ w_out, int lane,
                                                  int32_t *ids_copy = nullptr) {
  uint32_t key[VPL];
  float val[VPL];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0;
    val[i] = -INFINITY;
    if (e < E) {
      const uint16_t b = kFromOtherCtas ? __ldcg(row + e) : row[e];
      key[i] = (bf16_order_key(b) << 16) | (0xFFFFu - static_cast<uint32_t>(e));
      val[i] = bf16_bits_to_float(b);
      mx = fmaxf(mx, val[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  // the full softmax denominator only when the weights are not renormalized
  float den = 0.f;
  if (!renormalize) {
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (lane + 32 * i < E) den += expf(val[i] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  }
  // top_k rounds pick the keys (lane j keeps the j-th); the exponentials of
  // the chosen logits are then taken by their lanes side by side
  uint32_t my_key = 0;
  for (int j = 0; j < top_k; ++j) {
    uint32_t best = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) best = max(best, key[i]);
    best = __reduce_max_sync(0xffffffffu, best);
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (key[i] == best) key[i] = 0;
    if (lane == j) my_key = best;
  }
  const int my_id = static_cast<int>(0xFFFFu - (my_key & 0xFFFFu));
  const float my_p = lane < top_k ? expf(bf16_bits_to_float(bf16_from_order_key(my_key >> 16)) - mx) : 0.f;
  float kept = my_p;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
  if (lane < top_k) {
    ids_out[lane] = my_id;
    if (ids_copy != nullptr) ids_copy[lane] = my_id;
    w_out[lane] = renormalize ? my_p / kept : my_p / den;
  }
}

// VPL (keys per lane) bucket for E experts.
inline int topk_vpl(int E) { return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : E <= 512 ? 16 : 32; }

}  // namespace
}  // namespace moe
