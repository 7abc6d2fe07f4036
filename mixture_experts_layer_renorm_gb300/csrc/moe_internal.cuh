// moe_internal.cuh -- shared device helpers and the launch functions that
// moe_api.cu calls.  Internal to the CUDA library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
// The workspace starts with a control block: the status word at int 0 and the
// fused routing kernel's completion counters from int kCountersOffset on.
constexpr int kStatusBytes = 1024;
constexpr int kCountersOffset = 64;
constexpr int kRouteFusedMaxGroups = 64;   // token groups (<= 8 tokens each); one more counter for the align
constexpr int kDecodeCtlOffset = 192;     // the decode-layer kernel's grid-barrier counters (3 ints)
constexpr int kRouterCtlOffset = 196;     // the tensor-core router's tile counters when it splits K
constexpr int kRouterCtlCount = 60;       // (one per tile; it splits only up to this many tiles)
constexpr int kRouterMaxSplits = 4;

// Programmatic dependent launch.  Every kernel of the library is launched with
// launch_pdl, so it may become resident while the kernel before it in the
// stream is still running.  It calls griddep_wait() before it touches
// anything an earlier kernel writes (this waits for the whole earlier kernel
// and makes its writes visible) and griddep_launch_dependents() to let the
// next kernel start the same way.  Both are no-ops for a kernel launched
// without the attribute or after a kernel that does not signal.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// The same with the grid launched as clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t s, unsigned cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Device status codes (same numbering as moe_status_t).
constexpr int kStatusBadExpertId = 5;
constexpr int kStatusTimeout = 6;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// fp32 -> bf16 bits, round to nearest even (cvt.rn.bf16.f32).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// acc + the 8 products of two rows of 8 bf16 (16 bytes each), taken in order
// with the mixed-precision multiply-add (bf16 operands, fp32 sum: the product
// of two bf16 values is exact in fp32, so each step rounds once, as an fp32
// fma of the widened values would).
__device__ __forceinline__ float dot8_bf16(const uint4 &w, const uint4 &x, float acc) {
  asm("{\n\t.reg .b16 w0, w1, w2, w3, w4, w5, w6, w7, x0, x1, x2, x3, x4, x5, x6, x7;\n\t"
      "mov.b32 {w0, w1}, %1;\n\tmov.b32 {w2, w3}, %2;\n\t"
      "mov.b32 {w4, w5}, %3;\n\tmov.b32 {w6, w7}, %4;\n\t"
      "mov.b32 {x0, x1}, %5;\n\tmov.b32 {x2, x3}, %6;\n\t"
      "mov.b32 {x4, x5}, %7;\n\tmov.b32 {x6, x7}, %8;\n\t"
      "fma.rn.f32.bf16 %0, w0, x0, %0;\n\tfma.rn.f32.bf16 %0, w1, x1, %0;\n\t"
      "fma.rn.f32.bf16 %0, w2, x2, %0;\n\tfma.rn.f32.bf16 %0, w3, x3, %0;\n\t"
      "fma.rn.f32.bf16 %0, w4, x4, %0;\n\tfma.rn.f32.bf16 %0, w5, x5, %0;\n\t"
      "fma.rn.f32.bf16 %0, w6, x6, %0;\n\tfma.rn.f32.bf16 %0, w7, x7, %0;\n\t}"
      : "+f"(acc)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w));
  return acc;
}

// Record the first problem a kernel meets; later ones keep the first code.
__device__ __forceinline__ void report_status(int *status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// 8 bf16 in a uint4 -> 8 floats
__device__ __forceinline__ void bf16x8_to_float(const uint4 &v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Streaming 16-byte load that skips L1 (weights are read once per use).
__device__ __forceinline__ uint4 ld_stream_16(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ----------------------------------------------------------------------------
// Launch functions.  Each returns the cudaError_t of its launch(es).

// S0: logits [M,E] = bf16(x [M,H] . w_router[E,H]^T + bias)
cudaError_t launch_router_logits(const uint16_t *x, const uint16_t *w_router, const float *bias,
                                 int M, int E, int H, uint16_t *logits, cudaStream_t s);

// S1: warp-per-token softmax / top-k / renormalize
cudaError_t launch_topk_softmax(const uint16_t *logits, int M, int E, int top_k, int renormalize,
                                int32_t *topk_ids, float *topk_weights, cudaStream_t s);

// S2: align.  hist: scratch int32 [align_hist_entries(P, E)] (may be null when
// align_num_ctas(P) == 1).  status: device status word.
int align_num_ctas(long P);
long align_hist_entries(long P, int E);
cudaError_t launch_align(const int32_t *topk_ids, int P, int E, int B, int cap,
                         int32_t *sorted_ids, int32_t *expert_ids, int32_t *expert_offsets,
                         int32_t *n_post, int32_t *hist, int *status, cudaStream_t s);

// S3 / S4 on CUDA cores: weight-streaming grouped GEMV (decode-sized groups).
cudaError_t launch_gemv_w13_act(const uint16_t *x, const uint16_t *w13, const int32_t *sorted_ids,
                                const int32_t *expert_ids, const int32_t *n_post, int P, int top_k,
                                int E, int H, int I, int B, int cap, uint16_t *a, cudaStream_t s);
cudaError_t launch_gemv_w2_combine(const uint16_t *a, const uint16_t *w2, const int32_t *sorted_ids,
                                   const int32_t *expert_ids, const int32_t *n_post,
                                   const float *topk_weights, int P, int top_k, int E, int H, int I,
                                   int B, int cap, float *y_acc, cudaStream_t s);

// S3 / S4 on the tensor cores (tcgen05 + TMEM + TMA), block sizes 16..256 (multiples of 16
// that are powers of two).  status: device status word for bounded-wait timeouts (nullable).
bool tc_supports_block(int B);
cudaError_t launch_tc_w13_act(const uint16_t *x, const uint16_t *w13, const int32_t *sorted_ids,
                              const int32_t *expert_ids, const int32_t *n_post, int P, int top_k,
                              int E, int H, int I, int B, int cap, uint16_t *a, int ksplit,
                              float *h_acc, int *tile_cnt, int *status, int pf_experts,
                              float *zero_dst, long zero_n, cudaStream_t s);
// zero_dst / zero_n: an fp32 buffer (zero_n a multiple of 4, 16-byte aligned)
// GEMM 1 clears on the way, or null.
// ksplit > 1 splits each tile's K range across CTAs (GEMM 1: partial sums go
// through h_acc [P, 2I] fp32 and tile_cnt [cap/B * ceil(I/128)] ints, both zero
// on entry; GEMM 2 adds its partial sums into y_acc directly).
cudaError_t launch_tc_w2_combine(const uint16_t *a, const uint16_t *w2, const int32_t *sorted_ids,
                                 const int32_t *expert_ids, const int32_t *n_post,
                                 const float *topk_weights, int P, int top_k, int E, int H, int I,
                                 int B, int cap, float *y_acc, int ksplit, int *status,
                                 bool early_weights, cudaStream_t s);

// FP8 (E4M3) versions of S3 / S4: codes [rows, K] with one fp32 scale per row
// on both sides (w13s [E, 2I], sx [M]; w2s [E, H], sa [P]).  GEMM 1 writes a in
// bf16 as the bf16 path does; the caller quantizes it for GEMM 2.
cudaError_t launch_tc_w13_act_f8(const uint8_t *qx, const float *sx, const uint8_t *w13q,
                                 const float *w13s, const int32_t *sorted_ids,
                                 const int32_t *expert_ids, const int32_t *n_post, int P, int top_k,
                                 int E, int H, int I, int B, int cap, uint16_t *a, int ksplit,
                                 float *h_acc, int *tile_cnt, int *status, int pf_experts,
                                 float *zero_dst, long zero_n, cudaStream_t s);
cudaError_t launch_tc_w2_combine_f8(const uint8_t *qa, const float *sa, const uint8_t *w2q,
                                    const float *w2s, const int32_t *sorted_ids,
                                    const int32_t *expert_ids, const int32_t *n_post,
                                    const float *topk_weights, int P, int top_k, int E, int H,
                                    int I, int B, int cap, float *y_acc, int ksplit, int *status,
                                    bool early_weights, cudaStream_t s);
// Per-row dynamic E4M3 quantization of a bf16 [R, K] matrix (K a multiple of
// 16): s[r] = amax / 448 (1 for a zero row), q[r, :] = e4m3(src[r, :] / s[r]).
cudaError_t launch_quant_rows(const uint16_t *src, int R, int K, uint8_t *q, float *s,
                              cudaStream_t st);

// S0 on the tensor cores: logits [M,E] = bf16(x . w_router^T + bias), blocks of 128 tokens.
// One CTA whose bounded wait on an mbarrier nothing completes gives up after
// about limit_ms ms and records the timeout status (self-test of that path).
cudaError_t launch_selftest_timeout(int *status, int limit_ms, cudaStream_t s);
// With split_scratch (kRouterMaxSplits * E * roundup(M, 128) floats) and
// tile_cnt (zero, kRouterCtlCount ints, left zero) the K range of each tile
// is split over up to kRouterMaxSplits CTAs when the tiles leave SMs idle.
cudaError_t launch_tc_router(const uint16_t *x, const uint16_t *w_router, const float *bias, int M,
                             int E, int H, uint16_t *logits, int *status, float *split_scratch,
                             int *tile_cnt, cudaStream_t s);

// y = bf16(y_acc + residual)
cudaError_t launch_finalize(const float *y_acc, const uint16_t *residual, int M, int H, uint16_t *y,
                            cudaStream_t s);

// S0 + S1 + S2 in one launch (decode-sized batches).  logits_in given: no
// router.  counters: kRouteFusedMaxGroups + 1 ints in the workspace control
// block, zero between calls.  zero_buf (nullable): zero_n floats cleared on the side.
bool route_fused_supports(int M, int E, int top_k);
cudaError_t launch_route_fused(const uint16_t *x, const uint16_t *w_router, const float *bias,
                               const uint16_t *logits_in, int M, int E, int H, int top_k,
                               int renormalize, int B, uint16_t *logits_ws, int32_t *topk_ids,
                               float *topk_w, int32_t *sorted_ids, int32_t *expert_ids,
                               int32_t *expert_offsets, int32_t *n_post, int *counters,
                               int *status, float *zero_buf, long zero_n, bool skip_sort,
                               cudaStream_t s);

// The whole layer in one persistent kernel (decode-sized batches): router
// (or the given logits), top-k, grouping, GEMM 1 + SiLU-and-mul, GEMM 2 +
// combine, y written as bf16.  ctl: 3 ints in the workspace control block,
// zero between calls.  logits_buf [M, E], a_buf [M * top_k, I] and y_acc
// [M, H] fp32 are scratch (logits_buf receives the router's logits).
bool decode_layer_supports(int M, int E, int top_k, int H, int I);
cudaError_t launch_decode_layer(const uint16_t *x, const uint16_t *w_router,
                                const uint16_t *logits_in, const float *bias,
                                const uint16_t *w13, const uint16_t *w2,
                                const uint16_t *residual, int M, int E, int top_k, int H, int I,
                                int renormalize, uint16_t *y, int32_t *ids_out, float *wts_out,
                                uint16_t *logits_buf, uint16_t *a_buf, float *y_acc, int *ctl,
                                int *status, cudaStream_t s);

int num_sms();

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  The driver call happens once per (kernel, device, size);
// later launches only look the pair up in a table.
cudaError_t ensure_smem_limit(const void *fn, size_t bytes);

}  // namespace moe
