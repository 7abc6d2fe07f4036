// moe_api.cu -- host side of the C ABI declared in include/moe_api.h:
// argument checks, workspace layout, path choice and kernel launches.
//
// Nothing here allocates device memory or synchronises with the host (except
// moe_get_device_status); every launch goes to the caller's stream, so the
// calls can be captured in a CUDA graph.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moe_api.h"
#include "moe_internal.cuh"

namespace {

using moe::kMaxExperts;
using moe::kMaxTopK;

constexpr size_t kAlign = 256;
constexpr int kMaxDim = 65536;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool valid_block_size(int B) { return B >= 1 && B <= 256; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shapes shared by every entry point.
moe_status_t check_shapes(int M, int E, int top_k, int H, int I) {
  if (M < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (top_k < 1 || top_k > std::min(E, kMaxTopK)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (H < 16 || H > kMaxDim || H % 16 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (I < 16 || I > kMaxDim || I % 16 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(M) * top_k >= (1LL << 31) - kMaxExperts * 256LL)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

long capacity(long P, int E, int B) {
  const long cap = P + static_cast<long>(E) * (B - 1);
  return (cap + B - 1) / B * B;
}

// Workspace regions, each 256-byte aligned.  The status word is always at
// offset 0 so that moe_get_device_status can find it from the pointer alone.
struct WsLayout {
  size_t status, logits, ids, wts, sorted, eids, offsets, npost, hist, a, qx, sx, qa, sa, yacc,
      hacc, tcnt, rscr, total;
};

// S0: the tensor-core router from 256 tokens up, the CUDA-core one below.
constexpr int kTcRouterMinTokens = 256;

// Batches whose tensor-core router may split its tiles' K range (routing of
// more than 256 tokens, at most moe::kRouterCtlCount tiles of 128 tokens):
// the split scratch holds kRouterMaxSplits fp32 slices of the logits.
bool router_may_split(int M, int E) {
  return M > kTcRouterMinTokens &&
         ((M + 127) / 128) * ((E + 255) / 256) <= moe::kRouterCtlCount;
}
size_t router_scratch_bytes(int M, int E) {
  return router_may_split(M, E)
             ? sizeof(float) * moe::kRouterMaxSplits * static_cast<size_t>(E) * ((M + 127) / 128 * 128)
             : 0;
}

// Decode-sized batches (those the fused routing kernel serves) may split
// GEMM 1's K range; they reserve its fp32 partial sums and tile counters.
constexpr int kSplitMaxTokens = 256;

// fp8: the E4M3 codes and row scales of x and a (before y_acc, so that the
// span the routing kernel clears from y_acc on is the same in both layouts).
WsLayout ws_layout(int M, int E, int top_k, int H, int I, int B, bool fp8 = false) {
  const long P = static_cast<long>(M) * top_k;
  const long cap = capacity(P, E, B);
  WsLayout w{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = round_up(o + bytes, kAlign);
    return at;
  };
  w.status = take(moe::kStatusBytes);
  w.logits = take(sizeof(uint16_t) * static_cast<size_t>(M) * E);
  w.ids = take(sizeof(int32_t) * static_cast<size_t>(P));
  w.wts = take(sizeof(float) * static_cast<size_t>(P));
  w.sorted = take(sizeof(int32_t) * static_cast<size_t>(cap));
  w.eids = take(sizeof(int32_t) * static_cast<size_t>(cap / B));
  w.offsets = take(sizeof(int32_t) * static_cast<size_t>(E + 1));
  w.npost = take(sizeof(int32_t));
  w.hist = take(sizeof(int32_t) * static_cast<size_t>(moe::align_hist_entries(P, E)));
  w.a = take(sizeof(uint16_t) * static_cast<size_t>(P) * I);
  w.qx = take(fp8 ? static_cast<size_t>(M) * H : 0);
  w.sx = take(fp8 ? sizeof(float) * static_cast<size_t>(M) : 0);
  w.qa = take(fp8 ? static_cast<size_t>(P) * I : 0);
  w.sa = take(fp8 ? sizeof(float) * static_cast<size_t>(P) : 0);
  w.yacc = take(sizeof(float) * static_cast<size_t>(M) * H);
  // h_acc and the tile counters directly follow y_acc: one span to clear
  const bool split = M <= kSplitMaxTokens;
  w.hacc = take(split ? sizeof(float) * static_cast<size_t>(P) * 2 * I : 0);
  w.tcnt = take(split ? sizeof(int32_t) * static_cast<size_t>(cap / B) * ((I + 127) / 128) : 0);
  w.rscr = take(router_scratch_bytes(M, E));
  w.total = o;
  return w;
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Which grouped-GEMM implementation runs: the tcgen05 kernels for block sizes
// they tile (16, 32, 64, 128, 256), the CUDA-core weight-streaming kernels for
// any other block size.  MOE_FORCE_PATH=gemv|tc|tc1 overrides the choice (for
// measurements and tests); "tc" falls back to gemv where the block size is
// not tiled; "tc1" is "tc" without 2-SM tiles (k_gemm_tc.cu reads it).
enum class GemmPath { kGemv, kTensorCore };

int forced_path() {
  const char *v = std::getenv("MOE_FORCE_PATH");
  if (v == nullptr) return 0;
  if (std::strcmp(v, "gemv") == 0) return 1;
  if (std::strcmp(v, "tc") == 0 || std::strcmp(v, "tc1") == 0) return 2;
  return 0;
}

// The whole layer as one persistent kernel (k_decode_layer), for decode-sized
// batches.  Measured against the kernel chain below it does not win on this
// GPU (a tie at one token, slower from about eight tokens on, where its
// CUDA-core arithmetic and its three grid barriers outweigh the saved
// launches), so it runs only when MOE_DECODE_LAYER=on asks for it and the
// shape fits its shared-memory plan.
bool use_decode_layer(int M, int E, int top_k, int H, int I) {
  const char *v = std::getenv("MOE_DECODE_LAYER");
  if (v == nullptr || std::strcmp(v, "on") != 0) return false;
  return forced_path() == 0 && moe::decode_layer_supports(M, E, top_k, H, I);
}

GemmPath pick_path(int M, int E, int top_k, int B) {
  (void)M; (void)E; (void)top_k;
  if (!moe::tc_supports_block(B)) return GemmPath::kGemv;
  if (forced_path() == 1) return GemmPath::kGemv;
  return GemmPath::kTensorCore;
}

// A library-wide status word (one per device) for entry points without a
// workspace; moe_get_device_status reports it together with the workspace's.
static __device__ int g_lib_status;
std::mutex g_lib_status_mutex;
int *g_lib_status_ptr[64] = {};

int *lib_status() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_lib_status_mutex);
  if (g_lib_status_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lib_status) == cudaSuccess) g_lib_status_ptr[dev] = static_cast<int *>(p);
  }
  return g_lib_status_ptr[dev];
}

// split_scratch (nullable): the router's split scratch and the control block
// holding its tile counters (the workspace's), for entry points that have one.
moe_status_t run_router(const uint16_t *x, const uint16_t *w_router, const float *bias, int M,
                        int E, int H, uint16_t *logits, int *status, float *split_scratch,
                        int *control, cudaStream_t s) {
  if (M >= kTcRouterMinTokens && forced_path() != 1)
    return cuda_status(moe::launch_tc_router(
        x, w_router, bias, M, E, H, logits, status, split_scratch,
        split_scratch != nullptr && control != nullptr ? control + moe::kRouterCtlOffset : nullptr,
        s));
  return cuda_status(moe::launch_router_logits(x, w_router, bias, M, E, H, logits, s));
}

// S0 + S1 + S2.  Decode-sized batches take one fused launch (which also
// clears zero_buf, the combine accumulator, when given); larger ones run the
// router, top-k and align kernels.  *zeroed tells whether zero_buf was cleared.
// skip_sort (only moe_forward asks, for M * top_k * 4 <= E): the fused launch
// puts each pair in its own block instead of grouping by expert; the vLLM
// blog, "Small batches skip the sort".
constexpr int kFusedRouteMaxTokens = 256;

moe_status_t run_route(const uint16_t *x, const uint16_t *w_router, const uint16_t *router_logits,
                       const float *bias, int M, int E, int top_k, int H, int renormalize, int B,
                       uint16_t *logits_ws, int32_t *ids, float *wts, int32_t *sorted,
                       int32_t *eids, int32_t *offs, int32_t *npost, int32_t *hist, int *control,
                       float *router_scratch, float *zero_buf, long zero_n, bool *zeroed,
                       bool skip_sort, cudaStream_t s) {
  const long P = static_cast<long>(M) * top_k;
  const int cap = static_cast<int>(capacity(P, E, B));
  *zeroed = false;
  if (M <= kFusedRouteMaxTokens && moe::route_fused_supports(M, E, top_k) && forced_path() != 1) {
    *zeroed = zero_buf != nullptr;
    return cuda_status(moe::launch_route_fused(
        x, w_router, bias, router_logits, M, E, H, top_k, renormalize, B, logits_ws, ids, wts,
        sorted, eids, offs, npost, control + moe::kCountersOffset, control, zero_buf, zero_n,
        skip_sort, s));
  }
  const uint16_t *logits = router_logits;
  if (w_router) {
    moe_status_t st =
        run_router(x, w_router, bias, M, E, H, logits_ws, control, router_scratch, control, s);
    if (st != MOE_OK) return st;
    logits = logits_ws;
  }
  moe_status_t st =
      cuda_status(moe::launch_topk_softmax(logits, M, E, top_k, renormalize, ids, wts, s));
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_align(ids, static_cast<int>(P), E, B, cap, sorted, eids, offs,
                                       npost, hist, control, s));
}

// Splits of each tile's K range for a grouped GEMM with n_ctiles weight tiles
// per block: decode batches can have fewer tiles than SMs, or a last wave
// that leaves most SMs idle.  The block count is estimated on the host as the
// expected number of distinct experts, E (1 - (1 - top_k/E)^M).  Each split
// beyond the first is charged split_cost of a tile's time (the fp32 partial
// sums it adds, the finishing pass, the split scratch the routing kernel
// clears): 0.15 with bf16 operands, 0.30 with E4M3 ones, whose mainloop is
// half as long.  Measured against 0.03 on one box: Qwen3 decode M = 8
// 115.3 -> 110.4 us (E4M3 102.6 -> 85.3), M = 32 204.0 -> 200.0 (E4M3
// 143.4 -> 134.0), E60 tail M = 64 199.7 -> 189.8 (E4M3 144.0 -> 126.5),
// 64-layer stack M = 16 7.97 -> 7.48 ms; M = 1 and M = 64 unchanged.
constexpr double kSplitCostBf16 = 0.15;
constexpr double kSplitCostE4M3 = 0.30;

int pick_ksplit(int M, int E, int top_k, int n_ctiles, int nk, double split_cost) {
  if (M > kSplitMaxTokens) return 1;
  const double D = E * (1.0 - std::pow(1.0 - static_cast<double>(top_k) / E, M));
  const double tiles = std::max(1.0, std::ceil(D)) * n_ctiles;
  const double sms = moe::num_sms();
  int best = 1;
  double best_score = 0;
  for (int ks = 1; ks <= 4 && ks <= nk; ++ks) {
    const double units = tiles * ks;
    const double eff = units / (std::ceil(units / sms) * sms);  // busy fraction of the waves
    const double score = eff / (1.0 + split_cost * (ks - 1));
    if (score > best_score + 1e-9) {
      best_score = score;
      best = ks;
    }
  }
  return best;
}

// prefetch (moe_forward): GEMM 1 may bring the first wave's expert weights
// into L2 while routing runs, when at least 80 % of the experts are expected to
// be routed to (decode M = 64: 220.8 -> 217.6 us with it; 32 tokens, which
// 0.9 left out, 203.4 -> 201.7, E4M3 135.3 -> 133.4; a cap of 64 or 112 MB
// instead of 96 no better).
moe_status_t run_gemm1(const uint16_t *x, const uint16_t *w13, const int32_t *sorted,
                       const int32_t *eids, const int32_t *npost, int M, int top_k, int E, int H,
                       int I, int B, uint16_t *a, float *h_acc, int *tile_cnt, int *status,
                       bool prefetch, float *zero_dst, long zero_n, cudaStream_t s) {
  const long P = static_cast<long>(M) * top_k;
  const int cap = static_cast<int>(capacity(P, E, B));
  switch (pick_path(M, E, top_k, B)) {
    case GemmPath::kTensorCore: {
      const int ks = h_acc != nullptr
                         ? pick_ksplit(M, E, top_k, (I + 127) / 128, (H + 63) / 64, kSplitCostBf16)
                         : 1;
      const double D = E * (1.0 - std::pow(1.0 - static_cast<double>(top_k) / E, M));
      const int pf_experts = (prefetch && D >= 0.8 * E) ? E : 0;
      return cuda_status(moe::launch_tc_w13_act(x, w13, sorted, eids, npost, static_cast<int>(P),
                                                top_k, E, H, I, B, cap, a, ks, h_acc, tile_cnt,
                                                status, pf_experts, zero_dst, zero_n, s));
    }
    case GemmPath::kGemv:
    default:
      if (zero_dst != nullptr &&
          cudaMemsetAsync(zero_dst, 0, sizeof(float) * static_cast<size_t>(zero_n), s) != cudaSuccess)
        return MOE_ERR_CUDA;
      return cuda_status(moe::launch_gemv_w13_act(x, w13, sorted, eids, npost, static_cast<int>(P),
                                                  top_k, E, H, I, B, cap, a, s));
  }
}

// early_weights: GEMM 2 directly follows GEMM 1 of the same layer (moe_forward),
// so its weight loads may start before GEMM 1 has finished.
moe_status_t run_gemm2(const uint16_t *a, const uint16_t *w2, const int32_t *sorted,
                       const int32_t *eids, const int32_t *npost, const float *wts, int M,
                       int top_k, int E, int H, int I, int B, float *yacc, int *status,
                       bool early_weights, cudaStream_t s) {
  const long P = static_cast<long>(M) * top_k;
  const int cap = static_cast<int>(capacity(P, E, B));
  switch (pick_path(M, E, top_k, B)) {
    case GemmPath::kTensorCore: {
      const int ks = pick_ksplit(M, E, top_k, (H + 255) / 256, (I + 63) / 64, kSplitCostBf16);
      return cuda_status(moe::launch_tc_w2_combine(a, w2, sorted, eids, npost, wts,
                                                   static_cast<int>(P), top_k, E, H, I, B, cap,
                                                   yacc, ks, status, early_weights, s));
    }
    case GemmPath::kGemv:
    default:
      return cuda_status(moe::launch_gemv_w2_combine(a, w2, sorted, eids, npost, wts,
                                                     static_cast<int>(P), top_k, E, H, I, B, cap,
                                                     yacc, s));
  }
}

// The FP8 grouped GEMMs run on the tensor cores only (E4M3 tiles of the
// tcgen05 kernels); the K split follows the bf16 rule with 128-element stages.
moe_status_t run_gemm1_f8(const uint8_t *qx, const float *sx, const uint8_t *w13,
                          const float *w13s, const int32_t *sorted, const int32_t *eids,
                          const int32_t *npost, int M, int top_k, int E, int H, int I, int B,
                          uint16_t *a, float *h_acc, int *tile_cnt, int *status, bool prefetch,
                          float *zero_dst, long zero_n, cudaStream_t s) {
  const long P = static_cast<long>(M) * top_k;
  const int cap = static_cast<int>(capacity(P, E, B));
  const int ks = h_acc != nullptr
                     ? pick_ksplit(M, E, top_k, (I + 127) / 128, (H + 127) / 128, kSplitCostE4M3)
                     : 1;
  const double D = E * (1.0 - std::pow(1.0 - static_cast<double>(top_k) / E, M));
  const int pf_experts = (prefetch && D >= 0.8 * E) ? E : 0;
  return cuda_status(moe::launch_tc_w13_act_f8(qx, sx, w13, w13s, sorted, eids, npost,
                                               static_cast<int>(P), top_k, E, H, I, B, cap, a, ks,
                                               h_acc, tile_cnt, status, pf_experts, zero_dst,
                                               zero_n, s));
}

moe_status_t run_gemm2_f8(const uint8_t *qa, const float *sa, const uint8_t *w2, const float *w2s,
                          const int32_t *sorted, const int32_t *eids, const int32_t *npost,
                          const float *wts, int M, int top_k, int E, int H, int I, int B,
                          float *yacc, int *status, bool early_weights, cudaStream_t s) {
  const long P = static_cast<long>(M) * top_k;
  const int cap = static_cast<int>(capacity(P, E, B));
  const int ks = pick_ksplit(M, E, top_k, (H + 255) / 256, (I + 127) / 128, kSplitCostE4M3);
  return cuda_status(moe::launch_tc_w2_combine_f8(qa, sa, w2, w2s, sorted, eids, npost, wts,
                                                  static_cast<int>(P), top_k, E, H, I, B, cap,
                                                  yacc, ks, status, early_weights, s));
}

size_t workspace_bytes(int M_max, int E, int top_k, int H, int I, int block_size_m, bool fp8) {
  if (check_shapes(M_max, E, top_k, H, I) != MOE_OK) return 0;
  if (block_size_m != 0 && !valid_block_size(block_size_m)) return 0;
  // a smaller batch may reserve split scratch that M_max does not: the GEMMs'
  // (up to kSplitMaxTokens tokens) or the router's (up to kRouterCtlCount
  // tiles of 128 tokens)
  const int M_split = std::min(M_max, kSplitMaxTokens);
  const int M_rsplit =
      std::min(M_max, moe::kRouterCtlCount / ((E + 255) / 256) * 128);
  auto need = [&](int B) {
    return std::max({ws_layout(M_max, E, top_k, H, I, B, fp8).total,
                     ws_layout(M_split, E, top_k, H, I, B, fp8).total,
                     ws_layout(M_rsplit, E, top_k, H, I, B, fp8).total});
  };
  if (block_size_m != 0) return need(block_size_m);
  size_t best = 0;
  for (int B : {16, 32, 64, 128, 256}) best = std::max(best, need(B));
  return best;
}

}  // namespace

extern "C" {

const char *moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_BAD_EXPERT_ID: return "MOE_ERR_DEVICE_BAD_EXPERT_ID";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
  }
  return "MOE_ERR_UNKNOWN";
}

int moe_pick_block_size(int M, int E, int top_k, int H, int I) {
  if (M <= 0 || E <= 0 || top_k <= 0) return 16;
  const double mean = static_cast<double>(M) * top_k / E;  // mean pairs per expert
  // Blocks a few times the mean group: where the layer streams weights, one
  // block per expert reads each expert's tiles once, and skewed routing
  // (a few experts with many pairs) gains most (Zipf prefill: 256 tokens
  // 193.8 -> 156.2 us with 64-token blocks, 512 tokens 218.4 -> 183.2 with
  // 128, 1024 tokens 243.9 -> 217.6 with 128); decode batches of a few pairs
  // per expert run the same with 16 or 32.
  if (mean <= 6) return 16;
  if (mean <= 12) return 32;
  if (mean <= 24) return 64;
  if (mean <= 64) return 128;
  // 256-token tiles (one N = 256 MMA per K step) pay off once their padding is
  // small next to the groups: from about 64 pairs per expert when both GEMMs
  // run them as 2-SM tiles (an even number of weight tiles: ceil(I/64) for
  // GEMM 1, ceil(H/128) for GEMM 2; E60 tail 1024 tokens 226.1 -> 214.7 us,
  // 2048 tokens 250.0 -> 229.7, Zipf prefill 2048 tokens 288.5 -> 280.6),
  // else from about 1024
  const bool pairs = ((I + 63) / 64) % 2 == 0 && ((H + 127) / 128) % 2 == 0;
  if (pairs || mean >= 1024) return 256;
  return 128;
}

long moe_align_capacity(int M, int top_k, int E, int block_size_m) {
  if (M < 0 || E < 1 || E > kMaxExperts || top_k < 1 || top_k > std::min(E, kMaxTopK) ||
      !valid_block_size(block_size_m))
    return -1;
  return capacity(static_cast<long>(M) * top_k, E, block_size_m);
}

size_t moe_workspace_size(int M_max, int E, int top_k, int H, int I, int block_size_m) {
  return workspace_bytes(M_max, E, top_k, H, I, block_size_m, false);
}

size_t moe_workspace_size_fp8(int M_max, int E, int top_k, int H, int I, int block_size_m) {
  if (block_size_m != 0 && !moe::tc_supports_block(block_size_m)) return 0;
  return workspace_bytes(M_max, E, top_k, H, I, block_size_m, true);
}

moe_status_t moe_router_logits(const moe_bf16_t *x, const moe_bf16_t *w_router,
                               const float *router_bias, int M, int E, int H, moe_bf16_t *logits,
                               cudaStream_t stream) {
  if (M < 0 || E < 1 || E > kMaxExperts) return M < 0 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
  if (H < 16 || H > kMaxDim || H % 16 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return MOE_OK;
  if (!x || !w_router || !logits) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
  return run_router(x, w_router, router_bias, M, E, H, logits, lib_status(), nullptr, nullptr,
                    stream);
}

moe_status_t moe_topk_softmax(const moe_bf16_t *logits, int M, int E, int top_k, int renormalize,
                              int32_t *topk_ids, float *topk_weights, cudaStream_t stream) {
  if (M < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > kMaxExperts || top_k < 1 || top_k > std::min(E, kMaxTopK))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_weights) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      moe::launch_topk_softmax(logits, M, E, top_k, renormalize, topk_ids, topk_weights, stream));
}

moe_status_t moe_align_block_size(const int32_t *topk_ids, int M, int top_k, int E,
                                  int block_size_m, int32_t *sorted_token_ids, int32_t *expert_ids,
                                  int32_t *expert_offsets, int32_t *num_tokens_post_padded,
                                  void *ws, size_t ws_bytes, cudaStream_t stream) {
  if (M < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > kMaxExperts || top_k < 1 || top_k > std::min(E, kMaxTopK) ||
      !valid_block_size(block_size_m))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(M) * top_k >= (1LL << 31) - kMaxExperts * 256LL)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((M > 0 && !topk_ids) || !sorted_token_ids || !expert_ids || !expert_offsets ||
      !num_tokens_post_padded || !ws)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  const long P = static_cast<long>(M) * top_k;
  // the align needs only the status word and its histogram scratch
  const size_t need = round_up(moe::kStatusBytes, kAlign) +
                      sizeof(int32_t) * static_cast<size_t>(moe::align_hist_entries(P, E));
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int *status = at<int>(ws, 0);
  int32_t *hist = at<int32_t>(ws, round_up(moe::kStatusBytes, kAlign));
  const int cap = static_cast<int>(capacity(P, E, block_size_m));
  return cuda_status(moe::launch_align(topk_ids, static_cast<int>(P), E, block_size_m, cap,
                                       sorted_token_ids, expert_ids, expert_offsets,
                                       num_tokens_post_padded, hist, status, stream));
}

moe_status_t moe_grouped_gemm_w13_act(const moe_bf16_t *x, const moe_bf16_t *w13,
                                      const int32_t *sorted_token_ids, const int32_t *expert_ids,
                                      const int32_t *num_tokens_post_padded, int M, int top_k,
                                      int E, int H, int I, int block_size_m, moe_bf16_t *a,
                                      cudaStream_t stream) {
  moe_status_t st = check_shapes(M, E, top_k, H, I);
  if (st != MOE_OK) return st;
  if (!valid_block_size(block_size_m)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return MOE_OK;
  if (!x || !w13 || !sorted_token_ids || !expert_ids || !num_tokens_post_padded || !a)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13)) return MOE_ERR_INVALID_ARG;
  return run_gemm1(x, w13, sorted_token_ids, expert_ids, num_tokens_post_padded, M, top_k, E, H, I,
                   block_size_m, a, nullptr, nullptr, lib_status(), /*prefetch=*/false,
                   /*zero_dst=*/nullptr, 0, stream);
}

moe_status_t moe_grouped_gemm_w2_combine(const moe_bf16_t *a, const moe_bf16_t *w2,
                                         const int32_t *sorted_token_ids,
                                         const int32_t *expert_ids,
                                         const int32_t *num_tokens_post_padded,
                                         const float *topk_weights, const moe_bf16_t *residual,
                                         int M, int top_k, int E, int H, int I, int block_size_m,
                                         moe_bf16_t *y, void *ws, size_t ws_bytes,
                                         cudaStream_t stream) {
  moe_status_t st = check_shapes(M, E, top_k, H, I);
  if (st != MOE_OK) return st;
  if (!valid_block_size(block_size_m)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return MOE_OK;
  if (!a || !w2 || !sorted_token_ids || !expert_ids || !num_tokens_post_padded || !topk_weights ||
      !y || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(w2) || !aligned16(y) || (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(M, E, top_k, H, I, block_size_m);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  float *yacc = at<float>(ws, L.yacc);
  cudaError_t e = cudaMemsetAsync(yacc, 0, sizeof(float) * static_cast<size_t>(M) * H, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  st = run_gemm2(a, w2, sorted_token_ids, expert_ids, num_tokens_post_padded, topk_weights, M,
                 top_k, E, H, I, block_size_m, yacc, at<int>(ws, 0), /*early_weights=*/false,
                 stream);
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_finalize(yacc, residual, M, H, y, stream));
}

moe_status_t moe_forward(const moe_bf16_t *x, const moe_bf16_t *w_router,
                         const moe_bf16_t *router_logits, const float *router_bias,
                         const moe_bf16_t *w13, const moe_bf16_t *w2, const moe_bf16_t *residual,
                         int M, int E, int top_k, int H, int I, int renormalize, int block_size_m,
                         moe_bf16_t *y, int32_t *topk_ids_out, float *topk_weights_out,
                         moe_bf16_t *router_logits_out, void *ws, size_t ws_bytes,
                         cudaStream_t stream) {
  moe_status_t st = check_shapes(M, E, top_k, H, I);
  if (st != MOE_OK) return st;
  if (block_size_m != 0 && !valid_block_size(block_size_m)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((w_router == nullptr) == (router_logits == nullptr)) return MOE_ERR_INVALID_ARG;
  if (router_bias && !w_router) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!x || !w13 || !w2 || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13) || !aligned16(w2) || !aligned16(y) ||
      (residual && !aligned16(residual)) || (w_router && !aligned16(w_router)))
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  const int B = block_size_m != 0 ? block_size_m : moe_pick_block_size(M, E, top_k, H, I);
  const WsLayout L = ws_layout(M, E, top_k, H, I, B);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;

  const long P = static_cast<long>(M) * top_k;
  const int cap = static_cast<int>(capacity(P, E, B));
  int *status = at<int>(ws, L.status);
  int32_t *ids = topk_ids_out ? topk_ids_out : at<int32_t>(ws, L.ids);
  float *wts = topk_weights_out ? topk_weights_out : at<float>(ws, L.wts);
  uint16_t *logits_ws = router_logits_out ? router_logits_out : at<uint16_t>(ws, L.logits);
  if (use_decode_layer(M, E, top_k, H, I))
    return cuda_status(moe::launch_decode_layer(
        x, w_router, router_logits, router_bias, w13, w2, residual, M, E, top_k, H, I,
        renormalize, y, ids, wts, logits_ws, at<uint16_t>(ws, L.a), at<float>(ws, L.yacc),
        status + moe::kDecodeCtlOffset, status, stream));
  int32_t *sorted = at<int32_t>(ws, L.sorted);
  int32_t *eids = at<int32_t>(ws, L.eids);
  int32_t *offs = at<int32_t>(ws, L.offsets);
  int32_t *npost = at<int32_t>(ws, L.npost);
  float *yacc = at<float>(ws, L.yacc);
  const long yn = static_cast<long>(M) * H;
  // the fused routing kernel clears y_acc, and h_acc and the tile counters
  // behind it when GEMM 1 will split its K range (one span)
  const bool want_split = L.hacc != L.tcnt && pick_path(M, E, top_k, B) == GemmPath::kTensorCore &&
                          pick_ksplit(M, E, top_k, (I + 127) / 128, (H + 63) / 64, kSplitCostBf16) > 1;
  const long zn = want_split ? static_cast<long>((L.total - L.yacc) / sizeof(float)) : yn;
  bool zeroed = false;
  st = run_route(x, w_router, router_logits, router_bias, M, E, top_k, H, renormalize, B,
                 logits_ws, ids, wts, sorted, eids, offs, npost,
                 at<int32_t>(ws, L.hist), status,
                 router_may_split(M, E) ? at<float>(ws, L.rscr) : nullptr, yacc, zn, &zeroed,
                 /*skip_sort=*/P * 4 <= E, stream);
  if (st != MOE_OK) return st;
  uint16_t *a = at<uint16_t>(ws, L.a);
  const bool split_ok = zeroed && want_split;  // scratch reserved and cleared
  // not cleared by the routing kernel: GEMM 1 clears it on the way (GEMM 2
  // reads it only after GEMM 1 has completed)
  st = run_gemm1(x, w13, sorted, eids, npost, M, top_k, E, H, I, B, a,
                 split_ok ? at<float>(ws, L.hacc) : nullptr,
                 split_ok ? at<int>(ws, L.tcnt) : nullptr, status, /*prefetch=*/true,
                 zeroed ? nullptr : yacc, yn, stream);
  if (st != MOE_OK) return st;
  st = run_gemm2(a, w2, sorted, eids, npost, wts, M, top_k, E, H, I, B, yacc, status,
                 /*early_weights=*/true, stream);
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_finalize(yacc, residual, M, H, y, stream));
}

moe_status_t moe_route(const moe_bf16_t *x, const moe_bf16_t *w_router,
                       const moe_bf16_t *router_logits, const float *router_bias, int M, int E,
                       int top_k, int H, int renormalize, int block_size_m, int32_t *topk_ids,
                       float *topk_weights, int32_t *sorted_token_ids, int32_t *expert_ids,
                       int32_t *expert_offsets, int32_t *num_tokens_post_padded,
                       moe_bf16_t *router_logits_out, void *ws, size_t ws_bytes,
                       cudaStream_t stream) {
  if (M < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > kMaxExperts || top_k < 1 || top_k > std::min(E, kMaxTopK) ||
      !valid_block_size(block_size_m))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (w_router && (H < 16 || H > kMaxDim || H % 16 != 0)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(M) * top_k >= (1LL << 31) - kMaxExperts * 256LL)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((w_router == nullptr) == (router_logits == nullptr)) return MOE_ERR_INVALID_ARG;
  if (router_bias && !w_router) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if ((w_router && (!x || !aligned16(x) || !aligned16(w_router))) || !topk_ids || !topk_weights ||
      !sorted_token_ids || !expert_ids || !expert_offsets || !num_tokens_post_padded || !ws)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(M, E, top_k, 16, 16, block_size_m);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  bool zeroed = false;
  uint16_t *logits_ws = router_logits_out ? router_logits_out : at<uint16_t>(ws, L.logits);
  return run_route(x, w_router, router_logits, router_bias, M, E, top_k, H, renormalize,
                   block_size_m, logits_ws, topk_ids, topk_weights,
                   sorted_token_ids, expert_ids, expert_offsets, num_tokens_post_padded,
                   at<int32_t>(ws, L.hist), at<int>(ws, 0),
                   router_may_split(M, E) ? at<float>(ws, L.rscr) : nullptr, nullptr, 0, &zeroed,
                   /*skip_sort=*/false, stream);
}

moe_status_t moe_quantize_rows_fp8(const moe_bf16_t *src, int R, int K, uint8_t *q,
                                   float *scales, cudaStream_t stream) {
  if (R < 0) return MOE_ERR_INVALID_ARG;
  if (K < 16 || K > kMaxDim || K % 16 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (R == 0) return MOE_OK;
  if (!src || !q || !scales || !aligned16(src) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_quant_rows(src, R, K, q, scales, stream));
}

moe_status_t moe_grouped_gemm_w13_act_fp8(const uint8_t *qx, const float *x_scales,
                                          const uint8_t *w13, const float *w13_scales,
                                          const int32_t *sorted_token_ids,
                                          const int32_t *expert_ids,
                                          const int32_t *num_tokens_post_padded, int M,
                                          int top_k, int E, int H, int I, int block_size_m,
                                          moe_bf16_t *a, cudaStream_t stream) {
  moe_status_t st = check_shapes(M, E, top_k, H, I);
  if (st != MOE_OK) return st;
  if (!moe::tc_supports_block(block_size_m)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return MOE_OK;
  if (!qx || !x_scales || !w13 || !w13_scales || !sorted_token_ids || !expert_ids ||
      !num_tokens_post_padded || !a)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(qx) || !aligned16(w13)) return MOE_ERR_INVALID_ARG;
  return run_gemm1_f8(qx, x_scales, w13, w13_scales, sorted_token_ids, expert_ids,
                      num_tokens_post_padded, M, top_k, E, H, I, block_size_m, a, nullptr,
                      nullptr, lib_status(), /*prefetch=*/false, /*zero_dst=*/nullptr, 0, stream);
}

moe_status_t moe_grouped_gemm_w2_combine_fp8(const uint8_t *qa, const float *a_scales,
                                             const uint8_t *w2, const float *w2_scales,
                                             const int32_t *sorted_token_ids,
                                             const int32_t *expert_ids,
                                             const int32_t *num_tokens_post_padded,
                                             const float *topk_weights,
                                             const moe_bf16_t *residual, int M, int top_k,
                                             int E, int H, int I, int block_size_m,
                                             moe_bf16_t *y, void *ws, size_t ws_bytes,
                                             cudaStream_t stream) {
  moe_status_t st = check_shapes(M, E, top_k, H, I);
  if (st != MOE_OK) return st;
  if (!moe::tc_supports_block(block_size_m)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return MOE_OK;
  if (!qa || !a_scales || !w2 || !w2_scales || !sorted_token_ids || !expert_ids ||
      !num_tokens_post_padded || !topk_weights || !y || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(qa) || !aligned16(w2) || !aligned16(y) || (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(M, E, top_k, H, I, block_size_m);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  float *yacc = at<float>(ws, L.yacc);
  cudaError_t e = cudaMemsetAsync(yacc, 0, sizeof(float) * static_cast<size_t>(M) * H, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  st = run_gemm2_f8(qa, a_scales, w2, w2_scales, sorted_token_ids, expert_ids,
                    num_tokens_post_padded, topk_weights, M, top_k, E, H, I, block_size_m, yacc,
                    at<int>(ws, 0), /*early_weights=*/false, stream);
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_finalize(yacc, residual, M, H, y, stream));
}

moe_status_t moe_forward_fp8(const moe_bf16_t *x, const moe_bf16_t *w_router,
                             const moe_bf16_t *router_logits, const float *router_bias,
                             const uint8_t *w13, const float *w13_scales, const uint8_t *w2,
                             const float *w2_scales, const moe_bf16_t *residual, int M, int E,
                             int top_k, int H, int I, int renormalize, int block_size_m,
                             moe_bf16_t *y, int32_t *topk_ids_out, float *topk_weights_out,
                             moe_bf16_t *router_logits_out, void *ws, size_t ws_bytes,
                             cudaStream_t stream) {
  moe_status_t st = check_shapes(M, E, top_k, H, I);
  if (st != MOE_OK) return st;
  if (block_size_m != 0 && !moe::tc_supports_block(block_size_m)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((w_router == nullptr) == (router_logits == nullptr)) return MOE_ERR_INVALID_ARG;
  if (router_bias && !w_router) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!x || !w13 || !w13_scales || !w2 || !w2_scales || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13) || !aligned16(w2) || !aligned16(y) ||
      (residual && !aligned16(residual)) || (w_router && !aligned16(w_router)))
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  const int B = block_size_m != 0 ? block_size_m : moe_pick_block_size(M, E, top_k, H, I);
  const WsLayout L = ws_layout(M, E, top_k, H, I, B, /*fp8=*/true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;

  const long P = static_cast<long>(M) * top_k;
  int *status = at<int>(ws, L.status);
  int32_t *ids = topk_ids_out ? topk_ids_out : at<int32_t>(ws, L.ids);
  float *wts = topk_weights_out ? topk_weights_out : at<float>(ws, L.wts);
  uint16_t *logits_ws = router_logits_out ? router_logits_out : at<uint16_t>(ws, L.logits);
  int32_t *sorted = at<int32_t>(ws, L.sorted);
  int32_t *eids = at<int32_t>(ws, L.eids);
  int32_t *offs = at<int32_t>(ws, L.offsets);
  int32_t *npost = at<int32_t>(ws, L.npost);
  float *yacc = at<float>(ws, L.yacc);
  uint8_t *qx = at<uint8_t>(ws, L.qx);
  float *sx = at<float>(ws, L.sx);
  uint8_t *qa = at<uint8_t>(ws, L.qa);
  float *sa = at<float>(ws, L.sa);
  const long yn = static_cast<long>(M) * H;
  const bool want_split =
      L.hacc != L.tcnt &&
      pick_ksplit(M, E, top_k, (I + 127) / 128, (H + 127) / 128, kSplitCostE4M3) > 1;
  const long zn = want_split ? static_cast<long>((L.total - L.yacc) / sizeof(float)) : yn;
  bool zeroed = false;
  st = run_route(x, w_router, router_logits, router_bias, M, E, top_k, H, renormalize, B,
                 logits_ws, ids, wts, sorted, eids, offs, npost, at<int32_t>(ws, L.hist), status,
                 router_may_split(M, E) ? at<float>(ws, L.rscr) : nullptr, yacc, zn, &zeroed,
                 /*skip_sort=*/P * 4 <= E, stream);
  if (st != MOE_OK) return st;
  st = cuda_status(moe::launch_quant_rows(x, M, H, qx, sx, stream));
  if (st != MOE_OK) return st;
  uint16_t *a = at<uint16_t>(ws, L.a);
  const bool split_ok = zeroed && want_split;
  st = run_gemm1_f8(qx, sx, w13, w13_scales, sorted, eids, npost, M, top_k, E, H, I, B, a,
                    split_ok ? at<float>(ws, L.hacc) : nullptr,
                    split_ok ? at<int>(ws, L.tcnt) : nullptr, status, /*prefetch=*/true,
                    zeroed ? nullptr : yacc, yn, stream);
  if (st != MOE_OK) return st;
  st = cuda_status(moe::launch_quant_rows(a, static_cast<int>(P), I, qa, sa, stream));
  if (st != MOE_OK) return st;
  st = run_gemm2_f8(qa, sa, w2, w2_scales, sorted, eids, npost, wts, M, top_k, E, H, I, B, yacc,
                    status, /*early_weights=*/true, stream);
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_finalize(yacc, residual, M, H, y, stream));
}

moe_status_t moe_selftest_device_timeout(void *ws, size_t ws_bytes, int limit_ms,
                                         cudaStream_t stream) {
  if (!ws || ws_bytes < static_cast<size_t>(moe::kStatusBytes)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_selftest_timeout(at<int>(ws, 0), limit_ms, stream));
}

moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws || ws_bytes < static_cast<size_t>(moe::kStatusBytes)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, stream));
}

moe_status_t moe_get_device_status(void *ws, cudaStream_t stream) {
  // ws == NULL: only the library-wide word, which the entry points without a
  // workspace (moe_router_logits, moe_grouped_gemm_w13_act, the _noalloc
  // combine) report into
  int host[2] = {0, 0};
  int *lib = lib_status();
  if (!ws && !lib) return MOE_ERR_CUDA;
  if (ws && cudaMemcpyAsync(&host[0], ws, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (lib && cudaMemcpyAsync(&host[1], lib, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (host[0] != 0 && cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (host[1] != 0 && cudaMemsetAsync(lib, 0, sizeof(int), stream) != cudaSuccess) return MOE_ERR_CUDA;
  if ((host[0] | host[1]) != 0 && cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status_t>(host[0] != 0 ? host[0] : host[1]);
}

}  // extern "C"

// ----------------------------------------------------------------------------
// GEMM 2 + combine without a caller workspace.
//
// Some callers cannot hand the library a workspace: plugin code running inside
// a host application that owns every device allocation and gives the plugin no
// allocator, or latency-critical code that may not call cudaMalloc (it can
// synchronise the device and its latency is unbounded).  For them the fp32
// accumulator of the combine lives in a fixed array compiled into this file.
// Every GPU that loads the library holds the array until the process exits.

namespace {

constexpr long kNoAllocAccElems = 1L << 21;  // 8 MiB of fp32: M * H <= 2,097,152

static __device__ __align__(256) float g_noalloc_acc[kNoAllocAccElems];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
float *g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_acc on the current device, looked up once per
// device.  In host code the array's name is only a host-side stand-in, so the
// kernels must be given this address instead.
moe_status_t noalloc_scratch(float **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_acc) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_grouped_gemm_w2_combine_noalloc(
    const moe_bf16_t *a, const moe_bf16_t *w2, const int32_t *sorted_token_ids,
    const int32_t *expert_ids, const int32_t *num_tokens_post_padded, const float *topk_weights,
    const moe_bf16_t *residual, int M, int top_k, int E, int H, int I, int block_size_m,
    moe_bf16_t *y, cudaStream_t stream) {
  moe_status_t st = check_shapes(M, E, top_k, H, I);
  if (st != MOE_OK) return st;
  if (!valid_block_size(block_size_m)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long>(M) * H > kNoAllocAccElems) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return MOE_OK;
  if (!a || !w2 || !sorted_token_ids || !expert_ids || !num_tokens_post_padded || !topk_weights || !y)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(w2) || !aligned16(y) || (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  float *acc = nullptr;
  st = noalloc_scratch(&acc);
  if (st != MOE_OK) return st;
  // the array keeps the previous call's sums: clear the part this call uses
  if (cudaMemsetAsync(acc, 0, sizeof(float) * static_cast<size_t>(M) * H, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  st = run_gemm2(a, w2, sorted_token_ids, expert_ids, num_tokens_post_padded, topk_weights, M,
                 top_k, E, H, I, block_size_m, acc, lib_status(), /*early_weights=*/false, stream);
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_finalize(acc, residual, M, H, y, stream));
}
