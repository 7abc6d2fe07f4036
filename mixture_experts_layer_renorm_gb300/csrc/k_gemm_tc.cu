// k_gemm_tc.cu -- S3 / S4 on the 5th-generation tensor cores (tcgen05): the
// grouped GEMMs of the layer with their fused epilogues.
//
// Page "Mixture of Experts in vLLM - From First Principles to fused_moe",
// sections "Each expert is now an ordinary GEMM", "One GEMM 1 program, step
// by step" and "The rest of the layer stays in pair order": every block of
// B = block_size_m entries of sorted_token_ids belongs to one expert; its
// rows are read in place through the pair id (GEMM 1: row p / top_k of x;
// GEMM 2: row p of the activation) and its results go straight to the pair's
// or token's final place.
//
// One CTA computes one block against a tile of weight rows, with the operands
// swapped so that the weight rows fill the MMA's M = 128 dimension and the
// block's B gathered rows are its N dimension (N = B in {16, ..., 256}):
//
//   GEMM 1: D_gate[128, B] = W13_e[i0 .. i0+127, :] . X_b^T
//           D_up  [128, B] = W13_e[I+i0 .. I+i0+127, :] . X_b^T
//           epilogue: a[p, i] = bf16(SiLU(bf16(gate)) * bf16(up)) -- the gate
//           row and its up row share a TMEM lane, so one thread forms a.
//   GEMM 2: D_0/1 [128, B] = W2_e[n0 .. n0+255, :] . A_b^T
//           epilogue: y_acc[t, n] += topk_weight[p] * D (fp32 red.add)
//
// 256-token blocks use one N = 256 MMA per K step on a single 128-row weight
// tile (GEMM 1: 64 gate rows over the matching 64 up rows, whose results the
// epilogue warp pairs trade through shared memory; GEMM 2: 128 rows of W2),
// so that two accumulators still fit TMEM: a chain of N = 128 MMAs into one
// accumulator leaves the tensor pipe idle between instructions.
//
// 2-SM tiles: where the weight tiles of a 256-token GEMM come in an even
// number, CTAs run in clusters of two on neighbouring weight tiles of the same
// block and the even CTA issues M = 256 MMAs (tcgen05 cta_group::2) over both
// CTAs' shared memory.  Each CTA gathers only its half of the block's rows
// (stages of 32 KB instead of 48, so six fit); the odd CTA's relay warp tells
// the even CTA's MMA lane when its half of a stage has landed, the MMA
// completions release both CTAs' stages (multicast commits), and each CTA's
// epilogue writes its own 128 rows from its own tensor memory.
//
// Persistent CTAs (one per SM, or pairs) walk the list of (block, weight tile) tiles;
// GEMM 2 with a large combine accumulator walks it in ranges of weight tiles
// so the live part of the accumulator stays in L2.  Every launch is a
// programmatic dependent launch: the CTAs wait (griddepcontrol.wait) only
// where they read what an earlier kernel wrote -- in a layer, GEMM 2's weights
// stream before GEMM 1 has finished, and decode GEMM 1 brings the first
// wave's expert weights into L2 while routing runs.
// Warp roles (480 threads): warp 0 -- one lane issues the TMA copies of the
// two 128 x 64 weight tiles (128-byte swizzle); warps 10-13 gather the block's
// rows with 16-byte cp.async into the same swizzled K-major layout (a TMA
// instruction costs too much issue time per 512 bytes to gather with it);
// warp 1 allocates TMEM and one lane issues tcgen05.mma; warps 2-9 are the
// epilogue, two per TMEM lane quarter splitting its columns (tcgen05.ld
// 32x32b); warp 14 relays stage completion in 2-SM tiles.  Waiting threads sleep in mbarrier.try_wait rather than spin.  Two
// accumulator buffers in TMEM let the epilogue of one tile
// overlap the mainloop of the next.  A ring of shared-memory stages with
// full/empty mbarriers connects the roles.  Every wait is bounded: after
// about 2 s the kernel records MOE_ERR_DEVICE_TIMEOUT in the status word,
// lets its own copies land and returns; it never traps.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kEpiWarps = 8;                         // warps 2..9: two per TMEM lane quarter
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kGatherWarp0 = 2 + kEpiWarps;          // warps 10..13 gather the block's rows
constexpr int kGatherWarps = 4;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kRelayWarp = kGatherWarp0 + kGatherWarps;  // warps 14, 15: 2-SM tiles, second CTA
constexpr int kRelayWarps = 2;                           // stage g is relayed by warp 14 + g % 2
constexpr int kTcThreads = 64 + kEpiThreads + kGatherThreads + 32 * kRelayWarps;
// 2-SM tiles: accumulator buffers per CTA
constexpr int kPairAccBufs = 2;
constexpr bool kPairTiles = true;  // 256-token tiles run as 2-SM tiles where they can
constexpr int kBK = 64;                              // K per stage: one 128-byte swizzle row
constexpr int kTileM = 128;                          // weight rows per MMA
constexpr uint32_t kATileBytes = kTileM * kBK * 2;   // 16 KB
constexpr int kSmemBudget = 220 * 1024;
constexpr int kMaxStages = 6;
constexpr long long kWaitLimitCycles = 4000000000ll;  // about 2 s at the SM clock
constexpr uint32_t kSuspendHintNs = 20000;           // a waiting thread sleeps until the phase completes

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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
// As mbar_try_wait, but the thread may stay suspended (off the issue slots the
// other roles need) for up to kSuspendHintNs unless the phase completes first.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// The same wait with cluster-scope acquire semantics: the phase's arrivals
// from the other CTA of a pair, made with release semantics at cluster scope,
// happen-before everything this thread does after the wait returns.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of the barrier; gives up after about 2 s of SM
// clock (or when another role already gave up), recording the timeout.
// cluster_acquire: the barrier collects arrivals from the other CTA of a pair.
__device__ bool wait_bounded_for(uint32_t bar, uint32_t parity, volatile int *abort, int *status,
                                 long long limit_cycles, bool cluster_acquire = false) {
  if (cluster_acquire ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (cluster_acquire ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait_sleep(bar, parity))
        return true;
    if (*abort) return false;
    if (clock64() - t0 > limit_cycles) {
      *abort = 1;
      report_status(status, kStatusTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort,
                                             int *status, bool cluster_acquire = false) {
  return wait_bounded_for(bar, parity, abort, status, kWaitLimitCycles, cluster_acquire);
}

// The failure path of wait_bounded, on its own: an mbarrier that nothing
// completes, waited for limit_cycles.
__global__ void k_selftest_timeout(int *status, long long limit_cycles) {
  __shared__ uint64_t bar;
  __shared__ volatile int abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)wait_bounded_for(smem_u32(&bar), 0, &abort, status, limit_cycles);
}

// ---------------------------------------------------------------- copies

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// Brings [src, src + bytes) into L2 (bytes a multiple of 16, src 16-byte aligned).
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Arrives on the barrier once every cp.async this thread issued so far has
// landed; the barrier's expected count already includes this arrival.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// Orders shared-memory writes made through the generic proxy (the row
// gathers), which this thread has observed through an mbarrier, before its
// following async-proxy accesses (the tensor core's operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] . B[smem]^T, E4M3 inputs, fp32 accumulate (K = 32 per
// instruction: the same 32 bytes of each row as a bf16 MMA's K = 16).
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on the barrier when every MMA this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// The same for a pair of CTAs (cta_group::2): an M = 256 MMA whose A rows
// 0-127 and B rows 0..N/2-1 come from the even CTA's shared memory and A rows
// 128-255 and B rows N/2..N-1 from the odd CTA's, at the same offsets; each
// CTA's tensor memory receives its 128 rows of D.  Issued by the even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on the barrier at this offset in both CTAs of the pair when
// every pair MMA this thread issued has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  const uint16_t both = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(both)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Address in CTA `rank` of the cluster of the shared variable at saddr here.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// One arrival on a barrier of another CTA of the cluster (address from
// map_to_cta), with release semantics at cluster scope: what this thread has
// observed before the arrival (tensor-memory loads it waited for) happens-
// before whatever the other CTA does after its cluster-scope acquire of the
// phase (every wait of the MMA lane on a barrier the other CTA arrives on).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The per-stage hand-off of the second CTA's rows to the first CTA's MMA.
// Its arrival is relaxed unless the library is built with
// -DMOE_STRICT_CLUSTER_ORDER: a release at cluster scope drains this SM's
// outstanding memory requests (the row gathers of the following stages among
// them) and measured 45 % slower GEMM 1 at M = 4096 and 16384 (one arrival per
// stage).  Without it the ordering rests on the hardware, not on the PTX
// memory model: the relaying thread has seen the stage's rows land in this
// CTA's own shared memory (its acquire of this CTA's barrier) and has made
// them visible to this CTA's tensor-core proxy (fence.proxy.async) before it
// issues the arrival; the first CTA issues the MMA only after the arrival
// reaches it, and this CTA's tensor core reads its half of the operands from
// its own shared memory.
__device__ __forceinline__ void mbar_arrive_stage_relay(uint32_t bar) {
#ifdef MOE_STRICT_CLUSTER_ORDER
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
#else
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
#endif
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core groups 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused with this swizzle)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;    // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;            // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;            // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor of kind::f8f6f4: E4M3 A and B (K-major), fp32 D, M x N
// (A and B format fields 0 = E4M3).
__host__ __device__ constexpr uint32_t umma_idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

template <int N, int MODE, bool P2 = false>
struct TcConfig {
  // Wide tiles (N = 256 token columns, GEMMs 1 and 2): ONE 128-row weight tile
  // per stage -- for GEMM 1 its 64 gate rows over the matching 64 up rows -- so
  // one accumulator takes N TMEM columns and two of them fit.  An N = 256 MMA
  // keeps the tensor pipe busy where a chain of dependent N = 128 MMAs into
  // one accumulator does not.  Narrower tiles use two 128-row weight tiles
  // (GEMM 1: gate and up, GEMM 2 and the router: 256 rows).
  static constexpr bool kWide = N == 256 && MODE != 2;
  static constexpr int kATiles = kWide ? 1 : 2;               // 128-row weight tiles per stage
  static constexpr int kRowsPerCTile = kWide && MODE == 0 ? 64 : kATiles * kTileM;  // output rows
  // 2-SM tiles (P2): each CTA of the pair holds half of the block's rows
  static constexpr int kBRows = P2 ? N / 2 : N;
  static constexpr uint32_t kBStageBytes = kBRows * kBK * 2;
  static constexpr uint32_t kStageBytes = kATiles * kATileBytes + kBStageBytes;
  // wide GEMM 1: gate and up of a channel sit in different TMEM lane quarters;
  // each pair of epilogue warps trades half of its bf16 values through a
  // double-buffered slot of 2 x 1 KB (4 pairs)
  // wide GEMM 2: per epilogue warp a 16 x 32 fp32 staging tile for 16-byte reductions
  static constexpr uint32_t kXchgBytes =
      !kWide ? 0 : MODE == 0 ? 4 * 2 * 2 * 32 * 32 : kEpiWarps * 16 * 32 * 4;
  static constexpr int kStages =
      ((kSmemBudget - static_cast<int>(kXchgBytes)) / static_cast<int>(kStageBytes)) < kMaxStages
          ? (kSmemBudget - static_cast<int>(kXchgBytes)) / static_cast<int>(kStageBytes)
          : kMaxStages;
  // accumulator buffers in TMEM: two (epilogue of one tile overlaps the
  // mainloop of the next) while both fit the 512 columns
  static constexpr uint32_t kAccCols = kATiles * N;
  static constexpr int kAccBufs = P2 ? kPairAccBufs : (2 * kAccCols <= 512) ? 2 : 1;
  static constexpr uint32_t kTmemCols = (kAccBufs * kAccCols <= 32) ? 32
                                        : (kAccBufs * kAccCols <= 64) ? 64
                                        : (kAccBufs * kAccCols <= 128) ? 128
                                        : (kAccBufs * kAccCols <= 256) ? 256 : 512;
  // 16-byte chunks of one stage's gathered rows per gather thread
  static constexpr int kChunksPerThread = kBRows * 8 / kGatherThreads;
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2]; tmem address,
  // abort flag; epilogue destination rows[N], weights[N]
  static constexpr uint32_t kCtlBytes = 8 * (2 * kStages + 4) + 16 + 8 * N;
  static constexpr uint32_t kSmemBytes = 1024 + kStages * kStageBytes + kXchgBytes + kCtlBytes;
  static_assert(kStages >= 3, "pipeline needs at least three stages");
  static_assert(kBRows * 8 % kGatherThreads == 0, "gather threads split a stage evenly");
  static_assert(!P2 || kWide, "2-SM tiles are 256-token tiles");
  static_assert(kAccBufs * kAccCols <= 512, "accumulators fit TMEM");
};

// Tile t of the persistent schedule: block b, weight tile c, and the K-stage
// range [kb0, kb1) of split sp (ksplit <= nk splits; the splits of one tile are
// neighbours in the schedule and run side by side).  With n_pass > 1 (GEMM 2
// with a large combine accumulator) the weight tiles are cut into n_pass
// ranges of ctp tiles, run one range after the other over every block: while
// a range runs only its columns of y_acc are live, small enough to stay in L2
// across the top_k additions each token receives.
struct TileCoord {
  int b, c, kb0, kb1;
};
struct TileSched {
  int n_ctiles, ksplit, nk, n_pass, ctp, per_pass;
};
__device__ __forceinline__ TileSched make_sched(int n_ctiles, int ksplit, int nk, int n_blocks,
                                                int n_pass) {
  TileSched s;
  s.n_ctiles = n_ctiles;
  s.ksplit = ksplit;
  s.nk = nk;
  s.n_pass = max(1, n_pass);
  s.ctp = (n_ctiles + s.n_pass - 1) / s.n_pass;
  s.per_pass = n_blocks * s.ctp * ksplit;
  return s;
}
__device__ __forceinline__ TileCoord tile_coord(int t, const TileSched &s) {
  int p = 0, ct = s.n_ctiles;
  if (s.n_pass > 1) {  // every range but the last holds ctp weight tiles
    p = min(t / s.per_pass, s.n_pass - 1);
    t -= p * s.per_pass;
    ct = min(s.ctp, s.n_ctiles - p * s.ctp);
  }
  const int per_b = ct * s.ksplit;
  TileCoord tc;
  tc.b = t / per_b;
  const int r = t - tc.b * per_b;
  const int cl = r / s.ksplit;
  tc.c = p * s.ctp + cl;
  const int sp = r - cl * s.ksplit;
  // balanced ranges: none is empty while ksplit <= nk (an empty range would
  // hand the epilogue an accumulator that no MMA of this tile wrote)
  tc.kb0 = sp * s.nk / s.ksplit;
  tc.kb1 = (sp + 1) * s.nk / s.ksplit;
  return tc;
}

// a = bf16( SiLU(bf16(gate)) * bf16(up) ) from fp32 GEMM-1 sums.
// The fast exponential and division (a few fp32 ulps) are far below the final
// bf16 rounding; 1 + exp(-g) = inf for very negative g gives SiLU = -0.
__device__ __forceinline__ uint16_t silu_mul_bf16(float gate, float up) {
  const float gb = bf16_bits_to_float(float_to_bf16_bits(gate));
  const float ub = bf16_bits_to_float(float_to_bf16_bits(up));
  const float silu = __fdividef(gb, 1.0f + __expf(-gb));
  return float_to_bf16_bits(silu * ub);
}

// Two fp32 values -> bf16x2 bits (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return static_cast<uint32_t>(float_to_bf16_bits(lo)) |
         (static_cast<uint32_t>(float_to_bf16_bits(hi)) << 16);
}

__device__ __forceinline__ void epilogue_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");  // the epilogue warps only
}
// Named barriers 2..5: the two warps of one exchange pair of the epilogue.
__device__ __forceinline__ void pair_bar_sync(int pair) {
  switch (pair) {
    case 0: asm volatile("bar.sync 2, 64;" ::: "memory"); break;
    case 1: asm volatile("bar.sync 3, 64;" ::: "memory"); break;
    case 2: asm volatile("bar.sync 4, 64;" ::: "memory"); break;
    default: asm volatile("bar.sync 5, 64;" ::: "memory"); break;
  }
}

// Persistent tiles (tile_coord): block, weight tile, K split; the weight tiles
// (and splits) of one block are neighbours, so concurrently running CTAs share
// the block's gathered rows and the expert's weights in L2.  With ksplit > 1
// (decode-sized GEMM 1 with too few tiles for the SMs) each split adds its
// fp32 partial gate/up sums into h_acc [P, 2I] and the last split of the tile
// forms a; h_acc and tile_cnt must be zero on entry and tile_cnt is left zero.
// early_weights: only the row gathers wait for the previous kernel (GEMM 2 in
// a layer); n_pass: ranges of weight tiles (GEMM 2); w_pf / pf_bytes: weights
// GEMM 1 brings into L2 before its dependency wait.
//
// MODE 0: GEMM 1 + SiLU-and-mul   rows = x[p / top_k], A = W13_e gate | up tiles,
//                                 a[p, i] = bf16(SiLU(bf16 gate) * bf16 up)
// MODE 1: GEMM 2 + combine        rows = a[p],         A = W2_e rows n0..n0+255,
//                                 y_acc[p / top_k, n] += topk_w[p] * o
// MODE 2: router logits           rows = x[t] (blocks of N consecutive tokens),
//                                 A = W_r rows e0..e0+255, logits[t, e] = bf16(D + bias[e])
//
// F8 (GEMM 1 and 2): E4M3 weights and E4M3 rows (src holds codes, one byte
// each), one fp32 scale per weight row (row_scale [E, a_rows]) and per source
// row (col_scale: per token for GEMM 1, per pair for GEMM 2); the sums are
// scaled by both before the epilogue's rounding or combine.  A stage then
// covers 128 K elements (the same 128 bytes per row).
template <int N, int MODE, bool P2, bool F8>
__global__ void __launch_bounds__(kTcThreads, 1)
k_gemm_tc(const __grid_constant__ CUtensorMap tmap_w, const uint16_t *__restrict__ src,
          int src_rows, const int32_t *__restrict__ sorted_ids, const int32_t *__restrict__ expert_ids,
          const int32_t *__restrict__ n_post_ptr, const float *__restrict__ vec, int P, int top_k,
          int E, int K, int R_out, int a_rows, int B, int cap, int n_ctiles, int ksplit,
          float *__restrict__ h_acc, int *__restrict__ tile_cnt, uint16_t *__restrict__ out16,
          float *__restrict__ y_acc, int H_out, int *status, int early_weights, int n_pass,
          const uint8_t *__restrict__ w_pf, long pf_bytes, float4 *__restrict__ zero_dst,
          long zero_n4, const float *__restrict__ row_scale, const float *__restrict__ col_scale) {
  using Cfg = TcConfig<N, MODE, P2>;
  constexpr int S = Cfg::kStages;
  static_assert(!F8 || MODE != 2, "the router runs in bf16");
  constexpr int kElt = F8 ? 1 : 2;              // bytes per element
  constexpr int kBKe = kBK * 2 / kElt;          // K elements per stage (128 bytes per row)
  // With early_weights (GEMM 2 right after GEMM 1 in one layer) only the row
  // gathers wait for the previous kernel: the weight tiles and the routing
  // lists it reads were final before GEMM 1 started, so the weights stream
  // while GEMM 1 drains.
  const bool early = MODE == 1 && early_weights != 0;
  // Decode GEMM 1 inside a layer: while routing still runs, the CTAs bring the
  // weights their first tiles will most likely read (the lowest experts' W13,
  // pf_bytes from w_pf) into L2; the host asks only when most of the experts
  // are routed to.  Weights never change, so this needs no wait.
  if (MODE == 0 && pf_bytes > 0 && threadIdx.x == 0) {
    const long slice = ((pf_bytes + gridDim.x - 1) / gridDim.x + 15) / 16 * 16;
    const long begin = (long)blockIdx.x * slice;
    const long end = min(pf_bytes, begin + slice);
    for (long o = begin; o < end; o += 65536) prefetch_l2_bulk(w_pf + o, (uint32_t)min(65536l, end - o));
  }
  // 2-SM tiles (P2, clusters of two): the pair's tile t covers weight tiles
  // c = 2 c2 (even CTA) and 2 c2 + 1 (odd CTA) of one block; the even CTA
  // issues M = 256 MMAs over both CTAs' shared memory, each CTA gathers half of
  // the block's rows and loads its own weight tile, and each CTA's epilogue
  // writes its own 128 rows.
  const int rank = P2 ? static_cast<int>(cluster_ctarank()) : 0;
  const int t0 = P2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tstride = P2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int n_cunits = P2 ? n_ctiles / 2 : n_ctiles;

  // Set-up that reads nothing an earlier kernel writes -- barriers, tensor
  // memory, the weight map's descriptor -- runs before the dependency wait,
  // while the previous kernel finishes.
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *a_tiles = smem;                                   // [S][kATiles][16 KB]
  uint8_t *b_tiles = smem + S * Cfg::kATiles * kATileBytes;  // [S][N * 128 B]
  uint8_t *xchg = b_tiles + S * Cfg::kBStageBytes;  // wide GEMM 1: [4 pairs][2][2 KB]; GEMM 2: [8 warps][2 KB]
  uint64_t *bars = reinterpret_cast<uint64_t *>(xchg + Cfg::kXchgBytes);
  uint64_t *full = bars;
  uint64_t *empty = bars + S;
  uint64_t *acc_full = bars + 2 * S;
  uint64_t *acc_empty = bars + 2 * S + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 4);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *dst_row = reinterpret_cast<int *>(tmem_slot + 4);     // epilogue's current block
  float *dst_w = reinterpret_cast<float *>(dst_row + N);
  volatile int *split_last = reinterpret_cast<volatile int *>(tmem_slot + 2);
  volatile int *epi_stop = reinterpret_cast<volatile int *>(tmem_slot + 3);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // the weight lane's expect_tx + one cp.async-completion arrival per gather thread
      // (2-SM tiles, even CTA: plus the odd CTA's relay arrival)
      mbar_init(smem_u32(&full[s]), 1 + kGatherThreads + (P2 && rank == 0 ? 1 : 0));
      mbar_init(smem_u32(&empty[s]), 1);      // one tcgen05.commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&acc_full[a]), 1);   // one tcgen05.commit
      // one arrive per epilogue warp (2-SM tiles, even CTA: of both CTAs)
      mbar_init(smem_u32(&acc_empty[a]), (P2 && rank == 0 ? 2 : 1) * kEpiWarps);
    }
    *abort = 0;
    *epi_stop = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if constexpr (P2) {
      tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (P2) cluster_sync();  // the other CTA's barriers exist before any arrival
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");

  if (!early) griddep_wait();
  griddep_launch_dependents();
  int n_blocks;
  if (MODE == 2) {
    n_blocks = (src_rows + N - 1) / N;
  } else {
    const int n_post = min(max(*n_post_ptr, 0), cap);
    n_blocks = n_post / B;
  }
  // This CTA's work: n_work tiles (block, weight tile, K-stage range), tiles
  // t0, t0 + tstride, ... of the persistent schedule, each split ksplit ways
  // along K.
  const int kspl = ksplit < 1 ? 1 : ksplit;
  const int nk = (K + kBKe - 1) / kBKe;
  const int Mt = MODE == 2 ? (src_rows + N - 1) / N * N : 0;  // router: tokens of all tiles
  const int n_tiles = n_blocks * n_cunits * kspl;
  const TileSched sched = make_sched(n_cunits, kspl, nk, n_blocks, MODE == 1 ? n_pass : 1);
  const int n_work = t0 < n_tiles ? (n_tiles - 1 - t0) / tstride + 1 : 0;
  auto work = [&](int j) {
    TileCoord tc = tile_coord(t0 + j * tstride, sched);
    if (P2) tc.c = 2 * tc.c + rank;
    return tc;
  };
  // GEMM 1 inside a layer clears the combine accumulator that GEMM 2 adds
  // into (zero_n4 float4s at zero_dst): each CTA its slice, the epilogue warps
  // while the first tile's mainloop runs (GEMM 2 reads it only after this
  // kernel has completed).
  auto zero_slice = [&](int tid, int nthreads) {
    const long slice = (zero_n4 + gridDim.x - 1) / gridDim.x;
    const long begin = static_cast<long>(blockIdx.x) * slice;
    const long end = min(zero_n4, begin + slice);
    for (long i = begin + tid; i < end; i += nthreads) zero_dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  };
  if (n_work == 0) {  // (both CTAs of a pair leave here together)
    // this kernel must not finish before the one it follows has: the next
    // kernels count on that when they reuse what it read
    if (early) griddep_wait();
    if (MODE == 0 && zero_n4 > 0) zero_slice(threadIdx.x, blockDim.x);
    // give back the tensor memory allocated above (a pair: both CTAs)
    tc_fence_before();
    __syncthreads();
    if constexpr (P2) {
      cluster_sync();
      if (warp == 1) tmem_dealloc_pair(tmem, Cfg::kTmemCols);
    } else {
      if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
    }
    return;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ weight tiles (TMA)
    // The next tile's expert id is loaded while this tile's copies go out.  An
    // id outside [0, E) needs no test here: its tiles lie outside the map and
    // read as zeros, and the epilogue writes nothing for that block.
    if (lane == 0) {
      int g = 0;
      bool stop = false;
      int e_next = MODE == 2 ? 0 : expert_ids[work(0).b];
      for (int j = 0; j < n_work && !stop; ++j) {
        const TileCoord tc = work(j);
        const int c = tc.c;
        const int e = e_next;
        if (MODE != 2 && j + 1 < n_work) e_next = expert_ids[work(j + 1).b];
        // weight rows of the stage's tile(s); wide GEMM 1 loads 64 gate rows
        // and the matching 64 up rows as the two halves of one 128-row tile
        // (the map's box is then 64 rows high)
        int row0, row1;
        bool two;
        if (Cfg::kWide) {
          row0 = c * Cfg::kRowsPerCTile;
          row1 = R_out + c * Cfg::kRowsPerCTile;
          two = MODE == 0;
        } else {
          row0 = MODE == 0 ? c * kTileM : c * 2 * kTileM;
          row1 = MODE == 0 ? R_out + c * kTileM : c * 2 * kTileM + kTileM;
          two = MODE == 0 || row1 < a_rows;
        }
        const uint32_t second = Cfg::kWide ? kATileBytes / 2 : kATileBytes;
        const uint32_t tx = Cfg::kWide ? kATileBytes : (two ? 2 : 1) * kATileBytes;
        for (int kb = tc.kb0; kb < tc.kb1; ++kb, ++g) {
          const int s = g % S;
          if (!wait_bounded(smem_u32(&empty[s]), ((g / S) & 1) ^ 1, abort, status)) {
            stop = true;
            break;
          }
          const uint32_t fb = smem_u32(&full[s]);
          const uint32_t a_s = smem_u32(a_tiles + s * Cfg::kATiles * kATileBytes);
          mbar_arrive_expect_tx(fb, tx);
          tma_load_3d(a_s, &tmap_w, kb * kBKe, row0, e, fb);
          if (two) tma_load_3d(a_s + second, &tmap_w, kb * kBKe, row1, e, fb);
        }
      }
      if constexpr (P2) {
        // the even CTA's MMAs release this CTA's stages with multicast
        // commits: wait for the last of them before leaving
        for (int g2 = g; g2 < g + S; ++g2)
          (void)wait_bounded(smem_u32(&empty[g2 % S]), ((g2 / S) & 1) ^ 1, abort, status);
      }
      // after an abort: let the copies already issued land before exit
      if (*abort) {
        for (int g2 = (g > S ? g - S : 0); g2 < g; ++g2) {
          const long long t0 = clock64();
          while (!mbar_try_wait(smem_u32(&full[g2 % S]), (g2 / S) & 1) &&
                 clock64() - t0 < kWaitLimitCycles) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp >= kRelayWarp) {
    // ------------------------------------------------------------ relay (2-SM tiles, odd CTA)
    // Once a stage of this CTA (its weight tile and its half of the rows) is
    // complete, one arrival on the even CTA's full barrier for that stage.
    // Stage g is relayed by warp kRelayWarp + g % kRelayWarps, so that the
    // arrivals' release of one stage overlaps the wait for the next.
    const int rw = warp - kRelayWarp;
    if (P2 && rank == 1 && lane == 0) {
      int g = 0;
      bool stop = false;
      for (int j = 0; j < n_work && !stop; ++j) {
        const TileCoord tc = work(j);
        for (int kb = tc.kb0; kb < tc.kb1; ++kb, ++g) {
          if (g % kRelayWarps != rw) continue;
          const int sf = g % S;
          if (!wait_bounded(smem_u32(&full[sf]), (g / S) & 1, abort, status)) {
            stop = true;
            break;
          }
          fence_proxy_async_smem();  // the rows were written by cp.async
          mbar_arrive_stage_relay(map_to_cta(smem_u32(&full[sf]), 0));
        }
      }
    }
    __syncwarp();
  } else if (warp >= kGatherWarp0) {
    // ------------------------------------------------------------ row gathers (cp.async)
    // Thread gt copies chunk (gt & 7) -- 16 bytes of the stage's 128-byte K
    // slice -- of rows gt/8, gt/8 + 16, ...; the hardware arrives on the
    // stage's full barrier for it when those copies land, so the thread moves
    // straight on to the next stage.
    const int gt = threadIdx.x - kGatherWarp0 * 32;
    const int ch = gt & 7;
    // Entries of sorted_token_ids (MODE 2: token ids) of this thread's rows in
    // tile t; the next tile's are loaded while this tile's rows are copied.
    // (2-SM tiles: this CTA's rows are the block's rows rank * N/2 + r)
    const int rbase = P2 ? rank * Cfg::kBRows : 0;
    auto fetch_ids = [&](int j, int (&ids)[Cfg::kChunksPerThread]) {
      const int b = work(j).b;
#pragma unroll
      for (int u = 0; u < Cfg::kChunksPerThread; ++u) {
        const int r = rbase + (gt >> 3) + 16 * u;
        if (MODE == 2) ids[u] = b * N + r;
        else ids[u] = r < B ? sorted_ids[(size_t)b * B + r] : -1;
      }
    };
    int ids_next[Cfg::kChunksPerThread];
    fetch_ids(0, ids_next);
    // the gathered rows are the previous kernel's output; the row ids (the
    // routing lists, final before GEMM 1 started) were loaded before the wait
    if (early) griddep_wait();
    int g = 0;
    bool stop = false;
    for (int j = 0; j < n_work && !stop; ++j) {
      const TileCoord tc = work(j);
      int rowv[Cfg::kChunksPerThread];
#pragma unroll
      for (int u = 0; u < Cfg::kChunksPerThread; ++u) {
        const int p = ids_next[u];
        int row = -1;
        if (MODE == 2) {
          if (p < src_rows) row = p;
        } else if (p >= 0 && p < P) {
          row = MODE == 0 ? p / top_k : p;
        }
        rowv[u] = row;
      }
      if (j + 1 < n_work) fetch_ids(j + 1, ids_next);
      for (int kb = tc.kb0; kb < tc.kb1; ++kb, ++g) {
        const int s = g % S;
        if (!wait_bounded(smem_u32(&empty[s]), ((g / S) & 1) ^ 1, abort, status)) {
          stop = true;
          break;
        }
        const uint32_t b_s = smem_u32(b_tiles + s * Cfg::kBStageBytes);
        const int kel = kb * kBKe + ch * (16 / kElt);  // first element of this thread's chunk
        const uint8_t *srcb = reinterpret_cast<const uint8_t *>(src);
#pragma unroll
        for (int u = 0; u < Cfg::kChunksPerThread; ++u) {
          const int r = (gt >> 3) + 16 * u;
          const bool ok = rowv[u] >= 0 && kel < K;
          const uint8_t *gp = ok ? srcb + ((size_t)rowv[u] * K + kel) * kElt : srcb;
          const uint32_t dst = b_s + (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
          cp_async_16(dst, gp, ok ? 16u : 0u);
        }
        cp_async_arrive_noinc(smem_u32(&full[s]));
      }
    }
    cp_async_wait<0>();  // nothing of ours still in flight at exit
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0 && (!P2 || rank == 0)) {
      constexpr uint32_t idesc = F8 ? umma_idesc_e4m3(P2 ? 2 * kTileM : kTileM, N)
                                    : umma_idesc_bf16(P2 ? 2 * kTileM : kTileM, N);
      int g = 0, i = 0;
      bool stop = false;
      for (int j = 0; j < n_work && !stop; ++j) {
        const TileCoord tc = work(j);
        const bool two = !Cfg::kWide && (MODE == 0 || tc.c * 2 * kTileM + kTileM < a_rows);
        const int acc = i % Cfg::kAccBufs;
        const uint32_t use = i / Cfg::kAccBufs;
        ++i;
        if (!wait_bounded(smem_u32(&acc_empty[acc]), (use & 1) ^ 1, abort, status, P2)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + acc * Cfg::kAccCols;
        for (int kb = tc.kb0; kb < tc.kb1; ++kb, ++g) {
          const int s = g % S;
          if (!wait_bounded(smem_u32(&full[s]), (g / S) & 1, abort, status, P2)) {
            stop = true;
            break;
          }
          fence_proxy_async_smem();  // the gathered rows were written by cp.async
          tc_fence_after();
          const uint32_t a0 = smem_u32(a_tiles + s * Cfg::kATiles * kATileBytes);
          const uint32_t a1 = a0 + kATileBytes;
          const uint32_t bt = smem_u32(b_tiles + s * Cfg::kBStageBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t accumulate = (kb > tc.kb0 || kk > 0) ? 1u : 0u;
            const uint64_t bd = sw128_kmajor_desc(bt + kk * 32);
            if constexpr (P2 && F8) {
              umma_e4m3_pair(d0, sw128_kmajor_desc(a0 + kk * 32), bd, idesc, accumulate);
            } else if constexpr (P2) {
              umma_bf16_pair(d0, sw128_kmajor_desc(a0 + kk * 32), bd, idesc, accumulate);
            } else if constexpr (F8) {
              umma_e4m3(d0, sw128_kmajor_desc(a0 + kk * 32), bd, idesc, accumulate);
              if (two) umma_e4m3(d0 + N, sw128_kmajor_desc(a1 + kk * 32), bd, idesc, accumulate);
            } else {
              umma_bf16(d0, sw128_kmajor_desc(a0 + kk * 32), bd, idesc, accumulate);
              if (two) umma_bf16(d0 + N, sw128_kmajor_desc(a1 + kk * 32), bd, idesc, accumulate);
            }
          }
          if constexpr (P2) umma_commit_pair(smem_u32(&empty[s]));
          else umma_commit(smem_u32(&empty[s]));
        }
        if constexpr (P2) umma_commit_pair(smem_u32(&acc_full[acc]));
        else umma_commit(smem_u32(&acc_full[acc]));
      }
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    // (exactly these warps meet the epilogue's named barriers)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // the two warps of a quarter split the column chunks
    const int et = threadIdx.x - 64;   // 0..255 over the epilogue warps
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    if (MODE == 0 && zero_n4 > 0) zero_slice(et, kEpiThreads);
    // F8 GEMM 2: the per-pair scales staged below are the previous kernel's
    // output (the quantization of a), unlike the routing lists
    if (F8 && early) griddep_wait();
    static_assert(N <= kEpiThreads, "one staged column per epilogue thread");
    int i = 0;
    // The next tile's block entries -- its expert id and this thread's entry
    // of sorted_token_ids (column et) -- are loaded while this tile is
    // processed, so that staging a tile waits for one load (the weight or
    // scale behind the entry) instead of two in a row.
    int pf_e = 0, pf_p = -1;
    auto prefetch = [&](int j) {
      if (MODE == 2 || j >= n_work) return;
      const int bb = work(j).b;
      pf_e = expert_ids[bb];
      pf_p = et < N && et < B ? sorted_ids[(size_t)bb * B + et] : -1;
    };
    prefetch(0);
    for (int jw = 0; jw < n_work; ++jw) {
      const TileCoord tc = work(jw);
      const int b = tc.b, c = tc.c;
      // a K range short of the whole tile: partial sums (GEMM 1 through h_acc)
      const bool partial = tc.kb0 > 0 || tc.kb1 < nk;
      // a block whose expert id lies outside [0, E) is computed (on zero
      // weights) but writes nothing
      const int e_cur = MODE == 2 ? 0 : pf_e;
      const int p_cur = pf_p;
      prefetch(jw + 1);
      const bool e_ok = MODE == 2 || (static_cast<unsigned>(e_cur) < static_cast<unsigned>(E));
      const bool two = !Cfg::kWide && (MODE == 0 || c * 2 * kTileM + kTileM < a_rows);
      // F8: the scales of the weight rows this thread's TMEM lane holds (1 for
      // a row past the end), loaded together with the staging below
      float s_lo = 1.f, s_hi = 1.f;
      if (F8 && e_ok) {
        const float *rs = row_scale + (size_t)e_cur * a_rows;
        if (MODE == 0 && Cfg::kWide) {
          const int chn = c * Cfg::kRowsPerCTile + (q & 1) * 32 + lane;  // gate rows in quarters 0-1
          if (chn < R_out) s_lo = rs[q < 2 ? chn : R_out + chn];
        } else if (MODE == 0) {
          const int chn = c * kTileM + q * 32 + lane;
          if (chn < R_out) {
            s_lo = rs[chn];
            s_hi = rs[R_out + chn];
          }
        } else if (MODE == 1) {
          const int n = c * Cfg::kRowsPerCTile + q * 32 + lane;  // h = 0 and h = 1 (two tiles)
          if (n < H_out) s_lo = rs[n];
          if (two && n + kTileM < H_out) s_hi = rs[n + kTileM];
        }
      }
      const int acc = i % Cfg::kAccBufs;
      const uint32_t use = i / Cfg::kAccBufs;
      ++i;
      // the block's destinations (and router weights), staged while the MMAs run
      epilogue_bar_sync();  // the previous tile's readers are done
      for (int j = et; j < N; j += kEpiThreads) {
        int d = -1;
        float wgt = 0.f;
        if (MODE == 2) {
          if (b * N + j < src_rows) d = b * N + j;
        } else if (j < B && e_ok) {
          const int p = p_cur;  // (j == et)
          if (p >= 0 && p < P) {
            d = MODE == 0 ? p : p / top_k;
            if (MODE == 1) wgt = vec[p];
            // F8: the source row's scale (GEMM 1: the token's; GEMM 2: the
            // pair's, folded into the router weight)
            if (F8) wgt = MODE == 0 ? col_scale[p / top_k] : wgt * col_scale[p];
          }
        }
        dst_row[j] = d;
        dst_w[j] = wgt;
      }
      epilogue_bar_sync();
      const bool ok = wait_bounded(smem_u32(&acc_full[acc]), use & 1, abort, status);
      tc_fence_after();
      // stop together: every epilogue warp meets the same named barriers
      if (!ok || *abort) *epi_stop = 1;
      epilogue_bar_sync();
      if (*epi_stop) break;
      const uint32_t d0 = tmem + lane_base + acc * Cfg::kAccCols;
      if (MODE == 0 && Cfg::kWide) {
        // TMEM lanes 0-63 hold the gate sums of channels c*64 .. c*64+63,
        // lanes 64-127 the up sums of the same channels.  Warp pair (gate
        // quarter q, up quarter q + 2) of one column half: per 32 columns each
        // warp rounds its values to bf16, hands 16 columns to the other warp
        // through the pair's slot, and forms a for the other 16.
        const bool is_gate = q < 2;
        const int pair = (q & 1) + 2 * half;
        const int chn = c * Cfg::kRowsPerCTile + (q & 1) * 32 + lane;
        const bool valid = chn < R_out;
        // [pair][buffer][direction][column half][lane] of 16 bytes (8 bf16 columns)
        uint4 *slot = reinterpret_cast<uint4 *>(xchg) + pair * (2 * 2 * 32 * 2);
        const float srow = s_lo;
#pragma unroll 1
        for (int j0 = 32 * half, it = 0; j0 < N; j0 += 64, ++it) {
          uint32_t lo[16], hi[16];
          tmem_ld_32x32b_x16(d0 + j0, lo);
          tmem_ld_32x32b_x16(d0 + j0 + 16, hi);
          tmem_ld_wait();
          if constexpr (F8) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              lo[jj] = __float_as_uint(__uint_as_float(lo[jj]) * srow * dst_w[j0 + jj]);
              hi[jj] = __float_as_uint(__uint_as_float(hi[jj]) * srow * dst_w[j0 + 16 + jj]);
            }
          }
          uint4 *buf = slot + (it & 1) * (2 * 32 * 2);
          // the gate warp gives away columns 16..31, the up warp columns 0..15
          {
            const uint32_t *g = is_gate ? hi : lo;
            uint4 *dst = buf + (is_gate ? 0 : 64) + lane;
            dst[0] = make_uint4(pack_bf16x2(__uint_as_float(g[0]), __uint_as_float(g[1])),
                                pack_bf16x2(__uint_as_float(g[2]), __uint_as_float(g[3])),
                                pack_bf16x2(__uint_as_float(g[4]), __uint_as_float(g[5])),
                                pack_bf16x2(__uint_as_float(g[6]), __uint_as_float(g[7])));
            dst[32] = make_uint4(pack_bf16x2(__uint_as_float(g[8]), __uint_as_float(g[9])),
                                pack_bf16x2(__uint_as_float(g[10]), __uint_as_float(g[11])),
                                pack_bf16x2(__uint_as_float(g[12]), __uint_as_float(g[13])),
                                pack_bf16x2(__uint_as_float(g[14]), __uint_as_float(g[15])));
          }
          pair_bar_sync(pair);
          const uint4 *src2 = buf + (is_gate ? 64 : 0) + lane;
          const uint4 r0 = src2[0], r1 = src2[32];
          const uint32_t other[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
          const uint32_t *mine = is_gate ? lo : hi;
          const int cbase = j0 + (is_gate ? 0 : 16);
          if constexpr (F8) {
            // E4M3 operands halve the mainloop and leave the epilogue the
            // longer path: all 16 values first, then the stores -- sixteen
            // independent chains (exp, reciprocal) that the scheduler
            // interleaves, where a value computed under its store's
            // condition costs a full chain each (measured: 0.50 -> 0.37 ms
            // at the 16384-token prefill).  With bf16 operands the mainloop
            // is the longer path and this form measured 3 % slower there.
            uint16_t res[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const float o = __uint_as_float((jj & 1) ? (other[jj >> 1] & 0xFFFF0000u) : (other[jj >> 1] << 16));
              const float m = __uint_as_float(mine[jj]);
              res[jj] = silu_mul_bf16(is_gate ? m : o, is_gate ? o : m);
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int p = dst_row[cbase + jj];
              if (valid && p >= 0) out16[(size_t)p * R_out + chn] = res[jj];
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const float o = __uint_as_float((jj & 1) ? (other[jj >> 1] & 0xFFFF0000u) : (other[jj >> 1] << 16));
              const float m = __uint_as_float(mine[jj]);
              const int p = dst_row[cbase + jj];
              if (valid && p >= 0)
                out16[(size_t)p * R_out + chn] = silu_mul_bf16(is_gate ? m : o, is_gate ? o : m);
            }
          }
        }
      } else if (MODE == 0) {
        const int chn = c * kTileM + q * 32 + lane;
        const bool valid = chn < R_out;
        const float sg = s_lo, su = s_hi;
#pragma unroll 1
        for (int j0 = 16 * half; j0 < N; j0 += 32) {
          uint32_t gt[16], up[16];
          tmem_ld_32x32b_x16(d0 + j0, gt);
          tmem_ld_32x32b_x16(d0 + N + j0, up);
          tmem_ld_wait();
          if constexpr (F8) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              gt[jj] = __float_as_uint(__uint_as_float(gt[jj]) * sg * dst_w[j0 + jj]);
              up[jj] = __float_as_uint(__uint_as_float(up[jj]) * su * dst_w[j0 + jj]);
            }
          }
          if (partial) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int p = dst_row[j0 + jj];
              if (valid && p >= 0) {
                // a partial sum over this split's K range: add it up in fp32
                atomicAdd(h_acc + (size_t)p * 2 * R_out + chn, __uint_as_float(gt[jj]));
                atomicAdd(h_acc + (size_t)p * 2 * R_out + R_out + chn, __uint_as_float(up[jj]));
              }
            }
          } else if constexpr (F8) {
            uint16_t res[16];  // the values first, then the stores (as above)
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              res[jj] = silu_mul_bf16(__uint_as_float(gt[jj]), __uint_as_float(up[jj]));
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int p = dst_row[j0 + jj];
              if (valid && p >= 0) out16[(size_t)p * R_out + chn] = res[jj];
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int p = dst_row[j0 + jj];
              if (valid && p >= 0)
                out16[(size_t)p * R_out + chn] =
                    silu_mul_bf16(__uint_as_float(gt[jj]), __uint_as_float(up[jj]));
            }
          }
        }
      } else {
        // work items (h, chunk of 16 columns), alternating between the two warps of a quarter
        const int n_chunks = N / 16;
        // Wide GEMM 2: the warp's 32 channels x 16 tokens pass through shared
        // memory so that each thread adds 4 consecutive channels of one token
        // with one 16-byte reduction (a quarter of the requests of per-channel
        // adds; measured faster for 256-token tiles, slower for narrower ones)
        float *scr = reinterpret_cast<float *>(xchg) + (warp - 2) * (16 * 32);  // [16 tokens][32 ch]
        const int q4 = lane & 7, cg = lane >> 3;
        // one item: 16 columns of one 128-row half; a warp takes every second
        // item and loads two before it waits, so one TMEM round trip serves two
        auto process = [&](int item, const uint32_t (&o)[16]) {
          const int h = item / n_chunks, j0 = (item - h * n_chunks) * 16;
          const int n = c * Cfg::kRowsPerCTile + h * kTileM + q * 32 + lane;
          const float srow = h == 0 ? s_lo : s_hi;
          if (MODE == 1 && Cfg::kWide) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) scr[jj * 32 + lane] = __uint_as_float(o[jj]) * srow;
            __syncwarp();
            const int n4 = n - lane + 4 * q4;  // first of this thread's 4 channels
            if (n4 < H_out) {                  // H_out is a multiple of 16: all 4 or none
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int col = cg * 4 + jj;
                const int d = dst_row[j0 + col];
                if (d >= 0) {
                  const float wgt = dst_w[j0 + col];
                  const float4 v = *reinterpret_cast<const float4 *>(scr + col * 32 + 4 * q4);
                  atomicAdd(reinterpret_cast<float4 *>(y_acc + (size_t)d * H_out + n4),
                            make_float4(wgt * v.x, wgt * v.y, wgt * v.z, wgt * v.w));
                }
              }
            }
            __syncwarp();  // the next item overwrites the staging rows
          } else {
            if constexpr (MODE == 2) {
              if (partial) {
                // a K range of the router's tile: its fp32 sums go to this split's
                // slice [Mt][a_rows] of h_acc, laid out like the logits (a warp's
                // lanes are consecutive experts: each store one 128-byte line);
                // the last split of the tile adds the slices in split order
                if (n < a_rows) {
                  const int sp = (tc.kb0 * kspl + nk - 1) / nk;  // this range's split (balanced ranges)
                  float *dst = h_acc + ((size_t)sp * Mt + (size_t)b * N + j0) * a_rows + n;
#pragma unroll
                  for (int jj = 0; jj < 16; ++jj) dst[(size_t)jj * a_rows] = __uint_as_float(o[jj]);
                }
                return;
              }
            }
            const bool valid = n < (MODE == 1 ? H_out : a_rows);
            const float bias = (MODE == 2 && valid && vec != nullptr) ? vec[n] : 0.f;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int d = dst_row[j0 + jj];
              if (valid && d >= 0) {
                if (MODE == 1)
                  atomicAdd(y_acc + (size_t)d * H_out + n, dst_w[j0 + jj] * (__uint_as_float(o[jj]) * srow));
                else
                  out16[(size_t)d * a_rows + n] = float_to_bf16_bits(__uint_as_float(o[jj]) + bias);
              }
            }
          }
        };
        const int n_items = (two ? 2 : 1) * n_chunks;
#pragma unroll 1
        for (int item = half; item < n_items; item += 4) {
          const int item2 = item + 2;
          uint32_t o[16], o2[16];
          {
            const int h = item / n_chunks, j0 = (item - h * n_chunks) * 16;
            tmem_ld_32x32b_x16(d0 + h * N + j0, o);
          }
          if (item2 < n_items) {
            const int h = item2 / n_chunks, j0 = (item2 - h * n_chunks) * 16;
            tmem_ld_32x32b_x16(d0 + h * N + j0, o2);
          }
          tmem_ld_wait();
          process(item, o);
          if (item2 < n_items) process(item2, o2);
        }
      }
      // this accumulator buffer may be overwritten once all epilogue warps are done with it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // (2-SM tiles: the MMAs are the even CTA's, so is the barrier)
        if (P2 && rank == 1) mbar_arrive_cluster(map_to_cta(smem_u32(&acc_empty[acc]), 0));
        else mbar_arrive(smem_u32(&acc_empty[acc]));
      }
      if (MODE == 0 && partial) {
        // The last part of this tile to finish (an atomic count of K stages
        // after a fence; nobody waits) reads the summed h back and writes a.
        __threadfence();
        epilogue_bar_sync();
        if (et == 0) {
          const int mine = tc.kb1 - tc.kb0;
          *split_last = atomicAdd(&tile_cnt[b * n_ctiles + c], mine) + mine == nk;
        }
        epilogue_bar_sync();
        if (*split_last) {
          __threadfence();
          const int chn = c * kTileM + q * 32 + lane;
          if (chn < R_out) {
            for (int j = half; j < N; j += 2) {
              const int p = dst_row[j];
              if (p < 0) continue;
              const float gs = __ldcg(h_acc + (size_t)p * 2 * R_out + chn);
              const float us = __ldcg(h_acc + (size_t)p * 2 * R_out + R_out + chn);
              out16[(size_t)p * R_out + chn] = silu_mul_bf16(gs, us);
            }
          }
          if (et == 0) tile_cnt[b * n_ctiles + c] = 0;
        }
      }
      if constexpr (MODE == 2) {
        if (partial) {
          // The router's tile cut along K: the last part to finish (counted in K
          // stages, as above) adds the splits' slices in split order -- the
          // same sum whichever part comes last -- and writes the logits.
          __threadfence();
          epilogue_bar_sync();
          if (et == 0) {
            const int mine = tc.kb1 - tc.kb0;
            *split_last = atomicAdd(&tile_cnt[b * n_ctiles + c], mine) + mine == nk;
          }
          epilogue_bar_sync();
          if (*split_last) {
            __threadfence();
            const int n_h = c * 2 * kTileM + kTileM < a_rows ? 2 : 1;
            for (int h = 0; h < n_h; ++h) {
              const int n = c * 2 * kTileM + h * kTileM + q * 32 + lane;
              if (n >= a_rows) continue;
              const float bias = vec != nullptr ? vec[n] : 0.f;
              for (int j0 = 16 * half; j0 < N; j0 += 32) {
                // every slice's 16 values loaded before any is added (one L2
                // round trip per chunk; the scratch holds kRouterMaxSplits
                // slices, those past kspl are not added), then added in split
                // order
                float v[kRouterMaxSplits][16];
#pragma unroll
                for (int sp = 0; sp < kRouterMaxSplits; ++sp) {
                  const float *src = h_acc + ((size_t)sp * Mt + (size_t)b * N + j0) * a_rows + n;
#pragma unroll
                  for (int jj = 0; jj < 16; ++jj) v[sp][jj] = __ldcg(src + (size_t)jj * a_rows);
                }
                float sum[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                  sum[jj] = 0.f;
#pragma unroll
                  for (int sp = 0; sp < kRouterMaxSplits; ++sp)
                    if (sp < kspl) sum[jj] += v[sp][jj];
                }
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                  const int d = dst_row[j0 + jj];
                  if (d >= 0) out16[(size_t)d * a_rows + n] = float_to_bf16_bits(sum[jj] + bias);
                }
              }
            }
            if (et == 0) tile_cnt[b * n_ctiles + c] = 0;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (P2) {
    cluster_sync();  // neither CTA leaves while the other may still signal it
    if (warp == 1) tmem_dealloc_pair(tmem, Cfg::kTmemCols);
  } else {
    if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over weights [E][rows][K] (bf16, or E4M3 codes with elt_bytes = 1;
// K contiguous), box of 128 bytes of K x box_rows x 1, 128-byte swizzle;
// out-of-range rows and columns read as zero.
cudaError_t encode_weight_map(CUtensorMap *map, const void *w, int K, int rows, int E,
                              int box_rows, int elt_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(E)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * elt_bytes,
                                 static_cast<cuuint64_t>(K) * elt_bytes * rows};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK * 2 / elt_bytes),
                             static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, elt_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                            3, const_cast<void *>(w),
                            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Encoded maps, keyed by (device, address, shape): a layer's weights keep
// their map from call to call, so the host encodes each one once.
struct MapEntry {
  int dev;
  const void *ptr;
  int K, rows, E, box_rows, elt;
  CUtensorMap map;
};
std::mutex g_map_mutex;
MapEntry g_maps[128];
int g_map_next = 0, g_map_count = 0;

cudaError_t make_weight_map(CUtensorMap *map, const void *w, int K, int rows, int E,
                            int box_rows = kTileM, int elt_bytes = 2) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  for (int i = 0; i < g_map_count; ++i) {
    const MapEntry &m = g_maps[i];
    if (m.dev == dev && m.ptr == w && m.K == K && m.rows == rows && m.E == E &&
        m.box_rows == box_rows && m.elt == elt_bytes) {
      *map = m.map;
      return cudaSuccess;
    }
  }
  err = encode_weight_map(map, w, K, rows, E, box_rows, elt_bytes);
  if (err != cudaSuccess) return err;
  MapEntry &m = g_maps[g_map_next];
  m = MapEntry{dev, w, K, rows, E, box_rows, elt_bytes, *map};
  g_map_next = (g_map_next + 1) % 128;
  if (g_map_count < 128) ++g_map_count;
  return cudaSuccess;
}

// Everything a launch of k_gemm_tc needs besides the weight map.
struct TcArgs {
  const uint16_t *src;
  int src_rows;
  const int32_t *sorted_ids, *expert_ids, *n_post;
  const float *vec;
  int P, top_k, E, K, R_out, a_rows, B, cap, n_ctiles, ksplit;
  float *h_acc;
  int *tile_cnt;
  uint16_t *out16;
  float *y_acc;
  int H_out;
  int *status;
  long max_blocks;  // host-side bound on the blocks (tiles = blocks * n_ctiles * ksplit)
  int early_weights;
  int n_pass;  // GEMM 2: ranges of weight tiles run one after the other (1: none)
  const uint8_t *w_pf = nullptr;  // GEMM 1: weights to bring into L2 before the dependency wait
  long pf_bytes = 0;
  float *zero_dst = nullptr;  // GEMM 1: fp32 buffer to clear (zero_n floats, a multiple of 4)
  long zero_n = 0;
  const float *row_scale = nullptr;  // E4M3 weights: per weight row
  const float *col_scale = nullptr;  // E4M3 rows: per token (GEMM 1) or pair (GEMM 2)
};

// Clusters of two CTAs of the 2-SM kernel that can be resident at once (0: none).
template <int N, int MODE, bool F8>
int max_pair_clusters() {
  static int cached[64];
  static bool known[64];
  static std::mutex m;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(m);
  if (!known[dev]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms() / 2 * 2);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = TcConfig<N, MODE, true>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_gemm_tc<N, MODE, true, F8>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    cached[dev] = n;
    known[dev] = true;
  }
  return cached[dev];
}

template <int N, int MODE, bool F8>
cudaError_t launch_tc_n(const CUtensorMap &map_w, const TcArgs &a, cudaStream_t s) {
  using Cfg = TcConfig<N, MODE>;
  cudaError_t err;
  if constexpr (Cfg::kWide) {
    // 256-token tiles with an even number of weight tiles: 2-SM tiles, as many
    // pairs of CTAs as can be resident at once
    // (MOE_FORCE_PATH=tc1 keeps one CTA per tile, for comparisons)
    const char *force = std::getenv("MOE_FORCE_PATH");
    const bool no_pairs = force != nullptr && std::strcmp(force, "tc1") == 0;
    if (kPairTiles && !no_pairs && a.ksplit == 1 && a.n_ctiles % 2 == 0) {
      auto kern2 = k_gemm_tc<N, MODE, true, F8>;
      err = ensure_smem_limit(reinterpret_cast<const void *>(kern2), TcConfig<N, MODE, true>::kSmemBytes);
      if (err != cudaSuccess) return err;
      const int units_max = max_pair_clusters<N, MODE, F8>();
      if (units_max > 0) {
        const int units =
            static_cast<int>(std::min<long>(a.max_blocks * (a.n_ctiles / 2), units_max));
        if (units <= 0) return cudaSuccess;
        return launch_pdl_cluster(kern2, dim3(2 * units), dim3(kTcThreads),
                                  TcConfig<N, MODE, true>::kSmemBytes, s, 2, map_w, a.src,
                                  a.src_rows, a.sorted_ids, a.expert_ids, a.n_post, a.vec, a.P,
                                  a.top_k, a.E, a.K, a.R_out, a.a_rows, a.B, a.cap, a.n_ctiles,
                                  a.ksplit, a.h_acc, a.tile_cnt, a.out16, a.y_acc, a.H_out,
                                  a.status, a.early_weights, a.n_pass, a.w_pf, a.pf_bytes,
                                  reinterpret_cast<float4 *>(a.zero_dst), a.zero_n / 4,
                                  a.row_scale, a.col_scale);
      }
    }
  }
  auto kern = k_gemm_tc<N, MODE, false, F8>;
  err = ensure_smem_limit(reinterpret_cast<const void *>(kern), Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  // persistent: one CTA per SM at most, each walking the tile list with stride gridDim.x
  const long units = a.max_blocks * a.n_ctiles * a.ksplit;
  const int grid = static_cast<int>(std::min<long>(units, num_sms()));
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(kern, dim3(grid), dim3(kTcThreads), Cfg::kSmemBytes, s, map_w, a.src,
                    a.src_rows, a.sorted_ids, a.expert_ids, a.n_post, a.vec, a.P, a.top_k, a.E,
                    a.K, a.R_out, a.a_rows, a.B, a.cap, a.n_ctiles, a.ksplit, a.h_acc, a.tile_cnt,
                    a.out16, a.y_acc, a.H_out, a.status, a.early_weights, a.n_pass, a.w_pf,
                    a.pf_bytes, reinterpret_cast<float4 *>(a.zero_dst), a.zero_n / 4, a.row_scale,
                    a.col_scale);
}

template <int MODE, bool F8 = false>
cudaError_t launch_tc(int N, const CUtensorMap &map_w, const TcArgs &a, cudaStream_t s) {
  switch (N) {
    case 16: return launch_tc_n<16, MODE, F8>(map_w, a, s);
    case 32: return launch_tc_n<32, MODE, F8>(map_w, a, s);
    case 64: return launch_tc_n<64, MODE, F8>(map_w, a, s);
    case 128: return launch_tc_n<128, MODE, F8>(map_w, a, s);
    case 256: return launch_tc_n<256, MODE, F8>(map_w, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool tc_supports_block(int B) { return B == 16 || B == 32 || B == 64 || B == 128 || B == 256; }

namespace {

// GEMM 1 on bf16 operands, or (F8) on E4M3 codes with per-row scales.
template <bool F8>
cudaError_t tc_w13_impl(const void *x, const void *w13, const float *w13_scale,
                        const float *x_scale, const int32_t *sorted_ids, const int32_t *expert_ids,
                        const int32_t *n_post, int P, int top_k, int E, int H, int I, int B,
                        int cap, uint16_t *a, int ksplit, float *h_acc, int *tile_cnt,
                        int *status, int pf_experts, float *zero_dst, long zero_n,
                        cudaStream_t s) {
  constexpr int elt = F8 ? 1 : 2;
  constexpr int bke = kBK * 2 / elt;  // K elements per stage
  // wide tiles (B = 256): 64 gate rows over 64 up rows per weight tile, no K split
  const bool wide = B == 256;
  CUtensorMap map_w;
  cudaError_t err = make_weight_map(&map_w, w13, H, 2 * I, E, wide ? kTileM / 2 : kTileM, elt);
  if (err != cudaSuccess) return err;
  const int nk = (H + bke - 1) / bke;
  // splits need the split-K scratch; 256-token tiles are not split
  if (wide || ksplit < 1 || ksplit > nk || h_acc == nullptr || tile_cnt == nullptr) ksplit = 1;
  TcArgs args{};
  args.src = static_cast<const uint16_t *>(x);
  args.src_rows = (P + top_k - 1) / top_k;
  args.sorted_ids = sorted_ids;
  args.expert_ids = expert_ids;
  args.n_post = n_post;
  args.P = P;
  args.top_k = top_k;
  args.E = E;
  args.K = H;
  args.R_out = I;
  args.a_rows = 2 * I;
  args.B = B;
  args.cap = cap;
  const int ct_rows = wide ? kTileM / 2 : kTileM;
  args.n_ctiles = (I + ct_rows - 1) / ct_rows;
  args.ksplit = ksplit;
  args.h_acc = h_acc;
  args.tile_cnt = tile_cnt;
  args.out16 = a;
  args.status = status;
  args.max_blocks = cap / B;
  args.zero_dst = zero_dst;
  args.zero_n = zero_dst != nullptr ? zero_n : 0;
  args.row_scale = w13_scale;
  args.col_scale = x_scale;
  if (pf_experts > 0) {
    // the first wave's experts: ceil(SMs / tiles per block) blocks, one expert
    // each at decode sizes, plus one for an expert without pairs among them
    const long per_e = 2l * I * H * elt;
    const int per_block = args.n_ctiles * std::max(ksplit, 1);
    const int wave = (num_sms() + per_block - 1) / per_block + 1;
    const int n_e = std::min(std::min(pf_experts, wave), E);
    args.w_pf = static_cast<const uint8_t *>(w13);
    args.pf_bytes = std::min<long>(n_e * per_e, 96l << 20);
  }
  return launch_tc<0, F8>(B, map_w, args, s);
}

}  // namespace

cudaError_t launch_tc_w13_act(const uint16_t *x, const uint16_t *w13, const int32_t *sorted_ids,
                              const int32_t *expert_ids, const int32_t *n_post, int P, int top_k,
                              int E, int H, int I, int B, int cap, uint16_t *a, int ksplit,
                              float *h_acc, int *tile_cnt, int *status, int pf_experts,
                              float *zero_dst, long zero_n, cudaStream_t s) {
  return tc_w13_impl<false>(x, w13, nullptr, nullptr, sorted_ids, expert_ids, n_post, P, top_k, E,
                            H, I, B, cap, a, ksplit, h_acc, tile_cnt, status, pf_experts, zero_dst,
                            zero_n, s);
}

cudaError_t launch_tc_w13_act_f8(const uint8_t *qx, const float *sx, const uint8_t *w13q,
                                 const float *w13s, const int32_t *sorted_ids,
                                 const int32_t *expert_ids, const int32_t *n_post, int P, int top_k,
                                 int E, int H, int I, int B, int cap, uint16_t *a, int ksplit,
                                 float *h_acc, int *tile_cnt, int *status, int pf_experts,
                                 float *zero_dst, long zero_n, cudaStream_t s) {
  return tc_w13_impl<true>(qx, w13q, w13s, sx, sorted_ids, expert_ids, n_post, P, top_k, E, H, I,
                           B, cap, a, ksplit, h_acc, tile_cnt, status, pf_experts, zero_dst,
                           zero_n, s);
}

// Ranges of GEMM 2's weight tiles run one after the other so that the live
// part of the fp32 combine accumulator (y_bytes in all) fits L2 beside the
// weight and activation streams; each extra range reads the activation again.
static int gemm2_passes(long y_bytes, int n_ctiles) {
  constexpr long kLiveBytes = 48l << 20;
  int n = static_cast<int>(std::min<long>((y_bytes + kLiveBytes - 1) / kLiveBytes, n_ctiles));
  n = std::max(n, 1);
  const int ctp = (n_ctiles + n - 1) / n;  // ranges actually needed with ctp tiles each
  return (n_ctiles + ctp - 1) / ctp;
}

namespace {

template <bool F8>
cudaError_t tc_w2_impl(const void *a, const void *w2, const float *w2_scale, const float *a_scale,
                       const int32_t *sorted_ids, const int32_t *expert_ids, const int32_t *n_post,
                       const float *topk_weights, int P, int top_k, int E, int H, int I, int B,
                       int cap, float *y_acc, int ksplit, int *status, bool early_weights,
                       cudaStream_t s) {
  constexpr int elt = F8 ? 1 : 2;
  constexpr int bke = kBK * 2 / elt;
  CUtensorMap map_w;
  cudaError_t err = make_weight_map(&map_w, w2, I, H, E, kTileM, elt);
  if (err != cudaSuccess) return err;
  const int nk = (I + bke - 1) / bke;
  TcArgs args{};
  args.src = static_cast<const uint16_t *>(a);
  args.src_rows = P;
  args.sorted_ids = sorted_ids;
  args.expert_ids = expert_ids;
  args.n_post = n_post;
  args.vec = topk_weights;
  args.P = P;
  args.top_k = top_k;
  args.E = E;
  args.K = I;
  args.R_out = H;
  args.a_rows = H;
  args.B = B;
  args.cap = cap;
  const int ct_rows = B == 256 ? kTileM : 2 * kTileM;  // wide tiles: one 128-row weight tile
  args.n_ctiles = (H + ct_rows - 1) / ct_rows;
  args.ksplit = std::max(1, std::min(ksplit, nk));  // the combine adds partial sums anyway
  args.y_acc = y_acc;
  args.H_out = H;
  args.status = status;
  args.max_blocks = cap / B;
  args.early_weights = early_weights ? 1 : 0;
  args.n_pass = gemm2_passes(static_cast<long>(P / top_k) * H * 4, args.n_ctiles);
  args.row_scale = w2_scale;
  args.col_scale = a_scale;
  return launch_tc<1, F8>(B, map_w, args, s);
}

}  // namespace

cudaError_t launch_tc_w2_combine(const uint16_t *a, const uint16_t *w2, const int32_t *sorted_ids,
                                 const int32_t *expert_ids, const int32_t *n_post,
                                 const float *topk_weights, int P, int top_k, int E, int H, int I,
                                 int B, int cap, float *y_acc, int ksplit, int *status,
                                 bool early_weights, cudaStream_t s) {
  return tc_w2_impl<false>(a, w2, nullptr, nullptr, sorted_ids, expert_ids, n_post, topk_weights,
                           P, top_k, E, H, I, B, cap, y_acc, ksplit, status, early_weights, s);
}

cudaError_t launch_tc_w2_combine_f8(const uint8_t *qa, const float *sa, const uint8_t *w2q,
                                    const float *w2s, const int32_t *sorted_ids,
                                    const int32_t *expert_ids, const int32_t *n_post,
                                    const float *topk_weights, int P, int top_k, int E, int H,
                                    int I, int B, int cap, float *y_acc, int ksplit, int *status,
                                    bool early_weights, cudaStream_t s) {
  return tc_w2_impl<true>(qa, w2q, w2s, sa, sorted_ids, expert_ids, n_post, topk_weights, P, top_k,
                          E, H, I, B, cap, y_acc, ksplit, status, early_weights, s);
}

cudaError_t launch_selftest_timeout(int *status, int limit_ms, cudaStream_t s) {
  int dev = 0, khz = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
  if (err != cudaSuccess) return err;
  const long long cycles = static_cast<long long>(std::max(1, std::min(limit_ms, 2000))) * khz;
  k_selftest_timeout<<<1, 32, 0, s>>>(status, cycles);
  return cudaGetLastError();
}

cudaError_t launch_tc_router(const uint16_t *x, const uint16_t *w_router, const float *bias, int M,
                             int E, int H, uint16_t *logits, int *status, float *split_scratch,
                             int *tile_cnt, cudaStream_t s) {
  CUtensorMap map_w;
  cudaError_t err = make_weight_map(&map_w, w_router, H, E, 1);
  if (err != cudaSuccess) return err;
  const int N = 128;
  TcArgs args{};
  args.src = x;
  args.src_rows = M;
  args.vec = bias;
  args.P = M;
  args.top_k = 1;
  args.E = 1;
  args.K = H;
  args.R_out = E;
  args.a_rows = E;
  args.B = N;
  args.n_ctiles = (E + 2 * kTileM - 1) / (2 * kTileM);
  // Each CTA streams the whole of W_r through its TMA unit (32 stages at
  // H = 2048): with fewer tiles than SMs, the tile's K range is split over
  // up to kRouterMaxSplits CTAs whose fp32 partial sums meet in split_scratch
  // (Zipf prefill, routing 512 tokens 34.4 -> 29.4 us, 4096 tokens 36.0 ->
  // 34.3; more than kRouterCtlCount tiles keep one CTA per tile).
  int ks = 1;
  const int units = ((M + N - 1) / N) * args.n_ctiles;
  const int nk = (H + kBK - 1) / kBK;
  if (split_scratch != nullptr && tile_cnt != nullptr && units <= kRouterCtlCount)
    ks = std::max(1, std::min({kRouterMaxSplits, num_sms() / units, nk}));
  args.ksplit = ks;
  args.h_acc = split_scratch;
  args.tile_cnt = tile_cnt;
  args.out16 = logits;
  args.status = status;
  args.max_blocks = (M + N - 1) / N;
  return launch_tc<2>(N, map_w, args, s);
}

}  // namespace moe
