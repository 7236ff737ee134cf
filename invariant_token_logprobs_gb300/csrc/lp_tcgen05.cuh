// lp_tcgen05.cuh: the sm_103a tensor-core pipeline shared by the fused kernels.
//
// A persistent grid of CTA pairs (thread-block clusters of 2, one CTA per SM)
// computes 256 x 256 fp32 tiles D = A B^T of two bf16 operands (K-major, or
// M/N-major for the backward's products) with
// tcgen05.mma.cta_group::2 (M=256, N=256, K=16, kind::f16) into tensor memory,
// and hands every finished tile to an epilogue.  CTA r of a pair holds rows
// 128r..128r+127 of the A box and rows 128r..128r+127 of the B box in its own
// shared memory and receives rows 128r.. of D in its own tensor memory, so an
// SM stages 32 KB per 64 of K (a single-CTA 128 x 256 tile needs 48 KB, and
// with the tensor core reading what TMA writes, shared-memory bandwidth is
// what bounds it).
//
// Roles (6 warps per CTA):
//   warp 0     TMA loader (both CTAs): this CTA's halves of the A and B blocks
//              into the operand ring, whose geometry is a template parameter
//              (Ring: 3 stages of 128 of K, each operand as two 64-wide boxes
//              with 128-byte swizzle, or 6 stages of 64); the bytes of both
//              CTAs complete one barrier in the leader CTA;
//   warp 1     tensor memory: 512 columns (two 128 x 256 fp32 accumulators)
//              allocated by both CTAs; one lane of the leader issues the MMAs
//              and commits them to barriers in both CTAs (multicast);
//   warps 2-5  epilogue (both CTAs): wait for a finished accumulator, run the
//              caller's epilogue on it (one row per thread), then arrive on the
//              leader's accumulator-empty barrier;
//   warp 6     (optional) a side job of the caller's, alongside the pipeline.
// While the epilogues drain one accumulator the MMAs fill the other.
//
// Every mbarrier wait is bounded by %globaltimer: a wait that gives up sets
// the call's error word and an abort flag in shared memory, the other roles of
// that CTA stop at their next wait (the roles of the other CTA give up on their
// own bounded waits), in-flight copies and MMAs are drained with bounded waits,
// tensor memory is freed and the CTAs return.
//
// The PTX below follows the public PTX ISA: tcgen05 (alloc, mma, commit, ld,
// fences), cp.async.bulk.tensor with .cta_group::2, mbarrier, mapa and
// barrier.cluster.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "lp_check.cuh"
#include "lp_internal.h"

namespace lp {
namespace tc {

constexpr int kBM = 128;       // rows of A per CTA (tensor-memory lanes); 256 per pair
constexpr int kBN = 256;       // columns of D per tile; 128 rows of B per CTA
constexpr int kBNHalf = kBN / 2;
constexpr int kAtomK = 64;     // bf16 per 128-byte swizzle row
constexpr int kUmmaK = 16;
constexpr int kThreads = 192;
constexpr int kEpilogueThreads = 128;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

static_assert(kBN == kTileN, "the vocabulary tile of the fused path is one MMA tile");

// Geometry of the operand ring: BK of K per stage (BK / 64 boxes of 128-byte
// swizzle rows side by side for a K-major operand), Stages stages.  Pair: the
// CTA is one of a 2-SM pair (cta_group::2, M = 256, this CTA's 128 rows of the
// tile's B); otherwise it works alone (cta_group::1, M = 128, all 256 rows of
// B, K-major operands only).
template <int BK, int Stages, bool Pair = true>
struct Ring {
  static constexpr bool kPair = Pair;
  static constexpr int kBK = BK;
  static constexpr int kAtoms = BK / kAtomK;
  static constexpr int kStages = Stages;
  static constexpr int kABytes = kBM * BK * 2;
  static constexpr int kBBytes = (Pair ? kBNHalf : kBN) * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kNumBars = 2 * Stages + 2 + 2 + 1;
  // bytes past the 1024-aligned dynamic shared-memory base the pipeline uses
  // (ring, barriers, tensor-memory slot); an epilogue may use what follows
  static constexpr int kSmemEnd = Stages * kStageBytes + 1024;
  // dynamic shared memory of a kernel whose epilogue uses none
  static constexpr int kSmemBytes = 1024 + Stages * kStageBytes + kNumBars * 8 + 16;
  // distance between the two 64-row boxes of an M- or N-major operand
  static constexpr uint32_t kMnBoxBytes = BK * 128;
  static_assert(BK % kAtomK == 0, "whole swizzle rows per stage");
  static_assert(kNumBars * 8 + 16 <= 1024, "barriers fit below kSmemEnd");
};

// 128 of K per stage, 3 stages: the fused forward and gradient kernels (both
// operands K-major).  With 64 and a 6-deep ring the fused kernel ran 4-5%
// slower: each W row was fetched 128 bytes at a time, while two adjacent
// 128-byte pieces requested together read HBM better (ring depth alone, 5 to
// 7 stages, changed nothing).
using WideRing = Ring<128, 3>;
// 64 of K per stage, 6 stages: the backward's products (M/N-major operands,
// 8 K blocks per grad_W unit), which ran ~1% faster this way.
using NarrowRing = Ring<64, 6>;
// One CTA per tile, 4 stages of 64 of K (16 KB of A, 32 KB of B each): the
// fused forward for batches of at most 128 rows, where the pair's second
// 128-row half would multiply only zero rows.
using SingleRing = Ring<64, 4, false>;

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, bits 10-12 = 1), A / B major-ness in bits 15 / 16 (0: K-major,
// 1: M- or N-major), N >> 3 in bits 17-22, M >> 4 in bits 24-28; M = 256 for
// the CTA pair.
__host__ __device__ constexpr uint32_t idesc(bool a_mn, bool b_mn, int m = 2 * kBM) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(kBN >> 3) << 17) | (uint32_t(m >> 4) << 24);
}
constexpr uint32_t kIdesc = idesc(false, false);

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
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

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// The part of wait_bar after a first try found the phase incomplete.
static __device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, uint32_t* err,
                                                  uint32_t role_bit) {
  const uint64_t t0 = global_timer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(err, role_bit);
      return false;
    }
  }
}

// Bounded wait for the phase of `bar` with parity `parity`.  Returns false when
// the CTA is aborting or this wait gave up (then it raises the abort).  The
// first try is inline: a phase that is already complete costs no call (the
// MMA issuer's wait per K block is on the products' critical path).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t* err, uint32_t role_bit) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, abort_flag, err, role_bit);
}

// Bounded wait used while draining after an abort; never raises anything.
static __device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer() - t0 > kWaitLimitNs) return;
  }
}

// TMA load of a box into this CTA's shared memory; the transferred bytes are
// counted on `bar`, a shared::cluster address that may lie in the peer CTA.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// The same into a CTA that works alone, counted on its own barrier.
__device__ __forceinline__ void tma_load_2d_local(uint32_t dst, const CUtensorMap* map, int c0,
                                                  int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` (same offset) in both CTAs of the pair once every MMA issued
// so far by this thread has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  const uint16_t both = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(bar),
      "h"(both)
      : "memory");
}

// The same for a CTA that works alone.
__device__ __forceinline__ void tc_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tc_mma_single(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t accumulate, uint32_t instr) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(instr), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t accumulate, uint32_t instr = kIdesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(instr), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 128 bytes (64 K elements), 8-row groups 1024 bytes
// apart; a stage holds kAtoms such boxes along K, each (rows x 128 bytes)
// after the previous.  Start address >> 4 in bits 0-13, leading-dimension
// offset (unused for this layout, set to 16 bytes) in bits 16-29, stride
// offset 1024 >> 4 in bits 32-45, descriptor version 1 in bits 46-47, swizzle
// mode 2 (128-byte) in bits 61-63.  The box base is 1024-byte aligned, so the
// K offset of each 16-element MMA step within a box is added to the start
// address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16 >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Shared-memory matrix descriptor of an M- or N-major bf16 tile of 128 (MN) x
// BK (K) written by TMA with 128-byte swizzle as two boxes of 64 (MN) x BK
// (K): in each box, K row r sits at r * 128 bytes (64 contiguous MN
// elements), so a swizzle atom is 64 MN elements x 8 K rows (1024 bytes).  The
// leading-dimension offset (bits 16-29) is the distance between atoms along
// MN (the second box, box_bytes = BK * 128); the stride offset (bits 32-45)
// the distance between 8-row groups along K (1024 bytes).  Each 16-element MMA
// step along K adds 2048 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t box_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(box_bytes >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// 64 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_load64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, "
      "%45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, "
      "%62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 1024-aligned base of the dynamic shared memory (the pipeline's ring).
__device__ __forceinline__ uint8_t* pipeline_smem_base() {
  extern __shared__ uint8_t smem_raw[];
  return reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

// ------------------------------------------------------------------ pipeline
//
// Sched (work list, the same on every CTA):
//   int units() const;
//   void coords(int u, uint32_t rank, int& a_row, int& b_row, int& kb0, int& kb1) const;
//     rows of this CTA's A and B boxes and the K blocks [kb0, kb1) of unit u
//     (kb1 > kb0 always).
//   Optional, for K split into segments that do not start on a K block:
//   int k_offset(int u) const;
//     first K element of the unit's segment (a multiple of 16): K block kb
//     covers K elements k_offset + kb * BK ..;
//   int k_steps_last(int u) const;
//     MMA steps (16 K each, 1 .. BK / 16) of the unit's last K block: the
//     steps past the segment's end are not issued, so the elements loaded
//     there (the next segment's) add nothing.
// Epi (one per epilogue thread):
//   void consume(int u, uint32_t taddr, uint32_t rank, int lane_grp, int lane);
//     read the finished 128 x 256 accumulator (this thread's lane at taddr,
//     columns taddr + 0..255, with tmem_load64; warp-collective) and use it;
//   void after_release(int u, uint32_t rank, int lane_grp, int lane);
//     work that no longer needs tensor memory (after the accumulator is freed);
//   void finish(int lane_grp, int lane);
//     once after the last unit (e.g. wait for asynchronous stores).
// Side (optional): a kernel launched with more than kThreads threads gives
//   each warp past the epilogue warps side(lane) to run once, alongside the
//   pipeline (work that needs neither shared nor tensor memory).
//
// Called by every thread of a CTA of a 2-CTA cluster launched with kThreads
// threads (or more, for a Side) and at least R::kSmemBytes of dynamic shared
// memory; R is the ring geometry (WideRing or NarrowRing).  `withhold_first_load`
// (tests of the bounded waits only): the leader CTA of pair 0 announces but
// never issues its first TMA load, so that stage never fills and the waits
// on it give up after their time bound.
//
// Operand layouts: K-major (kAMn / kBMn false) operands are [rows, K] with K
// contiguous and their tensor maps have boxes of 64 K x 128 rows
// (encode_bf16_2d with box_rows 128), kAtoms per stage along K; M- or N-major
// operands (true) are [K, rows] with the rows contiguous and their tensor maps
// have boxes of 64 rows x R::kBK K (box_rows R::kBK), two per stage along the
// rows.
struct NoSide {
  __device__ __forceinline__ void operator()(int) const {}
};

// Whether a Sched has the optional segment members (k_offset, k_steps_last).
template <class S, class = void>
struct HasKSegments : std::false_type {};
template <class S>
struct HasKSegments<S, std::void_t<decltype(std::declval<const S&>().k_offset(0)),
                                   decltype(std::declval<const S&>().k_steps_last(0))>>
    : std::true_type {};

template <class R, class Sched, class Epi, bool kAMn = false, bool kBMn = false,
          class Side = NoSide>
__device__ __forceinline__ void run_pair_pipeline(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                                  const Sched& sch, Epi& epi, uint32_t* err,
                                                  int withhold_first_load = 0,
                                                  const Side& side = Side()) {
  constexpr int kBK = R::kBK;
  constexpr int kAtoms = R::kAtoms;
  constexpr int kStages = R::kStages;
  constexpr int kABytes = R::kABytes;
  constexpr int kBBytes = R::kBBytes;
  constexpr int kStageBytes = R::kStageBytes;
  constexpr int kNumBars = R::kNumBars;
  constexpr bool kPair = R::kPair;
  static_assert(kPair || (!kAMn && !kBMn), "a lone CTA takes K-major operands only");
  // the MMA issuer steps descriptors by address / 16 within 14 bits: every
  // shared address of the ring (all of a CTA's shared memory) is below 2^18
  static_assert(232448 < (1 << 18), "shared memory per CTA below 2^18 bytes");
  uint8_t* smem = pipeline_smem_base();
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // 0: leader (issues the MMAs), 1: peer; a lone CTA is its own leader
  const uint32_t rank = kPair ? cluster_rank() : 0u;
  const int pair = kPair ? blockIdx.x >> 1 : blockIdx.x;  // this CTA's (pair's) place in the grid
  const int n_pairs = kPair ? gridDim.x >> 1 : gridDim.x;
  const int units = sch.units();

  // The error word of this call starts at zero; a wait can only give up (and
  // set it) a full time bound after every CTA of the grid has started.
  if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), (kPair ? 2 : 1) * kEpilogueThreads);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmB)) : "memory");
  }
  if (warp == 1) {
    if constexpr (kPair) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if constexpr (kPair) cluster_sync();  // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA loader
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pending = 0;         // stages with a load in flight (leader: bit mask)
      uint32_t pending_parity = 0;  // parity of that load's phase
      bool ok = true;
      for (int u = pair; ok && u < units; u += n_pairs) {
        int a_row, b_row, kb0, kb1;
        sch.coords(u, rank, a_row, b_row, kb0, kb1);
        int k_off = 0;
        if constexpr (HasKSegments<Sched>::value) k_off = sch.k_offset(u);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int k0 = k_off + kb * kBK;  // first K element of the block
          if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, err, kErrLoader)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * kStageBytes);
          const uint32_t leader_full = kPair ? cluster_addr(full_bar(stage), 0) : full_bar(stage);
          if (rank == 0) {
            mbar_arrive_expect_tx(full_bar(stage), (kPair ? 2 : 1) * kStageBytes);
            pending |= 1u << stage;
            pending_parity = (pending_parity & ~(1u << stage)) | (phase << stage);
          }
          // checked build: a negative coordinate is recorded and its copy
          // withheld (the stage's bounded waits then give up: no fault)
          const bool withheld = (withhold_first_load != 0 && pair == 0 && rank == 0 &&
                                 u == pair && kb == kb0) ||
                                !LP_CHECK(a_row >= 0 && b_row >= 0 && k0 >= 0, kChkTmaCoord);
          if (!withheld && !kPair) {
            // a lone CTA: its 128 rows of A and all 256 rows of the B tile (two
            // 128-row boxes per 64 of K), counted on its own barrier
#pragma unroll
            for (int i = 0; i < kAtoms; ++i) {
              tma_load_2d_local(sa + i * (kABytes / kAtoms), tmA, k0 + i * kAtomK, a_row,
                                leader_full);
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_2d_local(sa + kABytes + i * (kBBytes / kAtoms) + h * (kBBytes / kAtoms / 2),
                                  tmB, k0 + i * kAtomK, b_row + h * kBNHalf, leader_full);
            }
          } else if (!withheld) {
            if (kAMn) {
              tma_load_2d(sa, tmA, a_row, k0, leader_full);
              tma_load_2d(sa + kABytes / 2, tmA, a_row + 64, k0, leader_full);
            } else {
#pragma unroll
              for (int i = 0; i < kAtoms; ++i)
                tma_load_2d(sa + i * (kABytes / kAtoms), tmA, k0 + i * kAtomK, a_row,
                            leader_full);
            }
            if (kBMn) {
              tma_load_2d(sa + kABytes, tmB, b_row, k0, leader_full);
              tma_load_2d(sa + kABytes + kBBytes / 2, tmB, b_row + 64, k0, leader_full);
            } else {
#pragma unroll
              for (int i = 0; i < kAtoms; ++i)
                tma_load_2d(sa + kABytes + i * (kBBytes / kAtoms), tmB, k0 + i * kAtomK,
                            b_row, leader_full);
            }
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && rank == 0) {  // let every issued copy land before the pair can exit
        for (int s = 0; s < kStages; ++s)
          if (pending & (1u << s)) drain_wait(full_bar(s), (pending_parity >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      if (rank == 0) {
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int u = pair; ok && u < units; u += n_pairs) {
          int a_row, b_row, kb0, kb1;
          sch.coords(u, rank, a_row, b_row, kb0, kb1);
          if (!wait_bar(tempty_bar(acc), acc_phase ^ 1u, abort_flag, err, kErrMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
          int last_steps = kBK / kUmmaK;
          if constexpr (HasKSegments<Sched>::value) last_steps = sch.k_steps_last(u);
          for (int kb = kb0; kb < kb1; ++kb) {
            const int n_steps = kb == kb1 - 1 ? last_steps : kBK / kUmmaK;
            if (!wait_bar(full_bar(stage), phase, abort_flag, err, kErrMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * kStageBytes);
            const uint32_t sb = sa + kABytes;
            // The descriptors of the stage's first step; a later step's differ
            // only in the start address field (address / 16, bits 0-13), and
            // shared addresses stay below 2^18, so adding the step's offset / 16
            // gives exactly the step's descriptor (no carry out of the field)
            // with one add instead of rebuilding it.
            const uint64_t da = kAMn ? sw128_mn_desc(sa, R::kMnBoxBytes) : sw128_desc(sa);
            const uint64_t db = kBMn ? sw128_mn_desc(sb, R::kMnBoxBytes) : sw128_desc(sb);
            // one MMA step (16 K) of the stage
            auto issue = [&](int k) {
              // K-major: box k / 4 of the stage, 32 bytes per step within it;
              // M- or N-major: 8 K rows of 128 bytes per step
              constexpr int kSteps = kAtomK / kUmmaK;
              const uint32_t offA = kAMn ? k * 2048
                                         : (k / kSteps) * (kABytes / kAtoms) +
                                               (k % kSteps) * kUmmaK * 2;
              const uint32_t offB = kBMn ? k * 2048
                                         : (k / kSteps) * (kBBytes / kAtoms) +
                                               (k % kSteps) * kUmmaK * 2;
              const uint64_t ad = da + (offA >> 4);
              const uint64_t bd = db + (offB >> 4);
              if constexpr (kPair)
                tc_mma(d_tmem, ad, bd, (kb != kb0 || k != 0) ? 1u : 0u, idesc(kAMn, kBMn));
              else
                tc_mma_single(d_tmem, ad, bd, (kb != kb0 || k != 0) ? 1u : 0u,
                              idesc(false, false, kBM));
            };
            // whole blocks through the unrolled steps (the issuing thread's
            // instruction count per MMA matters: a loop that can exit early
            // cost the products several percent); a segment's last block
            // issues only its steps
            if (n_steps == kBK / kUmmaK) {
#pragma unroll
              for (int k = 0; k < kBK / kUmmaK; ++k) issue(k);
            } else {
#pragma unroll
              for (int k = 0; k < kBK / kUmmaK; ++k)
                if (k < n_steps) issue(k);
            }
            // frees the stage (in both CTAs of a pair)
            if constexpr (kPair) tc_commit_pair(empty_bar(stage));
            else tc_commit_local(empty_bar(stage));
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          // accumulator ready (in both CTAs of a pair)
          if constexpr (kPair) tc_commit_pair(tfull_bar(acc));
          else tc_commit_local(tfull_bar(acc));
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
        // arrives once every MMA issued here is done
        if constexpr (kPair) tc_commit_pair(drain_bar);
        else tc_commit_local(drain_bar);
      }
      drain_wait(drain_bar, 0);
    }
  } else if (warp < 2 + kEpilogueThreads / 32) {
    // -------------------------------------------------------------- epilogue
    const int lane_grp = warp & 3;  // tensor-memory lanes 32*lane_grp .. +31
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(lane_grp * 32) << 16);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = pair; u < units; u += n_pairs) {
      // one lane waits, the warp follows (tcgen05.ld is warp-collective)
      int go = 1;
      if (lane == 0) go = wait_bar(tfull_bar(acc), acc_phase, abort_flag, err, kErrEpilogue);
      go = __shfl_sync(0xffffffffu, go, 0);
      if (!go) break;
      tc_fence_after();
      epi.consume(u, t_lane + static_cast<uint32_t>(acc * kBN), rank, lane_grp, lane);
      tc_fence_before();
      if constexpr (kPair) mbar_arrive_cluster(cluster_addr(tempty_bar(acc), 0));
      else mbar_arrive_local(tempty_bar(acc));
      epi.after_release(u, rank, lane_grp, lane);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    epi.finish(lane_grp, lane);
  } else {
    side(lane);
  }

  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if constexpr (kPair) cluster_sync();  // no remote arrive or copy into either CTA is still pending
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (kPair)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(kTmemCols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(kTmemCols)
                   : "memory");
  }
}

// ------------------------------------------------------------ host helpers

// 2-D bf16 tensor map over [rows, cols] (cols contiguous, row stride ld
// elements) with a box of [box_rows, 64] and 128-byte swizzle; out-of-range
// elements read as zero.  Returns false if the CUDA driver rejects it.
bool encode_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                    int box_rows);

// 3-D fp32 tensor map over [S, rows, cols] (cols contiguous, row stride ld
// elements, S matrices split_stride elements apart) with 32 x 32 x 1 boxes and
// 128-byte swizzle, for bulk stores of output tiles; elements outside the
// tensor are not written.  Returns false if the CUDA driver rejects it (e.g. a
// stride that is not a multiple of 16 bytes).
bool encode_f32_3d_store(CUtensorMap* map, void* base, int64_t S, int64_t rows, int64_t cols,
                         int64_t ld, int64_t split_stride);

// The same over bf16 [S, rows, cols] with 64 x 32 x 1 boxes (128-byte rows).
bool encode_bf16_3d_store(CUtensorMap* map, void* base, int64_t S, int64_t rows, int64_t cols,
                          int64_t ld, int64_t split_stride);

// Persistent grid (in CTAs, even) for `units` units on `sm_count` SMs under the
// process-wide CTA limit: one CTA pair per two SMs, never more pairs than units.
int pair_grid(int sm_count, int64_t units);

// The same in CTAs for CTAs that work alone (SingleRing): one per SM.
int single_grid(int sm_count, int64_t units);

// Let `kernel` launch with `bytes` of dynamic shared memory (once per kernel
// and context).
cudaError_t set_smem_limit(const void* kernel, int bytes);

}  // namespace tc
}  // namespace lp
