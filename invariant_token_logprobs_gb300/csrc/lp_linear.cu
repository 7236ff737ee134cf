// lp_linear.cu: fused LM-head projection + selected-token log-probability
// ("linear_logp", rlkernel.linear_logp.bitwise.v1 in the backend readbacks of
// the RL-Kernel H100 PCP evidence record, h100-pcp.json, section "validation").
//
// z = H W^T (bf16 inputs, fp32 accumulation) is formed one 256 x 256 tile at a
// time in tensor memory and reduced on the spot to a per-row state
// (max, sum-exp, sum-exp*(z-max), target logit); the T x V logits never reach
// global memory.
//
// Tiling.  The vocabulary is cut into four quarters [floor(qV/4),
// floor((q+1)V/4)); each quarter into 256-column tiles counted from the
// quarter's first column (the last tile of a quarter is masked past the
// quarter's end).  Rows are cut into 256-row blocks.  A work unit is one
// (row block, quarter, tile); its per-row state goes to the workspace, and a
// second kernel merges the tiles of each quarter (rebased to the quarter's
// maximum, float64 sums in a fixed tree) and then the quarters as
// (Q0 + Q1) + (Q2 + Q3).  Every value depends only on the row and on the fixed
// tile grid of its quarter: not on T, the row's offset, the shard, the grid
// size or the order in which CTAs pick up tiles.
//
// Kernel structure: persistent CTA pairs (thread-block clusters of 2, one CTA
// per SM), each CTA with 6 warps.  The pair computes a 256 x 256 tile with
// tcgen05.mma.cta_group::2 (M=256, N=256, K=16, kind::f16 bf16 x bf16 -> f32):
// CTA r holds rows 128r..128r+127 of the H tile and rows 128r..128r+127 of the
// W tile in its own shared memory, and receives rows 128r.. of the result in
// its own tensor memory.  Each SM so stages 32 KB per 64-wide K block instead
// of the 48 KB a single-CTA 128 x 256 tile needs: with the tensor core reading
// what TMA writes, shared-memory bandwidth is what bounds a single-CTA tile.
//   warp 0     TMA loader (both CTAs): its CTA's halves of the H and W boxes
//              (64 x 128 each, 128-byte swizzle) into a 6-stage ring; the
//              bytes of both CTAs complete one barrier in the leader CTA;
//   warp 1     tensor memory: 512 columns (two 128 x 256 fp32 accumulators)
//              allocated by both CTAs; one lane of the leader CTA issues the
//              MMAs and commits them to barriers in both CTAs (multicast);
//   warps 2-5  epilogue (both CTAs): tcgen05.ld of the finished accumulator,
//              one row per thread, online reduction in column order, state
//              store, then an arrive on the leader's accumulator-empty barrier.
// While the epilogues drain one accumulator the MMAs fill the other.  Units
// are taken round-robin in (tile, row block) order so that the pairs that
// share a W tile run at the same time and W is read from HBM about once.
//
// Temperature: with inv_tau != 1 every logit leaving tensor memory is first
// multiplied by inv_tau; with inv_tau == 1 nothing changes.
//
// Every wait on an mbarrier is bounded by %globaltimer: a wait that gives up
// sets the workspace error word and an abort flag in shared memory, the other
// roles of that CTA stop at their next wait (the roles of the other CTA give up
// on their own bounded waits), in-flight copies and MMAs are drained with
// bounded waits, tensor memory is freed and the CTAs return.  The merge kernel
// then writes NaN for every row.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "lp_device.cuh"
#include "lp_internal.h"

namespace lp {
namespace {

constexpr int kBM = 128;       // rows of H per CTA (tensor-memory lanes); 256 per pair
constexpr int kBN = kTileN;    // vocabulary columns per tile (pair); 128 W rows per CTA
constexpr int kBNHalf = kBN / 2;
constexpr int kBK = 64;        // K per pipeline stage: 64 bf16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;
constexpr int kStages = 6;
constexpr int kABytes = kBM * kBK * 2;       // 16 KB
constexpr int kBBytes = kBNHalf * kBK * 2;   // 16 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kEpilogueThreads = 128;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kNumBars * 8 + 16;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28; M = 256 for the CTA pair.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (uint32_t(kBN >> 3) << 17) | (uint32_t((2 * kBM) >> 4) << 24);

struct LinearArgs {
  const int64_t* targets;
  float4* chunks;  // [T][n_q][n_tiles_q]
  uint32_t* err;
  int64_t V;       // full vocabulary size
  int64_t w_row0;  // global vocabulary index of W row 0
  float inv_tau;   // every logit is multiplied by it (1: no temperature)
  int T;
  int n_mb;        // 256-row blocks
  int n_kb;
  int q_first;
  int n_q;
  int n_tiles_q;
  int total_tiles;
};

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

// Bounded wait for the phase of `bar` with parity `parity`.  Returns false when
// the CTA is aborting or this wait gave up (then it raises the abort).
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      uint32_t* err, uint32_t role_bit) {
  if (mbar_try_wait(bar, parity)) return true;
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

// Bounded wait used while draining after an abort; never raises anything.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
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

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
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

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
// Start address >> 4 in bits 0-13, leading-dimension offset (unused for this
// layout, set to 16 bytes) in bits 16-29, stride offset 1024 >> 4 in bits
// 32-45, descriptor version 1 in bits 46-47, swizzle mode 2 (128-byte) in
// bits 61-63.  The tile base is 1024-byte aligned, so the K offset of each
// 16-element MMA step is added to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16 >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// 64 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_load64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      :         "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Add the 64 logits of a fully valid piece to the online state (whose maximum
// already covers them): e = 2^(x log2e - m log2e) (one fma, one ex2.approx.ftz),
// s += e, u += e (x - m), in packed f32x2 arithmetic with four lane sums.  Used
// only when every logit of the piece is finite, which a product of finite bf16
// inputs always is.
__device__ __forceinline__ void accumulate_piece_packed(const float (&v)[64], Online& st) {
  const float mL = __fmul_rn(st.m, kLog2e);
  uint64_t mm, ll, nml, zero;
  asm("mov.b64 %0, {%1, %1};" : "=l"(mm) : "f"(st.m));
  asm("mov.b64 %0, {%1, %1};" : "=l"(ll) : "f"(kLog2e));
  asm("mov.b64 %0, {%1, %1};" : "=l"(nml) : "f"(-mL));
  asm("mov.b64 %0, {%1, %1};" : "=l"(zero) : "f"(0.f));
  uint64_t s2[2] = {zero, zero}, u2[2] = {zero, zero};
#pragma unroll
  for (int i = 0; i < 64; i += 2) {
    uint64_t x2, d2, a2, e2;
    float a0, a1, e0, e1;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x2) : "f"(v[i]), "f"(v[i + 1]));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d2) : "l"(x2), "l"(mm));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(a2) : "l"(x2), "l"(ll), "l"(nml));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a2));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(a0));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(e2) : "f"(e0), "f"(e1));
    const int k = (i >> 1) & 1;
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(s2[k]) : "l"(e2));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(u2[k]) : "l"(e2), "l"(d2));
  }
  float sa[4], ua[4];
  asm("mov.b64 {%0, %1}, %2;" : "=f"(sa[0]), "=f"(sa[1]) : "l"(s2[0]));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(sa[2]), "=f"(sa[3]) : "l"(s2[1]));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(ua[0]), "=f"(ua[1]) : "l"(u2[0]));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(ua[2]), "=f"(ua[3]) : "l"(u2[1]));
  st.s = __fadd_rn(st.s, __fadd_rn(__fadd_rn(sa[0], sa[1]), __fadd_rn(sa[2], sa[3])));
  st.u = __fadd_rn(st.u, __fadd_rn(__fadd_rn(ua[0], ua[1]), __fadd_rn(ua[2], ua[3])));
}

__device__ __forceinline__ void decode_tile(const LinearArgs& a, int u, int& mb, int& ql, int& j) {
  mb = u % a.n_mb;
  const int g = u / a.n_mb;
  ql = g / a.n_tiles_q;
  j = g % a.n_tiles_q;
}

// ------------------------------------------------------------------- kernel
// ------------------------------------------------------------------- kernel

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    lp_linear_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const LinearArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
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
  const uint32_t rank = cluster_rank();  // 0: leader (issues the MMAs), 1: peer
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;

  // The error word of this call starts at zero; a wait can only give up (and
  // set it) a full time bound after every CTA of the grid has started.
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * kEpilogueThreads);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync();  // both CTAs' barriers initialised and tensor memory allocated
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
      for (int u = pair; ok && u < a.total_tiles; u += n_pairs) {
        int mb, ql, j;
        decode_tile(a, u, mb, ql, j);
        const int a_row = mb * (2 * kBM) + static_cast<int>(rank) * kBM;
        const int b_row = static_cast<int>(quarter_begin(a.V, a.q_first + ql) - a.w_row0) +
                          j * kBN + static_cast<int>(rank) * kBNHalf;
        for (int kb = 0; kb < a.n_kb; ++kb) {
          if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, a.err, kErrLoader)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * kStageBytes);
          const uint32_t leader_full = cluster_addr(full_bar(stage), 0);
          if (rank == 0) {
            mbar_arrive_expect_tx(full_bar(stage), 2 * kStageBytes);
            pending |= 1u << stage;
            pending_parity = (pending_parity & ~(1u << stage)) | (phase << stage);
          }
          tma_load_2d(sa, &tmA, kb * kBK, a_row, leader_full);
          tma_load_2d(sa + kABytes, &tmB, kb * kBK, b_row, leader_full);
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
        for (int u = pair; ok && u < a.total_tiles; u += n_pairs) {
          if (!wait_bar(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.err, kErrMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
          for (int kb = 0; kb < a.n_kb; ++kb) {
            if (!wait_bar(full_bar(stage), phase, abort_flag, a.err, kErrMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * kStageBytes);
            const uint32_t sb = sa + kABytes;
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k) {
              tc_mma(d_tmem, sw128_desc(sa + k * kUmmaK * 2), sw128_desc(sb + k * kUmmaK * 2),
                     (kb | k) != 0 ? 1u : 0u);
            }
            tc_commit_pair(empty_bar(stage));  // frees the stage in both CTAs
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit_pair(tfull_bar(acc));  // accumulator ready in both CTAs
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
        tc_commit_pair(drain_bar);  // arrives once every MMA issued here is done
      }
      drain_wait(drain_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int lane_grp = warp & 3;  // tensor-memory lanes 32*lane_grp .. +31
    const int row_in_tile = static_cast<int>(rank) * kBM + lane_grp * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(lane_grp * 32) << 16);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = pair; u < a.total_tiles; u += n_pairs) {
      int mb, ql, j;
      decode_tile(a, u, mb, ql, j);
      const int q = a.q_first + ql;
      const int64_t row = static_cast<int64_t>(mb) * (2 * kBM) + row_in_tile;
      const int64_t y = row < a.T ? a.targets[row] : -1;
      const int64_t qc0 = quarter_begin(a.V, q);
      const int64_t qw = quarter_begin(a.V, q + 1) - qc0;
      const int64_t tile_c0 = qc0 + static_cast<int64_t>(j) * kBN;
      const int valid = static_cast<int>(
          max(static_cast<int64_t>(0), min(static_cast<int64_t>(kBN), qw - int64_t(j) * kBN)));
      const int64_t yl64 = y - tile_c0;
      const int yl = (y >= 0 && yl64 >= 0 && yl64 < valid) ? static_cast<int>(yl64) : -1;

      // one lane waits, the warp follows (tcgen05.ld is warp-collective)
      int go = 1;
      if (lane == 0) go = wait_bar(tfull_bar(acc), acc_phase, abort_flag, a.err, kErrEpilogue);
      go = __shfl_sync(0xffffffffu, go, 0);
      if (!go) break;
      tc_fence_after();

      Online st;
      st.reset();
      float t = neg_inf();
#pragma unroll 1
      for (int p = 0; p < kBN / 64; ++p) {
        float v[64];
        __syncwarp();
        tmem_load64(t_lane + static_cast<uint32_t>(acc * kBN + p * 64), v);
        if (a.inv_tau != 1.f) {
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = __fmul_rn(v[i], a.inv_tau);
        }
        if (p * 64 + 64 > valid) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (p * 64 + i >= valid) v[i] = neg_inf();
        }
        const bool mine = yl >= p * 64 && yl < p * 64 + 64;
        if (__any_sync(0xffffffffu, mine)) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (mine && yl == p * 64 + i) t = v[i];
        }
        float bm = v[0];
#pragma unroll
        for (int i = 1; i < 64; ++i) bm = fmax_nan(bm, v[i]);
        st.raise_to(bm);
        if (p * 64 + 64 <= valid) {
          accumulate_piece_packed(v, st);
        } else if (st.active()) {
          float sa[4] = {0.f, 0.f, 0.f, 0.f};
          float ua[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            float e, d;
            term(v[i], st.m, e, d);
            sa[i & 3] = __fadd_rn(sa[i & 3], e);
            ua[i & 3] = __fmaf_rn(e, d, ua[i & 3]);
          }
          st.s = __fadd_rn(st.s, __fadd_rn(__fadd_rn(sa[0], sa[1]), __fadd_rn(sa[2], sa[3])));
          st.u = __fadd_rn(st.u, __fadd_rn(__fadd_rn(ua[0], ua[1]), __fadd_rn(ua[2], ua[3])));
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(cluster_addr(tempty_bar(acc), 0));
      if (row < a.T) {
        a.chunks[(row * a.n_q + ql) * a.n_tiles_q + j] = make_float4(st.m, st.s, st.u, t);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync();  // no remote arrive or copy into either CTA is still pending
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}


// Merge the tile states of each quarter and then either finalise the row from
// its four quarters or store the quarter states of a shard.  One block per
// row, one warp per quarter: the quarter's maximum is exact (order-free); lane
// l rebases tiles l, l+32, l+64, ... to it and sums them, and the 32 lane sums
// are combined by a fixed shuffle tree.  The result depends only
// on the quarter's tile states.
__global__ void __launch_bounds__(128)
    lp_tile_merge_kernel(const float4* __restrict__ chunks, const int64_t* __restrict__ targets,
                         const uint32_t* __restrict__ err, int n_q, int n_tiles_q, int64_t V,
                         float* __restrict__ logp, float* __restrict__ entropy,
                         float4* __restrict__ partials_out) {
  __shared__ float4 qs[kQuarters];
  const int ql = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  if (ql < n_q) {
    const float4* c = chunks + (row * n_q + ql) * n_tiles_q;
    float M = neg_inf();
    for (int j = lane; j < n_tiles_q; j += 32) M = fmaxf(M, c[j].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float S = 0.f, U = 0.f;
    float t = neg_inf();
    for (int j = lane; j < n_tiles_q; j += 32) {
      const float4 x = c[j];
      float s, u;
      rebase(x.x, x.y, x.z, M, s, u);
      S = __fadd_rn(S, s);
      U = __fadd_rn(U, u);
      t = fmax_nan(t, x.w);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      S = __fadd_rn(S, __shfl_down_sync(0xffffffffu, S, off));
      U = __fadd_rn(U, __shfl_down_sync(0xffffffffu, U, off));
      t = fmax_nan(t, __shfl_down_sync(0xffffffffu, t, off));
    }
    if (lane == 0) {
      const int64_t y = targets[row];
      if (y < 0 || y >= V) t = quiet_nan();
      float4 st = make_float4(M, S, U, t);
      if (*err != 0u) st.y = quiet_nan();  // a pipeline wait gave up: no result
      if (partials_out != nullptr)
        partials_out[row * n_q + ql] = st;
      else
        qs[ql] = st;
    }
  }
  if (partials_out != nullptr) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    const float4 q4[kQuarters] = {qs[0], qs[1], qs[2], qs[3]};
    float lp, ent;
    finalise(q4, lp, ent);
    logp[row] = lp;
    if (entropy != nullptr) entropy[row] = ent;
  }
}

// ------------------------------------------------------------ host helpers

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over [rows, cols] (cols contiguous) with a box of
// [box_rows, 64] and 128-byte swizzle; out-of-range elements read as zero.
bool encode_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                    int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t linear_workspace_bytes(int64_t T, int64_t V_total, int n_q) {
  return kWorkspaceHeader +
         static_cast<size_t>(n_q) * static_cast<size_t>(tiles_per_quarter(V_total)) *
             static_cast<size_t>(T) * sizeof(float4);
}

lp_status launch_linear(const Device& dev, const void* H, int64_t ld_h, const void* W,
                        int64_t ld_w, const int64_t* targets, int64_t T, int64_t d,
                        int64_t V_total, int q_first, int n_q, float inv_tau, float* logp,
                        float* entropy, float* partials_out, void* workspace,
                        cudaStream_t stream) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(lp_linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
  });
  if (attr_err != cudaSuccess) return LP_ERR_CUDA;

  const int64_t w_row0 = quarter_begin(V_total, q_first);
  // An empty shard (only possible when V < 4) still maps one row; all of its
  // tiles are masked.
  const int64_t w_rows = max(quarter_begin(V_total, q_first + n_q) - w_row0, int64_t(1));
  CUtensorMap tmA, tmB;
  if (!encode_bf16_2d(&tmA, H, T, d, ld_h, kBM)) return LP_ERR_CUDA;
  if (!encode_bf16_2d(&tmB, W, w_rows, d, ld_w, kBNHalf)) return LP_ERR_CUDA;

  LinearArgs a;
  a.targets = targets;
  a.chunks = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) + kWorkspaceHeader);
  a.err = static_cast<uint32_t*>(workspace);
  a.V = V_total;
  a.w_row0 = w_row0;
  a.inv_tau = inv_tau;
  a.T = static_cast<int>(T);
  a.n_mb = static_cast<int>((T + 2 * kBM - 1) / (2 * kBM));
  a.n_kb = static_cast<int>((d + kBK - 1) / kBK);
  a.q_first = q_first;
  a.n_q = n_q;
  a.n_tiles_q = static_cast<int>(tiles_per_quarter(V_total));
  const int64_t total = int64_t(a.n_mb) * n_q * a.n_tiles_q;
  if (total >= (int64_t(1) << 31)) return LP_ERR_INVALID_ARGUMENT;
  a.total_tiles = static_cast<int>(total);

  // one CTA pair per two SMs (clusters of 2), never more pairs than units
  int pairs = dev.sm_count / 2;
  const int limit = persistent_grid_limit();
  if (limit > 0 && (limit + 1) / 2 < pairs) pairs = (limit + 1) / 2;
  if (total < pairs) pairs = static_cast<int>(total);
  if (pairs < 1) pairs = 1;
  const int grid = 2 * pairs;

  cudaEvent_t ev_start, ev_stop;
  timing_events(&ev_start, &ev_stop);
  if (ev_start != nullptr && cudaEventRecord(ev_start, stream) != cudaSuccess) return LP_ERR_CUDA;
  lp_linear_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, a);
  if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
  if (ev_stop != nullptr && cudaEventRecord(ev_stop, stream) != cudaSuccess) return LP_ERR_CUDA;
  lp_tile_merge_kernel<<<static_cast<unsigned>(T), 128, 0, stream>>>(
      a.chunks, targets, a.err, n_q, a.n_tiles_q, V_total, logp, entropy,
      reinterpret_cast<float4*>(partials_out));
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

// --------------------------------------------- fixed scratch for the no-alloc call
//
// lp_linear_logprob_noalloc runs the same two kernels as lp_linear_logprob, but
// with its workspace in this file-scope device array instead of memory the
// caller allocates.  Every device that loads the library holds the array until
// the process exits.  All calls on a device share it and it keeps the last
// call's contents; the only part that must start at zero (the error word in
// its header) is cleared by each call's kernel.  Two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array and may return wrong results.

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

size_t static_scratch_bytes() { return kStaticScratchBytes; }

// Device address of g_static_scratch on the current device.  In host code the
// array's name is only a host-side stand-in; the device address comes from
// cudaGetSymbolAddress, called once per device with that device current (the
// first no-alloc call on each device does it).
lp_status static_scratch(int ordinal, void** out) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static void* addr[kMaxDev] = {};
  if (ordinal < 0 || ordinal >= kMaxDev) return LP_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[ordinal] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LP_ERR_CUDA;
    }
    addr[ordinal] = p;
  }
  *out = addr[ordinal];
  return LP_OK;
}

}  // namespace lp
