// lp_backward.cu: gradient of the fused LM-head logprob/entropy loss.
//
// For L = sum_t g_logp[t] logp[t] + g_ent[t] entropy[t] with z = H W^T and
// p = softmax(z / tau):
//   G[t, v] = dL/dz[t, v]
//           = (g_logp[t] (delta(v, y_t) - p[t, v])
//              - g_ent[t] p[t, v] (log p[t, v] + entropy[t])) / tau
//   dL/dH = G W,   dL/dW = G^T H.
// This is the training side of the operator whose forward is lp_linear.cu (the
// trainer of the RL-Kernel H100 PCP evidence record back-propagates through
// these log-probabilities: h100-pcp.json, section "comparison",
// train/grad_norm).
//
// Steps, all on the tensor-core pair pipeline of lp_tcgen05.cuh:
//   1. unless the caller passes the forward's log Z and entropy per row, the
//      forward kernels again, keeping them;
//   2. lp_grad_kernel: z tiles recomputed in tensor memory; the epilogue forms
//      G in fp32 and stores it in bf16 as G [T, V];
//   3. lp_gemm_kernel<K-major A, N-major B>: dH = G W, reading W [V, d] as an
//      N-major operand, over fixed vocabulary ranges (partial products in
//      fp32): 7 per quarter of the vocabulary when V % 64 == 0, else 19 of the
//      whole vocabulary;
//   4. lp_gemm_kernel<M-major A, N-major B>: dW = G^T H, reading G [T, V] as an
//      M-major operand and H [T, d] as an N-major one.  A seventh warp per CTA
//      adds the ranges of dH meanwhile — each quarter's in order, then
//      (Q0 + Q1) + (Q2 + Q3) — (lp_split_sum_kernel does it on its own when
//      dW is not asked for), and the last CTA to finish fills dW with NaN if
//      a wait of the call gave up.
// Both products write their output through TMA bulk stores from a swizzled
// staging area (dW may instead be added into a main gradient with the TMA
// reduction).  No operand is transposed in memory.  Every output element is
// produced by one CTA pair with a fixed K order and split sums are added in a
// fixed order: the results are deterministic, and a row of dH depends only on
// that row's inputs (not on T or its offset).  A call may cover a shard of
// whole vocabulary quarters (W's rows of the shard, global targets, the merged
// rows' statistics): its dW rows are those of the whole call, and its dH is
// the quarter tree's subtree of its quarters, to be merged by
// launch_merge_grad_h.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "lp_check.cuh"
#include "lp_device.cuh"
#include "lp_internal.h"
#include "lp_tcgen05.cuh"

namespace lp {
namespace {

using namespace tc;

// Ring geometry of the gradient kernel (both operands K-major, like the fused
// forward) and of the two products (M/N-major operands).  The gradient kernel
// picks its form by batch as the fused forward does (up to 128 rows: one CTA
// per tile; one 256-row block: the narrow ring; more: the wide ring, which
// with the 256-bit G stores below saves ~8 us per call at T = 512).  The products ran ~1% faster on
// the narrow ring (both products; the dH product alone on the wide ring: no
// change).
using GradHRing = NarrowRing;  // dH = G W (A K-major)
using GradWRing = NarrowRing;  // dW = G^T H (A M-major)
template <bool kAMn>
using GemmRing = std::conditional_t<kAMn, GradWRing, GradHRing>;
constexpr int kGemmBK = GradHRing::kBK;  // K block of both products
static_assert(GradWRing::kBK == kGemmBK, "one K block for the product work list");
// the products' staging area starts where either ring ends
static_assert(WideRing::kSmemEnd == NarrowRing::kSmemEnd, "one staging offset");
constexpr int kGemmRingEnd = NarrowRing::kSmemEnd;

// Fixed vocabulary ranges of the dH product (split K).  When every quarter of
// the vocabulary starts on a 16-column boundary (V % 64 == 0) each quarter is
// cut into kRangesPerQuarter ranges, summed in order within the quarter, and
// the quarter sums are added as (Q0 + Q1) + (Q2 + Q3): a shard of whole
// quarters computes one subtree of that order, so the shards' partial dH merge
// to the bits of one GPU.  Otherwise the whole vocabulary is cut into
// kSplitsDH ranges summed in order.  Constants, so the bits never depend on
// the GPU or the batch; 7 per quarter makes the 32 output tiles of T = 512,
// d = 4096 11.8 waves of 76 CTA pairs, 19 exactly 8.
constexpr int kSplitsDH = 19;
constexpr int kRangesPerQuarter = 7;
constexpr int kMaxSplitsDH = 4 * kRangesPerQuarter;
static_assert(kMaxSplitsDH >= kSplitsDH, "partial buffers for either order");

inline int64_t round8(int64_t x) { return (x + 7) / 8 * 8; }

// ------------------------------------------------------------------ gradient

struct GradTiles {  // same work list as the forward kernel: (row block, quarter, tile)
  int64_t V;       // full vocabulary size
  int64_t w_row0;  // global vocabulary index of W's row 0 and of G's column 0
  int q_first;     // first quarter of this call (a shard's quarters: q_first ..)
  int n_mb;
  int n_kb;
  int n_tiles_q;
  int total;
  __device__ __forceinline__ int units() const { return total; }
  __device__ __forceinline__ void decode(int u, int& mb, int& q, int& j) const {
    mb = u % n_mb;
    const int g = u / n_mb;
    q = g / n_tiles_q;
    j = g % n_tiles_q;
  }
  __device__ __forceinline__ void coords(int u, uint32_t rank, int& a_row, int& b_row, int& kb0,
                                         int& kb1) const {
    int mb, q, j;
    decode(u, mb, q, j);
    a_row = mb * (2 * kBM) + static_cast<int>(rank) * kBM;
    b_row = static_cast<int>(quarter_begin(V, q_first + q) - w_row0) + j * kBN +
            static_cast<int>(rank) * kBNHalf;
    kb0 = 0;
    kb1 = n_kb;
  }
};

struct GradArgs {
  GradTiles tiles;
  const int64_t* targets;
  const float* g_logp;    // [T] or NULL
  const float* g_ent;     // [T] or NULL
  const float* lse;       // [T] log Z of the scaled logits
  const float* ent;       // [T] entropy
  __nv_bfloat16* G;       // [T][ld_g], column c: vocabulary index w_row0 + c
  uint32_t* err;
  uint32_t* ticket;       // finish counter of the dW product, zeroed here
  int64_t ld_g;
  float inv_tau;
  int T;
};

// One 256-bit store (p 32-byte aligned).
__device__ __forceinline__ void store_32_bytes(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

struct GradEpilogue {
  const GradArgs* a;

  __device__ __forceinline__ void consume(int u, uint32_t taddr, uint32_t rank, int lane_grp,
                                          int lane) {
    int mb, q, j;
    a->tiles.decode(u, mb, q, j);
    const int64_t row = static_cast<int64_t>(mb) * (2 * kBM) + rank * kBM + lane_grp * 32 + lane;
    const bool row_ok = row < a->T;
    const int64_t qc0 = quarter_begin(a->tiles.V, a->tiles.q_first + q);
    const int64_t qw = quarter_begin(a->tiles.V, a->tiles.q_first + q + 1) - qc0;
    const int64_t c0 = qc0 + static_cast<int64_t>(j) * kBN;
    const int valid = static_cast<int>(
        max(static_cast<int64_t>(0), min(static_cast<int64_t>(kBN), qw - int64_t(j) * kBN)));
    float gl = 0.f, ge = 0.f, log_z = 0.f, ent = 0.f;
    int yl = -1;
    if (row_ok) {
      const int64_t y = a->targets[row];
      const bool y_ok = y >= 0 && y < a->tiles.V;
      gl = (a->g_logp != nullptr && y_ok) ? a->g_logp[row] : 0.f;
      ge = a->g_ent != nullptr ? a->g_ent[row] : 0.f;
      log_z = a->lse[row];
      ent = a->ent[row];
      const int64_t yl64 = y - c0;
      if (y_ok && yl64 >= 0 && yl64 < valid) yl = static_cast<int>(yl64);
    }
    const float scale = a->inv_tau;
#pragma unroll 1
    for (int p = 0; p < kBN / 64; ++p) {
      float v[64];
      __syncwarp();
      tmem_load64(taddr + static_cast<uint32_t>(p * 64), v);
      if (!row_ok || p * 64 >= valid) continue;
      uint32_t pk[32];  // G of columns 2i, 2i+1 as packed bf16x2
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        float g2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float zs = __fmul_rn(v[i + h], scale);                   // z / tau
          const float lp = __fsub_rn(zs, log_z);                         // log p
          const float pr = exp_fast(lp);                                 // p
          // -p (g_logp + g_ent (log p + entropy)) + g_logp [v == y], then / tau
          float g = -__fmul_rn(pr, __fmaf_rn(ge, __fadd_rn(lp, ent), gl));
          if (p * 64 + i + h == yl) g = __fadd_rn(g, gl);
          g2[h] = __fmul_rn(g, scale);
        }
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(g2[0], g2[1]);
        pk[i >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      const int n = min(64, valid - p * 64);
      const int64_t col0 = c0 + p * 64 - a->tiles.w_row0;  // column of G
      if (!LP_CHECK(row < a->T && col0 >= 0 && col0 + n <= a->ld_g, kChkGStore)) continue;
      __nv_bfloat16* grow = a->G + row * a->ld_g + col0;
      // a thread writes its row's 128 bytes: as four whole 32-byte sectors when
      // aligned (half the store transactions of 16-byte stores; the L1 cycles
      // they free matter to the ring), else 16 or 2 bytes at a time
      if (n == 64 && ((reinterpret_cast<uintptr_t>(grow) & 31u) == 0)) {
#pragma unroll
        for (int i = 0; i < 32; i += 8)
          store_32_bytes(grow + 2 * i, pk + i);
      } else if (n == 64 && ((reinterpret_cast<uintptr_t>(grow) & 15u) == 0)) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<uint4*>(grow + 2 * i) = make_uint4(pk[i], pk[i + 1], pk[i + 2], pk[i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          if (i < n) {
            const uint16_t bits = static_cast<uint16_t>(pk[i >> 1] >> (16 * (i & 1)));
            grow[i] = *reinterpret_cast<const __nv_bfloat16*>(&bits);
          }
        }
      }
    }
  }
  __device__ __forceinline__ void after_release(int, uint32_t, int, int) {}
  __device__ __forceinline__ void finish(int, int) {}
};

template <class R>
__device__ __forceinline__ void grad_body(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                          const GradArgs& a) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.ticket = 0u;
  GradEpilogue epi{&a};
  run_pair_pipeline<R>(tmA, tmB, a.tiles, epi, a.err);
}

template <class R>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    lp_grad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ GradArgs a) {
  grad_body<R>(&tmA, &tmB, a);
}

// Batches of at most 128 rows: one CTA per tile, as in the fused forward.
__global__ void __launch_bounds__(kThreads, 1)
    lp_grad_single_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ GradArgs a) {
  grad_body<SingleRing>(&tmA, &tmB, a);
}

// ---------------------------------------------------------------------- GEMM

// C[M, N] (fp32, row stride ldc) = A[M, K] B[N, K]^T for the K blocks of split
// s; split s writes C + s * split_stride.  Units: (row block, column block,
// split), with the row block or the column block fastest (the operand that is
// shared by consecutive units stays in L2).
struct GemmTiles {
  int n_mb, n_nb, n_split, n_kb, kb_per_split, total;
  int nb_fastest;
  // K in segments of seg_w elements (seg_w a multiple of 16; 0: one segment,
  // all of K), each of n_kb K blocks in seg_splits splits; split s is split
  // s % seg_splits of segment s / seg_splits
  int seg_w, seg_splits;
  __device__ __forceinline__ int units() const { return total; }
  __device__ __forceinline__ void decode(int u, int& mb, int& nb, int& s) const {
    if (nb_fastest) {
      nb = u % n_nb;
      const int g = u / n_nb;
      mb = g % n_mb;
      s = g / n_mb;
    } else {
      mb = u % n_mb;
      const int g = u / n_mb;
      nb = g % n_nb;
      s = g / n_nb;
    }
  }
  __device__ __forceinline__ void coords(int u, uint32_t rank, int& a_row, int& b_row, int& kb0,
                                         int& kb1) const {
    int mb, nb, s;
    decode(u, mb, nb, s);
    a_row = mb * (2 * kBM) + static_cast<int>(rank) * kBM;
    b_row = nb * kBN + static_cast<int>(rank) * kBNHalf;
    kb0 = (s % seg_splits) * kb_per_split;
    kb1 = min(n_kb, kb0 + kb_per_split);
  }
};

// The work list with its segments' K offsets and last-block steps (the dH
// product); the dW product (one segment, K = T) takes GemmTiles alone and
// issues every K block whole.
struct SegGemmTiles : GemmTiles {
  __device__ __forceinline__ int k_offset(int u) const {
    int mb, nb, s;
    decode(u, mb, nb, s);
    return (s / seg_splits) * seg_w;
  }
  __device__ __forceinline__ int k_steps_last(int u) const {
    constexpr int kFull = kGemmBK / kUmmaK;
    if (seg_w == 0) return kFull;
    int mb, nb, s;
    decode(u, mb, nb, s);
    const int kb1 = min(n_kb, (s % seg_splits + 1) * kb_per_split);
    if (kb1 < n_kb) return kFull;
    return (seg_w - (n_kb - 1) * kGemmBK + kUmmaK - 1) / kUmmaK;
  }
};

// A 16-byte load that skips L1 and leaves L2 first in line for eviction: the
// split sum reads each partial once, and in the dW product it must not push
// out the operand blocks that consecutive units re-read from L2.
__device__ __forceinline__ float4 load_once(const float4* p) {
  float4 v;
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z),
                     __fadd_rn(a.w, b.w));
}

// out[i] = the fixed-order sum of the n_seg * seg_len partials part[s][i]
// (n_seg 1, 2 or 4; n_seg * seg_len <= kMaxSplitsDH): each segment's seg_len
// partials (the ranges of one quarter, or of the whole vocabulary) in order,
// then the segment sums as S0, S0 + S1 or (S0 + S1) + (S2 + S3); for i = i0,
// i0 + stride, ... < n4 (float4 elements: n4 = n / 4, part and out 16-byte
// aligned); NaN when an error word of the kernels that made the partials
// (words 0..2 of the call) is set.
__device__ __forceinline__ void split_sum(const float4* __restrict__ part, int64_t n4, int n_seg,
                                          int seg_len, const uint32_t* __restrict__ err,
                                          float4* __restrict__ out, int64_t i0, int64_t stride) {
  const bool failed = (err[0] | err[1] | err[2]) != 0u;
  const int n_split = n_seg * seg_len;
  const bool shape_ok = LP_CHECK(n_split <= kMaxSplitsDH && seg_len >= 1 &&
                                     (n_seg == 1 || n_seg == 2 || n_seg == 4),
                                 kChkSplitIndex);
  for (int64_t i = i0; i < n4; i += stride) {
    float4 x[kMaxSplitsDH];
#pragma unroll
    for (int k = 0; k < kMaxSplitsDH; ++k)
      if (k < n_split)
        x[k] = shape_ok ? load_once(part + k * n4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    // the running segment's sum, the even segment before it, S0 + S1, S2 + S3
    float4 cur = x[0], left = x[0], s01 = x[0], s23 = x[0];
    int seg = 0;
    int next_seg = seg_len;  // first partial of the next segment
#pragma unroll
    for (int k = 1; k < kMaxSplitsDH; ++k) {
      if (k < n_split) {
        if (k == next_seg) {  // segment seg is complete
          if ((seg & 1) == 0) left = cur;
          else if (seg == 1) s01 = add4(left, cur);
          else s23 = add4(left, cur);
          ++seg;
          next_seg += seg_len;
          cur = x[k];
        } else {
          cur = add4(cur, x[k]);
        }
      }
    }
    float4 s;
    if (n_seg == 1) s = cur;
    else if (n_seg == 2) s = add4(left, cur);
    else s = add4(s01, add4(left, cur));
    const float q = quiet_nan();
    out[i] = failed ? make_float4(q, q, q, q) : s;
  }
}

// The split sum of dH as the side warp of the dW product: the product is
// bound by its tensor work and stores, the sum by HBM reads, so the two
// overlap.  part == nullptr: nothing to do.
struct SplitSumSide {
  const float4* part;
  int64_t n4;
  int n_seg;
  int seg_len;
  const uint32_t* err;
  float4* out;
  __device__ __forceinline__ void operator()(int lane) const {
    if (part == nullptr) return;
    split_sum(part, n4, n_seg, seg_len, err, out, static_cast<int64_t>(blockIdx.x) * 32 + lane,
              static_cast<int64_t>(gridDim.x) * 32);
  }
};

// Threads of a product CTA: the pipeline's six warps and the side warp.
constexpr int kGemmThreads = kThreads + 32;

struct GemmArgs {
  GemmTiles tiles;
  CUtensorMap tmC;  // bulk-store map of C
  int64_t M;
  int64_t N;
  int n_split;      // matrices of C (split products)
  uint32_t* err;
  int out_bf16;     // C is bf16 (32 x 64 boxes) instead of fp32 (32 x 32 boxes)
  int out_add;      // fp32 boxes are added into C (TMA reduction) instead of stored
  SplitSumSide side;
  // NaN fill of poison_out[0, poison_n) (C's type) by the last CTA to finish
  // when any of the call's four error words is set (ticket == nullptr: none);
  // the ticket is zero at launch and counts finished CTAs.
  uint32_t* ticket;
  const uint32_t* err_all;
  void* poison_out;
  int64_t poison_n;
  int withhold_first_load;  // fault injection for tests of the bounded waits
};

// Epilogue of the products.  Each warp owns 32 rows of the tile and writes
// them in boxes of 32 rows x 128 bytes (32 fp32 columns, or 64 bf16 columns
// rounded to nearest even): a box is staged in shared memory with the 128-byte
// swizzle of C's store map (16-byte chunk c of row r at chunk c ^ (r % 8)), and
// one lane issues its TMA bulk store.  The warp's two staging buffers
// alternate, one per store, each reused once the store that last read it has
// finished reading.  Boxes wholly outside C are skipped (the map clips partial
// ones).  C's row stride is a multiple of 16 bytes (d % 8 == 0).
constexpr int kBoxFloats = 32 * 32;
constexpr int kBoxes = 2;  // staging buffers per epilogue warp
// dynamic shared memory of the product kernels: alignment slack, the
// pipeline, then 4 warps' staging buffers
constexpr int kGemmSmemBytes = 1024 + kGemmRingEnd + 4 * kBoxes * kBoxFloats * 4;
static_assert(kGemmSmemBytes <= 232448, "fits the 227 KB per-CTA limit");

__device__ __forceinline__ void bulk_store_3d(const CUtensorMap* map, int c0, int c1, int c2,
                                              uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// The box added element by element into C (an fp32 add in the memory system;
// every element of C is the target of exactly one box of one launch, so the
// result does not depend on timing) instead of stored.
__device__ __forceinline__ void bulk_reduce_add_3d(const CUtensorMap* map, int c0, int c1, int c2,
                                                   uint32_t src) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], "
      "[%4];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

struct GemmEpilogue {
  const GemmArgs* a;
  int next = 0;  // staging buffer of this warp's next store

  __device__ __forceinline__ void consume(int u, uint32_t taddr, uint32_t rank, int lane_grp,
                                          int lane) {
    int mb, nb, s;
    a->tiles.decode(u, mb, nb, s);
    const int64_t row0 = static_cast<int64_t>(mb) * (2 * kBM) + rank * kBM + lane_grp * 32;
    const int64_t n0 = static_cast<int64_t>(nb) * kBN;
    float* stg = reinterpret_cast<float*>(pipeline_smem_base() + kGemmRingEnd) +
                 lane_grp * kBoxes * kBoxFloats;
    if (row0 >= a->M) return;
#pragma unroll 1
    for (int p = 0; p < kBN / 64; ++p) {
      if (n0 + p * 64 >= a->N) break;
      float v[64];
      __syncwarp();
      tmem_load64(taddr + static_cast<uint32_t>(p * 64), v);
      if (a->out_bf16) {
        // the 64 columns of this piece as one box of 32 rows x 64 bf16
        float* box = stg + next * kBoxFloats;
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kBoxes - 1) : "memory");
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * c + 2 * h], v[8 * c + 2 * h + 1]);
            w[h] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          *reinterpret_cast<uint4*>(box + lane * 32 + ((c ^ (lane & 7)) * 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0 && LP_CHECK(n0 + p * 64 < a->N && row0 < a->M && s >= 0 &&
                                      s < a->n_split, kChkOutBox))
          bulk_store_3d(&a->tmC, static_cast<int>(n0 + p * 64), static_cast<int>(row0), s,
                        smem_u32(box));
        if (++next == kBoxes) next = 0;
        continue;
      }
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int64_t col = n0 + p * 64 + b * 32;
        if (col >= a->N) continue;
        float* box = stg + next * kBoxFloats;
        // the store that last read this buffer (kBoxes stores ago) has read it
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kBoxes - 1) : "memory");
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int k = b * 8 + c;
          *reinterpret_cast<float4*>(box + lane * 32 + ((c ^ (lane & 7)) * 4)) =
              make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0 && LP_CHECK(col < a->N && row0 < a->M && s >= 0 && s < a->n_split,
                                  kChkOutBox)) {
          if (a->out_add)
            bulk_reduce_add_3d(&a->tmC, static_cast<int>(col), static_cast<int>(row0), s,
                               smem_u32(box));
          else
            bulk_store_3d(&a->tmC, static_cast<int>(col), static_cast<int>(row0), s, smem_u32(box));
        }
        if (++next == kBoxes) next = 0;
      }
    }
  }
  __device__ __forceinline__ void after_release(int, uint32_t, int, int) {}
  __device__ __forceinline__ void finish(int, int lane) {
    // every bulk store of this warp has written global memory
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }
};

// The last CTA of the grid to get here fills poison_out with NaN if a wait of
// the call gave up: every CTA counts itself in after its own work, so the last
// one sees every error word of the launch (and of the kernels before it).
__device__ __forceinline__ void poison_if_failed(const GemmArgs& a) {
  uint32_t* flag = reinterpret_cast<uint32_t*>(pipeline_smem_base());  // the ring is idle now
  if (threadIdx.x == 0) {
    uint32_t failed = 0u;
    __threadfence();
    if (atomicAdd(a.ticket, 1u) == gridDim.x - 1) {
      __threadfence();
      const volatile uint32_t* e = a.err_all;
      failed = (e[0] | e[1] | e[2] | e[3]) != 0u ? 1u : 0u;
    }
    *flag = failed;
  }
  __syncthreads();
  if (*flag == 0u) return;
  for (int64_t i = threadIdx.x; i < a.poison_n; i += blockDim.x) {
    if (a.out_bf16)
      reinterpret_cast<uint16_t*>(a.poison_out)[i] = 0x7fc0u;  // bf16 NaN
    else
      reinterpret_cast<float*>(a.poison_out)[i] = quiet_nan();
  }
}

template <bool kAMn, bool kBMn>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    lp_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ GemmArgs a) {
  GemmEpilogue epi{&a};
  if constexpr (kAMn) {
    run_pair_pipeline<GemmRing<kAMn>, GemmTiles, GemmEpilogue, kAMn, kBMn, SplitSumSide>(
        &tmA, &tmB, a.tiles, epi, a.err, a.withhold_first_load, a.side);
  } else {
    const SegGemmTiles tiles{a.tiles};
    run_pair_pipeline<GemmRing<kAMn>, SegGemmTiles, GemmEpilogue, kAMn, kBMn, SplitSumSide>(
        &tmA, &tmB, tiles, epi, a.err, a.withhold_first_load, a.side);
  }
  if (a.ticket != nullptr) poison_if_failed(a);
}

// ------------------------------------------------------------- plain kernels

// dH's split sum on its own (when dW is not asked for).
__global__ void lp_split_sum_kernel(const float4* __restrict__ part, int64_t n4, int n_seg,
                                    int seg_len, const uint32_t* __restrict__ err,
                                    float4* __restrict__ out) {
  split_sum(part, n4, n_seg, seg_len, err, out,
            static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
            static_cast<int64_t>(gridDim.x) * blockDim.x);
}

// grad_H = the shards' partial dH in the order of one GPU's quarter tree:
// P0, P0 + P1 or (P0 + P1) + (P2 + P3) (n_shards 1, 2 or 4), float4 elements.
struct ShardParts {
  const float4* p[4];
};
__global__ void lp_merge_grad_h_kernel(ShardParts parts, int n_shards, int64_t n4,
                                       float4* out) {  // out may be one of the parts
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = parts.p[0][i];
    if (n_shards == 1) {
      out[i] = a;
    } else if (n_shards == 2) {
      out[i] = add4(a, parts.p[1][i]);
    } else {
      out[i] = add4(add4(a, parts.p[1][i]), add4(parts.p[2][i], parts.p[3][i]));
    }
  }
}

struct BackwardLayout {
  int64_t V8;
  size_t off_lse, off_logp, off_ent, off_g, off_dh, total;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Whether the dH product splits K by quarters (and how many partials it writes
// at most) for a vocabulary of V_total.
bool quarter_splits(int64_t V_total) { return V_total % 64 == 0; }
int max_splits_dh(int64_t V_total) {
  return quarter_splits(V_total) ? kMaxSplitsDH : kSplitsDH;
}

// V: the columns of this call (a shard's, or all V_total)
BackwardLayout backward_layout(int64_t T, int64_t d, int64_t V, int64_t V_total) {
  BackwardLayout L;
  L.V8 = round8(V);
  // the forward's workspace (for recomputed statistics; a shard has them
  // given), or only the header with the error words
  size_t o = align256(V == V_total ? linear_workspace_bytes(T, d, V, 4) : kWorkspaceHeader);
  L.off_lse = o; o = align256(o + sizeof(float) * T);
  L.off_logp = o; o = align256(o + sizeof(float) * T);
  L.off_ent = o; o = align256(o + sizeof(float) * T);
  L.off_g = o; o = align256(o + 2 * static_cast<size_t>(T) * L.V8);
  L.off_dh = o;
  o = align256(o + sizeof(float) * max_splits_dh(V_total) * static_cast<size_t>(T) * d);
  L.total = o;
  return L;
}

// C = A B^T over the pipeline.  A is [M, K] (K-major, row stride ld_a) or,
// with kAMn, [K, M] (M contiguous); B likewise with N.
// What a product launch does besides C = A B^T: the side warps' split sum and
// the last CTA's NaN fill (both off by default).
struct GemmExtras {
  SplitSumSide side{nullptr, 0, 1, 1, nullptr, nullptr};
  uint32_t* ticket = nullptr;
  const uint32_t* err_all = nullptr;
  void* poison_out = nullptr;
  int64_t poison_n = 0;
  int withhold_first_load = 0;
};

// K is split into n_seg = K / seg_w segments of seg_w elements (seg_w == 0:
// one segment, all of K), each into at most n_split splits of whole K blocks
// (fewer when the segment has fewer blocks); *n_split_out = the splits of one
// segment.  Every segment starts on a multiple of 16 elements and, for the
// K-major A, on a 16-byte boundary.
template <bool kAMn, bool kBMn>
lp_status launch_gemm(const Device& dev, const void* A, int64_t M, int64_t ld_a, const void* B,
                      int64_t N, int64_t ld_b, int64_t K, int64_t seg_w, int n_split, void* C,
                      int64_t ldc, int64_t split_stride, uint32_t* err, cudaStream_t stream,
                      int* n_split_out, bool nb_fastest, int out_mode = LP_GRAD_W_FLOAT32,
                      const GemmExtras& x = GemmExtras()) {
  static PerContextOnce attr;
  if (attr.run(dev.ctx_id, [] {
        return set_smem_limit(reinterpret_cast<const void*>(lp_gemm_kernel<kAMn, kBMn>),
                              kGemmSmemBytes);
      }) != cudaSuccess)
    return LP_ERR_CUDA;
  CUtensorMap tmA, tmB;
  using R = GemmRing<kAMn>;
  const bool okA = kAMn ? encode_bf16_2d(&tmA, A, K, M, ld_a, R::kBK)
                        : encode_bf16_2d(&tmA, A, M, K, ld_a, kBM);
  const bool okB = kBMn ? encode_bf16_2d(&tmB, B, K, N, ld_b, R::kBK)
                        : encode_bf16_2d(&tmB, B, N, K, ld_b, kBNHalf);
  if (!okA || !okB) return LP_ERR_CUDA;
  GemmArgs g;
  g.tiles.n_mb = static_cast<int>((M + 2 * kBM - 1) / (2 * kBM));
  g.tiles.n_nb = static_cast<int>((N + kBN - 1) / kBN);
  const int64_t n_seg = seg_w > 0 ? K / seg_w : 1;
  if (seg_w > 0 && (seg_w % kUmmaK != 0 || n_seg * seg_w != K || seg_w >= (int64_t(1) << 30)))
    return LP_ERR_INVALID_ARGUMENT;
  const int64_t seg_len = seg_w > 0 ? seg_w : K;
  g.tiles.n_kb = static_cast<int>((seg_len + R::kBK - 1) / R::kBK);
  g.tiles.kb_per_split = (g.tiles.n_kb + n_split - 1) / n_split;
  // every split gets at least one K block (the count depends on the segment
  // length alone)
  const int seg_splits = (g.tiles.n_kb + g.tiles.kb_per_split - 1) / g.tiles.kb_per_split;
  g.tiles.seg_w = static_cast<int>(seg_w);
  g.tiles.seg_splits = seg_splits;
  n_split = static_cast<int>(n_seg) * seg_splits;
  g.tiles.n_split = n_split;
  g.tiles.nb_fastest = nb_fastest ? 1 : 0;
  if (n_split_out != nullptr) *n_split_out = seg_splits;
  const int64_t total = int64_t(g.tiles.n_mb) * g.tiles.n_nb * n_split;
  if (total >= (int64_t(1) << 31)) return LP_ERR_INVALID_ARGUMENT;
  g.tiles.total = static_cast<int>(total);
  g.M = M;
  g.N = N;
  g.err = err;
  g.n_split = n_split;
  const bool out_bf16 = out_mode == LP_GRAD_W_BFLOAT16;
  g.out_bf16 = out_bf16 ? 1 : 0;
  g.out_add = out_mode == LP_GRAD_W_FLOAT32_ACCUMULATE ? 1 : 0;
  g.side = x.side;
  g.ticket = x.ticket;
  g.err_all = x.err_all;
  g.poison_out = x.poison_out;
  g.poison_n = x.poison_n;
  g.withhold_first_load = x.withhold_first_load;
  const bool ok_c = out_bf16 ? encode_bf16_3d_store(&g.tmC, C, n_split, M, N, ldc, split_stride)
                             : encode_f32_3d_store(&g.tmC, C, n_split, M, N, ldc, split_stride);
  if (!ok_c) return LP_ERR_CUDA;
  lp_gemm_kernel<kAMn, kBMn>
      <<<pair_grid(dev.sm_count, total), kGemmThreads, kGemmSmemBytes, stream>>>(tmA, tmB, g);
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

// Batches of fewer than kSmallRows rows run the whole backward on copies
// padded with zero rows to kSmallRows (zero upstream gradients, so the padded
// rows add nothing to grad_W and their grad_H rows are dropped): with a row
// extent this small the operand loads of all three tensor-core kernels ran
// slowly (T = 1: ~1040 us against ~880 us at T = 16).  The padded rows carry
// exactly the zeros the loads filled in before, so the results are the same
// bits.
constexpr int64_t kSmallRows = 16;

struct SmallLayout {
  size_t inner;  // workspace of the padded backward (at offset 0)
  size_t off_h, off_y, off_gl, off_ge, off_lse, off_ent, off_gh, total;
};

SmallLayout small_layout(int64_t d, int64_t V, int64_t V_total) {
  SmallLayout L;
  const int64_t d8 = (d + 7) / 8 * 8;
  size_t o = align256(backward_layout(kSmallRows, d, V, V_total).total);
  L.inner = o;
  L.off_h = o; o = align256(o + 2 * static_cast<size_t>(kSmallRows * d8));
  L.off_y = o; o = align256(o + 8 * kSmallRows);
  L.off_gl = o; o = align256(o + 4 * kSmallRows);
  L.off_ge = o; o = align256(o + 4 * kSmallRows);
  L.off_lse = o; o = align256(o + 4 * kSmallRows);
  L.off_ent = o; o = align256(o + 4 * kSmallRows);
  L.off_gh = o; o = align256(o + 4 * static_cast<size_t>(kSmallRows * d));
  L.total = o;
  return L;
}

// Zero-padded kSmallRows-row copies of the backward's per-row inputs: H (rows
// d8 = d rounded up to 8 wide, zeros past column d), targets (0 past T), and
// the optional per-row floats (0 past T).
__global__ void lp_pad_backward_kernel(const uint16_t* __restrict__ H, int64_t ld_h, int64_t d,
                                       int64_t T, const int64_t* __restrict__ y,
                                       const float* __restrict__ gl, const float* __restrict__ ge,
                                       const float* __restrict__ lse, const float* __restrict__ ent,
                                       uint4* __restrict__ H_out, int64_t* __restrict__ y_out,
                                       float* __restrict__ gl_out, float* __restrict__ ge_out,
                                       float* __restrict__ lse_out, float* __restrict__ ent_out) {
  const int64_t d16 = (d + 7) / 8;
  const int64_t n = kSmallRows * d16;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / d16, c = i % d16;
    if (LP_CHECK(c * 8 < ld_h, kChkCopyIndex))
      H_out[i] = r < T ? load_row_chunk(H + r * ld_h, d, c) : make_uint4(0u, 0u, 0u, 0u);
  }
  if (blockIdx.x == 0 && threadIdx.x < kSmallRows) {
    const int r = threadIdx.x;
    const bool in = r < T;
    y_out[r] = in ? y[r] : 0;
    if (gl != nullptr) gl_out[r] = in ? gl[r] : 0.f;
    if (ge != nullptr) ge_out[r] = in ? ge[r] : 0.f;
    if (lse != nullptr) lse_out[r] = in ? lse[r] : 0.f;
    if (ent != nullptr) ent_out[r] = in ? ent[r] : 0.f;
  }
}

// grad_h [T, d] = the first T rows of gh [kSmallRows, d].
__global__ void lp_copy_rows_kernel(const float* __restrict__ gh, int64_t n,
                                    float* __restrict__ grad_h) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    grad_h[i] = gh[i];
}

}  // namespace

size_t linear_backward_workspace_bytes(int64_t T, int64_t d, int64_t V, int64_t V_total) {
  if (T > 0 && T < kSmallRows) return small_layout(d, V, V_total).total;
  return backward_layout(T, d, V, V_total).total;
}

lp_status launch_linear_backward(const Device& dev, const void* H, int64_t ld_h, const void* W,
                                 int64_t ld_w, const int64_t* targets, int64_t T, int64_t d,
                                 int64_t V, int64_t V_total, int q_first, int n_q,
                                 const TauArgs& tau, const float* saved_lse,
                                 const float* saved_entropy, const float* g_logp,
                                 const float* g_ent, float* grad_h, void* grad_w,
                                 int grad_w_mode, void* workspace, cudaStream_t stream) {
  if (T > 0 && T < kSmallRows) {
    const SmallLayout S = small_layout(d, V, V_total);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    const int64_t d8 = (d + 7) / 8 * 8;
    uint4* h16 = reinterpret_cast<uint4*>(base + S.off_h);
    int64_t* y16 = reinterpret_cast<int64_t*>(base + S.off_y);
    float* gl16 = g_logp != nullptr ? reinterpret_cast<float*>(base + S.off_gl) : nullptr;
    float* ge16 = g_ent != nullptr ? reinterpret_cast<float*>(base + S.off_ge) : nullptr;
    float* lse16 = saved_lse != nullptr ? reinterpret_cast<float*>(base + S.off_lse) : nullptr;
    float* ent16 = saved_entropy != nullptr ? reinterpret_cast<float*>(base + S.off_ent) : nullptr;
    float* gh16 = reinterpret_cast<float*>(base + S.off_gh);
    lp_pad_backward_kernel<<<static_cast<unsigned>((kSmallRows * d8 / 8 + 255) / 256), 256, 0,
                             stream>>>(static_cast<const uint16_t*>(H), ld_h, d, T, targets,
                                       g_logp, g_ent, saved_lse, saved_entropy, h16, y16, gl16,
                                       ge16, lse16, ent16);
    if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
    const lp_status st =
        launch_linear_backward(dev, h16, d8, W, ld_w, y16, kSmallRows, d, V, V_total, q_first,
                               n_q, tau, lse16, ent16, gl16, ge16, gh16, grad_w, grad_w_mode,
                               workspace, stream);
    if (st != LP_OK) return st;
    lp_copy_rows_kernel<<<static_cast<unsigned>((T * d + 255) / 256), 256, 0, stream>>>(
        gh16, T * d, grad_h);
    return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
  }
  static PerContextOnce attr;
  if (attr.run(dev.ctx_id, [] {
        cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(lp_grad_kernel<WideRing>),
                                       WideRing::kSmemBytes);
        if (e == cudaSuccess)
          e = set_smem_limit(reinterpret_cast<const void*>(lp_grad_kernel<NarrowRing>),
                             NarrowRing::kSmemBytes);
        if (e == cudaSuccess)
          e = set_smem_limit(reinterpret_cast<const void*>(lp_grad_single_kernel),
                             SingleRing::kSmemBytes);
        return e;
      }) != cudaSuccess)
    return LP_ERR_CUDA;

  // a shard (n_q < 4) comes with the merged rows' statistics
  if (n_q < 4 && (saved_lse == nullptr || saved_entropy == nullptr)) return LP_ERR_INVALID_ARGUMENT;
  const BackwardLayout L = backward_layout(T, d, V, V_total);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);  // words 0..3, one per pipeline kernel
  const float* lse = saved_lse;
  const float* ent = saved_entropy;
  auto* G = reinterpret_cast<__nv_bfloat16*>(ws + L.off_g);
  float* dh_part = reinterpret_cast<float*>(ws + L.off_dh);

  // 1. forward statistics (log Z, entropy) of every row, unless given
  if (lse == nullptr || ent == nullptr) {
    float* lse_ws = reinterpret_cast<float*>(ws + L.off_lse);
    float* ent_ws = reinterpret_cast<float*>(ws + L.off_ent);
    lp_status st0 = launch_linear_stats(dev, H, ld_h, W, ld_w, targets, T, d, V, 0, 4, tau,
                                        reinterpret_cast<float*>(ws + L.off_logp), ent_ws,
                                        nullptr, lse_ws, workspace, stream);
    if (st0 != LP_OK) return st0;
    lse = lse_ws;
    ent = ent_ws;
  } else {
    // the error words of this call start at zero (the forward kernel would
    // have cleared them)
    if (cudaMemsetAsync(err, 0, 4 * sizeof(uint32_t), stream) != cudaSuccess) return LP_ERR_CUDA;
  }
  lp_status st = LP_OK;

  // 2. G
  {
    CUtensorMap tmA, tmB;
    if (!encode_bf16_2d(&tmA, H, T, d, ld_h, kBM)) return LP_ERR_CUDA;
    if (!encode_bf16_2d(&tmB, W, V, d, ld_w, kBNHalf)) return LP_ERR_CUDA;
    GradArgs g;
    g.tiles.V = V_total;
    g.tiles.w_row0 = quarter_begin(V_total, q_first);
    g.tiles.q_first = q_first;
    g.tiles.n_mb = static_cast<int>((T + 2 * kBM - 1) / (2 * kBM));
    const bool single = T <= kBM;
    const bool wide = g.tiles.n_mb > 1;
    const int bk = wide ? WideRing::kBK : single ? SingleRing::kBK : NarrowRing::kBK;
    g.tiles.n_kb = static_cast<int>((d + bk - 1) / bk);
    g.tiles.n_tiles_q = static_cast<int>(tiles_per_quarter(V_total));
    const int64_t total = int64_t(g.tiles.n_mb) * n_q * g.tiles.n_tiles_q;
    if (total >= (int64_t(1) << 31)) return LP_ERR_INVALID_ARGUMENT;
    g.tiles.total = static_cast<int>(total);
    g.targets = targets;
    g.g_logp = g_logp;
    g.g_ent = g_ent;
    g.lse = lse;
    g.ent = ent;
    g.G = G;
    g.err = err + 1;
    g.ticket = err + 4;
    g.ld_g = L.V8;
    g.inv_tau = tau.inv_hi;
    g.T = static_cast<int>(T);
    const int grid = single ? single_grid(dev.sm_count, total) : pair_grid(dev.sm_count, total);
    if (wide)
      lp_grad_kernel<WideRing><<<grid, kThreads, WideRing::kSmemBytes, stream>>>(tmA, tmB, g);
    else if (single)
      lp_grad_single_kernel<<<grid, kThreads, SingleRing::kSmemBytes, stream>>>(tmA, tmB, g);
    else
      lp_grad_kernel<NarrowRing><<<grid, kThreads, NarrowRing::kSmemBytes, stream>>>(tmA, tmB, g);
    if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
  }

  // 3. dH = G W (W read N-major) over fixed vocabulary ranges: per quarter
  // when the quarters start on 16-column boundaries (a shard's quarters are
  // then the subtree of one GPU's order), else over the whole vocabulary
  const bool by_quarter = quarter_splits(V_total);
  const int64_t seg_w = by_quarter ? V_total / 4 : 0;
  const int n_seg = by_quarter ? n_q : 1;
  int seg_splits = 0;
  // row blocks fastest: the pairs of one W range run together
  st = launch_gemm<false, true>(dev, G, T, L.V8, W, d, ld_w, V, seg_w,
                                by_quarter ? kRangesPerQuarter : kSplitsDH, dh_part, d, T * d,
                                err + 2, stream, &seg_splits, false);
  if (st != LP_OK) return st;
  // T * d is a multiple of 4 (d % 8 == 0); dh_part and grad_h are 16-byte aligned
  const SplitSumSide sum{reinterpret_cast<const float4*>(dh_part), T * d / 4, n_seg, seg_splits,
                         err, reinterpret_cast<float4*>(grad_h)};
  if (grad_w == nullptr) {
    // 128-thread blocks, three resident per SM at this kernel's registers (one
    // wave): ~10 us faster per call than four waves of 256-thread blocks
    lp_split_sum_kernel<<<dev.sm_count * 3, 128, 0, stream>>>(sum.part, sum.n4, sum.n_seg,
                                                              sum.seg_len, err, sum.out);
    return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
  }

  // 4. dW = G^T H (G read M-major, H read N-major), dH's split sum alongside;
  // NaN in dW if any wait of the call gave up
  GemmExtras x;
  x.side = sum;
  x.ticket = err + 4;  // zeroed by lp_grad_kernel
  x.err_all = err;
  x.poison_out = grad_w;
  x.poison_n = V * d;
  x.withhold_first_load = fault_injection() == 2 ? 1 : 0;
  // column blocks fastest: a block of G is used by 16 consecutive units
  return launch_gemm<true, true>(dev, G, V, L.V8, H, d, ld_h, T, 0, 1, grad_w, d, 0, err + 3,
                                 stream, nullptr, true, grad_w_mode, x);
}

lp_status launch_merge_grad_h(const Device& dev, const float* const* shard_grad_h, int n_shards,
                              int64_t n, float* grad_h, cudaStream_t stream) {
  ShardParts parts{};
  for (int i = 0; i < 4; ++i)
    parts.p[i] = reinterpret_cast<const float4*>(shard_grad_h[i < n_shards ? i : 0]);
  const int64_t n4 = n / 4;
  const int64_t blocks = std::min<int64_t>((n4 + 255) / 256, int64_t(dev.sm_count) * 8);
  lp_merge_grad_h_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, stream>>>(
      parts, n_shards, n4, reinterpret_cast<float4*>(grad_h));
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

cudaError_t take_check_word_backward(uint32_t* out) { return take_check_word(out); }

}  // namespace lp
