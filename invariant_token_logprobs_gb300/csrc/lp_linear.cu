// lp_linear.cu: fused LM-head projection + selected-token log-probability
// ("linear_logp", rlkernel.linear_logp.bitwise.v1 in the backend readbacks of
// the RL-Kernel H100 PCP evidence record, h100-pcp.json, section "validation").
//
// z = H W^T (bf16 inputs, fp32 accumulation) is formed one 256 x 256 tile at a
// time in tensor memory by the CTA-pair pipeline of lp_tcgen05.cuh (or, for
// batches of at most 128 rows, one 128 x 256 tile per CTA alone) and reduced
// on the spot to a per-row state (max, sum-exp, sum-exp*(z-max), target logit);
// the T x V logits never reach global memory.
//
// Tiling.  The vocabulary is cut into four quarters [floor(qV/4),
// floor((q+1)V/4)); each quarter into 256-column tiles counted from the
// quarter's first column (the last tile of a quarter is masked past the
// quarter's end).  Rows are cut into 256-row blocks (128 for lone CTAs).  A
// work unit is one (row block, quarter, tile); its per-row state goes to the
// workspace, and a second kernel merges the tiles of each quarter (rebased to
// the quarter's maximum, summed in a fixed tree) and then the quarters as
// (Q0 + Q1) + (Q2 + Q3).  Every value depends only on the row and on the fixed tile grid
// of its quarter: not on T, the row's offset, the shard, the grid size or the
// order in which CTAs pick up tiles.  Units are taken round-robin in
// (tile, row block) order so that the pairs that share a W tile run at the
// same time and W is read from HBM about once.
//
// Epilogue: one row per thread, 64 columns at a time (tcgen05.ld x64); the
// running maximum is raised once per 64 columns and the exponentials of a fully
// valid piece are summed in packed f32x2 arithmetic.
//
// Temperature: maxima are taken over raw logits and every difference z - m is
// multiplied by fl(1/tau) before the exponential; with tau == 1 no
// multiplication is made.
//
// A pipeline wait that gives up sets the workspace error word (see
// lp_tcgen05.cuh); the merge kernel then writes NaN for every row.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "lp_check.cuh"
#include "lp_device.cuh"
#include "lp_internal.h"
#include "lp_tcgen05.cuh"

namespace lp {

// ------------------------------------------------------------ host helpers

namespace tc {

namespace {
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
}  // namespace

bool encode_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                    int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kAtomK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_f32_3d_store(CUtensorMap* map, void* base, int64_t S, int64_t rows, int64_t cols,
                         int64_t ld, int64_t split_stride) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  if (((ld * 4) % 16) != 0 || ((split_stride * 4) % 16) != 0 ||
      (reinterpret_cast<uintptr_t>(base) % 16) != 0)
    return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(S)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 4,
                                 static_cast<cuuint64_t>(S > 1 ? split_stride : rows * ld) * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_3d_store(CUtensorMap* map, void* base, int64_t S, int64_t rows, int64_t cols,
                          int64_t ld, int64_t split_stride) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  if (((ld * 2) % 16) != 0 || ((split_stride * 2) % 16) != 0 ||
      (reinterpret_cast<uintptr_t>(base) % 16) != 0)
    return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(S)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2,
                                 static_cast<cuuint64_t>(S > 1 ? split_stride : rows * ld) * 2};
  const cuuint32_t box[3] = {64, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same for CTAs that work alone: one per SM.
int single_grid(int sm_count, int64_t units) {
  int ctas = sm_count;
  const int limit = persistent_grid_limit();
  if (limit > 0 && limit < ctas) ctas = limit;
  if (units < ctas) ctas = static_cast<int>(units);
  if (ctas < 1) ctas = 1;
  return ctas;
}

int pair_grid(int sm_count, int64_t units) {
  int pairs = sm_count / 2;
  const int limit = persistent_grid_limit();
  if (limit > 0 && (limit + 1) / 2 < pairs) pairs = (limit + 1) / 2;
  if (units < pairs) pairs = static_cast<int>(units);
  if (pairs < 1) pairs = 1;
  return 2 * pairs;
}

cudaError_t set_smem_limit(const void* kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace tc

namespace {

using namespace tc;

// Work list of the fused logprob kernels: unit u = (row block mb, quarter ql
// of this call, tile j), row block fastest.
struct QuarterTiles {
  int64_t V;       // full vocabulary size
  int64_t w_row0;  // global vocabulary index of W row 0
  int n_mb;        // row blocks
  int mb_rows;     // rows per block: 256 for CTA pairs, 128 for CTAs alone
  int n_kb;        // K blocks of the ring
  int q_first;
  int n_tiles_q;
  int total;

  __device__ __forceinline__ int units() const { return total; }
  __device__ __forceinline__ void decode(int u, int& mb, int& ql, int& j) const {
    mb = u % n_mb;
    const int g = u / n_mb;
    ql = g / n_tiles_q;
    j = g % n_tiles_q;
  }
  __device__ __forceinline__ void coords(int u, uint32_t rank, int& a_row, int& b_row, int& kb0,
                                         int& kb1) const {
    int mb, ql, j;
    decode(u, mb, ql, j);
    a_row = mb * mb_rows + static_cast<int>(rank) * kBM;
    b_row = static_cast<int>(quarter_begin(V, q_first + ql) - w_row0) + j * kBN +
            static_cast<int>(rank) * kBNHalf;
    kb0 = 0;
    kb1 = n_kb;
  }
  // Columns of tile j of quarter q that lie inside the quarter, and the
  // tile's first global column.
  __device__ __forceinline__ void tile_span(int ql, int j, int& valid, int64_t& c0) const {
    const int q = q_first + ql;
    const int64_t qc0 = quarter_begin(V, q);
    const int64_t qw = quarter_begin(V, q + 1) - qc0;
    c0 = qc0 + static_cast<int64_t>(j) * kBN;
    valid = static_cast<int>(
        max(static_cast<int64_t>(0), min(static_cast<int64_t>(kBN), qw - int64_t(j) * kBN)));
  }
};

struct LinearArgs {
  QuarterTiles tiles;
  const int64_t* targets;
  float4* chunks;  // [T][n_q][n_tiles_q]
  uint32_t* err;
  float inv_tau;   // differences z - m are multiplied by it (1: no temperature)
  float tau;       // stored in the quarter states
  int T;
  int n_q;
  int withhold_first_load;  // fault injection for tests of the bounded waits
};

// Add the 64 logits of a fully valid piece to the online state (whose maximum
// already covers them): d = (x - m) / tau, e = 2^(d log2e) (ex2.approx.ftz),
// s += e, u += e d, in packed f32x2 arithmetic with four lane sums.  Used only
// when every logit of the piece is finite, which a product of finite bf16
// inputs always is.
template <bool kScaled>
__device__ __forceinline__ void accumulate_piece_packed(const float (&v)[64], Online& st,
                                                        float inv_tau) {
  const uint64_t mm = pk2(st.m, st.m);
  const uint64_t ll = pk2(kLog2e, kLog2e);
  const uint64_t it = pk2(inv_tau, inv_tau);
  const uint64_t zero = pk2(0.f, 0.f);
  uint64_t s2[2] = {zero, zero}, u2[2] = {zero, zero};
#pragma unroll
  for (int i = 0; i < 64; i += 2) {
    uint64_t d2 = sub2(pk2(v[i], v[i + 1]), mm);
    if (kScaled) d2 = mul2(d2, it);
    float a0, a1;
    upk2(mul2(d2, ll), a0, a1);
    const uint64_t e2 = pk2(exp2_approx(a0), exp2_approx(a1));
    const int k = (i >> 1) & 1;
    s2[k] = add2(s2[k], e2);
    u2[k] = fma2(e2, d2, u2[k]);
  }
  float sa[4], ua[4];
  upk2(s2[0], sa[0], sa[1]);
  upk2(s2[1], sa[2], sa[3]);
  upk2(u2[0], ua[0], ua[1]);
  upk2(u2[1], ua[2], ua[3]);
  st.s = __fadd_rn(st.s, __fadd_rn(__fadd_rn(sa[0], sa[1]), __fadd_rn(sa[2], sa[3])));
  st.u = __fadd_rn(st.u, __fadd_rn(__fadd_rn(ua[0], ua[1]), __fadd_rn(ua[2], ua[3])));
}

// Epilogue of the logprob kernel: the tile's per-row state.
struct StateEpilogue {
  const LinearArgs* a;
  Online st;
  float t;

  __device__ __forceinline__ void consume(int u, uint32_t taddr, uint32_t rank, int lane_grp,
                                          int lane) {
    int mb, ql, j;
    a->tiles.decode(u, mb, ql, j);
    const int64_t row =
        static_cast<int64_t>(mb) * a->tiles.mb_rows + rank * kBM + lane_grp * 32 + lane;
    const int64_t y = row < a->T ? a->targets[row] : -1;
    int valid;
    int64_t tile_c0;
    a->tiles.tile_span(ql, j, valid, tile_c0);
    const int64_t yl64 = y - tile_c0;
    const int yl = (y >= 0 && yl64 >= 0 && yl64 < valid) ? static_cast<int>(yl64) : -1;

    st.reset();
    t = neg_inf();
    const float inv_tau = a->inv_tau;
#pragma unroll 1
    for (int p = 0; p < kBN / 64; ++p) {
      float v[64];
      __syncwarp();
      tmem_load64(taddr + static_cast<uint32_t>(p * 64), v);
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
      st.raise_to(bm, inv_tau);
      if (p * 64 + 64 <= valid) {
        if (inv_tau == 1.f)
          accumulate_piece_packed<false>(v, st, inv_tau);
        else
          accumulate_piece_packed<true>(v, st, inv_tau);
      } else if (st.active()) {
        float sa[4] = {0.f, 0.f, 0.f, 0.f};
        float ua[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float e, d;
          term(v[i], st.m, inv_tau, e, d);
          sa[i & 3] = __fadd_rn(sa[i & 3], e);
          ua[i & 3] = __fmaf_rn(e, d, ua[i & 3]);
        }
        st.s = __fadd_rn(st.s, __fadd_rn(__fadd_rn(sa[0], sa[1]), __fadd_rn(sa[2], sa[3])));
        st.u = __fadd_rn(st.u, __fadd_rn(__fadd_rn(ua[0], ua[1]), __fadd_rn(ua[2], ua[3])));
      }
    }
  }

  __device__ __forceinline__ void finish(int, int) {}

  __device__ __forceinline__ void after_release(int u, uint32_t rank, int lane_grp, int lane) {
    int mb, ql, j;
    a->tiles.decode(u, mb, ql, j);
    const int64_t row =
        static_cast<int64_t>(mb) * a->tiles.mb_rows + rank * kBM + lane_grp * 32 + lane;
    if (row < a->T) {
      const int64_t idx = (row * a->n_q + ql) * a->tiles.n_tiles_q + j;
      if (LP_CHECK(ql < a->n_q && j < a->tiles.n_tiles_q &&
                       idx < int64_t(a->T) * a->n_q * a->tiles.n_tiles_q,
                   kChkStateIndex))
        a->chunks[idx] = make_float4(st.m, st.s, st.u, t);
    }
  }
};

// The pipeline follows the batch.  With one 256-row block (T <= 256) the
// kernel streams W from HBM: up to 128 rows one CTA per tile (SingleRing), so
// no tensor core multiplies the zero rows a pair's second half would hold;
// 129..256 rows a pair with the 6 x 64 ring, which ran ~2% faster there than
// 3 x 128 (T = 1: 205 against 209 us).  From two blocks on the kernel is
// tensor-bound and the 3 x 128 ring is 4-12% faster (T = 512: 370 against
// 386 us; T = 2048: 1365 against 1540 us).  Every form issues the MMAs of an
// accumulator element in the same K order, so the bits do not change.
// Batches of at most this many rows run one CTA per tile and 128-row block.
// Above 128 rows a pair does the same tensor work with less shared-memory
// traffic per SM: lone CTAs at T = 192 / 256 took 238 / 242 us against 216 /
// 222 us as pairs (same bits).
constexpr int64_t kSingleMaxRows = kBM;

template <class R>
__device__ __forceinline__ void linear_body(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                            const LinearArgs& a) {
  // words 1..3 of the error header belong to the backward's kernels; a call
  // of this kernel starts them at zero too
  if (blockIdx.x == 0 && threadIdx.x == 0) a.err[1] = a.err[2] = a.err[3] = 0u;
  // the merge kernel (a programmatic dependent of this grid) may be scheduled
  // now: it waits for this grid to finish before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  StateEpilogue epi{&a};
  run_pair_pipeline<R>(tmA, tmB, a.tiles, epi, a.err, a.withhold_first_load);
}

template <class R>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    lp_linear_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const __grid_constant__ LinearArgs a) {
  linear_body<R>(&tmA, &tmB, a);
}

__global__ void __launch_bounds__(kThreads, 1)
    lp_linear_single_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ LinearArgs a) {
  linear_body<SingleRing>(&tmA, &tmB, a);
}

// Merge the tile states of each quarter and then either finalise the row from
// its four quarters or store the quarter states of a shard.  One block per
// row, one warp per quarter: the quarter's maximum is exact (order-free); lane
// l rebases tiles l, l+32, l+64, ... to it and sums them, and the 32 lane sums
// are combined by a fixed shuffle tree.  The result depends only on the
// quarter's tile states.  When `lse` is given, the row's log-partition
// log Z = M / tau + log S is also written there.
__global__ void __launch_bounds__(128)
    lp_tile_merge_kernel(const float4* __restrict__ chunks, const int64_t* __restrict__ targets,
                         const uint32_t* __restrict__ err, int n_q, int n_tiles_q, int64_t V,
                         float inv_tau, float tau, int64_t T, float* __restrict__ logp,
                         float* __restrict__ entropy, QuarterState* __restrict__ partials_out,
                         float* __restrict__ lse) {
  __shared__ __align__(16) QuarterState qs[kQuarters];
  // launched as a programmatic dependent of the fused kernel: wait for that
  // grid to finish and its stores to be visible (a no-op in a plain launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int ql = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  if (!LP_CHECK(row < T, kChkRowIndex)) return;
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
      const float delta = __fmul_rn(__fsub_rn(x.x, M), inv_tau);
      if (x.x != neg_inf() && !(delta < kExpClampLo)) {  // NaN goes on
        const float a = exp_neg(delta);
        S = __fadd_rn(S, __fmul_rn(a, x.y));
        U = __fadd_rn(U, __fmul_rn(a, __fmaf_rn(delta, x.y, x.z)));
      }
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
      QuarterState st{M, S, 0.f, U, t, tau, 0.f, 0.f};
      if (*err != 0u) st.s_hi = quiet_nan();  // a pipeline wait gave up: no result
      if (partials_out != nullptr) {
        if (LP_CHECK(row * n_q + ql < T * n_q, kChkStateIndex))
          store_state(&partials_out[row * n_q + ql], st);
      }
      else
        store_state(&qs[ql], st);
    }
  }
  if (partials_out != nullptr) return;
  __syncthreads();
  if (threadIdx.x < 4) {
    const QuarterState mine = load_state(&qs[threadIdx.x]);
    float lp, ent, lz;
    finalise_quad(mine, 0xfu, lp, ent, lz);
    if (threadIdx.x == 0) {
      logp[row] = lp;
      if (entropy != nullptr) entropy[row] = ent;
      if (lse != nullptr) lse[row] = lz;
    }
  }
}

// Batches of fewer than kPadRows rows are first copied into a zero-padded
// block of kPadRows rows in the workspace: with a row extent this small the
// operand loads ran ~1.6x slower (T = 1..9: 300-330 us against 200 us padded,
// at d = 4096, V = 151936); from 16 rows on the unpadded loads are as fast.
// The zero rows change nothing (the loads fill rows past the end with zeros
// anyway); the results are the same bits.
constexpr int64_t kPadRows = 16;

size_t chunk_bytes(int64_t T, int64_t V_total, int n_q) {
  return static_cast<size_t>(n_q) * static_cast<size_t>(tiles_per_quarter(V_total)) *
         static_cast<size_t>(T) * sizeof(float4);
}

// dst [rows_out, d8] (dense, d8 = d rounded up to 8) = H [T, d] (row stride
// ld_h, a multiple of 8) with zeros past column d and past row T; 16 bytes per
// thread and step (both 16-byte aligned).
__global__ void lp_pad_rows_kernel(const uint16_t* __restrict__ H, int64_t ld_h, int64_t T,
                                   int64_t d, int64_t rows_out, uint4* __restrict__ dst) {
  const int64_t d16 = (d + 7) / 8;
  const int64_t n = rows_out * d16;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / d16, c = i % d16;
    if (LP_CHECK(i < rows_out * d16 && c * 8 < ld_h, kChkCopyIndex))
      dst[i] = r < T ? load_row_chunk(H + r * ld_h, d, c) : make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace

size_t linear_workspace_bytes(int64_t T, int64_t d, int64_t V_total, int n_q) {
  size_t bytes = kWorkspaceHeader + chunk_bytes(T, V_total, n_q);
  if (T > 0 && T < kPadRows)
    bytes = (bytes + 255) / 256 * 256 + static_cast<size_t>(kPadRows * ((d + 7) / 8 * 8)) * 2;
  return bytes;
}

lp_status launch_linear_stats(const Device& dev, const void* H, int64_t ld_h, const void* W,
                              int64_t ld_w, const int64_t* targets, int64_t T, int64_t d,
                              int64_t V_total, int q_first, int n_q, const TauArgs& tau,
                              float* logp, float* entropy, float* partials_out, float* lse,
                              void* workspace, cudaStream_t stream) {
  static PerContextOnce attr;
  if (attr.run(dev.ctx_id, [] {
        cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(lp_linear_kernel<WideRing>),
                                       WideRing::kSmemBytes);
        if (e == cudaSuccess)
          e = set_smem_limit(reinterpret_cast<const void*>(lp_linear_kernel<NarrowRing>),
                             NarrowRing::kSmemBytes);
        if (e == cudaSuccess)
          e = set_smem_limit(reinterpret_cast<const void*>(lp_linear_single_kernel),
                             SingleRing::kSmemBytes);
        return e;
      }) != cudaSuccess)
    return LP_ERR_CUDA;

  const int64_t w_row0 = quarter_begin(V_total, q_first);
  // An empty shard (only possible when V < 4) still maps one row; all of its
  // tiles are masked.
  const int64_t w_rows = max(quarter_begin(V_total, q_first + n_q) - w_row0, int64_t(1));
  int64_t h_rows = T;
  if (T > 0 && T < kPadRows) {
    const size_t off = (kWorkspaceHeader + chunk_bytes(T, V_total, n_q) + 255) / 256 * 256;
    void* padded = static_cast<uint8_t*>(workspace) + off;
    const int64_t d8 = (d + 7) / 8 * 8;
    lp_pad_rows_kernel<<<static_cast<unsigned>((kPadRows * d8 / 8 + 255) / 256), 256, 0,
                         stream>>>(static_cast<const uint16_t*>(H), ld_h, T, d, kPadRows,
                                   static_cast<uint4*>(padded));
    if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
    H = padded;
    ld_h = d8;
    h_rows = kPadRows;
  }
  CUtensorMap tmA, tmB;
  if (!encode_bf16_2d(&tmA, H, h_rows, d, ld_h, kBM)) return LP_ERR_CUDA;
  if (!encode_bf16_2d(&tmB, W, w_rows, d, ld_w, kBNHalf)) return LP_ERR_CUDA;

  LinearArgs a;
  a.tiles.V = V_total;
  a.tiles.w_row0 = w_row0;
  const bool single = T <= kSingleMaxRows;  // one CTA per tile: no pair half of zero rows
  a.tiles.mb_rows = single ? kBM : 2 * kBM;
  a.tiles.n_mb = static_cast<int>((T + a.tiles.mb_rows - 1) / a.tiles.mb_rows);
  const bool wide = !single && a.tiles.n_mb > 1;
  const int bk = wide ? WideRing::kBK : single ? SingleRing::kBK : NarrowRing::kBK;
  a.tiles.n_kb = static_cast<int>((d + bk - 1) / bk);
  a.tiles.q_first = q_first;
  a.tiles.n_tiles_q = static_cast<int>(tiles_per_quarter(V_total));
  const int64_t total = int64_t(a.tiles.n_mb) * n_q * a.tiles.n_tiles_q;
  if (total >= (int64_t(1) << 31)) return LP_ERR_INVALID_ARGUMENT;
  a.tiles.total = static_cast<int>(total);
  a.targets = targets;
  a.chunks = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) + kWorkspaceHeader);
  a.err = static_cast<uint32_t*>(workspace);
  a.inv_tau = tau.inv_hi;
  a.tau = tau.tau;
  a.T = static_cast<int>(T);
  a.n_q = n_q;
  a.withhold_first_load = fault_injection() == 1 ? 1 : 0;

  const int grid = single ? single_grid(dev.sm_count, total) : pair_grid(dev.sm_count, total);
  cudaEvent_t ev_start, ev_stop;
  timing_events(&ev_start, &ev_stop);
  if (ev_start != nullptr && cudaEventRecord(ev_start, stream) != cudaSuccess) return LP_ERR_CUDA;
  if (wide)
    lp_linear_kernel<WideRing><<<grid, kThreads, WideRing::kSmemBytes, stream>>>(tmA, tmB, a);
  else if (single)
    lp_linear_single_kernel<<<grid, kThreads, SingleRing::kSmemBytes, stream>>>(tmA, tmB, a);
  else
    lp_linear_kernel<NarrowRing><<<grid, kThreads, NarrowRing::kSmemBytes, stream>>>(tmA, tmB, a);
  if (cudaGetLastError() != cudaSuccess) return LP_ERR_CUDA;
  if (ev_stop != nullptr && cudaEventRecord(ev_stop, stream) != cudaSuccess) return LP_ERR_CUDA;
  // the merge as a programmatic dependent launch: its launch overlaps the
  // tail of the fused kernel instead of following it (~2 us per call at
  // T <= 128; no change at T = 512)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, lp_tile_merge_kernel, static_cast<const float4*>(a.chunks), targets,
                         static_cast<const uint32_t*>(a.err), n_q, a.tiles.n_tiles_q, V_total,
                         a.inv_tau, a.tau, T, logp, entropy,
                         reinterpret_cast<QuarterState*>(partials_out), lse) != cudaSuccess)
    return LP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

lp_status launch_linear(const Device& dev, const void* H, int64_t ld_h, const void* W,
                        int64_t ld_w, const int64_t* targets, int64_t T, int64_t d,
                        int64_t V_total, int q_first, int n_q, const TauArgs& tau, float* logp,
                        float* entropy, float* partials_out, void* workspace,
                        cudaStream_t stream) {
  return launch_linear_stats(dev, H, ld_h, W, ld_w, targets, T, d, V_total, q_first, n_q,
                             tau, logp, entropy, partials_out, nullptr, workspace, stream);
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

// Device address of g_static_scratch in the calling thread's current context.
// In host code the array's name is only a host-side stand-in; the device
// address comes from cudaGetSymbolAddress with the context current.  The
// address belongs to the module as loaded into that context, so it is cached
// per context id and looked up again in a context not seen before (another
// device, a context the caller created, or the primary context re-created after
// cudaDeviceReset).  The first no-alloc call in each context does the look-up.
lp_status static_scratch(void** out) {
  constexpr int kSlots = 16;
  static std::mutex mu;
  static uint64_t ids[kSlots] = {};
  static void* addr[kSlots] = {};
  static int next = 0;
  uint64_t ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (ctx != 0)
    for (int i = 0; i < kSlots; ++i)
      if (ids[i] == ctx) {
        *out = addr[i];
        return LP_OK;
      }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return LP_ERR_CUDA;
  }
  // the look-up makes the device's primary context current when none was
  if (ctx == 0) ctx = current_context_id();
  if (ctx != 0) {
    ids[next] = ctx;
    addr[next] = p;
    next = (next + 1) % kSlots;
  }
  *out = p;
  return LP_OK;
}

cudaError_t take_check_word_linear(uint32_t* out) { return take_check_word(out); }

}  // namespace lp
