// lp_logits.cu: selected-token log-probabilities from given fp32 logits.
//
// The computation the RL-Kernel logprob prior-art report (report.json) times
// for every candidate: logp = z[y] - logsumexp(z) per row of shared logits,
// here with the per-row entropy as a side output.  It is bound by the HBM read
// of the logits (4 bytes per element, read once).
//
// Work unit: one CTA of 256 threads per (row, vocabulary quarter).  Thread i
// owns the 4-column groups g = i, i + 256, i + 512, ... counted from the
// quarter's first column; it reads them eight groups (128 bytes) at a time
// with 128-bit non-caching loads, so a warp reads 512 contiguous bytes per
// load.  A thread keeps an online state (max m, count of values equal to m,
// sum of exp((z - m)/tau) over the others, and the entropy sum), raising its
// maximum once per batch of 32 values; the terms are formed two at a time in
// f32x2 arithmetic, each exponential with the hardware 2^x.  The running
// maximum's own terms (exactly e^0 = 1) are counted instead of summed, so the
// large terms never swamp the small ones' low bits, and every rescaling of a
// thread's sums (a raised maximum, the CTA maximum) uses the accurate
// polynomial exp of lp_device.cuh.  The 256 thread states are rebased to the
// CTA maximum and summed as float pairs (hi + lo) in a fixed tree (warp
// shuffles, then 8 warp partials in a fixed pairing).  Which thread owns which
// column depends only on the column's offset inside its quarter, so a row's
// quarter state is the same whatever the row's position, batch or shard.
//
// Finalising variant: the 4 CTAs of a row form a thread-block cluster; each
// writes its 32-byte quarter state into the shared memory of cluster rank 0
// (DSMEM), and after the cluster barrier four lanes of rank 0 merge
// (Q0 + Q1) + (Q2 + Q3) with float pairs.  Partials variant: each CTA writes
// its quarter state to global memory for lp_merge_partials.
//
// Temperature: the maximum is taken over raw logits and each difference
// z - m is multiplied by 1/tau = inv_hi + inv_lo; with tau == 1 no
// multiplication is made and the results are those of the unscaled entry
// points.
#include <cuda_runtime.h>

#include "lp_check.cuh"
#include "lp_device.cuh"
#include "lp_internal.h"

namespace lp {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBatch = 8;  // 4-float groups per thread per batch (32 values)
// Resident CTAs per SM the kernels are compiled for: 5 caps them at 51
// registers a thread (48 used, a 16-byte spill) where they took 58 and fitted
// 4 per SM.  The fifth CTA keeps more loads in flight: 98.6 us against
// 101.3 us for the 1024 x 151936 logits; 6 (40 registers) spilled and ran
// 126 us.
constexpr int kCtasPerSm = 5;

__device__ __forceinline__ float4 load_stream(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Group g (columns 4g .. 4g+3 of the quarter, w < 2^31 columns); columns >= w
// read as -inf.  A whole group of a 16-byte aligned quarter is one 128-bit
// load, others are scalar loads of the same values.
__device__ __forceinline__ void load_group(const float* __restrict__ q0, int w, int g, bool vec,
                                           float (&v)[4]) {
  const int c = g * 4;
  if (vec && c + 3 < w) {
    const float4 x = load_stream(q0 + c);
    v[0] = x.x;
    v[1] = x.y;
    v[2] = x.z;
    v[3] = x.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (c + i < w) ? __ldg(q0 + c + i) : neg_inf();
  }
}

// Per-thread online state of the logits path: the running maximum m, the
// number c of values equal to it (each contributes exactly exp(0) = 1), the sum
// s of exp((z - m) / tau) over the other values, and u.  Keeping the maximal
// terms out of s keeps every rounding of the running sums relative to the
// smaller terms: a row dominated by a few large logits (the peaked workload)
// loses nothing to adding small terms onto a term of 1.
struct LogitsOnline {
  float m, c, s, u;
  __device__ __forceinline__ void reset() {
    m = neg_inf();
    c = 0.f;
    s = 0.f;
    u = 0.f;
  }
  __device__ __forceinline__ void raise_to(float bm, float inv_hi, float inv_lo) {
    if (!(bm <= m)) {
      if (m == neg_inf()) {
        c = 0.f;
        s = 0.f;
        u = 0.f;
      } else {
        const float delta = scale_diff(__fsub_rn(m, bm), inv_hi, inv_lo);  // < 0
        if (delta < kExpClampLo) {  // the old terms vanish (delta may be -inf); NaN goes on
          s = 0.f;
          u = 0.f;
        } else {
          const float a = exp_neg(delta);
          const float tot = __fadd_rn(c, s);
          u = __fmul_rn(a, __fmaf_rn(delta, tot, u));
          s = __fmul_rn(a, tot);
        }
        c = 0.f;
      }
      m = bm;
    }
  }
};

// Add one batch of values (all <= st.m) to the online state: per value
// d = (z - m) / tau, f = [d == 0] (the running maximum's term, exactly 1) to
// the count, e = exp(d) for the others to s, and e d to u.  The lanes hold
// f - e and (f - e) d (negated sums; f d = 0), two values per f32x2
// operation, four lanes.  The exponential of a single term is the hardware
// 2^x: on this GPU it measured a -5e-8 relative bias for |x| > 1 (-0.4 ulp),
// but the terms that carry a row's sum are exact (each thread's maximum, e^0
// = 1) or rescaled with the accurate exp; over every row of the peaked
// workload the logp error stays within 3e-9 of the output's own float
// rounding, and the per-term polynomial exp (unbiased) cost 12 us of 113 in
// FMA-pipe work.
template <bool kScaled>
__device__ __forceinline__ void accumulate_batch(const float (&v)[kBatch][4], LogitsOnline& st,
                                                 float inv_hi, float inv_lo) {
  const uint64_t mm = pk2(st.m, st.m);
  const uint64_t ih = pk2(inv_hi, inv_hi), il = pk2(inv_lo, inv_lo);
  const uint64_t zero = pk2(0.f, 0.f);
  uint64_t sn2[2] = {zero, zero}, c2[2] = {zero, zero}, un2[2] = {zero, zero};
#pragma unroll
  for (int k = 0; k < kBatch; ++k)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint64_t d2 = sub2(pk2(v[k][2 * h], v[k][2 * h + 1]), mm);
      if (kScaled) {  // finite before scaling: -inf * a negative 1/tau low part
        float sa, sb;
        upk2(d2, sa, sb);
        d2 = pk2(fmax_nan(sa, -3.402823466e38f), fmax_nan(sb, -3.402823466e38f));
        d2 = fma2(d2, il, mul2(d2, ih));
      }
      // f = [d == 0]; dc = d made finite for the entropy term (e dc = 0 for a
      // -inf logit); e = 2^(dc log2 e) with the hardware 2^x
      float da, db;
      upk2(d2, da, db);
      const uint64_t dc2 = pk2(fmax_nan(da, -3.402823466e38f), fmax_nan(db, -3.402823466e38f));
      const uint64_t f2 = pk2(ge_one_zero(da, 0.f), ge_one_zero(db, 0.f));
      float ya, yb;
      upk2(mul2(dc2, pk2(kLog2e, kLog2e)), ya, yb);
      const uint64_t fme2 = sub2(f2, pk2(exp2_approx(ya), exp2_approx(yb)));
      sn2[h] = add2(sn2[h], fme2);
      c2[h] = add2(c2[h], f2);
      un2[h] = fma2(fme2, dc2, un2[h]);
    }
  float sa[4], ca[4], ua[4];
  upk2(sn2[0], sa[0], sa[1]);
  upk2(sn2[1], sa[2], sa[3]);
  upk2(c2[0], ca[0], ca[1]);
  upk2(c2[1], ca[2], ca[3]);
  upk2(un2[0], ua[0], ua[1]);
  upk2(un2[1], ua[2], ua[3]);
  st.s = __fsub_rn(st.s, __fadd_rn(__fadd_rn(sa[0], sa[1]), __fadd_rn(sa[2], sa[3])));
  st.c = __fadd_rn(st.c, __fadd_rn(__fadd_rn(ca[0], ca[1]), __fadd_rn(ca[2], ca[3])));
  st.u = __fsub_rn(st.u, __fadd_rn(__fadd_rn(ua[0], ua[1]), __fadd_rn(ua[2], ua[3])));
}

// The quarter state (M, S = S_hi + S_lo, U) of the w columns starting at q0
// for softmax(z / tau); valid in thread 0.
template <bool kScaled>
__device__ __forceinline__ void quarter_state(const float* __restrict__ q0, int64_t w,
                                              float inv_hi, float inv_lo, QuarterState& out) {
  __shared__ float red_m[kWarps], red_hi[kWarps], red_lo[kWarps], red_u[kWarps];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const bool vec = (reinterpret_cast<uintptr_t>(q0) & 15u) == 0;
  const int wi = static_cast<int>(w);
  const int n_groups = (wi + 3) / 4;

  LogitsOnline st;
  st.reset();
  for (int g0 = 0; g0 < n_groups; g0 += kThreads * kBatch) {
    float v[kBatch][4];
    if (vec && (g0 + kThreads * kBatch) * 4 <= wi) {  // every group of the batch is whole
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float4 x = load_stream(q0 + (g0 + k * kThreads + tid) * 4);
        v[k][0] = x.x;
        v[k][1] = x.y;
        v[k][2] = x.z;
        v[k][3] = x.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < kBatch; ++k) load_group(q0, wi, g0 + k * kThreads + tid, vec, v[k]);
    }
    // batch maximum, three operands per instruction
    float bm = fmax3_nan(v[0][0], v[0][1], v[0][2]);
    bm = fmax_nan(bm, v[0][3]);
#pragma unroll
    for (int k = 1; k < kBatch; ++k) {
      bm = fmax3_nan(bm, v[k][0], v[k][1]);
      bm = fmax3_nan(bm, v[k][2], v[k][3]);
    }
    st.raise_to(bm, inv_hi, inv_lo);
    if (st.m != neg_inf()) accumulate_batch<kScaled>(v, st, inv_hi, inv_lo);
  }

  // CTA maximum (order-free), then every thread's sum rebased to it as a float
  // pair and the pairs summed in a fixed tree (shuffles, then the 8 warp sums
  // in a fixed pairing).
  float M = st.m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red_m[warp] = M;
  __syncthreads();
  M = red_m[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) M = fmaxf(M, red_m[i]);

  float hi = 0.f, lo = 0.f, u = 0.f;
  const float delta = scale_diff(__fsub_rn(st.m, M), inv_hi, inv_lo);
  // a thread whose maximum lies more than 87 below the CTA's (after scaling;
  // possibly -inf) adds nothing; NaN goes on
  if (st.m != neg_inf() && !(delta < kExpClampLo)) {
    const float a = exp_neg(delta);  // 1 for the thread(s) holding the maximum
    float thi, tlo;
    two_sum(st.c, st.s, thi, tlo);
    mul_pair(a, thi, tlo, hi, lo);
    u = __fmul_rn(a, __fmaf_rn(delta, thi, st.u));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ohi = __shfl_down_sync(0xffffffffu, hi, off);
    const float olo = __shfl_down_sync(0xffffffffu, lo, off);
    u = __fadd_rn(u, __shfl_down_sync(0xffffffffu, u, off));
    add_pair(hi, lo, ohi, olo, hi, lo);
  }
  if (lane == 0) {
    red_hi[warp] = hi;
    red_lo[warp] = lo;
    red_u[warp] = u;
  }
  __syncthreads();
  if (tid == 0) {
    // fixed pairwise tree over the warp sums: ((0+1)+(2+3))+((4+5)+(6+7)) for 8
    static_assert((kWarps & (kWarps - 1)) == 0, "a power of two of warps");
    float h[kWarps], l[kWarps], uu[kWarps];
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      h[i] = red_hi[i];
      l[i] = red_lo[i];
      uu[i] = red_u[i];
    }
#pragma unroll
    for (int width = kWarps / 2; width >= 1; width /= 2)
#pragma unroll
      for (int i = 0; i < width; ++i) {
        add_pair(h[2 * i], l[2 * i], h[2 * i + 1], l[2 * i + 1], h[i], l[i]);
        uu[i] = __fadd_rn(uu[2 * i], uu[2 * i + 1]);
      }
    out.s_hi = h[0];
    out.s_lo = l[0];
    out.u = uu[0];
    out.m = M;
  }
}

// RAW target logit of a quarter: z[y] if y is in [c0, c1), -inf if y is
// another valid column, NaN if y is outside [0, V).  The load is issued before
// the quarter's stream of loads (asm volatile keeps it there), so its latency
// is hidden by the reduction.
__device__ __forceinline__ float quarter_target(const float* __restrict__ q0, int64_t y,
                                                int64_t c0, int64_t c1, int64_t V) {
  if (y < 0 || y >= V) return quiet_nan();
  if (y >= c0 && y < c1) {
    float t;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(t) : "l"(q0 + (y - c0)));
    return t;
  }
  return neg_inf();
}

// Quarter state of the w columns at q0 (thread 0 holds it), the target taken
// from targets[row]; temperature tau with 1/tau = inv_hi + inv_lo.
__device__ __forceinline__ QuarterState quarter_state_any(const float* __restrict__ q0, int64_t w,
                                                          const int64_t* __restrict__ targets,
                                                          int64_t row, int64_t c0, int64_t V,
                                                          const TauArgs& tau) {
  float t = 0.f;
  if (threadIdx.x == 0) t = quarter_target(q0, targets[row], c0, c0 + w, V);
  QuarterState st{};
  if (tau.inv_hi == 1.f && tau.inv_lo == 0.f)
    quarter_state<false>(q0, w, tau.inv_hi, tau.inv_lo, st);
  else
    quarter_state<true>(q0, w, tau.inv_hi, tau.inv_lo, st);
  if (threadIdx.x == 0) {
    st.t = t;
    st.tau = tau.tau;
  }
  return st;
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads, kCtasPerSm)
    lp_logits_final_kernel(const float* __restrict__ logits, int64_t ld,
                           const int64_t* __restrict__ targets, int64_t T, int64_t V, TauArgs tau,
                           float* __restrict__ logp, float* __restrict__ entropy,
                           float* __restrict__ lse) {
  __shared__ __align__(16) QuarterState qstates[kQuarters];
  const int q = blockIdx.x & 3;
  const int64_t row = blockIdx.x >> 2;
  const int64_t c0 = quarter_begin(V, q);
  int64_t c1 = quarter_begin(V, q + 1);
  // checked build: the row exists and its quarter lies inside the row stride
  // (a failed test reads nothing: an empty quarter of row 0)
  const bool geo_ok = LP_CHECK(row < T && c1 <= ld, row < T ? kChkLogitsLoad : kChkRowIndex);
  const int64_t r = geo_ok ? row : 0;
  if (!geo_ok) c1 = c0;
  const float* q0 = logits + r * ld + c0;

  const QuarterState st = quarter_state_any(q0, c1 - c0, targets, r, c0, V, tau);
  if (threadIdx.x == 0) {
    const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(&qstates[q]));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(0));
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(st.m),
                 "f"(st.s_hi), "f"(st.s_lo), "f"(st.u)
                 : "memory");
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote + 16u),
                 "f"(st.t), "f"(st.tau), "f"(0.f), "f"(0.f)
                 : "memory");
  }
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (q == 0 && threadIdx.x < 4) {
    const QuarterState mine = load_state(&qstates[threadIdx.x]);
    float lp, ent, lz;
    finalise_quad(mine, 0xfu, lp, ent, lz);
    if (threadIdx.x == 0 && geo_ok) {
      logp[row] = lp;
      if (entropy != nullptr) entropy[row] = ent;
      if (lse != nullptr) lse[row] = lz;
    }
  }
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    lp_logits_partials_kernel(const float* __restrict__ logits_shard, int64_t ld,
                              const int64_t* __restrict__ targets, int64_t T, int64_t V,
                              int q_first, int n_q, TauArgs tau,
                              QuarterState* __restrict__ partials) {
  const int ql = blockIdx.x % n_q;
  const int64_t row = blockIdx.x / n_q;
  const int q = q_first + ql;
  const int64_t shard_c0 = quarter_begin(V, q_first);
  const int64_t c0 = quarter_begin(V, q);
  int64_t c1 = quarter_begin(V, q + 1);
  const bool geo_ok =
      LP_CHECK(row < T && c1 - shard_c0 <= ld, row < T ? kChkLogitsLoad : kChkRowIndex);
  const int64_t r = geo_ok ? row : 0;
  if (!geo_ok) c1 = c0;
  const float* q0 = logits_shard + r * ld + (c0 - shard_c0);

  const QuarterState st = quarter_state_any(q0, c1 - c0, targets, r, c0, V, tau);
  if (threadIdx.x == 0 && geo_ok && LP_CHECK(row * n_q + ql < T * n_q, kChkStateIndex))
    store_state(&partials[row * n_q + ql], st);
}

// One thread per (row, quarter), four consecutive lanes per row.
__global__ void __launch_bounds__(128)
    lp_merge_partials_kernel(const QuarterState* __restrict__ p0,
                             const QuarterState* __restrict__ p1,
                             const QuarterState* __restrict__ p2,
                             const QuarterState* __restrict__ p3, int n_shards, int64_t T,
                             float* __restrict__ logp, float* __restrict__ entropy,
                             float* __restrict__ lse) {
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x / 4) + (threadIdx.x >> 2);
  const int q = threadIdx.x & 3;
  const QuarterState* shard[4] = {p0, p1, p2, p3};
  const int per = kQuarters / n_shards;
  QuarterState st{neg_inf(), 0.f, 0.f, 0.f, neg_inf(), 1.f, 0.f, 0.f};
  if (row < T &&
      LP_CHECK(q / per < n_shards && row * per + (q % per) < T * per, kChkStateIndex))
    st = load_state(&shard[q / per][row * per + (q % per)]);
  float lp, ent, lz;
  finalise_quad(st, 0xffffffffu, lp, ent, lz);
  if (row < T && q == 0) {
    logp[row] = lp;
    if (entropy != nullptr) entropy[row] = ent;
    if (lse != nullptr) lse[row] = lz;
  }
}

// dL/dz of L = sum_t g_logp[t] logp[t] + g_ent[t] entropy[t] over given
// logits, the logits-path twin of the fused backward's gradient epilogue:
// with zs = z / tau, log p = zs - log Z and p = exp(log p),
//   G = (g_logp (delta(v, y) - p) - g_ent p (log p + entropy)) / tau,
// where a term with p = 0 (a -inf logit, or one far below the maximum) is 0
// and a row whose target is outside [0, V) has no logp term.  log Z and the
// entropy are the forward's (lp_logprob_from_logits_lse).  One CTA per (row,
// kGradChunk columns); whole chunks of 16-byte-aligned rows load four float4
// per thread before computing, the rest goes 4 bytes at a time.  The logits
// may be a vocabulary shard: its V columns are global columns col0 .. col0 +
// V - 1 of a vocabulary of V_total (every element depends only on its own
// logit and the row's log Z and entropy, so shards give the bits of the whole).
constexpr int kGradVec = 4;                          // float4 per thread and chunk
constexpr int64_t kGradChunk = kThreads * 4 * kGradVec;  // 4096 columns

__device__ __forceinline__ float logits_grad(float z, int64_t col, int64_t y, float inv_tau,
                                             float log_z, float ent, float gl, float ge) {
  // col and y: shard-relative (y outside the shard never matches)
  const float zs = inv_tau == 1.f ? z : __fmul_rn(z, inv_tau);
  const float lp = __fsub_rn(zs, log_z);
  const float p = exp_fast(lp);
  float g = p == 0.f ? 0.f : -__fmul_rn(p, __fmaf_rn(ge, __fadd_rn(lp, ent), gl));
  if (col == y) g = __fadd_rn(g, gl);
  return inv_tau == 1.f ? g : __fmul_rn(g, inv_tau);
}

__global__ void __launch_bounds__(kThreads)
    lp_logits_grad_kernel(const float* __restrict__ logits, int64_t ld,
                          const int64_t* __restrict__ targets, int64_t T, int64_t V,
                          int64_t col0, int64_t V_total, int64_t chunks, float inv_tau,
                          const float* __restrict__ lse,
                          const float* __restrict__ entropy, const float* __restrict__ g_logp,
                          const float* __restrict__ g_ent, float* __restrict__ grad,
                          int64_t ld_grad) {
  const int64_t row = blockIdx.x / chunks;
  const int64_t c0 = (blockIdx.x % chunks) * kGradChunk;
  if (!LP_CHECK(row < T && V <= ld && V <= ld_grad, kChkRowIndex)) return;
  const int64_t c1 = min(V, c0 + kGradChunk);
  const int64_t y_global = targets[row];
  const bool y_ok = y_global >= 0 && y_global < V_total;
  const int64_t y = y_global - col0;  // this shard's column of the target
  const float gl = (g_logp != nullptr && y_ok) ? g_logp[row] : 0.f;
  const float ge = g_ent != nullptr ? g_ent[row] : 0.f;
  const float log_z = lse[row];
  const float ent = entropy[row];
  const float* zr = logits + row * ld;
  float* gr = grad + row * ld_grad;
  const int tid = threadIdx.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(zr) | reinterpret_cast<uintptr_t>(gr)) & 15u) == 0;
  if (vec && c1 - c0 == kGradChunk) {
    float4 z[kGradVec];
#pragma unroll
    for (int k = 0; k < kGradVec; ++k) z[k] = load_stream(zr + c0 + 4 * (tid + k * kThreads));
#pragma unroll
    for (int k = 0; k < kGradVec; ++k) {
      const int64_t col = c0 + 4 * (tid + k * kThreads);
      float4 g;
      g.x = logits_grad(z[k].x, col, y, inv_tau, log_z, ent, gl, ge);
      g.y = logits_grad(z[k].y, col + 1, y, inv_tau, log_z, ent, gl, ge);
      g.z = logits_grad(z[k].z, col + 2, y, inv_tau, log_z, ent, gl, ge);
      g.w = logits_grad(z[k].w, col + 3, y, inv_tau, log_z, ent, gl, ge);
      *reinterpret_cast<float4*>(gr + col) = g;
    }
    return;
  }
  for (int64_t col = c0 + tid; col < c1; col += kThreads)
    gr[col] = logits_grad(zr[col], col, y, inv_tau, log_z, ent, gl, ge);
}

}  // namespace

lp_status launch_logits_final(const float* logits, int64_t ld, const int64_t* targets,
                              int64_t T, int64_t V, const TauArgs& tau, float* logp,
                              float* entropy, float* lse, cudaStream_t stream) {
  const int64_t blocks = T * kQuarters;
  lp_logits_final_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
      logits, ld, targets, T, V, tau, logp, entropy, lse);
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

lp_status launch_logits_backward(const float* logits, int64_t ld, const int64_t* targets,
                                 int64_t T, int64_t V, int64_t col0, int64_t V_total,
                                 const TauArgs& tau, const float* lse, const float* entropy,
                                 const float* g_logp, const float* g_ent, float* grad,
                                 int64_t ld_grad, cudaStream_t stream) {
  const int64_t chunks = (V + kGradChunk - 1) / kGradChunk;
  if (T * chunks >= (int64_t(1) << 31)) return LP_ERR_INVALID_ARGUMENT;
  lp_logits_grad_kernel<<<static_cast<unsigned>(T * chunks), kThreads, 0, stream>>>(
      logits, ld, targets, T, V, col0, V_total, chunks, tau.inv_hi, lse, entropy, g_logp, g_ent,
      grad, ld_grad);
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

lp_status launch_logits_partials(const float* logits_shard, int64_t ld,
                                 const int64_t* targets, int64_t T, int64_t V_total,
                                 int q_first, int n_q, const TauArgs& tau, float* partials,
                                 cudaStream_t stream) {
  const int64_t blocks = T * n_q;
  lp_logits_partials_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
      logits_shard, ld, targets, T, V_total, q_first, n_q, tau,
      reinterpret_cast<QuarterState*>(partials));
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

lp_status launch_merge_partials(const float* const* shard_partials, int n_shards, int64_t T,
                                float* logp, float* entropy, float* lse, cudaStream_t stream) {
  const QuarterState* p[4] = {nullptr, nullptr, nullptr, nullptr};
  for (int i = 0; i < n_shards; ++i)
    p[i] = reinterpret_cast<const QuarterState*>(shard_partials[i]);
  const int threads = 128;  // 32 rows per block, one thread per quarter
  const int64_t blocks = (T + threads / 4 - 1) / (threads / 4);
  lp_merge_partials_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      p[0], p[1], p[2], p[3], n_shards, T, logp, entropy, lse);
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

}  // namespace lp

namespace lp {
cudaError_t take_check_word_logits(uint32_t* out) { return take_check_word(out); }
}  // namespace lp
