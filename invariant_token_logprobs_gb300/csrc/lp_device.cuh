// lp_device.cuh: arithmetic shared by every kernel of liblp.
//
// The per-row state of a slice of the vocabulary, for the distribution
// softmax(z / tau), is (m, s, u, t):
//   m  the slice's maximum RAW logit (before the temperature),
//   s  sum over the slice of exp((z - m) / tau),
//   u  sum over the slice of exp((z - m) / tau) * (z - m) / tau,
//   t  the RAW target logit z[y] when y lies in the slice, -inf when it does
//      not, NaN when y is outside [0, V).
// From the states of the four vocabulary quarters the row's results follow:
//   logp    = (t - M) / tau - log S
//   entropy = log S - U / S
// with M the largest m and S, U the quarter sums rebased to M.  This is
// log-sum-exp of the selected-token log-probability of the RL-Kernel logprob
// prior-art report (report.json, "candidates") split into slices; entropy uses
// -sum p log p = log Z - sum p z.  The temperature enters only through the
// differences z - m (exact or nearly so for the terms that matter) and
// (t - M) / tau, which is formed with float pairs (~44 bits): no logit is
// rounded after scaling.
//
// A quarter state leaves a kernel as 8 floats (32 bytes, QuarterState):
// m, s_hi, s_lo, u, t, tau, 0, 0, with s = s_hi + s_lo held as an unevaluated
// float pair so that the sum keeps ~40 bits between kernels.
//
// Every kernel that forms or merges states goes through the functions below,
// so a slice's state has one bit pattern whichever kernel or call produced it.
// The library is compiled with --fmad=false and the arithmetic here uses
// explicit rounding intrinsics: no multiply-add is contracted differently in
// different kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lp {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kQuarters = 4;

__host__ __device__ __forceinline__ int64_t quarter_begin(int64_t V, int q) {
  return (static_cast<int64_t>(q) * V) / kQuarters;
}

// 2^x with the hardware approximation (flushes subnormal results to zero).
__device__ __forceinline__ float exp2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// exp(x) through the hardware 2^x: e^x = 2^(x log2 e).  Used where the
// results feed the bf16-tolerance fused path.
__device__ __forceinline__ float exp_fast(float x) { return exp2_approx(__fmul_rn(x, kLog2e)); }

// max that returns NaN when either operand is NaN.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Three-operand max that returns NaN when any operand is NaN.
__device__ __forceinline__ float fmax3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 1.0f when a >= b, else 0.0f (NaN compares false).
__device__ __forceinline__ float ge_one_zero(float a, float b) {
  float r;
  asm("set.ge.f32.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }

// Chunk c (8 bf16 values, 16 bytes) of a row of d bf16 values starting at row
// (16-byte aligned): read whole when it lies inside the row, value by value
// with zeros past d otherwise, so nothing past the row's d values is read.
__device__ __forceinline__ uint4 load_row_chunk(const uint16_t* __restrict__ row, int64_t d,
                                                int64_t c) {
  if (c * 8 + 8 <= d) return *reinterpret_cast<const uint4*>(row + c * 8);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t k = c * 8 + 2 * i;
    const uint32_t lo = k < d ? row[k] : 0u;
    const uint32_t hi = k + 1 < d ? row[k + 1] : 0u;
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ float quiet_nan() { return __int_as_float(0x7fffffffu); }

// ------------------------------------------------------------ packed f32 pairs
// Two floats in one 64-bit register, for the f32x2 arithmetic of sm_100+.

__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// ------------------------------------------------- exp for arguments x <= 0
//
// e^x by Cody and Waite's argument reduction and a polynomial (the textbook
// method, e.g. J.-M. Muller, "Elementary Functions", ch. 11):
//   n = round(x log2 e), r = x - n ln2 with ln2 = L1 + L2 split so that n L1
//   is exact (L1 has 16 significant bits), |r| <= ln2 / 2, e^x = p(r) 2^n.
// p(r) = 1 + r + r^2 (c2 + c3 r + ... + c6 r^4) is the minimax approximation
// of e^r on [-ln2/2, ln2/2] in relative error with the first two coefficients
// held at exactly 1 (so p(0) = 1: the maximal term of a sum is exactly 1),
// computed with the Remez exchange algorithm: relative error 3.1e-9 before
// float32 rounding.  The rounding to an integer uses the float addition of
// 1.5 * 2^23 (+127, the exponent bias): the sum's low mantissa bits are then
// n + 127, which shifted into the exponent field give 2^n directly.
// Arguments are clamped to [-87, 0] first (2^n stays a normal float); below
// -87 the result, ~1e-38, is negligible against the maximal term 1 of every
// sum it enters.  NaN stays NaN.  With float32 fma Horner steps the relative
// error is at most ~0.55 ulp and unbiased (mean ~2e-10); the hardware 2^x, by
// comparison, measured -5e-8 (-0.4 ulp) biased on this GPU for |x| > 1.  Used
// for every rescaling of a sum (raised maxima, rebases to a common maximum).
constexpr float kExpClampLo = -87.0f;
constexpr float kExpMagic = 12583039.0f;     // 1.5 * 2^23 + 127
constexpr float kLn2Hi = 0.693145751953125f;
constexpr float kLn2Lo = 1.42860677e-06f;
constexpr float kP2 = 0.49999993451708435f, kP3 = 0.1666652068983302f,
                kP4 = 0.04166838736126115f, kP5 = 0.008368709824171195f,
                kP6 = 0.0013814613260779772f;

__device__ __forceinline__ float exp_neg(float x) {
  const float xc = fmax_nan(x, kExpClampLo);
  const float t = __fmaf_rn(xc, kLog2e, kExpMagic);
  const float n = __fsub_rn(t, kExpMagic);
  float r = __fmaf_rn(n, -kLn2Hi, xc);
  r = __fmaf_rn(n, -kLn2Lo, r);
  float p = __fmaf_rn(kP6, r, kP5);
  p = __fmaf_rn(p, r, kP4);
  p = __fmaf_rn(p, r, kP3);
  p = __fmaf_rn(p, r, kP2);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  return __fmul_rn(p, __int_as_float(__float_as_int(t) << 23));
}

// -------------------------------------------------- float pairs (hi + lo)

// Error-free sum: hi + lo == a + b exactly, hi = fl(a + b) (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float& hi, float& lo) {
  hi = __fadd_rn(a, b);
  const float bb = __fsub_rn(hi, a);
  lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, bb)), __fsub_rn(b, bb));
}

// (a_hi + a_lo) + (b_hi + b_lo) as a normalised pair.
__device__ __forceinline__ void add_pair(float a_hi, float a_lo, float b_hi, float b_lo,
                                         float& hi, float& lo) {
  float s, e;
  two_sum(a_hi, b_hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a_lo, b_lo));
  hi = __fadd_rn(s, e);
  lo = __fsub_rn(e, __fsub_rn(hi, s));
}

// a * (x_hi + x_lo) as a pair (the product's rounding error kept by an fma).
__device__ __forceinline__ void mul_pair(float a, float x_hi, float x_lo, float& hi, float& lo) {
  const float p = __fmul_rn(a, x_hi);
  const float e = __fmaf_rn(a, x_hi, -p);
  const float l = __fmaf_rn(a, x_lo, e);
  hi = __fadd_rn(p, l);
  lo = __fsub_rn(l, __fsub_rn(hi, p));
}

// d / tau for a difference d <= 0 of raw logits: d * (1/tau) with 1/tau given
// as a float pair inv_hi + inv_lo, so that no rounding of 1/tau biases every
// term the same way.  With inv_hi == 1, inv_lo == 0 this is d itself.
__device__ __forceinline__ float scale_diff(float d, float inv_hi, float inv_lo) {
  return __fmaf_rn(d, inv_lo, __fmul_rn(d, inv_hi));
}

// -------------------------------------------------------------- states

struct QuarterState {
  float m, s_hi, s_lo, u, t, tau, r0, r1;
};
static_assert(sizeof(QuarterState) == 32, "quarter states are 32 bytes");

__device__ __forceinline__ void store_state(QuarterState* dst, const QuarterState& q) {
  float4* p = reinterpret_cast<float4*>(dst);
  p[0] = make_float4(q.m, q.s_hi, q.s_lo, q.u);
  p[1] = make_float4(q.t, q.tau, 0.f, 0.f);
}

__device__ __forceinline__ QuarterState load_state(const QuarterState* src) {
  const float4* p = reinterpret_cast<const float4*>(src);
  const float4 a = p[0], b = p[1];
  return QuarterState{a.x, a.y, a.z, a.w, b.x, b.y, 0.f, 0.f};
}

// Online state of one thread over a sequence of logits of the fused path
// (bf16 tolerance): s includes the maximal term.
struct Online {
  float m, s, u;
  __device__ __forceinline__ void reset() {
    m = neg_inf();
    s = 0.f;
    u = 0.f;
  }
  // Raise the running maximum to bm (a maximum over the next values, computed
  // with fmax_nan).  NaN in bm makes the state NaN from here on.
  __device__ __forceinline__ void raise_to(float bm, float inv_tau) {
    if (!(bm <= m)) {
      if (m == neg_inf()) {
        s = 0.f;
        u = 0.f;
      } else {
        const float delta = __fmul_rn(__fsub_rn(m, bm), inv_tau);  // < 0
        if (delta < kExpClampLo) {  // the old terms vanish (delta may be -inf); NaN goes on
          s = 0.f;
          u = 0.f;
        } else {
          const float a = exp_fast(delta);
          u = __fmul_rn(a, __fmaf_rn(delta, s, u));
          s = __fmul_rn(a, s);
        }
      }
      m = bm;
    }
  }
  __device__ __forceinline__ bool active() const { return m != neg_inf(); }
};

// One logit's terms relative to the running maximum m on the fused path:
// d = (x - m) / tau clamped so that e * d is 0 for a -inf logit (never
// 0 * inf) while NaN stays NaN, and e = exp(d).
__device__ __forceinline__ void term(float x, float m, float inv_tau, float& e, float& d) {
  d = fmax_nan(__fmul_rn(__fsub_rn(x, m), inv_tau), -3.402823466e38f);
  e = exp_fast(d);
}

// ------------------------------------------------ float-pair exp and log
//
// Values held as an unevaluated pair hi + lo of floats (|lo| <= ulp(hi) / 2),
// about 44 significant bits, for the once-per-row finalisation.  Float64
// transcendentals are slow on this GPU; these use only float operations.

struct F2 {
  float hi, lo;
};

__device__ __forceinline__ F2 f2_norm(float hi, float lo) {  // |hi| >= |lo|
  const float s = __fadd_rn(hi, lo);
  return F2{s, __fsub_rn(lo, __fsub_rn(s, hi))};
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  return f2_norm(s, __fadd_rn(e, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
  const float p = __fmul_rn(a.hi, b.hi);
  const float e = __fmaf_rn(a.hi, b.hi, -p);
  return f2_norm(p, __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, e)));
}

// e^x for x = x.hi + x.lo with -87 <= x.hi <= 0: n = round(x log2 e),
// r = x - n ln2 (ln2 split in three, n L1 exact), e^r = 1 + r + r^2 P(r) with
// P(r) = 1/2 + r (1/3! + r/4! + ... + r^6/9!) (Taylor, truncation < 1e-11 for
// |r| <= ln2/2), the leading terms carried as pairs; e^x = e^r 2^n.
// Relative error about 1e-10.
constexpr float kLn2A = 0.693145751953125f;       // 16 significant bits
constexpr float kLn2B = 1.4286068203094172e-06f;  // next 24 bits
constexpr float kLn2C = 5.497923e-14f;            // remainder (ln2 - A - B)
__device__ __forceinline__ F2 exp_f2(F2 x) {
  const float t = __fmaf_rn(x.hi, kLog2e, kExpMagic);
  const float n = __fsub_rn(t, kExpMagic);
  const float r1 = __fmaf_rn(n, -kLn2A, x.hi);  // exact
  const float pb = __fmul_rn(n, kLn2B);
  const float pbe = __fmaf_rn(n, kLn2B, -pb);
  F2 r;
  two_sum(r1, -pb, r.hi, r.lo);
  r = f2_norm(r.hi, __fadd_rn(r.lo, __fsub_rn(x.lo, __fmaf_rn(n, kLn2C, pbe))));
  float q = 1.0f / 362880.0f;  // 1/9!
  q = __fmaf_rn(q, r.hi, 1.0f / 40320.0f);
  q = __fmaf_rn(q, r.hi, 1.0f / 5040.0f);
  q = __fmaf_rn(q, r.hi, 1.0f / 720.0f);
  q = __fmaf_rn(q, r.hi, 1.0f / 120.0f);
  q = __fmaf_rn(q, r.hi, 1.0f / 24.0f);
  q = __fmaf_rn(q, r.hi, 1.0f / 6.0f);
  F2 P;
  two_sum(0.5f, __fmul_rn(r.hi, q), P.hi, P.lo);
  P.lo = __fadd_rn(P.lo, __fmaf_rn(r.hi, q, -__fmul_rn(r.hi, q)));
  F2 r2;  // r^2 including 2 r.hi r.lo
  r2.hi = __fmul_rn(r.hi, r.hi);
  r2.lo = __fmaf_rn(r.hi, r.hi, -r2.hi);
  r2.lo = __fmaf_rn(__fmul_rn(2.0f, r.hi), r.lo, r2.lo);
  const F2 tail = f2_mul(r2, P);
  F2 e = f2_add(F2{1.0f, 0.0f}, r);
  e = f2_add(e, tail);
  const float scale = __int_as_float(__float_as_int(t) << 23);  // 2^n
  return F2{__fmul_rn(e.hi, scale), __fmul_rn(e.lo, scale)};
}

// log S for S = S.hi + S.lo >= 1 (finite): y = logf(S.hi) (CUDA's logf), then
// one Newton step on e^y = S in pairs, log S = y + (S e^-y - 1) (the next
// term, -(S e^-y - 1)^2 / 2, is below 1e-14).  Absolute error about 1e-10.
__device__ __forceinline__ F2 log_f2(F2 S) {
  const float y = logf(S.hi);
  const F2 E = exp_f2(F2{-y, 0.0f});
  const F2 w = f2_add(f2_mul(S, E), F2{-1.0f, 0.0f});
  return f2_add(F2{y, 0.0f}, w);
}

// ------------------------------------------------------------- finalise
//
// The four quarter states of a row sit in four consecutive lanes of a warp
// (lane & 3 == quarter); `mask` names every lane taking part (groups of four).
// Each lane rebases its quarter to the row maximum with float pairs,
//   delta_q = (m_q - M) / tau,  a_q = exp(delta_q),  S_q = a_q (s_hi + s_lo),
//   U_q = a_q (u + delta_q (s_hi + s_lo)),
// and the sums are formed as (Q0 + Q1) + (Q2 + Q3) with two xor-shuffles
// (pair addition is commutative, so every lane of the group holds the same
// bits).  Every lane then has the row's logp = (t - M) / tau - log S, entropy
// = log S - U / S and log Z = M / tau + log S, each rounded to float once.
// States of different temperatures, NaN anywhere, or no finite logit give NaN.
__device__ __forceinline__ void finalise_quad(const QuarterState& q, unsigned mask, float& logp,
                                              float& entropy, float& log_z) {
  float M = q.m;
  M = fmax_nan(M, __shfl_xor_sync(mask, M, 1));
  M = fmax_nan(M, __shfl_xor_sync(mask, M, 2));
  float t = q.t;
  t = fmax_nan(t, __shfl_xor_sync(mask, t, 1));
  t = fmax_nan(t, __shfl_xor_sync(mask, t, 2));
  int same_tau = q.tau == __shfl_xor_sync(mask, q.tau, 1);
  same_tau &= q.tau == __shfl_xor_sync(mask, q.tau, 2);
  same_tau &= __shfl_xor_sync(mask, same_tau, 1);
  same_tau &= __shfl_xor_sync(mask, same_tau, 2);

  // 1/tau as a pair (tau == 1: exactly 1, 0)
  const float inv_hi = __frcp_rn(q.tau);
  const float inv_lo = __fdiv_rn(__fmaf_rn(-inv_hi, q.tau, 1.0f), q.tau);
  const F2 inv{inv_hi, inv_lo};

  F2 S{0.0f, 0.0f};
  float U = 0.0f;
  if (q.m != neg_inf() && M == M) {
    F2 d;
    two_sum(q.m, -M, d.hi, d.lo);  // exact
    // a quarter more than 87 below the row maximum after scaling adds nothing
    // (the scaled difference may even overflow); NaN goes on
    if (!(__fmul_rn(d.hi, inv_hi) < kExpClampLo)) {
      d = f2_mul(d, inv);
      const F2 a = exp_f2(d);
      S = f2_mul(a, F2{q.s_hi, q.s_lo});
      U = __fmul_rn(a.hi, __fmaf_rn(d.hi, q.s_hi, q.u));
    }
  }
  F2 o;
  o.hi = __shfl_xor_sync(mask, S.hi, 1);
  o.lo = __shfl_xor_sync(mask, S.lo, 1);
  S = f2_add(S, o);
  U = __fadd_rn(U, __shfl_xor_sync(mask, U, 1));
  o.hi = __shfl_xor_sync(mask, S.hi, 2);
  o.lo = __shfl_xor_sync(mask, S.lo, 2);
  S = f2_add(S, o);
  U = __fadd_rn(U, __shfl_xor_sync(mask, U, 2));

  if (!same_tau || !(M > neg_inf()) || !(S.hi > 0.0f) || U != U || S.hi != S.hi ||
      S.hi > 3.402823466e38f) {  // NaN somewhere, or empty
    logp = quiet_nan();
    entropy = quiet_nan();
    log_z = quiet_nan();
    return;
  }
  const F2 log_s = log_f2(S);
  F2 tm;
  two_sum(t, -M, tm.hi, tm.lo);
  const F2 lp = f2_add(f2_mul(tm, inv), F2{-log_s.hi, -log_s.lo});
  logp = t == neg_inf() ? neg_inf() : t != t ? quiet_nan() : __fadd_rn(lp.hi, lp.lo);
  entropy = __fadd_rn(log_s.hi, __fsub_rn(log_s.lo, __fdiv_rn(U, S.hi)));
  const F2 lz = f2_add(f2_mul(F2{M, 0.0f}, inv), log_s);
  log_z = __fadd_rn(lz.hi, lz.lo);
}

}  // namespace lp
