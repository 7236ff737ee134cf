// lp_device.cuh: arithmetic shared by every kernel of liblp.
//
// The per-row state of a slice of the vocabulary is (m, s, u, t):
//   m  the slice's maximum logit,
//   s  sum over the slice of exp(z - m),
//   u  sum over the slice of exp(z - m) * (z - m),
//   t  the target logit z[y] when y lies in the slice, -inf when it does not,
//      NaN when y is outside [0, V).
// From the states of the four vocabulary quarters the row's results follow:
//   logp    = (t - M) - log S
//   entropy = log S - U / S
// with M the largest m and S, U the quarter sums rebased to M.  This is
// log-sum-exp of the selected-token log-probability of the RL-Kernel logprob
// prior-art report (report.json, "candidates") split into slices; entropy uses
// -sum p log p = log Z - sum p z.
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
constexpr double kLn2 = 0.6931471805599453;
constexpr int kQuarters = 4;

__host__ __device__ __forceinline__ int64_t quarter_begin(int64_t V, int q) {
  return (static_cast<int64_t>(q) * V) / kQuarters;
}

// exp(x) as exp2(x * log2 e) with CUDA's exp2f.
__device__ __forceinline__ float exp_f(float x) { return exp2f(__fmul_rn(x, kLog2e)); }

// 2^x with the hardware approximation (flushes subnormal results to zero).
__device__ __forceinline__ float exp2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// max that returns NaN when either operand is NaN.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

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

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }
__device__ __forceinline__ float quiet_nan() { return __int_as_float(0x7fffffffu); }

// Online state of one thread over a sequence of logits.
struct Online {
  float m, s, u;
  __device__ __forceinline__ void reset() {
    m = neg_inf();
    s = 0.f;
    u = 0.f;
  }
  // Raise the running maximum to bm (a maximum over the next values, computed
  // with fmax_nan).  NaN in bm makes the state NaN from here on.
  __device__ __forceinline__ void raise_to(float bm) {
    if (!(bm <= m)) {
      if (m == neg_inf()) {
        s = 0.f;
        u = 0.f;
      } else {
        const float delta = __fsub_rn(m, bm);  // < 0
        const float a = exp_f(delta);
        u = __fmul_rn(a, __fmaf_rn(delta, s, u));
        s = __fmul_rn(a, s);
      }
      m = bm;
    }
  }
  __device__ __forceinline__ bool active() const { return m != neg_inf(); }
};

// One logit's terms relative to the running maximum m: e = exp(x - m) and the
// clamped difference d = x - m, so that e * d is 0 for a -inf logit (never
// 0 * inf) while NaN stays NaN.
__device__ __forceinline__ void term(float x, float m, float& e, float& d) {
  d = fmax_nan(__fsub_rn(x, m), -3.402823466e38f);
  e = exp_f(d);
}

// Rebase (m, s, u) to a common maximum M >= m: returns (s', u') with
// s' = e^(m-M) s and u' = e^(m-M) (u + (m - M) s).  An empty state (m = -inf)
// contributes nothing.
__device__ __forceinline__ void rebase(float m, float s, float u, float M, float& s_out,
                                       float& u_out) {
  if (m == neg_inf()) {
    s_out = 0.f;
    u_out = 0.f;
    return;
  }
  const float delta = __fsub_rn(m, M);
  const float a = exp_f(delta);
  s_out = __fmul_rn(a, s);
  u_out = __fmul_rn(a, __fmaf_rn(delta, s, u));
}

// exp(delta) for delta <= 0 given exactly in double, through float: the
// relative error is that of rounding delta to float plus CUDA's expf, a few
// times 1e-7 for the terms that matter (|delta| of order 1); terms with large
// |delta| are negligible in the sums they enter.  Double-precision
// transcendentals are slow on this GPU and the four quarters need only this.
__device__ __forceinline__ double exp_nonpos(double delta) {
  return static_cast<double>(expf(static_cast<float>(delta)));
}

// log(S) for finite S > 0: with S = m 2^e, m in [0.5, 1) (frexp),
// log S = log m + e ln 2, log m taken with CUDA's logf (|log m| < 0.7, so its
// absolute error is about 1e-7) and the rest in double.  log S itself can be
// ~12 or more, where a float would carry an error of ~1e-6.
__device__ __forceinline__ double log_pos(double S) {
  int e;
  const double m = frexp(S, &e);
  return __dadd_rn(static_cast<double>(logf(static_cast<float>(m))),
                   __dmul_rn(static_cast<double>(e), kLn2));
}

// Final merge of the four quarter states, fixed order (Q0 + Q1) + (Q2 + Q3),
// in float64 (the exponentials and the logarithm through float, above), and
// the row's results.
__device__ __forceinline__ void finalise(const float4 (&q)[kQuarters], float& logp,
                                         float& entropy) {
  const float M = fmaxf(fmaxf(q[0].x, q[1].x), fmaxf(q[2].x, q[3].x));
  double S_q[kQuarters], U_q[kQuarters];
#pragma unroll
  for (int i = 0; i < kQuarters; ++i) {
    if (q[i].x == neg_inf()) {
      S_q[i] = 0.0;
      U_q[i] = 0.0;
    } else {
      const double delta = __dsub_rn(static_cast<double>(q[i].x), static_cast<double>(M));
      const double a = exp_nonpos(delta);
      S_q[i] = __dmul_rn(a, static_cast<double>(q[i].y));
      U_q[i] = __dmul_rn(a, __fma_rn(delta, static_cast<double>(q[i].y),
                                     static_cast<double>(q[i].z)));
    }
  }
  const double S = __dadd_rn(__dadd_rn(S_q[0], S_q[1]), __dadd_rn(S_q[2], S_q[3]));
  const double U = __dadd_rn(__dadd_rn(U_q[0], U_q[1]), __dadd_rn(U_q[2], U_q[3]));
  const float t = fmax_nan(fmax_nan(q[0].w, q[1].w), fmax_nan(q[2].w, q[3].w));
  if (!(M > neg_inf()) || !(S > 0.0)) {  // no distribution, or NaN somewhere
    logp = quiet_nan();
    entropy = quiet_nan();
    return;
  }
  const double log_s = log_pos(S);
  logp = __double2float_rn(
      __dsub_rn(__dsub_rn(static_cast<double>(t), static_cast<double>(M)), log_s));
  entropy = __double2float_rn(__dsub_rn(log_s, __ddiv_rn(U, S)));
}

}  // namespace lp
