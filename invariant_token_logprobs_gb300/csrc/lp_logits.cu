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
// load.  A thread keeps an online (max, sum-exp, sum-exp*(z-max)) state,
// raising its maximum once per batch of 32 values, and sums each batch in four
// column-lane accumulators before adding it to the state.  The 256 thread
// states are rebased to the CTA maximum and summed in a fixed tree (warp
// shuffles, then 8 warp partials in a fixed pairing).  Which thread owns which
// column depends only on the column's offset inside its quarter, so a row's
// quarter state is the same whatever the row's position, batch or shard.
//
// Finalising variant: the 4 CTAs of a row form a thread-block cluster; each
// writes its quarter state into the shared memory of cluster rank 0 (DSMEM),
// and after the cluster barrier rank 0 merges (Q0 + Q1) + (Q2 + Q3).  Partials
// variant: each CTA writes its quarter state to global memory for
// lp_merge_partials.
//
// Temperature: with inv_tau != 1 every logit is first multiplied by inv_tau
// (fl(z * fl(1/tau))); with inv_tau == 1 the results are exactly those of the
// unscaled computation.
#include <cuda_runtime.h>

#include "lp_device.cuh"
#include "lp_internal.h"

namespace lp {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBatch = 8;  // 4-float groups per thread per batch

__device__ __forceinline__ float4 load_stream(const float* p) {
  float4 v;
  asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(p));
  return v;
}

// Group g (columns 4g .. 4g+3 of the quarter); columns >= w read as -inf.
__device__ __forceinline__ void load_group(const float* __restrict__ q0, int64_t w, int64_t g,
                                           bool vec, float (&v)[4]) {
  const int64_t c = g * 4;
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

// State (M, S, U) of the w columns starting at q0, each logit multiplied by
// inv_tau first when kScaled; valid in thread 0.
template <bool kScaled>
__device__ __forceinline__ void quarter_state(const float* __restrict__ q0, int64_t w,
                                              float inv_tau, float& M_out, float& S_out,
                                              float& U_out) {
  __shared__ float red_m[kWarps], red_s[kWarps], red_u[kWarps];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const bool vec = (reinterpret_cast<uintptr_t>(q0) & 15u) == 0;
  const int64_t n_groups = (w + 3) / 4;

  Online st;
  st.reset();
  for (int64_t g0 = 0; g0 < n_groups; g0 += int64_t(kThreads) * kBatch) {
    float v[kBatch][4];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) load_group(q0, w, g0 + k * kThreads + tid, vec, v[k]);
    if (kScaled) {
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) v[k][i] = __fmul_rn(v[k][i], inv_tau);
    }
    float bm = v[0][0];
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
#pragma unroll
      for (int i = 0; i < 4; ++i) bm = fmax_nan(bm, v[k][i]);
    st.raise_to(bm);
    if (st.active()) {
      float sa[4] = {0.f, 0.f, 0.f, 0.f};
      float ua[4] = {0.f, 0.f, 0.f, 0.f};
      // e = 2^(x log2e - m log2e): one fma and one ex2.approx.ftz per logit;
      // d = x - m clamped so that a -inf logit adds e * d = 0, NaN stays NaN
      const float mL = __fmul_rn(st.m, kLog2e);
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float d = fmax_nan(__fsub_rn(v[k][i], st.m), -3.402823466e38f);
          const float e = exp2_approx(__fmaf_rn(v[k][i], kLog2e, -mL));
          sa[i] = __fadd_rn(sa[i], e);
          ua[i] = __fmaf_rn(e, d, ua[i]);
        }
      st.s = __fadd_rn(st.s, __fadd_rn(__fadd_rn(sa[0], sa[1]), __fadd_rn(sa[2], sa[3])));
      st.u = __fadd_rn(st.u, __fadd_rn(__fadd_rn(ua[0], ua[1]), __fadd_rn(ua[2], ua[3])));
    }
  }

  // CTA maximum (order-free), then rebase and fixed-tree sums.
  float m = st.m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) red_m[warp] = m;
  __syncthreads();
  float M = red_m[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) M = fmaxf(M, red_m[i]);

  float s, u;
  if (M == neg_inf()) {
    s = 0.f;
    u = 0.f;
  } else {
    rebase(st.m, st.s, st.u, M, s, u);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    s = __fadd_rn(s, __shfl_down_sync(0xffffffffu, s, off));
    u = __fadd_rn(u, __shfl_down_sync(0xffffffffu, u, off));
  }
  if (lane == 0) {
    red_s[warp] = s;
    red_u[warp] = u;
  }
  __syncthreads();
  if (tid == 0) {
    static_assert(kWarps == 8, "fixed pairing below assumes 8 warps");
    S_out = __fadd_rn(__fadd_rn(__fadd_rn(red_s[0], red_s[1]), __fadd_rn(red_s[2], red_s[3])),
                      __fadd_rn(__fadd_rn(red_s[4], red_s[5]), __fadd_rn(red_s[6], red_s[7])));
    U_out = __fadd_rn(__fadd_rn(__fadd_rn(red_u[0], red_u[1]), __fadd_rn(red_u[2], red_u[3])),
                      __fadd_rn(__fadd_rn(red_u[4], red_u[5]), __fadd_rn(red_u[6], red_u[7])));
    M_out = M;
  }
}

// Target logit of a quarter: z[y] * inv_tau if y is in [c0, c1), -inf if y is
// another valid column, NaN if y is outside [0, V).
__device__ __forceinline__ float quarter_target(const float* __restrict__ q0, int64_t y,
                                                int64_t c0, int64_t c1, int64_t V,
                                                float inv_tau) {
  if (y < 0 || y >= V) return quiet_nan();
  if (y >= c0 && y < c1) return __fmul_rn(__ldg(q0 + (y - c0)), inv_tau);
  return neg_inf();
}

__device__ __forceinline__ void quarter_state_any(const float* __restrict__ q0, int64_t w,
                                                  float inv_tau, float& M, float& S, float& U) {
  if (inv_tau == 1.f)
    quarter_state<false>(q0, w, inv_tau, M, S, U);
  else
    quarter_state<true>(q0, w, inv_tau, M, S, U);
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads)
    lp_logits_final_kernel(const float* __restrict__ logits, int64_t ld,
                           const int64_t* __restrict__ targets, int64_t V, float inv_tau,
                           float* __restrict__ logp, float* __restrict__ entropy) {
  __shared__ float4 qstates[kQuarters];
  const int q = blockIdx.x & 3;
  const int64_t row = blockIdx.x >> 2;
  const int64_t c0 = quarter_begin(V, q);
  const int64_t c1 = quarter_begin(V, q + 1);
  const float* q0 = logits + row * ld + c0;

  float M, S, U;
  quarter_state_any(q0, c1 - c0, inv_tau, M, S, U);
  if (threadIdx.x == 0) {
    const float t = quarter_target(q0, targets[row], c0, c1, V, inv_tau);
    const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(&qstates[q]));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(0));
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(M),
                 "f"(S), "f"(U), "f"(t)
                 : "memory");
  }
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (q == 0 && threadIdx.x == 0) {
    const float4 qs[kQuarters] = {qstates[0], qstates[1], qstates[2], qstates[3]};
    float lp, ent;
    finalise(qs, lp, ent);
    logp[row] = lp;
    if (entropy != nullptr) entropy[row] = ent;
  }
}

__global__ void __launch_bounds__(kThreads)
    lp_logits_partials_kernel(const float* __restrict__ logits_shard, int64_t ld,
                              const int64_t* __restrict__ targets, int64_t V, int q_first,
                              int n_q, float inv_tau, float4* __restrict__ partials) {
  const int ql = blockIdx.x % n_q;
  const int64_t row = blockIdx.x / n_q;
  const int q = q_first + ql;
  const int64_t shard_c0 = quarter_begin(V, q_first);
  const int64_t c0 = quarter_begin(V, q);
  const int64_t c1 = quarter_begin(V, q + 1);
  const float* q0 = logits_shard + row * ld + (c0 - shard_c0);

  float M, S, U;
  quarter_state_any(q0, c1 - c0, inv_tau, M, S, U);
  if (threadIdx.x == 0) {
    const float t = quarter_target(q0, targets[row], c0, c1, V, inv_tau);
    partials[row * n_q + ql] = make_float4(M, S, U, t);
  }
}

__global__ void lp_merge_partials_kernel(const float4* __restrict__ p0,
                                         const float4* __restrict__ p1,
                                         const float4* __restrict__ p2,
                                         const float4* __restrict__ p3, int n_shards,
                                         int64_t T, float* __restrict__ logp,
                                         float* __restrict__ entropy) {
  const int64_t row = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= T) return;
  const float4* shard[4] = {p0, p1, p2, p3};
  const int per = kQuarters / n_shards;
  float4 qs[kQuarters];
#pragma unroll
  for (int q = 0; q < kQuarters; ++q) qs[q] = shard[q / per][row * per + (q % per)];
  float lp, ent;
  finalise(qs, lp, ent);
  logp[row] = lp;
  if (entropy != nullptr) entropy[row] = ent;
}

}  // namespace

lp_status launch_logits_final(const float* logits, int64_t ld, const int64_t* targets,
                              int64_t T, int64_t V, float inv_tau, float* logp, float* entropy,
                              cudaStream_t stream) {
  const int64_t blocks = T * kQuarters;
  lp_logits_final_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
      logits, ld, targets, V, inv_tau, logp, entropy);
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

lp_status launch_logits_partials(const float* logits_shard, int64_t ld,
                                 const int64_t* targets, int64_t T, int64_t V_total,
                                 int q_first, int n_q, float inv_tau, float* partials,
                                 cudaStream_t stream) {
  const int64_t blocks = T * n_q;
  lp_logits_partials_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
      logits_shard, ld, targets, V_total, q_first, n_q, inv_tau,
      reinterpret_cast<float4*>(partials));
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

lp_status launch_merge_partials(const float* const* shard_partials, int n_shards, int64_t T,
                                float* logp, float* entropy, cudaStream_t stream) {
  const float4* p[4] = {nullptr, nullptr, nullptr, nullptr};
  for (int i = 0; i < n_shards; ++i) p[i] = reinterpret_cast<const float4*>(shard_partials[i]);
  const int threads = 128;
  const int64_t blocks = (T + threads - 1) / threads;
  lp_merge_partials_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      p[0], p[1], p[2], p[3], n_shards, T, logp, entropy);
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

}  // namespace lp
