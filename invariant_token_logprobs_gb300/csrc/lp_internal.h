// lp_internal.h: launchers shared between the C-ABI front end (lp_api.cu) and
// the kernel translation units.  Arguments reaching these functions have
// already been validated by the front end.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/lp.h"

namespace lp {

// Header at the start of every fused-path workspace.
constexpr size_t kWorkspaceHeader = 256;
// Vocabulary tile width of the fused path (columns of z per tensor-memory tile).
constexpr int kTileN = 256;

// Error bits of the workspace error word.
constexpr uint32_t kErrLoader = 1u;
constexpr uint32_t kErrMma = 2u;
constexpr uint32_t kErrEpilogue = 4u;

// Quarter range [q_first, q_first + n_q) of shard `shard_index` of `n_shards`.
inline void shard_quarters(int shard_index, int n_shards, int& q_first, int& n_q) {
  n_q = 4 / n_shards;
  q_first = shard_index * n_q;
}

// Tiles of kTileN columns per quarter; the same for every quarter (a quarter
// one column narrower than the widest gets a masked tail).
inline int64_t tiles_per_quarter(int64_t V) {
  const int64_t wmax = (V + 3) / 4;
  return (wmax + kTileN - 1) / kTileN;
}

struct Device {
  int ordinal;
  int sm_count;
  uint64_t ctx_id;  // current_context_id() at the time of the call
};
lp_status current_device(Device* dev);  // checks compute capability 10.3

// Identifier of the CUDA context current on the calling thread, 0 when none is
// current or it cannot be read.  Identifiers are unique for the life of the
// process: the primary context re-created after cudaDeviceReset, or a context
// the caller created with the driver API, gets a new one.
uint64_t current_context_id();

// Runs a setter once per CUDA context.  Function attributes (the dynamic
// shared-memory limit of a kernel) and device addresses of module variables
// belong to the module as loaded into one context, so they are set or looked
// up again whenever the calling thread's context is one not seen before.
// A context id of 0 (unknown) runs the setter every time.
class PerContextOnce {
 public:
  template <class F>
  cudaError_t run(uint64_t ctx_id, F&& set) {
    std::lock_guard<std::mutex> lock(mu_);
    if (ctx_id != 0)
      for (int i = 0; i < kSlots; ++i)
        if (ids_[i] == ctx_id) return cudaSuccess;
    const cudaError_t e = set();
    if (e == cudaSuccess && ctx_id != 0) {
      ids_[next_] = ctx_id;
      next_ = (next_ + 1) % kSlots;
    }
    return e;
  }

 private:
  static constexpr int kSlots = 16;
  std::mutex mu_;
  uint64_t ids_[kSlots] = {};
  int next_ = 0;
};

// Temperature of a call: tau itself (stored in every quarter state) and 1/tau
// as a float pair inv_hi + inv_lo (inv_hi = fl(1/tau), inv_lo the rest); tau
// == 1 gives (1, 1, 0), for which the kernels skip every multiplication.
struct TauArgs {
  float tau;
  float inv_hi;
  float inv_lo;
};

// logits path
lp_status launch_logits_final(const float* logits, int64_t ld, const int64_t* targets,
                              int64_t T, int64_t V, const TauArgs& tau, float* logp,
                              float* entropy, float* lse, cudaStream_t stream);
// the logits' V columns are global columns col0 .. col0 + V - 1 of V_total
lp_status launch_logits_backward(const float* logits, int64_t ld, const int64_t* targets,
                                 int64_t T, int64_t V, int64_t col0, int64_t V_total,
                                 const TauArgs& tau, const float* lse, const float* entropy,
                                 const float* g_logp, const float* g_ent, float* grad,
                                 int64_t ld_grad, cudaStream_t stream);
lp_status launch_logits_partials(const float* logits_shard, int64_t ld,
                                 const int64_t* targets, int64_t T, int64_t V_total,
                                 int q_first, int n_q, const TauArgs& tau, float* partials,
                                 cudaStream_t stream);
lp_status launch_merge_partials(const float* const* shard_partials, int n_shards, int64_t T,
                                float* logp, float* entropy, float* lse, cudaStream_t stream);

// fused path
size_t linear_workspace_bytes(int64_t T, int64_t d, int64_t V_total, int n_q);
lp_status launch_linear(const Device& dev, const void* H, int64_t ld_h, const void* W,
                        int64_t ld_w, const int64_t* targets, int64_t T, int64_t d,
                        int64_t V_total, int q_first, int n_q, const TauArgs& tau, float* logp,
                        float* entropy, float* partials_out, void* workspace,
                        cudaStream_t stream);

// fixed device scratch of the no-alloc fused call: its device address in the
// calling thread's current context
size_t static_scratch_bytes();
lp_status static_scratch(void** out);

// As launch_linear, and when `lse` is not NULL also writes per row the
// log-sum-exp log Z of the (tempered) logits.
lp_status launch_linear_stats(const Device& dev, const void* H, int64_t ld_h, const void* W,
                              int64_t ld_w, const int64_t* targets, int64_t T, int64_t d,
                              int64_t V_total, int q_first, int n_q, const TauArgs& tau,
                              float* logp,
                              float* entropy, float* partials_out, float* lse,
                              void* workspace, cudaStream_t stream);

// backward of the fused path over the quarters [q_first, q_first + n_q) of a
// vocabulary of V_total (V = their columns = W's rows; all four: the whole
// vocabulary); a shard's grad_h is its partial dH (the subtree sum of its
// quarters), merged by launch_merge_grad_h
size_t linear_backward_workspace_bytes(int64_t T, int64_t d, int64_t V, int64_t V_total);
lp_status launch_linear_backward(const Device& dev, const void* H, int64_t ld_h, const void* W,
                                 int64_t ld_w, const int64_t* targets, int64_t T, int64_t d,
                                 int64_t V, int64_t V_total, int q_first, int n_q,
                                 const TauArgs& tau, const float* saved_lse,
                                 const float* saved_entropy, const float* g_logp,
                                 const float* g_ent, float* grad_h, void* grad_w,
                                 int grad_w_mode, void* workspace, cudaStream_t stream);
// grad_h [n] = the n_shards (1, 2, 4) partial dH in the quarter tree's order
// (n a multiple of 4, every pointer 16-byte aligned)
lp_status launch_merge_grad_h(const Device& dev, const float* const* shard_grad_h, int n_shards,
                              int64_t n, float* grad_h, cudaStream_t stream);

// Read and clear the check word of each translation unit (lp_check.cuh).
cudaError_t take_check_word_logits(uint32_t* out);
cudaError_t take_check_word_linear(uint32_t* out);
cudaError_t take_check_word_backward(uint32_t* out);

int persistent_grid_limit();
int fault_injection();
void timing_events(cudaEvent_t* start, cudaEvent_t* stop);

}  // namespace lp
