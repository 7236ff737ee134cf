// lp_api.cu: the C-ABI front end of liblp (declared in include/lp.h).
//
// Every entry point validates its arguments on the host, in this order:
// sizes and null pointers (LP_ERR_INVALID_ARGUMENT), alignment
// (LP_ERR_MISALIGNED), workspace size (LP_ERR_WORKSPACE_TOO_SMALL), and only
// then the current device (LP_ERR_UNSUPPORTED_DEVICE unless compute capability
// 10.3).  Nothing is enqueued before all checks pass.  There is no fallback
// path of any kind: on another device, or without a device, calls fail.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "lp_check.cuh"
#include "lp_device.cuh"
#include "lp_internal.h"

namespace lp {

namespace {
std::atomic<int> g_grid_limit{0};
std::atomic<int> g_fault_injection{0};
std::atomic<cudaEvent_t> g_ev_start{nullptr};
std::atomic<cudaEvent_t> g_ev_stop{nullptr};

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_state[kMaxDevices];  // 0 unknown, 1 supported, 2 unsupported
std::atomic<int> g_dev_sms[kMaxDevices];

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
}  // namespace

int persistent_grid_limit() { return g_grid_limit.load(std::memory_order_relaxed); }
int fault_injection() { return g_fault_injection.load(std::memory_order_relaxed); }

void timing_events(cudaEvent_t* start, cudaEvent_t* stop) {
  *start = g_ev_start.load(std::memory_order_acquire);
  *stop = g_ev_stop.load(std::memory_order_acquire);
}

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  cudaGetLastError();
  return nullptr;
}
}  // namespace

uint64_t current_context_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return static_cast<uint64_t>(id);
}

lp_status current_device(Device* dev) {
  int ordinal = 0;
  if (cudaGetDevice(&ordinal) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of a missing device
    return LP_ERR_UNSUPPORTED_DEVICE;
  }
  if (ordinal < 0 || ordinal >= kMaxDevices) return LP_ERR_UNSUPPORTED_DEVICE;
  int state = g_dev_state[ordinal].load(std::memory_order_acquire);
  if (state == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, ordinal) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, ordinal) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ordinal) != cudaSuccess) {
      cudaGetLastError();
      return LP_ERR_CUDA;
    }
    g_dev_sms[ordinal].store(sms, std::memory_order_relaxed);
    state = (major == 10 && minor == 3) ? 1 : 2;
    g_dev_state[ordinal].store(state, std::memory_order_release);
  }
  if (state != 1) return LP_ERR_UNSUPPORTED_DEVICE;
  dev->ordinal = ordinal;
  dev->sm_count = g_dev_sms[ordinal].load(std::memory_order_relaxed);
  dev->ctx_id = current_context_id();
  return LP_OK;
}

namespace {

// The temperature arguments of a call: false unless tau is finite and > 0 and
// 1/tau is a finite positive float.  1/tau is split into inv_hi = fl(1/tau)
// and inv_lo = fl(1/tau - inv_hi), both from float64.
bool make_tau(float temperature, TauArgs* out) {
  if (!(temperature > 0.0f) || !(temperature < 3.402823466e38f)) return false;
  const double r = 1.0 / static_cast<double>(temperature);
  if (!(r > 0.0) || r > 3.402823466e38) return false;
  const float hi = static_cast<float>(r);
  if (!(hi > 0.0f) || !(hi < 3.402823466e38f)) return false;
  out->tau = temperature;
  out->inv_hi = hi;
  out->inv_lo = static_cast<float>(r - static_cast<double>(hi));
  return true;
}

lp_status check_shard(int shard_index, int n_shards) {
  if (!(n_shards == 1 || n_shards == 2 || n_shards == 4)) return LP_ERR_INVALID_ARGUMENT;
  if (shard_index < 0 || shard_index >= n_shards) return LP_ERR_INVALID_ARGUMENT;
  return LP_OK;
}

lp_status check_fused_args(const void* H, int64_t ld_h, const void* W, int64_t ld_w,
                           const int64_t* targets, int64_t T, int64_t d, int64_t V) {
  if (T < 0 || T > kMaxDim || d < 1 || d > kMaxDim || V < 1 || V > kMaxDim)
    return LP_ERR_INVALID_ARGUMENT;
  if (ld_h < d || ld_w < d) return LP_ERR_INVALID_ARGUMENT;
  if (T == 0) return LP_OK;
  if (H == nullptr || W == nullptr || targets == nullptr) return LP_ERR_INVALID_ARGUMENT;
  if (!aligned(H, 16) || !aligned(W, 16) || (ld_h % 8) != 0 || (ld_w % 8) != 0 ||
      !aligned(targets, 8))
    return LP_ERR_MISALIGNED;
  return LP_OK;
}

}  // namespace
}  // namespace lp


extern "C" {

const char* lp_status_string(lp_status status) {
  switch (status) {
    case LP_OK: return "LP_OK";
    case LP_ERR_INVALID_ARGUMENT: return "LP_ERR_INVALID_ARGUMENT";
    case LP_ERR_MISALIGNED: return "LP_ERR_MISALIGNED";
    case LP_ERR_UNSUPPORTED_DEVICE: return "LP_ERR_UNSUPPORTED_DEVICE";
    case LP_ERR_WORKSPACE_TOO_SMALL: return "LP_ERR_WORKSPACE_TOO_SMALL";
    case LP_ERR_CUDA: return "LP_ERR_CUDA";
    case LP_ERR_TIMEOUT: return "LP_ERR_TIMEOUT";
  }
  return "LP_ERR_UNKNOWN";
}

const char* lp_backend_id(void) {
  return lp::kChecked ? "lp.sm103a.bitwise.v1+checked" : "lp.sm103a.bitwise.v1";
}

lp_status lp_get_check_word(uint32_t* word_out) {
  if (word_out == nullptr) return LP_ERR_INVALID_ARGUMENT;
  *word_out = 0;
  lp::Device dev;
  const lp_status st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return LP_ERR_CUDA;
  uint32_t a = 0, b = 0, c = 0;
  if (lp::take_check_word_logits(&a) != cudaSuccess ||
      lp::take_check_word_linear(&b) != cudaSuccess ||
      lp::take_check_word_backward(&c) != cudaSuccess) {
    cudaGetLastError();
    return LP_ERR_CUDA;
  }
  *word_out = a | b | c;
  return LP_OK;
}

lp_status lp_set_persistent_grid_limit(int max_ctas) {
  if (max_ctas < 0) return LP_ERR_INVALID_ARGUMENT;
  lp::g_grid_limit.store(max_ctas, std::memory_order_relaxed);
  return LP_OK;
}

lp_status lp_set_fault_injection(int mode) {
  if (mode < 0 || mode > 2) return LP_ERR_INVALID_ARGUMENT;
  lp::g_fault_injection.store(mode, std::memory_order_relaxed);
  return LP_OK;
}

lp_status lp_set_kernel_timing_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return LP_ERR_INVALID_ARGUMENT;
  lp::g_ev_start.store(static_cast<cudaEvent_t>(start_event), std::memory_order_release);
  lp::g_ev_stop.store(static_cast<cudaEvent_t>(stop_event), std::memory_order_release);
  return LP_OK;
}

lp_status lp_vocab_shard_range(int64_t vocab_total, int shard_index, int n_shards,
                               int64_t* begin, int64_t* end) {
  if (vocab_total < 1 || vocab_total > lp::kMaxDim || begin == nullptr || end == nullptr)
    return LP_ERR_INVALID_ARGUMENT;
  const lp_status st = lp::check_shard(shard_index, n_shards);
  if (st != LP_OK) return st;
  int q_first, n_q;
  lp::shard_quarters(shard_index, n_shards, q_first, n_q);
  *begin = lp::quarter_begin(vocab_total, q_first);
  *end = lp::quarter_begin(vocab_total, q_first + n_q);
  return LP_OK;
}

lp_status lp_logprob_from_logits_temperature(const float* logits, int64_t ld_logits,
                                             const int64_t* targets, int64_t T, int64_t V,
                                             float temperature, float* logp_out,
                                             float* entropy_out, void* stream) {
  lp::TauArgs tau;
  if (!lp::make_tau(temperature, &tau)) return LP_ERR_INVALID_ARGUMENT;
  if (T < 0 || T > lp::kMaxDim / 4 || V < 1 || V > lp::kMaxDim || ld_logits < V)
    return LP_ERR_INVALID_ARGUMENT;
  if (T == 0) return LP_OK;
  if (logits == nullptr || targets == nullptr || logp_out == nullptr)
    return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(logits, 4) || !lp::aligned(targets, 8) || !lp::aligned(logp_out, 4) ||
      !lp::aligned(entropy_out, 4))
    return LP_ERR_MISALIGNED;
  lp::Device dev;
  const lp_status st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_logits_final(logits, ld_logits, targets, T, V, tau, logp_out,
                                 entropy_out, nullptr, static_cast<cudaStream_t>(stream));
}

lp_status lp_logprob_from_logits_lse(const float* logits, int64_t ld_logits,
                                     const int64_t* targets, int64_t T, int64_t V,
                                     float temperature, float* logp_out, float* entropy_out,
                                     float* lse_out, void* stream) {
  lp::TauArgs tau;
  if (!lp::make_tau(temperature, &tau)) return LP_ERR_INVALID_ARGUMENT;
  if (T < 0 || T > lp::kMaxDim / 4 || V < 1 || V > lp::kMaxDim || ld_logits < V)
    return LP_ERR_INVALID_ARGUMENT;
  if (T == 0) return LP_OK;
  if (logits == nullptr || targets == nullptr || logp_out == nullptr || entropy_out == nullptr ||
      lse_out == nullptr)
    return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(logits, 4) || !lp::aligned(targets, 8) || !lp::aligned(logp_out, 4) ||
      !lp::aligned(entropy_out, 4) || !lp::aligned(lse_out, 4))
    return LP_ERR_MISALIGNED;
  lp::Device dev;
  const lp_status st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_logits_final(logits, ld_logits, targets, T, V, tau, logp_out, entropy_out,
                                 lse_out, static_cast<cudaStream_t>(stream));
}

namespace {
// The logits-path backward over columns col0 .. col0 + V - 1 of a vocabulary
// of V_total (the whole vocabulary, or one shard of it).
lp_status logits_backward_checked(const float* logits, int64_t ld_logits, const int64_t* targets,
                                  int64_t T, int64_t V, int64_t col0, int64_t V_total,
                                  float temperature, const float* saved_lse,
                                  const float* saved_entropy, const float* grad_logp,
                                  const float* grad_entropy, float* grad_logits, int64_t ld_grad,
                                  void* stream) {
  lp::TauArgs tau;
  if (!lp::make_tau(temperature, &tau)) return LP_ERR_INVALID_ARGUMENT;
  if (T < 0 || T > lp::kMaxDim / 4 || V < 1 || V > lp::kMaxDim || ld_logits < V || ld_grad < V)
    return LP_ERR_INVALID_ARGUMENT;
  if (T == 0) return LP_OK;
  if (logits == nullptr || targets == nullptr || saved_lse == nullptr ||
      saved_entropy == nullptr || grad_logits == nullptr ||
      (grad_logp == nullptr && grad_entropy == nullptr))
    return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(logits, 4) || !lp::aligned(targets, 8) || !lp::aligned(saved_lse, 4) ||
      !lp::aligned(saved_entropy, 4) || !lp::aligned(grad_logp, 4) ||
      !lp::aligned(grad_entropy, 4) || !lp::aligned(grad_logits, 4))
    return LP_ERR_MISALIGNED;
  // grad_logits must not overlap the logits (they are read through the
  // read-only path while the gradient is written)
  const uintptr_t z0 = reinterpret_cast<uintptr_t>(logits);
  const uintptr_t z1 = z0 + 4 * static_cast<uintptr_t>((T - 1) * ld_logits + V);
  const uintptr_t g0 = reinterpret_cast<uintptr_t>(grad_logits);
  const uintptr_t g1 = g0 + 4 * static_cast<uintptr_t>((T - 1) * ld_grad + V);
  if (g0 < z1 && z0 < g1) return LP_ERR_INVALID_ARGUMENT;
  lp::Device dev;
  const lp_status st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_logits_backward(logits, ld_logits, targets, T, V, col0, V_total, tau,
                                    saved_lse, saved_entropy, grad_logp, grad_entropy, grad_logits,
                                    ld_grad, static_cast<cudaStream_t>(stream));
}
}  // namespace

lp_status lp_logprob_from_logits_backward(const float* logits, int64_t ld_logits,
                                          const int64_t* targets, int64_t T, int64_t V,
                                          float temperature, const float* saved_lse,
                                          const float* saved_entropy, const float* grad_logp,
                                          const float* grad_entropy, float* grad_logits,
                                          int64_t ld_grad, void* stream) {
  return logits_backward_checked(logits, ld_logits, targets, T, V, 0, V, temperature, saved_lse,
                                 saved_entropy, grad_logp, grad_entropy, grad_logits, ld_grad,
                                 stream);
}

lp_status lp_logprob_partials_from_logits_backward(
    const float* logits_shard, int64_t ld_logits, const int64_t* targets, int64_t T,
    int64_t vocab_total, int shard_index, int n_shards, float temperature,
    const float* saved_lse, const float* saved_entropy, const float* grad_logp,
    const float* grad_entropy, float* grad_shard, int64_t ld_grad, void* stream) {
  int64_t begin = 0, end = 0;
  const lp_status st = lp_vocab_shard_range(vocab_total, shard_index, n_shards, &begin, &end);
  if (st != LP_OK) return st;
  return logits_backward_checked(logits_shard, ld_logits, targets, T, end - begin, begin,
                                 vocab_total, temperature, saved_lse, saved_entropy, grad_logp,
                                 grad_entropy, grad_shard, ld_grad, stream);
}

lp_status lp_logprob_partials_from_logits_temperature(const float* logits_shard,
                                                      int64_t ld_logits, const int64_t* targets,
                                                      int64_t T, int64_t vocab_total,
                                                      int shard_index, int n_shards,
                                                      float temperature, float* partials_out,
                                                      void* stream) {
  lp::TauArgs tau;
  if (!lp::make_tau(temperature, &tau)) return LP_ERR_INVALID_ARGUMENT;
  lp_status st = lp::check_shard(shard_index, n_shards);
  if (st != LP_OK) return st;
  if (T < 0 || T > lp::kMaxDim / 4 || vocab_total < 1 || vocab_total > lp::kMaxDim)
    return LP_ERR_INVALID_ARGUMENT;
  int64_t b, e;
  lp_vocab_shard_range(vocab_total, shard_index, n_shards, &b, &e);
  if (ld_logits < e - b || ld_logits < 1) return LP_ERR_INVALID_ARGUMENT;
  if (T == 0) return LP_OK;
  // an empty shard (vocab_total < 4 only) reads no logits and may pass NULL
  if ((logits_shard == nullptr && e > b) || targets == nullptr || partials_out == nullptr)
    return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(logits_shard, 4) || !lp::aligned(targets, 8) ||
      !lp::aligned(partials_out, 16))
    return LP_ERR_MISALIGNED;
  lp::Device dev;
  st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  int q_first, n_q;
  lp::shard_quarters(shard_index, n_shards, q_first, n_q);
  return lp::launch_logits_partials(logits_shard, ld_logits, targets, T, vocab_total, q_first,
                                    n_q, tau, partials_out, static_cast<cudaStream_t>(stream));
}

lp_status lp_merge_partials(const float* const* shard_partials, int n_shards, int64_t T,
                            float* logp_out, float* entropy_out, void* stream) {
  if (!(n_shards == 1 || n_shards == 2 || n_shards == 4)) return LP_ERR_INVALID_ARGUMENT;
  if (T < 0 || T > lp::kMaxDim) return LP_ERR_INVALID_ARGUMENT;
  if (T == 0) return LP_OK;
  if (shard_partials == nullptr || logp_out == nullptr) return LP_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < n_shards; ++i) {
    if (shard_partials[i] == nullptr) return LP_ERR_INVALID_ARGUMENT;
    if (!lp::aligned(shard_partials[i], 16)) return LP_ERR_MISALIGNED;
  }
  if (!lp::aligned(logp_out, 4) || !lp::aligned(entropy_out, 4)) return LP_ERR_MISALIGNED;
  lp::Device dev;
  const lp_status st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_merge_partials(shard_partials, n_shards, T, logp_out, entropy_out, nullptr,
                                   static_cast<cudaStream_t>(stream));
}

lp_status lp_merge_partials_lse(const float* const* shard_partials, int n_shards, int64_t T,
                                float* logp_out, float* entropy_out, float* lse_out,
                                void* stream) {
  if (!(n_shards == 1 || n_shards == 2 || n_shards == 4)) return LP_ERR_INVALID_ARGUMENT;
  if (T < 0 || T > lp::kMaxDim) return LP_ERR_INVALID_ARGUMENT;
  if (T == 0) return LP_OK;
  if (shard_partials == nullptr || logp_out == nullptr || entropy_out == nullptr ||
      lse_out == nullptr)
    return LP_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < n_shards; ++i) {
    if (shard_partials[i] == nullptr) return LP_ERR_INVALID_ARGUMENT;
    if (!lp::aligned(shard_partials[i], 16)) return LP_ERR_MISALIGNED;
  }
  if (!lp::aligned(logp_out, 4) || !lp::aligned(entropy_out, 4) || !lp::aligned(lse_out, 4))
    return LP_ERR_MISALIGNED;
  lp::Device dev;
  const lp_status st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_merge_partials(shard_partials, n_shards, T, logp_out, entropy_out, lse_out,
                                   static_cast<cudaStream_t>(stream));
}

size_t lp_linear_logprob_workspace_size(int64_t T, int64_t d, int64_t V) {
  if (T < 0 || d < 1 || d > lp::kMaxDim || V < 1 || V > lp::kMaxDim) return 0;
  return lp::linear_workspace_bytes(T, d, V, 4);
}

size_t lp_linear_logprob_partials_workspace_size(int64_t T, int64_t d, int64_t vocab_total,
                                                 int n_shards) {
  if (T < 0 || d < 1 || d > lp::kMaxDim || vocab_total < 1 || vocab_total > lp::kMaxDim)
    return 0;
  if (!(n_shards == 1 || n_shards == 2 || n_shards == 4)) return 0;
  return lp::linear_workspace_bytes(T, d, vocab_total, 4 / n_shards);
}

lp_status lp_linear_logprob_temperature(const void* H, int64_t ld_h, const void* W, int64_t ld_w,
                                        const int64_t* targets, int64_t T, int64_t d, int64_t V,
                                        float temperature, float* logp_out, float* entropy_out,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  lp::TauArgs tau;
  if (!lp::make_tau(temperature, &tau)) return LP_ERR_INVALID_ARGUMENT;
  lp_status st = lp::check_fused_args(H, ld_h, W, ld_w, targets, T, d, V);
  if (st != LP_OK || T == 0) return st;
  if (logp_out == nullptr || workspace == nullptr) return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(logp_out, 4) || !lp::aligned(entropy_out, 4) || !lp::aligned(workspace, 256))
    return LP_ERR_MISALIGNED;
  if (workspace_bytes < lp::linear_workspace_bytes(T, d, V, 4)) return LP_ERR_WORKSPACE_TOO_SMALL;
  lp::Device dev;
  st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_linear(dev, H, ld_h, W, ld_w, targets, T, d, V, 0, 4, tau, logp_out,
                           entropy_out, nullptr, workspace, static_cast<cudaStream_t>(stream));
}

lp_status lp_linear_logprob_noalloc(const void* H, int64_t ld_h, const void* W, int64_t ld_w,
                                    const int64_t* targets, int64_t T, int64_t d, int64_t V,
                                    float* logp_out, float* entropy_out, void* stream) {
  lp_status st = lp::check_fused_args(H, ld_h, W, ld_w, targets, T, d, V);
  if (st != LP_OK || T == 0) return st;
  if (logp_out == nullptr) return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(logp_out, 4) || !lp::aligned(entropy_out, 4)) return LP_ERR_MISALIGNED;
  if (lp::linear_workspace_bytes(T, d, V, 4) > lp::static_scratch_bytes())
    return LP_ERR_WORKSPACE_TOO_SMALL;
  lp::Device dev;
  st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  void* scratch = nullptr;
  st = lp::static_scratch(&scratch);
  if (st != LP_OK) return st;
  lp::TauArgs tau;
  lp::make_tau(1.0f, &tau);
  return lp::launch_linear(dev, H, ld_h, W, ld_w, targets, T, d, V, 0, 4, tau, logp_out,
                           entropy_out, nullptr, scratch, static_cast<cudaStream_t>(stream));
}

lp_status lp_linear_logprob_lse(const void* H, int64_t ld_h, const void* W, int64_t ld_w,
                                const int64_t* targets, int64_t T, int64_t d, int64_t V,
                                float temperature, float* logp_out, float* entropy_out,
                                float* lse_out, void* workspace, size_t workspace_bytes,
                                void* stream) {
  lp::TauArgs tau;
  if (!lp::make_tau(temperature, &tau)) return LP_ERR_INVALID_ARGUMENT;
  lp_status st = lp::check_fused_args(H, ld_h, W, ld_w, targets, T, d, V);
  if (st != LP_OK || T == 0) return st;
  if (logp_out == nullptr || entropy_out == nullptr || lse_out == nullptr || workspace == nullptr)
    return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(logp_out, 4) || !lp::aligned(entropy_out, 4) || !lp::aligned(lse_out, 4) ||
      !lp::aligned(workspace, 256))
    return LP_ERR_MISALIGNED;
  if (workspace_bytes < lp::linear_workspace_bytes(T, d, V, 4)) return LP_ERR_WORKSPACE_TOO_SMALL;
  lp::Device dev;
  st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_linear_stats(dev, H, ld_h, W, ld_w, targets, T, d, V, 0, 4, tau, logp_out,
                                 entropy_out, nullptr, lse_out, workspace,
                                 static_cast<cudaStream_t>(stream));
}

lp_status lp_linear_logprob_partials_temperature(const void* H, int64_t ld_h,
                                                 const void* W_shard, int64_t ld_w,
                                                 const int64_t* targets, int64_t T, int64_t d,
                                                 int64_t vocab_total, int shard_index,
                                                 int n_shards, float temperature,
                                                 float* partials_out, void* workspace,
                                                 size_t workspace_bytes, void* stream) {
  lp::TauArgs tau;
  if (!lp::make_tau(temperature, &tau)) return LP_ERR_INVALID_ARGUMENT;
  lp_status st = lp::check_shard(shard_index, n_shards);
  if (st != LP_OK) return st;
  st = lp::check_fused_args(H, ld_h, W_shard, ld_w, targets, T, d, vocab_total);
  if (st != LP_OK || T == 0) return st;
  if (partials_out == nullptr || workspace == nullptr) return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(partials_out, 16) || !lp::aligned(workspace, 256)) return LP_ERR_MISALIGNED;
  int q_first, n_q;
  lp::shard_quarters(shard_index, n_shards, q_first, n_q);
  if (workspace_bytes < lp::linear_workspace_bytes(T, d, vocab_total, n_q))
    return LP_ERR_WORKSPACE_TOO_SMALL;
  lp::Device dev;
  st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_linear(dev, H, ld_h, W_shard, ld_w, targets, T, d, vocab_total, q_first, n_q,
                           tau, nullptr, nullptr, partials_out, workspace,
                           static_cast<cudaStream_t>(stream));
}

lp_status lp_logprob_from_logits(const float* logits, int64_t ld_logits, const int64_t* targets,
                                 int64_t T, int64_t V, float* logp_out, float* entropy_out,
                                 void* stream) {
  return lp_logprob_from_logits_temperature(logits, ld_logits, targets, T, V, 1.0f, logp_out,
                                            entropy_out, stream);
}

lp_status lp_logprob_partials_from_logits(const float* logits_shard, int64_t ld_logits,
                                          const int64_t* targets, int64_t T,
                                          int64_t vocab_total, int shard_index, int n_shards,
                                          float* partials_out, void* stream) {
  return lp_logprob_partials_from_logits_temperature(logits_shard, ld_logits, targets, T,
                                                     vocab_total, shard_index, n_shards, 1.0f,
                                                     partials_out, stream);
}

lp_status lp_linear_logprob(const void* H, int64_t ld_h, const void* W, int64_t ld_w,
                            const int64_t* targets, int64_t T, int64_t d, int64_t V,
                            float* logp_out, float* entropy_out, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return lp_linear_logprob_temperature(H, ld_h, W, ld_w, targets, T, d, V, 1.0f, logp_out,
                                       entropy_out, workspace, workspace_bytes, stream);
}

lp_status lp_linear_logprob_partials(const void* H, int64_t ld_h, const void* W_shard,
                                     int64_t ld_w, const int64_t* targets, int64_t T, int64_t d,
                                     int64_t vocab_total, int shard_index, int n_shards,
                                     float* partials_out, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  return lp_linear_logprob_partials_temperature(H, ld_h, W_shard, ld_w, targets, T, d,
                                                vocab_total, shard_index, n_shards, 1.0f,
                                                partials_out, workspace, workspace_bytes, stream);
}

size_t lp_linear_logprob_backward_workspace_size(int64_t T, int64_t d, int64_t V) {
  if (T < 0 || d < 1 || V < 1 || V > lp::kMaxDim || d > lp::kMaxDim) return 0;
  return lp::linear_backward_workspace_bytes(T, d, V, V);
}

lp_status lp_linear_logprob_backward_ex(const void* H, int64_t ld_h, const void* W, int64_t ld_w,
                                        const int64_t* targets, int64_t T, int64_t d, int64_t V,
                                        float temperature, const float* saved_lse,
                                        const float* saved_entropy, const float* grad_logp,
                                        const float* grad_entropy, float* grad_H, void* grad_W,
                                        int grad_W_dtype, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  lp::TauArgs tau;
  if (!lp::make_tau(temperature, &tau)) return LP_ERR_INVALID_ARGUMENT;
  if (grad_W_dtype != LP_GRAD_W_FLOAT32 && grad_W_dtype != LP_GRAD_W_BFLOAT16 &&
      grad_W_dtype != LP_GRAD_W_FLOAT32_ACCUMULATE)
    return LP_ERR_INVALID_ARGUMENT;
  lp_status st = lp::check_fused_args(H, ld_h, W, ld_w, targets, T, d, V);
  if (st != LP_OK || T == 0) return st;
  if (grad_H == nullptr || workspace == nullptr) return LP_ERR_INVALID_ARGUMENT;
  if (grad_logp == nullptr && grad_entropy == nullptr) return LP_ERR_INVALID_ARGUMENT;
  if ((saved_lse == nullptr) != (saved_entropy == nullptr)) return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(saved_lse, 4) || !lp::aligned(saved_entropy, 4)) return LP_ERR_MISALIGNED;
  if (T > (int64_t(1) << 24)) return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(grad_logp, 4) || !lp::aligned(grad_entropy, 4) || !lp::aligned(grad_H, 16) ||
      !lp::aligned(grad_W, 16) || !lp::aligned(workspace, 256))
    return LP_ERR_MISALIGNED;
  if (workspace_bytes < lp::linear_backward_workspace_bytes(T, d, V, V))
    return LP_ERR_WORKSPACE_TOO_SMALL;
  lp::Device dev;
  st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_linear_backward(dev, H, ld_h, W, ld_w, targets, T, d, V, V, 0, 4, tau,
                                    saved_lse, saved_entropy, grad_logp, grad_entropy, grad_H,
                                    grad_W, grad_W_dtype, workspace,
                                    static_cast<cudaStream_t>(stream));
}

size_t lp_linear_logprob_partials_backward_workspace_size(int64_t T, int64_t d,
                                                          int64_t vocab_total, int n_shards) {
  if (T < 0 || d < 1 || d > lp::kMaxDim || vocab_total < 1 || vocab_total > lp::kMaxDim)
    return 0;
  if (!(n_shards == 1 || n_shards == 2 || n_shards == 4)) return 0;
  size_t most = 0;  // the widest shard's
  for (int i = 0; i < n_shards; ++i) {
    int64_t b = 0, e = 0;
    lp_vocab_shard_range(vocab_total, i, n_shards, &b, &e);
    if (e > b) most = std::max(most, lp::linear_backward_workspace_bytes(T, d, e - b, vocab_total));
  }
  return most;
}

lp_status lp_linear_logprob_partials_backward(
    const void* H, int64_t ld_h, const void* W_shard, int64_t ld_w, const int64_t* targets,
    int64_t T, int64_t d, int64_t vocab_total, int shard_index, int n_shards, float temperature,
    const float* saved_lse, const float* saved_entropy, const float* grad_logp,
    const float* grad_entropy, float* grad_H_partial, void* grad_W_shard, int grad_W_dtype,
    void* workspace, size_t workspace_bytes, void* stream) {
  lp::TauArgs tau;
  if (!lp::make_tau(temperature, &tau)) return LP_ERR_INVALID_ARGUMENT;
  if (grad_W_dtype != LP_GRAD_W_FLOAT32 && grad_W_dtype != LP_GRAD_W_BFLOAT16 &&
      grad_W_dtype != LP_GRAD_W_FLOAT32_ACCUMULATE)
    return LP_ERR_INVALID_ARGUMENT;
  lp_status st = lp::check_shard(shard_index, n_shards);
  if (st != LP_OK) return st;
  st = lp::check_fused_args(H, ld_h, W_shard, ld_w, targets, T, d, vocab_total);
  if (st != LP_OK) return st;
  // the quarters must start on 16-column boundaries for a shard to compute a
  // subtree of the single-GPU order of grad_H
  if (n_shards > 1 && vocab_total % 64 != 0) return LP_ERR_INVALID_ARGUMENT;
  if (T == 0) return LP_OK;
  if (grad_H_partial == nullptr || workspace == nullptr || saved_lse == nullptr ||
      saved_entropy == nullptr || (grad_logp == nullptr && grad_entropy == nullptr))
    return LP_ERR_INVALID_ARGUMENT;
  if (T > (int64_t(1) << 24)) return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(saved_lse, 4) || !lp::aligned(saved_entropy, 4) ||
      !lp::aligned(grad_logp, 4) || !lp::aligned(grad_entropy, 4) ||
      !lp::aligned(grad_H_partial, 16) || !lp::aligned(grad_W_shard, 16) ||
      !lp::aligned(workspace, 256))
    return LP_ERR_MISALIGNED;
  int q_first, n_q;
  lp::shard_quarters(shard_index, n_shards, q_first, n_q);
  const int64_t begin = lp::quarter_begin(vocab_total, q_first);
  const int64_t end = lp::quarter_begin(vocab_total, q_first + n_q);
  if (end == begin) return LP_ERR_INVALID_ARGUMENT;  // only vocab_total < 4, n_shards 4
  if (workspace_bytes < lp::linear_backward_workspace_bytes(T, d, end - begin, vocab_total))
    return LP_ERR_WORKSPACE_TOO_SMALL;
  lp::Device dev;
  st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_linear_backward(dev, H, ld_h, W_shard, ld_w, targets, T, d, end - begin,
                                    vocab_total, q_first, n_q, tau, saved_lse, saved_entropy,
                                    grad_logp, grad_entropy, grad_H_partial, grad_W_shard,
                                    grad_W_dtype, workspace,
                                    static_cast<cudaStream_t>(stream));
}

lp_status lp_merge_grad_h_partials(const float* const* shard_grad_h, int n_shards, int64_t T,
                                   int64_t d, float* grad_H, void* stream) {
  if (!(n_shards == 1 || n_shards == 2 || n_shards == 4)) return LP_ERR_INVALID_ARGUMENT;
  if (T < 0 || T > lp::kMaxDim || d < 1 || d > lp::kMaxDim) return LP_ERR_INVALID_ARGUMENT;
  if (d % 8 != 0) return LP_ERR_MISALIGNED;
  if (T == 0) return LP_OK;
  if (shard_grad_h == nullptr || grad_H == nullptr) return LP_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < n_shards; ++i) {
    if (shard_grad_h[i] == nullptr) return LP_ERR_INVALID_ARGUMENT;
    if (!lp::aligned(shard_grad_h[i], 16)) return LP_ERR_MISALIGNED;
  }
  if (!lp::aligned(grad_H, 16)) return LP_ERR_MISALIGNED;
  lp::Device dev;
  const lp_status st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  return lp::launch_merge_grad_h(dev, shard_grad_h, n_shards, T * d, grad_H,
                                 static_cast<cudaStream_t>(stream));
}

lp_status lp_linear_logprob_backward(const void* H, int64_t ld_h, const void* W, int64_t ld_w,
                                     const int64_t* targets, int64_t T, int64_t d, int64_t V,
                                     float temperature, const float* saved_lse,
                                     const float* saved_entropy, const float* grad_logp,
                                     const float* grad_entropy, float* grad_H, float* grad_W,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  return lp_linear_logprob_backward_ex(H, ld_h, W, ld_w, targets, T, d, V, temperature, saved_lse,
                                       saved_entropy, grad_logp, grad_entropy, grad_H, grad_W,
                                       LP_GRAD_W_FLOAT32, workspace, workspace_bytes, stream);
}

lp_status lp_get_device_error(const void* workspace, size_t workspace_bytes, uint32_t* word_out,
                              void* stream) {
  if (workspace == nullptr || workspace_bytes < lp::kWorkspaceHeader)
    return LP_ERR_INVALID_ARGUMENT;
  if (!lp::aligned(workspace, 256)) return LP_ERR_MISALIGNED;
  lp::Device dev;
  const lp_status st = lp::current_device(&dev);
  if (st != LP_OK) return st;
  uint32_t words[4] = {0, 0, 0, 0};  // one word per pipeline kernel of a call
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(words, workspace, sizeof(words), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return LP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LP_ERR_CUDA;
  const uint32_t word = words[0] | words[1] | words[2] | words[3];
  if (word_out != nullptr) *word_out = word;
  return word == 0 ? LP_OK : LP_ERR_TIMEOUT;
}

}  // extern "C"
