// lp_check.cuh: the checked build of liblp.
//
// Compiled with -DLP_CHECKED (the library _build_checked/liblp.so), every
// kernel tests the indexes and coordinates it computes for global memory
// accesses and TMA copies against the extents the host derived from the call's
// arguments.  A failed test never traps: it ORs the access's bit into this
// translation unit's check word and the access is skipped.  lp_get_check_word
// reads (and clears) the check words of all translation units.  In the normal
// build LP_CHECK(cond, bit) is the constant true, so the tests cost nothing.
// This is the stand-in for a memory checker on GPUs where none may run.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lp {

#ifdef LP_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// Bits of the check word: which access failed its test.
constexpr uint32_t kChkLogitsLoad = 1u << 0;     // a logit read outside its row's quarter
constexpr uint32_t kChkRowIndex = 1u << 1;       // a per-row input or output outside [0, T)
constexpr uint32_t kChkStateIndex = 1u << 2;     // a quarter or tile state outside its buffer
constexpr uint32_t kChkTmaCoord = 1u << 3;       // a TMA load coordinate negative
constexpr uint32_t kChkGStore = 1u << 4;         // a store of G outside [T, ld_g]
constexpr uint32_t kChkOutBox = 1u << 5;         // a product's output box outside C
constexpr uint32_t kChkSplitIndex = 1u << 6;     // a split-sum read or write outside its buffer
constexpr uint32_t kChkCopyIndex = 1u << 7;      // a padding / row-copy access outside its buffer

// One check word per translation unit (each .cu file is its own module).
static __device__ uint32_t g_check_word;

__device__ __forceinline__ bool check_ok(bool ok, uint32_t bit) {
  if (!kChecked) return true;
  if (!ok) atomicOr(&g_check_word, bit);
  return ok;
}

#define LP_CHECK(cond, bit) (::lp::kChecked ? ::lp::check_ok((cond), (bit)) : true)

// Host: read this translation unit's check word in the current context and
// clear it.
static inline cudaError_t take_check_word(uint32_t* out) {
  uint32_t w = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&w, g_check_word, sizeof(w));
  if (e == cudaSuccess) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_check_word, &zero, sizeof(zero));
  }
  *out = w;
  return e;
}

}  // namespace lp
