// Bounds checks of the checked build (the library compiled with
// -DQATTN_CHECK=1; build.build(checked=True)).  QATTN_IN_BOUNDS(cond) guards a
// device access whose index the kernel computes: when cond is false the access
// is skipped and the failure recorded in this translation unit's check word,
// which qattn_get_error() reads (QATTN_ERR_BOUNDS).  Nothing traps, so a
// failing check leaves the context usable.  In the normal build the macro is
// `true` and the compiler drops the test.
#pragma once
#include <cuda_runtime.h>

namespace qattn {

#if defined(QATTN_CHECK) && QATTN_CHECK
static __device__ unsigned int g_check_word;
__device__ __forceinline__ bool check_fail() {
  atomicOr(&g_check_word, 1u);
  return false;
}
#define QATTN_IN_BOUNDS(cond) ((cond) ? true : ::qattn::check_fail())
constexpr bool kChecked = true;
// Reads and clears this translation unit's check word (host).
static inline unsigned int check_take_local() {
  unsigned int v = 0;
  const unsigned int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_check_word, sizeof v) != cudaSuccess) return 0;
  if (v != 0) cudaMemcpyToSymbol(g_check_word, &zero, sizeof zero);
  return v;
}
#else
#define QATTN_IN_BOUNDS(cond) true
constexpr bool kChecked = false;
static inline unsigned int check_take_local() { return 0; }
#endif

}  // namespace qattn
