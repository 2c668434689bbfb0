// debug_bounds.cuh -- the debug build's access checks (libqnre_debug.so, built
// with QNRE_DEBUG_BOUNDS=1).  A kernel checks each load or store against the
// byte range of the buffer it belongs to; an access outside it is counted and
// skipped, never performed.  Nothing here traps: the kernel runs to its end and
// the host reads the count.  The release build (QNRE_DEBUG_BOUNDS=0) compiles
// every check to `true`.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#ifndef QNRE_DEBUG_BOUNDS
#define QNRE_DEBUG_BOUNDS 0
#endif

namespace qnre {

struct Extent {
  uintptr_t lo, hi;  // [lo, hi) in bytes
};

inline Extent extent_of(const void* p, uint64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Extent{a, a + static_cast<uintptr_t>(bytes)};
}

#if QNRE_DEBUG_BOUNDS
// One counter per translation unit (internal linkage).
static __device__ unsigned long long g_bounds_violations;

// true when [p, p + n) lies inside e; else counts one violation
__device__ __forceinline__ bool access_ok(const void* p, int n, Extent e) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  if (a >= e.lo && a + n <= e.hi) return true;
  atomicAdd(&g_bounds_violations, 1ull);
  return false;
}

// This translation unit's count (reset to 0 when `reset`); synchronises the device.
static inline cudaError_t read_bounds_violations(unsigned long long* count, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(count, g_bounds_violations, sizeof(*count));
  if (e == cudaSuccess && reset) {
    const unsigned long long zero = 0;
    e = cudaMemcpyToSymbol(g_bounds_violations, &zero, sizeof(zero));
  }
  return e;
}
// Test hook of the debug build: QNRE_DEBUG_SHRINK_OUTPUT=<n> takes n bytes off
// the end of every output range the checks use, so the stores to the last n
// bytes of each output are counted and skipped although they lie inside the
// buffer.  It is the checks' positive control: no access leaves the real buffer.
inline uint64_t debug_shrink_bytes() {
  const char* s = std::getenv("QNRE_DEBUG_SHRINK_OUTPUT");
  return s ? std::strtoull(s, nullptr, 10) : 0;
}
inline Extent output_extent(uintptr_t lo, uintptr_t hi) {
  const uint64_t n = debug_shrink_bytes();
  return Extent{lo, hi - (n < hi - lo ? n : hi - lo)};
}

#define QNRE_ACCESS_OK(p, n, e) ::qnre::access_ok((p), (n), (e))
#else
#define QNRE_ACCESS_OK(p, n, e) true
#endif

}  // namespace qnre
