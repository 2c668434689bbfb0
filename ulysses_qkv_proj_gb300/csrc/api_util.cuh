// api_util.cuh -- argument-checking helpers shared by the C ABI translation units.
#pragma once

#include "../../include/qnre.h"

#include <cuda_runtime.h>

#include <cstdint>

namespace qnre {
namespace api {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct ByteRange {
  uintptr_t lo, hi;  // [lo, hi); empty when lo == hi
};

inline bool overlaps(ByteRange a, ByteRange b) { return a.lo < b.hi && b.lo < a.hi; }

inline ByteRange span(const void* p, uint64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + static_cast<uintptr_t>(bytes)};
}

inline int dtype_size(int32_t dt) {
  switch (dt) {
    case QNRE_DTYPE_BF16: return 2;
    case QNRE_DTYPE_FP16: return 2;
    case QNRE_DTYPE_FP32: return 4;
    default: return 0;
  }
}

inline qnre_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? QNRE_OK : QNRE_ERR_CUDA; }

// Checks common to every strided rank-4 view; fills the byte span of its
// storage.  Extents 0 and 1 (batch, sequence) may be 0 (an empty call).
inline qnre_status_t check_view(const qnre_tensor4_t* t, ByteRange* range) {
  if (t == nullptr || t->data == nullptr) return QNRE_ERR_INVALID_ARG;
  const int esz = dtype_size(t->dtype);
  if (esz == 0) return QNRE_ERR_UNSUPPORTED;
  bool empty = false;
  uint64_t last = 0;
  for (int i = 0; i < 4; ++i) {
    if (t->shape[i] < (i < 2 ? 0 : 1) || t->stride[i] < 1) return QNRE_ERR_INVALID_ARG;
    if (t->shape[i] > (int64_t{1} << 40) || t->stride[i] > (int64_t{1} << 40)) return QNRE_ERR_CAPACITY;
    if (t->shape[i] == 0) {
      empty = true;
      continue;
    }
    last += static_cast<uint64_t>(t->shape[i] - 1) * static_cast<uint64_t>(t->stride[i]);
    if (last > (uint64_t{1} << 56)) return QNRE_ERR_CAPACITY;
  }
  if (!aligned(t->data, static_cast<uintptr_t>(esz))) return QNRE_ERR_ALIGNMENT;
  *range = empty ? ByteRange{0, 0} : span(t->data, (last + 1) * static_cast<uint64_t>(esz));
  return QNRE_OK;
}

// Head rows of this view can be copied as 16-byte vectors.
inline bool rows_vectorisable(const qnre_tensor4_t* t, int esz) {
  if (t->stride[3] != 1) return false;
  if ((t->shape[3] * esz) % 16 != 0) return false;
  if (!aligned(t->data, 16)) return false;
  for (int i = 0; i < 3; ++i)
    if ((t->stride[i] * esz) % 16 != 0) return false;
  return true;
}

}  // namespace api
}  // namespace qnre
