// layout_copy.cuh -- launcher of the head-row copy kernel behind every Ulysses
// layout entry point (head-chunk pack and merge, scatter/gather heads, the
// output sequence-chunk pack and the composed head-chunk exchanges).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace qnre {

// One launch copies head rows of `units` copy units each.  A "segment" is one
// (slot, component) pair: slot = r*head_count + j names head j of rank r's
// band, component c selects one of up to three sources (q | k | v).  Rows are
// addressed by a sequence index s < S and a batch index z < Z1*Z0 split as
// z = z1*Z0 + z0.  All strides are in bytes:
//   src = src[c] + r*src_rank[c] + (src_head_offset + j)*src_head[c]
//                + z1*src_z1[c] + z0*src_z0[c] + s*src_s[c] + u*src_unit
//   dst = dst    + r*dst_rank    + (dst_head_offset + j)*dst_head + c*dst_comp
//                + z1*dst_z1     + z0*dst_z0     + s*dst_s     + u*unit_bytes
struct LayoutCopyPlan {
  const void* src[3];
  long long src_rank[3], src_head[3], src_z1[3], src_z0[3], src_s[3];
  long long src_unit;
  int src_head_offset;
  void* dst;
  long long dst_rank, dst_head, dst_comp, dst_z1, dst_z0, dst_s;
  int dst_head_offset;
  long long Z1, Z0, S;
  int head_count;   // heads per band (j < head_count)
  int ranks;        // r < ranks
  int comps;        // 1 or 3
  int units;        // copy units per head row
  int unit_bytes;   // 16 (vector path), 4 or 2 (element path)
  // Byte ranges [lo, hi) of each source and of the output, from the entry
  // point's own extent checks.  The debug build checks every access against
  // them (and refuses a plan without them); the release build ignores them.
  uintptr_t src_lo[3], src_hi[3];
  uintptr_t dst_lo, dst_hi;
  // 1: cache-streaming loads and stores (the copy runs beside a kernel whose
  // L2 working set it should not displace); 0: the default policy.
  int streaming;
};

cudaError_t launch_layout_copy(const LayoutCopyPlan& plan, cudaStream_t stream);

// Up to kLayoutCopyMaxBatch plans in one launch: they must share S, Z1, Z0,
// unit_bytes and streaming, and write disjoint bytes (their blocks run in any
// order).
constexpr int kLayoutCopyMaxBatch = 8;
cudaError_t launch_layout_copy_batch(const LayoutCopyPlan* plans, int n, cudaStream_t stream);

// Debug build: accesses the copy kernels skipped because they fell outside a
// plan's byte ranges (reset to 0 when `reset`).  Synchronises the device.
// cudaErrorNotSupported in the release build.
cudaError_t layout_copy_bounds_violations(unsigned long long* count, bool reset);

}  // namespace qnre
