// head_chunk.cuh -- launcher of the segment-copy kernel behind the head-chunk
// pack and merge entry points.
#pragma once

#include <cuda_runtime.h>

namespace qnre {

// One launch copies `segments` head rows per (b, s): segment = slot*comps + c,
// slot = r*head_count + j.  All strides are in bytes.
struct SegCopyPlan {
  const void* src[3];
  long long src_sb[3], src_ss[3], src_sh[3];
  long long src_sd;           // bytes between consecutive copy units along d
  void* dst;
  long long dst_sb, dst_ss;   // contiguous destination
  long long B, S;
  int segments;
  int units;                  // copy units per head row
  int unit_bytes;             // 16 (vector path), 4 or 2 (element path)
  int comps;
  int head_count;
  int src_heads_per_rank, src_head_offset;
  int dst_heads_per_rank, dst_head_offset;
  long long dst_seg_bytes;    // bytes of one head row (D elements) in dst
};

cudaError_t launch_seg_copy(const SegCopyPlan& plan, cudaStream_t stream);

}  // namespace qnre
