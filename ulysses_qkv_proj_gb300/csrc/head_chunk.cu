// head_chunk.cu -- head-chunk pack and merge ("Head-Chunk Layout and Transport
// Primitives", flashinfer.comm API reference: pack_ulysses_qkv_head_chunk and
// merge_ulysses_output_head_chunk) as memory-bound copy kernels for sm_103a.
//
// Both are gathers of whole D-element head rows.  The grid is
//   x: one "segment" = one (slot, component) head row of the output,
//   y: a run of sequence positions, z: batch,
// so blocks that run together cover every segment of the same rows: the
// output rows are written as long contiguous runs and the source rows are read
// as 2*D-byte pieces.  Each thread copies 16-byte vectors (when the rows are
// 16-byte aligned with unit innermost stride) at a fixed column of the segment
// while it walks the rows, so the index arithmetic is hoisted out of the loop;
// four rows are in flight per thread.  Offsets are 64-bit.
#include "head_chunk.cuh"

#include <cuda_runtime.h>

#include <cstdint>

namespace qnre {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

struct SegCopyArgs {
  // Source of the segment's rows: byte address of element (b, s=0, head, d=0)
  // is src_base[c] + b*src_sb[c] + head*src_sh[c]; rows advance by src_ss[c].
  const char* src[3];
  long long src_sb[3], src_ss[3], src_sh[3];
  long long src_sd;      // bytes between consecutive units along d
  char* dst;
  long long dst_sb, dst_ss;  // bytes (contiguous output)
  long long S;               // rows per batch entry
  int units;                 // units per segment row (D elements or D*esz/16 vectors)
  int rows_per_block;
  // segment decomposition
  int comps;        // 3 for pack (q|k|v), 1 for merge
  int head_count;   // heads per destination band
  int src_heads_per_rank;  // H_local (pack) or head_count (merge)
  int src_head_offset;     // head_offset (pack) or 0 (merge)
  int dst_heads_per_rank;  // head_count (pack) or local_heads (merge)
  int dst_head_offset;     // 0 (pack) or head_offset (merge)
  long long dst_seg_bytes; // bytes of one (head, comp) segment row in dst
};

template <typename U>
__global__ void __launch_bounds__(kThreads) seg_copy_kernel(const SegCopyArgs a) {
  const int seg = blockIdx.x;
  const int c = seg % a.comps;
  const int slot = seg / a.comps;                 // r*head_count + j
  const int r = slot / a.head_count;
  const int j = slot - r * a.head_count;
  const int src_head = r * a.src_heads_per_rank + a.src_head_offset + j;
  const int dst_head = r * a.dst_heads_per_rank + a.dst_head_offset + j;
  const long long b = blockIdx.z;
  const long long s_begin = static_cast<long long>(blockIdx.y) * a.rows_per_block;
  long long s_end = s_begin + a.rows_per_block;
  if (s_end > a.S) s_end = a.S;

  const char* src = a.src[c] + b * a.src_sb[c] + src_head * a.src_sh[c];
  char* dst = a.dst + b * a.dst_sb + static_cast<long long>(dst_head) * (a.dst_seg_bytes * a.comps) +
              static_cast<long long>(c) * a.dst_seg_bytes;
  const long long ss = a.src_ss[c];
  const long long ds = a.dst_ss;

  if (a.units <= kThreads) {
    const int rows_per_iter = kThreads / a.units;
    const int lr = threadIdx.x / a.units;
    const int u = threadIdx.x - lr * a.units;
    if (lr >= rows_per_iter) return;
    const char* sp = src + u * a.src_sd;
    char* dp = dst + static_cast<long long>(u) * sizeof(U);
    const long long step = rows_per_iter;
    for (long long s = s_begin + lr; s < s_end; s += step * kUnroll) {
      U v[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const long long sk = s + k * step;
        if (sk < s_end) v[k] = *reinterpret_cast<const U*>(sp + sk * ss);
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const long long sk = s + k * step;
        if (sk < s_end) *reinterpret_cast<U*>(dp + sk * ds) = v[k];
      }
    }
  } else {
    const long long n = (s_end - s_begin) * a.units;
    for (long long e = threadIdx.x; e < n; e += kThreads) {
      const long long s = s_begin + e / a.units;
      const long long u = e % a.units;
      *reinterpret_cast<U*>(dst + s * ds + u * static_cast<long long>(sizeof(U))) =
          *reinterpret_cast<const U*>(src + s * ss + u * a.src_sd);
    }
  }
}

}  // namespace

cudaError_t launch_seg_copy(const SegCopyPlan& p, cudaStream_t stream) {
  SegCopyArgs a{};
  for (int c = 0; c < 3; ++c) {
    a.src[c] = static_cast<const char*>(p.src[c]);
    a.src_sb[c] = p.src_sb[c];
    a.src_ss[c] = p.src_ss[c];
    a.src_sh[c] = p.src_sh[c];
  }
  a.src_sd = p.src_sd;
  a.dst = static_cast<char*>(p.dst);
  a.dst_sb = p.dst_sb;
  a.dst_ss = p.dst_ss;
  a.S = p.S;
  a.units = p.units;
  a.comps = p.comps;
  a.head_count = p.head_count;
  a.src_heads_per_rank = p.src_heads_per_rank;
  a.src_head_offset = p.src_head_offset;
  a.dst_heads_per_rank = p.dst_heads_per_rank;
  a.dst_head_offset = p.dst_head_offset;
  a.dst_seg_bytes = p.dst_seg_bytes;

  long long rows_per_block = 64;
  while ((p.S + rows_per_block - 1) / rows_per_block > 65535) rows_per_block *= 2;
  a.rows_per_block = static_cast<int>(rows_per_block);
  const dim3 grid(static_cast<unsigned>(p.segments),
                  static_cast<unsigned>((p.S + rows_per_block - 1) / rows_per_block),
                  static_cast<unsigned>(p.B));
  switch (p.unit_bytes) {
    case 16: seg_copy_kernel<uint4><<<grid, kThreads, 0, stream>>>(a); break;
    case 4: seg_copy_kernel<uint32_t><<<grid, kThreads, 0, stream>>>(a); break;
    case 2: seg_copy_kernel<uint16_t><<<grid, kThreads, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace qnre
