// layout_copy.cu -- the head-row copy kernel behind the Ulysses layout entry
// points ("Head-Chunk Layout and Transport Primitives" and "Ulysses
// Context-Parallel All-to-All", flashinfer.comm API reference), for sm_103a.
//
// Every one of those transforms moves whole D-element head rows between two
// layouts whose addresses are affine in (rank, head, batch, sequence), so one
// kernel serves them all.  The grid is
//   x: segment = (slot, component) head row,  y: runs of 128 sequence rows,
//   z: batch (split into two affine indices),
// so blocks that run together cover every segment of the same rows and the
// output is written as long contiguous runs.  Each thread copies 16-byte
// vectors (when rows are 16-byte aligned with unit innermost stride) at a fixed
// column of the segment while it walks the rows, so all index arithmetic is
// hoisted out of the loop; four rows are in flight per thread.  Offsets are
// 64-bit.  Plans marked `streaming` (the schedule calls, which run beside the
// projection) load and store with .cs: every copied byte is touched once, so
// its lines are the first to leave L2 and the tensor-core kernel beside the
// copy keeps more of its operands there; other plans use the default policy,
// which copies alone run about 2 % faster with.
//
// Launch overlap.  A launch of 100-300 MB loses about 5 us to its start (the
// previous grid's last blocks draining, then this grid's first loads filling
// the memory pipeline).  Every copy is a programmatic dependent launch: its
// blocks may be scheduled while the previous grid in the stream drains, and
// wait (griddepcontrol.wait) until that grid has completed and its writes are
// visible before they load anything the copy depends on.  Plans that run alone
// first ask L2 for the lines of their block's source rows (prefetch.global.L2, a
// hint with no effect on results: L2 is where this GPU keeps global memory
// coherent, so a line written by the previous grid is current there), so their
// DRAM reads overlap that drain.  Measured at the pages' shape: the per-chunk
// merge 84 -> 95 % and the output sequence pack 84 -> 93 % of the copy rate.
#include "layout_copy.cuh"

#include "debug_bounds.cuh"

#include <cuda_runtime.h>

#include <cstdint>

namespace qnre {
namespace {

#ifndef QNRE_COPY_UNROLL
#define QNRE_COPY_UNROLL 4
#endif
#ifndef QNRE_COPY_ROWS
#define QNRE_COPY_ROWS 128
#endif
#ifndef QNRE_COPY_PDL
#define QNRE_COPY_PDL 1  // launches may begin while the previous grid in the stream drains
#endif
#ifndef QNRE_COPY_PREFETCH
// plans that run alone prefetch their source rows into L2 before that wait (not
// in the debug build, whose point is that every address is checked before use)
#define QNRE_COPY_PREFETCH (!QNRE_DEBUG_BOUNDS)
#endif
constexpr int kThreads = 256;
constexpr int kUnroll = QNRE_COPY_UNROLL;  // rows in flight per thread
constexpr int kMaxBatch = kLayoutCopyMaxBatch;

struct Args {
  const char* src[3];
  long long src_rank[3], src_head[3], src_z1[3], src_z0[3], src_s[3];
  long long src_unit;
  int src_head_offset;
  char* dst;
  long long dst_rank, dst_head, dst_comp, dst_z1, dst_z0, dst_s;
  int dst_head_offset;
  int Z0;  // z = z1 * Z0 + z0 < 65536 (grid z)
  long long S;
  int rows_per_block;
  int head_count, comps, units;
#if QNRE_DEBUG_BOUNDS
  Extent src_ext[3], dst_ext;
#endif
};

#define QNRE_SRC_OK(p) QNRE_ACCESS_OK((p), sizeof(U), a.src_ext[c])
#define QNRE_DST_OK(p) QNRE_ACCESS_OK((p), sizeof(U), a.dst_ext)

__device__ __forceinline__ void prefetch_l2(const char* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <typename U, bool kStream>
__device__ __forceinline__ U ld_row(const char* p) {
  if constexpr (kStream) return __ldcs(reinterpret_cast<const U*>(p));
  else return *reinterpret_cast<const U*>(p);
}
template <typename U, bool kStream>
__device__ __forceinline__ void st_row(char* p, const U& v) {
  if constexpr (kStream) __stcs(reinterpret_cast<U*>(p), v);
  else *reinterpret_cast<U*>(p) = v;
}

// Rows [y * rows_per_block, +rows_per_block) of segment `seg` of batch row z.
// With kPrefetchOnly the block only asks L2 for the 128-byte lines of its source
// rows (a hint with no effect on results: L2 is where this GPU's global memory is
// kept coherent) and copies nothing.
template <typename U, bool kStream, bool kPrefetchOnly = false>
__device__ __forceinline__ void copy_block(const Args& a, int seg, int y, int z) {
  // 32-bit index arithmetic (every grid index fits); byte offsets are 64-bit
  const int slot = seg / a.comps;
  const int c = seg - slot * a.comps;
  const int r = slot / a.head_count;
  const int j = slot - r * a.head_count;
  const int z1 = z / a.Z0;
  const int z0 = z - z1 * a.Z0;
  const long long s_begin = static_cast<long long>(y) * a.rows_per_block;
  long long s_end = s_begin + a.rows_per_block;
  if (s_end > a.S) s_end = a.S;

  const char* src = a.src[c] + r * a.src_rank[c] + static_cast<long long>(a.src_head_offset + j) * a.src_head[c] +
                    z1 * a.src_z1[c] + z0 * a.src_z0[c];
  char* dst = a.dst + r * a.dst_rank + static_cast<long long>(a.dst_head_offset + j) * a.dst_head +
              static_cast<long long>(c) * a.dst_comp + z1 * a.dst_z1 + z0 * a.dst_z0;
  const long long ss = a.src_s[c];
  const long long ds = a.dst_s;

  if (a.units <= kThreads) {
    const int rows_per_iter = kThreads / a.units;
    const int lr = threadIdx.x / a.units;
    const int u = threadIdx.x - lr * a.units;
    if (lr >= rows_per_iter) return;
    const char* sp = src + u * a.src_unit;
    char* dp = dst + static_cast<long long>(u) * sizeof(U);
    const long long step = rows_per_iter;
    if constexpr (kPrefetchOnly) {
      if ((u * a.src_unit) % 128 == 0)
        for (long long s = s_begin + lr; s < s_end; s += step) prefetch_l2(sp + s * ss);
    } else {
      for (long long s = s_begin + lr; s < s_end; s += step * kUnroll) {
        U v[kUnroll];
        bool ok[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
          const long long sk = s + k * step;
          ok[k] = sk < s_end && QNRE_SRC_OK(sp + sk * ss);
          if (ok[k]) v[k] = ld_row<U, kStream>(sp + sk * ss);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
          const long long sk = s + k * step;
          if (ok[k] && QNRE_DST_OK(dp + sk * ds)) st_row<U, kStream>(dp + sk * ds, v[k]);
        }
      }
    }
  } else if constexpr (!kPrefetchOnly) {
    const long long n = (s_end - s_begin) * a.units;
    for (long long e = threadIdx.x; e < n; e += kThreads) {
      const long long s = s_begin + e / a.units;
      const long long u = e % a.units;
      const char* sp = src + s * ss + u * a.src_unit;
      char* dp = dst + s * ds + u * static_cast<long long>(sizeof(U));
      if (QNRE_SRC_OK(sp) && QNRE_DST_OK(dp)) st_row<U, kStream>(dp, ld_row<U, kStream>(sp));
    }
  }
}

// Programmatic dependent launch: wait until the grid this launch depends on has
// completed and its writes are visible (a no-op without such a dependency), then
// let the next launch in the stream begin its own set-up.
__device__ __forceinline__ void pdl_enter() {
#if QNRE_COPY_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

template <typename U, bool kStream>
__global__ void __launch_bounds__(kThreads) layout_copy_kernel(const Args a) {
  if (QNRE_COPY_PREFETCH && !kStream) copy_block<U, kStream, true>(a, blockIdx.x, blockIdx.y, blockIdx.z);
  pdl_enter();
  copy_block<U, kStream>(a, blockIdx.x, blockIdx.y, blockIdx.z);
}

// Several plans with the same rows and batch extents in one launch: block x
// runs segment blockIdx.x - first[p] of plan p.
struct BatchArgs {
  Args plan[kMaxBatch];
  int first[kMaxBatch + 1];  // first block of each plan; first[n] = grid x
  int n;
};

template <typename U, bool kStream>
__global__ void __launch_bounds__(kThreads) layout_copy_batch_kernel(const __grid_constant__ BatchArgs b) {
  const int x = blockIdx.x;
  int p = 0;
  while (p + 1 < b.n && x >= b.first[p + 1]) ++p;
  if (QNRE_COPY_PREFETCH && !kStream) copy_block<U, kStream, true>(b.plan[p], x - b.first[p], blockIdx.y, blockIdx.z);
  pdl_enter();
  copy_block<U, kStream>(b.plan[p], x - b.first[p], blockIdx.y, blockIdx.z);
}

}  // namespace

namespace {

// Kernel arguments of one plan; false when a grid extent is out of range.
bool make_args(const LayoutCopyPlan& p, Args* out, long long* segments) {
  Args a{};
  for (int c = 0; c < 3; ++c) {
    a.src[c] = static_cast<const char*>(p.src[c]);
    a.src_rank[c] = p.src_rank[c];
    a.src_head[c] = p.src_head[c];
    a.src_z1[c] = p.src_z1[c];
    a.src_z0[c] = p.src_z0[c];
    a.src_s[c] = p.src_s[c];
  }
  a.src_unit = p.src_unit;
  a.src_head_offset = p.src_head_offset;
  a.dst = static_cast<char*>(p.dst);
  a.dst_rank = p.dst_rank;
  a.dst_head = p.dst_head;
  a.dst_comp = p.dst_comp;
  a.dst_z1 = p.dst_z1;
  a.dst_z0 = p.dst_z0;
  a.dst_s = p.dst_s;
  a.dst_head_offset = p.dst_head_offset;
  a.S = p.S;
  a.head_count = p.head_count;
  a.comps = p.comps;
  a.units = p.units;
#if QNRE_DEBUG_BOUNDS
  if (p.dst_hi <= p.dst_lo) return false;  // the debug build checks every plan
  for (int c = 0; c < p.comps; ++c) {
    if (p.src_hi[c] <= p.src_lo[c]) return false;
    a.src_ext[c] = Extent{p.src_lo[c], p.src_hi[c]};
  }
  a.dst_ext = output_extent(p.dst_lo, p.dst_hi);
#endif

  // 128 rows per block: on the few SMs that copies get beside the persistent
  // fused kernel, longer blocks amortise each block's start-up (measured: the
  // benchmarked step 3.6 % shorter; full-GPU copies of the pages' shape 1.3 %
  // slower than with 64-row blocks, still 97 % of the measured copy rate)
  long long rows_per_block = QNRE_COPY_ROWS;
  while ((p.S + rows_per_block - 1) / rows_per_block > 65535) rows_per_block *= 2;
  a.rows_per_block = static_cast<int>(rows_per_block);
  *segments = static_cast<long long>(p.ranks) * p.head_count * p.comps;
  const long long zs = p.Z1 * p.Z0;
  if (*segments > 0x7FFFFFFFll || zs > 65535) return false;
  a.Z0 = static_cast<int>(p.Z0);
  *out = a;
  return true;
}

dim3 rows_grid(const LayoutCopyPlan& p, const Args& a, long long x) {
  return dim3(static_cast<unsigned>(x), static_cast<unsigned>((p.S + a.rows_per_block - 1) / a.rows_per_block),
              static_cast<unsigned>(p.Z1 * p.Z0));
}

}  // namespace

// Launch `kernel` on `grid` x kThreads, as a programmatic dependent launch when
// QNRE_COPY_PDL is on.
template <typename... KArgs, typename... Args2>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, cudaStream_t stream, Args2&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
#if QNRE_COPY_PDL
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
#else
  (void)attr;
#endif
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args2>(args)...);
}

template <typename U, bool kStream>
cudaError_t launch_one(const LayoutCopyPlan& p, const Args& a, long long segments, cudaStream_t stream) {
  return launch(layout_copy_kernel<U, kStream>, rows_grid(p, a, segments), stream, a);
}

cudaError_t launch_layout_copy(const LayoutCopyPlan& p, cudaStream_t stream) {
  if (p.S <= 0 || p.Z1 <= 0 || p.Z0 <= 0) return cudaSuccess;
  Args a;
  long long segments = 0;
  if (!make_args(p, &a, &segments)) return cudaErrorInvalidValue;
  const bool st = p.streaming != 0;
  switch (p.unit_bytes) {
    case 16: return st ? launch_one<uint4, true>(p, a, segments, stream) : launch_one<uint4, false>(p, a, segments, stream);
    case 4:
      return st ? launch_one<uint32_t, true>(p, a, segments, stream)
                : launch_one<uint32_t, false>(p, a, segments, stream);
    case 2:
      return st ? launch_one<uint16_t, true>(p, a, segments, stream)
                : launch_one<uint16_t, false>(p, a, segments, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_layout_copy_batch(const LayoutCopyPlan* plans, int n, cudaStream_t stream) {
  if (n < 1 || n > kMaxBatch) return cudaErrorInvalidValue;
  const LayoutCopyPlan& p0 = plans[0];
  for (int i = 1; i < n; ++i) {
    if (plans[i].S != p0.S || plans[i].Z1 != p0.Z1 || plans[i].Z0 != p0.Z0 ||
        plans[i].unit_bytes != p0.unit_bytes || plans[i].streaming != p0.streaming)
      return cudaErrorInvalidValue;
  }
  if (p0.S <= 0 || p0.Z1 <= 0 || p0.Z0 <= 0) return cudaSuccess;
  BatchArgs b{};
  long long x = 0;
  for (int i = 0; i < n; ++i) {
    long long segments = 0;
    if (!make_args(plans[i], &b.plan[i], &segments)) return cudaErrorInvalidValue;
    b.first[i] = static_cast<int>(x);
    x += segments;
    if (x > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  }
  b.first[n] = static_cast<int>(x);
  b.n = n;
  const dim3 grid = rows_grid(p0, b.plan[0], x);
  const bool st = p0.streaming != 0;
  switch (p0.unit_bytes) {
    case 16:
      return st ? launch(layout_copy_batch_kernel<uint4, true>, grid, stream, b)
                : launch(layout_copy_batch_kernel<uint4, false>, grid, stream, b);
    case 4:
      return st ? launch(layout_copy_batch_kernel<uint32_t, true>, grid, stream, b)
                : launch(layout_copy_batch_kernel<uint32_t, false>, grid, stream, b);
    case 2:
      return st ? launch(layout_copy_batch_kernel<uint16_t, true>, grid, stream, b)
                : launch(layout_copy_batch_kernel<uint16_t, false>, grid, stream, b);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t layout_copy_bounds_violations(unsigned long long* count, bool reset) {
#if QNRE_DEBUG_BOUNDS
  return read_bounds_violations(count, reset);
#else
  *count = 0;
  (void)reset;
  return cudaErrorNotSupported;
#endif
}

}  // namespace qnre
