// qnre_api.cu -- the extern "C" boundary of libqnre: argument checks, the plan
// object, TMA descriptor encoding and kernel launches.  Every check runs before
// anything is enqueued, so a rejected call has no effect.
#include "../../include/qnre.h"
#include "fused_qkv.cuh"
#include "api_util.cuh"
#include "layout_copy.cuh"
#include "debug_bounds.cuh"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#ifndef QNRE_RASTER_L2_MB
#define QNRE_RASTER_L2_MB 32  // L2 share for the resident x panels of a row-tile group
#endif
#include <cstdint>
#include <mutex>
#include <new>

namespace qnre {
cudaError_t sage2_bounds_violations(unsigned long long* count, bool reset);  // sage2.cu
}

struct qnre_plan_s {
  int hidden = 0;
  int num_heads = 0;
  int P = 0;
  int H_local = 0;
  qnre_layout_t layout = QNRE_LAYOUT_BSHD;
  int64_t max_tokens = 0;
  qnre_rope_t rope_style = QNRE_ROPE_ROTATE_HALF;
  unsigned flags = 0;
  int device = -1;
  int max_pairs = 0;  // CTA pairs the fused kernel runs (all_pairs minus any reserved)
  int all_pairs = 0;  // CTA pairs of the fused kernel that fit on the device at once
  int max_quads = 0;  // the same for clusters of two pairs (QNRE_FLAG_W_MULTICAST)
  int all_quads = 0;
  unsigned* d_status = nullptr;
};

namespace {

using namespace qnre;
using qnre::FusedArgs;

using api::aligned;
using api::ByteRange;
using api::from_cuda;
using api::overlaps;
using api::span;

// ------------------------------------------------------------------ TMA maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}

// 2-D bf16 row-major matrix [rows, cols], box = box_cols x box_rows, 128-byte swizzle.
bool encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                    uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Head-band output for TMA stores: bf16 [rows, H_local, width] (width 128 for a
// bshd q/k/v tensor, 384 for the fused payload), box 64 x 1 x 32 with the
// 128-byte swizzle the epilogue's staging uses.
bool encode_out_bf16(CUtensorMap* map, void* base, uint64_t rows, uint64_t H_local, uint64_t width) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {width, H_local, rows};
  const cuuint64_t strides[2] = {width * 2, H_local * width * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(qnre::kStoreRows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

const char* qnre_status_string(qnre_status_t s) {
  switch (s) {
    case QNRE_OK: return "QNRE_OK";
    case QNRE_ERR_INVALID_ARG: return "QNRE_ERR_INVALID_ARG: invalid argument";
    case QNRE_ERR_UNSUPPORTED: return "QNRE_ERR_UNSUPPORTED: unsupported configuration";
    case QNRE_ERR_ALIGNMENT: return "QNRE_ERR_ALIGNMENT: misaligned pointer or stride";
    case QNRE_ERR_ALIAS: return "QNRE_ERR_ALIAS: output overlaps an input";
    case QNRE_ERR_CAPACITY: return "QNRE_ERR_CAPACITY: size beyond the plan or index limits";
    case QNRE_ERR_CUDA: return "QNRE_ERR_CUDA: CUDA call failed";
    case QNRE_ERR_DEVICE: return "QNRE_ERR_DEVICE: device-side check fired";
  }
  return "QNRE_ERR_UNKNOWN";
}

qnre_status_t qnre_plan_create(qnre_plan_t* plan, int hidden, int num_heads, int head_dim, int P,
                               qnre_layout_t layout, int64_t max_tokens, qnre_rope_t rope_style,
                               unsigned flags) {
  if (plan == nullptr) return QNRE_ERR_INVALID_ARG;
  if (head_dim != QNRE_HEAD_DIM) return head_dim > 0 ? QNRE_ERR_UNSUPPORTED : QNRE_ERR_INVALID_ARG;
  if (num_heads < 1 || P < 1 || hidden < 1) return QNRE_ERR_INVALID_ARG;
  if (hidden != num_heads * head_dim || hidden % 64 != 0) return QNRE_ERR_INVALID_ARG;
  if (num_heads % P != 0) return QNRE_ERR_INVALID_ARG;
  if (layout != QNRE_LAYOUT_BSHD && layout != QNRE_LAYOUT_FUSED) return QNRE_ERR_INVALID_ARG;
  if (rope_style != QNRE_ROPE_ROTATE_HALF && rope_style != QNRE_ROPE_INTERLEAVED) return QNRE_ERR_INVALID_ARG;
  if ((flags & ~(QNRE_FLAG_EPILOGUE_OFF | QNRE_FLAG_W_MULTICAST | QNRE_FLAG_ONE_PAIR)) != 0) return QNRE_ERR_INVALID_ARG;
  if ((flags & QNRE_FLAG_W_MULTICAST) && (flags & QNRE_FLAG_ONE_PAIR)) return QNRE_ERR_INVALID_ARG;
  if (max_tokens < 1) return QNRE_ERR_INVALID_ARG;
  // The kernel's tile indices and TMA coordinates are 32-bit.
  if (max_tokens * static_cast<int64_t>(P) > (int64_t{1} << 31) - 256) return QNRE_ERR_CAPACITY;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return QNRE_ERR_CUDA;
  int major = 0, minor = 0, pairs = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return QNRE_ERR_CUDA;
  if (major != 10 || minor != 3) return QNRE_ERR_UNSUPPORTED;
  int quads = 0;
  if (qnre::prepare_fused_qkv_kernel(&pairs, &quads) != cudaSuccess) return QNRE_ERR_CUDA;
  if ((flags & QNRE_FLAG_W_MULTICAST) && quads < 1) return QNRE_ERR_UNSUPPORTED;
  if (encode_tiled_fn() == nullptr) return QNRE_ERR_CUDA;

  qnre_plan_s* p = new (std::nothrow) qnre_plan_s();
  if (p == nullptr) return QNRE_ERR_CUDA;
  if (cudaMalloc(&p->d_status, 16) != cudaSuccess) {
    delete p;
    return QNRE_ERR_CUDA;
  }
  if (cudaMemset(p->d_status, 0, 16) != cudaSuccess) {
    cudaFree(p->d_status);
    delete p;
    return QNRE_ERR_CUDA;
  }
  p->hidden = hidden;
  p->num_heads = num_heads;
  p->P = P;
  p->H_local = num_heads / P;
  p->layout = layout;
  p->max_tokens = max_tokens;
  p->rope_style = rope_style;
  p->flags = flags;
  p->device = dev;
  p->max_pairs = pairs;
  p->all_pairs = pairs;
  p->max_quads = quads;
  p->all_quads = quads;
  *plan = p;
  return QNRE_OK;
}

qnre_status_t qnre_plan_reserve_sms(qnre_plan_t plan, int sms) {
  if (plan == nullptr || sms < 0) return QNRE_ERR_INVALID_ARG;
  const int free_pairs = sms / 2 + sms % 2;  // SMs come free two at a time (one CTA pair)
  if (free_pairs >= plan->all_pairs) return QNRE_ERR_INVALID_ARG;
  plan->max_pairs = plan->all_pairs - free_pairs;
  const int free_quads = sms / 4 + (sms % 4 != 0 ? 1 : 0);  // four SMs at a time with two pairs per cluster
  plan->max_quads = plan->all_quads > free_quads ? plan->all_quads - free_quads : std::min(plan->all_quads, 1);
  return QNRE_OK;
}

qnre_status_t qnre_plan_destroy(qnre_plan_t plan) {
  if (plan == nullptr) return QNRE_OK;
  cudaError_t e = cudaSuccess;
  if (plan->d_status != nullptr) e = cudaFree(plan->d_status);
  delete plan;
  return from_cuda(e);
}

}  // extern "C"

namespace {

// The form a forward takes: clusters of one pair, or of two pairs sharing W
// through multicast (forced by a flag, else chosen when such clusters fit and
// the row tiles pair up: an odd last row tile is paired with an empty one, so
// odd counts take it only when that waste is small), and its work list.
struct LaunchShape {
  int pairs_per_cluster;  // 1 or 2
  int units;              // clusters launched
  int num_mp_tiles;       // row units of the raster
  int group_m;            // raster group, in row units
  int num_full, num_work; // whole items, all items (whole + halves)
};

// Longest load of any unit, in half tiles, when `units` units take the work
// list of qnre::plan_work round robin (unit u: items u, u + units, ...; items
// below num_full are whole tiles, the rest halves).  A unit's load is its whole
// tiles plus its items, and unit 0 has the most of both.
int makespan_halves(int num_full, int num_work, int units) {
  return (num_full + units - 1) / units + (num_work + units - 1) / units;
}

// The fewest units (<= max_units) whose work list finishes in as many half-tile
// rounds as max_units would: the SMs this leaves idle stay with kernels on
// other streams (the head-chunk copies beside the projection) at no cost to
// the projection.
int fewest_units(int num_tiles, int max_units, int* num_full, int* num_work) {
  qnre::plan_work(num_tiles, max_units, num_full, num_work);
  int best = std::min(*num_work, max_units);
  const int target = makespan_halves(*num_full, *num_work, best);
  for (int c = best - 1; c >= 1 && static_cast<long long>(c) * target >= 2LL * num_tiles; --c) {
    int nf = 0, nw = 0;
    qnre::plan_work(num_tiles, c, &nf, &nw);
    const int u = std::min(nw, c);
    if (makespan_halves(nf, nw, u) <= target) {
      best = u;
      *num_full = nf;
      *num_work = nw;
    }
  }
  return best;
}

LaunchShape launch_shape(const qnre_plan_s* plan, int m_tiles, int n_tiles, int group_m) {
  LaunchShape ls{};
  const bool multicast = !(plan->flags & QNRE_FLAG_ONE_PAIR) && plan->max_quads >= 1 &&
                         ((plan->flags & QNRE_FLAG_W_MULTICAST) || m_tiles % 2 == 0 || m_tiles >= 16);
  if (multicast) {
    // work item = (pair of adjacent row tiles, column tile); a short last round
    // is split into 256 x 128 halves like the one-pair kernel's
    ls.pairs_per_cluster = 2;
    ls.num_mp_tiles = (m_tiles + 1) / 2;
    ls.group_m = std::max(1, (group_m + 1) / 2);
    ls.units = fewest_units(ls.num_mp_tiles * n_tiles, plan->max_quads, &ls.num_full, &ls.num_work);
  } else {
    ls.pairs_per_cluster = 1;
    ls.num_mp_tiles = m_tiles;
    ls.group_m = group_m;
    ls.units = fewest_units(m_tiles * n_tiles, plan->max_pairs, &ls.num_full, &ls.num_work);
  }
  return ls;
}

// The fused forward; `ready` (device [P] words, or null) receives the
// per-destination publication counts.
qnre_status_t forward_impl(qnre_plan_t plan, int B, int S_local, const void* x, const void* w_qkv,
                           const void* q_norm_w, const void* k_norm_w, const float* cos_sin, int64_t n_pos,
                           const int32_t* positions, const qnre_out_t* out, unsigned* ready, qnre_stream_t stream) {
  if (plan == nullptr || out == nullptr) return QNRE_ERR_INVALID_ARG;
  if (B < 0 || S_local < 0) return QNRE_ERR_INVALID_ARG;
  const int64_t tokens_per_rank = static_cast<int64_t>(B) * S_local;
  if (tokens_per_rank > plan->max_tokens) return QNRE_ERR_CAPACITY;
  if (tokens_per_rank == 0) return QNRE_OK;
  if (x == nullptr || w_qkv == nullptr || q_norm_w == nullptr || k_norm_w == nullptr || cos_sin == nullptr)
    return QNRE_ERR_INVALID_ARG;
  if (n_pos < 1) return QNRE_ERR_INVALID_ARG;
  const bool bshd = plan->layout == QNRE_LAYOUT_BSHD;
  if (bshd ? (out->q == nullptr || out->k == nullptr || out->v == nullptr) : out->fused == nullptr)
    return QNRE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_qkv, 16) || !aligned(q_norm_w, 16) || !aligned(k_norm_w, 16) ||
      !aligned(cos_sin, 16) || (positions != nullptr && !aligned(positions, 4)))
    return QNRE_ERR_ALIGNMENT;
  if (bshd ? (!aligned(out->q, 16) || !aligned(out->k, 16) || !aligned(out->v, 16)) : !aligned(out->fused, 16))
    return QNRE_ERR_ALIGNMENT;

  const int P = plan->P;
  const int64_t T = tokens_per_rank * P;
  const int64_t K = plan->hidden;
  const int64_t N = 3 * K;
  if (n_pos > (int64_t{1} << 40)) return QNRE_ERR_CAPACITY;

  // Storage ranges: outputs must not overlap any input, nor each other.
  const uint64_t band_bytes = static_cast<uint64_t>(T) * K * 2;  // one of q/k/v over all ranks
  const ByteRange in[6] = {span(x, static_cast<uint64_t>(T) * K * 2), span(w_qkv, static_cast<uint64_t>(K) * N * 2),
                           span(q_norm_w, 256), span(k_norm_w, 256),
                           span(cos_sin, static_cast<uint64_t>(n_pos) * 512),
                           positions ? span(positions, static_cast<uint64_t>(T) * 4) : ByteRange{0, 0}};
  ByteRange outs[3];
  int n_out = 0;
  if (bshd) {
    outs[n_out++] = span(out->q, band_bytes);
    outs[n_out++] = span(out->k, band_bytes);
    outs[n_out++] = span(out->v, band_bytes);
  } else {
    outs[n_out++] = span(out->fused, 3 * band_bytes);
  }
  for (int i = 0; i < n_out; ++i) {
    for (const ByteRange& r : in)
      if (r.hi > r.lo && overlaps(outs[i], r)) return QNRE_ERR_ALIAS;
    for (int j = i + 1; j < n_out; ++j)
      if (overlaps(outs[i], outs[j])) return QNRE_ERR_ALIAS;
  }
  if (ready != nullptr) {
    if (!aligned(ready, 4)) return QNRE_ERR_ALIGNMENT;
    const ByteRange rr = span(ready, static_cast<uint64_t>(P) * 4);
    for (const ByteRange& r : in)
      if (r.hi > r.lo && overlaps(rr, r)) return QNRE_ERR_ALIAS;
    for (int i = 0; i < n_out; ++i)
      if (overlaps(rr, outs[i])) return QNRE_ERR_ALIAS;
  }

  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return QNRE_ERR_CUDA;
  if (cur != plan->device) return QNRE_ERR_INVALID_ARG;

  FusedArgs a;
  if (!encode_2d_bf16(&a.tmap_x, x, static_cast<uint64_t>(T), static_cast<uint64_t>(K), qnre::kBK, qnre::kBM))
    return QNRE_ERR_CUDA;
  if (!encode_2d_bf16(&a.tmap_w, w_qkv, static_cast<uint64_t>(K), static_cast<uint64_t>(N), 64, qnre::kBK))
    return QNRE_ERR_CUDA;
  a.q_norm_w = static_cast<const uint16_t*>(q_norm_w);
  a.k_norm_w = static_cast<const uint16_t*>(k_norm_w);
  a.cos_sin = cos_sin;
  a.positions = positions;
  a.out_q = static_cast<uint16_t*>(bshd ? out->q : nullptr);
  a.out_k = static_cast<uint16_t*>(bshd ? out->k : nullptr);
  a.out_v = static_cast<uint16_t*>(bshd ? out->v : nullptr);
  a.out_fused = static_cast<uint16_t*>(bshd ? nullptr : out->fused);
  a.status = plan->d_status;
  a.ready = ready;
  // TMA stores of whole 32-row head tiles (their row coordinate is 32-bit); the
  // debug build and the publishing form store rows one by one.
  {
    const int64_t band_rows = T * P;  // P * B * S_global rows of each band tensor
    bool ok = !QNRE_DEBUG_BOUNDS && ready == nullptr && band_rows < (int64_t{1} << 31);
    if (ok && bshd) {
      ok = encode_out_bf16(&a.tmap_out[0], out->q, band_rows, plan->H_local, 128) &&
           encode_out_bf16(&a.tmap_out[1], out->k, band_rows, plan->H_local, 128) &&
           encode_out_bf16(&a.tmap_out[2], out->v, band_rows, plan->H_local, 128);
    } else if (ok) {
      ok = encode_out_bf16(&a.tmap_out[0], out->fused, band_rows, plan->H_local, 384);
    }
    a.tma_store = ok ? 1 : 0;
  }
  // [P, B, P*S_local, H_local, D] = T * H * D elements (T = P*B*S_local tokens)
  a.out_elems = static_cast<long long>(T) * plan->num_heads * (bshd ? 128 : 384);
#if QNRE_DEBUG_BOUNDS
  {
    const long long shrink = static_cast<long long>(qnre::debug_shrink_bytes() / 2);
    a.out_elems -= shrink < a.out_elems ? shrink : a.out_elems;
  }
#endif
  a.n_pos = n_pos;
  a.T = static_cast<int>(T);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.H = plan->num_heads;
  a.H_local = plan->H_local;
  a.P = P;
  a.B = B;
  a.S = S_local;
  a.layout = bshd ? 0 : 1;
  a.rope_style = plan->rope_style == QNRE_ROPE_INTERLEAVED ? 1 : 0;
  a.epilogue_on = (plan->flags & QNRE_FLAG_EPILOGUE_OFF) ? 0 : 1;
  const int64_t m_tiles = (T + qnre::kPairM - 1) / qnre::kPairM;
  const int64_t n_tiles = (N + qnre::kBN - 1) / qnre::kBN;
  if (m_tiles * n_tiles > INT32_MAX) return QNRE_ERR_CAPACITY;
  a.num_m_tiles = static_cast<int>(m_tiles);
  a.num_n_tiles = static_cast<int>(n_tiles);
  a.num_tiles = a.num_m_tiles * a.num_n_tiles;
  // Raster: groups of group_m row tiles sweep every column tile, rows fastest.
  // The group's x panels (256 rows x hidden each) stay resident in L2 while W
  // streams past; keep them to about 32 MB of the 129 MB L2 (a budget of 28-32
  // MB ran the 32768-token, hidden-8192 projection fastest both alone and under
  // the power cap; 16, 40 and 48 MB were slower).
  const int64_t panel_bytes = static_cast<int64_t>(qnre::kPairM) * K * 2;
  a.group_m = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>(m_tiles, (static_cast<int64_t>(QNRE_RASTER_L2_MB) << 20) / panel_bytes)));
  a.num_k_blocks = static_cast<int>(K / qnre::kBK);
  const LaunchShape ls = launch_shape(plan, a.num_m_tiles, a.num_n_tiles, a.group_m);
  const bool multicast = ls.pairs_per_cluster == 2;
  const int units = ls.units;
  a.num_mp_tiles = ls.num_mp_tiles;
  a.group_m = ls.group_m;
  a.num_full = ls.num_full;
  a.num_work = ls.num_work;
  if (ready != nullptr &&
      cudaMemsetAsync(ready, 0, static_cast<size_t>(P) * 4, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QNRE_ERR_CUDA;
  return from_cuda(qnre::launch_fused_qkv(a, units, multicast ? 2 : 1, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

qnre_status_t qnre_forward(qnre_plan_t plan, int B, int S_local, const void* x, const void* w_qkv,
                           const void* q_norm_w, const void* k_norm_w, const float* cos_sin, int64_t n_pos,
                           const int32_t* positions, const qnre_out_t* out, qnre_stream_t stream) {
  return forward_impl(plan, B, S_local, x, w_qkv, q_norm_w, k_norm_w, cos_sin, n_pos, positions, out, nullptr,
                      stream);
}

qnre_status_t qnre_forward_publish(qnre_plan_t plan, int B, int S_local, const void* x, const void* w_qkv,
                                   const void* q_norm_w, const void* k_norm_w, const float* cos_sin, int64_t n_pos,
                                   const int32_t* positions, const qnre_out_t* out, unsigned* ready,
                                   qnre_stream_t stream) {
  if (ready == nullptr) return QNRE_ERR_INVALID_ARG;
  return forward_impl(plan, B, S_local, x, w_qkv, q_norm_w, k_norm_w, cos_sin, n_pos, positions, out, ready,
                      stream);
}

qnre_status_t qnre_plan_describe(qnre_plan_t plan, int B, int S_local, qnre_plan_info_t* info) {
  if (plan == nullptr || info == nullptr || B < 0 || S_local < 0) return QNRE_ERR_INVALID_ARG;
  const int64_t tokens_per_rank = static_cast<int64_t>(B) * S_local;
  if (tokens_per_rank > plan->max_tokens) return QNRE_ERR_CAPACITY;
  qnre_plan_info_t r{};
  r.device = plan->device;
  if (tokens_per_rank > 0) {
    const int64_t T = tokens_per_rank * plan->P;
    const int64_t N = 3 * static_cast<int64_t>(plan->num_heads) * QNRE_HEAD_DIM;
    r.row_tiles = static_cast<int>((T + qnre::kPairM - 1) / qnre::kPairM);
    r.col_tiles = static_cast<int>((N + qnre::kBN - 1) / qnre::kBN);
    const LaunchShape ls = launch_shape(plan, r.row_tiles, r.col_tiles, 1);
    r.pairs_per_cluster = ls.pairs_per_cluster;
    r.clusters = ls.units;
    r.sms = ls.units * 2 * ls.pairs_per_cluster;
    r.work_items = ls.num_work;
    r.half_items = ls.num_work - ls.num_full;
    r.launches = 1;
  }
  *info = r;
  return QNRE_OK;
}

qnre_status_t qnre_ready_target(qnre_plan_t plan, int B, int S_local, unsigned* target) {
  if (plan == nullptr || target == nullptr || B < 0 || S_local < 0) return QNRE_ERR_INVALID_ARG;
  const int64_t T = static_cast<int64_t>(B) * S_local * plan->P;
  const int64_t m_tiles = (T + qnre::kPairM - 1) / qnre::kPairM;
  const unsigned long long t = qnre::ready_target(m_tiles, plan->H_local);
  if (t > 0xFFFFFFFFull) return QNRE_ERR_CAPACITY;
  *target = static_cast<unsigned>(t);
  return QNRE_OK;
}

qnre_status_t qnre_wait_ready(qnre_plan_t plan, const unsigned* ready, unsigned target, uint64_t timeout_ns,
                              qnre_stream_t stream) {
  if (plan == nullptr || ready == nullptr) return QNRE_ERR_INVALID_ARG;
  if (!aligned(ready, 4)) return QNRE_ERR_ALIGNMENT;
  if (plan->P > 1024) return QNRE_ERR_CAPACITY;
  if (timeout_ns == 0 || timeout_ns > 10ull * 1000ull * 1000ull * 1000ull) return QNRE_ERR_INVALID_ARG;
  return from_cuda(qnre::launch_wait_ready(ready, plan->P, target, timeout_ns, plan->d_status,
                                           QNRE_DEVICE_READY_TIMEOUT, reinterpret_cast<cudaStream_t>(stream)));
}

qnre_status_t qnre_plan_device_status(qnre_plan_t plan, qnre_stream_t stream, unsigned* bits, int clear) {
  if (plan == nullptr || bits == nullptr) return QNRE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned host = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return QNRE_ERR_CUDA;
  if (cudaMemcpy(&host, plan->d_status, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess)
    return QNRE_ERR_CUDA;
  if (clear && cudaMemset(plan->d_status, 0, sizeof(unsigned)) != cudaSuccess) return QNRE_ERR_CUDA;
  *bits = host;
  return host ? QNRE_ERR_DEVICE : QNRE_OK;
}

qnre_status_t qnre_debug_bounds(unsigned long long* violations, int reset) {
  if (violations == nullptr) return QNRE_ERR_INVALID_ARG;
  *violations = 0;
#if QNRE_DEBUG_BOUNDS
  unsigned long long copies = 0, sage2 = 0;
  if (qnre::layout_copy_bounds_violations(&copies, reset != 0) != cudaSuccess ||
      qnre::sage2_bounds_violations(&sage2, reset != 0) != cudaSuccess)
    return QNRE_ERR_CUDA;
  *violations = copies + sage2;
  return QNRE_OK;
#else
  (void)reset;
  return QNRE_ERR_UNSUPPORTED;
#endif
}

// --------------------------------------------------------------------------
// Allocation-free forward.  Some callers cannot call cudaMalloc at the point
// where they run the projection: code inside a framework's memory pool that
// forbids raw device allocations, a runtime that has handed all device memory
// to its own allocator, or a process that must not allocate once it is
// serving.  qnre_plan_create allocates the plan's status word with cudaMalloc,
// so those callers cannot make a plan.  qnre_forward_noalloc needs no plan: its
// only scratch is the status word, kept in the static device array below, and
// it makes no device allocation at all.
// --------------------------------------------------------------------------
namespace {

// Scratch of the allocation-free forward: every GPU that loads this library
// holds these 256 bytes until the process exits.  A call uses the first 16
// (one 4-byte status word, padded like the plan's).
constexpr size_t kNoAllocScratchBytes = 256;
constexpr size_t kNoAllocStatusBytes = 16;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
struct NoAllocDevice {
  bool ready = false;
  void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int max_pairs = 0;
};
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// One-time set-up per device, with that device current: the kernel's
// shared-memory opt-in and the device address of the static scratch array
// (the array's name is only a host-side stand-in in host code).
qnre_status_t noalloc_setup(int dev, NoAllocDevice* out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return QNRE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& st = g_noalloc_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0, pairs = 0, quads = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return QNRE_ERR_CUDA;
    if (major != 10 || minor != 3) return QNRE_ERR_UNSUPPORTED;
    if (qnre::prepare_fused_qkv_kernel(&pairs, &quads) != cudaSuccess) return QNRE_ERR_CUDA;
    if (encode_tiled_fn() == nullptr) return QNRE_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QNRE_ERR_CUDA;
    st.scratch = p;
    st.max_pairs = pairs;
    st.ready = true;
  }
  *out = st;
  return QNRE_OK;
}

}  // namespace

qnre_status_t qnre_forward_noalloc(int hidden, int num_heads, int P, qnre_layout_t layout, qnre_rope_t rope_style,
                                   unsigned flags, int B, int S_local, const void* x, const void* w_qkv,
                                   const void* q_norm_w, const void* k_norm_w, const float* cos_sin, int64_t n_pos,
                                   const int32_t* positions, const qnre_out_t* out, unsigned* device_status_out,
                                   qnre_stream_t stream) {
  // The geometry checks of qnre_plan_create, without its allocation.
  if (num_heads < 1 || P < 1 || hidden < 1) return QNRE_ERR_INVALID_ARG;
  if (hidden != num_heads * QNRE_HEAD_DIM || hidden % 64 != 0 || num_heads % P != 0) return QNRE_ERR_INVALID_ARG;
  if (layout != QNRE_LAYOUT_BSHD && layout != QNRE_LAYOUT_FUSED) return QNRE_ERR_INVALID_ARG;
  if (rope_style != QNRE_ROPE_ROTATE_HALF && rope_style != QNRE_ROPE_INTERLEAVED) return QNRE_ERR_INVALID_ARG;
  if ((flags & ~QNRE_FLAG_EPILOGUE_OFF) != 0) return QNRE_ERR_INVALID_ARG;
  if (B < 0 || S_local < 0) return QNRE_ERR_INVALID_ARG;
  // Sizes beyond what this entry point serves: the status block must fit the
  // static scratch, and the token count must stay inside the kernel's 32-bit
  // tile and TMA coordinates (the same bound qnre_plan_create puts on max_tokens).
  if (kNoAllocStatusBytes > kNoAllocScratchBytes) return QNRE_ERR_CAPACITY;
  const int64_t tokens_per_rank = static_cast<int64_t>(B) * S_local;
  if (tokens_per_rank * static_cast<int64_t>(P) > (int64_t{1} << 31) - 256) return QNRE_ERR_CAPACITY;
  if (device_status_out != nullptr && !aligned(device_status_out, 4)) return QNRE_ERR_ALIGNMENT;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return QNRE_ERR_CUDA;
  NoAllocDevice st;
  const qnre_status_t s0 = noalloc_setup(dev, &st);
  if (s0 != QNRE_OK) return s0;

  // A plan on the host stack whose status word is the static scratch.
  qnre_plan_s plan;
  plan.hidden = hidden;
  plan.num_heads = num_heads;
  plan.P = P;
  plan.H_local = num_heads / P;
  plan.layout = layout;
  plan.max_tokens = tokens_per_rank > 0 ? tokens_per_rank : 1;
  plan.rope_style = rope_style;
  plan.flags = flags;
  plan.device = dev;
  plan.max_pairs = st.max_pairs;
  plan.d_status = static_cast<unsigned*>(st.scratch);

  const qnre_status_t s1 = qnre_forward(&plan, B, S_local, x, w_qkv, q_norm_w, k_norm_w, cos_sin, n_pos, positions,
                                        out, stream);
  if (s1 != QNRE_OK) return s1;  // nothing was enqueued
  if (tokens_per_rank == 0) {
    if (device_status_out == nullptr) return QNRE_OK;
    return from_cuda(cudaMemsetAsync(device_status_out, 0, sizeof(unsigned), reinterpret_cast<cudaStream_t>(stream)));
  }
  // The kernel ORs bits into the status word, so it must be zero when the next
  // call's kernel starts: hand this call's word to the caller, then clear it,
  // both in stream order behind the kernel.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (device_status_out != nullptr &&
      cudaMemcpyAsync(device_status_out, st.scratch, sizeof(unsigned), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return QNRE_ERR_CUDA;
  return from_cuda(cudaMemsetAsync(st.scratch, 0, kNoAllocStatusBytes, s));
}

}  // extern "C"
