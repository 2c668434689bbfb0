// layout_api.cu -- extern "C" entry points of the Ulysses layout transforms:
// head-chunk pack and merge, ordinary scatter/gather heads over P virtual
// ranks, the output sequence-chunk pack, and the two head-chunk exchanges
// composed over P virtual ranks.  Each one validates its arguments, maps the
// transform onto the affine head-row copy (layout_copy.cuh) and launches once.
#include "../../include/qnre.h"
#include "api_util.cuh"
#include "layout_copy.cuh"

#include <cuda_runtime.h>

#include <cstdint>
#include <initializer_list>

namespace {

using namespace qnre;
using namespace qnre::api;

cudaStream_t as_stream(qnre_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Source side of a plan from up to three strided [*, *, heads, D] views that
// share one shape.  Chooses 16-byte vectors when every view and the output allow.
void set_sources(LayoutCopyPlan& p, const qnre_tensor4_t* const* views, int n, int esz, bool vec) {
  for (int c = 0; c < 3; ++c) {
    const qnre_tensor4_t* t = views[c < n ? c : 0];
    p.src[c] = t->data;
    p.src_head[c] = t->stride[2] * esz;
    p.src_z0[c] = t->stride[0] * esz;
    p.src_s[c] = t->stride[1] * esz;
    p.src_z1[c] = 0;
  }
  p.unit_bytes = vec ? 16 : esz;
  p.units = static_cast<int>(vec ? views[0]->shape[3] * esz / 16 : views[0]->shape[3]);
  p.src_unit = vec ? 16 : views[0]->stride[3] * esz;
}

// Byte ranges the debug build checks every access against: the same extents
// the alias checks use (source c < n, the output).
void set_ranges(LayoutCopyPlan& p, const ByteRange* in, int n, ByteRange out) {
  for (int c = 0; c < 3; ++c) {
    p.src_lo[c] = in[c < n ? c : 0].lo;
    p.src_hi[c] = in[c < n ? c : 0].hi;
  }
  p.dst_lo = out.lo;
  p.dst_hi = out.hi;
}

bool all_vectorisable(const qnre_tensor4_t* const* views, int n, int esz, const void* out) {
  if (!aligned(out, 16)) return false;
  for (int c = 0; c < n; ++c)
    if (!rows_vectorisable(views[c], esz)) return false;
  return true;
}

// Contiguous operand checks for the P-virtual-rank transforms.
qnre_status_t check_contig(const void* in, uint64_t in_elems, const void* out, uint64_t out_elems, int esz,
                           bool* vec, int64_t D) {
  if (in == nullptr || out == nullptr) return QNRE_ERR_INVALID_ARG;
  if (!aligned(in, static_cast<uintptr_t>(esz)) || !aligned(out, static_cast<uintptr_t>(esz)))
    return QNRE_ERR_ALIGNMENT;
  if (overlaps(span(in, in_elems * esz), span(out, out_elems * esz))) return QNRE_ERR_ALIAS;
  *vec = aligned(in, 16) && aligned(out, 16) && (D * esz) % 16 == 0;
  return QNRE_OK;
}

bool dims_ok(std::initializer_list<int64_t> dims) {
  for (int64_t d : dims)
    if (d < 0 || d > (int64_t{1} << 31)) return false;
  return true;
}

// ---- head-chunk pack and merge, shared by the single-chunk and schedule calls

struct PackPlan {
  LayoutCopyPlan plan{};
  ByteRange out_range{0, 0};
  bool same_unit = true;  // one launch covers q, k and v
  bool empty = false;     // B == 0 or S == 0: nothing to copy
};

// Validation and copy plan of one pack_ulysses_qkv_head_chunk call.
qnre_status_t pack_plan(const qnre_tensor4_t* q, const qnre_tensor4_t* k, const qnre_tensor4_t* v, int world_size,
                        int head_offset, int head_count, void* out, PackPlan* pp) {
  const qnre_tensor4_t* X[3] = {q, k, v};
  ByteRange in[3];
  for (int c = 0; c < 3; ++c) {
    const qnre_status_t st = check_view(X[c], &in[c]);
    if (st != QNRE_OK) return st;
  }
  for (int c = 1; c < 3; ++c) {
    if (X[c]->dtype != q->dtype) return QNRE_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
      if (X[c]->shape[i] != q->shape[i]) return QNRE_ERR_INVALID_ARG;
  }
  if (out == nullptr) return QNRE_ERR_INVALID_ARG;
  const int64_t B = q->shape[0], S = q->shape[1], H = q->shape[2], D = q->shape[3];
  if (world_size < 1 || H % world_size != 0) return QNRE_ERR_INVALID_ARG;
  const int64_t H_local = H / world_size;
  if (head_offset < 0 || head_count < 1 || head_offset + static_cast<int64_t>(head_count) > H_local)
    return QNRE_ERR_INVALID_ARG;
  if (B > 65535) return QNRE_ERR_CAPACITY;
  const int esz = dtype_size(q->dtype);
  if (!aligned(out, static_cast<uintptr_t>(esz))) return QNRE_ERR_ALIGNMENT;
  const int64_t slots = static_cast<int64_t>(world_size) * head_count;
  const ByteRange o = span(out, static_cast<uint64_t>(B) * S * slots * 3 * D * esz);
  for (int c = 0; c < 3; ++c)
    if (overlaps(o, in[c])) return QNRE_ERR_ALIAS;
  pp->out_range = o;
  pp->empty = B == 0 || S == 0;
  if (pp->empty) return QNRE_OK;

  const bool vec = all_vectorisable(X, 3, esz, out);
  LayoutCopyPlan& p = pp->plan;
  p = LayoutCopyPlan{};
  set_sources(p, X, 3, esz, vec);
  for (int c = 0; c < 3; ++c) p.src_rank[c] = H_local * X[c]->stride[2] * esz;
  p.src_head_offset = head_offset;
  p.dst = out;
  p.dst_rank = static_cast<long long>(head_count) * 3 * D * esz;
  p.dst_head = 3 * D * esz;
  p.dst_comp = D * esz;
  p.dst_head_offset = 0;
  p.dst_z1 = 0;
  p.dst_z0 = S * slots * 3 * D * esz;
  p.dst_s = slots * 3 * D * esz;
  p.Z1 = 1;
  p.Z0 = B;
  p.S = S;
  p.head_count = head_count;
  p.ranks = world_size;
  p.comps = 3;
  set_ranges(p, in, 3, o);
  pp->same_unit = vec || (k->stride[3] == q->stride[3] && v->stride[3] == q->stride[3]);
  return QNRE_OK;
}

// One pack: a single launch, or (element path with different innermost
// strides) one launch per component.
qnre_status_t launch_pack(const PackPlan& pp, const qnre_tensor4_t* q, const qnre_tensor4_t* k,
                          const qnre_tensor4_t* v, void* out, qnre_stream_t stream) {
  if (pp.same_unit) return from_cuda(launch_layout_copy(pp.plan, as_stream(stream)));
  const qnre_tensor4_t* X[3] = {q, k, v};
  const int esz = dtype_size(q->dtype);
  const int64_t D = q->shape[3];
  for (int c = 0; c < 3; ++c) {
    LayoutCopyPlan pc = pp.plan;
    pc.src[0] = X[c]->data;
    pc.src_rank[0] = pp.plan.src_rank[c];
    pc.src_head[0] = pp.plan.src_head[c];
    pc.src_z0[0] = pp.plan.src_z0[c];
    pc.src_s[0] = pp.plan.src_s[c];
    pc.src_lo[0] = pp.plan.src_lo[c];
    pc.src_hi[0] = pp.plan.src_hi[c];
    pc.src_unit = X[c]->stride[3] * esz;
    pc.dst = static_cast<char*>(out) + static_cast<int64_t>(c) * D * esz;
    pc.comps = 1;
    const cudaError_t e = launch_layout_copy(pc, as_stream(stream));
    if (e != cudaSuccess) return QNRE_ERR_CUDA;
  }
  return QNRE_OK;
}

// Validation and copy plan of one merge_ulysses_output_head_chunk call.
qnre_status_t merge_plan(const qnre_tensor4_t* received, int world_size, int local_heads, int head_offset,
                         void* out, LayoutCopyPlan* plan, bool* empty) {
  ByteRange in;
  const qnre_status_t st = check_view(received, &in);
  if (st != QNRE_OK) return st;
  if (out == nullptr) return QNRE_ERR_INVALID_ARG;
  const int64_t B = received->shape[0], S = received->shape[1], WC = received->shape[2], D = received->shape[3];
  if (world_size < 1 || WC % world_size != 0) return QNRE_ERR_INVALID_ARG;
  const int64_t head_count = WC / world_size;
  if (local_heads < 1 || head_offset < 0 || head_offset + head_count > local_heads) return QNRE_ERR_INVALID_ARG;
  if (B > 65535) return QNRE_ERR_CAPACITY;
  const int esz = dtype_size(received->dtype);
  if (!aligned(out, static_cast<uintptr_t>(esz))) return QNRE_ERR_ALIGNMENT;
  const int64_t out_heads = static_cast<int64_t>(world_size) * local_heads;
  const ByteRange o = span(out, static_cast<uint64_t>(B) * S * out_heads * D * esz);
  if (overlaps(o, in)) return QNRE_ERR_ALIAS;
  *empty = B == 0 || S == 0;
  if (*empty) return QNRE_OK;

  const qnre_tensor4_t* X[1] = {received};
  const bool vec = all_vectorisable(X, 1, esz, out);
  LayoutCopyPlan& p = *plan;
  p = LayoutCopyPlan{};
  set_sources(p, X, 1, esz, vec);
  p.src_rank[0] = head_count * received->stride[2] * esz;
  p.src_head_offset = 0;
  p.dst = out;
  p.dst_rank = static_cast<long long>(local_heads) * D * esz;
  p.dst_head = D * esz;
  p.dst_comp = 0;
  p.dst_head_offset = head_offset;
  p.dst_z0 = S * out_heads * D * esz;
  p.dst_s = out_heads * D * esz;
  p.Z1 = 1;
  p.Z0 = B;
  p.S = S;
  p.head_count = static_cast<int>(head_count);
  p.ranks = world_size;
  p.comps = 1;
  set_ranges(p, &in, 1, o);
  return QNRE_OK;
}

}  // namespace

extern "C" {

qnre_status_t ulysses_pack_head_chunk(const qnre_tensor4_t* q, const qnre_tensor4_t* k, const qnre_tensor4_t* v,
                                      int world_size, int head_offset, int head_count, void* out,
                                      qnre_stream_t stream) {
  PackPlan pp;
  const qnre_status_t st = pack_plan(q, k, v, world_size, head_offset, head_count, out, &pp);
  if (st != QNRE_OK || pp.empty) return st;
  return launch_pack(pp, q, k, v, out, stream);
}

qnre_status_t ulysses_merge_output_head_chunk(const qnre_tensor4_t* received, int world_size, int local_heads,
                                              int head_offset, void* out, qnre_stream_t stream) {
  LayoutCopyPlan p{};
  bool empty = false;
  const qnre_status_t st = merge_plan(received, world_size, local_heads, head_offset, out, &p, &empty);
  if (st != QNRE_OK || empty) return st;
  return from_cuda(launch_layout_copy(p, as_stream(stream)));
}

qnre_status_t ulysses_pack_head_chunk_schedule(const qnre_tensor4_t* q, const qnre_tensor4_t* k,
                                               const qnre_tensor4_t* v, int world_size, int num_chunks,
                                               const int* head_offsets, const int* head_counts, void* const* outs,
                                               qnre_stream_t stream) {
  if (num_chunks < 1 || head_offsets == nullptr || head_counts == nullptr || outs == nullptr)
    return QNRE_ERR_INVALID_ARG;
  if (num_chunks > kLayoutCopyMaxBatch) return QNRE_ERR_CAPACITY;
  PackPlan pp[kLayoutCopyMaxBatch];
  bool batch = true;
  for (int i = 0; i < num_chunks; ++i) {
    const qnre_status_t st = pack_plan(q, k, v, world_size, head_offsets[i], head_counts[i], outs[i], &pp[i]);
    if (st != QNRE_OK) return st;
    pp[i].plan.streaming = 1;  // schedule calls run beside the projection
    batch = batch && pp[i].same_unit && pp[i].plan.unit_bytes == pp[0].plan.unit_bytes;
  }
  for (int i = 0; i < num_chunks; ++i)
    for (int j = i + 1; j < num_chunks; ++j)
      if (overlaps(pp[i].out_range, pp[j].out_range)) return QNRE_ERR_ALIAS;
  if (pp[0].empty) return QNRE_OK;  // every chunk shares the views' (B, S)
  if (batch) {
    LayoutCopyPlan plans[kLayoutCopyMaxBatch];
    for (int i = 0; i < num_chunks; ++i) plans[i] = pp[i].plan;
    return from_cuda(launch_layout_copy_batch(plans, num_chunks, as_stream(stream)));
  }
  for (int i = 0; i < num_chunks; ++i) {  // mixed copy units: chunk by chunk
    const qnre_status_t st = launch_pack(pp[i], q, k, v, outs[i], stream);
    if (st != QNRE_OK) return st;
  }
  return QNRE_OK;
}

qnre_status_t ulysses_merge_output_head_chunk_schedule(const qnre_tensor4_t* const* received, int world_size,
                                                       int local_heads, int num_chunks, const int* head_offsets,
                                                       void* out, qnre_stream_t stream) {
  if (num_chunks < 1 || received == nullptr || head_offsets == nullptr) return QNRE_ERR_INVALID_ARG;
  if (num_chunks > kLayoutCopyMaxBatch) return QNRE_ERR_CAPACITY;
  LayoutCopyPlan plans[kLayoutCopyMaxBatch];
  int64_t lo[kLayoutCopyMaxBatch], hi[kLayoutCopyMaxBatch];
  bool empty = false, batch = true;
  for (int i = 0; i < num_chunks; ++i) {
    if (received[i] == nullptr) return QNRE_ERR_INVALID_ARG;
    const qnre_status_t st =
        merge_plan(received[i], world_size, local_heads, head_offsets[i], out, &plans[i], &empty);
    if (st != QNRE_OK) return st;
    plans[i].streaming = 1;
    for (int d : {0, 1, 3})
      if (received[i]->shape[d] != received[0]->shape[d]) return QNRE_ERR_INVALID_ARG;
    if (received[i]->dtype != received[0]->dtype) return QNRE_ERR_INVALID_ARG;
    lo[i] = head_offsets[i];
    hi[i] = head_offsets[i] + received[i]->shape[2] / world_size;
    batch = batch && plans[i].unit_bytes == plans[0].unit_bytes;
  }
  for (int i = 0; i < num_chunks; ++i)  // one launch runs the chunks in any order: their bands must be disjoint
    for (int j = i + 1; j < num_chunks; ++j)
      if (lo[i] < hi[j] && lo[j] < hi[i]) return QNRE_ERR_INVALID_ARG;
  if (empty) return QNRE_OK;
  if (batch) return from_cuda(launch_layout_copy_batch(plans, num_chunks, as_stream(stream)));
  for (int i = 0; i < num_chunks; ++i) {
    const cudaError_t e = launch_layout_copy(plans[i], as_stream(stream));
    if (e != cudaSuccess) return QNRE_ERR_CUDA;
  }
  return QNRE_OK;
}

qnre_status_t ulysses_scatter_heads(const void* x, int P, int B, int S_local, int H, int D, int32_t dtype, void* out,
                                    qnre_stream_t stream) {
  if (P < 1 || B < 0 || S_local < 0 || H < 1 || D < 1 || H % P != 0) return QNRE_ERR_INVALID_ARG;
  const int esz = dtype_size(dtype);
  if (esz == 0) return QNRE_ERR_UNSUPPORTED;
  if (!dims_ok({P, B, S_local, H, D}) || static_cast<int64_t>(P) * B > 65535) return QNRE_ERR_CAPACITY;
  const int64_t H_l = H / P;
  const uint64_t n = static_cast<uint64_t>(P) * B * S_local * H * D;
  bool vec = false;
  const qnre_status_t st = check_contig(x, n, out, n, esz, &vec, D);
  if (st != QNRE_OK) return st;
  if (n == 0) return QNRE_OK;
  LayoutCopyPlan p{};
  const int64_t e = esz;
  for (int c = 0; c < 3; ++c) {
    p.src[c] = x;
    p.src_rank[c] = H_l * D * e;
    p.src_head[c] = D * e;
    p.src_z1[c] = static_cast<int64_t>(B) * S_local * H * D * e;
    p.src_z0[c] = static_cast<int64_t>(S_local) * H * D * e;
    p.src_s[c] = static_cast<int64_t>(H) * D * e;
  }
  p.src_unit = vec ? 16 : e;
  p.dst = out;
  p.dst_rank = static_cast<int64_t>(B) * P * S_local * H_l * D * e;
  p.dst_head = D * e;
  p.dst_z1 = static_cast<int64_t>(S_local) * H_l * D * e;
  p.dst_z0 = static_cast<int64_t>(P) * S_local * H_l * D * e;
  p.dst_s = H_l * D * e;
  p.Z1 = P;
  p.Z0 = B;
  p.S = S_local;
  p.head_count = static_cast<int>(H_l);
  p.ranks = P;
  p.comps = 1;
  p.unit_bytes = vec ? 16 : esz;
  p.units = static_cast<int>(vec ? D * e / 16 : D);
  const ByteRange in = span(x, n * esz);
  set_ranges(p, &in, 1, span(out, n * esz));
  return from_cuda(launch_layout_copy(p, as_stream(stream)));
}

qnre_status_t ulysses_gather_heads(const void* y, int P, int B, int S_global, int H_local, int D, int32_t dtype,
                                   void* out, qnre_stream_t stream) {
  if (P < 1 || B < 0 || S_global < 0 || H_local < 1 || D < 1 || S_global % P != 0) return QNRE_ERR_INVALID_ARG;
  const int esz = dtype_size(dtype);
  if (esz == 0) return QNRE_ERR_UNSUPPORTED;
  if (!dims_ok({P, B, S_global, H_local, D}) || static_cast<int64_t>(P) * B > 65535) return QNRE_ERR_CAPACITY;
  const int64_t S = S_global / P;
  const int64_t H = static_cast<int64_t>(P) * H_local;
  const uint64_t n = static_cast<uint64_t>(P) * B * S_global * H_local * D;
  bool vec = false;
  const qnre_status_t st = check_contig(y, n, out, n, esz, &vec, D);
  if (st != QNRE_OK) return st;
  if (n == 0) return QNRE_OK;
  LayoutCopyPlan p{};
  const int64_t e = esz;
  for (int c = 0; c < 3; ++c) {
    p.src[c] = y;
    p.src_rank[c] = static_cast<int64_t>(B) * S_global * H_local * D * e;
    p.src_head[c] = D * e;
    p.src_z1[c] = S * H_local * D * e;
    p.src_z0[c] = static_cast<int64_t>(S_global) * H_local * D * e;
    p.src_s[c] = static_cast<int64_t>(H_local) * D * e;
  }
  p.src_unit = vec ? 16 : e;
  p.dst = out;
  p.dst_rank = static_cast<int64_t>(H_local) * D * e;
  p.dst_head = D * e;
  p.dst_z1 = static_cast<int64_t>(B) * S * H * D * e;
  p.dst_z0 = S * H * D * e;
  p.dst_s = H * D * e;
  p.Z1 = P;
  p.Z0 = B;
  p.S = S;
  p.head_count = H_local;
  p.ranks = P;
  p.comps = 1;
  p.unit_bytes = vec ? 16 : esz;
  p.units = static_cast<int>(vec ? D * e / 16 : D);
  const ByteRange in = span(y, n * esz);
  set_ranges(p, &in, 1, span(out, n * esz));
  return from_cuda(launch_layout_copy(p, as_stream(stream)));
}

qnre_status_t ulysses_pack_output_sequence_chunk(const qnre_tensor4_t* x, int world_size, void* out,
                                                 qnre_stream_t stream) {
  ByteRange in;
  const qnre_status_t st = check_view(x, &in);
  if (st != QNRE_OK) return st;
  if (out == nullptr) return QNRE_ERR_INVALID_ARG;
  const int64_t B = x->shape[0], S_g = x->shape[1], cnt = x->shape[2], D = x->shape[3];
  if (world_size < 1 || S_g % world_size != 0) return QNRE_ERR_INVALID_ARG;
  if (B > 65535) return QNRE_ERR_CAPACITY;
  const int esz = dtype_size(x->dtype);
  if (!aligned(out, static_cast<uintptr_t>(esz))) return QNRE_ERR_ALIGNMENT;
  const ByteRange o = span(out, static_cast<uint64_t>(B) * S_g * cnt * D * esz);
  if (overlaps(o, in)) return QNRE_ERR_ALIAS;
  if (B == 0 || S_g == 0) return QNRE_OK;
  const int64_t S = S_g / world_size;
  const qnre_tensor4_t* X[1] = {x};
  const bool vec = all_vectorisable(X, 1, esz, out);
  LayoutCopyPlan p{};
  set_sources(p, X, 1, esz, vec);
  p.src_rank[0] = S * x->stride[1] * esz;  // rank r's chunk starts at row r*S_local
  p.src_head_offset = 0;
  p.dst = out;
  p.dst_rank = B * S * cnt * D * esz;
  p.dst_head = D * esz;
  p.dst_z0 = S * cnt * D * esz;
  p.dst_s = cnt * D * esz;
  p.Z1 = 1;
  p.Z0 = B;
  p.S = S;
  p.head_count = static_cast<int>(cnt);
  p.ranks = world_size;
  p.comps = 1;
  set_ranges(p, &in, 1, o);
  return from_cuda(launch_layout_copy(p, as_stream(stream)));
}

qnre_status_t ulysses_gather_output_head_chunk(const void* x, int P, int B, int S_global, int head_count, int D,
                                               int32_t dtype, int local_heads, int head_offset, void* out,
                                               qnre_stream_t stream) {
  if (P < 1 || B < 0 || S_global < 0 || head_count < 1 || D < 1 || S_global % P != 0) return QNRE_ERR_INVALID_ARG;
  if (local_heads < 1 || head_offset < 0 || head_offset + head_count > local_heads) return QNRE_ERR_INVALID_ARG;
  const int esz = dtype_size(dtype);
  if (esz == 0) return QNRE_ERR_UNSUPPORTED;
  if (!dims_ok({P, B, S_global, head_count, D, local_heads}) || static_cast<int64_t>(P) * B > 65535)
    return QNRE_ERR_CAPACITY;
  const int64_t S = S_global / P;
  const uint64_t n_in = static_cast<uint64_t>(P) * B * S_global * head_count * D;
  const uint64_t n_out = static_cast<uint64_t>(P) * B * S * P * local_heads * D;
  bool vec = false;
  const qnre_status_t st = check_contig(x, n_in, out, n_out, esz, &vec, D);
  if (st != QNRE_OK) return st;
  if (n_in == 0) return QNRE_OK;
  LayoutCopyPlan p{};
  const int64_t e = esz;
  for (int c = 0; c < 3; ++c) {
    p.src[c] = x;
    p.src_rank[c] = static_cast<int64_t>(B) * S_global * head_count * D * e;
    p.src_head[c] = D * e;
    p.src_z1[c] = S * head_count * D * e;
    p.src_z0[c] = static_cast<int64_t>(S_global) * head_count * D * e;
    p.src_s[c] = static_cast<int64_t>(head_count) * D * e;
  }
  p.src_unit = vec ? 16 : e;
  p.dst = out;
  p.dst_rank = static_cast<int64_t>(local_heads) * D * e;
  p.dst_head = D * e;
  p.dst_head_offset = head_offset;
  p.dst_z1 = static_cast<int64_t>(B) * S * P * local_heads * D * e;
  p.dst_z0 = S * P * local_heads * D * e;
  p.dst_s = static_cast<int64_t>(P) * local_heads * D * e;
  p.Z1 = P;
  p.Z0 = B;
  p.S = S;
  p.head_count = head_count;
  p.ranks = P;
  p.comps = 1;
  p.unit_bytes = vec ? 16 : esz;
  p.units = static_cast<int>(vec ? D * e / 16 : D);
  const ByteRange in = span(x, n_in * esz);
  set_ranges(p, &in, 1, span(out, n_out * esz));
  return from_cuda(launch_layout_copy(p, as_stream(stream)));
}

qnre_status_t ulysses_scatter_qkv_head_chunk(const qnre_tensor4_t* q, const qnre_tensor4_t* k,
                                             const qnre_tensor4_t* v, int P, int head_offset, int head_count,
                                             void* out, qnre_stream_t stream) {
  const qnre_tensor4_t* X[3] = {q, k, v};
  ByteRange in[3];
  for (int c = 0; c < 3; ++c) {
    const qnre_status_t st = check_view(X[c], &in[c]);
    if (st != QNRE_OK) return st;
  }
  for (int c = 1; c < 3; ++c) {
    if (X[c]->dtype != q->dtype) return QNRE_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
      if (X[c]->shape[i] != q->shape[i]) return QNRE_ERR_INVALID_ARG;
  }
  if (out == nullptr || P < 1) return QNRE_ERR_INVALID_ARG;
  const int64_t PB = q->shape[0], S = q->shape[1], H = q->shape[2], D = q->shape[3];
  if (PB % P != 0 || H % P != 0) return QNRE_ERR_INVALID_ARG;
  const int64_t B = PB / P, H_local = H / P;
  if (head_offset < 0 || head_count < 1 || head_offset + static_cast<int64_t>(head_count) > H_local)
    return QNRE_ERR_INVALID_ARG;
  if (PB > 65535) return QNRE_ERR_CAPACITY;
  const int esz = dtype_size(q->dtype);
  if (!aligned(out, static_cast<uintptr_t>(esz))) return QNRE_ERR_ALIGNMENT;
  // out [P, B, P*S, head_count, 3D]: P * PB * S head rows of 3D elements
  const ByteRange o = span(out, static_cast<uint64_t>(P) * PB * S * head_count * 3 * D * esz);
  for (int c = 0; c < 3; ++c)
    if (overlaps(o, in[c])) return QNRE_ERR_ALIAS;
  if (PB == 0 || S == 0) return QNRE_OK;

  const bool vec = all_vectorisable(X, 3, esz, out);
  LayoutCopyPlan p{};
  set_sources(p, X, 3, esz, vec);
  for (int c = 0; c < 3; ++c) {
    p.src_rank[c] = H_local * X[c]->stride[2] * esz;
    p.src_z1[c] = B * X[c]->stride[0] * esz;  // batch index z = r_s*B + b
  }
  p.src_head_offset = head_offset;
  const int64_t row = static_cast<int64_t>(head_count) * 3 * D * esz;
  p.dst = out;
  p.dst_rank = B * P * S * row;
  p.dst_head = 3 * D * esz;
  p.dst_comp = D * esz;
  p.dst_z1 = S * row;
  p.dst_z0 = P * S * row;
  p.dst_s = row;
  p.Z1 = P;
  p.Z0 = B;
  p.S = S;
  p.head_count = head_count;
  p.ranks = P;
  p.comps = 3;
  set_ranges(p, in, 3, o);
  const bool same_unit = vec || (k->stride[3] == q->stride[3] && v->stride[3] == q->stride[3]);
  if (same_unit) return from_cuda(launch_layout_copy(p, as_stream(stream)));
  for (int c = 0; c < 3; ++c) {
    LayoutCopyPlan pc = p;
    pc.src[0] = X[c]->data;
    pc.src_rank[0] = p.src_rank[c];
    pc.src_head[0] = p.src_head[c];
    pc.src_z1[0] = p.src_z1[c];
    pc.src_z0[0] = p.src_z0[c];
    pc.src_s[0] = p.src_s[c];
    pc.src_lo[0] = p.src_lo[c];
    pc.src_hi[0] = p.src_hi[c];
    pc.src_unit = X[c]->stride[3] * esz;
    pc.dst = static_cast<char*>(out) + static_cast<int64_t>(c) * D * esz;
    pc.comps = 1;
    const cudaError_t e = launch_layout_copy(pc, as_stream(stream));
    if (e != cudaSuccess) return QNRE_ERR_CUDA;
  }
  return QNRE_OK;
}

}  // extern "C"
