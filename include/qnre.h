/*
 * qnre.h -- C ABI of libqnre: the single-GPU data-parallel core of the Ulysses
 * sequence-parallel attention front end, for NVIDIA GB300 (sm_103a).
 *
 * Sources (pages, by title and section):
 *   [FUSED] flashinfer.comm API reference v0.7.4, "Fused QKV Projection + Norm +
 *           RoPE + Head Exchange" (QkvNormRopeExchangeOverlap and its Notes).
 *   [MATH]  "QKV projection + RMSNorm + RoPE overlapped with the Ulysses head
 *           exchange" (flashinfer PR #6332 commit text, on the docs PR #4240
 *           page), "Description" and "Assumptions" / "Operator math".
 *   [ULY]   flashinfer.comm API reference, "Ulysses Context-Parallel All-to-All".
 *   [PACK]  flashinfer.comm API reference, "Head-Chunk Layout and Transport
 *           Primitives", pack_ulysses_qkv_head_chunk.
 *   [MERGE] same section, merge_ulysses_output_head_chunk.
 *   [XCHG]  flashinfer.comm API reference, UlyssesCommunicator.scatter_qkv_head_chunk,
 *           gather_output_head_chunk and exchange_chunks.
 *   [LOWP]  flashinfer.comm API reference, "Prepared Low-Precision QKV Exchange"
 *           (UlyssesCommunicator.prepare_qkv / scatter_qkv) and its
 *           "Low-Precision Implementation Primitives" list.
 *   [PR5027] "allocation-stable, head-chunked Ulysses communication primitives"
 *           (flashinfer PR #5027), Description: uneven schedules, positive-stride
 *           non-contiguous views, storage-range alias checks, int32 limits.
 *
 * On one GPU the P Ulysses ranks are virtual: every rank's input shard and
 * every rank's receive buffer live in this GPU's memory, and the head exchange
 * is the address each result is stored to.  No call communicates.
 *
 * Conventions for every call:
 *   - Pointers marked "device" point to memory of the current CUDA device; the
 *     caller owns all of it.  No call allocates device memory except
 *     qnre_plan_create (the plan's 16-byte status word).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns without waiting for it.  Stream order holds for
 *     every call.  The layout copies (pack, merge, scatter/gather, sequence
 *     pack, the composed exchanges) and the three Sage2 kernels are
 *     programmatic dependent launches: their blocks may be scheduled while
 *     the previous kernel in the stream drains, and each waits until that
 *     kernel has completed and its writes are visible before it reads
 *     anything.  Layout copies launched alone (not the *_schedule calls) first
 *     hint L2 to fetch their source lines, which never changes a result.
 *   - Arguments are validated before anything is launched: a call that returns
 *     an error has enqueued nothing and written nothing.
 *   - bf16 values are IEEE bfloat16 bit patterns (the high half of a float32).
 *   - Status codes: QNRE_OK on success, else the first failed check.
 */
#ifndef QNRE_H_
#define QNRE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QNRE_HEAD_DIM 128

typedef struct CUstream_st* qnre_stream_t; /* == cudaStream_t */

typedef enum {
  QNRE_OK = 0,
  QNRE_ERR_INVALID_ARG = 1, /* bad shape, count, offset, NULL pointer, unknown enum */
  QNRE_ERR_UNSUPPORTED = 2, /* valid request this build does not serve (head_dim != 128, dtype) */
  QNRE_ERR_ALIGNMENT = 3,   /* a pointer or stride breaks the stated byte alignment */
  QNRE_ERR_ALIAS = 4,       /* an output's storage range overlaps an input's */
  QNRE_ERR_CAPACITY = 5,    /* B*S_local > max_tokens, or a size that overflows 64-bit offsets */
  QNRE_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed (no device, launch failure) */
  QNRE_ERR_DEVICE = 7       /* a device-side check fired (see qnre_plan_device_status) */
} qnre_status_t;

typedef enum { QNRE_LAYOUT_BSHD = 0, QNRE_LAYOUT_FUSED = 1 } qnre_layout_t;

/* RoPE pairing.  ROTATE_HALF rotates (i, i+64); INTERLEAVED rotates (2i, 2i+1)
 * (the pairing the [MATH] page names).  Both read cos_i = cos_sin[p][i] and
 * sin_i = cos_sin[p][64+i], i < 64. */
typedef enum { QNRE_ROPE_ROTATE_HALF = 0, QNRE_ROPE_INTERLEAVED = 1 } qnre_rope_t;

typedef enum { QNRE_DTYPE_BF16 = 0, QNRE_DTYPE_FP16 = 1, QNRE_DTYPE_FP32 = 2 } qnre_dtype_t;

/* Plan flags. */
#define QNRE_FLAG_EPILOGUE_OFF 0x1u /* store the bare projection for q, k and v (no norm, no RoPE).
                                       A diagnostic: with integer-coded inputs the result is exact,
                                       so band placement can be compared bit for bit. */
#define QNRE_FLAG_W_MULTICAST 0x2u  /* always run the fused kernel in clusters of two CTA pairs
                                       that take adjacent 256-row tiles of the same column tile
                                       and share each W tile through one TMA multicast load.
                                       Without this flag the plan still picks that form when it
                                       fits and the row tiles pair up (an even count, or 16 or
                                       more).  Results are bit-identical either way.
                                       QNRE_ERR_UNSUPPORTED at plan creation if such clusters
                                       cannot be resident. */
#define QNRE_FLAG_ONE_PAIR 0x4u     /* always run the fused kernel one CTA pair per cluster (no
                                       W multicast); not together with QNRE_FLAG_W_MULTICAST. */

/* Device-side status bits (qnre_plan_device_status). */
#define QNRE_DEVICE_BAD_POSITION 0x1u /* a token's position was outside [0, n_pos): its q and k rows
                                         were written as NaN and the table was not read */
#define QNRE_DEVICE_WAIT_TIMEOUT 0x2u /* a pipeline wait inside the kernel ran past its time limit; the
                                         kernel stopped early and its outputs are incomplete */
#define QNRE_DEVICE_READY_TIMEOUT 0x4u /* qnre_wait_ready gave up before every readiness word reached
                                          its target */
#define QNRE_DEVICE_BOUNDS 0x8u /* debug build only (libqnre_debug.so): a computed output row fell
                                   outside its output tensor and was not stored */

typedef struct qnre_plan_s* qnre_plan_t;

/* Output buffers of qnre_forward (device, bf16, caller-owned, 16-byte aligned).
 *   QNRE_LAYOUT_BSHD : q, k, v each [P, B, S_global, H_local, 128]; fused unused.
 *   QNRE_LAYOUT_FUSED: fused [P, B, S_global, H_local, 384], q|k|v along the last
 *                      axis; q, k, v unused.
 * Index [r, b, row, hl, :] is virtual rank r's receive slot: head r*H_local + hl
 * of the token at global row `row` of batch row b. */
typedef struct {
  void* q;
  void* k;
  void* v;
  void* fused;
} qnre_out_t;

/* A strided rank-4 view (device).  shape[i] >= 1 and stride[i] >= 1 are in
 * elements; element (a, b, c, d) lives at data + (a*stride[0] + b*stride[1] +
 * c*stride[2] + d*stride[3]) * element_size. */
typedef struct {
  void* data;
  int64_t shape[4];
  int64_t stride[4];
  int32_t dtype; /* qnre_dtype_t */
} qnre_tensor4_t;

/* Human-readable name of a status code (static storage; never NULL). */
const char* qnre_status_string(qnre_status_t status);

/*
 * qnre_plan_create -- prepare the fused QKV projection + RMSNorm + RoPE + head-band
 * scatter for one geometry.  [FUSED] constructor: hidden = num_heads*head_dim, a
 * multiple of 64; num_heads divisible by the world size (P here); head_dim = 128;
 * bf16 only; max_tokens = the largest B*S_local of any call.
 *
 *   plan       out: receives the plan handle (host object).  Unchanged on error.
 *   hidden     model width; must equal num_heads*128.
 *   num_heads  attention heads H (>= 1, H % P == 0).
 *   head_dim   must be 128 (else QNRE_ERR_UNSUPPORTED).
 *   P          virtual Ulysses ranks (>= 1).
 *   layout     QNRE_LAYOUT_BSHD or QNRE_LAYOUT_FUSED.
 *   max_tokens largest B*S_local per rank accepted by qnre_forward (>= 1).
 *   rope_style QNRE_ROPE_ROTATE_HALF or QNRE_ROPE_INTERLEAVED.
 *   flags      0, or QNRE_FLAG_EPILOGUE_OFF and at most one of QNRE_FLAG_W_MULTICAST,
 *              QNRE_FLAG_ONE_PAIR.
 *
 * Binds to the current CUDA device: queries it, sets the kernel's shared-memory
 * limit, and allocates the plan's 16-byte device status word (the only device
 * allocation the library makes; it is released by qnre_plan_destroy).
 * Errors: QNRE_ERR_INVALID_ARG, QNRE_ERR_UNSUPPORTED, QNRE_ERR_CUDA (no device,
 * not an sm_103 GPU).
 */
qnre_status_t qnre_plan_create(qnre_plan_t* plan, int hidden, int num_heads, int head_dim, int P,
                               qnre_layout_t layout, int64_t max_tokens, qnre_rope_t rope_style,
                               unsigned flags);

/* Release a plan.  The caller must make sure no launched forward still runs.
 * NULL is accepted (no-op). */
qnre_status_t qnre_plan_destroy(qnre_plan_t plan);

/*
 * qnre_plan_reserve_sms -- leave `sms` SMs free of the fused kernel's
 * persistent grid, for work the caller runs beside it on other streams (the
 * pages' producers run "over every SM (no reserved SMs)" only on some
 * architectures: [FUSED] Notes, per-architecture gates).  The count is rounded
 * up to whole clusters of the form the call runs: CTA pairs (2 SMs) or two
 * pairs sharing W (4 SMs; at least one such cluster always remains).  The
 * fused kernel then runs on the remaining clusters; results are bit-identical
 * for every setting (each tile's arithmetic does not depend on which cluster
 * runs it).  0 (the default) reserves nothing.  In either case a forward
 * launches the fewest of the clusters it may use that finish its work list in
 * as many rounds as all of them would (qnre_plan_describe reports the count):
 * the clusters that would only idle through the last round are left to other
 * streams.
 * Host-only; applies to later calls of this plan.
 * Errors: QNRE_ERR_INVALID_ARG for a NULL plan, sms < 0, or a request that would
 * leave no CTA pair.
 */
qnre_status_t qnre_plan_reserve_sms(qnre_plan_t plan, int sms);

/*
 * qnre_plan_describe -- how a forward of (B, S_local) with this plan runs (the
 * pages' sessions report their resolved path and launches per call: [FUSED]
 * Notes, describe()).  Host-only; no GPU work.  An empty call (B*S_local == 0)
 * reports zeros.
 * Errors: QNRE_ERR_INVALID_ARG (NULL plan or info, negative sizes),
 * QNRE_ERR_CAPACITY (B*S_local > max_tokens).
 */
typedef struct {
  int device;            /* CUDA device the plan is bound to */
  int pairs_per_cluster; /* 1, or 2: two CTA pairs sharing each W tile by TMA multicast */
  int clusters;          /* clusters the kernel launches (persistent grid): the fewest of
                            those available that finish in as many rounds as all of them */
  int sms;               /* SMs those clusters occupy */
  int row_tiles;         /* 256-token row tiles of the projection */
  int col_tiles;         /* 256-column tiles (two heads each) */
  int work_items;        /* items of the work list (whole tiles or row-tile pairs, and halves) */
  int half_items;        /* 256 x 128 half items among them (a short last round, small problems) */
  int launches;          /* kernel launches of one qnre_forward */
} qnre_plan_info_t;

qnre_status_t qnre_plan_describe(qnre_plan_t plan, int B, int S_local, qnre_plan_info_t* info);

/*
 * qnre_forward -- the fused op on all P virtual ranks at once.  [FUSED], [MATH]:
 *   Y = x W (bf16 operands, fp32 accumulation) with W's columns grouped
 *   Q | K | V (column g*H*128 + h*128 + d);
 *   q, k heads: n_d = Y_d / sqrt(mean_d Y^2 + 1e-6) * w_{q|k}[d]  (fp32),
 *   then RoPE with the token's cos/sin row (fp32); v heads: Y unchanged;
 *   one rounding to bf16, stored to rank h / H_local, local head h % H_local,
 *   global row r_s*S_local + s, for the token at (r_s, b, s).
 *
 *   plan      from qnre_plan_create.
 *   B, S_local batch rows and tokens per rank; B*S_local <= max_tokens.
 *             B*S_local == 0 is an empty call: QNRE_OK, nothing launched.
 *   x         device bf16 [P, B, S_local, hidden] (rank r_s's shard first), 16-B aligned.
 *   w_qkv     device bf16 [hidden, 3*H*128] row-major, 16-B aligned.
 *   q_norm_w, k_norm_w  device bf16 [128] each, 16-B aligned.
 *   cos_sin   device fp32 [n_pos, 128], row p = [cos_0..cos_63 | sin_0..sin_63], 16-B aligned.
 *   n_pos     rows of cos_sin (>= 1).
 *   positions device int32 [P, B, S_local] cos/sin row of every token, or NULL for
 *             row = token index in [P, B, S_local] order.  A position outside
 *             [0, n_pos) is a device-side error: that token's q and k rows are
 *             written as NaN and QNRE_DEVICE_BAD_POSITION is raised.
 *   out       host pointer to the output buffers (see qnre_out_t); outputs must not
 *             overlap x, w_qkv, the norm weights, cos_sin or positions.
 *   stream    CUDA stream.
 *
 * Every output element is written exactly once.  Device-side errors do not
 * surface in the return value (the call does not wait); read them with
 * qnre_plan_device_status.
 */
qnre_status_t qnre_forward(qnre_plan_t plan, int B, int S_local, const void* x, const void* w_qkv,
                           const void* q_norm_w, const void* k_norm_w, const float* cos_sin,
                           int64_t n_pos, const int32_t* positions, const qnre_out_t* out,
                           qnre_stream_t stream);

/*
 * Readiness words ([FUSED], [MATH] "Description": the producer publishes
 * per-chunk readiness words as it stores each destination's band, and a
 * one-CTA wait kernel on a consumer stream acquires them).  Here one word per
 * virtual rank counts the head rows stored into that rank's band.
 *
 * qnre_forward_publish -- qnre_forward that also publishes readiness.
 *   ready   device, [P] uint32, 4-byte aligned, caller-owned; must not overlap any
 *           input or output.  The call zeroes it in stream order, then the kernel
 *           adds to ready[r] (release at GPU scope) each time an epilogue warp has
 *           stored its rows of one head of rank r.  When the forward is complete,
 *           every word equals qnre_ready_target(plan, B, S_local).
 * Other arguments, checks and errors: as qnre_forward.
 */
qnre_status_t qnre_forward_publish(qnre_plan_t plan, int B, int S_local, const void* x, const void* w_qkv,
                                   const void* q_norm_w, const void* k_norm_w, const float* cos_sin,
                                   int64_t n_pos, const int32_t* positions, const qnre_out_t* out,
                                   unsigned* ready, qnre_stream_t stream);

/* The value every readiness word reaches when a forward of (B, S_local) with this
 * plan has stored all of that rank's band.  Host-only; no GPU work. */
qnre_status_t qnre_ready_target(qnre_plan_t plan, int B, int S_local, unsigned* target);

/*
 * qnre_wait_ready -- enqueue on `stream` a one-CTA kernel that waits until every
 * ready[r] (r < P) is >= target, with acquire loads, so work enqueued after it on
 * `stream` sees the bands.  The wait is bounded: after timeout_ns (1 ns .. 10 s)
 * it stops, raises QNRE_DEVICE_READY_TIMEOUT in the plan's status word and
 * returns, leaving the context usable.
 *   ready   device [P] uint32 written by qnre_forward_publish.
 * A wait kernel that runs while its producer is still running (on another
 * stream) depends on both being resident at once, which nothing guarantees on
 * one GPU; order the wait after the producer unless the caller knows they fit.
 */
qnre_status_t qnre_wait_ready(qnre_plan_t plan, const unsigned* ready, unsigned target, uint64_t timeout_ns,
                              qnre_stream_t stream);

/* Read (and, if clear != 0, reset) the plan's device status bits
 * (QNRE_DEVICE_*).  Waits for `stream`, then copies 4 bytes to the host.
 * Returns QNRE_ERR_DEVICE when any bit is set, QNRE_OK otherwise. */
qnre_status_t qnre_plan_device_status(qnre_plan_t plan, qnre_stream_t stream, unsigned* bits,
                                      int clear);

/* qnre_debug_bounds -- the debug build's count of skipped accesses.
 * libqnre_debug.so (the same sources built with QNRE_DEBUG_BOUNDS=1) checks
 * every load and store of the layout copy kernels and of the Sage2 kernels
 * against the byte range of the buffer the call was given for it (the same
 * ranges the alias checks use), and every head-row store of the fused epilogue
 * against its output tensor.  An access outside its range is not performed:
 * the layout and Sage2 kernels count it here, the fused kernel raises
 * QNRE_DEVICE_BOUNDS in the plan's status word.  Nothing traps; the calls'
 * results are then incomplete, and a correct build never counts anything.
 *   violations  host, out: accesses skipped since the last reset (all kernels,
 *               all streams, this device).
 *   reset       non-zero: set the count to 0 after reading it.
 * Synchronises the device (a symbol copy).  Errors: QNRE_ERR_INVALID_ARG for a
 * NULL pointer, QNRE_ERR_UNSUPPORTED in the release build (libqnre.so, which
 * has no checks), QNRE_ERR_CUDA when the copy fails. */
qnre_status_t qnre_debug_bounds(unsigned long long* violations, int reset);

/*
 * qnre_forward_noalloc -- qnre_forward without a plan and without any device
 * allocation.  The pages have no counterpart: this entry point exists for
 * callers that cannot call cudaMalloc when they run the projection (a
 * framework whose memory pool forbids raw device allocations, a runtime that
 * has handed all device memory to its own allocator, a server that must not
 * allocate once it is running).  qnre_plan_create allocates the plan's device
 * status word, so such callers cannot make a plan; this call keeps that word
 * in a static device array of the library instead.
 *
 *   hidden, num_heads, P, layout, rope_style, flags
 *             the geometry qnre_plan_create takes (head_dim is 128), with the
 *             same rules and error codes; flags is 0 or QNRE_FLAG_EPILOGUE_OFF
 *             (this call always runs the fused kernel one CTA pair per cluster).
 *   B .. out  as in qnre_forward (there is no max_tokens; see the limit below).
 *   device_status_out  device pointer to one unsigned (4-byte aligned), or NULL:
 *             receives this call's QNRE_DEVICE_* bits, in stream order.
 *   stream    CUDA stream.
 *
 * Scratch and limits: the library holds a 256-byte static device array on
 * every GPU that loads it, until the process exits; a call uses 16 bytes of it.
 * Sizes beyond what the call serves are rejected with QNRE_ERR_CAPACITY: a
 * status block larger than the array, or P*B*S_local tokens beyond 2^31 - 256.
 * The call makes no cudaMalloc, cudaFree or other allocating call.
 *
 * Set-up: the first call on each device (with that device current) looks up
 * the array's device address with cudaGetSymbolAddress and sets the kernel's
 * shared-memory limit.  Make that first call before any stream capture.
 *
 * Sharing: every call on a device uses the same array.  After its kernel, a
 * call copies the status word to device_status_out and clears it, so the next
 * call starts from zero; calls that overlap on the GPU (different streams, no
 * ordering between them) race on the word and may see each other's bits.
 * A rejected call enqueues nothing.
 */
qnre_status_t qnre_forward_noalloc(int hidden, int num_heads, int P, qnre_layout_t layout,
                                   qnre_rope_t rope_style, unsigned flags, int B, int S_local,
                                   const void* x, const void* w_qkv, const void* q_norm_w,
                                   const void* k_norm_w, const float* cos_sin, int64_t n_pos,
                                   const int32_t* positions, const qnre_out_t* out,
                                   unsigned* device_status_out, qnre_stream_t stream);

/*
 * ulysses_pack_head_chunk -- [PACK]: select local head band
 * [head_offset, head_offset + head_count) inside every destination rank's
 * H/world_size head slice of q, k and v, fusing q|k|v along the last axis:
 *
 *   out[b, s, r*head_count + j, c*D + d] = X_c[b, s, r*(H/world_size) + head_offset + j, d]
 *   for X_0 = q, X_1 = k, X_2 = v, r < world_size, j < head_count.
 *
 *   q, k, v     host pointers to views [B, S_local, H, D] with positive strides, equal
 *               shapes and dtype (bf16, fp16 or fp32); they may overlap each other
 *               (e.g. slices of one fused projection buffer).
 *   world_size  >= 1, H % world_size == 0.
 *   head_offset, head_count  0 <= head_offset, head_count >= 1,
 *               head_offset + head_count <= H/world_size.
 *   out         device, contiguous [B, S_local, world_size*head_count, 3*D] of the
 *               same dtype; must not overlap the storage range of q, k or v.
 *   stream      CUDA stream.
 *
 * Element-size-aligned pointers are required (QNRE_ERR_ALIGNMENT otherwise);
 * 16-byte aligned rows with unit innermost stride take the vectorised path.
 * Offsets are 64-bit, so the pages' int32 payload limit ([PR5027]) does not
 * apply.  B*S_local == 0 is an empty call (QNRE_OK, nothing launched).
 */
qnre_status_t ulysses_pack_head_chunk(const qnre_tensor4_t* q, const qnre_tensor4_t* k,
                                      const qnre_tensor4_t* v, int world_size, int head_offset,
                                      int head_count, void* out, qnre_stream_t stream);

/*
 * ulysses_merge_output_head_chunk -- [MERGE]: write one gathered output head band
 * into the full output, leaving every other element untouched:
 *
 *   out[b, s, r*local_heads + head_offset + j, d] = received[b, s, r*head_count + j, d]
 *   for r < world_size, j < head_count = received.shape[2] / world_size.
 *
 *   received    host pointer to a view [B, S_local, world_size*head_count, D] with
 *               positive strides (the pages' input is contiguous; any positive
 *               strides are accepted).
 *   world_size  >= 1, divides received.shape[2].
 *   local_heads heads per rank in out (>= 1).
 *   head_offset 0 <= head_offset, head_offset + head_count <= local_heads.
 *   out         device, contiguous [B, S_local, world_size*local_heads, D] of the same
 *               dtype; must not overlap received's storage range.
 *   stream      CUDA stream.
 *
 * Same alignment, vectorisation and int32 rules as ulysses_pack_head_chunk.
 */
qnre_status_t ulysses_merge_output_head_chunk(const qnre_tensor4_t* received, int world_size,
                                              int local_heads, int head_offset, void* out,
                                              qnre_stream_t stream);

/*
 * Schedule forms ([PR5027] Description: uneven head schedules; [HC] example
 * schedule): every chunk of a schedule in one launch, with the same results as
 * calling the single-chunk function for each chunk in order.
 *
 * ulysses_pack_head_chunk_schedule -- chunk i = (head_offsets[i], head_counts[i])
 *   of the same q, k, v views into outs[i] (as ulysses_pack_head_chunk).
 *   head_offsets, head_counts, outs   host arrays of num_chunks entries.
 * ulysses_merge_output_head_chunk_schedule -- chunk i merges received[i] (its own
 *   head count = shape[2] / world_size) at band head_offsets[i] of the same out
 *   (as ulysses_merge_output_head_chunk).
 *   received, head_offsets   host arrays of num_chunks entries; the received views
 *   share B, S, D and dtype.
 * Errors: each chunk's checks as in the single-chunk call; num_chunks < 1 or a NULL
 * array -> QNRE_ERR_INVALID_ARG; num_chunks > 8 -> QNRE_ERR_CAPACITY; pack outputs
 * that overlap one another -> QNRE_ERR_ALIAS; merge bands that overlap one another
 * (the chunks run in any order) -> QNRE_ERR_INVALID_ARG.  Chunks whose copies need
 * different copy units (alignment or innermost strides) are launched one by one.
 * These calls are the ones meant to run beside the projection (the head-chunk
 * pipeline), so they load and store with the cache-streaming policy: the copied
 * lines leave L2 first and the projection's operands stay.  Alone they run as fast
 * as the single-chunk calls (within 1 %); beside the fused projection the step
 * gains.
 */
qnre_status_t ulysses_pack_head_chunk_schedule(const qnre_tensor4_t* q, const qnre_tensor4_t* k,
                                               const qnre_tensor4_t* v, int world_size, int num_chunks,
                                               const int* head_offsets, const int* head_counts,
                                               void* const* outs, qnre_stream_t stream);

qnre_status_t ulysses_merge_output_head_chunk_schedule(const qnre_tensor4_t* const* received, int world_size,
                                                       int local_heads, int num_chunks, const int* head_offsets,
                                                       void* out, qnre_stream_t stream);

/*
 * ulysses_scatter_heads -- [ULY] scatter_heads for all P virtual ranks at once:
 * [B, S_local, H, D] per rank -> [B, S_global, H_local, D] per rank, where rank r
 * keeps heads [r*H_local, (r+1)*H_local) of the whole sequence:
 *
 *   out[r, b, r_s*S_local + s, hl, d] = x[r_s, b, s, r*H_local + hl, d]
 *
 *   x       device, contiguous [P, B, S_local, H, D] (rank r_s's shard first).
 *   P       virtual ranks (>= 1), H % P == 0 (else QNRE_ERR_INVALID_ARG).  P == 1 copies.
 *   dtype   qnre_dtype_t of x and out.
 *   out     device, contiguous [P, B, P*S_local, H/P, D]; must not overlap x.
 * P*B <= 65535.  B*S_local == 0 is an empty call.
 */
qnre_status_t ulysses_scatter_heads(const void* x, int P, int B, int S_local, int H, int D, int32_t dtype,
                                    void* out, qnre_stream_t stream);

/*
 * ulysses_gather_heads -- [ULY] gather_heads for all P virtual ranks, the inverse
 * of ulysses_scatter_heads:
 *
 *   out[r_s, b, s, r*H_local + hl, d] = y[r, b, r_s*S_local + s, hl, d]
 *
 *   y       device, contiguous [P, B, S_global, H_local, D]; S_global % P == 0.
 *   out     device, contiguous [P, B, S_global/P, P*H_local, D]; must not overlap y.
 */
qnre_status_t ulysses_gather_heads(const void* y, int P, int B, int S_global, int H_local, int D, int32_t dtype,
                                   void* out, qnre_stream_t stream);

/*
 * ulysses_pack_output_sequence_chunk -- the sequence split of one attention-output
 * band that the output exchange sends ([XCHG] gather_output_head_chunk: the NCCL
 * path packs the sequence split into staging; chunk r goes to rank r, which owns
 * sequence rows [r*S_local, (r+1)*S_local)):
 *
 *   out[r, b, s, j, d] = x[b, r*S_local + s, j, d],   S_local = S_global / world_size
 *
 *   x           host pointer to a view [B, S_global, head_count, D], positive strides.
 *   world_size  >= 1, divides S_global.
 *   out         device, contiguous [world_size, B, S_local, head_count, D]; must not
 *               overlap x.
 */
qnre_status_t ulysses_pack_output_sequence_chunk(const qnre_tensor4_t* x, int world_size, void* out,
                                                 qnre_stream_t stream);

/*
 * ulysses_gather_output_head_chunk -- [XCHG] gather_output_head_chunk for all P
 * virtual ranks at once: the sequence-split pack on every rank, the exchange and
 * the merge into each rank's full output, as one copy.  Only the band is written:
 *
 *   out[r2, b, s, r*local_heads + head_offset + j, d] = x[r, b, r2*S_local + s, j, d]
 *
 *   x           device, contiguous [P, B, S_global, head_count, D]: rank r's attention
 *               output band over the whole sequence.  S_global % P == 0.
 *   local_heads, head_offset  0 <= head_offset, head_offset + head_count <= local_heads.
 *   out         device, contiguous [P, B, S_global/P, P*local_heads, D]; other heads
 *               keep their values; must not overlap x.
 */
qnre_status_t ulysses_gather_output_head_chunk(const void* x, int P, int B, int S_global, int head_count, int D,
                                               int32_t dtype, int local_heads, int head_offset, void* out,
                                               qnre_stream_t stream);

/*
 * ulysses_scatter_qkv_head_chunk -- [XCHG] scatter_qkv_head_chunk for all P virtual
 * ranks at once: the head-chunk pack on every rank and the exchange of its
 * destination slots, as one copy.  Rank r receives band
 * [head_offset, head_offset + head_count) of its head slice for the whole sequence:
 *
 *   out[r, b, r_s*S_local + s, j, c*D + d] = X_c[r_s*B + b, s, r*H_local + head_offset + j, d]
 *
 *   q, k, v     host pointers to views [P*B, S_local, H, D] (rank r_s's batch rows
 *               first), positive strides, equal shapes and dtype.
 *   P           virtual ranks; P divides the first extent and H.
 *   out         device, contiguous [P, B, P*S_local, head_count, 3*D]; must not overlap
 *               q, k or v.
 */
qnre_status_t ulysses_scatter_qkv_head_chunk(const qnre_tensor4_t* q, const qnre_tensor4_t* k,
                                             const qnre_tensor4_t* v, int P, int head_offset, int head_count,
                                             void* out, qnre_stream_t stream);

/*
 * Sage2 low-precision QKV exchange over P virtual ranks ([LOWP]): FP32
 * statistics over the global sequence, INT8 Q per group of 32 tokens, INT8
 * (K - global per-channel mean of K) per group of 64 tokens, FP8 E4M3 V with a
 * per-channel scale, written into every destination rank's exchanged layout.
 * Arithmetic (readings of the page): stored scale = amax / 127 (INT8) or
 * amax / 448 (E4M3) in fp32; code = x * (127 / amax) (or x * (448 / amax))
 * rounded to nearest even, saturated, the reciprocal taken once per group or
 * channel and 0 when amax is 0; the K mean is sum / U, the sum taken in a fixed
 * order (rows of a source rank in chunks of 256, chunks in order, ranks in
 * order); rows at or beyond U are code 0 and take no part in any amax.
 *
 * ulysses_sage2_workspace_bytes -- bytes of scratch ulysses_sage2_scatter_qkv
 * needs for (P, B, L, H, D); host-only, touches no device.
 *
 * ulysses_sage2_scatter_qkv --
 *   q, k, v        host pointers to views [P*B, L, H, D] (rank r_s's batch rows first),
 *                  bf16 or fp16, equal shapes; channel axis contiguous, every row and
 *                  the base 16-byte aligned ([LOWP] scatter_qkv).  Rows at or beyond
 *                  the used prefix must be zero (they enter the K sum).
 *   P              virtual ranks, divides H and the first extent.  S = P*L.
 *   used_sequence  U in (0, S].
 *   q_out, k_out   device int8 [P, B, S, H/P, D], 16-byte aligned.
 *   v_out          device E4M3 codes [P, B, D, H/P, S_pad], S_pad = S rounded up to 64,
 *                  16-byte aligned; the padding is written as code 0.
 *   q_scale        device fp32 [P, B, H/P, ceil(U/32)];  k_scale fp32 [P, B, H/P, ceil(U/64)];
 *   v_scale        device fp32 [P, B, H/P, D].
 *   workspace      device scratch of at least ulysses_sage2_workspace_bytes, 16-byte
 *                  aligned, caller-owned; overwritten by the call.
 * Every output element is written.  No output may overlap an input, another output
 * or the workspace (QNRE_ERR_ALIAS).  D must be 64 or 128 (QNRE_ERR_UNSUPPORTED
 * otherwise); S above 65535*64, P*B or H above 65535 give QNRE_ERR_CAPACITY.
 * Three launches on `stream`; inputs must be finite.
 */
qnre_status_t ulysses_sage2_workspace_bytes(int P, int B, int L, int H, int D, uint64_t* bytes);

qnre_status_t ulysses_sage2_scatter_qkv(const qnre_tensor4_t* q, const qnre_tensor4_t* k,
                                        const qnre_tensor4_t* v, int P, int used_sequence, void* q_out,
                                        void* k_out, void* v_out, float* q_scale, float* k_scale,
                                        float* v_scale, void* workspace, uint64_t workspace_bytes,
                                        qnre_stream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* QNRE_H_ */
