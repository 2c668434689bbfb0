// sage2.cu -- Sage2 low-precision QKV exchange over P virtual ranks for sm_103a
// ("Prepared Low-Precision QKV Exchange", flashinfer.comm API reference):
// FP32 statistics over the global sequence, INT8 Q in groups of 32 tokens, INT8
// K minus its global per-channel mean in groups of 64 tokens, FP8 E4M3 V with a
// per-channel scale, all written straight into every destination rank's
// exchanged layout.
//
// Three launches, each deterministic:
//   1. stats_partial: one CTA per (16 or 32 heads, 256-row chunk of a source
//      rank, batch); each thread owns 8 channels of one head (16-byte loads,
//      eight rows in flight) and sums K / takes max|V| down them row by row;
//   2. stats_final: four warps per (head, batch, 32 channels); warp w adds a
//      quarter of the (source rank, chunk) sums in order, the quarters are added
//      in warp order -> K mean = sum / U, V scale = max / 448 and the V
//      reciprocal 448 / max;
//   3. quantize: one CTA per (head, 64-row global group, batch); each thread
//      owns 8 channels of 4 (D = 128) or 2 (D = 64) consecutive rows and lands
//      all of its V, Q and K chunks in shared memory with 16-byte asynchronous
//      copies before touching any (48 KiB in flight per CTA at D = 128, four
//      CTAs per SM); two Q groups and one K group reduce their amax across the
//      CTA; each group or channel takes one reciprocal (127 / amax, 448 /
//      amax), every value one fp32 multiply and one rounding (INT8: nearest
//      even, by an fp32 add of 1.5 * 2^23; E4M3: nearest even, saturating).
//      Maxima are taken on the packed 16-bit inputs, where they are exact.  V
//      codes are turned around in shared memory so that each channel's 64
//      codes leave as whole 16-byte stores.
// Every float decision (sums, maxima, scales, quotients) is a single IEEE fp32
// operation in a fixed order, so the codes are reproducible bit for bit.
#include "../../include/qnre.h"
#include "api_util.cuh"
#include "debug_bounds.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <utility>

#ifndef QNRE_SAGE2_QUANT_MIN_BLOCKS
#define QNRE_SAGE2_QUANT_MIN_BLOCKS 4  // resident quantize CTAs per SM the register budget aims at
#endif

namespace {

using namespace qnre::api;
using qnre::Extent;

constexpr int kChunk = 256;  // rows per statistics chunk
constexpr int kQGroup = 32;
constexpr int kKGroup = 64;
constexpr int kVPad = 64;
constexpr int kVRowWords = 17;  // 64 code bytes + one pad word per staged V channel row

struct View {
  const char* data;
  long long sz, ss, sh;  // bytes: batch (z = r_s*B + b), sequence, head; d is contiguous
};

// ---------------------------------------------------------------------------
// Packed 16-bit floats (two per word, element 2p in the low half): conversions
// and lane-wise max / min (exact: a max or min of 16-bit values is one of them).
// ---------------------------------------------------------------------------
template <bool BF16>
__device__ __forceinline__ float lo16(uint32_t w) {
  if (BF16) return __uint_as_float(w << 16);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
template <bool BF16>
__device__ __forceinline__ float hi16(uint32_t w) {
  if (BF16) return __uint_as_float(w & 0xFFFF0000u);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
template <bool BF16, bool MAX>
__device__ __forceinline__ uint32_t minmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  if (BF16) {
    __nv_bfloat162 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    const __nv_bfloat162 m = MAX ? __hmax2(x, y) : __hmin2(x, y);
    memcpy(&r, &m, 4);
  } else {
    __half2 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    const __half2 m = MAX ? __hmax2(x, y) : __hmin2(x, y);
    memcpy(&r, &m, 4);
  }
  return r;
}
template <bool BF16>
__device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
  return minmax2<BF16, true>(a, b);
}
template <bool BF16>
__device__ __forceinline__ uint32_t min2(uint32_t a, uint32_t b) {
  return minmax2<BF16, false>(a, b);
}
template <bool BF16>
__device__ __forceinline__ uint4 max2(uint4 a, uint4 b) {
  return make_uint4(max2<BF16>(a.x, b.x), max2<BF16>(a.y, b.y), max2<BF16>(a.z, b.z), max2<BF16>(a.w, b.w));
}
template <bool BF16>
__device__ __forceinline__ uint4 min2(uint4 a, uint4 b) {
  return make_uint4(min2<BF16>(a.x, b.x), min2<BF16>(a.y, b.y), min2<BF16>(a.z, b.z), min2<BF16>(a.w, b.w));
}
// |x| of both halves of every word (clears the sign bits)
__device__ __forceinline__ uint4 abs2(uint4 a) {
  return make_uint4(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu, a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu);
}
template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    f[2 * p] = lo16<BF16>(w[p]);
    f[2 * p + 1] = hi16<BF16>(w[p]);
  }
}

// top / amax, or 0 when amax is 0 (then every code of the group or channel is 0).
__device__ __forceinline__ float reciprocal(float amax, float top) {
  return amax > 0.f ? __fdiv_rn(top, amax) : 0.f;
}

// The three launches are programmatic dependent launches: each waits here until
// the grid before it in the stream has completed and its writes are visible,
// before it reads anything, then lets the next launch begin its set-up.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// 1. Chunk statistics
// ---------------------------------------------------------------------------
struct StatsArgs {
  View k, v;
  float* ksum;  // [P, chunks, B, H, D]
  float* vmax;  // [P, chunks, B, H, D]: max |V| over the chunk's rows below U
  int P, B, L, H, D, chunks, U;
#if QNRE_DEBUG_BOUNDS
  Extent k_ext, v_ext, ws_ext;
#endif
};

// One CTA: one 256-row chunk of one source rank, 256 / (D / 8) heads.  Thread t
// owns 8 channels (16 bytes) of one head and walks the chunk's rows in order,
// so each column's sum is the same row-by-row fp32 sum the oracle takes.
// kStatsRows rows of K and V are loaded before any is added (2 x 8 x 16 bytes
// in flight per thread), enough to keep HBM busy even when the grid is small.
constexpr int kStatsRows = 8;
template <bool BF16>
__global__ void __launch_bounds__(256, 2) stats_partial_kernel(const StatsArgs a) {
  pdl_enter();
  const int tpr = a.D / 8;  // threads per head row
  const int h = blockIdx.x * (256 / tpr) + threadIdx.x / tpr;
  if (h >= a.H) return;
  const int c0 = (threadIdx.x % tpr) * 8;
  const int chunk = blockIdx.y, z = blockIdx.z;  // z = r_s * B + b
  const int r_s = z / a.B, b = z - r_s * a.B;
  const int l0 = chunk * kChunk, l1 = min(a.L, l0 + kChunk);
  // local rows below live_end lie below U in the global sequence
  const int live_end = min(l1, max(l0, a.U - r_s * a.L));
  const char* kp = a.k.data + z * a.k.sz + h * a.k.sh + c0 * 2;
  const char* vp = a.v.data + z * a.v.sz + h * a.v.sh + c0 * 2;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  uint4 vm = make_uint4(0, 0, 0, 0);
  int l = l0;
  for (; l + kStatsRows <= l1; l += kStatsRows) {
    uint4 kw[kStatsRows], vw[kStatsRows];
#pragma unroll
    for (int u = 0; u < kStatsRows; ++u) {
      const char* ku = kp + static_cast<long long>(l + u) * a.k.ss;
      const char* vu = vp + static_cast<long long>(l + u) * a.v.ss;
      kw[u] = QNRE_ACCESS_OK(ku, 16, a.k_ext) ? *reinterpret_cast<const uint4*>(ku) : make_uint4(0, 0, 0, 0);
      vw[u] = QNRE_ACCESS_OK(vu, 16, a.v_ext) ? *reinterpret_cast<const uint4*>(vu) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kStatsRows; ++u) {
      float f[8];
      unpack8<BF16>(kw[u], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
      if (l + u < live_end) vm = max2<BF16>(vm, abs2(vw[u]));
    }
  }
  for (; l < l1; ++l) {
    const char* ku = kp + static_cast<long long>(l) * a.k.ss;
    const char* vu = vp + static_cast<long long>(l) * a.v.ss;
    const uint4 kw = QNRE_ACCESS_OK(ku, 16, a.k_ext) ? *reinterpret_cast<const uint4*>(ku) : make_uint4(0, 0, 0, 0);
    const uint4 vw = QNRE_ACCESS_OK(vu, 16, a.v_ext) ? *reinterpret_cast<const uint4*>(vu) : make_uint4(0, 0, 0, 0);
    float f[8];
    unpack8<BF16>(kw, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
    if (l < live_end) vm = max2<BF16>(vm, abs2(vw));
  }
  float vf[8];
  unpack8<BF16>(vm, vf);
  const long long o = ((((static_cast<long long>(r_s) * a.chunks + chunk) * a.B + b) * a.H + h) * a.D) + c0;
  if (!QNRE_ACCESS_OK(a.ksum + o, 32, a.ws_ext) || !QNRE_ACCESS_OK(a.vmax + o, 32, a.ws_ext)) return;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a.ksum[o + i] = acc[i];
    a.vmax[o + i] = vf[i];
  }
}

// ---------------------------------------------------------------------------
// 2. Global statistics
// ---------------------------------------------------------------------------
struct FinalArgs {
  const float* ksum;
  const float* vmax;
  float* kmean;    // [B, H, D]
  float* vinv;     // [B, H, D]: 448 / max |V| (0 where the max is 0)
  float* v_scale;  // [P, B, H_l, D]
  int P, B, H, H_l, D, chunks, U;
#if QNRE_DEBUG_BOUNDS
  Extent ws_ext, v_scale_ext;
#endif
};

// One CTA of four warps per (head, batch, 32 channels): warp w sums its quarter
// of the (source rank, chunk) partials in order, 16 loads in flight per thread,
// and the four quarter sums are added in warp order, so the K sum is the same
// fixed-order fp32 sum on every run.
constexpr int kFinalWarps = 4;
__global__ void __launch_bounds__(32 * kFinalWarps) stats_final_kernel(const FinalArgs a) {
  pdl_enter();
  const int lane = threadIdx.x & 31, wq = threadIdx.x >> 5;
  const int d = blockIdx.z * 32 + lane, h = blockIdx.x, b = blockIdx.y;
  // partial (r, c) sits at ((r * chunks + c) * B + b) * H * D + h * D + d: linear in
  // i = r * chunks + c with step B * H * D
  const long long step = static_cast<long long>(a.B) * a.H * a.D;
  const int n = a.P * a.chunks;
  const int per = (n + kFinalWarps - 1) / kFinalWarps;
  const int i0 = min(n, wq * per), i1 = min(n, i0 + per);
  const long long base = (static_cast<long long>(b) * a.H + h) * a.D + d;
  const float* kp = a.ksum + base + i0 * step;
  const float* vp = a.vmax + base + i0 * step;
  float part = 0.f, vm = 0.f;
  constexpr int kAhead = 16;  // loads in flight per thread; the sum still runs in order
  int i = i0;
  for (; i + kAhead <= i1; i += kAhead, kp += kAhead * step, vp += kAhead * step) {
    float ks[kAhead], vs[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      ks[u] = kp[u * step];
      vs[u] = vp[u * step];
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      part = __fadd_rn(part, ks[u]);
      vm = fmaxf(vm, vs[u]);
    }
  }
  for (; i < i1; ++i, kp += step, vp += step) {
    part = __fadd_rn(part, *kp);
    vm = fmaxf(vm, *vp);
  }
  __shared__ float ps[kFinalWarps][32], pv[kFinalWarps][32];
  ps[wq][lane] = part;
  pv[wq][lane] = vm;
  __syncthreads();
  if (wq != 0) return;
  float total = 0.f;
#pragma unroll
  for (int w = 0; w < kFinalWarps; ++w) {
    total = __fadd_rn(total, ps[w][lane]);
    vm = fmaxf(vm, pv[w][lane]);
  }
  const long long o = (static_cast<long long>(b) * a.H + h) * a.D + d;
  if (QNRE_ACCESS_OK(a.kmean + o, 4, a.ws_ext)) a.kmean[o] = __fdiv_rn(total, static_cast<float>(a.U));
  if (QNRE_ACCESS_OK(a.vinv + o, 4, a.ws_ext)) a.vinv[o] = reciprocal(vm, 448.0f);
  const int r = h / a.H_l, hl = h - r * a.H_l;
  float* vs = a.v_scale + ((static_cast<long long>(r) * a.B + b) * a.H_l + hl) * a.D + d;
  if (QNRE_ACCESS_OK(vs, 4, a.v_scale_ext)) *vs = __fdiv_rn(vm, 448.0f);
}

// ---------------------------------------------------------------------------
// 3. Codes
// ---------------------------------------------------------------------------
struct QuantArgs {
  View q, k, v;
  const float* kmean;  // [B, H, D]
  const float* vinv;   // [B, H, D]: 448 / max |V| over the used sequence, 0 where that max is 0
  int8_t* q_out;       // [P, B, S, H_l, D]
  int8_t* k_out;
  uint8_t* v_out;  // [P, B, D, H_l, S_pad]
  float* q_scale;  // [P, B, H_l, wq]
  float* k_scale;  // [P, B, H_l, wk]
  int P, B, L, H, H_l, D, S, S_pad, U, wq, wk;
#if QNRE_DEBUG_BOUNDS
  Extent src_ext[3];  // v, q, k (landing order)
  Extent q_out_ext, k_out_ext, v_out_ext, q_scale_ext, k_scale_ext;
#endif
};

// Max over the CTA's 256 threads (holds two barriers).
__device__ __forceinline__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
  return m;
}

// INT8 code of x * inv: the product is rounded to fp32 first (one multiply),
// then to the nearest integer, ties to even, by adding 1.5 * 2^23: for
// |y| < 2^22 the sum's unit in the last place is 1, so the fp32 addition itself
// rounds y to an integer, and the low byte of the sum's bits is that integer
// in two's complement.  |y| <= 127 (1 + 2^-23)^2 < 127.5 because |x| <= amax
// and inv = 127 / amax, so the codes stay in [-127, 127] with no clamp.
__device__ __forceinline__ uint32_t int8_bits(float x, float inv) {
  return __float_as_uint(__fadd_rn(__fmul_rn(x, inv), 12582912.0f));
}
// low bytes of four words -> one word (a in byte 0)
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// 16-byte asynchronous copy global -> shared (L1 bypassed) and its group fences.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(a), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// eight consecutive floats (16-byte aligned) as two 16-byte loads
__device__ __forceinline__ void load_f8(const float* p, float (&f)[8]) {
  const float4 x = reinterpret_cast<const float4*>(p)[0], y = reinterpret_cast<const float4*>(p)[1];
  f[0] = x.x;
  f[1] = x.y;
  f[2] = x.z;
  f[3] = x.w;
  f[4] = y.x;
  f[5] = y.y;
  f[6] = y.z;
  f[7] = y.w;
}

template <int RPT>
constexpr int quantize_smem_bytes() {  // V, Q, K landing slots
  return 3 * RPT * 256 * 16;
}

// One CTA: one 64-row global group of one head.  Thread t owns 8 channels
// (16 bytes) of RPT consecutive rows (RPT = 4 for D = 128, 2 for D = 64).
// Every thread first issues all of its V, Q and K copies into shared memory
// (three commit groups, in that order; rows at or past U are zero-filled
// instead) and then consumes only the chunks it copied itself, so shared
// memory is a landing zone that keeps 3 * RPT * 16 bytes per thread in flight
// without holding registers; only the group maxima cross threads.  Shared
// layout [tensor][u][thread][16 B]: a warp's 16-byte accesses for one
// (tensor, u) are contiguous, so they are conflict free.
template <int RPT, bool BF16>
__global__ void __launch_bounds__(256, QNRE_SAGE2_QUANT_MIN_BLOCKS) quantize_kernel(const QuantArgs a) {
  pdl_enter();
  extern __shared__ uint4 land[];  // [3][RPT][256]
  __shared__ float red[8];
  constexpr int kTpr = 4 * RPT;  // threads per row: 16 for D = 128, 8 for D = 64
  const int tid = threadIdx.x;
  const int j = tid / kTpr, cv = tid - j * kTpr;
  // heads vary fastest across the grid, so CTAs that run together read
  // neighbouring heads of the same rows (long contiguous runs per row)
  const int h = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int r = h / a.H_l, hl = h - r * a.H_l;
  const int s0 = g * kKGroup, sr = s0 + j * RPT;  // this thread's first row
  const int c0 = cv * 8;
  const int n_live = max(0, min(RPT, a.U - sr));  // rows sr .. sr + n_live - 1 lie below U
  const long long stat = (static_cast<long long>(b) * a.H + h) * a.D + c0;
  auto slot = [&](int c, int u) -> uint4& { return land[(c * RPT + u) * 256 + tid]; };
  {
    int zr[RPT], lr[RPT];  // batch index r_s*B + b and local row of each row (rows are consecutive)
    {
      int r_s = sr / a.L, l = sr - r_s * a.L;
#pragma unroll
      for (int u = 0; u < RPT; ++u) {
        zr[u] = r_s * a.B + b;
        lr[u] = l;
        if (++l == a.L) {
          l = 0;
          ++r_s;
        }
      }
    }
    const View* src[3] = {&a.v, &a.q, &a.k};
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      const View& t = *src[c];
      const char* base = t.data + h * t.sh + c0 * 2;
#pragma unroll
      for (int u = 0; u < RPT; ++u) {
        const char* gp = base + static_cast<long long>(zr[u]) * t.sz + static_cast<long long>(lr[u]) * t.ss;
        if (u < n_live && QNRE_ACCESS_OK(gp, 16, a.src_ext[c]))
          cp_async16(&slot(c, u), gp);
        else
          slot(c, u) = make_uint4(0, 0, 0, 0);  // a dead row reads as +0
      }
      cp_async_commit();
    }
  }
  uint32_t* vt = reinterpret_cast<uint32_t*>(land);  // transposed V codes, over the V landing slots
  static_assert(32 * RPT * kVRowWords * 4 <= RPT * 256 * 16, "D = 32 * RPT staged rows fit the V landing slots");

  // V: E4M3 codes with the channel's reciprocal, two rows per conversion; for
  // each of the 8 channels, RPT consecutive rows are RPT contiguous bytes (one
  // word per channel).  Dead rows are +0 and encode as 0x00.
  uint32_t vword[8];
  {
    float vinv[8];
    load_f8(a.vinv + stat, vinv);
    cp_async_wait<2>();
    uint32_t pr[RPT / 2][8];
#pragma unroll
    for (int u = 0; u < RPT; u += 2) {
      float v0[8], v1[8];
      unpack8<BF16>(slot(0, u), v0);
      unpack8<BF16>(slot(0, u + 1), v1);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        pr[u / 2][i] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(v0[i], vinv[i]), __fmul_rn(v1[i], vinv[i])), __NV_SATFINITE,
            __NV_E4M3));  // row u in the low byte
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) vword[i] = RPT == 4 ? __byte_perm(pr[0][i], pr[RPT / 2 - 1][i], 0x5410) : pr[0][i];
  }

  const long long sc_base = (static_cast<long long>(r) * a.B + b) * a.H_l + hl;
  const long long row_step = static_cast<long long>(a.H_l) * a.D;  // bytes between output rows
  const long long out0 = ((static_cast<long long>(r) * a.B + b) * a.S + sr) * row_step + hl * a.D + c0;

  // Q: group maximum (exact in the 16-bit domain), then codes (8 bytes per row).
  {
    cp_async_wait<1>();
    uint4 m4 = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < RPT; ++u) m4 = max2<BF16>(m4, abs2(slot(1, u)));
    const uint32_t m2 = max2<BF16>(max2<BF16>(m4.x, m4.y), max2<BF16>(m4.z, m4.w));
    const float xmax = fmaxf(lo16<BF16>(m2), hi16<BF16>(m2));
    const bool first_half = (j * RPT) < kQGroup;  // rows [0, 32) form Q group 2g, rows [32, 64) group 2g + 1
    const float m0 = block_max(first_half ? xmax : 0.f, red);
    const float m1 = block_max(first_half ? 0.f : xmax, red);
    const float inv = reciprocal(first_half ? m0 : m1, 127.0f);
    // every thread has read its V landing slots (block_max holds barriers):
    // reuse them to turn the V codes around into [channel][64 rows] rows of
    // kVRowWords words, so the global stores write whole 64-byte rows
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (RPT == 4) vt[(c0 + i) * kVRowWords + j] = vword[i];
      else reinterpret_cast<uint16_t*>(vt)[(c0 + i) * kVRowWords * 2 + j] = static_cast<uint16_t>(vword[i]);
    }
    if (tid == 0) {
      const int gq = 2 * g;
      float* qs = a.q_scale + sc_base * a.wq + gq;
      if (gq < a.wq && QNRE_ACCESS_OK(qs, 4, a.q_scale_ext)) qs[0] = __fdiv_rn(m0, 127.0f);
      if (gq + 1 < a.wq && QNRE_ACCESS_OK(qs + 1, 4, a.q_scale_ext)) qs[1] = __fdiv_rn(m1, 127.0f);
    }
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
      int8_t* qd = a.q_out + out0 + u * row_step;
      if (sr + u < a.S && QNRE_ACCESS_OK(qd, 8, a.q_out_ext)) {
        float f[8];
        unpack8<BF16>(slot(1, u), f);  // dead rows are +0 and encode as 0
        uint32_t t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = int8_bits(f[i], inv);
        *reinterpret_cast<uint2*>(qd) =
            make_uint2(pack_low_bytes(t[0], t[1], t[2], t[3]), pack_low_bytes(t[4], t[5], t[6], t[7]));
      }
    }
  }

  // K - mean: per channel, max |k - mean| over the live rows equals
  // max(|kmax - mean|, |kmin - mean|) because fp32 subtraction is monotone.
  {
    float mean[8];
    load_f8(a.kmean + stat, mean);
    cp_async_wait<0>();
    float xmax = 0.f;
    if (n_live > 0) {
      uint4 kmx = slot(2, 0), kmn = kmx;  // per-channel max and min over the live rows
#pragma unroll
      for (int u = 1; u < RPT; ++u) {
        if (u < n_live) {
          const uint4 w = slot(2, u);
          kmx = max2<BF16>(kmx, w);
          kmn = min2<BF16>(kmn, w);
        }
      }
      float fh[8], fl[8];
      unpack8<BF16>(kmx, fh);
      unpack8<BF16>(kmn, fl);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        xmax = fmaxf(xmax, fmaxf(fabsf(__fsub_rn(fh[i], mean[i])), fabsf(__fsub_rn(fl[i], mean[i]))));
    }
    const float m = block_max(xmax, red);
    const float inv = reciprocal(m, 127.0f);
    float* ks = a.k_scale + sc_base * a.wk + g;
    if (tid == 0 && g < a.wk && QNRE_ACCESS_OK(ks, 4, a.k_scale_ext)) *ks = __fdiv_rn(m, 127.0f);
    // the transposed V codes are complete (block_max's barriers): 16-byte stores
    for (int idx = tid; idx < a.D * 4; idx += 256) {
      const int c = idx >> 2, part = idx & 3;
      const uint32_t* row = vt + c * kVRowWords + part * 4;
      uint8_t* dst = a.v_out + (((static_cast<long long>(r) * a.B + b) * a.D + c) * a.H_l + hl) * a.S_pad + s0 +
                     part * 16;
      if (QNRE_ACCESS_OK(dst, 16, a.v_out_ext)) *reinterpret_cast<uint4*>(dst) = make_uint4(row[0], row[1], row[2], row[3]);
    }
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
      int8_t* kd = a.k_out + out0 + u * row_step;
      if (sr + u < a.S && QNRE_ACCESS_OK(kd, 8, a.k_out_ext)) {
        uint2 code = make_uint2(0, 0);  // rows at or past U are code 0
        if (u < n_live) {
          float f[8];
          unpack8<BF16>(slot(2, u), f);
          uint32_t t[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = int8_bits(__fsub_rn(f[i], mean[i]), inv);
          code = make_uint2(pack_low_bytes(t[0], t[1], t[2], t[3]), pack_low_bytes(t[4], t[5], t[6], t[7]));
        }
        *reinterpret_cast<uint2*>(kd) = code;
      }
    }
  }
}

// 48 KiB of dynamic shared memory needs the opt-in, once per device (the
// attribute is per device; setting it twice is harmless, so races are benign).
qnre_status_t quantize_opt_in() {
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> done[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QNRE_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_acquire)) return QNRE_OK;
  const cudaFuncAttribute attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  if (cudaFuncSetAttribute(quantize_kernel<4, true>, attr, quantize_smem_bytes<4>()) != cudaSuccess ||
      cudaFuncSetAttribute(quantize_kernel<4, false>, attr, quantize_smem_bytes<4>()) != cudaSuccess ||
      cudaFuncSetAttribute(quantize_kernel<2, true>, attr, quantize_smem_bytes<2>()) != cudaSuccess ||
      cudaFuncSetAttribute(quantize_kernel<2, false>, attr, quantize_smem_bytes<2>()) != cudaSuccess)
    return QNRE_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) done[dev].store(true, std::memory_order_release);
  return QNRE_OK;
}

struct Geometry {
  int P, B, L, H, H_l, D, S, S_pad, U, wq, wk, chunks;
  uint64_t ws_bytes;
};

qnre_status_t geometry(int P, int B, int L, int H, int D, int U, Geometry* g) {
  if (P < 1 || B < 1 || L < 1 || H < 1 || H % P != 0) return QNRE_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return QNRE_ERR_UNSUPPORTED;
  const int64_t S = static_cast<int64_t>(P) * L;
  // grid limits: H (x), L/256 and S/64 (y, <= 65535), P*B (z, <= 65535)
  if (S > int64_t{65535} * kKGroup || static_cast<int64_t>(P) * B > 65535 || H > 65535) return QNRE_ERR_CAPACITY;
  if (U < 1 || U > S) return QNRE_ERR_INVALID_ARG;
  g->P = P;
  g->B = B;
  g->L = L;
  g->H = H;
  g->H_l = H / P;
  g->D = D;
  g->S = static_cast<int>(S);
  g->S_pad = static_cast<int>((S + kVPad - 1) / kVPad * kVPad);
  g->U = U;
  g->wq = (U + kQGroup - 1) / kQGroup;
  g->wk = (U + kKGroup - 1) / kKGroup;
  g->chunks = (L + kChunk - 1) / kChunk;
  const uint64_t bhd = static_cast<uint64_t>(B) * H * D;
  g->ws_bytes = (2 * static_cast<uint64_t>(P) * g->chunks * bhd + 2 * bhd) * sizeof(float);
  return QNRE_OK;
}

}  // namespace

extern "C" {

qnre_status_t ulysses_sage2_workspace_bytes(int P, int B, int L, int H, int D, uint64_t* bytes) {
  if (bytes == nullptr) return QNRE_ERR_INVALID_ARG;
  Geometry g;
  const qnre_status_t st = geometry(P, B, L, H, D, 1, &g);
  if (st != QNRE_OK) return st;
  *bytes = g.ws_bytes;
  return QNRE_OK;
}

qnre_status_t ulysses_sage2_scatter_qkv(const qnre_tensor4_t* q, const qnre_tensor4_t* k, const qnre_tensor4_t* v,
                                        int P, int used_sequence, void* q_out, void* k_out, void* v_out,
                                        float* q_scale, float* k_scale, float* v_scale, void* workspace,
                                        uint64_t workspace_bytes, qnre_stream_t stream) {
  const qnre_tensor4_t* X[3] = {q, k, v};
  ByteRange in[3];
  for (int c = 0; c < 3; ++c) {
    const qnre_status_t st = check_view(X[c], &in[c]);
    if (st != QNRE_OK) return st;
    if (X[c]->dtype != QNRE_DTYPE_BF16 && X[c]->dtype != QNRE_DTYPE_FP16) return QNRE_ERR_UNSUPPORTED;
    if (X[c]->dtype != q->dtype) return QNRE_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
      if (X[c]->shape[i] != q->shape[i]) return QNRE_ERR_INVALID_ARG;
    // head rows: channel axis contiguous, rows 16-byte aligned
    if (X[c]->stride[3] != 1 || !aligned(X[c]->data, 16)) return QNRE_ERR_ALIGNMENT;
    for (int i = 0; i < 3; ++i)
      if ((X[c]->stride[i] * 2) % 16 != 0) return QNRE_ERR_ALIGNMENT;
  }
  if (P < 1 || q->shape[0] % P != 0) return QNRE_ERR_INVALID_ARG;
  if (q->shape[0] == 0 || q->shape[1] == 0) return QNRE_ERR_INVALID_ARG;
  if (q->shape[0] > 65535 || q->shape[1] > (int64_t{1} << 30) || q->shape[2] > 65535) return QNRE_ERR_CAPACITY;
  Geometry g;
  qnre_status_t st = geometry(P, static_cast<int>(q->shape[0] / P), static_cast<int>(q->shape[1]),
                              static_cast<int>(q->shape[2]), static_cast<int>(q->shape[3]), used_sequence, &g);
  if (st != QNRE_OK) return st;
  if (!q_out || !k_out || !v_out || !q_scale || !k_scale || !v_scale || !workspace) return QNRE_ERR_INVALID_ARG;
  if (workspace_bytes < g.ws_bytes) return QNRE_ERR_CAPACITY;
  if (!aligned(q_out, 16) || !aligned(k_out, 16) || !aligned(v_out, 16) || !aligned(q_scale, 4) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(workspace, 16))
    return QNRE_ERR_ALIGNMENT;
  const uint64_t n_qk = static_cast<uint64_t>(P) * g.B * g.S * g.H_l * g.D;
  const ByteRange outs[7] = {span(q_out, n_qk), span(k_out, n_qk),
                             span(v_out, static_cast<uint64_t>(P) * g.B * g.D * g.H_l * g.S_pad),
                             span(q_scale, static_cast<uint64_t>(P) * g.B * g.H_l * g.wq * 4),
                             span(k_scale, static_cast<uint64_t>(P) * g.B * g.H_l * g.wk * 4),
                             span(v_scale, static_cast<uint64_t>(P) * g.B * g.H_l * g.D * 4),
                             span(workspace, g.ws_bytes)};
  for (int i = 0; i < 7; ++i) {
    for (int c = 0; c < 3; ++c)
      if (overlaps(outs[i], in[c])) return QNRE_ERR_ALIAS;
    for (int j = i + 1; j < 7; ++j)
      if (overlaps(outs[i], outs[j])) return QNRE_ERR_ALIAS;
  }
  st = quantize_opt_in();
  if (st != QNRE_OK) return st;

  auto view = [](const qnre_tensor4_t* t) {
    View w;
    w.data = static_cast<const char*>(t->data);
    w.sz = t->stride[0] * 2;
    w.ss = t->stride[1] * 2;
    w.sh = t->stride[2] * 2;
    return w;
  };
  const bool bf16 = q->dtype == QNRE_DTYPE_BF16;
  float* ws = static_cast<float*>(workspace);
  const uint64_t partial = static_cast<uint64_t>(P) * g.chunks * g.B * g.H * g.D;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  StatsArgs sa;
  sa.k = view(k);
  sa.v = view(v);
  sa.ksum = ws;
  sa.vmax = ws + partial;
  sa.P = P;
  sa.B = g.B;
  sa.L = g.L;
  sa.H = g.H;
  sa.D = g.D;
  sa.chunks = g.chunks;
  sa.U = g.U;
#if QNRE_DEBUG_BOUNDS
  sa.k_ext = Extent{in[1].lo, in[1].hi};
  sa.v_ext = Extent{in[2].lo, in[2].hi};
  sa.ws_ext = Extent{outs[6].lo, outs[6].hi};
#endif
  const int heads_per_cta = 256 / (g.D / 8);
  const dim3 sgrid((g.H + heads_per_cta - 1) / heads_per_cta, g.chunks, P * g.B);
  if ((bf16 ? launch_pdl(stats_partial_kernel<true>, sgrid, dim3(256), 0, s, sa)
            : launch_pdl(stats_partial_kernel<false>, sgrid, dim3(256), 0, s, sa)) != cudaSuccess)
    return QNRE_ERR_CUDA;

  FinalArgs fa;
  fa.ksum = sa.ksum;
  fa.vmax = sa.vmax;
  fa.kmean = ws + 2 * partial;
  fa.vinv = fa.kmean + static_cast<uint64_t>(g.B) * g.H * g.D;
  fa.v_scale = v_scale;
  fa.P = P;
  fa.B = g.B;
  fa.H = g.H;
  fa.H_l = g.H_l;
  fa.D = g.D;
  fa.chunks = g.chunks;
  fa.U = g.U;
#if QNRE_DEBUG_BOUNDS
  fa.ws_ext = Extent{outs[6].lo, outs[6].hi};
  fa.v_scale_ext = Extent{outs[5].lo, outs[5].hi};
#endif
  if (launch_pdl(stats_final_kernel, dim3(g.H, g.B, g.D / 32), dim3(32 * kFinalWarps), 0, s, fa) != cudaSuccess)
    return QNRE_ERR_CUDA;

  QuantArgs qa;
  qa.q = view(q);
  qa.k = view(k);
  qa.v = view(v);
  qa.kmean = fa.kmean;
  qa.vinv = fa.vinv;
  qa.q_out = static_cast<int8_t*>(q_out);
  qa.k_out = static_cast<int8_t*>(k_out);
  qa.v_out = static_cast<uint8_t*>(v_out);
  qa.q_scale = q_scale;
  qa.k_scale = k_scale;
  qa.P = P;
  qa.B = g.B;
  qa.L = g.L;
  qa.H = g.H;
  qa.H_l = g.H_l;
  qa.D = g.D;
  qa.S = g.S;
  qa.S_pad = g.S_pad;
  qa.U = g.U;
  qa.wq = g.wq;
  qa.wk = g.wk;
#if QNRE_DEBUG_BOUNDS
  qa.src_ext[0] = Extent{in[2].lo, in[2].hi};
  qa.src_ext[1] = Extent{in[0].lo, in[0].hi};
  qa.src_ext[2] = Extent{in[1].lo, in[1].hi};
  qa.q_out_ext = qnre::output_extent(outs[0].lo, outs[0].hi);
  qa.k_out_ext = qnre::output_extent(outs[1].lo, outs[1].hi);
  qa.v_out_ext = qnre::output_extent(outs[2].lo, outs[2].hi);
  qa.q_scale_ext = Extent{outs[3].lo, outs[3].hi};
  qa.k_scale_ext = Extent{outs[4].lo, outs[4].hi};
#endif
  const dim3 qgrid(g.H, g.S_pad / kKGroup, g.B);
  cudaError_t e;
  if (g.D == 128 && bf16) e = launch_pdl(quantize_kernel<4, true>, qgrid, dim3(256), quantize_smem_bytes<4>(), s, qa);
  else if (g.D == 128) e = launch_pdl(quantize_kernel<4, false>, qgrid, dim3(256), quantize_smem_bytes<4>(), s, qa);
  else if (bf16) e = launch_pdl(quantize_kernel<2, true>, qgrid, dim3(256), quantize_smem_bytes<2>(), s, qa);
  else e = launch_pdl(quantize_kernel<2, false>, qgrid, dim3(256), quantize_smem_bytes<2>(), s, qa);
  return from_cuda(e);
}

}  // extern "C"

namespace qnre {

cudaError_t sage2_bounds_violations(unsigned long long* count, bool reset) {
#if QNRE_DEBUG_BOUNDS
  return read_bounds_violations(count, reset);
#else
  *count = 0;
  (void)reset;
  return cudaErrorNotSupported;
#endif
}

}  // namespace qnre
