// fused_qkv.cu -- fused QKV projection + per-head RMSNorm + RoPE + head-band
// scatter on the sm_103a tensor cores.
//
// What it computes ("Fused QKV Projection + Norm + RoPE + Head Exchange",
// flashinfer.comm API reference; operator math from "QKV projection + RMSNorm +
// RoPE overlapped with the Ulysses head exchange", Assumptions):
//   Y = x W, bf16 x bf16 -> fp32; W's columns grouped Q | K | V, head-major;
//   q/k heads: RMSNorm over the 128-wide head (eps 1e-6, shared [128] weight),
//   then RoPE from the token's fp32 cos/sin row; v heads unchanged;
//   bf16 result of head h of token (r_s, b, s) goes to virtual rank h / H_local,
//   local head h % H_local, global row r_s * S + s.
//
// How (this kernel's design, not the pages'):
//   * persistent grid of CTA pairs, one CTA per SM; a pair owns a 256-token x
//     256-column tile (= 2 heads), tiles walked in a grouped raster so
//     concurrent pairs share x and W panels in L2;
//   * kPC = 1: clusters of one pair.  kPC = 2: clusters of two pairs on
//     adjacent row tiles of the same column tile, which need the same W
//     blocks: pair q loads W block q of each CTA's half once, by TMA multicast
//     into the matching CTA of both pairs, and a stage is released only when
//     both pairs' MMAs have committed it;
//   * warp 0 of each CTA: one thread issues TMA loads of its 128 x-rows
//     (K-major) and its W columns (N-major) into a 5-stage ring (128-byte
//     swizzle); a pair's loads complete on its leader CTA's stage barrier;
//   * warp 1 of the leader: one thread issues tcgen05.mma.cta_group::2 (M=256,
//     N=256, K=16, bf16 in, fp32 accumulate in each CTA's tensor memory),
//     double-buffering the accumulator so the epilogue of tile i overlaps the
//     main loop of tile i+1; commits are multicast to both CTAs;
//   * warps 2-5 of each CTA: epilogue; thread i owns TMEM lane i = token row i
//     of that CTA's half and reads a head's 128 accumulator columns once into
//     registers, so they are thread-local: the RMS sum,
//     the scale and both RoPE pairings need no cross-thread traffic; the bf16
//     rows go into an 8 KiB per-warp staging buffer (two 32 x 128-byte halves,
//     128-byte swizzle), and when the warp's 32 tokens lie in one (rank, batch)
//     segment one lane writes them into the head's band with two TMA tensor
//     stores (box 64 columns x 32 consecutive band rows); otherwise (a segment
//     edge, the ragged end, the publishing form, the debug build) each store
//     instruction writes two whole 256-byte head rows; then both CTAs release
//     the accumulator on the leader.
//   * every mbarrier wait has a time limit; on expiry the kernel raises a
//     status bit, tells the peer CTA to stop, drains its own in-flight copies
//     and MMAs, frees its tensor memory and returns.
#include "fused_qkv.cuh"
#include "ptx.cuh"
#include "../../include/qnre.h"

#include <cuda_bf16.h>

namespace qnre {
namespace {

constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s per wait
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kPairM, kBN, /*b_mn_major=*/true);
constexpr uint32_t kIdescHalf = ptx::idesc_bf16_f32(kPairM, kBNHalf, /*b_mn_major=*/true);
constexpr uint64_t kDrainGraceNs = 50ull * 1000ull;  // in-flight TMA settles in microseconds

struct SmemLayout {
  uint32_t a;      // kStages x kABytes
  uint32_t b;      // kStages x kBBytes
  uint32_t full;   // kStages mbarriers: TMA -> MMA (the leader's count both CTAs' bytes)
  uint32_t empty;  // kStages mbarriers: MMA -> TMA (both CTAs, multicast commit)
  uint32_t tfull;  // 2 mbarriers: MMA -> epilogue (both CTAs, multicast commit)
  uint32_t tempty; // 2 mbarriers: epilogues of both CTAs -> MMA (leader)
  uint32_t drain;  // 1 mbarrier: MMA completion on abort (leader)
  uint32_t abort;  // abort word (shared address)
  uint32_t rank;   // 0 = pair leader, 1 = peer
  uint32_t crank;  // rank in the cluster (pair q = crank / 2)
  uint32_t leader; // cluster rank of this CTA's pair leader
  uint32_t ncta;   // CTAs in the cluster (2 or 4)
};

__device__ __forceinline__ void raise_abort(const SmemLayout& L, volatile uint32_t* abort_flag, unsigned* status) {
  *abort_flag = 1u;
  for (uint32_t r = 0; r < L.ncta; ++r)
    if (r != L.crank) ptx::st_shared_cluster_u32(ptx::mapa_shared(L.abort, r), 1u);
  atomicOr(status, QNRE_DEVICE_WAIT_TIMEOUT);
}

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, const SmemLayout& L,
                                             volatile uint32_t* abort_flag, unsigned* status,
                                             bool honour_abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (ptx::global_timer_ns() - t0 > kWaitLimitNs) {
        if (honour_abort) raise_abort(L, abort_flag, status);
        return false;
      }
    }
  }
}

#ifndef QNRE_X_POLICY
#define QNRE_X_POLICY 0  // L2 priority of the x loads: 0 evict_last, 1 evict_normal, 2 evict_first
#endif
#ifndef QNRE_W_POLICY
#define QNRE_W_POLICY 0  // the same for the W loads
#endif
__device__ __forceinline__ uint64_t l2_policy(int kind) {
  return kind == 0 ? ptx::l2_policy_evict_last() : (kind == 1 ? ptx::l2_policy_evict_normal() : ptx::l2_policy_evict_first());
}

__device__ __forceinline__ void grace_spin(uint64_t ns) {
  const uint64_t t0 = ptx::global_timer_ns();
  while (ptx::global_timer_ns() - t0 < ns) {
  }
}

// Raster position -> (row unit, column tile); a row unit is one 256-row tile,
// or two adjacent ones when two pairs share a cluster.
__device__ __forceinline__ void tile_coords(int tile, const FusedArgs& a, int num_m, int& m_blk, int& n_blk) {
  const int per_group = a.group_m * a.num_n_tiles;
  const int group = tile / per_group;
  const int first_m = group * a.group_m;
  const int gm = min(a.group_m, num_m - first_m);
  const int within = tile - group * per_group;
  m_blk = first_m + within % gm;
  n_blk = within / gm;
}

// One work item: rows [m_blk*256, +256), columns [col0, col0 + width).
struct Work {
  int m_blk;
  int col0;
  int width;  // kBN or kBNHalf
};

template <int kPC>
__device__ __forceinline__ Work work_coords(int w, const FusedArgs& a, uint32_t pair_in_cluster) {
  int m_blk, n_blk;
  if (kPC == 2) {  // work item = (row-tile pair, column tile); pair q takes row tile 2 * unit + q
    const int q = static_cast<int>(pair_in_cluster);
    if (w < a.num_full) {
      tile_coords(w, a, a.num_mp_tiles, m_blk, n_blk);
      return {2 * m_blk + q, n_blk * kBN, kBN};
    }
    const int j = w - a.num_full;
    tile_coords(a.num_full + (j >> 1), a, a.num_mp_tiles, m_blk, n_blk);
    return {2 * m_blk + q, n_blk * kBN + (j & 1) * kBNHalf, kBNHalf};
  }
  if (w < a.num_full) {
    tile_coords(w, a, a.num_m_tiles, m_blk, n_blk);
    return {m_blk, n_blk * kBN, kBN};
  }
  const int j = w - a.num_full;
  tile_coords(a.num_full + (j >> 1), a, a.num_m_tiles, m_blk, n_blk);
  return {m_blk, n_blk * kBN + (j & 1) * kBNHalf, kBNHalf};
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Compiler-level barrier: the registers count as rewritten here, so no use of
// them is scheduled above the preceding tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

__device__ __forceinline__ void rotate(float& a, float& b, float c, float s) {
  const float na = a * c - b * s;
  const float nb = b * c + a * s;
  a = na;
  b = nb;
}

// --------------------------------------------------------------------------
// Producer (both CTAs): TMA loads of this CTA's x rows and W columns.
// --------------------------------------------------------------------------
template <int kPC>
__device__ void run_producer(const FusedArgs& a, const SmemLayout& L, volatile uint32_t* abort_flag) {
  uint32_t g = 0;
  uint32_t used_mask = 0, parity_mask = 0;  // per stage: ever loaded / parity of its last load
  const uint64_t pol_x = l2_policy(QNRE_X_POLICY);
  const uint64_t pol_w = l2_policy(QNRE_W_POLICY);
  const uint32_t full_leader = ptx::mapa_shared(L.full, L.leader);
  const uint32_t q = L.crank >> 1;  // pair in the cluster
  const int unit = blockIdx.x / (2 * kPC);
  const int num_units = gridDim.x / (2 * kPC);
  bool ok = true;
  for (int w = unit; ok && w < a.num_work; w += num_units) {
    const Work t = work_coords<kPC>(w, a, q);
    const int row0 = t.m_blk * kPairM + static_cast<int>(L.rank) * kBM;
    const int bcols = t.width / 2;  // this CTA's share of the tile's columns
    const int col0 = t.col0 + static_cast<int>(L.rank) * bcols;
    const uint32_t tx = 2u * static_cast<uint32_t>(kABytes + bcols * kBK * 2);
    for (int kb = 0; kb < a.num_k_blocks; ++kb, ++g) {
      const uint32_t s = g % kStages;
      const uint32_t ph = (g / kStages) & 1u;
      if (!bounded_wait(L.empty + 8 * s, ph ^ 1u, L, abort_flag, a.status, true)) {
        ok = false;
        break;
      }
      if (L.rank == 0) ptx::mbar_arrive_expect_tx(L.full + 8 * s, tx);
      const uint32_t bar = full_leader + 8 * s;
      ptx::tma_load_2d_pair(L.a + s * kABytes, &a.tmap_x, bar, kb * kBK, row0, pol_x);
      if (kPC == 2) {
        // both pairs need this CTA's share of the W tile: pair q loads 64-column
        // block q of it once, into this CTA and its counterpart in the other pair
        // (a half tile has one block per CTA, loaded by pair 0)
        const uint16_t mask = static_cast<uint16_t>((1u << L.rank) | (1u << (L.rank + 2)));
        if (static_cast<int>(q) < bcols / 64)
          ptx::tma_load_2d_pair_multicast(L.b + s * kBBytes + q * (64 * kBK * 2), &a.tmap_w, bar,
                                          col0 + static_cast<int>(q) * 64, kb * kBK, mask, pol_w);
      } else {
        for (int j = 0; j < bcols / 64; ++j) {
          ptx::tma_load_2d_pair(L.b + s * kBBytes + j * (64 * kBK * 2), &a.tmap_w, bar, col0 + j * 64, kb * kBK,
                                pol_w);
        }
      }
      used_mask |= 1u << s;
      parity_mask = (parity_mask & ~(1u << s)) | (ph << s);
    }
  }
  if (!ok) {
    // Abort: let every load already issued land before the CTA can exit.  The
    // leader's stage barriers count both CTAs' bytes; the peer cannot observe
    // its own loads, so both also wait a short grace period.
    if (L.rank == 0) {
      for (uint32_t s = 0; s < kStages; ++s) {
        if (used_mask & (1u << s)) {
          bounded_wait(L.full + 8 * s, (parity_mask >> s) & 1u, L, abort_flag, a.status, false);
        }
      }
    }
    grace_spin(kDrainGraceNs);
  }
}

// --------------------------------------------------------------------------
// MMA issuer (leader CTA only): tcgen05.mma over the stage ring into the TMEM
// accumulators of both CTAs.
// --------------------------------------------------------------------------
template <int kPC>
__device__ void run_mma(const FusedArgs& a, const SmemLayout& L, uint32_t tmem_base,
                        volatile uint32_t* abort_flag) {
  uint32_t g = 0;
  uint32_t it = 0;
  bool ok = true;
  const int unit = blockIdx.x / (2 * kPC);
  const int num_units = gridDim.x / (2 * kPC);
  // a stage is free once every pair that reads it has consumed it: with two
  // pairs the W blocks were multicast into all four CTAs
  const uint16_t empty_mask = kPC == 2 ? 0xF : 0x3;
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (2 * (L.crank >> 1)));
  for (int w = unit; ok && w < a.num_work; w += num_units, ++it) {
    const uint32_t acc = it & 1u;
    const uint32_t aph = (it >> 1) & 1u;
    const uint32_t idesc = w < a.num_full ? kIdesc : kIdescHalf;
    if (!bounded_wait(L.tempty + 8 * acc, aph ^ 1u, L, abort_flag, a.status, true)) {
      ok = false;
      break;
    }
    ptx::tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + acc * kAccCols;
    for (int kb = 0; kb < a.num_k_blocks; ++kb, ++g) {
      const uint32_t s = g % kStages;
      const uint32_t ph = (g / kStages) & 1u;
      if (!bounded_wait(L.full + 8 * s, ph, L, abort_flag, a.status, true)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      const uint32_t a_base = L.a + s * kABytes;
      const uint32_t b_base = L.b + s * kBBytes;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        // A: K-major, rows of 128 B (64 bf16), 8-row groups 1024 B apart;
        //    the k-th 16-wide slice starts 32 B into the swizzled row.
        const uint64_t adesc = ptx::smem_desc_sw128(a_base + kk * 32, 16, 1024);
        // B: N-major, 64-column blocks of kBK rows x 128 B (LBO = 8 KiB apart),
        //    8-row k groups 1024 B apart; the k-th 16-row slice starts 2 KiB in.
        const uint64_t bdesc = ptx::smem_desc_sw128(b_base + kk * 2048, 64 * kBK * 2, 1024);
        ptx::umma_f16_pair(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
      }
      ptx::umma_commit_pair_multicast(L.empty + 8 * s, empty_mask);  // frees the stage
    }
    if (!ok) break;
    ptx::umma_commit_pair_multicast(L.tfull + 8 * acc, pair_mask);  // accumulators ready in both CTAs
  }
  if (!ok) {
    ptx::umma_commit_pair(L.drain);
    bounded_wait(L.drain, 0, L, abort_flag, a.status, false);
  }
}

// --------------------------------------------------------------------------
// Epilogue: TMEM -> registers -> norm / RoPE -> bf16 -> band destination.
// --------------------------------------------------------------------------
template <int kPC>
__device__ void run_epilogue(const FusedArgs& a, const SmemLayout& L, uint32_t tmem_base,
                             const float* norm_w, uint4* epi_stage, volatile uint32_t* abort_flag) {
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int sub = warp & 3;  // TMEM lane quarter this warp may access
  const int row = sub * 32 + lane;
  const int S_g = a.P * a.S;
  const int three_h = 3 * a.H;
  const uint32_t tempty_leader = ptx::mapa_shared(L.tempty, L.leader);
  // This warp's staging: two 32 x 128-byte halves (columns 0-63, 64-127) in the
  // 128-byte swizzle layout: 16-byte chunk c of row i sits at chunk (c ^ (i & 7))
  // of that row, so neither the row-wise writes below nor the reads of either
  // store path collide in a bank, and a TMA store can read each half directly.
  uint4* stage = epi_stage + (warp - 2) * (kEpiWarpBytes / 16);
  const uint32_t stage_saddr = ptx::smem_addr(stage);
  bool store_pending = false;  // lane 0: a TMA store may still be reading the staging
  const int unit = blockIdx.x / (2 * kPC);
  const int num_units = gridDim.x / (2 * kPC);
  uint32_t it = 0;
  for (int w = unit; w < a.num_work; w += num_units, ++it) {
    const uint32_t acc = it & 1u;
    const uint32_t aph = (it >> 1) & 1u;
    if (!bounded_wait(L.tfull + 8 * acc, aph, L, abort_flag, a.status, true)) break;
    ptx::tc_fence_after_sync();

    const Work tw = work_coords<kPC>(w, a, L.crank >> 1);
    if (kPC == 2 && tw.m_blk >= a.num_m_tiles) {
      // the second pair's row tile past an odd tile count: its accumulator holds
      // the product of zero rows; nothing is stored or published
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(tempty_leader + 8 * acc);
      continue;
    }
    const int t = tw.m_blk * kPairM + static_cast<int>(L.rank) * kBM + row;
    const bool valid = t < a.T;
    const int s_loc = valid ? t % a.S : 0;
    const int tb = valid ? t / a.S : 0;
    const int b = tb % a.B;
    const int r_s = tb / a.B;
    long long pos = 0;
    bool bad_pos = false;
    if (valid && a.epilogue_on) {
      pos = a.positions != nullptr ? static_cast<long long>(a.positions[t]) : static_cast<long long>(t);
      bad_pos = pos < 0 || pos >= a.n_pos;
    }
    const long long dest_row = static_cast<long long>(r_s) * a.S + s_loc;  // global row in batch b
    // The warp's 32 tokens t - lane .. t - lane + 31 go to 32 consecutive rows of
    // every head band when they are all valid and lie in one (rank, batch)
    // segment: then one TMA store box covers them (lane 0's token is the first).
    const int t_first = t - lane;
    const bool tma_rows = !QNRE_DEBUG_BOUNDS && a.tma_store && a.ready == nullptr &&
                          t_first + (kStoreRows - 1) < a.T && (t_first % a.S) + (kStoreRows - 1) < a.S;

#pragma unroll 1
    for (int hh = 0; hh < tw.width / 128; ++hh) {
      const int ch = tw.col0 / 128 + hh;  // head column index in [0, 3H)
      if (ch >= three_h) break;
      const int g = ch / a.H;
      const int h = ch - g * a.H;
      const int r = h / a.H_local;
      const int hl = h - r * a.H_local;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + acc * kAccCols + hh * 128;
      uint16_t* dst;
      if (a.layout == 0) {
        uint16_t* base = g == 0 ? a.out_q : (g == 1 ? a.out_k : a.out_v);
        dst = base + ((((static_cast<long long>(r) * a.B + b) * S_g + dest_row) * a.H_local + hl) * 128);
      } else {
        dst = a.out_fused +
              ((((static_cast<long long>(r) * a.B + b) * S_g + dest_row) * a.H_local + hl) * 384 + g * 128);
      }
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      const bool normed = g < 2 && a.epilogue_on;
#if QNRE_DEBUG_BOUNDS
      // debug build: a head row outside its output tensor is reported and not stored
      bool row_ok = valid;
      if (valid) {
        const long long off = dst - (a.layout == 0 ? (g == 0 ? a.out_q : (g == 1 ? a.out_k : a.out_v)) : a.out_fused);
        if (off < 0 || off + 128 > a.out_elems) {
          atomicOr(a.status, QNRE_DEVICE_BOUNDS);
          row_ok = false;
        }
      }
#else
      const bool row_ok = valid;
#endif

      // One read of the head's 128 accumulator columns: v[j] holds columns
      // [32j, 32j + 32) of this thread's token.
      uint32_t v[4][32];
      ptx::tmem_ld_32x32b_x32(taddr, v[0]);
      ptx::tmem_ld_32x32b_x32(taddr + 32, v[1]);
      ptx::tmem_ld_32x32b_x32(taddr + 64, v[2]);
      ptx::tmem_ld_32x32b_x32(taddr + 96, v[3]);
      ptx::tmem_ld_wait();
      reg_fence(v[0]);
      reg_fence(v[1]);
      reg_fence(v[2]);
      reg_fence(v[3]);
      // q, k: mean square of the head row (columns 0-31 with 32-63, then 64-95
      // with 96-127, one pair of squares at a time).
      float scale = 1.0f;
      if (normed) {
        float ss = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float x0 = __uint_as_float(v[2 * half][i]);
            const float x1 = __uint_as_float(v[2 * half + 1][i]);
            ss = fmaf(x0, x0, ss);
            ss = fmaf(x1, x1, ss);
          }
        }
        scale = rsqrtf(ss * (1.0f / 128.0f) + 1e-6f);
      }
      const float* wn = norm_w + (g < 2 ? g : 0) * 128;
      const float4* cs = reinterpret_cast<const float4*>(a.cos_sin + pos * 128);
      const bool nan_out = normed && bad_pos;
      const bool rope = normed && !bad_pos;

      // Scale, rotate, round and stage 64 columns per step: rotate-half pairs
      // column i with i + 64, so step p takes columns [32p, 32p + 32) and
      // [64 + 32p, 96 + 32p) (v[p], v[2 + p]); interleaved pairs are adjacent, so
      // step p takes [64p, 64p + 64) (v[2p], v[2p + 1]).  The call sites below
      // fix which register blocks (vl, vh) a step pairs, so no register is
      // selected at run time.
      auto step = [&](const uint32_t(&vl)[32], const uint32_t(&vh)[32], const int p, const bool rh) {
        const int c_lo = rh ? 32 * p : 64 * p;
        const int c_hi = rh ? 64 + 32 * p : 64 * p + 32;
        float lo[32], hi[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          lo[i] = __uint_as_float(vl[i]);
          hi[i] = __uint_as_float(vh[i]);
        }
        if (normed) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            lo[i] = (lo[i] * scale) * wn[c_lo + i];
            hi[i] = (hi[i] * scale) * wn[c_hi + i];
          }
        }
        if (rope) {
          if (rh) {
            // pair (c_lo + i, c_hi + i) uses angle index 32p + i
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 c = __ldg(cs + 8 * p + i4);
              const float4 sn = __ldg(cs + 16 + 8 * p + i4);
              rotate(lo[4 * i4 + 0], hi[4 * i4 + 0], c.x, sn.x);
              rotate(lo[4 * i4 + 1], hi[4 * i4 + 1], c.y, sn.y);
              rotate(lo[4 * i4 + 2], hi[4 * i4 + 2], c.z, sn.z);
              rotate(lo[4 * i4 + 3], hi[4 * i4 + 3], c.w, sn.w);
            }
          } else {
            // pairs (2i, 2i+1) over columns [64p, 64p + 64): angle index 32p + i
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 c = __ldg(cs + 8 * p + i4);
              const float4 sn = __ldg(cs + 16 + 8 * p + i4);
              float* pv = i4 < 4 ? lo : hi;
              const int o = (i4 & 3) * 8;
              rotate(pv[o + 0], pv[o + 1], c.x, sn.x);
              rotate(pv[o + 2], pv[o + 3], c.y, sn.y);
              rotate(pv[o + 4], pv[o + 5], c.z, sn.z);
              rotate(pv[o + 6], pv[o + 7], c.w, sn.w);
            }
          }
        }
        if (nan_out) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            lo[i] = __uint_as_float(0x7FC00000u);
            hi[i] = __uint_as_float(0x7FC00000u);
          }
        }
        // The previous head's TMA store must have read the staging before it
        // is rewritten.
        if (p == 0 && store_pending) {
          ptx::bulk_wait_group_read_all();
          store_pending = false;
        }
        __syncwarp();
        // Stage the bf16 row in this warp's buffer: row `lane`, 16-byte chunk c
        // (8 columns) in half c / 8 at swizzled chunk (c % 8) ^ (lane % 8).
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 u;
          u.x = pack_bf16x2(lo[8 * j + 0], lo[8 * j + 1]);
          u.y = pack_bf16x2(lo[8 * j + 2], lo[8 * j + 3]);
          u.z = pack_bf16x2(lo[8 * j + 4], lo[8 * j + 5]);
          u.w = pack_bf16x2(lo[8 * j + 6], lo[8 * j + 7]);
          const int cl = c_lo / 8 + j;
          stage[(cl >> 3) * (kEpiHalfBytes / 16) + lane * 8 + ((cl & 7) ^ (lane & 7))] = u;
          uint4 w;
          w.x = pack_bf16x2(hi[8 * j + 0], hi[8 * j + 1]);
          w.y = pack_bf16x2(hi[8 * j + 2], hi[8 * j + 3]);
          w.z = pack_bf16x2(hi[8 * j + 4], hi[8 * j + 5]);
          w.w = pack_bf16x2(hi[8 * j + 6], hi[8 * j + 7]);
          const int ch2 = c_hi / 8 + j;
          stage[(ch2 >> 3) * (kEpiHalfBytes / 16) + lane * 8 + ((ch2 & 7) ^ (lane & 7))] = w;
        }
      };
      if (a.rope_style == 0) {
        step(v[0], v[2], 0, true);
        step(v[1], v[3], 1, true);
      } else {
        step(v[0], v[1], 0, false);
        step(v[2], v[3], 1, false);
      }
      if (tma_rows) {
        // Two TMA stores (columns 0-63 and 64-127) write the warp's 32 rows of
        // this head into its band: box 64 x 1 x 32 at (column, local head,
        // flattened (rank, batch, global row)).  The staging writes are made
        // visible to the async proxy first.
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const CUtensorMap* map = &a.tmap_out[a.layout == 0 ? g : 0];
          const int col = a.layout == 0 ? 0 : g * 128;
          const int grow = static_cast<int>((static_cast<long long>(r) * a.B + b) * S_g + dest_row);
          ptx::tma_store_3d(map, stage_saddr, col, hl, grow);
          ptx::tma_store_3d(map, stage_saddr + kEpiHalfBytes, col + 64, hl, grow);
          ptx::bulk_commit_group();
          store_pending = true;
        }
      } else {
        // Write the warp's 32 head rows back two rows per instruction: lanes
        // 0-15 cover row 2i and lanes 16-31 row 2i+1, 256 contiguous bytes each.
        __syncwarp();
        const int half = lane >> 4;
        const int chunk = lane & 15;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          const int src_row = 2 * i + half;
          uint4* rd = reinterpret_cast<uint4*>(__shfl_sync(0xffffffffu, reinterpret_cast<long long>(d4), src_row));
          const int rv = __shfl_sync(0xffffffffu, row_ok ? 1 : 0, src_row);
          const uint4 u =
              stage[(chunk >> 3) * (kEpiHalfBytes / 16) + src_row * 8 + ((chunk & 7) ^ (src_row & 7))];
          if (rv) rd[chunk] = u;
        }
      }
      __syncwarp();
      if (a.ready != nullptr) {
        // This warp's 32 rows of the head are stored: publish them to rank r
        // (release at GPU scope orders every lane's stores before the count).
        __syncwarp();
        if (lane == 0) ptx::red_add_release_gpu(a.ready + r, 1u);
      }
    }
    if (bad_pos && valid) atomicOr(a.status, QNRE_DEVICE_BAD_POSITION);

    // Hand the accumulator back to the leader's MMA thread.
    ptx::tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster(tempty_leader + 8 * acc);
  }
  // Every TMA store has completed before the CTA (and its shared memory) ends.
  if (lane == 0 && store_pending) ptx::bulk_wait_group_all();
  __syncwarp();
}

template <int kPC>
__global__ void __launch_bounds__(kThreads, 1) fused_qkv_kernel(const __grid_constant__ FusedArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;

  SmemLayout L;
  L.a = raw + pad;
  L.b = L.a + kStages * kABytes;
  const uint32_t bar0 = L.b + kStages * kBBytes + kEpiStageBytes;
  L.full = bar0;
  L.empty = L.full + 8 * kStages;
  L.tfull = L.empty + 8 * kStages;
  L.tempty = L.tfull + 16;
  L.drain = L.tempty + 16;
  uint4* epi_stage = reinterpret_cast<uint4*>(smem + kStages * kStageBytes);  // 1024-byte aligned
  uint8_t* bar_ptr = smem + kStages * kStageBytes + kEpiStageBytes;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * kStages + 5));
  volatile uint32_t* abort_flag = tmem_holder + 1;
  L.abort = ptx::smem_addr(tmem_holder + 1);
  L.crank = ptx::cluster_ctarank();
  L.rank = L.crank & 1u;
  L.leader = L.crank & ~1u;
  L.ncta = 2u * kPC;
  float* norm_w = reinterpret_cast<float*>(bar_ptr + kBarBytes);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    ptx::prefetch_tensormap(&args.tmap_x);
    ptx::prefetch_tensormap(&args.tmap_w);
    if (args.tma_store) {
      for (int i = 0; i < (args.layout == 0 ? 3 : 1); ++i) ptx::prefetch_tensormap(&args.tmap_out[i]);
    }
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(L.full + 8 * s, 1);   // the leader's expect_tx arrival
      ptx::mbar_init(L.empty + 8 * s, kPC);  // one multicast commit from each pair that reads the stage
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(L.tfull + 8 * i, 1);   // one multicast commit
      ptx::mbar_init(L.tempty + 8 * i, 8);  // four epilogue warps in each CTA
    }
    ptx::mbar_init(L.drain, 1);
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(tmem_holder), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  if (threadIdx.x >= 64) {
    const int d = threadIdx.x - 64;  // 0..127
    norm_w[d] = bf16_bits_to_float(args.q_norm_w[d]);
    norm_w[128 + d] = bf16_bits_to_float(args.k_norm_w[d]);
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers initialised before any remote use
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) run_producer<kPC>(args, L, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && L.rank == 0) run_mma<kPC>(args, L, tmem_base, abort_flag);
    __syncwarp();
  } else {
    run_epilogue<kPC>(args, L, tmem_base, norm_w, epi_stage, abort_flag);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while its peer may still signal it or use its memory
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

namespace {

template <int kPC>
cudaLaunchConfig_t fused_config(int units, cudaLaunchAttribute* attr, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * kPC * units);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * kPC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int kPC>
cudaError_t max_clusters(int sms, int* clusters) {
  cudaError_t e = cudaFuncSetAttribute(fused_qkv_kernel<kPC>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = fused_config<kPC>(sms / (2 * kPC), attr, nullptr);
  return cudaOccupancyMaxActiveClusters(clusters, fused_qkv_kernel<kPC>, &cfg);
}

}  // namespace

cudaError_t prepare_fused_qkv_kernel(int* max_pairs, int* max_quads) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  int pairs = 0, quads = 0;
  if ((e = max_clusters<1>(sms, &pairs)) != cudaSuccess) return e;
  if (pairs < 1) return cudaErrorInvalidConfiguration;
  if (max_clusters<2>(sms, &quads) != cudaSuccess) {
    cudaGetLastError();  // four-CTA clusters unavailable: the one-pair kernel still serves
    quads = 0;
  }
  *max_pairs = pairs;
  *max_quads = quads;
  return cudaSuccess;
}

cudaError_t launch_fused_qkv(const FusedArgs& args, int units, int pairs_per_cluster, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  if (pairs_per_cluster == 2) {
    const cudaLaunchConfig_t cfg = fused_config<2>(units, attr, stream);
    return cudaLaunchKernelEx(&cfg, fused_qkv_kernel<2>, args);
  }
  const cudaLaunchConfig_t cfg = fused_config<1>(units, attr, stream);
  return cudaLaunchKernelEx(&cfg, fused_qkv_kernel<1>, args);
}

}  // namespace qnre

namespace qnre {
namespace {

// One CTA; thread r watches destination rank r's readiness count.  The wait is
// bounded by the global timer, so a count that never arrives ends the kernel
// with a status bit instead of a hang.
__global__ void wait_ready_kernel(const unsigned* ready, int P, unsigned target, unsigned long long timeout_ns,
                                  unsigned* status, unsigned timeout_bit) {
  const int r = threadIdx.x;
  if (r >= P) return;
  const uint64_t t0 = ptx::global_timer_ns();
  while (ptx::ld_acquire_gpu(ready + r) < target) {
    if (ptx::global_timer_ns() - t0 > timeout_ns) {
      atomicOr(status, timeout_bit);
      return;
    }
    __nanosleep(256);
  }
}

}  // namespace

cudaError_t launch_wait_ready(const unsigned* ready, int P, unsigned target, unsigned long long timeout_ns,
                              unsigned* status, unsigned timeout_bit, cudaStream_t stream) {
  wait_ready_kernel<<<1, ((P + 31) / 32) * 32, 0, stream>>>(ready, P, target, timeout_ns, status, timeout_bit);
  return cudaGetLastError();
}

}  // namespace qnre
