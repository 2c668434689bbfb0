// fused_qkv.cuh -- kernel arguments and launcher of the fused QKV projection +
// per-head RMSNorm + RoPE + head-band scatter (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace qnre {

// Tile geometry.  A cluster of two CTAs (an SM pair) owns a 256 x 256 tile of
// Y = x W: 256 tokens by two 128-wide heads.  Each CTA holds 128 of the rows
// (its own A half and its own accumulator rows) and 128 of the columns of the
// B tile; the pair's tcgen05.mma (cta_group::2) combines them.  A token's whole
// head row is one TMEM lane of one CTA.
#ifndef QNRE_DEBUG_BOUNDS
#define QNRE_DEBUG_BOUNDS 0  // 1: debug build, every output store checked against its buffer's extent
#endif

constexpr int kBM = 128;                      // rows per CTA (256 per pair)
constexpr int kPairM = 2 * kBM;
constexpr int kBN = 256;                      // columns per tile (two heads)
constexpr int kBNHalf = kBN / 2;              // B columns held by each CTA
constexpr int kBK = 64;                       // one 128-byte swizzle row of bf16
#ifndef QNRE_FUSED_STAGES
#define QNRE_FUSED_STAGES 5
#endif
constexpr int kStages = QNRE_FUSED_STAGES;  // 32 KiB per stage per CTA
constexpr int kThreads = 192;                 // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kABytes = kBM * kBK * 2;        // 16 KiB
constexpr int kBBytes = kBNHalf * kBK * 2;    // 16 KiB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kAccCols = kBN;                 // fp32 accumulator columns per buffer
constexpr int kTmemCols = 2 * kAccCols;       // double-buffered accumulator
constexpr int kBarBytes = 256;                // mbarriers + small words
// One 32-row bf16 head tile per epilogue warp, as two 32 x 128-byte halves
// (columns 0-63 and 64-127) in the 128-byte swizzle layout that TMA stores read.
constexpr int kEpiHalfBytes = 32 * 128;
constexpr int kEpiWarpBytes = 2 * kEpiHalfBytes;
constexpr int kEpiStageBytes = 4 * kEpiWarpBytes;
constexpr int kStoreRows = 32;  // rows per TMA store box (one epilogue warp's tokens)
constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + kBarBytes +
                           2 * 128 * 4 /*norm weights*/ + kEpiStageBytes;
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds the sm_103a limit");

struct FusedArgs {
  CUtensorMap tmap_x;  // bf16 [T, K], box 64 x 128, 128-byte swizzle
  CUtensorMap tmap_w;  // bf16 [K, N], box 64 x 64, 128-byte swizzle
  // Head-band outputs for TMA stores (when tma_store): bshd q, k, v as
  // [P*B*S_g, H_local, 128], or the fused payload (index 0) as
  // [P*B*S_g, H_local, 384]; box 64 x 1 x 32, 128-byte swizzle.
  CUtensorMap tmap_out[3];
  int tma_store;  // 1: warps whose 32 tokens sit in one segment store their head rows with TMA
  const uint16_t* q_norm_w;
  const uint16_t* k_norm_w;
  const float* cos_sin;
  const int32_t* positions;
  uint16_t* out_q;
  uint16_t* out_k;
  uint16_t* out_v;
  uint16_t* out_fused;
  unsigned* status;
  unsigned* ready;  // per destination rank, or null: per-warp head-row publication counts
  long long out_elems;  // elements of each output tensor (q, k and v each, or the fused payload)
  long long n_pos;
  int T, K, N, H, H_local, P, B, S;
  int layout;       // 0 bshd, 1 fused
  int rope_style;   // 0 rotate-half, 1 interleaved
  int epilogue_on;  // 0: bare projection
  int num_m_tiles, num_n_tiles, num_tiles, group_m, num_k_blocks;  // m tiles are 256 rows
  // Row units of the raster: num_m_tiles, or ceil(num_m_tiles / 2) when two
  // pairs share a cluster and take adjacent row tiles of the same column tile.
  int num_mp_tiles;
  // Work list: items [0, num_full) are whole 256x256 tiles in raster order; items
  // [num_full, num_work) split the remaining tiles into 256x128 halves (one head
  // each), so a short last round or a small problem spreads over more pairs.
  int num_full, num_work;
};

// Enqueue the fused kernel: `units` clusters of `pairs_per_cluster` CTA pairs
// (1, or 2 sharing W through TMA multicast) walk the work list persistently.
cudaError_t launch_fused_qkv(const FusedArgs& args, int units, int pairs_per_cluster, cudaStream_t stream);

// Split of num_tiles pair tiles over at most max_pairs pairs: how many stay
// whole, and how many work items (whole + halves) that makes.
inline void plan_work(int num_tiles, int max_pairs, int* num_full, int* num_work) {
  if (2 * num_tiles <= max_pairs) {  // small problem: every tile in two halves
    *num_full = 0;
    *num_work = 2 * num_tiles;
    return;
  }
  const int rem = num_tiles % max_pairs;
  if (rem > 0 && 2 * rem <= max_pairs) {  // short last round: halve its tiles
    *num_full = num_tiles - rem;
    *num_work = *num_full + 2 * rem;
    return;
  }
  *num_full = num_tiles;
  *num_work = num_tiles;
}

// Readiness count a complete forward publishes to each destination rank:
// every epilogue warp of every pair tile adds 1 per head of that rank it stored.
inline unsigned long long ready_target(long long num_m_tiles, int H_local) {
  return static_cast<unsigned long long>(num_m_tiles) * 2 /*CTAs*/ * 4 /*epilogue warps*/ * 3 /*q,k,v*/ * H_local;
}

// Enqueue a one-CTA wait: thread r spins (with acquire loads) until ready[r] >=
// target or `timeout_ns` passes; on expiry it ORs `timeout_bit` into *status.
cudaError_t launch_wait_ready(const unsigned* ready, int P, unsigned target, unsigned long long timeout_ns,
                              unsigned* status, unsigned timeout_bit, cudaStream_t stream);

// One-time per-device kernel setup (shared-memory opt-in); returns how many
// clusters of one CTA pair (*max_pairs) and of two pairs (*max_quads) fit on
// the current device at once (*max_quads may be 0).
cudaError_t prepare_fused_qkv_kernel(int* max_pairs, int* max_quads);

}  // namespace qnre
