// Kernels of the fused linear cross-entropy for sm_103a.
//
// One persistent, warp-specialised tcgen05 GEMM template serves the four
// contractions of the method (source: "Long-Sequence MoE RL Training: From
// First Principles to MI300X", section 3):
//
//   MODE_FWD  Z = H W^T tile by tile (M = tokens, N = vocab, K = Hd); the
//             epilogue folds each tile into a per-row running max and sum of
//             exponentials (the log-sum-exp recurrence) and picks out the
//             target logit.  Z is never written.
//   MODE_DZ   the same logit tiles recomputed for one token chunk; the
//             epilogue forms dZ = g (exp(z - lse) - onehot) in registers and
//             stores it as bf16 into the [chunk x V] dZ slice.
//   MODE_DHW  both contractions of that dZ slice in one launch:
//               dH[chunk] = dZ W        (M = tokens, N = Hd, K = vocab)
//               dW (+)= dZ^T H[chunk]   (M = vocab,  N = Hd, K = tokens)
//             Tiles are handed out by a global atomic counter, the long dH
//             tiles first, so the short dW tiles fill the SMs that the dH
//             tiles leave idle at the end of their last wave.
//   MODE_SCORE MODE_FWD that also keeps each row's largest logit and its id
//             (the greedy token), for scoring without a loss.
//
// SM pairs: every kernel runs as clusters of two CTAs on two SMs that compute
// one 256 x 256 output tile together with cta_group::2 MMAs (M = 256, N = 256,
// K = 16).  CTA rank r of the pair stages rows 128*r .. +127 of the A tile and
// rows 128*r .. +127 of the B tile (B's N dimension) in its own shared memory;
// the tensor cores of the pair read both halves, so each SM streams half of B
// instead of all of it.  Rank r's TMEM holds rows 128*r .. +127 of the fp32
// accumulator (all 256 columns).
//
// CTA layout: 6 warps per CTA.  Warp 0: TMA producer (one elected thread) in
// both CTAs; their loads are counted on the even CTA's stage barrier.  Warp 1:
// TMEM allocator in both CTAs; in the even CTA also the MMA issuer (one
// elected thread), whose commits arrive on the barriers of both CTAs.  Warps
// 2..5: epilogue; warp w reads TMEM lanes 32*(w%4) .. +31 of its own CTA and
// signals the even CTA when the accumulator may be overwritten.
//
// K blocks are 64 deep: one bf16 K block of a row is 128 bytes, the width of
// the 128-byte TMA / UMMA swizzle.  Operand halves pass through a ring of
// NSTAGE shared-memory stages; the accumulator is double-buffered in TMEM
// (2 x 256 columns) so that the epilogue of one tile overlaps the MMAs of the
// next.  Exception: MODE_DHW's dH tiles are 256 x 512 when Hd allows (two N =
// 256 MMAs per A slice, both accumulators, the ring re-cut in WIDE_NSTAGE
// larger stages), which moves fewer operand bytes per FLOP on their long K loop.
//
// Work is handed out dynamically for the forward units and the MODE_DHW tiles
// (a global counter and a small ring in shared memory, see "work-index ring")
// and statically for the dZ recompute's tiles.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace flce {

constexpr int BM = 128;                         // tile rows held by one CTA (the pair MMA has M = 256)
constexpr int BN = 256;                         // N of the pair MMA
constexpr int BN_HALF = BN / 2;                 // rows of B staged by each CTA of the pair
constexpr int BK = 64;
constexpr int NSTAGE = 6;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN_HALF * BK * 2;       // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB per CTA
constexpr uint32_t PAIR_TX_BYTES = 2 * STAGE_BYTES;  // both CTAs' loads of a stage
// MODE_DHW wide dH tiles (256 tokens x 512 hidden columns per pair): a stage holds
// the A block and two 128-column halves of B, and the same 192 KB of shared
// memory is cut into 4 such stages instead of 6.
constexpr int WIDE_NSTAGE = 4;
constexpr int WIDE_B_BYTES = 2 * B_BYTES;                  // 32 KB
constexpr int WIDE_STAGE_BYTES = A_BYTES + WIDE_B_BYTES;   // 48 KB per CTA
constexpr uint32_t WIDE_PAIR_TX_BYTES = 2 * WIDE_STAGE_BYTES;
static_assert(WIDE_NSTAGE * WIDE_STAGE_BYTES <= NSTAGE * STAGE_BYTES, "wide stages fit the ring");
static_assert(WIDE_STAGE_BYTES % 1024 == 0, "128-byte swizzle atoms stay 1024-byte aligned");
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int STAGING_BOX_BYTES = 32 * 128;     // 32 rows x 128 bytes
constexpr int STAGING_BYTES = kEpiWarps * 2 * STAGING_BOX_BYTES;
constexpr uint32_t TMEM_COLS = 512;
constexpr int kTileRing = 8;                    // MODE_DHW: tile indices in flight inside a CTA
// full[NSTAGE], empty[NSTAGE], tmem_full[2], tmem_empty[2], drain, tile_full[R], tile_empty[R]
constexpr int kBarriers = 2 * NSTAGE + 5 + 2 * kTileRing;
constexpr int kSmemTail = 512;                  // barriers + TMEM slot + abort flag + tile ring
constexpr uint64_t kDrainTimeoutNs = 2000000000ull;
constexpr uint64_t kAbortSettleNs = 200000ull;   // 200 us: far longer than any TMA load takes
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum Mode : int { MODE_FWD = 0, MODE_DZ = 1, MODE_DHW = 2, MODE_SCORE = 3 };

// MODE_SCORE is MODE_FWD plus a per-row argmax of the logits.
__host__ __device__ constexpr bool is_forward(int mode) { return mode == MODE_FWD || mode == MODE_SCORE; }

// Device status codes (match flce_status in include/flce.h).
constexpr int kStatusTargetRange = 6;
constexpr int kStatusTimeout = 7;

__host__ __device__ constexpr int smem_bytes_for(int mode) {
  return 1024 + NSTAGE * STAGE_BYTES + (is_forward(mode) ? 0 : STAGING_BYTES) + kSmemTail;
}
static_assert(smem_bytes_for(MODE_DHW) <= 232448, "shared memory per CTA");
static_assert(kBarriers * 8 + 8 + kTileRing * 4 <= kSmemTail, "smem tail");

// DzPanels: the backward's [chunk x V] bf16 dZ block is stored as V_pad / 64
// panels of 64 vocab columns, each panel [chunk rows x 64 columns] row-major
// (128 bytes per row), panel after panel.  Its three tensor maps are 3-D
// {64 columns, rows, panels}; every box the kernels move (32 x 64 stored, 128 x 64
// and 64 x 64 loaded) is then one contiguous run of memory instead of 32..128
// rows 2 V bytes apart.
struct GemmParams {
  // MODE_FWD / MODE_DZ: A = H (K-major), B = W (K-major), tmOut = dZ store (panels).
  // MODE_DHW dH tiles: A = dZ (K-major, panels), B = W (MN-major); dH written through dH_out.
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmOut;
  // MODE_DHW dW tiles: A = dZ (MN-major, panels), B = H (MN-major), tmOut2 = dW store / reduce.
  CUtensorMap tmA2;
  CUtensorMap tmB2;
  CUtensorMap tmOut2;
  int32_t num_m_pairs;   // 256-row tile pairs along M (tokens); MODE_DHW: dH tiles
  int32_t num_n_blocks;
  int32_t num_k_blocks;
  int32_t n_split;       // MODE_FWD: vocab ranges per token block
  int32_t split_group;   // MODE_FWD: vocab ranges side by side in the unit order (divides n_split)
  int32_t dynamic_units; // MODE_FWD: 1 = units from the work-index ring, 0 = strided over the pairs
  int32_t num_units;
  int32_t row0;          // first row of the launch in the A / B2 operand maps (0 for MODE_FWD)
  int32_t rows;          // rows of the launch (T for MODE_FWD); over a row list: the chunk's capacity
  int32_t T;
  int32_t V;
  int32_t part_stride;   // MODE_FWD: row stride of one split's partials
  int32_t reduce_out;    // MODE_DHW: dW tiles 0 = store, 1 = reduce-add into the output
  int32_t n_dh_tiles;    // MODE_DHW: dH tiles come first in the tile order ...
  int32_t n_dw_tiles;    // ... then the dW tiles
  int32_t num_k_blocks2; // MODE_DHW: K blocks of a dW tile (tokens of the chunk / 64)
  int32_t dh_wide;       // MODE_DHW: 1 = dH tiles are 256 x 512 (both TMEM accumulators), 0 = 256 x 256
  int64_t vocab_offset;  // global id of local vocab row 0 (a vocab shard); 0 for the full vocabulary
  int64_t ignore_index;
  const int64_t* targets;
  const float* lse;      // MODE_DZ
  const float* g;        // MODE_DZ
  float2* partials;      // MODE_FWD [n_split][part_stride] of (max*log2e, sum of 2^(z*log2e - max))
  float* zy;             // MODE_FWD [T] target logit
  float* best_val;       // MODE_SCORE [n_split][part_stride]: largest logit of the row's vocab range
  int32_t* best_idx;     // MODE_SCORE [n_split][part_stride]: its global vocab id (lowest on ties)
  int32_t* tile_counter; // MODE_DHW tiles / forward units handed out so far; zero before the launch
  int32_t* status;
  uint64_t timeout_ns;
  // Over a list of rows (the backward skips rows whose upstream gradient is zero;
  // the forward of flce_forward_valid skips rows with an ignored target): the launch
  // holds list positions index0 .. index0 + rows - 1 of the row list, whose length a
  // prep kernel writes to *rows_dev; token rows of H / dH come gathered in buffers
  // of their own, and targets, lse and g are read through row_index.
  // rows_dev == nullptr: rows row0 .. row0 + rows - 1.
  const int32_t* rows_dev;
  const int32_t* row_index;
  int32_t index0;
  uint16_t* dH_out;      // MODE_DHW: dH [T, Hd] bf16 (row stride dH_ld elements); dH tiles write their
  int64_t dH_ld;         //   rows straight to their tokens' rows through the row list
  int32_t Hd;
  float* dW_zero;        // MODE_DHW: dW, zero-filled here when the list is empty
  int64_t dW_elems;
};

// Extent of one launch: the host's figures, or, over compacted rows, the ones
// that follow from the chunk's share of the row list.
struct Counts {
  int rows;           // rows of the chunk
  int num_m_pairs;    // 256-row pairs along M (unit modes) / dH tiles' token pairs
  int num_units;      // unit modes (forward, scoring, dZ recompute): work units
  int n_dh_tiles;     // MODE_DHW
  int num_k_blocks2;  // MODE_DHW: K blocks of a dW tile
};

template <int MODE>
__device__ __forceinline__ Counts counts_of(const GemmParams& p) {
  Counts c;
  if (!p.rows_dev) {
    c.rows = p.rows;
    c.num_m_pairs = p.num_m_pairs;
    c.num_units = p.num_units;
    c.n_dh_tiles = p.n_dh_tiles;
    c.num_k_blocks2 = p.num_k_blocks2;
    return c;
  }
  c.rows = min(max(*p.rows_dev - p.index0, 0), p.rows);
  c.num_m_pairs = (c.rows + 2 * BM - 1) / (2 * BM);
  c.num_units = c.num_m_pairs * (is_forward(MODE) ? p.n_split : p.num_n_blocks);
  c.n_dh_tiles = c.num_m_pairs * (p.dh_wide ? p.num_n_blocks / 2 : p.num_n_blocks);
  c.num_k_blocks2 = (c.rows + BK - 1) / BK;
  return c;
}

struct Unit {
  int m_blk;
  int n_lo;
  int n_hi;
  int split;
};

// Work unit of a pair; m_blk is this CTA's 128-row block (2 * pair + rank).
template <int MODE>
__device__ __forceinline__ Unit decode_unit(const GemmParams& p, const Counts& c, int u, uint32_t rank) {
  Unit r;
  if constexpr (is_forward(MODE)) {
    // Units in groups of G = p.split_group vocab ranges: (token pair 0, range
    // 0 .. G-1), (token pair 1, range 0 .. G-1), ..., then the next G ranges.
    // Two schedules (chosen on the host from measurements):
    //  * range-major (G = 1) with the units from the work-index ring, when the
    //    in-flight pairs' H blocks (512 * Hd bytes each) fit in L2: the pairs
    //    then hold consecutive token pairs of one range and share each W tile
    //    (forward DRAM reads 5.5-7.7 GB at 65,536 x 2048 x 124,160, against
    //    13.5-14.5 GB with G = 2);
    //  * otherwise G = 4 (or 2) with the units strided over the pairs (pair c
    //    takes units c, c + pairs, ...), which puts the units sharing an H block
    //    on neighbouring clusters (at 131,072 x 4096 x 124,160 the forward takes
    //    78-79 ms with G = 4 and 80-81 ms with G = 2, against 86-90 ms from the
    //    ring with G = 1, 2 or 4).
    const int G = p.split_group;
    const int gsz = G * c.num_m_pairs;
    const int grp = u / gsz;
    const int rr = u - grp * gsz;
    const int split = grp * G + rr % G;
    const int base = p.num_n_blocks / p.n_split;
    const int rem = p.num_n_blocks % p.n_split;
    r.m_blk = 2 * (rr / G) + static_cast<int>(rank);
    r.split = split;
    r.n_lo = split * base + min(split, rem);
    r.n_hi = r.n_lo + base + (split < rem ? 1 : 0);
  } else {
    const int nb = u / c.num_m_pairs;  // token blocks fastest: the W tile is shared in L2
    r.m_blk = 2 * (u - nb * c.num_m_pairs) + static_cast<int>(rank);
    r.n_lo = nb;
    r.n_hi = nb + 1;
    r.split = 0;
  }
  return r;
}

// One MODE_DHW tile: family 0 = dH, family 1 = dW; Hd blocks fastest so that
// CTAs running side by side share the dZ rows (dH) or dZ columns (dW) in L2.
// With p.dh_wide, a dH tile covers 512 hidden columns (nb counts 512-column
// blocks) and uses both TMEM accumulators.
struct Tile {
  int family;
  int m_blk;
  int nb;
  int num_k;
  bool wide;
};

__device__ __forceinline__ Tile decode_dhw(const GemmParams& p, const Counts& c, int t, uint32_t rank) {
  Tile r;
  r.family = t < c.n_dh_tiles ? 0 : 1;
  r.wide = r.family == 0 && p.dh_wide != 0;
  const int u = r.family ? t - c.n_dh_tiles : t;
  const int nbl = r.wide ? p.num_n_blocks / 2 : p.num_n_blocks;
  const int pair = u / nbl;
  r.nb = u - pair * nbl;
  r.m_blk = 2 * pair + static_cast<int>(rank);
  r.num_k = r.family ? c.num_k_blocks2 : p.num_k_blocks;
  return r;
}

__device__ __forceinline__ void raise_status(int32_t* status, int code) { atomicCAS(status, 0, code); }

struct SmemLayout {
  uint8_t* stages;
  uint8_t* staging;
  uint64_t* bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  volatile int* tile_ring;
};

template <int MODE>
__device__ __forceinline__ SmemLayout carve_smem(uint8_t* raw) {
  SmemLayout s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.stages = base;
  s.staging = base + NSTAGE * STAGE_BYTES;
  uint8_t* tail = s.staging + (is_forward(MODE) ? 0 : STAGING_BYTES);
  s.bars = reinterpret_cast<uint64_t*>(tail);
  s.tmem_slot = reinterpret_cast<uint32_t*>(tail + kBarriers * 8);
  s.abort_flag = reinterpret_cast<volatile int*>(tail + kBarriers * 8 + 4);
  s.tile_ring = reinterpret_cast<volatile int*>(tail + kBarriers * 8 + 8);
  return s;
}

__device__ __forceinline__ uint32_t bar_full(const SmemLayout& s, int i) { return ptx::smem_u32(s.bars + i); }
__device__ __forceinline__ uint32_t bar_empty(const SmemLayout& s, int i) {
  return ptx::smem_u32(s.bars + NSTAGE + i);
}
__device__ __forceinline__ uint32_t bar_tfull(const SmemLayout& s, int i) {
  return ptx::smem_u32(s.bars + 2 * NSTAGE + i);
}
__device__ __forceinline__ uint32_t bar_tempty(const SmemLayout& s, int i) {
  return ptx::smem_u32(s.bars + 2 * NSTAGE + 2 + i);
}
__device__ __forceinline__ uint32_t bar_drain(const SmemLayout& s) { return ptx::smem_u32(s.bars + 2 * NSTAGE + 4); }
__device__ __forceinline__ uint32_t bar_tile_full(const SmemLayout& s, int i) {
  return ptx::smem_u32(s.bars + 2 * NSTAGE + 5 + i);
}
__device__ __forceinline__ uint32_t bar_tile_empty(const SmemLayout& s, int i) {
  return ptx::smem_u32(s.bars + 2 * NSTAGE + 5 + kTileRing + i);
}

__device__ __forceinline__ void abort_cta(const GemmParams& p, const SmemLayout& s) {
  *s.abort_flag = 1;
  raise_status(p.status, kStatusTimeout);
}

// ----------------------------------------------------------------------------- operand loads (one K block)
// Each CTA of the pair loads its A rows (its m_blk) and its half of B (N rows
// nb*256 + 128*rank ..); `full` is the even CTA's stage barrier, as a
// shared::cluster address, which counts the bytes of both CTAs.
// K-major H and W for the logits (forward and recompute).
__device__ __forceinline__ void load_logits_stage(const GemmParams& p, uint32_t a_dst, uint32_t b_dst,
                                                  uint32_t full, int m_blk, int nb, int k0, uint32_t rank) {
  ptx::tma_load_2d_pair(a_dst, &p.tmA, k0, p.row0 + m_blk * BM, full);
  ptx::tma_load_2d_pair(b_dst, &p.tmB, k0, nb * BN + static_cast<int>(rank) * BN_HALF, full);
}

// dH tile: dZ rows (K-major, K = vocab) and W as MN-major 64-column boxes.
// The dZ block is stored in 64-column panels (see DzPanels): K block k0 / 64
// of 128 token rows is one contiguous 16 KB piece of panel k0 / 64.
__device__ __forceinline__ void load_dh_stage(const GemmParams& p, uint32_t a_dst, uint32_t b_dst, uint32_t full,
                                              int m_blk, int nb, int k0, uint32_t rank) {
  ptx::tma_load_3d_pair(a_dst, &p.tmA, 0, m_blk * BM, k0 / BK, full);
#pragma unroll
  for (int j = 0; j < BN_HALF / 64; ++j)
    ptx::tma_load_2d_pair(b_dst + j * 8192, &p.tmB, nb * BN + static_cast<int>(rank) * BN_HALF + j * 64, k0, full);
}

// dW tile: dZ^T (MN-major 64-vocab boxes, K = tokens) and H[chunk] as MN-major boxes.
// 64 vocab rows x 64 tokens of dZ^T are 64 consecutive 128-byte rows of one panel.
__device__ __forceinline__ void load_dw_stage(const GemmParams& p, uint32_t a_dst, uint32_t b_dst, uint32_t full,
                                              int m_blk, int nb, int k0, uint32_t rank) {
#pragma unroll
  for (int j = 0; j < BM / 64; ++j)
    ptx::tma_load_3d_pair(a_dst + j * 8192, &p.tmA2, 0, k0, (m_blk * BM) / 64 + j, full);
#pragma unroll
  for (int j = 0; j < BN_HALF / 64; ++j)
    ptx::tma_load_2d_pair(b_dst + j * 8192, &p.tmB2, nb * BN + static_cast<int>(rank) * BN_HALF + j * 64,
                          p.row0 + k0, full);
}

// Wide dH tile: the A block as for dH, and B as two halves of 128 hidden
// columns each (the pair MMA's N = 256 halves of this CTA for hidden columns
// nb*512 + 128*rank .. and nb*512 + 256 + 128*rank ..), 16 KB apart.
__device__ __forceinline__ void load_dh_wide_stage(const GemmParams& p, uint32_t a_dst, uint32_t b_dst,
                                                   uint32_t full, int m_blk, int nbw, int k0, uint32_t rank) {
  ptx::tma_load_3d_pair(a_dst, &p.tmA, 0, m_blk * BM, k0 / BK, full);
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int j = 0; j < BN_HALF / 64; ++j)
      ptx::tma_load_2d_pair(b_dst + h * B_BYTES + j * 8192, &p.tmB,
                            nbw * 2 * BN + h * BN + static_cast<int>(rank) * BN_HALF + j * 64, k0, full);
}

// Stage ring of one role (producer or MMA issuer).  Each stage's barriers keep
// their own phase (bit i of `parity` is the parity of the next use of stage i),
// so the ring can be re-cut: NSTAGE stages of STAGE_BYTES, or WIDE_NSTAGE
// stages of WIDE_STAGE_BYTES for wide dH tiles, over the same shared memory.
struct Ring {
  uint32_t stage = 0, parity = 0, used = 0;
  int nst = NSTAGE;
  __device__ __forceinline__ uint32_t stage_bytes() const {
    return nst == NSTAGE ? static_cast<uint32_t>(STAGE_BYTES) : static_cast<uint32_t>(WIDE_STAGE_BYTES);
  }
  __device__ __forceinline__ uint32_t parity_of(uint32_t i) const { return (parity >> i) & 1u; }
  __device__ __forceinline__ void advance() {
    used |= 1u << stage;
    parity ^= 1u << stage;
    if (++stage == static_cast<uint32_t>(nst)) stage = 0;
  }
};

// The producer's side: before the ring is re-cut, every load it issued must
// have been consumed (the MMAs released the stage), since the new stages
// overlap the old ones.  Returns false when a wait ran out.
__device__ __forceinline__ bool producer_recut(const GemmParams& p, const SmemLayout& s, Ring& r, int nst) {
  if (r.nst == nst) return true;
  for (uint32_t i = 0; i < static_cast<uint32_t>(r.nst); ++i)
    if (r.used & (1u << i))
      if (!ptx::wait_bounded_cluster(bar_empty(s, i), r.parity_of(i) ^ 1u, p.timeout_ns, s.abort_flag)) {
        abort_cta(p, s);
        return false;
      }
  r.nst = nst;
  r.stage = 0;
  return true;
}

// The MMA issuer's side of a re-cut (it has consumed every stage it waited on).
__device__ __forceinline__ void mma_recut(Ring& r, int nst) {
  if (r.nst == nst) return;
  r.nst = nst;
  r.stage = 0;
}

// The even CTA's stage barriers count both CTAs' loads: waiting on the
// last-armed phase of each stage means no TMA write of either CTA is in
// flight.  (The odd CTA's loads are consumed by the same MMAs.)
__device__ __forceinline__ void producer_drain(const SmemLayout& s, const Ring& r, uint32_t rank) {
  if (rank != 0) return;
  for (uint32_t i = 0; i < static_cast<uint32_t>(NSTAGE); ++i)
    if (r.used & (1u << i)) ptx::wait_bounded(bar_full(s, i), r.parity_of(i) ^ 1u, kDrainTimeoutNs, nullptr);
}

// Loads the K blocks of one tile; `kind` 0 = logits, 1 = dH, 2 = dW, 3 = wide dH
// (the ring must be cut for the kind: WIDE_NSTAGE stages for 3, NSTAGE otherwise).
__device__ __forceinline__ bool produce_tile(const GemmParams& p, const SmemLayout& s, Ring& ps, int kind,
                                             int m_blk, int nb, int num_k, uint32_t rank) {
  const uint32_t tx = kind == 3 ? WIDE_PAIR_TX_BYTES : PAIR_TX_BYTES;
  for (int kb = 0; kb < num_k; ++kb) {
    if (!ptx::wait_bounded_cluster(bar_empty(s, ps.stage), ps.parity_of(ps.stage) ^ 1u, p.timeout_ns,
                                   s.abort_flag)) {
      abort_cta(p, s);
      return false;
    }
    const uint32_t full_local = bar_full(s, ps.stage);
    if (rank == 0) ptx::mbar_arrive_expect_tx(full_local, tx);
    const uint32_t full = ptx::mapa(full_local, 0);
    const uint32_t a_dst = ptx::smem_u32(s.stages + ps.stage * ps.stage_bytes());
    const uint32_t b_dst = a_dst + A_BYTES;
    const int k0 = kb * BK;
    if (kind == 0)
      load_logits_stage(p, a_dst, b_dst, full, m_blk, nb, k0, rank);
    else if (kind == 1)
      load_dh_stage(p, a_dst, b_dst, full, m_blk, nb, k0, rank);
    else if (kind == 2)
      load_dw_stage(p, a_dst, b_dst, full, m_blk, nb, k0, rank);
    else
      load_dh_wide_stage(p, a_dst, b_dst, full, m_blk, nb, k0, rank);
    ps.advance();
  }
  return true;
}

// ----------------------------------------------------------------------------- MMA (one tile)
// Issues the K loop of one pair tile into the accumulator at d_tmem (rows
// 0..127 in the even CTA's TMEM, 128..255 in the odd CTA's); each stage is
// released to both CTAs' producers when its MMAs complete.  K-major
// operand: the 16-deep slice is 32 bytes further along the swizzled 128-byte
// row, 8-row groups 1024 bytes apart.  MN-major operand: the slice is 16 rows
// (2048 bytes) further, 64-wide MN blocks 8 KB apart.
__device__ __forceinline__ bool mma_tile(const GemmParams& p, const SmemLayout& s, uint32_t d_tmem, int num_k,
                                         uint32_t a_mn, uint32_t b_mn, uint32_t idesc, Ring& r) {
  for (int kb = 0; kb < num_k; ++kb) {
    if (!ptx::wait_bounded(bar_full(s, r.stage), r.parity_of(r.stage), p.timeout_ns, s.abort_flag)) {
      abort_cta(p, s);
      return false;
    }
    ptx::tc_fence_after();
    const uint32_t a_addr = ptx::smem_u32(s.stages + r.stage * r.stage_bytes());
    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
    for (int k = 0; k < BK / 16; ++k) {
      const uint64_t a_desc = a_mn ? ptx::smem_desc_sw128(a_addr + k * 2048, 8192, 1024)
                                   : ptx::smem_desc_sw128(a_addr + k * 32, 16, 1024);
      const uint64_t b_desc = b_mn ? ptx::smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                   : ptx::smem_desc_sw128(b_addr + k * 32, 16, 1024);
      ptx::mma_bf16_pair(d_tmem, a_desc, b_desc, idesc, (kb | k) != 0 ? 1u : 0u);
    }
    ptx::mma_commit_pair(bar_empty(s, r.stage), 0x3);
    r.advance();
  }
  return true;
}

// Wide dH tile: per 16-deep slice, the K-major A slice is multiplied with both
// MN-major B halves, into the accumulators at d0 (hidden columns 0..255 of the
// 512) and d1 (256..511).
__device__ __forceinline__ bool mma_tile_wide(const GemmParams& p, const SmemLayout& s, uint32_t d0, uint32_t d1,
                                              int num_k, uint32_t idesc, Ring& r) {
  for (int kb = 0; kb < num_k; ++kb) {
    if (!ptx::wait_bounded(bar_full(s, r.stage), r.parity_of(r.stage), p.timeout_ns, s.abort_flag)) {
      abort_cta(p, s);
      return false;
    }
    ptx::tc_fence_after();
    const uint32_t a_addr = ptx::smem_u32(s.stages + r.stage * r.stage_bytes());
    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
    for (int k = 0; k < BK / 16; ++k) {
      const uint64_t a_desc = ptx::smem_desc_sw128(a_addr + k * 32, 16, 1024);
      const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
      ptx::mma_bf16_pair(d0, a_desc, ptx::smem_desc_sw128(b_addr + k * 2048, 8192, 1024), idesc, acc);
      ptx::mma_bf16_pair(d1, a_desc, ptx::smem_desc_sw128(b_addr + B_BYTES + k * 2048, 8192, 1024), idesc, acc);
    }
    ptx::mma_commit_pair(bar_empty(s, r.stage), 0x3);
    r.advance();
  }
  return true;
}

// ----------------------------------------------------------------------------- epilogue pieces
// TMEM load of 32 columns for this warp's 32 rows, completed before return.
__device__ __forceinline__ void tmem_load32_sync(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  ptx::tmem_ld32(taddr, r);
  ptx::tmem_wait_ld32(r);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// Write eight 16-byte chunks (32 words) of this lane's staging row using the
// 128-byte swizzle the TMA store expects: chunk k of row r lands at
// r*128 + ((k ^ (r % 8)) * 16).
__device__ __forceinline__ void stage_row_words(uint32_t buf, int lane, const uint32_t (&w)[32]) {
  const uint32_t row = buf + lane * 128;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    ptx::st_shared_v4(row + ((k ^ (lane & 7)) << 4), w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

// Stages one 32-row x 128-byte box in a staging buffer (alternating two per
// warp) and stores or reduce-adds it with TMA at (x, yrow), or, with panel >= 0,
// stores it at (0, yrow, panel) of a map over 64-column panels.
__device__ __forceinline__ void store_box(const CUtensorMap* tm, bool reduce, uint32_t staging0,
                                          uint32_t& box_count, int lane, const uint32_t (&w)[32], int x, int yrow,
                                          int panel = -1) {
  const uint32_t buf = staging0 + (box_count & 1u) * STAGING_BOX_BYTES;
  if (lane == 0) ptx::bulk_wait_read<1>();
  __syncwarp();
  stage_row_words(buf, lane, w);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (panel >= 0)
      ptx::tma_store_3d(tm, buf, 0, yrow, panel);
    else if (reduce)
      ptx::tma_reduce_add_2d(tm, buf, x, yrow);
    else
      ptx::tma_store_2d(tm, buf, x, yrow);
    ptx::bulk_commit();
  }
  ++box_count;
}

// dZ tile store: 4 boxes of 64 columns.  Each accumulator value z becomes
// g (2^(z log2e - lse log2e) - [col == y]), columns at or past V become 0 (the
// last panel's tail is read back as K by the dH tiles), and box j goes to
// panel x0 / 64 + j of the dZ block.
__device__ __forceinline__ void epi_dz_tile(const CUtensorMap* tm, uint32_t tcol, int x0, int yrow,
                                            uint32_t staging0, uint32_t& box_count, int lane, float gt, float lse2,
                                            int y, int V) {
#pragma unroll 1
  for (int j = 0; j < BN / 64; ++j) {
    uint32_t w[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float v[32];
      tmem_load32_sync(tcol + j * 64 + h * 32, v);
      const int col0 = x0 + j * 64 + h * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = ptx::ex2(fmaf(v[i], kLog2e, -lse2));
      const int yo = y - col0;
      if (static_cast<unsigned>(yo) < 32u) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i == yo) v[i] -= 1.0f;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= gt;
      if (col0 + 32 > V) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i >= V) v[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) w[h * 16 + i] = ptx::pack_bf16x2(v[2 * i], v[2 * i + 1]);
    }
    store_box(tm, false, staging0, box_count, lane, w, x0 + j * 64, yrow, x0 / 64 + j);
  }
}

// bf16 dH tile rows (256 columns from x0) written straight to their tokens' rows
// of dH: lane l of the warp holds chunk row l, whose token is `token` (< 0: no
// row).  Each 64-column piece is staged (one row per lane, 128-byte swizzle) and
// read back four rows per instruction, 8 lanes per 128-byte row segment, so every
// store covers whole segments.  Columns >= Hd are not written.
__device__ __forceinline__ void epi_dh_rows(uint16_t* dH, int64_t ld, int Hd, int token, uint32_t tcol, int x0,
                                            uint32_t staging0, uint32_t& box_count, int lane) {
  const int sub = lane >> 3;   // row within a group of four
  const int piece = lane & 7;  // 16-byte piece of the row segment
  // The staging buffers may still be read by this warp's TMA stores of a dW tile.
  if (lane == 0) ptx::bulk_wait_read<0>();
  __syncwarp();
#pragma unroll 1
  for (int j = 0; j < BN / 64; ++j) {
    uint32_t w[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float v[32];
      tmem_load32_sync(tcol + j * 64 + h * 32, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) w[h * 16 + i] = ptx::pack_bf16x2(v[2 * i], v[2 * i + 1]);
    }
    const uint32_t buf = staging0 + (box_count & 1u) * STAGING_BOX_BYTES;
    __syncwarp();
    stage_row_words(buf, lane, w);
    __syncwarp();
    const int col = x0 + j * 64 + piece * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + sub;
      const int tok = __shfl_sync(0xffffffffu, token, r);
      uint32_t a, b, c, d;
      ptx::ld_shared_v4(buf + r * 128 + ((piece ^ (r & 7)) << 4), a, b, c, d);
      if (tok >= 0 && col < Hd) ptx::st_global_v4(dH + static_cast<int64_t>(tok) * ld + col, a, b, c, d);
    }
    ++box_count;
  }
}

// fp32 tile store or TMA reduce-add (dW): 8 boxes of 32 columns.
__device__ __forceinline__ void epi_f32_tile(const CUtensorMap* tm, bool reduce, uint32_t tcol, int x0, int yrow,
                                             uint32_t staging0, uint32_t& box_count, int lane) {
#pragma unroll 1
  for (int j = 0; j < BN / 32; ++j) {
    float v[32];
    tmem_load32_sync(tcol + j * 32, v);
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
    store_box(tm, reduce, staging0, box_count, lane, w, x0 + j * 32, yrow);
  }
}

// ----------------------------------------------------------------------------- work-index ring
// Dynamic schedule (MODE_DHW tiles, MODE_FWD / MODE_SCORE units): the even CTA's
// producer takes the next index from the launch's global counter, writes it into
// slot i % kTileRing of both CTAs' rings and arrives on both CTAs' tile_full
// barriers; the consumers (the even CTA's MMA thread, the odd CTA's producer and
// all eight epilogue warps) read their own ring and arrive on the even CTA's
// tile_empty barrier.  An index past the last one ends every role's loop.  The
// pairs then work on a contiguous window of the index order at any time, however
// their speeds differ, which keeps operand blocks they share in L2.
__device__ __forceinline__ uint32_t ring_addr(const SmemLayout& s, int slot) {
  return ptx::smem_u32(const_cast<int*>(s.tile_ring + slot));
}

// The even CTA's producer: claims the i-th index of this pair into *t.
__device__ __forceinline__ bool ring_claim(const GemmParams& p, const SmemLayout& s, int i, int* t) {
  const int slot = i % kTileRing;
  const uint32_t ph = static_cast<uint32_t>(i / kTileRing) & 1u;
  if (!ptx::wait_bounded_cluster(bar_tile_empty(s, slot), ph ^ 1u, p.timeout_ns, s.abort_flag)) {
    abort_cta(p, s);
    return false;
  }
  *t = atomicAdd(p.tile_counter, 1);
  s.tile_ring[slot] = *t;
  ptx::st_shared_cluster_u32(ptx::mapa(ring_addr(s, slot), 1), static_cast<uint32_t>(*t));
  ptx::mbar_arrive_cluster(ptx::mapa(bar_tile_full(s, slot), 0));
  ptx::mbar_arrive_cluster(ptx::mapa(bar_tile_full(s, slot), 1));
  return true;
}

// A consumer: reads the i-th index of this pair into *t and releases the slot
// (one arrival per calling thread, or per warp through lane 0 with `per_warp`).
__device__ __forceinline__ bool ring_take(const GemmParams& p, const SmemLayout& s, int i, int* t, bool per_warp,
                                          int lane) {
  const int slot = i % kTileRing;
  const uint32_t ph = static_cast<uint32_t>(i / kTileRing) & 1u;
  if (!ptx::wait_bounded_cluster(bar_tile_full(s, slot), ph, p.timeout_ns, s.abort_flag)) {
    abort_cta(p, s);
    return false;
  }
  *t = s.tile_ring[slot];
  if (per_warp) __syncwarp();
  if (!per_warp || lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(bar_tile_empty(s, slot), 0));
  return true;
}

// ----------------------------------------------------------------------------- MODE_FWD / MODE_DZ / MODE_SCORE loops
// Forward units (token pair x vocab range) come from the work-index ring; the
// dZ recompute's single-tile units are strided statically (pair c takes units
// c, c + pairs, c + 2 * pairs, ...).
template <int MODE>
__device__ __forceinline__ bool next_unit(const GemmParams& p, const SmemLayout& s, int i, int* u, int role,
                                          uint32_t rank, int lane) {
  if constexpr (is_forward(MODE)) {
    if (p.dynamic_units) {
      // role 0: producer, 1: MMA issuer, 2: epilogue warp
      if (role == 0 && rank == 0) return ring_claim(p, s, i, u);
      return ring_take(p, s, i, u, role == 2, lane);
    }
  }
  *u = static_cast<int>(blockIdx.x >> 1) + i * static_cast<int>(gridDim.x >> 1);
  return true;
}
template <int MODE>
__device__ __forceinline__ void producer_loop(const GemmParams& p, const Counts& c, const SmemLayout& s,
                                              uint32_t rank) {
  Ring ps;
  bool ok = true;
  for (int i = 0; ok; ++i) {
    int u;
    if (!next_unit<MODE>(p, s, i, &u, 0, rank, 0) || u >= c.num_units) break;
    const Unit un = decode_unit<MODE>(p, c, u, rank);
    for (int nb = un.n_lo; nb < un.n_hi && ok; ++nb)
      ok = produce_tile(p, s, ps, 0, un.m_blk, nb, p.num_k_blocks, rank);
  }
  producer_drain(s, ps, rank);
}

// Even CTA only.
template <int MODE>
__device__ __forceinline__ void mma_loop(const GemmParams& p, const Counts& c, const SmemLayout& s,
                                         uint32_t tmem_base) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(2 * BM, BN, 0, 0);
  Ring ring;
  uint32_t acc = 0, acc_phase = 0;
  bool ok = true;
  for (int i = 0; ok; ++i) {
    int u;
    if (!next_unit<MODE>(p, s, i, &u, 1, 0, 0) || u >= c.num_units) break;
    const Unit un = decode_unit<MODE>(p, c, u, 0);
    for (int nb = un.n_lo; nb < un.n_hi && ok; ++nb) {
      if (!ptx::wait_bounded_cluster(bar_tempty(s, acc), acc_phase ^ 1u, p.timeout_ns, s.abort_flag)) {
        abort_cta(p, s);
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      ok = mma_tile(p, s, tmem_base + acc * BN, p.num_k_blocks, 0, 0, idesc, ring);
      if (!ok) break;
      ptx::mma_commit_pair(bar_tfull(s, acc), 0x3);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  // Wait for every MMA issued so far before TMEM is freed.
  ptx::mma_commit_pair(bar_drain(s), 0x1);
  ptx::wait_bounded(bar_drain(s), 0, kDrainTimeoutNs, nullptr);
}

// Tells the even CTA that this warp has read its rows of accumulator `acc`.
__device__ __forceinline__ void release_accumulator(const SmemLayout& s, uint32_t acc, int lane) {
  ptx::tc_fence_before();
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(bar_tempty(s, acc), 0));
}

template <int MODE>
__device__ __forceinline__ void epilogue_loop(const GemmParams& p, const Counts& c, const SmemLayout& s,
                                              uint32_t tmem_base, int warp, int lane, uint32_t rank) {
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  const int row_in_tile = q * 32 + lane;
  const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  uint32_t acc = 0, acc_phase = 0;
  uint32_t box_count = 0;
  const uint32_t staging0 = ptx::smem_u32(s.staging + q * 2 * STAGING_BOX_BYTES);
  bool ok = true;

  for (int i = 0; ok; ++i) {
    int u;
    if (!next_unit<MODE>(p, s, i, &u, 2, rank, lane) || u >= c.num_units) break;
    const Unit un = decode_unit<MODE>(p, c, u, rank);
    const bool active = un.m_blk * BM < c.rows;       // the odd CTA of a ragged last pair has no rows
    const int t_local = un.m_blk * BM + row_in_tile;  // token within the launch

    float m_run = -INFINITY, s_run = 0.0f, zy = 0.0f;
    bool have_zy = false;
    int y = -1;
    float gt = 0.0f, lse2 = 0.0f;
    float best = -INFINITY;
    int best_col = -1;
    // y: the target's local vocab column when this launch's vocab rows own it, else -1
    if constexpr (is_forward(MODE)) {
      if (t_local < c.rows) {
        const int64_t target = p.targets[p.row_index ? p.row_index[t_local] : t_local];
        const int64_t yy = target - p.vocab_offset;
        if (target != p.ignore_index && yy >= 0 && yy < p.V) y = static_cast<int>(yy);
      }
    } else {
      if (t_local < c.rows) {
        const int t = p.row_index ? p.row_index[p.index0 + t_local] : p.row0 + t_local;
        gt = p.g[t];
        lse2 = p.lse[t] * kLog2e;
        const int64_t yy = p.targets[t] - p.vocab_offset;
        if (yy >= 0 && yy < p.V) y = static_cast<int>(yy);
      }
    }

    for (int nb = un.n_lo; nb < un.n_hi; ++nb) {
      if (!ptx::wait_bounded_cluster(bar_tfull(s, acc), acc_phase, p.timeout_ns, s.abort_flag)) {
        abort_cta(p, s);
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tcol = lane_addr + acc * BN;

      if (active) {
        if constexpr (is_forward(MODE)) {
          const int n0 = nb * BN;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_load32_sync(tcol + c * 32, v);
            const int col0 = n0 + c * 32;
            if (col0 + 32 > p.V) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j >= p.V) v[j] = -INFINITY;
            }
            const int yo = y - col0;
            if (static_cast<unsigned>(yo) < 32u) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j == yo) zy = v[j];
              have_zy = true;
            }
            float mx = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) mx = fmaxf(mx, v[j]);
            if constexpr (MODE == MODE_SCORE) {
              // strictly larger: equal values keep the earlier (lower) column
              if (mx > best) {
                int jj = 0;
#pragma unroll
                for (int j = 31; j >= 0; --j)
                  if (v[j] == mx) jj = j;
                best = mx;
                best_col = col0 + jj;
              }
            }
            const float m_new = fmaxf(m_run, mx * kLog2e);
            float acc_s = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) acc_s += ptx::ex2(fmaf(v[j], kLog2e, -m_new));
            s_run = s_run * ptx::ex2(m_run - m_new) + acc_s;
            m_run = m_new;
          }
        } else {
          epi_dz_tile(&p.tmOut, tcol, nb * BN, un.m_blk * BM + q * 32, staging0, box_count, lane, gt, lse2,
                              y, p.V);
        }
      }
      release_accumulator(s, acc, lane);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }

    if constexpr (is_forward(MODE)) {
      if (ok && t_local < c.rows) {
        p.partials[static_cast<size_t>(un.split) * p.part_stride + t_local] = make_float2(m_run, s_run);
        if (have_zy) p.zy[t_local] = zy;
        if constexpr (MODE == MODE_SCORE) {
          p.best_val[static_cast<size_t>(un.split) * p.part_stride + t_local] = best;
          p.best_idx[static_cast<size_t>(un.split) * p.part_stride + t_local] =
              static_cast<int32_t>(p.vocab_offset + best_col);
        }
      }
    }
  }
  if (lane == 0) ptx::bulk_wait<0>();
  __syncwarp();
}

// ----------------------------------------------------------------------------- MODE_DHW loops (dynamic schedule)

__device__ __forceinline__ void dhw_producer(const GemmParams& p, const Counts& c, const SmemLayout& s,
                                             uint32_t rank) {
  Ring ps;
  const int total = c.n_dh_tiles + p.n_dw_tiles;
  for (int i = 0;; ++i) {
    int t;
    if (!(rank == 0 ? ring_claim(p, s, i, &t) : ring_take(p, s, i, &t, false, 0))) break;
    if (t >= total) break;
    const Tile ti = decode_dhw(p, c, t, rank);
    // Wide dH tiles (all first in the tile order) use the ring cut in WIDE_NSTAGE
    // stages; the first dW tile after them re-cuts it, once per launch.
    if (!producer_recut(p, s, ps, ti.wide ? WIDE_NSTAGE : NSTAGE)) break;
    if (!produce_tile(p, s, ps, ti.wide ? 3 : 1 + ti.family, ti.m_blk, ti.nb, ti.num_k, rank)) break;
  }
  producer_drain(s, ps, rank);
}

// Even CTA only.
__device__ __forceinline__ void dhw_mma(const GemmParams& p, const Counts& c, const SmemLayout& s,
                                        uint32_t tmem_base) {
  constexpr uint32_t idesc_dh = ptx::idesc_bf16_f32(2 * BM, BN, 0, 1);
  constexpr uint32_t idesc_dw = ptx::idesc_bf16_f32(2 * BM, BN, 1, 1);
  const int total = c.n_dh_tiles + p.n_dw_tiles;
  Ring ring;
  // Accumulator uses so far: use n is buffer n % 2 with phase (n / 2) % 2.  A wide
  // dH tile takes two consecutive uses (both buffers), a 256-column tile one.
  uint32_t n_acc = 0;
  for (int i = 0;; ++i) {
    int t;
    if (!ring_take(p, s, i, &t, false, 0)) break;
    if (t >= total) break;
    const Tile ti = decode_dhw(p, c, t, 0);
    const int uses = ti.wide ? 2 : 1;
    bool ok = true;
    for (int h = 0; h < uses && ok; ++h) {
      const uint32_t n = n_acc + h;
      ok = ptx::wait_bounded_cluster(bar_tempty(s, n & 1u), ((n >> 1) & 1u) ^ 1u, p.timeout_ns, s.abort_flag);
    }
    if (!ok) {
      abort_cta(p, s);
      break;
    }
    ptx::tc_fence_after();
    mma_recut(ring, ti.wide ? WIDE_NSTAGE : NSTAGE);
    const uint32_t d0 = tmem_base + (n_acc & 1u) * BN;
    if (ti.wide) {
      const uint32_t d1 = tmem_base + ((n_acc + 1) & 1u) * BN;
      if (!mma_tile_wide(p, s, d0, d1, ti.num_k, idesc_dh, ring)) break;
    } else {
      if (!mma_tile(p, s, d0, ti.num_k, static_cast<uint32_t>(ti.family), 1u, ti.family ? idesc_dw : idesc_dh,
                    ring))
        break;
    }
    for (int h = 0; h < uses; ++h) ptx::mma_commit_pair(bar_tfull(s, (n_acc + h) & 1u), 0x3);
    n_acc += uses;
  }
  ptx::mma_commit_pair(bar_drain(s), 0x1);
  ptx::wait_bounded(bar_drain(s), 0, kDrainTimeoutNs, nullptr);
}

__device__ __forceinline__ void dhw_epilogue(const GemmParams& p, const Counts& c, const SmemLayout& s,
                                             uint32_t tmem_base, int warp, int lane, uint32_t rank) {
  const int q = warp & 3;
  const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  const uint32_t staging0 = ptx::smem_u32(s.staging + q * 2 * STAGING_BOX_BYTES);
  const int total = c.n_dh_tiles + p.n_dw_tiles;
  uint32_t n_acc = 0, box_count = 0;  // accumulator uses, as in dhw_mma
  for (int i = 0;; ++i) {
    int t;
    if (!ring_take(p, s, i, &t, true, lane)) break;
    if (t >= total) break;
    const Tile ti = decode_dhw(p, c, t, rank);
    const int uses = ti.wide ? 2 : 1;
    bool ok = true;
    // One 256-column accumulator at a time: a wide tile's second half is read
    // after its first half has been stored and released.
    for (int h = 0; h < uses && ok; ++h) {
      const uint32_t n = n_acc + h;
      if (!ptx::wait_bounded_cluster(bar_tfull(s, n & 1u), (n >> 1) & 1u, p.timeout_ns, s.abort_flag)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tcol = lane_addr + (n & 1u) * BN;
      if (ti.family == 0) {
        const int x0 = ti.wide ? ti.nb * 2 * BN + h * BN : ti.nb * BN;
        if (ti.m_blk * BM < c.rows) {
          const int r = ti.m_blk * BM + q * 32 + lane;  // row of the chunk
          const int token = r < c.rows ? (p.row_index ? p.row_index[p.index0 + r] : p.row0 + r) : -1;
          epi_dh_rows(p.dH_out, p.dH_ld, p.Hd, token, tcol, x0, staging0, box_count, lane);
        }
      } else {
        if (ti.m_blk * BM < p.V)
          epi_f32_tile(&p.tmOut2, p.reduce_out != 0, tcol, ti.nb * BN, ti.m_blk * BM + q * 32, staging0,
                       box_count, lane);
      }
      release_accumulator(s, n & 1u, lane);
    }
    if (!ok) {
      abort_cta(p, s);
      break;
    }
    n_acc += uses;
  }
  if (lane == 0) ptx::bulk_wait<0>();
  __syncwarp();
}

// ----------------------------------------------------------------------------- the GEMM kernel
template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const Counts c = counts_of<MODE>(p);
  if (p.rows_dev && c.rows == 0) {
    // An empty chunk of the row list: nothing to compute.  Every CTA sees the same
    // count and leaves before any barrier, TMEM or cluster operation.  When the
    // list is empty altogether, the first chunk's dW (stored, not added to) is zero.
    if constexpr (MODE == MODE_DHW) {
      if (!p.reduce_out && p.dW_zero) {
        const int64_t n4 = p.dW_elems / 4;
        float4* d4 = reinterpret_cast<float4*>(p.dW_zero);
        const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride)
          d4[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int64_t i = n4 * 4 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.dW_elems;
             i += stride)
          p.dW_zero[i] = 0.0f;
      }
    }
    return;
  }
  const SmemLayout s = carve_smem<MODE>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      ptx::mbar_init(bar_full(s, i), 1);
      ptx::mbar_init(bar_empty(s, i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar_tfull(s, i), 1);
      ptx::mbar_init(bar_tempty(s, i), 2 * kEpiWarps);
    }
    ptx::mbar_init(bar_drain(s), 1);
    for (int i = 0; i < kTileRing; ++i) {
      ptx::mbar_init(bar_tile_full(s, i), 1);
      ptx::mbar_init(bar_tile_empty(s, i), 2 + 2 * kEpiWarps);
    }
    *s.abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&p.tmA);
    ptx::prefetch_tmap(&p.tmB);
    if (MODE == MODE_DZ) ptx::prefetch_tmap(&p.tmOut);
    if (MODE == MODE_DHW) {
      ptx::prefetch_tmap(&p.tmA2);
      ptx::prefetch_tmap(&p.tmB2);
      ptx::prefetch_tmap(&p.tmOut2);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(s.tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  // Both CTAs' barriers are initialised and their TMEM allocated before any
  // cross-CTA signal.
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *s.tmem_slot;

  if (warp == 0) {
    if (ptx::elect_one()) {
      if constexpr (MODE == MODE_DHW)
        dhw_producer(p, c, s, rank);
      else
        producer_loop<MODE>(p, c, s, rank);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0 && ptx::elect_one()) {
      if constexpr (MODE == MODE_DHW)
        dhw_mma(p, c, s, tmem_base);
      else
        mma_loop<MODE>(p, c, s, tmem_base);
    }
    __syncwarp();
  } else {
    if constexpr (MODE == MODE_DHW)
      dhw_epilogue(p, c, s, tmem_base, warp, lane, rank);
    else
      epilogue_loop<MODE>(p, c, s, tmem_base, warp, lane, rank);
  }

  // After an abort the odd CTA's loads may not have been consumed (they are
  // counted on the even CTA's barriers): give any TMA write still in flight
  // time to land before shared memory is released.
  if (warp == 0 && *s.abort_flag) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < kAbortSettleNs) {
    }
  }
  // No CTA leaves while its peer may still signal its barriers or use the
  // pair's TMEM.
  ptx::tc_fence_before();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ----------------------------------------------------------------------------- forward finalize
// Per row: merge the vocab-range partials in split order into lse, then
// loss_t = lse - z_y and logp_t = z_y - lse on valid rows.  Each block also
// writes the fixed-order sum of its rows' losses and its count of valid rows.
constexpr int kFinalizeThreads = 256;

struct FinalizeParams {
  const float2* partials;
  const float* zy;
  const int64_t* targets;
  float* lse;
  float* logp;
  float* loss_rows;      // [T] when reduction is NONE, else nullptr
  double* block_sum;     // [num_blocks]
  int64_t* block_count;  // [num_blocks]
  int32_t* status;
  const int32_t* pos;    // row-list position of each token, -1 when not listed; nullptr: position t
  int64_t ignore_index;
  int32_t T;
  int32_t V;
  int32_t n_split;
  int32_t part_stride;
};

__global__ void __launch_bounds__(kFinalizeThreads) fwd_finalize_kernel(const FinalizeParams p) {
  __shared__ double sh_sum[kFinalizeThreads];
  __shared__ long long sh_cnt[kFinalizeThreads];
  const int t = blockIdx.x * kFinalizeThreads + threadIdx.x;
  double my_loss = 0.0;
  long long my_cnt = 0;
  const int i = (t < p.T && p.pos) ? p.pos[t] : t;  // the row's slot in the partials
  if (t < p.T && i < 0) {
    // not listed (an ignored target): nothing was computed for the row
    p.lse[t] = 0.0f;
    p.logp[t] = 0.0f;
    if (p.loss_rows) p.loss_rows[t] = 0.0f;
  } else if (t < p.T) {
    float M = -INFINITY;
    for (int sp = 0; sp < p.n_split; ++sp) M = fmaxf(M, p.partials[static_cast<size_t>(sp) * p.part_stride + i].x);
    float S = 0.0f;
    for (int sp = 0; sp < p.n_split; ++sp) {
      const float2 pr = p.partials[static_cast<size_t>(sp) * p.part_stride + i];
      S += pr.y * exp2f(pr.x - M);
    }
    const float lse = (M + log2f(S)) * kLn2;
    const int64_t y = p.targets[t];
    bool valid = y != p.ignore_index;
    if (valid && (y < 0 || y >= p.V)) {
      raise_status(p.status, kStatusTargetRange);
      valid = false;
    }
    float loss_t = 0.0f, logp_t = 0.0f;
    if (valid) {
      const float z = p.zy[i];
      loss_t = lse - z;
      logp_t = z - lse;
      my_loss = static_cast<double>(loss_t);
      my_cnt = 1;
    }
    p.lse[t] = lse;
    p.logp[t] = logp_t;
    if (p.loss_rows) p.loss_rows[t] = loss_t;
  }
  sh_sum[threadIdx.x] = my_loss;
  sh_cnt[threadIdx.x] = my_cnt;
  __syncthreads();
  for (int w = kFinalizeThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      sh_sum[threadIdx.x] += sh_sum[threadIdx.x + w];
      sh_cnt[threadIdx.x] += sh_cnt[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.block_sum[blockIdx.x] = sh_sum[0];
    p.block_count[blockIdx.x] = sh_cnt[0];
  }
}

// Scoring: per row, lse and logp as fwd_finalize_kernel (no loss reduction)
// and the argmax merged over the vocab ranges in order (lowest id on ties).
__global__ void __launch_bounds__(kFinalizeThreads) score_finalize_kernel(
    const float2* partials, const float* zy, const float* best_val, const int32_t* best_idx, const int64_t* targets,
    int T, int V, int64_t ignore_index, int n_split, int part_stride, float* lse_out, float* logp_out,
    int64_t* argmax_out, int32_t* status, const int32_t* pos) {
  const int t = blockIdx.x * kFinalizeThreads + threadIdx.x;
  if (t >= T) return;
  const int r = pos ? pos[t] : t;  // the row's slot in the partials; < 0: not listed, nothing computed
  if (r < 0) {
    if (lse_out) lse_out[t] = 0.0f;
    logp_out[t] = 0.0f;
    if (argmax_out) argmax_out[t] = -1;
    return;
  }
  float M = -INFINITY;
  for (int sp = 0; sp < n_split; ++sp) M = fmaxf(M, partials[static_cast<size_t>(sp) * part_stride + r].x);
  float S = 0.0f;
  float bv = -INFINITY;
  int32_t bi = 0;
  for (int sp = 0; sp < n_split; ++sp) {
    const size_t i = static_cast<size_t>(sp) * part_stride + r;
    const float2 pr = partials[i];
    S += pr.y * exp2f(pr.x - M);
    if (best_val[i] > bv) {
      bv = best_val[i];
      bi = best_idx[i];
    }
  }
  const float lse = (M + log2f(S)) * kLn2;
  const int64_t y = targets[t];
  bool valid = y != ignore_index;
  if (valid && (y < 0 || y >= V)) {
    raise_status(status, kStatusTargetRange);
    valid = false;
  }
  if (lse_out) lse_out[t] = lse;
  logp_out[t] = valid ? zy[r] - lse : 0.0f;
  if (argmax_out) argmax_out[t] = bi;
}

// Vocab shard forward: per row, merge the shard's split partials into the
// shard's log-sum-exp and report the target logit when the shard owns the target.
__global__ void __launch_bounds__(kFinalizeThreads) fwd_shard_finalize_kernel(
    const float2* partials, const float* zy, const int64_t* targets, int T, int64_t vocab_offset, int V_shard,
    int n_split, int part_stride, float* shard_lse, float* shard_zy) {
  const int t = blockIdx.x * kFinalizeThreads + threadIdx.x;
  if (t >= T) return;
  float M = -INFINITY;
  for (int sp = 0; sp < n_split; ++sp) M = fmaxf(M, partials[static_cast<size_t>(sp) * part_stride + t].x);
  float S = 0.0f;
  for (int sp = 0; sp < n_split; ++sp) {
    const float2 pr = partials[static_cast<size_t>(sp) * part_stride + t];
    S += pr.y * exp2f(pr.x - M);
  }
  const int64_t yy = targets[t] - vocab_offset;
  shard_lse[t] = (M + log2f(S)) * kLn2;
  shard_zy[t] = (yy >= 0 && yy < V_shard) ? zy[t] : 0.0f;
}

// Cross-shard combine, step 1: shard r's log-sum-exp becomes the partial
// (lse_r * log2e, 1) of split r, and the target logits are summed in shard
// order (only the owning shard reports a non-zero one).  fwd_finalize_kernel
// then merges the partials exactly as it merges the vocab ranges of one launch.
__global__ void __launch_bounds__(kFinalizeThreads) combine_shards_kernel(const float* shard_lse,
                                                                         const float* shard_zy, int n_shards, int T,
                                                                         float2* partials, int part_stride,
                                                                         float* zy) {
  const int t = blockIdx.x * kFinalizeThreads + threadIdx.x;
  if (t >= T) return;
  float z = 0.0f;
  for (int r = 0; r < n_shards; ++r) {
    partials[static_cast<size_t>(r) * part_stride + t] =
        make_float2(shard_lse[static_cast<size_t>(r) * T + t] * kLog2e, 1.0f);
    z += shard_zy[static_cast<size_t>(r) * T + t];
  }
  zy[t] = z;
}

// One block: fixed-order sum of the block partials into the scalar loss and n_valid.
constexpr int kReduceThreads = 1024;

__global__ void __launch_bounds__(kReduceThreads) fwd_reduce_kernel(const double* block_sum, const int64_t* block_count,
                                                                    int num_blocks, int reduction, float* loss,
                                                                    int64_t* n_valid) {
  __shared__ double sh_sum[kReduceThreads];
  __shared__ long long sh_cnt[kReduceThreads];
  double a = 0.0;
  long long c = 0;
  for (int i = threadIdx.x; i < num_blocks; i += kReduceThreads) {
    a += block_sum[i];
    c += block_count[i];
  }
  sh_sum[threadIdx.x] = a;
  sh_cnt[threadIdx.x] = c;
  __syncthreads();
  for (int w = kReduceThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      sh_sum[threadIdx.x] += sh_sum[threadIdx.x + w];
      sh_cnt[threadIdx.x] += sh_cnt[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double total = sh_sum[0];
    const long long n = sh_cnt[0];
    if (reduction == 1) loss[0] = n > 0 ? static_cast<float>(total / static_cast<double>(n)) : 0.0f;
    if (reduction == 2) loss[0] = static_cast<float>(total);
    if (n_valid) n_valid[0] = n;
  }
}

// ----------------------------------------------------------------------------- backward prep
// One block: count valid rows (fixed-order tree), flag out-of-range targets,
// then write the per-token upstream weight g_t.  dloss may be null (no loss
// gradient); dlogp, when given, is a gradient on the logp output, and since
// logp_t = -loss_t on valid rows it enters g_t with a minus sign.
__global__ void __launch_bounds__(kReduceThreads) bwd_prep_kernel(const float* dloss, const float* dlogp,
                                                                  const int64_t* targets, int T, int V,
                                                                  int64_t ignore_index, int reduction, float* g,
                                                                  int32_t* row_index, int32_t* row_count,
                                                                  int32_t* status) {
  __shared__ long long sh_cnt[kReduceThreads];
  long long c = 0;
  bool bad = false;
  for (int t = threadIdx.x; t < T; t += kReduceThreads) {
    const int64_t y = targets[t];
    if (y != ignore_index) {
      if (y >= 0 && y < V)
        ++c;
      else
        bad = true;
    }
  }
  if (bad) raise_status(status, kStatusTargetRange);
  sh_cnt[threadIdx.x] = c;
  __syncthreads();
  for (int w = kReduceThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh_cnt[threadIdx.x] += sh_cnt[threadIdx.x + w];
    __syncthreads();
  }
  const long long n = sh_cnt[0];
  __syncthreads();
  const float d0 = dloss ? dloss[0] : 0.0f;
  const float scalar = (reduction == 1) ? (n > 0 ? d0 / static_cast<float>(n) : 0.0f) : (reduction == 2 ? d0 : 0.0f);
  // g_t, and the list of the rows whose g_t is not zero (their dZ rows are the only
  // non-zero ones) in token order: rounds of kReduceThreads consecutive tokens, each
  // placed by a ballot within its warp and a scan of the 32 warp counts.
  static_assert(kReduceThreads == 1024, "one warp scans the 32 warp counts");
  __shared__ int warp_off[kReduceThreads / 32];
  __shared__ int round_total;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  int base = 0;
  for (int r0 = 0; r0 < T; r0 += kReduceThreads) {
    const int t = r0 + static_cast<int>(threadIdx.x);
    float gt = 0.0f;
    if (t < T) {
      const int64_t y = targets[t];
      const bool valid = (y != ignore_index) && y >= 0 && y < V;
      gt = reduction == 0 ? (dloss ? dloss[t] : 0.0f) : scalar;
      if (dlogp) gt -= dlogp[t];
      gt = valid ? gt : 0.0f;
      g[t] = gt;
    }
    const bool keep = t < T && gt != 0.0f;
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) warp_off[warp] = __popc(m);
    __syncthreads();
    if (warp == 0) {
      const int v = warp_off[lane];
      int inc = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
      }
      warp_off[lane] = inc - v;
      if (lane == 31) round_total = inc;
    }
    __syncthreads();
    if (keep) row_index[base + warp_off[warp] + __popc(m & ((1u << lane) - 1u))] = t;
    base += round_total;
    __syncthreads();  // warp_off and round_total are rewritten by the next round
  }
  if (threadIdx.x == 0) *row_count = base;
}

// The list of rows with a valid target, in token order, for flce_forward_valid:
// row_index[position] = token, pos[token] = position or -1, *row_count = length.
// Rounds of kReduceThreads tokens, placed by warp ballots and a scan of the
// warp counts.  A target outside [0, V) that is not ignore_index is flagged
// and the row left out.
__global__ void __launch_bounds__(kReduceThreads) fwd_list_kernel(const int64_t* targets, int T, int V,
                                                                  int64_t ignore_index, int32_t* row_index,
                                                                  int32_t* pos, int32_t* row_count,
                                                                  int32_t* status) {
  static_assert(kReduceThreads == 1024, "one warp scans the 32 warp counts");
  __shared__ int warp_off[kReduceThreads / 32];
  __shared__ int round_total;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  int base = 0;
  bool bad = false;
  for (int r0 = 0; r0 < T; r0 += kReduceThreads) {
    const int t = r0 + static_cast<int>(threadIdx.x);
    bool keep = false;
    if (t < T) {
      const int64_t y = targets[t];
      if (y != ignore_index) {
        keep = y >= 0 && y < V;
        bad = bad || !keep;
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) warp_off[warp] = __popc(m);
    __syncthreads();
    if (warp == 0) {
      const int v = warp_off[lane];
      int inc = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
      }
      warp_off[lane] = inc - v;
      if (lane == 31) round_total = inc;
    }
    __syncthreads();
    if (t < T) {
      const int at = base + warp_off[warp] + __popc(m & ((1u << lane) - 1u));
      pos[t] = keep ? at : -1;
      if (keep) row_index[at] = t;
    }
    base += round_total;
    __syncthreads();
  }
  if (bad) raise_status(status, kStatusTargetRange);
  if (threadIdx.x == 0) *row_count = base;
}

// Rows list positions index0 .. index0 + rows - 1 of H, gathered into the chunk
// buffer Hc, 16 bytes at a time; Hc rows rows .. min(cap, round_up(rows, 256)) - 1
// (read by the chunk's last tile pair, and as the K tail of its dW tiles) are zeroed.
constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) gather_rows_kernel(const uint4* H, const int32_t* row_index,
                                                                   const int32_t* row_count, int index0, int cap,
                                                                   int row_vecs, uint4* Hc) {
  const int rows = min(max(*row_count - index0, 0), cap);
  const int fill = min(cap, (rows + 2 * BM - 1) / (2 * BM) * (2 * BM));
  const int64_t n = static_cast<int64_t>(fill) * row_vecs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < n; v += stride) {
    const int i = static_cast<int>(v / row_vecs);
    const int j = static_cast<int>(v - static_cast<int64_t>(i) * row_vecs);
    Hc[v] = i < rows ? H[static_cast<int64_t>(row_index[index0 + i]) * row_vecs + j] : make_uint4(0, 0, 0, 0);
  }
}

// ----------------------------------------------------------------------------- self-test of the bounded wait
// One thread waits, with the same bounded wait the GEMMs use, on an mbarrier
// that nothing arrives on, and records FLCE_ERR_TIMEOUT in the status word
// when the limit runs out (and 0 if the wait ever succeeded, which it cannot).
__global__ void wait_selftest_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = ptx::smem_u32(&bar);
  ptx::mbar_init(b, 1);
  ptx::fence_barrier_init();
  const bool ok = ptx::wait_bounded(b, 0, timeout_ns, nullptr);
  *status = ok ? 0 : kStatusTimeout;
}

}  // namespace flce
