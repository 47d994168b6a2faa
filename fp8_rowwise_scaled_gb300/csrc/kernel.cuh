// kernel.cuh -- persistent, warp-specialised FP8 rowwise-scaled grouped GEMM for sm_103a.
//
// Operation (MSLK #471 "Back the FP8 rowwise grouped GEMM ops with FlyDSL on ROCm",
// commit introducing the rowwise scaling scheme): for every row r of group g,
//   out[r, n] = bf16_rne((acc[r, n] * scale_a[r]) * scale_b[g, n]),
//   acc[r, n] = sum_k A[r, k] * B[g, n, k]   (e4m3 x e4m3, fp32 accumulator in TMEM)
// The K loop accumulates unscaled; the two scales are applied once, in the epilogue,
// on the fp32 accumulator (never rounded before that).
//
// CTA organisation (one CTA per SM, persistent over output tiles):
//   loader warp(s)   TMA (one elected thread) or cp.async (4 warps) fill an S-stage
//                    ring of 128-byte-swizzled shared-memory tiles (full/empty mbarriers)
//   MMA warp         allocates TMEM; one thread issues tcgen05.mma (K = 32 per
//                    instruction, 4 per 128-byte stage) into a ring of 2-8 TMEM
//                    accumulator buffers (kNumAcc), and tcgen05.commit releases stages
//                    and buffers
//   prefetch warp    (swap-AB plans) asks L2 for the CTA's first weight tiles while the
//                    kernel before it on the stream finishes
//   4/8 epilogue     tcgen05.ld the accumulator, scale, convert to bf16, store with
//   warps            row / column predicates; padding rows get +0.0
//
// Group/tile scheduler (MSLK #471, commits on the packed and padded layouts and on the
// group resolution step): each CTA reads the [G] metadata once, prefix-sums it in shared
// memory, and enumerates output tiles over groups that have rows, so an empty group
// generates no tile.  Within a group tiles run n-major (all m-tiles of one weight
// n-tile are consecutive), so concurrently running CTAs share a weight tile in L2.
//
// Tile shapes:
//   normal  (kSwap = false): MMA M = 128 activation rows, MMA N = kTileN weight rows.
//   swap-AB (kSwap = true) : MMA M = 128 weight rows, MMA N = kTileN activation rows;
//                            for few rows per group the weights fill the 128-row side.
//   CTA pair (kPair = true): a cluster of two CTAs on two SMs computes a 256 x 256 tile
//                            with one cta_group::2 MMA of M = 256 issued by the leader
//                            (rank 0).  Each CTA loads its own 128 activation rows and
//                            half of the 256 weight rows per K block -- 32 KB instead of
//                            the 48 KB a 128 x 256 tile needs per SM -- and its TMEM gets
//                            the 128 x 256 accumulator of its own rows.  Both CTAs' loads
//                            complete on the leader's full barrier; the leader's commits
//                            arrive on both CTAs' barriers; both epilogues arrive on the
//                            leader's accumulator-empty barrier.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace mslkb {

constexpr int kMaxGroups = 1024;
constexpr int kBK = 128;  // bytes (= e4m3 elements) of K per pipeline stage
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusClamped = 2u;
constexpr uint32_t kStatusBadSlice = 4u;  // ragged K: a slice bound not on 16 elements
constexpr uint32_t kStatusBounds = 8u;    // checked builds: an index outside its buffer

struct GemmParams {
  const uint8_t* A;        // [rows, K] e4m3
  const uint8_t* B;        // [G, N, K] e4m3
  const float* scale_a;    // [rows]
  const float* scale_b;    // [G, N]
  const int64_t* meta;     // [G] m_sizes (stacked), zero_start_index_M (dynamic), or int32
                           // inclusive offsets (offsets layout; ragged N / K over N / K)
  uint16_t* out;           // [rows, N] bf16 bits
  uint32_t* status;        // device status word
  int32_t rows;            // rows of A: total_M (stacked), G * E (dynamic, ragged N), M
                           // (ragged K)
  int32_t G;
  int32_t N;               // columns of the output (total_N for ragged N)
  int32_t K;               // row length of A and B (total_K for ragged K)
  int32_t E;               // slab height: expected_m (dynamic), M (ragged N / K)
  int32_t num_kb;          // ceil(K / 128)
  int32_t copy_width;      // cp.async loader: bytes per copy (16, 8, 4) or 1 (byte loads)
  int32_t meta_kind;       // stacked: 0 int64 m_sizes, 1 int32 inclusive offsets;
                           // dynamic: 0 int64 zero_start_index_M, 2 none (full slabs)
  int32_t kb_per_chunk;    // K blocks the tensor core sums before the epilogue takes over
  int32_t split_k;         // 1: split the last waves' tiles along K over all CTAs
  float* sk_ws;            // split tiles: fp32 partial sums, 2 slots per CTA
  uint32_t* sk_cnt;        // split tiles: arrival counters, one per (tile, epilogue warp)
  uint64_t timeout_ns;     // give-up time of one pipeline wait
  int32_t test_stall;      // test hook: CTA 0 (CTA pairs: the first pair) withholds its
                           // first stage (TMA kernels), so the MMA wait runs out and the
                           // timeout path runs
  int32_t w_pair;          // swap-AB: 1 when the weight map of two K blocks per box (the
                           // kernel's tmB2) is valid, i.e. K is a multiple of 128
  int32_t prefetch_kb;     // swap-AB: K blocks of weights each CTA asks L2 to prefetch
                           // before the dependency wait (0: none)
  const int64_t* spec_meta;  // metadata the speculative schedule reads (= meta, unless a
                             // test points it elsewhere)
  uint32_t* tile_ctr;      // CTA pairs: {tiles claimed, leaders finished}, zero between
                           // calls (the last leader to finish resets both); null: every
                           // pair takes its tiles in a fixed stride
};

template <int kTileN_, int kStages_, bool kSwap_, bool kTma_, bool kDynamic_, int kEpiWarps_ = 4,
          bool kPair_ = false, int kRagged_ = 0, bool kBlockScale_ = false>
struct KernelCfg {
  static constexpr int kTileN = kTileN_;     // MMA N
  static constexpr int kStages = kStages_;
  static constexpr bool kSwap = kSwap_;
  static constexpr bool kTma = kTma_;
  static constexpr bool kDynamic = kDynamic_;
  // CTA pair (cluster of two, cta_group::2): the leader CTA issues one MMA of M = 256
  // rows whose A rows and B (weight) rows are split in halves over the two CTAs' shared
  // memory; each CTA's TMEM receives the 128 x kTileN accumulator of its own rows.  Each
  // SM then loads half of the weight tile per K block instead of all of it.
  static constexpr bool kPair = kPair_;
  static constexpr int kCtas = kPair ? 2 : 1;
  // Ragged layouts (MSLK #471, grouped-mm commits): 1 = groups partition N (A [G, M, K],
  // B [total_N, K], out [M, total_N]); 2 = groups slice K (A [M, total_K], B [N, total_K],
  // out [G, M, N]).  Group ranges come from int32 inclusive offsets.
  static constexpr bool kRagN = kRagged_ == 1;
  static constexpr bool kRagK = kRagged_ == 2;
  static constexpr bool kRagged = kRagged_ != 0;
  // Block scaling (groupwise; MSLK #471, commit introducing the rowwise scheme beside the
  // block scheme), stacked or slab (dynamic, batched) layouts: scale_a [rows of A, K/128],
  // scale_b [G, N/128, K/128]; every K block's
  // partial sum is scaled on its way from TMEM into the fp32 registers (one K block per
  // TMEM chunk), and the epilogue applies no further scale.
  static constexpr bool kBlockScale = kBlockScale_;
  static constexpr int kScaleBlock = 128;
  static constexpr int kMmaM = 128;                           // accumulator rows per CTA
  static constexpr int kActRows = kSwap ? kTileN : kMmaM;     // activation rows per CTA
  static constexpr int kWRows = kSwap ? kMmaM : kTileN / kCtas;  // weight rows per CTA
  static constexpr int kTileAct = kActRows * kCtas;  // activation rows per output tile
  static constexpr int kTileW = kWRows * kCtas;      // weight rows (columns) per output tile
  static constexpr int kActBytes = kActRows * kBK;
  static constexpr int kWBytes = kWRows * kBK;
  static constexpr int kStageBytes = kActBytes + kWBytes;  // one CTA's bytes per stage
  static constexpr int kLoaderWarps = kTma ? 1 : 4;
  static constexpr int kLoaderThreads = 32 * kLoaderWarps;
  static constexpr int kMmaWarp = kLoaderWarps;
  static constexpr int kEpiWarps = kEpiWarps_;            // 4, or 8 (two per TMEM quadrant)
  // Register split (128 x 256 tiles fed by TMA, 128 accumulator columns per thread):
  // warpgroup 0 = TMA warp, MMA warp and two idle warps, dropping to kRegsLow; the 8
  // epilogue warps (warpgroups 1-2) rise to kRegsHigh, enough for 128 fp32 accumulators
  // plus 64 columns of TMEM loads in flight.
  // Budget: launched with 384 x 168 registers = 128 x 40 + 256 x 232; per SM sub-partition
  // one warpgroup-0 warp and two epilogue warps: (40 + 232 + 232) x 32 <= 16384.
  static constexpr bool kRegSplit = kTma && !kSwap && kEpiWarps == 8 && kTileN == 256;
  // Swap-AB plans (weight streaming) carry one more warp, which prefetches the CTA's first
  // weight tiles into L2 while the kernel before it on the stream finishes (below)
  static constexpr bool kSpecWarp = kSwap && kTma && !kRagged;
  static constexpr int kIdleWarps = kRegSplit ? 2 : (kSpecWarp ? 1 : 0);
  static constexpr int kSpecWarpIdx = kLoaderWarps + 1;
  // Ragged K: one of the register split's spare warps takes each loaded stage and zeroes
  // the bytes of its tiles that lie outside the tile's K slice (the first block is loaded
  // from the 128-byte boundary below the slice start, the last runs past its end), then
  // hands the stage to the MMA thread through a barrier of its own, so that the MMA thread
  // issues whole blocks only
  static constexpr bool kEdgeWarp = kRagK && kRegSplit;
  static constexpr int kEdgeWarpIdx = kLoaderWarps + 1;
  static constexpr int kEpiWarp0 = kLoaderWarps + 1 + kIdleWarps;
  static constexpr int kThreads = 32 * (kLoaderWarps + 1 + kIdleWarps + kEpiWarps);
  static constexpr int kLaunchRegs = kRegSplit ? 168 : 0;  // required at launch (0: any)
  static constexpr int kRegsLow = 40;
  static constexpr int kRegsHigh = 232;
  // accumulator columns one epilogue thread owns (and keeps in fp32 registers)
  static constexpr int kThreadCols = kSwap ? kTileN : kTileN / (kEpiWarps / 4);
  static constexpr int kAccCols = kTileN;  // fp32 TMEM columns of one accumulator
  // K blocks per chunk under block scaling, each summed into an accumulator of its own (so
  // that each gets its own scales): the swap-AB tiles put two side by side in a chunk
  // buffer and so commit and hand over once per two blocks; 128-row tiles fill TMEM with
  // one.  Without block scaling a chunk buffer is one accumulator summing
  // GemmParams::kb_per_chunk blocks.
  static constexpr int kBSSub = (kBlockScale && kSwap) ? 2 : 1;
  static constexpr int kBufCols = kAccCols * kBSSub;  // fp32 TMEM columns of a chunk buffer
  // TMEM chunk buffers the MMA can run ahead of the epilogue by: two for 256-column
  // buffers (all 512 columns), more for narrower ones (up to 8: the swap-AB tiles, which
  // under block scaling hand over a buffer every one or two K blocks and need the slack)
  static constexpr int kNumAcc = (kBufCols >= 256) ? 2 : (kBufCols >= 128) ? 4 : 8;
  static constexpr int kTmemCols = (kNumAcc * kBufCols <= 32)    ? 32
                                   : (kNumAcc * kBufCols <= 64)  ? 64
                                   : (kNumAcc * kBufCols <= 128) ? 128
                                   : (kNumAcc * kBufCols <= 256) ? 256
                                                                 : 512;
  static constexpr int kCpLag = kStages - 2;  // cp.async groups kept in flight per thread
  static constexpr uint32_t kIdesc = ptx::idesc_e4m3_f32(kMmaM * kCtas, kTileN);
  // CTA pairs, a group's last <= 128 rows: the tile transposed, the weights as the M = 256
  // operand (each CTA's 128 weight rows, as in a whole tile) and the tile's rows, rounded
  // up to 16, as N (half of them in each CTA).  Each CTA's accumulator holds its 128 output
  // columns (TMEM lanes) x the tile's rows (TMEM columns): the tensor core computes the
  // remainder's rows only, not 128 (at the power cap the time follows the MACs computed).

  // 128-row tiles write the output through shared memory and TMA stores: each epilogue
  // warp stages 32 rows x 32 columns of bf16 (2 KB, 64-byte swizzle) at a time
  static constexpr bool kTmaStore = !kSwap;
  static constexpr int kStageOutBytes = 32 * 32 * 2;

  // shared memory layout, from a 1024-byte aligned base
  static constexpr int kOffAct = 0;
  static constexpr int kOffW = kStages * kActBytes;
  static constexpr int kOffOut = kOffW + kStages * kWBytes;
  static constexpr int kOffBar = kOffOut + (kTmaStore ? kEpiWarps * kStageOutBytes : 0);
  // CTA pairs: a ring of tile numbers that the leader's loader claims from a global
  // counter and hands to the pair's other roles (slots, then a full and an empty barrier
  // per slot)
  static constexpr int kTQ = kPair ? 4 : 0;
  static constexpr int kNumBars = 2 * kStages + 2 * kNumAcc + 2 * kTQ + (kEdgeWarp ? kStages : 0);
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem address, abort flag
  static constexpr int kOffWork = kOffMisc + 16;           // the CTA's Work (below)
  static constexpr int kOffTQ = kOffWork + 64;             // the tile ring (pairs)
  static constexpr int kOffSched = kOffTQ + 16;
  static constexpr int kSchedBytes = 2 * 4 * (kMaxGroups + 1);
  static constexpr int kOffSpec = kOffSched + kSchedBytes;  // the prefetch warp's tables
  static constexpr int kSmemBytes =
      kOffSpec + (kSpecWarp ? kSchedBytes : 0) + 1024;  // + alignment slack

  static_assert(kTileN % 16 == 0 && kTileN >= 16 && kTileN <= 256, "MMA N for M = 128");
  static_assert(kActBytes % 1024 == 0 && kWBytes % 1024 == 0, "swizzle atoms");
  static_assert(kStages >= 3, "pipeline depth");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kNumAcc * kBufCols <= 512, "the accumulators must fit TMEM");
  static_assert(kEpiWarps == 4 || (kEpiWarps == 8 && !kSwap), "epilogue warp split");
  static_assert(!kPair || (kTma && !kSwap && kTileN == 256 && kActBytes == kWBytes),
                "CTA pairs: 256 x 256 tiles, TMA (operand tiles of one size: a transposed "
                "tile swaps their descriptors)");
  static_assert(!kRagged || (kTma && !kPair && !kDynamic), "ragged layouts: TMA, single CTAs");
  static_assert(!kBlockScale || (kTma && !kPair && !kRagged && kBK == kScaleBlock &&
                                 (!kSwap || kTileN <= 32)),
                "block scaling: stacked or slab TMA tiles (swap-AB up to 32 rows), one K block "
                "per scale block");
  static_assert(kThreadCols % 16 == 0, "TMEM load granularity");
  static_assert(!kRegSplit || (kThreads == 384 && kEpiWarp0 == 4 &&
                               128 * kRegsLow + 256 * kRegsHigh == kThreads * kLaunchRegs),
                "register split budget");
};

struct TileCoord {
  int32_t g;          // group
  int32_t m0;         // first activation row of this CTA (global row index)
  int32_t n0;         // first weight row / output column
  int32_t valid_end;  // rows < valid_end get the product
  int32_t zero_end;   // rows in [valid_end, zero_end) get +0.0 (padding)
  bool half;          // CTA pairs: a group's last <= 128 rows, run as a transposed tile
                      // (m0 is then the tile's first row in both CTAs)
  int32_t tr_n;       // ... its rows rounded up to 16: the MMA's N, half of them per CTA
  int32_t orow_delta; // output row = A row + orow_delta
  int32_t srow_delta; // scale_a index = A row + srow_delta
  int32_t n_begin;    // columns in [n_begin, n_end) belong to the tile's group
  int32_t n_end;
  int32_t bz;         // third coordinate of the weight tensor map
  int32_t sb_off;     // scale_b index of column 0 of the group
  int32_t k0;         // first K element of the contraction
  int32_t k_len;      // K elements of the contraction
  int32_t k_skip;     // ragged K: elements of the first K block before the slice starts
  int32_t nkb;        // K blocks of the contraction
};

// CTA pairs: a group's rows run in 256-row tiles, except that a last piece of at most 128
// rows runs as a 128-row tile (64 rows per CTA), so short remainders cost half a tile.
// Rows [0, cover) of a group of `cnt` rows lie inside its tiles.
template <class Cfg>
__device__ __forceinline__ int32_t tile_cover(int32_t cnt) {
  const int32_t full = (cnt + Cfg::kTileAct - 1) / Cfg::kTileAct * Cfg::kTileAct;
  if constexpr (Cfg::kPair) {
    const int32_t rem = cnt % Cfg::kTileAct;
    if (rem > 0 && rem <= Cfg::kTileAct / 2) return full - Cfg::kTileAct / 2;
  }
  return full;
}

// Shared-memory scheduler tables.
//   rowinfo[g]: stacked -> first row of group g (G + 1 entries, clamped prefix);
//               dynamic -> valid rows v_g of slab g;
//               ragged N / K -> first column / first K element of group g (G + 1 entries).
//   tile_pre[g]: exclusive prefix of output tiles over groups (G + 1 entries).
struct Sched {
  const int32_t* rowinfo;
  const int32_t* tile_pre;
  int32_t G;
  int32_t E;
  int32_t n_tiles_n;
  int32_t total;
  int32_t N;
  int32_t K;
  int32_t num_kb;
};

// Output tiles of group g (ntn: weight tiles across N).
template <class Cfg>
__device__ __forceinline__ int64_t group_tiles(const int32_t* rowinfo, int32_t g, int32_t E,
                                               int64_t ntn) {
  if constexpr (Cfg::kRagN) {
    // every slab row, over the group's own columns; the group's tiles start on the 8-column
    // grid below its first column, so that every output store is 16-byte aligned
    const int32_t c0 = rowinfo[g], c1 = rowinfo[g + 1];
    const int64_t cols = c1 > c0 ? static_cast<int64_t>(c1) - (c0 & ~7) : 0;
    return ((E + Cfg::kTileAct - 1) / Cfg::kTileAct) * ((cols + Cfg::kTileW - 1) / Cfg::kTileW);
  } else if constexpr (Cfg::kRagK) {  // a whole [M, N] slab per group
    return ((E + Cfg::kTileAct - 1) / Cfg::kTileAct) * ntn;
  } else {
    int64_t cnt;
    if constexpr (Cfg::kDynamic) cnt = rowinfo[g];
    else cnt = static_cast<int64_t>(rowinfo[g + 1]) - rowinfo[g];
    return ((cnt + Cfg::kTileAct - 1) / Cfg::kTileAct) * ntn;
  }
}

template <class Cfg>
__device__ __forceinline__ int32_t group_rows(const Sched& s, int32_t g) {
  if constexpr (Cfg::kDynamic) return s.rowinfo[g];
  else return s.rowinfo[g + 1] - s.rowinfo[g];
}

// crank: this CTA's rank in its pair (0 without pairs); a pair's output tile spans
// kTileAct rows, of which CTA r owns [m0 + r * kActRows, m0 + (r + 1) * kActRows).
template <class Cfg>
__device__ __forceinline__ TileCoord decode_tile(const Sched& s, int32_t t, uint32_t crank) {
  // largest g with tile_pre[g] <= t  (tile_pre[0] = 0 <= t < tile_pre[G] = total)
  int32_t lo = 0, hi = s.G;
  while (hi - lo > 1) {
    int32_t mid = (lo + hi) >> 1;
    if (s.tile_pre[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int32_t g = lo;
  TileCoord c;
  c.g = g;
  c.half = false;
  c.tr_n = 0;
  if constexpr (Cfg::kRagged) {
    const int32_t mt = (s.E + Cfg::kTileAct - 1) / Cfg::kTileAct;
    const int32_t local = t - s.tile_pre[g];
    const int32_t n_idx = local / mt;
    const int32_t m_idx = local - n_idx * mt;
    const int32_t lo_g = s.rowinfo[g], hi_g = s.rowinfo[g + 1];
    if constexpr (Cfg::kRagN) {
      // A rows of slab g; output rows are slab-local; columns of the group only
      c.m0 = g * s.E + m_idx * Cfg::kTileAct;
      c.valid_end = c.zero_end = g * s.E + s.E;
      c.orow_delta = -g * s.E;
      c.srow_delta = 0;
      c.n0 = (lo_g & ~7) + n_idx * Cfg::kTileW;  // on the 8-column grid (16-byte stores)
      c.n_begin = lo_g;
      c.n_end = hi_g;
      c.sb_off = 0;
      c.k0 = 0;
      c.k_len = s.K;
      c.k_skip = 0;
      c.nkb = s.num_kb;
    } else {
      // A rows shared by the groups; output slab g and scales of group g; the K slice
      c.m0 = m_idx * Cfg::kTileAct;
      c.valid_end = c.zero_end = s.E;
      c.orow_delta = g * s.E;
      c.srow_delta = g * s.E;
      c.n0 = n_idx * Cfg::kTileW;
      c.n_begin = 0;
      c.n_end = s.N;
      c.sb_off = g * s.N;
      // a slice whose bounds are off the 16-element TMA grid is not computed (+0.0).  The
      // K blocks are loaded from the 128-element boundary at or below the slice start
      // (TMA boxes that start inside a 128-byte line fetch two lines per row: measured 26 %
      // slower on the weight-gradient shape); the MMA skips what lies before the slice in
      // the first block and past it in the last.
      c.k_len = ((lo_g | hi_g) & 15) ? 0 : hi_g - lo_g;
      c.k0 = lo_g & ~(kBK - 1);
      c.k_skip = c.k_len > 0 ? lo_g - c.k0 : 0;
      c.nkb = c.k_len > 0 ? (c.k_skip + c.k_len + kBK - 1) / kBK : 0;
    }
    c.bz = 0;
    return c;
  }
  const int32_t cnt = group_rows<Cfg>(s, g);
  const int32_t mt = (cnt + Cfg::kTileAct - 1) / Cfg::kTileAct;
  const int32_t local = t - s.tile_pre[g];
  const int32_t n_idx = local / mt;
  const int32_t m_idx = local - n_idx * mt;
  c.orow_delta = 0;
  c.srow_delta = 0;
  c.n_begin = 0;
  c.n_end = s.N;
  c.bz = g;
  c.sb_off = g * s.N;
  c.k0 = 0;
  c.k_len = s.K;
  c.k_skip = 0;
  c.nkb = s.num_kb;
  const int32_t base = Cfg::kDynamic ? g * s.E : s.rowinfo[g];
  if constexpr (Cfg::kPair) {
    const int32_t rem = cnt - m_idx * Cfg::kTileAct;  // rows from this tile's first on
    c.half = rem <= Cfg::kTileAct / 2;
    if (c.half) c.tr_n = (rem + 15) & ~15;
  }
  // (a transposed tile's m0 is its first row in both CTAs: each CTA's loader adds its own
  // share, crank * tr_n / 2, for the rows it holds)
  c.m0 = base + m_idx * Cfg::kTileAct + (c.half ? 0 : static_cast<int32_t>(crank) * Cfg::kActRows);
  c.n0 = n_idx * Cfg::kTileW;
  c.valid_end = base + cnt;
  c.zero_end = Cfg::kDynamic ? base + s.E : base + cnt;
  return c;
}

// Work of one CTA (all CTAs derive the same split).  With T tiles and P CTAs, the tiles
// of all full waves but the last, [0, dp), run whole: tile t on CTA t % P.  The remaining
// P + T % P tiles (all T when T < 2P) are cut into (tile, K-block) units, and each CTA
// takes one contiguous range of those units, so every CTA gets the same amount of K work
// (stream-K).  A tile whose units fall to several CTAs is finished by whichever of them
// arrives last, from the fp32 partial sums the others published.
struct Work {
  int32_t dp_tiles;  // tiles run whole
  int32_t n_dp;      // whole tiles of this CTA
  int32_t nkb;       // K blocks per tile
  int32_t sk_ctas;   // CTAs sharing the split region: min(P, units), each range non-empty
  int64_t units;     // K-block units of the split region
  int64_t sk_begin;  // this CTA's unit range
  int64_t sk_end;
  int32_t n_items;   // work items of this CTA
};

static_assert(sizeof(Work) <= 64, "Work must fit its shared-memory slot");

struct Item {
  int32_t tile;
  int32_t kb0;       // K blocks [kb0, kb1) of the tile
  int32_t kb1;
  int32_t sk_tile;   // index of a tile shared with other CTAs, else -1
};

// c: this worker (a CTA, or a CTA pair), P: the number of workers
__device__ __forceinline__ Work make_work(int32_t T, int32_t nkb, bool split, int32_t c,
                                          int32_t P) {
  Work w;
  w.nkb = nkb;
  int32_t dp = T;
  if (split && nkb > 0 && T % P != 0) dp = T >= 2 * P ? (T / P - 1) * P : 0;
  w.dp_tiles = dp;
  w.n_dp = c < dp ? (dp - 1 - c) / P + 1 : 0;
  w.units = static_cast<int64_t>(T - dp) * nkb;
  w.sk_ctas = static_cast<int32_t>(w.units < P ? w.units : P);
  w.sk_begin = c < w.sk_ctas ? w.units * c / w.sk_ctas : w.units;
  w.sk_end = c < w.sk_ctas ? w.units * (c + 1) / w.sk_ctas : w.units;
  const int32_t n_sk = w.sk_end > w.sk_begin
                           ? static_cast<int32_t>((w.sk_end - 1) / nkb - w.sk_begin / nkb + 1)
                           : 0;
  w.n_items = w.n_dp + n_sk;
  return w;
}

__device__ __forceinline__ Item work_item(const Work& w, int32_t i, int32_t c, int32_t P) {
  Item it;
  if (i < w.n_dp) {
    it.tile = c + i * P;
    it.kb0 = 0;
    it.kb1 = w.nkb;
    it.sk_tile = -1;
    return it;
  }
  const int64_t t = w.sk_begin / w.nkb + (i - w.n_dp);
  const int64_t u0 = w.sk_begin > t * w.nkb ? w.sk_begin : t * w.nkb;
  const int64_t u1 = w.sk_end < (t + 1) * w.nkb ? w.sk_end : (t + 1) * w.nkb;
  it.tile = w.dp_tiles + static_cast<int32_t>(t);
  it.kb0 = static_cast<int32_t>(u0 - t * w.nkb);
  it.kb1 = static_cast<int32_t>(u1 - t * w.nkb);
  it.sk_tile = (it.kb0 == 0 && it.kb1 == w.nkb) ? -1 : static_cast<int32_t>(t);
  return it;
}

// CTA whose unit range holds split-region unit u: the largest c with
// floor(units * c / sk_ctas) <= u
__device__ __forceinline__ int32_t unit_owner(const Work& w, int64_t u) {
  return static_cast<int32_t>(((u + 1) * w.sk_ctas - 1) / w.units);
}

// Bounded mbarrier wait: false if the CTA is aborting or the wait gave up, in which
// case the abort flag and the device status word are set.  kCluster: acquire at cluster
// scope (a barrier that the other CTA of a pair arrives on).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                         uint32_t* status, uint64_t timeout_ns) {
  auto try_wait = [&]() {
    return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
  };
  if (try_wait()) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (try_wait()) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (ptx::globaltimer_ns() - t0 > timeout_ns) {
        *abort = 1u;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Bounded wait (one thread) for a global counter to reach `want`, with acquire semantics:
// false if the CTA is aborting or the wait gave up (the abort flag and the device status
// word are then set).
__device__ __forceinline__ bool wait_count(const uint32_t* cnt, uint32_t want,
                                           volatile uint32_t* abort, uint32_t* status,
                                           uint64_t timeout_ns) {
  if (ptx::ld_acquire_gpu_u32(cnt) >= want) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    ptx::nanosleep(32);
    if (ptx::ld_acquire_gpu_u32(cnt) >= want) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (ptx::globaltimer_ns() - t0 > timeout_ns) {
        *abort = 1u;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Checked builds (compiled with MSLKB_CHECKED): every global access of the kernels is tested
// against the extents of the buffers the call passed.  An index outside them sets
// kStatusBounds in the device status word, together with one bit (16 + site) naming the kind
// of access, and the access is not made as asked: a load reads element 0 of its buffer
// instead, a store is dropped, a TMA copy takes coordinate 0 on the faulty axis (a TMA box
// may lie partly or wholly past the tensor's extent -- zero fill -- but its innermost
// coordinate must be 16-byte aligned and a store's start must not be negative).  Product
// builds compile none of the tests: the helpers return their argument.
enum CheckSite : uint32_t {
  kCkMeta = 0,        // group metadata (m_sizes, offsets, zero_start_index_M)
  kCkTmaX = 1,        // TMA load or prefetch: K coordinate out of range
  kCkTmaY = 2,        // TMA load or prefetch: row / column / group coordinate out of range
  kCkTmaAlign = 3,    // TMA load or prefetch: K coordinate not 16-byte aligned
  kCkScale = 4,       // scale_a / scale_b
  kCkStore = 5,       // direct output store
  kCkTmaStore = 6,    // TMA output store
  kCkSplit = 7,       // split-tile workspace and counters
};
__device__ __forceinline__ void ck_fail(const GemmParams& p, uint32_t site) {
#ifdef MSLKB_CHECKED
  atomicOr(p.status, kStatusBounds | (1u << (16 + site)));
#else
  (void)p;
  (void)site;
#endif
}
__device__ __forceinline__ int64_t ck_index(const GemmParams& p, int64_t i, int64_t n,
                                            uint32_t site) {
#ifdef MSLKB_CHECKED
  if (i < 0 || i >= n) {
    ck_fail(p, site);
    return 0;
  }
#else
  (void)p;
  (void)n;
  (void)site;
#endif
  return i;
}
__device__ __forceinline__ bool ck_range(const GemmParams& p, int64_t i, int64_t count,
                                         int64_t n) {
#ifdef MSLKB_CHECKED
  if (i < 0 || count < 0 || i + count > n) {
    ck_fail(p, kCkStore);
    return false;
  }
#else
  (void)p;
  (void)i;
  (void)count;
  (void)n;
#endif
  return true;
}
// TMA load coordinate on an axis of `n` elements.  x (the K axis, one byte per element) must
// start inside [lo, n) on a multiple of 16.  A box on the other axes may reach past the end,
// or lie wholly past it (the second CTA of a pair on a group's last rows, the second half of
// an N-tail weight tile): those elements read zero fill.  A start more than one box (256
// rows) past the end is a coordinate gone wrong.
__device__ __forceinline__ int32_t ck_tma(const GemmParams& p, int32_t v, int32_t lo, int64_t n,
                                          bool inner) {
#ifdef MSLKB_CHECKED
  if (v < lo || v >= (inner ? n : n + 256)) {
    ck_fail(p, inner ? kCkTmaX : kCkTmaY);
    return 0;
  }
  if (inner && (v & 15) != 0) {
    ck_fail(p, kCkTmaAlign);
    return 0;
  }
#else
  (void)p;
  (void)lo;
  (void)n;
  (void)inner;
#endif
  return v;
}

// A pointer into [base, base + n) (a load through it reads *base instead otherwise).
template <class T>
__device__ __forceinline__ const T* ck_ptr(const GemmParams& p, const T* ptr, const T* base,
                                           int64_t n) {
  return base + ck_index(p, ptr - base, n, kCkScale);
}
// A TMA store of a 32 x 32 bf16 block at (x, y) into an [rows, cols] output: false (and the
// status bits) if it would start before the output, off a 16-byte boundary, or reach past its
// last row.  Columns at or past `cols` are clipped by the copy (a block of an N-tail tile may
// lie wholly past N and write nothing).
__device__ __forceinline__ bool ck_tma_store(const GemmParams& p, int32_t x, int32_t y,
                                             int64_t rows, int64_t cols) {
#ifdef MSLKB_CHECKED
  if (x < 0 || x >= cols + 256 || (x & 7) != 0 || y < 0 || y + 32 > rows) {
    ck_fail(p, kCkTmaStore);
    return false;
  }
#else
  (void)p;
  (void)x;
  (void)y;
  (void)rows;
  (void)cols;
#endif
  return true;
}

// Buffer extents of a call, in elements (for the checked build's tests).
template <class Cfg>
__device__ __forceinline__ int64_t ext_scale_a(const GemmParams& p) {
  if constexpr (Cfg::kRagged) return static_cast<int64_t>(p.G) * p.E;
  else if constexpr (Cfg::kBlockScale) return static_cast<int64_t>(p.rows) * p.num_kb;
  else return p.rows;
}
template <class Cfg>
__device__ __forceinline__ int64_t ext_scale_b(const GemmParams& p) {
  if constexpr (Cfg::kRagN) return p.N;
  else if constexpr (Cfg::kBlockScale)
    return static_cast<int64_t>(p.G) * (p.N / Cfg::kScaleBlock) * p.num_kb;
  else return static_cast<int64_t>(p.G) * p.N;
}
template <class Cfg>
__device__ __forceinline__ int64_t ext_out_rows(const GemmParams& p) {
  if constexpr (Cfg::kRagN) return p.E;
  else if constexpr (Cfg::kRagK) return static_cast<int64_t>(p.G) * p.E;
  else return p.rows;
}

// Two TMEM values into two fp32 register accumulators with one packed (f32x2) operation:
// round-to-nearest adds, or (block scaling) fused multiply-adds by the K block's scale.
// Each lane of the pair rounds exactly as the scalar operation would.
template <bool kScale>
__device__ __forceinline__ void accum2(float& a0, float& a1, uint32_t v0, uint32_t v1,
                                       float s0, float s1) {
  const float2 v = make_float2(__uint_as_float(v0), __uint_as_float(v1));
  float2 a = make_float2(a0, a1);
  if constexpr (kScale) a = __ffma2_rn(v, make_float2(s0, s1), a);
  else a = __fadd2_rn(a, v);
  a0 = a.x;
  a1 = a.y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

// Inclusive warp scan of 64-bit values.
__device__ __forceinline__ int64_t warp_incl_scan(int64_t v, uint32_t lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int64_t o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= static_cast<uint32_t>(d)) v += o;
  }
  return v;
}

// One warp builds the scheduler tables from the [G] metadata (lane l takes a
// contiguous chunk of groups; chunks are combined with warp scans).  kSpec: a speculative
// build ahead of the dependency wait, whose metadata may still change -- its reads skip
// L1 (so no stale line is left there) and it reports nothing in the status word.
template <class Cfg, bool kSpec = false>
__device__ void build_sched(const GemmParams& p, int32_t* rowinfo, int32_t* tile_pre,
                            uint32_t lane) {
  const int64_t* meta = kSpec ? p.spec_meta : p.meta;
  const int32_t G = p.G;
  const int32_t per = (G + 31) / 32;
  const int32_t g0 = min(G, static_cast<int32_t>(lane) * per);
  const int32_t g1 = min(G, g0 + per);
  const int64_t ntn = (p.N + Cfg::kTileW - 1) / Cfg::kTileW;
  bool clamped = false;
  if constexpr (Cfg::kDynamic) {
    for (int32_t g = g0; g < g1; ++g) {
      // full slabs (batched layout) read no metadata
      int64_t v = p.meta_kind == 2 ? p.E
                  : (kSpec ? __ldcg(reinterpret_cast<const long long*>(meta) + ck_index(p, g, G, kCkMeta))
                           : meta[ck_index(p, g, G, kCkMeta)]);
      v = v < 0 ? 0 : (v > p.E ? p.E : v);
      rowinfo[g] = static_cast<int32_t>(v);
    }
  } else {
    // rows of group g: m_sizes[g], or the step between successive int32 inclusive
    // offsets (offsets[-1] = 0)
    const int32_t* offs = reinterpret_cast<const int32_t*>(meta);
    auto ld32 = [&](int32_t g) -> int64_t {
      return kSpec ? __ldcg(offs + ck_index(p, g, G, kCkMeta)) : offs[ck_index(p, g, G, kCkMeta)];
    };
    auto count = [&](int32_t g) -> int64_t {
      if (p.meta_kind == 1) return ld32(g) - (g > 0 ? ld32(g - 1) : 0);
      return kSpec ? __ldcg(reinterpret_cast<const long long*>(meta) + ck_index(p, g, G, kCkMeta))
                   : meta[ck_index(p, g, G, kCkMeta)];
    };
    // ragged layouts partition the columns (N) or the contraction (K) instead of the rows
    const int64_t total = Cfg::kRagN ? p.N : (Cfg::kRagK ? p.K : p.rows);
    // clamped exclusive prefix: off_g = min(sum_{h<g} max(m_h, 0), total_M).  Each count
    // is read from global memory once, kept in the table as min(max(m, 0), total) (a count
    // above the total clamps everything after it anyway), and replaced by its prefix.
    int64_t my_sum = 0;
    for (int32_t g = g0; g < g1; ++g) {
      const int64_t m = count(g);
      if (m < 0 || m > total) clamped = true;
      const int64_t mc = m < 0 ? 0 : (m > total ? total : m);
      rowinfo[g] = static_cast<int32_t>(mc);
      my_sum += mc;
    }
    int64_t run = warp_incl_scan(my_sum, lane) - my_sum;
    for (int32_t g = g0; g < g1; ++g) {
      const int64_t mc = rowinfo[g];
      rowinfo[g] = static_cast<int32_t>(run < total ? run : total);
      run += mc;
    }
    if (lane == 31) {  // the last chunk ends at G, so run is the sum over all groups
      if (run > total) clamped = true;
      rowinfo[G] = static_cast<int32_t>(run < total ? run : total);
    }
  }
  __syncwarp();
  int64_t my_tiles = 0;
  bool bad_slice = false;
  for (int32_t g = g0; g < g1; ++g) {
    my_tiles += group_tiles<Cfg>(rowinfo, g, p.E, ntn);
    if constexpr (Cfg::kRagK) bad_slice |= ((rowinfo[g] | rowinfo[g + 1]) & 15) != 0;
  }
  const int64_t incl = warp_incl_scan(my_tiles, lane);
  int64_t tp = incl - my_tiles;
  for (int32_t g = g0; g < g1; ++g) {
    tile_pre[g] = static_cast<int32_t>(tp);
    tp += group_tiles<Cfg>(rowinfo, g, p.E, ntn);
  }
  if (lane == 31) tile_pre[G] = static_cast<int32_t>(incl);
  const bool any_clamped = __any_sync(0xffffffffu, clamped);
  const bool any_bad = __any_sync(0xffffffffu, bad_slice);
  if constexpr (!kSpec) {
    if (any_clamped && lane == 0 && blockIdx.x == 0) atomicOr(p.status, kStatusClamped);
    if (any_bad && lane == 0 && blockIdx.x == 0) atomicOr(p.status, kStatusBadSlice);
  }
}

// The 16-byte chunk `chunk` of every row of one stage's activation and weight tiles set to
// zero by the 32 lanes of a warp (rows strided over the lanes), made visible to the tensor
// core's reads, and the lanes converged again.
template <class Cfg>
__device__ __forceinline__ void zero_stage_chunk(uint32_t sa_base, uint32_t sw_base,
                                                 uint32_t chunk, uint32_t lane) {
  for (int row = static_cast<int>(lane); row < Cfg::kActRows; row += 32)
    ptx::st_shared_v4(sa_base + row * 128u + ((chunk ^ (row & 7u)) << 4), 0u, 0u, 0u, 0u);
  for (int row = static_cast<int>(lane); row < Cfg::kWRows; row += 32)
    ptx::st_shared_v4(sw_base + row * 128u + ((chunk ^ (row & 7u)) << 4), 0u, 0u, 0u, 0u);
  ptx::fence_proxy_async_smem();
  __syncwarp();
}

// Ragged K, the first K block of a slice that starts `lo` bytes into it and ends at `hi`
// (<= 128): the block was loaded from the 128-byte boundary below the slice start, and
// before lo and past hi lie other groups' K (or TMA zero fill).  Whole 32-byte steps
// outside [lo, hi) are not issued; in a half-used step the unused 16 bytes of every row of
// both operands are zeroed first (slices start and end on a 16-element boundary; both
// operands, since 0 x NaN is NaN; 128-byte swizzle: chunk c of row r sits at c ^ (r & 7)).
// The first issued step overwrites the accumulator.  Out of line: once per tile, off the
// MMA warp's per-block path.  Called by every lane of the MMA warp: the zeroing is shared,
// lane 0 issues the MMAs.
template <class Cfg>
__device__ __noinline__ void mma_ragk_first_block(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t sa_base,
                                                  uint32_t sw_base, int32_t lo, int32_t hi,
                                                  uint32_t lane) {
  if (lo & 16) zero_stage_chunk<Cfg>(sa_base, sw_base, static_cast<uint32_t>(lo >> 4) - 1u, lane);
  if (hi & 16) zero_stage_chunk<Cfg>(sa_base, sw_base, static_cast<uint32_t>(hi >> 4), lane);
  if (lane != 0) return;
  const int k_first = lo / 32;
  const int k_end = (hi + 31) / 32;
  for (int k = k_first; k < k_end; ++k)
    ptx::mma_f8f6f4(d_tmem, a_desc + 2u * k, b_desc + 2u * k, Cfg::kIdesc,
                    k > k_first ? 1u : 0u);
}

// K blocks per accumulation chunk that the unrolled MMA path below serves (the default
// chunk; other chunk lengths take the general loop).
constexpr int kUnrolledChunkKb = 8;

// One whole accumulation chunk of kUnrolledChunkKb K blocks whose first block sits in
// stage kS0 of the ring, the ring's phase for that pass being `phase`.  Stage numbers,
// barrier addresses, descriptor offsets and accumulate flags are all compile-time here, so
// per K block the MMA thread only waits, fences, issues its four MMAs and commits.  The
// tensor core's queue hides little of what this thread does between two blocks' MMAs
// (measured on GB300: back-to-back 128 x 256 x 32 MMAs take the nominal 128 cycles each,
// but a wait, a commit and a few dozen instructions of loop bookkeeping per block leave
// the tensor core idle); with the loads replaced by bare barrier arrivals, a 128 x 256
// tile's MMA stream takes ~669 cycles per K block of four MMAs in the general loop below
// and ~565 in this form, a CTA pair's ~696 and ~562 (512 at the nominal rate).  The
// chunk's commit to its TMEM buffer's barrier goes before the last stage's commit.  The
// barrier addresses follow the kernel's layout: the barrier that says stage s is ready at
// s_wait + 8 s (its full barrier, s_bar + 8 s; on ragged-K tiles with the edge warp its
// ready barrier), its empty barrier at s_bar + 8 (kStages + s).
template <class Cfg, int kS0, int kJ = 0>
__device__ __forceinline__ bool mma_chunk_unrolled(const GemmParams& p, uint32_t s_bar,
                                                   uint32_t s_wait, uint32_t tfull,
                                                   uint32_t d_buf, uint32_t idesc,
                                                   uint32_t a_lo0, uint32_t b_lo0,
                                                   uint32_t phase, volatile uint32_t* abort) {
  if constexpr (kJ == kUnrolledChunkKb) {
    return true;
  } else {
    // block kJ of the chunk: its stage, and whether the ring wrapped since the chunk's start
    // (s_wait: the barriers that say a stage is ready, one per stage from there)
    constexpr int kSt = (kS0 + kJ) % Cfg::kStages;
    constexpr uint32_t kFlip = static_cast<uint32_t>(((kS0 + kJ) / Cfg::kStages) & 1);
    if (!wait_bar(s_wait + 8u * kSt, phase ^ kFlip, abort, p.status, p.timeout_ns)) return false;
    ptx::tc_fence_after_sync();
    // the stage's operand tiles, then K steps of 32 bytes inside the 128-byte swizzled row
    // (+2 in 16-byte descriptor units each)
    static_assert(kBK / 32 == 4, "four MMAs per stage");
    constexpr uint32_t kAOff =
        static_cast<uint32_t>(((Cfg::kSwap ? Cfg::kWBytes : Cfg::kActBytes) * kSt) >> 4);
    constexpr uint32_t kBOff =
        static_cast<uint32_t>(((Cfg::kSwap ? Cfg::kActBytes : Cfg::kWBytes) * kSt) >> 4);
    ptx::mma_f8f6f4_lo<Cfg::kPair, kAOff + 0, kBOff + 0>(d_buf, a_lo0, b_lo0, idesc,
                                                        kJ > 0 ? 1u : 0u);
    ptx::mma_f8f6f4_lo<Cfg::kPair, kAOff + 2, kBOff + 2>(d_buf, a_lo0, b_lo0, idesc, 1u);
    ptx::mma_f8f6f4_lo<Cfg::kPair, kAOff + 4, kBOff + 4>(d_buf, a_lo0, b_lo0, idesc, 1u);
    ptx::mma_f8f6f4_lo<Cfg::kPair, kAOff + 6, kBOff + 6>(d_buf, a_lo0, b_lo0, idesc, 1u);
    const uint32_t empty = s_bar + 8u * (Cfg::kStages + kSt);
    if constexpr (Cfg::kPair) {
      if constexpr (kJ == kUnrolledChunkKb - 1) ptx::mma_commit_pair(tfull, 0x3);
      ptx::mma_commit_pair(empty, 0x3);
    } else {
      if constexpr (kJ == kUnrolledChunkKb - 1) ptx::mma_commit(tfull);
      ptx::mma_commit(empty);
    }
    return mma_chunk_unrolled<Cfg, kS0, kJ + 1>(p, s_bar, s_wait, tfull, d_buf, idesc, a_lo0,
                                                b_lo0, phase, abort);
  }
}

// mma_chunk_unrolled for the runtime stage `stage` (one instance per ring position).
template <class Cfg, int kS = 0>
__device__ __forceinline__ bool mma_chunk_at(int stage, const GemmParams& p, uint32_t s_bar,
                                             uint32_t s_wait, uint32_t tfull, uint32_t d_buf,
                                             uint32_t idesc, uint32_t a_lo0, uint32_t b_lo0,
                                             uint32_t phase, volatile uint32_t* abort) {
  if constexpr (kS + 1 < Cfg::kStages) {
    if (stage != kS)
      return mma_chunk_at<Cfg, kS + 1>(stage, p, s_bar, s_wait, tfull, d_buf, idesc, a_lo0,
                                       b_lo0, phase, abort);
  }
  return mma_chunk_unrolled<Cfg, kS>(p, s_bar, s_wait, tfull, d_buf, idesc, a_lo0, b_lo0,
                                     phase, abort);
}

// Block scaling on 128-row tiles: every K block sums into an accumulator of its own (a TMEM
// buffer, kNumAcc of them in a ring), so each block is a chunk of one: wait for the buffer to
// be drained, wait for the stage, four MMAs that start the accumulator afresh, commit the
// buffer to the epilogue (which frees the stage once it sees the commit).  The general loop
// does that with runtime stage, phase, buffer and descriptor bookkeeping per block; this
// issues kUnrolledChunkKb blocks in a row with all of it fixed at compile time, one instance
// per ring position kS0 and buffer kB0 of the first block.  use_par: parity of the number of
// times the first block's buffer was used before (the epilogue's hand-backs).
template <class Cfg, int kS0, int kB0, int kJ = 0>
__device__ __forceinline__ bool mma_bs_run_unrolled(const GemmParams& p, uint32_t s_bar,
                                                    uint32_t tmem_base, uint32_t a_lo0,
                                                    uint32_t b_lo0, uint32_t phase,
                                                    uint32_t use_par, volatile uint32_t* abort) {
  if constexpr (kJ == kUnrolledChunkKb) {
    return true;
  } else {
    constexpr int kSt = (kS0 + kJ) % Cfg::kStages;
    constexpr uint32_t kFlip = static_cast<uint32_t>(((kS0 + kJ) / Cfg::kStages) & 1);
    constexpr int kBuf = (kB0 + kJ) % Cfg::kNumAcc;
    constexpr uint32_t kUseFlip = static_cast<uint32_t>(((kB0 + kJ) / Cfg::kNumAcc) & 1);
    const uint32_t tempty = s_bar + 8u * (2 * Cfg::kStages + Cfg::kNumAcc + kBuf);
    const uint32_t tfull = s_bar + 8u * (2 * Cfg::kStages + kBuf);
    if (!wait_bar(tempty, (use_par ^ kUseFlip) ^ 1u, abort, p.status, p.timeout_ns))
      return false;
    ptx::tc_fence_after_sync();
    if (!wait_bar(s_bar + 8u * kSt, phase ^ kFlip, abort, p.status, p.timeout_ns)) return false;
    ptx::tc_fence_after_sync();
    constexpr uint32_t kAOff = static_cast<uint32_t>((Cfg::kActBytes * kSt) >> 4);
    constexpr uint32_t kBOff = static_cast<uint32_t>((Cfg::kWBytes * kSt) >> 4);
    const uint32_t d_buf = tmem_base + static_cast<uint32_t>(kBuf * Cfg::kBufCols);
    ptx::mma_f8f6f4_lo<false, kAOff + 0, kBOff + 0>(d_buf, a_lo0, b_lo0, Cfg::kIdesc, 0u);
    ptx::mma_f8f6f4_lo<false, kAOff + 2, kBOff + 2>(d_buf, a_lo0, b_lo0, Cfg::kIdesc, 1u);
    ptx::mma_f8f6f4_lo<false, kAOff + 4, kBOff + 4>(d_buf, a_lo0, b_lo0, Cfg::kIdesc, 1u);
    ptx::mma_f8f6f4_lo<false, kAOff + 6, kBOff + 6>(d_buf, a_lo0, b_lo0, Cfg::kIdesc, 1u);
    ptx::mma_commit(tfull);
    return mma_bs_run_unrolled<Cfg, kS0, kB0, kJ + 1>(p, s_bar, tmem_base, a_lo0, b_lo0, phase,
                                                      use_par, abort);
  }
}

// mma_bs_run_unrolled for the runtime ring position `stage` and first buffer `buf`.
template <class Cfg, int kS = 0, int kB = 0>
__device__ __forceinline__ bool mma_bs_run_at(int stage, int buf, const GemmParams& p,
                                              uint32_t s_bar, uint32_t tmem_base,
                                              uint32_t a_lo0, uint32_t b_lo0, uint32_t phase,
                                              uint32_t use_par, volatile uint32_t* abort) {
  if constexpr (kB + 1 < Cfg::kNumAcc) {
    if (buf != kB)
      return mma_bs_run_at<Cfg, kS, kB + 1>(stage, buf, p, s_bar, tmem_base, a_lo0, b_lo0,
                                            phase, use_par, abort);
  }
  if constexpr (kS + 1 < Cfg::kStages) {
    if (stage != kS)
      return mma_bs_run_at<Cfg, kS + 1, kB>(stage, buf, p, s_bar, tmem_base, a_lo0, b_lo0,
                                            phase, use_par, abort);
  }
  return mma_bs_run_unrolled<Cfg, kS, kB>(p, s_bar, tmem_base, a_lo0, b_lo0, phase, use_par,
                                          abort);
}

// cp.async loader: one 16-byte chunk of a swizzled tile row.
__device__ __forceinline__ void load_chunk(uint32_t dst, const uint8_t* row_ptr, bool row_ok,
                                           int32_t k, int32_t K, int32_t width,
                                           const uint8_t* any_valid) {
  if (width == 16) {
    const bool ok = row_ok && k < K;  // K % 16 == 0 on this path
    ptx::cp_async<16>(dst, ok ? row_ptr + k : any_valid, ok ? 16u : 0u);
  } else if (width == 8) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int32_t kk = k + 8 * h;
      const bool ok = row_ok && kk < K;  // K % 8 == 0 on this path
      ptx::cp_async<8>(dst + 8 * h, ok ? row_ptr + kk : any_valid, ok ? 8u : 0u);
    }
  } else if (width == 4) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int32_t kk = k + 4 * h;
      const bool ok = row_ok && kk < K;  // K % 4 == 0 on this path
      ptx::cp_async<4>(dst + 4 * h, ok ? row_ptr + kk : any_valid, ok ? 4u : 0u);
    }
  } else {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int32_t kk = k + i;
      const uint32_t b = (row_ok && kk < K) ? static_cast<uint32_t>(__ldg(row_ptr + kk)) : 0u;
      w[i >> 2] |= b << (8 * (i & 3));
    }
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3])
                 : "memory");
  }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmParams p,
                        const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC,
                        const __grid_constant__ CUtensorMap tmB2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_act = ptx::smem_addr(smem + Cfg::kOffAct);
  const uint32_t s_w = ptx::smem_addr(smem + Cfg::kOffW);
  const uint32_t s_bar = ptx::smem_addr(smem + Cfg::kOffBar);
  const uint32_t s_out = ptx::smem_addr(smem + Cfg::kOffOut);
  auto full_bar = [&](int s) { return s_bar + 8u * s; };
  auto empty_bar = [&](int s) { return s_bar + 8u * (Cfg::kStages + s); };
  auto tfull_bar = [&](int b) { return s_bar + 8u * (2 * Cfg::kStages + b); };
  auto tempty_bar = [&](int b) { return s_bar + 8u * (2 * Cfg::kStages + Cfg::kNumAcc + b); };
  auto tq_full_bar = [&](int i) {
    return s_bar + 8u * (2 * Cfg::kStages + 2 * Cfg::kNumAcc + i);
  };
  auto tq_empty_bar = [&](int i) {
    return s_bar + 8u * (2 * Cfg::kStages + 2 * Cfg::kNumAcc + Cfg::kTQ + i);
  };
  // ragged K: stage s loaded and trimmed to the tile's K slice (the MMA thread waits on
  // these instead of the full barriers)
  const uint32_t s_ready = s_bar + 8u * (2 * Cfg::kStages + 2 * Cfg::kNumAcc + 2 * Cfg::kTQ);
  auto ready_bar = [&](int s) { return s_ready + 8u * s; };
  volatile int32_t* tq = reinterpret_cast<volatile int32_t*>(smem + Cfg::kOffTQ);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffMisc + 4);
  int32_t* rowinfo = reinterpret_cast<int32_t*>(smem + Cfg::kOffSched);
  int32_t* tile_pre = rowinfo + (kMaxGroups + 1);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  // CTA pairs: this CTA's rank in its pair; work is divided among pairs
  const uint32_t crank = Cfg::kPair ? ptx::cluster_ctarank() : 0u;
  const int32_t worker = static_cast<int32_t>(blockIdx.x) / Cfg::kCtas;
  const int32_t workers = static_cast<int32_t>(gridDim.x) / Cfg::kCtas;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      ptx::mbar_init(full_bar(s), Cfg::kTma ? 1u : static_cast<uint32_t>(Cfg::kLoaderThreads));
      ptx::mbar_init(empty_bar(s), 1u);
    }
    for (int b = 0; b < Cfg::kNumAcc; ++b) {
      ptx::mbar_init(tfull_bar(b), 1u);
      // pairs: the leader's MMA waits for the epilogue warps of both CTAs
      ptx::mbar_init(tempty_bar(b), static_cast<uint32_t>(Cfg::kEpiWarps * Cfg::kCtas));
    }
    if constexpr (Cfg::kEdgeWarp)
      for (int st = 0; st < Cfg::kStages; ++st) ptx::mbar_init(ready_bar(st), 1u);
    for (int i = 0; i < Cfg::kTQ; ++i) {
      ptx::mbar_init(tq_full_bar(i), 1u);
      // on the leader: its MMA thread and epilogue warps, the peer's loader and epilogue
      // warps (the peer's empty barriers go unused)
      ptx::mbar_init(tq_empty_bar(i), static_cast<uint32_t>(2 + 2 * Cfg::kEpiWarps));
    }
    *abort_flag = 0u;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if constexpr (Cfg::kTma) {
    if (warp == 0 && lane == 0 && p.num_kb > 0) {
      ptx::prefetch_tensormap(&tmA);
      ptx::prefetch_tensormap(&tmB);
      if constexpr (Cfg::kSwap && !Cfg::kRagged && !Cfg::kBlockScale) {
        if (p.w_pair != 0) ptx::prefetch_tensormap(&tmB2);
      }
    }
  }
  if (warp == Cfg::kMmaWarp) {
    if constexpr (Cfg::kPair) {
      ptx::tmem_alloc_pair(ptx::smem_addr(tmem_holder), Cfg::kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_addr(tmem_holder), Cfg::kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  if constexpr (Cfg::kPair) {
    // the peer signals this CTA's barriers only after both have initialised theirs
    ptx::tc_fence_before_sync();
    ptx::cluster_sync();
    ptx::tc_fence_after_sync();
  }
  // Everything above is CTA-local.  With programmatic dependent launch the next kernel on
  // the stream may begin launching now; every global-memory access whose result matters
  // (the metadata, operands, scales, output, split workspace, status word) waits for the
  // kernels this one depends on to complete, below.
  if (threadIdx.x == 0) ptx::griddep_launch_dependents();
  // Swap-AB plans stream weights, and with programmatic dependent launch this CTA may be
  // resident while the kernel before it finishes.  Meanwhile the prefetch warp works out
  // the CTA's first K blocks from a speculative read of the group metadata and asks L2 to
  // prefetch their weight tiles.  Only a hint: the real schedule below reads the metadata
  // again after the dependency wait, and every load goes through L2 (coherent with
  // whatever the earlier kernel writes).  The warp keeps its own tables and takes no part
  // in the setup barriers, so a CTA that starts late is not held up by it; its next and
  // last barrier is the teardown's.
  const bool spec_warp = Cfg::kSpecWarp && warp == static_cast<uint32_t>(Cfg::kSpecWarpIdx);
  if constexpr (Cfg::kSpecWarp) {
    if (spec_warp && p.num_kb > 0 && p.prefetch_kb > 0) {
      int32_t* s_rows = reinterpret_cast<int32_t*>(smem + Cfg::kOffSpec);
      int32_t* s_tpre = s_rows + (kMaxGroups + 1);
      build_sched<Cfg, true>(p, s_rows, s_tpre, lane);
      __syncwarp();
      if (lane == 0) {
        Sched ss;
        ss.rowinfo = s_rows;
        ss.tile_pre = s_tpre;
        ss.G = p.G;
        ss.E = p.E;
        ss.n_tiles_n = (p.N + Cfg::kWRows - 1) / Cfg::kWRows;
        ss.total = s_tpre[p.G];
        ss.N = p.N;
        ss.K = p.K;
        ss.num_kb = p.num_kb;
        const Work w = make_work(ss.total, p.num_kb, p.split_k != 0, worker, workers);
        int32_t budget = p.prefetch_kb;
        for (int32_t i = 0; i < w.n_items && budget > 0; ++i) {
          const Item it = work_item(w, i, worker, workers);
          const TileCoord c = decode_tile<Cfg>(ss, it.tile, 0u);
          for (int32_t kb = it.kb0; kb < it.kb1 && budget > 0; ++kb, --budget)
            ptx::tma_prefetch_3d(&tmB, ck_tma(p, kb * kBK, 0, p.K, true),
                                 ck_tma(p, c.n0, 0, p.N, false),
                                 ck_tma(p, c.g, 0, p.G, false));
        }
      }
      __syncwarp();
    }
  }
  // setup barriers: every warp but the prefetch warp
  auto setup_sync = [&]() {
    if constexpr (Cfg::kSpecWarp) {
      if (!spec_warp) ptx::named_bar_sync(1, Cfg::kThreads - 32);
    } else {
      __syncthreads();
    }
  };
  if (!spec_warp) ptx::griddep_wait();
  if (warp == Cfg::kEpiWarp0) build_sched<Cfg>(p, rowinfo, tile_pre, lane);
  ptx::tc_fence_before_sync();
  setup_sync();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = spec_warp ? 0u : *tmem_holder;

  Sched sched;
  sched.rowinfo = rowinfo;
  sched.tile_pre = tile_pre;
  sched.G = p.G;
  sched.E = p.E;
  sched.n_tiles_n = (p.N + Cfg::kWRows - 1) / Cfg::kWRows;
  sched.total = spec_warp ? 0 : tile_pre[p.G];
  sched.N = p.N;
  sched.K = p.K;
  sched.num_kb = p.num_kb;
  const bool has_k = p.num_kb > 0;
  // CTA pairs with a claim counter take their tiles in claim order: a pair that finishes a
  // tile early (a group's half-used last tile) takes the next unclaimed one, so the tiles in
  // flight stay a window of consecutive tiles and the pairs that share a weight tile stay in
  // step on it (with tiles in a fixed stride they drift apart and re-read weights from DRAM).
  // Item i of every role is slot i % kTQ of the tile ring: the leader's loader claims and
  // writes it into both CTAs; the leader's MMA thread and epilogue warps and the peer's
  // loader and epilogue warps take it.  Every wait is bounded.  The results do not depend
  // on which pair runs which tile.
  const bool dyn = Cfg::kPair && p.tile_ctr != nullptr && has_k;
  auto whole_tile = [&](int32_t t) {
    Item it;
    it.tile = t;
    it.kb0 = 0;
    it.kb1 = p.num_kb;
    it.sk_tile = -1;
    return it;
  };
  // the leader's loader: claim item i (a tile number, or -1 past the last tile).  The
  // claim for item i + 1 is issued while item i's last loads go out (claim_early), so its
  // round trip to the counter does not hold up the next tile's first load.
  uint32_t claim_u = 0;
  bool claimed = false;
  auto claim_early = [&]() {
    claim_u = atomicAdd(p.tile_ctr, 1u);
    claimed = true;
  };
  auto tq_claim = [&](int32_t i, bool& ok) -> int32_t {
    const int slot = i % (Cfg::kTQ > 0 ? Cfg::kTQ : 1);
    const uint32_t par = static_cast<uint32_t>(((i / (Cfg::kTQ > 0 ? Cfg::kTQ : 1)) & 1) ^ 1);
    if (!claimed) claim_early();
    claimed = false;
    if (!wait_bar<true>(tq_empty_bar(slot), par, abort_flag, p.status, p.timeout_ns)) {
      ok = false;
      return -1;
    }
    const uint32_t u = claim_u;
    const int32_t t = u < static_cast<uint32_t>(sched.total) ? static_cast<int32_t>(u) : -1;
    tq[slot] = t;
    ptx::st_shared_cluster_u32(ptx::mapa_shared(ptx::smem_addr(const_cast<int32_t*>(tq + slot)), 1u),
                               static_cast<uint32_t>(t));
    ptx::mbar_arrive(tq_full_bar(slot));
    ptx::mbar_arrive_cluster(ptx::mapa_shared(tq_full_bar(slot), 1u));
    return t;
  };
  // any other role (one thread): take item i
  auto tq_take = [&](int32_t i, bool& ok) -> int32_t {
    const int slot = i % (Cfg::kTQ > 0 ? Cfg::kTQ : 1);
    const uint32_t par = static_cast<uint32_t>((i / (Cfg::kTQ > 0 ? Cfg::kTQ : 1)) & 1);
    const bool got = crank == 0
                         ? wait_bar(tq_full_bar(slot), par, abort_flag, p.status, p.timeout_ns)
                         : wait_bar<true>(tq_full_bar(slot), par, abort_flag, p.status,
                                          p.timeout_ns);
    if (!got) {
      ok = false;
      return -1;
    }
    const int32_t t = tq[slot];
    if (crank == 0) ptx::mbar_arrive(tq_empty_bar(slot));
    else ptx::mbar_arrive_cluster(ptx::mapa_shared(tq_empty_bar(slot), 0u));
    return t;
  };
  // the work split lives in shared memory: every role reads it, none keeps it in registers
  Work* work_smem = reinterpret_cast<Work*>(smem + Cfg::kOffWork);
  if (threadIdx.x == 0)
    *work_smem = make_work(sched.total, p.num_kb, p.split_k != 0 && !Cfg::kPair && !Cfg::kRagged,
                           worker, workers);
  setup_sync();
  const Work& work = *work_smem;

  if (warp < static_cast<uint32_t>(Cfg::kEpiWarp0)) {
  // producer side: loader warp(s), MMA warp, and idle warps (register split: two; the
  // prefetch warp, whose work is done)
  if constexpr (Cfg::kRegSplit) ptx::setmaxnreg_dec<Cfg::kRegsLow>();
  if (warp < static_cast<uint32_t>(Cfg::kLoaderWarps)) {
    // ------------------------------------------------------------------ loader
    if constexpr (Cfg::kTma) {
      if (lane == 0 && has_k) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        // swap-AB plans stream each weight tile once past a few activation rows: the
        // weights are marked evict-first in L2, the activations evict-last (measured on
        // GB300: +2-4 % on the weight-streaming shapes, a loss on the 128-row tiles)
        const uint64_t pol_act = ptx::l2_policy_evict_last();
        const uint64_t pol_w = ptx::l2_policy_evict_first();
        // test hook: the first CTA (CTA pairs: both CTAs of the first pair) skips one stage
        bool withhold = p.test_stall != 0 && worker == 0;
        for (int32_t i = 0; ok && (dyn || i < work.n_items); ++i) {
          Item it;
          if (dyn) {
            const int32_t t = crank == 0 ? tq_claim(i, ok) : tq_take(i, ok);
            if (t < 0) break;
            it = whole_tile(t);
          } else {
            it = work_item(work, i, worker, workers);
          }
          const TileCoord c = decode_tile<Cfg>(sched, it.tile, crank);
          const int32_t kb_end = Cfg::kRagK ? c.nkb : it.kb1;  // a ragged-K tile's own K
          const int32_t kb_claim = max(it.kb0, kb_end - 4);    // pairs: next tile's claim
          // pairs: this CTA's first activation row (a transposed tile: its share of the rows)
          const int32_t a_row =
              c.m0 + (Cfg::kPair && c.half ? static_cast<int32_t>(crank) * (c.tr_n / 2) : 0);
          for (int32_t kb = it.kb0; kb < kb_end; ++kb) {
            if (dyn && crank == 0 && kb == kb_claim) claim_early();
            if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
              ok = false;
              break;
            }
            if constexpr (Cfg::kPair) {
              if (withhold) {
                // neither CTA of the pair arrives or loads: the leader's full barrier for this
                // stage never completes, so the leader's MMA wait runs out
                withhold = false;
              } else {
                // both CTAs' bytes complete on the leader's full barrier, which expects them all
                const uint32_t fb = ptx::mapa_shared(full_bar(stage), 0u);
                if (crank == 0) ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * Cfg::kStageBytes);
                const int32_t x = ck_tma(p, kb * kBK, 0, p.K, true);
                ptx::tma_load_2d_pair(s_act + stage * Cfg::kActBytes, &tmA, fb, x,
                                      ck_tma(p, a_row, 0, p.rows, false));
                // (the second CTA's half of an N-tail tile may lie wholly past N: zero fill)
                ptx::tma_load_3d_pair(
                    s_w + stage * Cfg::kWBytes, &tmB, fb, x,
                    ck_tma(p, c.n0 + static_cast<int32_t>(crank) * Cfg::kWRows, 0, p.N, false),
                    ck_tma(p, c.g, 0, p.G, false));
              }
            } else if (withhold) {
              withhold = false;  // this stage's full barrier never completes
            } else if (Cfg::kSwap && !Cfg::kRagged && !Cfg::kBlockScale && p.w_pair != 0 &&
                       stage + 1 < Cfg::kStages && kb + 1 < kb_end) {
              // Swap-AB: the weights of K blocks kb and kb + 1 in one TMA operation (a box of
              // two K blocks of a 4-D view of B, which lands as the two stages' weight tiles
              // one after the other): an SM's weight stream is capped by its rate of TMA
              // operations, 16 KB ones reaching about two thirds of what 32 KB ones do.  The
              // next stage must be free as well; stage s's barrier takes both blocks' weight
              // bytes (the MMA thread consumes s before s + 1), s + 1's its activations only.
              if (!wait_bar(empty_bar(stage + 1), phase ^ 1u, abort_flag, p.status,
                            p.timeout_ns)) {
                ok = false;
                break;
              }
              ptx::mbar_arrive_expect_tx(full_bar(stage), Cfg::kActBytes + 2 * Cfg::kWBytes);
              ptx::mbar_arrive_expect_tx(full_bar(stage + 1), Cfg::kActBytes);
              const int32_t x = ck_tma(p, kb * kBK, 0, p.K, true);
              const int32_t x1 = ck_tma(p, (kb + 1) * kBK, 0, p.K, true);
              const int32_t ya = ck_tma(p, c.m0, 0, p.rows, false);
              const int32_t yb = ck_tma(p, c.n0, 0, p.N, false);
              const int32_t zb = ck_tma(p, c.bz, 0, p.G, false);
              ptx::tma_load_2d_hint(s_act + stage * Cfg::kActBytes, &tmA, full_bar(stage), x,
                                    ya, pol_act);
              ptx::tma_load_2d_hint(s_act + (stage + 1) * Cfg::kActBytes, &tmA,
                                    full_bar(stage + 1), x1, ya, pol_act);
              ptx::tma_load_4d_hint(s_w + stage * Cfg::kWBytes, &tmB2, full_bar(stage), 0, yb,
                                    ck_tma(p, kb, 0, p.num_kb, false), zb, pol_w);
              ++stage;  // the loop's own step below moves past stage + 1
              ++kb;
            } else {
              ptx::mbar_arrive_expect_tx(full_bar(stage), Cfg::kStageBytes);
              // k0: a ragged-K slice starts on a multiple of 16 elements (16 bytes)
              const int32_t x = ck_tma(p, c.k0 + kb * kBK, 0, p.K, true);
              const int32_t ya = ck_tma(p, c.m0, 0, p.rows, false);
              const int32_t yb = ck_tma(p, c.n0, 0, p.N, false);
              const int32_t zb = ck_tma(p, c.bz, 0, Cfg::kRagged ? 1 : p.G, false);
              if constexpr (Cfg::kSwap) {
                ptx::tma_load_2d_hint(s_act + stage * Cfg::kActBytes, &tmA, full_bar(stage), x,
                                      ya, pol_act);
                ptx::tma_load_3d_hint(s_w + stage * Cfg::kWBytes, &tmB, full_bar(stage), x, yb,
                                      zb, pol_w);
              } else {
                ptx::tma_load_2d(s_act + stage * Cfg::kActBytes, &tmA, full_bar(stage), x, ya);
                ptx::tma_load_3d(s_w + stage * Cfg::kWBytes, &tmB, full_bar(stage), x, yb, zb);
              }
            }
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        // tail: wait until the MMA has released every stage it was given
        for (int i = 0; ok && i < Cfg::kStages; ++i) {
          ok = wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else {
      if (has_k) {
        const uint32_t tid = threadIdx.x;  // 0 .. kLoaderThreads - 1
        int stage = 0;
        uint32_t phase = 0;
        int64_t fills = 0;  // stages issued by this thread
        bool ok = true;
        for (int32_t i = 0; ok && i < work.n_items; ++i) {
          const Item it = work_item(work, i, worker, workers);
          const TileCoord c = decode_tile<Cfg>(sched, it.tile, crank);
          const uint8_t* b_group = p.B + static_cast<size_t>(c.g) * p.N * p.K;
          for (int32_t kb = it.kb0; kb < it.kb1; ++kb) {
            if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
              ok = false;
              break;
            }
            const int32_t k0 = kb * kBK;
            constexpr int kChunks = (Cfg::kActRows + Cfg::kWRows) * 8;
            for (int i = tid; i < kChunks; i += Cfg::kLoaderThreads) {
              const int r_all = i >> 3;
              const int ch = i & 7;
              const bool is_act = r_all < Cfg::kActRows;
              const int r = is_act ? r_all : r_all - Cfg::kActRows;
              const uint32_t dst = (is_act ? s_act + stage * Cfg::kActBytes
                                           : s_w + stage * Cfg::kWBytes) +
                                   r * 128 + (static_cast<uint32_t>(ch ^ (r & 7)) << 4);
              const uint8_t* row_ptr;
              bool row_ok;
              if (is_act) {
                const int32_t R = c.m0 + r;
                row_ok = R < p.rows;
                row_ptr = p.A + static_cast<size_t>(row_ok ? R : 0) * p.K;
              } else {
                const int32_t n = c.n0 + r;
                row_ok = n < p.N;
                row_ptr = b_group + static_cast<size_t>(row_ok ? n : 0) * p.K;
              }
              load_chunk(dst, row_ptr, row_ok, k0 + ch * 16, p.K, p.copy_width, p.A);
            }
            ptx::cp_async_commit();
            if (fills >= Cfg::kCpLag) {
              ptx::cp_async_wait<Cfg::kCpLag>();
              ptx::fence_proxy_async_smem();
              ptx::mbar_arrive(full_bar(static_cast<int>((fills - Cfg::kCpLag) % Cfg::kStages)));
            }
            ++fills;
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        ptx::cp_async_wait<0>();
        ptx::fence_proxy_async_smem();
        if (ok) {
          for (int64_t f = (fills > Cfg::kCpLag ? fills - Cfg::kCpLag : 0); f < fills; ++f)
            ptx::mbar_arrive(full_bar(static_cast<int>(f % Cfg::kStages)));
          if (tid == 0) {
            for (int i = 0; ok && i < Cfg::kStages; ++i) {
              ok = wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns);
              if (++stage == Cfg::kStages) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
        }
      }
    }
  } else if (warp == static_cast<uint32_t>(Cfg::kMmaWarp)) {
    // ------------------------------------------------------------------ MMA issuer
    // The tensor core sums at most kb_per_chunk K blocks into one TMEM chunk buffer
    // (two buffers, alternating); the epilogue adds every chunk into fp32 registers with
    // round-to-nearest, so the tensor core's own accumulation only ever spans a chunk.
    // A pair's MMAs are issued by its leader (rank 0) alone.
    // Ragged K without the edge warp: the whole warp walks the loop (every lane waits on the
    // same barriers), so that the zeroing of a slice's half-used 32-byte steps is shared by
    // 32 lanes; lane 0 alone issues the MMAs and commits.  Other kernels (and ragged K with
    // the edge warp, which trims the stages and passes them on through the ready barriers):
    // lane 0 alone.
    constexpr bool kWarpWalks = Cfg::kRagK && !Cfg::kEdgeWarp;
    const bool issuer = lane == 0;
    // a wait's outcome, made the same for every lane walking the loop (so that a wait that
    // runs out just as its barrier completes cannot send the lanes different ways)
    auto warp_agrees = [&](bool ok_lane) -> bool {
      if constexpr (kWarpWalks) return __all_sync(0xffffffffu, ok_lane);
      else return ok_lane;
    };
    // the barriers that say a stage is ready for the MMAs
    const uint32_t s_wait = Cfg::kEdgeWarp ? s_ready : s_bar;
    if ((issuer || kWarpWalks) && has_k && crank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t chunk = 0;  // chunks issued by this CTA: buffer = chunk % kNumAcc
      bool ok = true;
      const int32_t kpc = Cfg::kBlockScale ? Cfg::kBSSub : p.kb_per_chunk;
      // the unrolled chunk path (128-row and pair tiles, ragged K with the edge warp; the
      // other ragged-K tiles, block scaling and the swap-AB tiles keep the general loop)
      constexpr bool kUnrolledMma = !Cfg::kSwap && !kWarpWalks && !Cfg::kBlockScale;
      const uint32_t a_lo0 = ptx::sw128_kmajor_desc_lo(Cfg::kSwap ? s_w : s_act);
      const uint32_t b_lo0 = ptx::sw128_kmajor_desc_lo(Cfg::kSwap ? s_act : s_w);
      for (int32_t i = 0; ok && (dyn || i < work.n_items); ++i) {
        Item it;
        if (dyn) {
          const int32_t t = tq_take(i, ok);
          if (t < 0) break;
          it = whole_tile(t);
        } else {
          it = work_item(work, i, worker, workers);
        }
        uint32_t idesc = Cfg::kIdesc;
        if constexpr (Cfg::kRagN && !Cfg::kSwap) {
          // a group's last column tile: the MMA's N cut to the group's columns in it,
          // rounded up to 16 (the accumulator's other columns are never stored; swap-AB
          // tiles hold the columns on the MMA's M side)
          const TileCoord tc = decode_tile<Cfg>(sched, it.tile, 0u);
          const int32_t cols = tc.n_end - tc.n0;
          if (cols < Cfg::kTileN) idesc = ptx::idesc_e4m3_f32(Cfg::kMmaM, (cols + 15) & ~15);
        }
        uint32_t a_lo = a_lo0, b_lo = b_lo0;
        bool tr = false;  // CTA pairs: a transposed tile (a group's last <= 128 rows)
        if constexpr (Cfg::kPair) {
          const TileCoord tc = decode_tile<Cfg>(sched, it.tile, 0u);
          if (tc.half) {
            idesc = ptx::idesc_e4m3_f32(Cfg::kMmaM * Cfg::kCtas, tc.tr_n);
            a_lo = b_lo0;
            b_lo = a_lo0;
            tr = true;
          }
        }
        int32_t kb_end = it.kb1;
        int32_t k_len = 0;  // ragged K: the slice, counted from the first block's start
        int32_t k_skip = 0;
        if constexpr (Cfg::kRagK) {
          const TileCoord c = decode_tile<Cfg>(sched, it.tile, 0u);
          kb_end = c.nkb;
          k_skip = c.k_skip;
          k_len = c.k_skip + c.k_len;
        }
        for (int32_t kb0 = it.kb0; ok && kb0 < kb_end; kb0 += kpc) {
          if constexpr (Cfg::kBlockScale && !Cfg::kSwap) {
            if (kb_end - kb0 >= kUnrolledChunkKb) {
              // the next kUnrolledChunkKb blocks, one accumulator each, from the unrolled path
              if (!mma_bs_run_at<Cfg>(stage, static_cast<int>(chunk % Cfg::kNumAcc), p, s_bar,
                                      tmem_base, a_lo0, b_lo0, phase,
                                      (chunk / Cfg::kNumAcc) & 1u, abort_flag)) {
                ok = false;
                break;
              }
              const int adv = stage + kUnrolledChunkKb;
              stage = adv % Cfg::kStages;
              phase ^= static_cast<uint32_t>((adv / Cfg::kStages) & 1);
              chunk += kUnrolledChunkKb;
              kb0 += kUnrolledChunkKb - kpc;  // the loop adds kpc (= 1) back
              continue;
            }
          }
          const int buf = static_cast<int>(chunk % Cfg::kNumAcc);
          const uint32_t use = chunk / Cfg::kNumAcc;  // how often this buffer was used before
          if (!warp_agrees(wait_bar<Cfg::kPair>(tempty_bar(buf), (use & 1u) ^ 1u, abort_flag,
                                                p.status, p.timeout_ns))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after_sync();
          const uint32_t d_buf = tmem_base + static_cast<uint32_t>(buf * Cfg::kBufCols);
          const int32_t kb1 = min(kb_end, kb0 + kpc);
          if constexpr (kUnrolledMma) {
            if (kb1 - kb0 == kUnrolledChunkKb) {
              // a whole default-length chunk: the compile-time unrolled path
              if (!mma_chunk_at<Cfg>(stage, p, s_bar, s_wait, tfull_bar(buf), d_buf, idesc,
                                     a_lo, b_lo, phase, abort_flag)) {
                ok = false;
                break;
              }
              const int adv = stage + kUnrolledChunkKb;
              stage = adv % Cfg::kStages;
              phase ^= static_cast<uint32_t>((adv / Cfg::kStages) & 1);
              ++chunk;
              continue;
            }
          }
          for (int32_t kb = kb0; kb < kb1; ++kb) {
            if (!warp_agrees(wait_bar(s_wait + 8u * static_cast<uint32_t>(stage), phase,
                                      abort_flag, p.status, p.timeout_ns))) {
              ok = false;
              break;
            }
            // block scaling: K block kb0 + j sums into sub-accumulator j of the buffer, from
            // zero; otherwise the chunk's blocks all add into the one accumulator
            const uint32_t d_tmem =
                d_buf + (Cfg::kBlockScale ? static_cast<uint32_t>((kb - kb0) * Cfg::kAccCols) : 0u);
            const bool first_of_acc = Cfg::kBlockScale || kb == kb0;
            ptx::tc_fence_after_sync();
            const uint64_t act_desc = ptx::sw128_kmajor_desc(s_act + stage * Cfg::kActBytes);
            const uint64_t w_desc = ptx::sw128_kmajor_desc(s_w + stage * Cfg::kWBytes);
            const uint64_t a_desc = (Cfg::kSwap || tr) ? w_desc : act_desc;
            const uint64_t b_desc = (Cfg::kSwap || tr) ? act_desc : w_desc;
            int nmma = kBK / 32;
            if (kWarpWalks && kb == 0 && k_skip != 0) {
              // a slice that starts inside its first block: that block's MMAs come from
              // the out-of-line edge path
              mma_ragk_first_block<Cfg>(d_tmem, a_desc, b_desc, s_act + stage * Cfg::kActBytes,
                                        s_w + stage * Cfg::kWBytes, k_skip,
                                        min(kBK, k_len), lane);
              if (issuer) ptx::mma_commit(empty_bar(stage));
              if (++stage == Cfg::kStages) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            if constexpr (kWarpWalks) {
              // the last block of a K slice: the bytes past the slice belong to the next
              // group (or are TMA zero fill past total_K).  Whole 32-byte steps past it are
              // not issued; in a half-used step the unused 16 bytes of every row of both
              // operands are zeroed first (the slice ends on a 16-element boundary).
              const int32_t r = k_len - kb * kBK;
              if (r < kBK) {
                nmma = (r + 31) / 32;
                if (r & 16)
                  zero_stage_chunk<Cfg>(s_act + stage * Cfg::kActBytes,
                                        s_w + stage * Cfg::kWBytes,
                                        static_cast<uint32_t>(r >> 4), lane);
              }
            }
#pragma unroll
            for (int k = 0; k < kBK / 32; ++k) {
              if (k >= nmma || !issuer) break;
              // advance 32 bytes of K inside the 128-byte swizzled row: +2 in 16-byte units
              if constexpr (Cfg::kPair)
                ptx::mma_f8f6f4_pair(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc,
                                     (!first_of_acc || k > 0) ? 1u : 0u);
              else
                ptx::mma_f8f6f4(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc,
                                (!first_of_acc || k > 0) ? 1u : 0u);
            }
            // pairs: the stage is free in both CTAs once the MMAs reading it complete.
            // Block scaling (one K block = one stage per chunk) has one commit per block:
            // the epilogue frees the stage once it sees the chunk's accumulator commit.
            if constexpr (Cfg::kPair) ptx::mma_commit_pair(empty_bar(stage), 0x3);
            else if constexpr (!Cfg::kBlockScale) {
              if (issuer) ptx::mma_commit(empty_bar(stage));
            }
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if constexpr (Cfg::kPair) ptx::mma_commit_pair(tfull_bar(buf), 0x3);
          else if (issuer) ptx::mma_commit(tfull_bar(buf));
          ++chunk;
        }
      }
    }
    __syncwarp();
  } else if (Cfg::kEdgeWarp && warp == static_cast<uint32_t>(Cfg::kEdgeWarpIdx)) {
    // ------------------------------------------------------------------ ragged-K edges
    // Every stage in the MMA thread's order: wait (lane 0, bounded) until it is loaded,
    // zero the 16-byte chunks of every row of both operand tiles that lie outside the
    // tile's K slice (before the slice start in its first block, past its end in its last;
    // both operands, since 0 x NaN is NaN; 128-byte swizzle: chunk c of row r sits at
    // c ^ (r & 7)), make that visible to the tensor core and pass the stage on.
    if (has_k) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int32_t i = 0; ok && i < work.n_items; ++i) {
        const Item it = work_item(work, i, worker, workers);
        const TileCoord c = decode_tile<Cfg>(sched, it.tile, 0u);
        const int32_t k_end = c.k_skip + c.k_len;  // slice end, from the first block's start
        for (int32_t kb = it.kb0; kb < c.nkb; ++kb) {
          uint32_t got = 1u;
          if (lane == 0)
            got = wait_bar(full_bar(stage), phase, abort_flag, p.status, p.timeout_ns) ? 1u : 0u;
          if (__shfl_sync(0xffffffffu, got, 0) == 0u) {
            ok = false;
            break;
          }
          const uint32_t c_lo = kb == 0 ? static_cast<uint32_t>(c.k_skip) >> 4 : 0u;
          const int32_t hi = k_end - kb * kBK;
          const uint32_t c_hi = hi < kBK ? static_cast<uint32_t>(hi) >> 4 : 8u;
          if (c_lo > 0u || c_hi < 8u) {
            const uint32_t sa = s_act + static_cast<uint32_t>(stage * Cfg::kActBytes);
            const uint32_t sw = s_w + static_cast<uint32_t>(stage * Cfg::kWBytes);
            for (int row = static_cast<int>(lane); row < Cfg::kActRows + Cfg::kWRows; row += 32) {
              const uint32_t base = row < Cfg::kActRows ? sa + static_cast<uint32_t>(row) * 128u
                                                        : sw + static_cast<uint32_t>(row - Cfg::kActRows) * 128u;
              const uint32_t sw_row = static_cast<uint32_t>(row) & 7u;  // kActRows % 8 == 0
              for (uint32_t ch = 0; ch < 8u; ++ch)
                if (ch < c_lo || ch >= c_hi)
                  ptx::st_shared_v4(base + ((ch ^ sw_row) << 4), 0u, 0u, 0u, 0u);
            }
            ptx::fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ready_bar(stage));
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  }
  } else {
    if constexpr (Cfg::kRegSplit) ptx::setmaxnreg_inc<Cfg::kRegsHigh>();
    // ------------------------------------------------------------------ epilogue
    const uint32_t q = warp & 3u;  // TMEM lane quadrant this warp may access
    const uint32_t ew = warp - Cfg::kEpiWarp0;
    const int32_t col_base = static_cast<int32_t>(ew >> 2) * Cfg::kThreadCols;  // column slice
    if constexpr (Cfg::kDynamic) {
      // rows of each slab past its last computed tile: pure padding, written +0.0
      const int32_t gw = blockIdx.x * Cfg::kEpiWarps + ew;
      const int32_t nw = gridDim.x * Cfg::kEpiWarps;
      for (int32_t g = 0; g < p.G; ++g) {
        const int32_t v = rowinfo[g];
        const int32_t covered = tile_cover<Cfg>(v);
        const int32_t z0 = g * p.E + (covered < p.E ? covered : p.E);
        const int32_t z1 = (g + 1) * p.E;
        for (int32_t r = z0 + gw; r < z1; r += nw) {
          uint16_t* orow = p.out + static_cast<size_t>(r) * p.N;
          for (int32_t col = lane * 8; col < p.N; col += 256)
            if (ck_range(p, static_cast<int64_t>(r) * p.N + col, 8, ext_out_rows<Cfg>(p) * p.N))
              *reinterpret_cast<uint4*>(orow + col) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    uint32_t chunk = 0;
    uint32_t kbs_done = 0;  // block scaling: K blocks taken over (their stages freed)
    bool ok = true;
    const int32_t kpc = Cfg::kBlockScale ? Cfg::kBSSub : p.kb_per_chunk;
    for (int32_t i = 0; ok && (dyn || i < work.n_items); ++i) {
      Item it;
      if (dyn) {
        // lane 0 takes the item for the warp
        int32_t t = -1;
        bool took = true;
        if (lane == 0) t = tq_take(i, took);
        t = __shfl_sync(0xffffffffu, t, 0);
        took = __shfl_sync(0xffffffffu, took ? 1 : 0, 0) != 0;
        if (!took) {
          ok = false;
          break;
        }
        if (t < 0) break;
        it = whole_tile(t);
      } else {
        it = work_item(work, i, worker, workers);
      }
      TileCoord c = decode_tile<Cfg>(sched, it.tile, crank);
      // an empty reduction (K = 0) writes +0.0 to every owned row, whatever the scales
      if (!has_k) c.valid_end = c.m0;
      // a ragged-K tile contracting over nothing (an empty or skipped slice) is all +0.0
      const int32_t kb_end = Cfg::kRagK ? c.nkb : it.kb1;
      if (Cfg::kRagK && c.nkb == 0) c.valid_end = c.m0;
      // this warp's rows (row_off from c.m0) and output columns (ocol from c.n0).  A CTA
      // pair's transposed tile (a group's last <= 128 rows) leaves each CTA its 128 output
      // columns as TMEM lanes and the tile's rows (from c.m0) as TMEM columns from 0: the
      // four warps of column slice 0 (32 output columns each) hold it all, the others sit out
      int32_t row_off = static_cast<int32_t>(32u * q);
      int32_t ocol = col_base;
      bool active = true;
      const bool tr = Cfg::kPair && c.half;
      if constexpr (Cfg::kPair) {
        if (tr) active = col_base == 0;
      }
      // scales this thread needs, loaded before the chunk waits so their latency hides
      // behind the MMA: scale_a of its row, and scale_b of column (col0 + lane) for each
      // 32-column piece, broadcast by shuffle when the piece is stored
      float sa_pre = 0.0f;
      // block scaling: the scale of each K block (this thread's row x its columns' 128-block)
      // is loaded one chunk ahead, so its latency hides behind the chunk wait
      const float* bs_a = nullptr;
      const float* bs_b = nullptr;
      float bsa_next = 0.0f;  // the next K block's scale_a and scale_b, loaded a block ahead
      float bsb_next = 0.0f;  // and multiplied only when the block is drained
      // swap-AB: the next chunk's scales of each of its K blocks, loaded a chunk ahead
      float sw_bs_next[Cfg::kBSSub];
      float sw_row_next[Cfg::kBSSub];
#pragma unroll
      for (int j = 0; j < Cfg::kBSSub; ++j) sw_bs_next[j] = sw_row_next[j] = 0.0f;
      float sb_pre[Cfg::kSwap ? 1 : Cfg::kThreadCols / 32];
      // swap-AB: scale_b of this thread's weight row, and scale_a of row m0 + 32 pc + lane
      float sw_sb = 0.0f;
      float sw_sa[(Cfg::kTileN + 31) / 32];
      if constexpr (Cfg::kSwap && !Cfg::kBlockScale) {
        const int32_t n = c.n0 + static_cast<int32_t>(32u * q + lane);
        sw_sb = (n >= c.n_begin && n < c.n_end)
                    ? __ldg(p.scale_b + ck_index(p, c.sb_off + n, ext_scale_b<Cfg>(p), kCkScale))
                    : 0.0f;
#pragma unroll
        for (int pc = 0; pc < (Cfg::kTileN + 31) / 32; ++pc) {
          constexpr int kCols = Cfg::kTileN < 32 ? Cfg::kTileN : 32;
          const int32_t Rl = c.m0 + pc * 32 + static_cast<int32_t>(lane);
          sw_sa[pc] = (lane < static_cast<uint32_t>(kCols) && Rl < c.valid_end)
                          ? __ldg(p.scale_a + ck_index(p, Rl + c.srow_delta,
                                                       ext_scale_a<Cfg>(p), kCkScale))
                          : 0.0f;
        }
      }
      if constexpr (!Cfg::kSwap && !Cfg::kBlockScale) {
        if (Cfg::kPair && tr) {
          // a transposed tile: sa_pre holds scale_b of this thread's output column and
          // sb_pre[pc] scale_a of the tile's row 32 pc + lane (loaded here, ahead of the
          // chunk waits, so that nothing more stays live across the drains)
          const int32_t m_t = c.m0;
          const int32_t v_end = c.valid_end;  // (K = 0 set it to m0: every row +0.0)
          const int32_t n = c.n0 + static_cast<int32_t>(crank) * Cfg::kWRows +
                            static_cast<int32_t>(32u * q + lane);
          if (active && n < c.n_end)
            sa_pre = __ldg(ck_ptr(p, p.scale_b + c.sb_off + n, p.scale_b, ext_scale_b<Cfg>(p)));
#pragma unroll
          for (int pc = 0; pc < Cfg::kThreadCols / 32; ++pc) {
            const int32_t Rl = m_t + pc * 32 + static_cast<int32_t>(lane);
            sb_pre[pc] = (active && Rl < v_end)
                             ? __ldg(p.scale_a + ck_index(p, Rl + c.srow_delta,
                                                          ext_scale_a<Cfg>(p), kCkScale))
                             : 0.0f;
          }
        } else {
          const int32_t R = c.m0 + row_off + static_cast<int32_t>(lane);
          if (active && R < c.valid_end)
            sa_pre = __ldg(p.scale_a + ck_index(p, R + c.srow_delta, ext_scale_a<Cfg>(p), kCkScale));
          const float* sb_g = p.scale_b + c.sb_off;
#pragma unroll
          for (int pc = 0; pc < Cfg::kThreadCols / 32; ++pc) {
            const int32_t col = c.n0 + ocol + pc * 32 + static_cast<int32_t>(lane);
            sb_pre[pc] = (active && col < c.n_end)
                             ? __ldg(ck_ptr(p, sb_g + col, p.scale_b, ext_scale_b<Cfg>(p)))
                             : 0.0f;
          }
        }
      }
      if constexpr (Cfg::kBlockScale && !Cfg::kSwap) {
        // the K-block scales are applied chunk by chunk: the epilogue multiplies by 1
        const int32_t R = c.m0 + row_off + static_cast<int32_t>(lane);
        const bool rv = active && R < c.valid_end;
        const int32_t nblk = p.N / Cfg::kScaleBlock;
        bs_a = p.scale_a + static_cast<size_t>(rv ? R : 0) * p.num_kb;
        // (columns of a tile past N are never stored: clamp their block into range)
        const int32_t blk = min((c.n0 + ocol) / Cfg::kScaleBlock, nblk - 1);
        bs_b = p.scale_b + (static_cast<size_t>(c.g) * nblk + blk) * p.num_kb;
        if (rv && it.kb0 < kb_end) {
          bsa_next = __ldg(ck_ptr(p, bs_a + it.kb0, p.scale_a, ext_scale_a<Cfg>(p)));
          bsb_next = __ldg(ck_ptr(p, bs_b + it.kb0, p.scale_b, ext_scale_b<Cfg>(p)));
        }
        sa_pre = 1.0f;
#pragma unroll
        for (int pc = 0; pc < Cfg::kThreadCols / 32; ++pc) sb_pre[pc] = 1.0f;
      }
      // swap-AB with block scaling: this thread's weight row owns one 128-column block of
      // scale_b; lane j holds scale_a of activation row m0 + j (broadcast by shuffle)
      if constexpr (Cfg::kBlockScale && Cfg::kSwap) {
        const int32_t nw = c.n0 + static_cast<int32_t>(32u * q + lane);
        const int32_t nblk = p.N / Cfg::kScaleBlock;
        const int32_t blk = min(nw / Cfg::kScaleBlock, nblk - 1);
        bs_b = p.scale_b + (static_cast<size_t>(c.g) * nblk + blk) * p.num_kb;
        const int32_t Rl = c.m0 + static_cast<int32_t>(lane);
        const bool rv = lane < static_cast<uint32_t>(Cfg::kTileN) && Rl < c.valid_end;
        bs_a = p.scale_a + static_cast<size_t>(rv ? Rl : 0) * p.num_kb;
        if (it.kb0 < kb_end) {
#pragma unroll
          for (int j = 0; j < Cfg::kBSSub; ++j) {
            const int32_t kbj = min(it.kb0 + j, kb_end - 1);
            sw_bs_next[j] = __ldg(ck_ptr(p, bs_b + kbj, p.scale_b, ext_scale_b<Cfg>(p)));
            sw_row_next[j] = __ldg(ck_ptr(p, bs_a + kbj, p.scale_a, ext_scale_a<Cfg>(p)));
          }
        }
      }
      // fp32 accumulator of this thread (round-to-nearest adds of the TMEM chunks)
      float acc[Cfg::kThreadCols];
#pragma unroll
      for (int j = 0; j < Cfg::kThreadCols; ++j) acc[j] = 0.0f;
      // A split tile: the CTAs holding its K blocks (the owner, c_first, holds the first),
      // each piece's partial sums in the workspace (slot 0 of its CTA: the first tile of
      // that CTA's range, which every CTA after c_first starts inside this tile), and the
      // count the non-owners add themselves to.
      int32_t sk_first = 0, sk_last = 0;
      if (it.sk_tile >= 0) {
        const int64_t u_first = static_cast<int64_t>(it.sk_tile) * work.nkb;
        sk_first = unit_owner(work, u_first);
        sk_last = unit_owner(work, u_first + work.nkb - 1);
      }
      constexpr size_t kPerWarp = 32 * Cfg::kThreadCols;
      auto piece = [&](int32_t cta) -> float* {
        return p.sk_ws + (static_cast<size_t>(ck_index(p, cta, gridDim.x, kCkSplit) * 2) * Cfg::kEpiWarps +
                          ew) * kPerWarp;
      };
      uint32_t* const cnt =
          it.sk_tile >= 0 ? p.sk_cnt + static_cast<size_t>(ck_index(p, it.sk_tile, 2 * gridDim.x, kCkSplit)) *
                                           Cfg::kEpiWarps + ew
                          : nullptr;
      // The owner of a split tile whose other pieces are already counted in -- they are
      // their CTAs' first items and normally finished long before the owner's own piece --
      // loads them now (narrow TMA swap-AB accumulators: up to kPre pieces in registers), so
      // that after its own drain only the adds remain.
      constexpr int kPre = (Cfg::kTma && Cfg::kThreadCols <= 32) ? 64 / Cfg::kThreadCols : 0;
      float pre[kPre > 0 ? kPre : 1][Cfg::kThreadCols];
      int32_t n_pre = 0;  // pieces loaded early
      if constexpr (kPre > 0) {
        if (it.sk_tile >= 0 && static_cast<int32_t>(blockIdx.x) == sk_first &&
            sk_last - sk_first <= kPre) {
          uint32_t ready = 0;
          if (lane == 0)
            ready = ptx::ld_acquire_gpu_u32(cnt) >= static_cast<uint32_t>(sk_last - sk_first);
          ready = __shfl_sync(0xffffffffu, ready, 0);
          __syncwarp();
          if (ready) {
#pragma unroll
            for (int b = 0; b < kPre; ++b) {
              if (b < sk_last - sk_first) {
                const float* src = piece(sk_first + 1 + b) + lane;
#pragma unroll
                for (int j = 0; j < Cfg::kThreadCols; ++j) pre[b][j] = __ldcg(src + j * 32);
              }
            }
            n_pre = sk_last - sk_first;
          }
        }
      }
      // TMEM data is needed only when this warp's lanes hold rows with computed values
      bool warp_any;
      if constexpr (!Cfg::kSwap) {
        warp_any = active && (tr || c.m0 + row_off < c.valid_end);  // lane 0's row
      } else {
        warp_any = c.n0 + static_cast<int32_t>(32u * q) < p.N && c.m0 < c.valid_end;
      }
      if (has_k) {
        for (int32_t kb0 = it.kb0; kb0 < kb_end; kb0 += kpc) {
          const int buf = static_cast<int>(chunk % Cfg::kNumAcc);
          const uint32_t use = chunk / Cfg::kNumAcc;
          const int32_t nsub = min(kpc, kb_end - kb0);  // K blocks in this chunk
          // block scaling: the scale of K block kb0 (128-row tiles), or of each of the
          // chunk's blocks (swap-AB), loaded one chunk ahead
          float bs = 1.0f;      // this thread's scale of the block (swap-AB: its column's)
          float bs_row = 0.0f;  // swap-AB: lane j's activation-row scale
          float sub_bs[Cfg::kBSSub];
          float sub_row[Cfg::kBSSub];
          if constexpr (Cfg::kBlockScale && Cfg::kSwap) {
            // this chunk's scales were loaded a chunk ago; the next chunk's go out now
#pragma unroll
            for (int j = 0; j < Cfg::kBSSub; ++j) {
              sub_bs[j] = sw_bs_next[j];
              sub_row[j] = sw_row_next[j];
            }
            if (kb0 + kpc < kb_end) {
#pragma unroll
              for (int j = 0; j < Cfg::kBSSub; ++j) {
                const int32_t kbj = min(kb0 + kpc + j, kb_end - 1);
                sw_bs_next[j] = __ldg(ck_ptr(p, bs_b + kbj, p.scale_b, ext_scale_b<Cfg>(p)));
                sw_row_next[j] = __ldg(ck_ptr(p, bs_a + kbj, p.scale_a, ext_scale_a<Cfg>(p)));
              }
            }
          } else if constexpr (Cfg::kBlockScale) {
            // (the product is taken here, a block after its loads were issued, so that the
            // loads' latency never holds up the wait and drain below)
            bs = bsa_next * bsb_next;
            if (kb0 + 1 < kb_end && bs_a != nullptr) {
              bsa_next = __ldg(ck_ptr(p, bs_a + kb0 + 1, p.scale_a, ext_scale_a<Cfg>(p)));
              bsb_next = __ldg(ck_ptr(p, bs_b + kb0 + 1, p.scale_b, ext_scale_b<Cfg>(p)));
            }
          }
          // scale of accumulator column j (block scaling; swap-AB: row j's times column's)
          auto cs = [&](int j) -> float {
            if constexpr (Cfg::kBlockScale && Cfg::kSwap)
              return __shfl_sync(0xffffffffu, bs_row, j) * bs;
            else
              return bs;
          };
          if (!wait_bar(tfull_bar(buf), use & 1u, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          // block scaling: the chunk's K blocks are this CTA's blocks kbs_done.. and lived in
          // the stages of those numbers mod kStages, whose MMAs have completed -- one lane
          // frees them for the loader
          if constexpr (Cfg::kBlockScale) {
            if (ew == 0 && lane == 0)
              for (int32_t j = 0; j < nsub; ++j)
                ptx::mbar_arrive(empty_bar(static_cast<int>((kbs_done + j) % Cfg::kStages)));
            kbs_done += static_cast<uint32_t>(nsub);
          }
          ptx::tc_fence_after_sync();
          if (warp_any) {
            const uint32_t t_buf = tmem_base + ((32u * q) << 16) +
                                   static_cast<uint32_t>(buf * Cfg::kBufCols + col_base);
            // one accumulator at t_acc into the fp32 registers (with the scale in bs / cs)
            auto drain = [&](uint32_t t_acc) {
              if constexpr (Cfg::kRegSplit && Cfg::kThreadCols % 64 == 0) {
                // two 32-column loads in flight per wait
#pragma unroll
                for (int pc = 0; pc < Cfg::kThreadCols / 64; ++pc) {
                  uint32_t v0[32], v1[32];
                  ptx::tmem_ld_x32(t_acc + static_cast<uint32_t>(pc * 64), v0);
                  ptx::tmem_ld_x32(t_acc + static_cast<uint32_t>(pc * 64 + 32), v1);
                  ptx::tmem_ld_wait();
#pragma unroll
                  for (int j = 0; j < 32; j += 2) {
                    accum2<Cfg::kBlockScale>(acc[pc * 64 + j], acc[pc * 64 + j + 1], v0[j],
                                             v0[j + 1], bs, bs);
                    accum2<Cfg::kBlockScale>(acc[pc * 64 + 32 + j], acc[pc * 64 + 33 + j], v1[j],
                                             v1[j + 1], bs, bs);
                  }
                }
              } else if constexpr (Cfg::kThreadCols % 32 == 0 && Cfg::kThreadCols < 128) {
                // 128 accumulators per thread leave no room for 32 more load registers at
                // the 168-register limit of 10+ warps: those drain 16 columns at a time
#pragma unroll
                for (int pc = 0; pc < Cfg::kThreadCols / 32; ++pc) {
                  uint32_t v[32];
                  ptx::tmem_ld_x32(t_acc + static_cast<uint32_t>(pc * 32), v);
                  ptx::tmem_ld_wait();
#pragma unroll
                  for (int j = 0; j < 32; j += 2)
                    accum2<Cfg::kBlockScale>(acc[pc * 32 + j], acc[pc * 32 + j + 1], v[j], v[j + 1],
                                             cs(pc * 32 + j), cs(pc * 32 + j + 1));
                }
              } else {
#pragma unroll
                for (int pc = 0; pc < Cfg::kThreadCols / 16; ++pc) {
                  uint32_t v[16];
                  ptx::tmem_ld_x16(t_acc + static_cast<uint32_t>(pc * 16), v);
                  ptx::tmem_ld_wait();
#pragma unroll
                  for (int j = 0; j < 16; j += 2)
                    accum2<Cfg::kBlockScale>(acc[pc * 16 + j], acc[pc * 16 + j + 1], v[j], v[j + 1],
                                             cs(pc * 16 + j), cs(pc * 16 + j + 1));
                }
              }
            };
            if constexpr (Cfg::kBlockScale && Cfg::kSwap) {
#pragma unroll
              for (int j = 0; j < Cfg::kBSSub; ++j) {
                if (j < nsub) {
                  bs = sub_bs[j];
                  bs_row = sub_row[j];
                  drain(t_buf + static_cast<uint32_t>(j * Cfg::kAccCols));
                }
              }
            } else {
              drain(t_buf);
            }
          }
          ptx::tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            if constexpr (Cfg::kPair) ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(buf), 0u));
            else ptx::mbar_arrive(tempty_bar(buf));
          }
          ++chunk;
        }
        if (!ok) break;
      }
      if (it.sk_tile >= 0) {
        // One piece of a split tile.  The tile's owner is the CTA whose piece holds its first
        // K block (c_first); every other piece is the first split item of its CTA, whose
        // epilogue warps publish their partial sums and count themselves in.  The owner's
        // warps keep theirs in registers, wait (bounded) for the others' counts and add the
        // pieces in CTA order -- ((p_first + p_next) + ...) + p_last -- and store the tile.
        // (No cycle: a non-owner piece is processed before any wait of its CTA.)
        const int32_t c_first = sk_first;
        const int32_t c_last = sk_last;
        if (static_cast<int32_t>(blockIdx.x) != c_first) {
          float* mine = piece(blockIdx.x) + lane;
#pragma unroll
          for (int j = 0; j < Cfg::kThreadCols; ++j) __stcg(mine + j * 32, acc[j]);
          // the warp barrier orders every lane's stores before lane 0's count, which
          // releases them at GPU scope
          __syncwarp();
          if (lane == 0) ptx::red_add_release_gpu(cnt, 1u);
          continue;
        }
        if constexpr (kPre > 0) {
          if (n_pre > 0) {
#pragma unroll
            for (int b = 0; b < kPre; ++b) {
              if (b < n_pre) {
#pragma unroll
                for (int j = 0; j < Cfg::kThreadCols; ++j) acc[j] += pre[b][j];
              }
            }
          }
        }
        if (n_pre == 0) {
          // the owner: its count acquires the others' releases; the warp barrier after it
          // hands them on to every lane
          uint32_t got_all = 1u;
          if (lane == 0)
            got_all = wait_count(cnt, static_cast<uint32_t>(c_last - c_first), abort_flag,
                                 p.status, p.timeout_ns) ? 1u : 0u;
          got_all = __shfl_sync(0xffffffffu, got_all, 0);
          if (!got_all) {
            ok = false;
            break;
          }
          __syncwarp();
          // the other pieces added to the owner's in CTA order; the loads of up to kBatch
          // pieces are in flight together before their adds
          constexpr int kBatch = Cfg::kThreadCols >= 64 ? 1 : 64 / Cfg::kThreadCols;
          if constexpr (kBatch == 1) {
            // wide accumulators: no registers to spare, one piece at a time
            for (int32_t cta = c_first + 1; cta <= c_last; ++cta) {
              const float* src = piece(cta) + lane;
#pragma unroll
              for (int j = 0; j < Cfg::kThreadCols; ++j) acc[j] += __ldcg(src + j * 32);
            }
          } else {
            for (int32_t c0 = c_first + 1; c0 <= c_last; c0 += kBatch) {
              float v[kBatch][Cfg::kThreadCols];
#pragma unroll
              for (int b = 0; b < kBatch; ++b) {
                if (c0 + b <= c_last) {
                  const float* src = piece(c0 + b) + lane;
#pragma unroll
                  for (int j = 0; j < Cfg::kThreadCols; ++j) v[b][j] = __ldcg(src + j * 32);
                }
              }
#pragma unroll
              for (int b = 0; b < kBatch; ++b) {
                if (c0 + b <= c_last) {
#pragma unroll
                  for (int j = 0; j < Cfg::kThreadCols; ++j) acc[j] += v[b][j];
                }
              }
            }
          }
        }
        if (lane == 0) *cnt = 0u;  // ready for the next call
      }
      if (!active) continue;
      if constexpr (Cfg::kPair) {
        if (tr) {
          // thread = output column n (its TMEM lane), acc[j] = the tile's row m_t + j.  For
          // each pair of rows, lanes 2i and 2i + 1 trade one value, so that each lane stores
          // two adjacent columns of one row: even lanes row 2k, odd lanes row 2k + 1
          // (scales: sa_pre = this column's scale_b, sb_pre[pc] = scale_a of row 32 pc + lane)
          const int32_t m_t = c.m0;
          const int32_t v_end = c.valid_end;  // (K = 0 set it to m0: every row +0.0)
          const bool odd = (lane & 1u) != 0u;
          // the first of the two columns this lane stores (N % 8 == 0: both in range)
          const int32_t n_st = c.n0 + static_cast<int32_t>(crank) * Cfg::kWRows +
                               static_cast<int32_t>(32u * q + (lane & ~1u));
          const float sb = sa_pre;
#pragma unroll
          for (int pc = 0; pc < Cfg::kThreadCols / 32; ++pc) {
            const int32_t r0 = m_t + pc * 32;
            if (r0 >= c.zero_end) break;
            const float sa_l = sb_pre[pc];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float y0 = (acc[pc * 32 + 2 * k] * __shfl_sync(0xffffffffu, sa_l, 2 * k)) * sb;
              const float y1 =
                  (acc[pc * 32 + 2 * k + 1] * __shfl_sync(0xffffffffu, sa_l, 2 * k + 1)) * sb;
              const float other = __shfl_xor_sync(0xffffffffu, odd ? y0 : y1, 1);
              const int32_t R = r0 + 2 * k + (odd ? 1 : 0);
              if (R < c.zero_end && n_st < c.n_end) {
                const int64_t o_idx = static_cast<int64_t>(R + c.orow_delta) * p.N + n_st;
                if (ck_range(p, o_idx, 2, ext_out_rows<Cfg>(p) * p.N))
                  *reinterpret_cast<uint32_t*>(p.out + o_idx) =
                      R < v_end ? (odd ? pack_bf16x2(other, y1) : pack_bf16x2(y0, other)) : 0u;
              }
            }
          }
          continue;
        }
      }
      if constexpr (!Cfg::kSwap) {
        // thread = one activation row
        const int32_t R = c.m0 + row_off + static_cast<int32_t>(lane);
        const bool row_val = R < c.valid_end;
        const bool row_zero = !row_val && R < c.zero_end;
        const int32_t R_first = c.m0 + row_off;
        // TMA stores clip at the output's last column only: a block that reaches outside a
        // ragged-N group's columns takes the predicated path
        if (Cfg::kTmaStore && R_first + 31 < c.zero_end && c.n0 + ocol >= c.n_begin &&
            (c.n_end == p.N || c.n0 + ocol + Cfg::kThreadCols <= c.n_end)) {
          // all 32 rows of this warp are owned: stage 32 x 32 bf16 blocks in shared memory
          // (64-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ ((r >> 1) & 3))
          // and let one lane store each block with TMA (whole lines, clipped at N)
          const uint32_t stg = s_out + ew * Cfg::kStageOutBytes;
#pragma unroll
          for (int pc = 0; pc < Cfg::kThreadCols / 32; ++pc) {
            const int32_t col0 = c.n0 + ocol + pc * 32;
            const float sb_l = sb_pre[pc];
            // the block's 32 columns scaled and packed first, while the previous block's TMA
            // store may still be reading the staging buffer
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float sb0 = __shfl_sync(0xffffffffu, sb_l, 2 * j);
              const float sb1 = __shfl_sync(0xffffffffu, sb_l, 2 * j + 1);
              w[j] = row_val ? pack_bf16x2((acc[pc * 32 + 2 * j] * sa_pre) * sb0,
                                           (acc[pc * 32 + 2 * j + 1] * sa_pre) * sb1)
                             : 0u;
            }
            if (lane == 0) ptx::bulk_wait_read_all();  // staging buffer free again
            __syncwarp();
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {  // 8 columns = one 16-byte chunk at a time
              const uint32_t a = stg + lane * 64u + ((static_cast<uint32_t>(ch) ^ ((lane >> 1) & 3u)) << 4);
              ptx::st_shared_v4(a, w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 &&
                ck_tma_store(p, col0, R_first + c.orow_delta, ext_out_rows<Cfg>(p), p.N)) {
              ptx::tma_store_2d(&tmC, stg, col0, R_first + c.orow_delta);
              ptx::bulk_commit();
            }
          }
        } else if (__any_sync(0xffffffffu, row_val || row_zero)) {
          // 8 output columns per 16-byte store, predicated per row and on the last column
          const float sa = sa_pre;
          uint16_t* orow =
              p.out + static_cast<size_t>(row_val || row_zero ? R + c.orow_delta : 0) * p.N;
#pragma unroll
          for (int pc = 0; pc < Cfg::kThreadCols / 32; ++pc) {
            const int32_t col0 = c.n0 + ocol + pc * 32;
            const float sb_l = sb_pre[pc];
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8) {
              float y[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float sb = __shfl_sync(0xffffffffu, sb_l, j8 * 8 + j);
                y[j] = (acc[pc * 32 + j8 * 8 + j] * sa) * sb;
              }
              const int32_t col = col0 + j8 * 8;  // a multiple of 8: 16-byte aligned
              const int64_t o_idx = static_cast<int64_t>(R + c.orow_delta) * p.N + col;
              if (col + 7 < c.n_end && col >= c.n_begin) {
                if ((row_val || row_zero) &&
                    ck_range(p, o_idx, 8, ext_out_rows<Cfg>(p) * p.N)) {
                  if (row_val) {
                    *reinterpret_cast<uint4*>(orow + col) =
                        make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                   pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
                  } else {
                    *reinterpret_cast<uint4*>(orow + col) = make_uint4(0u, 0u, 0u, 0u);
                  }
                }
              } else if (Cfg::kRagN && row_val && col < c.n_end && col + 7 >= c.n_begin) {
                // a ragged-N group starting or ending inside these 8 columns: its own
                // columns one by one
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (col + j >= c.n_begin && col + j < c.n_end &&
                      ck_range(p, o_idx + j, 1, ext_out_rows<Cfg>(p) * p.N))
                    orow[col + j] = __bfloat16_as_ushort(__float2bfloat16_rn(y[j]));
              }
            }
          }
        }
      } else {
        // thread = one weight row (output column n); accumulator columns are activation rows
        const int32_t n = c.n0 + static_cast<int32_t>(32u * q + lane);
        const bool col_ok = n >= c.n_begin && n < c.n_end;
        // block scaling: the scales were applied chunk by chunk
        const float sb = Cfg::kBlockScale ? 1.0f : sw_sb;
#pragma unroll
        for (int pc = 0; pc < (Cfg::kTileN + 31) / 32; ++pc) {
          constexpr int kCols = Cfg::kTileN < 32 ? Cfg::kTileN : 32;
          const int32_t m_first = c.m0 + pc * 32;
          if (m_first >= c.zero_end) break;
          // lane j holds scale_a of row m_first + j
          const float sa_l = Cfg::kBlockScale ? 1.0f : sw_sa[pc];
#pragma unroll
          for (int j = 0; j < kCols; ++j) {
            const float sa = __shfl_sync(0xffffffffu, sa_l, j);
            const int32_t R = m_first + j;
            if (R < c.valid_end) {
              const float y = (acc[pc * 32 + j] * sa) * sb;
              if (col_ok && ck_range(p, static_cast<int64_t>(R + c.orow_delta) * p.N + n, 1,
                                     ext_out_rows<Cfg>(p) * p.N))
                p.out[static_cast<size_t>(R + c.orow_delta) * p.N + n] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(y));
            } else if (R < c.zero_end) {
              if (col_ok && ck_range(p, static_cast<int64_t>(R + c.orow_delta) * p.N + n, 1,
                                     ext_out_rows<Cfg>(p) * p.N))
                p.out[static_cast<size_t>(R + c.orow_delta) * p.N + n] = 0;
            }
          }
        }
      }
    }
  }

  if constexpr (Cfg::kTmaStore) {
    if (warp >= static_cast<uint32_t>(Cfg::kEpiWarp0) && lane == 0) ptx::bulk_wait_all();
  }

  // ------------------------------------------------------------------ teardown
  ptx::tc_fence_before_sync();
  __syncthreads();
  bool aborting = *abort_flag != 0u;
  if constexpr (Cfg::kPair) {
    // neither CTA of a pair leaves while the other may still signal its barriers or read
    // its shared memory, and both wait out in-flight work if either gave up
    ptx::cluster_sync();
    const uint32_t peer_abort = ptx::ld_shared_cluster_u32(
        ptx::mapa_shared(ptx::smem_addr(smem + Cfg::kOffMisc + 4), crank ^ 1u));
    aborting = aborting || peer_abort != 0u;
    ptx::cluster_sync();
    // the last leader to get here (every claim is made by then) resets the claim counter
    // for the next call; teardown runs on the abort path too
    if (dyn && crank == 0 && threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(p.tile_ctr + 1, 1u) == static_cast<uint32_t>(workers - 1)) {
        volatile uint32_t* ctr = p.tile_ctr;
        ctr[0] = 0u;
        ctr[1] = 0u;
        __threadfence();
      }
    }
  }
  if (aborting) {
    // let any copy or MMA still in flight land before the memory is released
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 2000000ull) ptx::nanosleep(1000);
  }
  if (warp == static_cast<uint32_t>(Cfg::kMmaWarp)) {
    ptx::tc_fence_after_sync();
    if constexpr (Cfg::kPair) ptx::tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    else ptx::tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace mslkb
