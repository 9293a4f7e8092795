// mx_cast.cu -- persistent, warp-specialised MX-FP8 cast kernels for sm_103a.
//
// One pass over a bf16 matrix X (M x K, row-major) writes
//   q0  (M x K)  e4m3, blocks of 32 along rows     ("dim0")
//   q1  (K x M)  e4m3, blocks of 32 along columns  ("dim1", X's column-major copy)
// and the e8m0 scales of both, already in the 128x4 blocked layout that
// block-scaled GEMMs read.  This is the fused cast of pytorch/ao PR #1869
// "triton kernel to cast to mx across dim0 and dim1" (summary: read each tile
// once, write both copies and their scales from it), with the future-work
// items of that summary built in: an outer tile of 128, scales written
// swizzled, and coalesced writes of the column-major copy.  The grouped-M and
// 3D variants follow pytorch/ao PR #2990 "[mxfp8 moe training] add compile
// support" (padding bound rows + groups*128 with no host sync; 3D weights cast
// as the reshaped 2D matrix).
//
// Tile = 128 rows x 128 columns of X.  Such a tile yields exactly one 512-byte
// 128x4 blocked scale tile per direction, so the swizzle costs nothing.
//
// CTA roles (one CTA per SM, persistent over tiles):
//   warps 0-7  compute: dim0 and dim1 block maxima, scales, e4m3 packing.
//              dim0 bytes go straight to global memory (each warp store
//              writes four whole 128-byte rows of q0); dim1 bytes go to a
//              swizzled shared-memory staging tile
//   warp 8     producer: TMA loads of the bf16 tile (two 64-column halves,
//              128B swizzle) into a kStages-deep ring
//   warp 9     storer: TMA stores of the staged q1 tile, bulk copy of the
//              dim0 scale tile, and the dim1 scale tile (staged in plain
//              order, transposed to the blocked order on the way out);
//              grouped mode: warps 9-12, one lane per q1 row, which first
//              shift misaligned rows onto 16-byte chunks in place (group
//              starts are not 16-byte aligned) or copy strip edges out with
//              plain stores
// Modes (template kMode): fused 2D, dim0 only, dim1 only, the 3D per-expert
// forms of the three, and grouped-M; see the Mode enum.
// The depths were chosen by measurement on GB300: few input stages and many
// output staging buffers.  More loads in flight (4-5 stages) slowed the
// kernel by ~12%: outstanding writes, not reads, limit the mixed stream.
// Every wait is bounded (see mbar_wait); on time-out the CTA raises an abort
// flag, stops, lets its own copies in flight land (the TMA loads into its
// input ring and the bulk stores out of its staging) and reports through a
// device word.
#include <cuda_runtime.h>

#include <mutex>

#include "mx_common.cuh"
#include "mx_kernels.h"

namespace mx {

// Device-side watchdog word: set when any CTA gave up waiting.
__device__ int g_watchdog = 0;
// Claim counters (kClaim launches), one per stream in use (claim_counter).
constexpr int kClaimSlots = 64;
__device__ unsigned int g_claims[kClaimSlots];

namespace {

constexpr int kTile = 128;
constexpr int kHalfBytes = 128 * 128;      // 64 bf16 columns x 128 rows
constexpr int kInBytes = 2 * kHalfBytes;    // one bf16 tile
constexpr int kQBytes = 128 * 128;          // one e4m3 tile
constexpr int kQ1Half = 64 * 128;           // even / odd columns of a q1 tile
constexpr int kScaleTile = 512;
constexpr int kStages = 3;                 // input ring depth
constexpr int kStaging = 6;                // q1 / scale staging buffers
// claim schedule (mx_cast_kernel): the last kClaimRounds rounds are claimed,
// for launches of at least kClaimMinRounds rounds (fewer: static).  At
// 16384^2 (108 rounds) it takes 165.6 -> 164.6 us; claiming 6, 10 or 16
// rounds measured alike; at 8192^2 (27 rounds) it cost 0.65 us.
constexpr int64_t kClaimRounds = 6;
constexpr int64_t kClaimMinRounds = 32;
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kProducerWarp = kComputeWarps;
constexpr int kFirstStoreWarp = kComputeWarps + 1;

// Shared-memory layout, offsets from a 1024-byte aligned base (the 128B
// swizzle pattern repeats every 1024 bytes).
constexpr int kOffIn = 0;
constexpr int kOffQ1 = kOffIn + kStages * kInBytes;
constexpr int kOffS0 = kOffQ1 + kStaging * kQBytes;
constexpr int kOffS1 = kOffS0 + kStaging * kScaleTile;
// group table in smem up to kMaxSmemGroups groups (mx_kernels.h)
constexpr int kOffGTab = kOffS1 + kStaging * kScaleTile;
constexpr int kGTabBytes = ((2 * kMaxSmemGroups + 1) * 4 + 127) / 128 * 128;
constexpr int kOffBar = kOffGTab + kGTabBytes;
constexpr int kNumBars = 2 * kStages + 2 * kStaging + 1;   // + the diagnostic stall barrier
constexpr int kQ1GroupBoxRows = static_cast<int>(kQ1BoxRowsGrouped);  // grouped: per-warp q1 box rows
constexpr int kOffFlag = kOffBar + kNumBars * 8;
// claim schedule: the tile of each input stage and staging buffer, as the
// producer chose it (-1: no more tiles)
constexpr int kOffIds = kOffFlag + 16;     // flag: abort (+0), bad group offsets (+4)
constexpr int kSmemUsed = kOffIds + (kStages + kStaging) * 8;
constexpr int kStatusBadGroups = -5;        // MX_ERR_GROUPS
constexpr int kSmemBytes = kSmemUsed + 1024;

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// Modes: which copies a launch writes and where its scale tiles go.
//   kModeFused2D   dim0 + dim1, 2D blocked scales
//   kModeDim1      dim1 only
//   kModeDim0      dim0 only
//   kModeExperts   3D weights (E, N, K) as the (E*N, K) matrix: dim1, each
//                  expert's scales blocked on their own
//   kModeExperts0  the same for dim0
//   kModeExperts01 the same for dim0 + dim1
//   kModeGrouped   grouped-M activations: dim0 + dim1 per group
//   kModeGroupedBands  the same, with tall groups walked in bands (see
//                  GroupCursor); a separate instantiation, so that shapes
//                  whose runs are too short for bands pay nothing for them
enum Mode : int {
  kModeFused2D = 0, kModeDim1 = 1, kModeExperts = 2, kModeGrouped = 3, kModeGroupedBands = 7,
  kModeDim0 = 4, kModeExperts0 = 5, kModeExperts01 = 6
};
__host__ __device__ constexpr bool has_dim0(int m) {
  return m == kModeFused2D || m == kModeGrouped || m == kModeGroupedBands || m == kModeDim0 ||
         m == kModeExperts0 ||
         m == kModeExperts01;
}
__host__ __device__ constexpr bool has_dim1(int m) { return m != kModeDim0 && m != kModeExperts0; }
__host__ __device__ constexpr bool per_expert(int m) {
  return m == kModeExperts || m == kModeExperts0 || m == kModeExperts01;
}

// One store warp drains a staging buffer by TMA in the 2D / 3D modes.  In
// the grouped mode q1 cannot leave by TMA (group starts are not 16-byte
// aligned), so four store warps copy it out with plain stores, off the
// compute warps' path.
__host__ __device__ constexpr bool is_grouped(int m) { return m == kModeGrouped || m == kModeGroupedBands; }
__host__ __device__ constexpr int store_warps(int mode) { return is_grouped(mode) ? 4 : 1; }
__host__ __device__ constexpr int threads_of(int mode) {
  return (kComputeWarps + 1 + store_warps(mode)) * 32;
}

struct Tile {
  int32_t m0;       // first row of X
  int32_t k0;       // first column of X
  int32_t rows;     // rows of the tile that belong to it (grouped mode), else 128
  int32_t cont;     // grouped: bit 0 = previous tile of this CTA is the one above in
                    // the same column strip, bit 1 = next tile is the one below
  int32_t next_rows;  // grouped: rows of the tile below in the strip (when cont bit 1)
  uint8_t* s0_dst;  // 512-byte blocked tile for dim0 scales
  uint8_t* s1_dst;  // 512-byte blocked tile for dim1 scales (null: scattered)
};

struct Params {
  int64_t M, K;
  int32_t n_mt, n_kt;       // tiles along M and K
  int64_t n_tiles;          // 2D / 3D modes
  uint8_t* s0;
  uint8_t* s1;
  uint8_t* q0;              // dim0 data, written directly
  uint8_t* q1;              // grouped mode: plain stores of q1
  // experts (3D)
  int64_t N;                // rows per expert
  int64_t s1_expert_bytes;  // blk(K, N/32)
  int32_t s1_scatter;       // N % 128 != 0: scales written byte by byte
  int32_t nb4;              // ceil4(N / 32)
  int64_t s0_expert_bytes;  // blk(N, K/32)
  int32_t s0_scatter;       // N % 128 != 0: dim0 scales written byte by byte
  int32_t kb4;              // ceil4(K / 32)
  // grouped
  const int32_t* offs;
  const int64_t* row_offs;  // s0_row_offs (G + 1), from group_offsets_kernel (G > kMaxSmemGroups)
  const int32_t* status;
  int64_t* row_offs_out;    // G <= kMaxSmemGroups: written by CTA 0 of this kernel
  int64_t* col_offs_out;
  int32_t* status_out;
  int32_t G;
  int32_t k128;             // ceil128(K)
  int32_t q1_tma;           // grouped: q1 rows 16-byte aligned (M % 16 == 0), so
                            // whole 128-byte tiles may leave by TMA
  // output buffers, for the bounds-checked build's store checks
  Span sp_q0, sp_q1, sp_s0, sp_s1, sp_ro, sp_co, sp_st;
  // diagnostic stall (mx_kernels.h): CTA 0's producer at run position
  // stall_at, -1 in normal use
  int64_t stall_at;
  uint64_t stall_ns;
  // 2D / 3D modes with the claim schedule: this launch's tile counter (one
  // word of g_claims, zero between launches)
  unsigned int* claims;
};

// Group table of the grouped mode: tr[g] = padded tile-rows before group g
// (s0_row_offs[g] / 128), ends[g] = offs[g].  Cached in shared memory when
// G <= kMaxSmemGroups, else read from global memory.
struct GroupTab {
  const int32_t* tr_s;      // smem copy or null
  const int32_t* ends_s;
  const int64_t* row_offs;  // global
  const int32_t* ends;
  __device__ __forceinline__ int64_t tr(int g) const {
    return tr_s ? static_cast<int64_t>(tr_s[g]) : (row_offs[g] >> 7);
  }
  __device__ __forceinline__ int64_t end(int g) const {
    return ends_s ? static_cast<int64_t>(ends_s[g]) : static_cast<int64_t>(ends[g]);
  }
};



// q = a / b, r = a - q * b for non-negative a and positive b, in 32 bits
// when both fit (always, for tile counts of buffers that fit in memory).
// Used by the grouped schedule; the 2D and 3D schedules keep the plain
// division (with 32-bit division and counters the 3D kernel measured 3.6%
// slower).
__device__ __forceinline__ int64_t div_tiles(int64_t a, int64_t b, int64_t& r) {
  if (((a | b) >> 32) == 0) {
    const uint32_t q = static_cast<uint32_t>(a) / static_cast<uint32_t>(b);
    r = a - static_cast<int64_t>(q) * b;
    return q;
  }
  const int64_t q = a / b;
  r = a - q * b;
  return q;
}

// Per-role tile counter: 32-bit in the grouped mode (1.6 us faster at
// 16640 x 5120, G = 4, measured against the 64-bit counter).
template <int M> struct ItType { using T = int64_t; };
template <> struct ItType<kModeGrouped> { using T = uint32_t; };
template <> struct ItType<kModeGroupedBands> { using T = uint32_t; };

// Tile t of the launch in the 2D / 3D modes: row-major over (M tiles, K tiles).
template <int kMode>
__device__ __forceinline__ Tile get_tile(const Params& p, const GroupTab& tab, int64_t t) {
  Tile T;
  T.cont = 0;
  T.next_rows = 0;
  {
    const int32_t tm = static_cast<int32_t>(t / p.n_kt);
    const int32_t tk = static_cast<int32_t>(t - static_cast<int64_t>(tm) * p.n_kt);
    T.m0 = tm * kTile;
    T.k0 = tk * kTile;
    T.rows = kTile;
    // Per-expert dim0 scales with N % 128 == 0 sit exactly where the 2D
    // layout puts them (expert e's blk(N, K/32) bytes start at tile row e*N/128).
    T.s0_dst = has_dim0(kMode) && !(per_expert(kMode) && p.s0_scatter) ? p.s0 + t * kScaleTile
                                                                       : nullptr;
    if (!has_dim1(kMode)) {
      T.s1_dst = nullptr;
    } else if (per_expert(kMode)) {
      if (p.s1_scatter) {
        T.s1_dst = nullptr;
      } else {
        const int64_t e = T.m0 / p.N;
        const int64_t nt = (T.m0 - e * p.N) >> 7;
        T.s1_dst = p.s1 + e * p.s1_expert_bytes + (tk * (p.N >> 7) + nt) * kScaleTile;
      }
    } else {
      T.s1_dst = p.s1 + (static_cast<int64_t>(tk) * p.n_mt + tm) * kScaleTile;
    }
  }
  return T;
}

// Grouped mode: tiles are ordered by group, then K tile, then M tile within
// the group, so that a CTA's contiguous run of tiles walks down one column
// strip of a group (this lets q1 rows be written in whole 16-byte chunks, see
// copy_out_q1).  A group much taller than a run is cut into bands of tile-rows
// as tall as a run (band, then K tile, then M tile within the band): the 152
// runs in flight then cover whole tile-rows of X instead of one strip segment
// each from all over the matrix (131072 x 5120 with one group: 456 -> 432 us).
// Shorter groups keep one band (there the strips already line up: 16640 x
// 5120 with one group measured 60.4 us as one band, 61.7 us cut into bands).
// Every role walks its run in order, so it keeps a cursor (group, band, K
// tile, M tile) that advances one tile at a time: one search of the group
// table per run instead of a search and a division per tile (the search alone
// cost about 2 us per doubling of the group count at 16640 x 5120).
constexpr int64_t kBandMinRun = 64;   // runs shorter than this: no bands

template <bool kBands>
struct GroupCursor {
  int g;
  int64_t tr_g, n_tg, tk, tm, start, end;
  int64_t run;      // kBands: tiles per run (the band height of tall groups)
  int64_t bh;       // kBands: this group's band height, run or n_tg (one band)
  int64_t b0, bend; // kBands: first and end tile-row of the current band

  __device__ __forceinline__ void set_group(const GroupTab& tab, int gi) {
    g = gi;
    tr_g = tab.tr(gi);
    n_tg = tab.tr(gi + 1) - tr_g;
    start = gi ? tab.end(gi - 1) : 0;
    end = tab.end(gi);
    tm = 0;
    if (kBands) {
      bh = (run >= kBandMinRun && n_tg >= 2 * run) ? run : (n_tg > 0 ? n_tg : 1);
      b0 = 0;
      bend = n_tg < bh ? n_tg : bh;
    }
  }
  __device__ __forceinline__ void init(const Params& p, const GroupTab& tab, int64_t t,
                                       int64_t run_len) {
    run = run_len;
    int lo = 0, hi = p.G;                          // tr(lo)*n_kt <= t < tr(hi)*n_kt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tab.tr(mid) * p.n_kt <= t) lo = mid; else hi = mid;
    }
    set_group(tab, lo);
    tk = 0;
    if (n_tg <= 0) return;                         // past the last tile
    const int64_t tl = t - tr_g * p.n_kt;
    if (kBands) {
      int64_t in_band;
      const int64_t band = div_tiles(tl, bh * p.n_kt, in_band);
      b0 = band * bh;
      bend = n_tg - b0 < bh ? n_tg : b0 + bh;
      int64_t r;
      tk = div_tiles(in_band, bend - b0, r);
      tm = b0 + r;
    } else {
      tk = div_tiles(tl, n_tg, tm);
    }
  }
  __device__ __forceinline__ void next(const Params& p, const GroupTab& tab) {
    if (++tm < (kBands ? bend : n_tg)) return;
    tm = kBands ? b0 : 0;
    if (++tk < p.n_kt) return;
    tk = 0;
    if (kBands) {
      b0 = bend;
      if (b0 < n_tg) {                             // next band of the group
        bend = n_tg - b0 < bh ? n_tg : b0 + bh;
        tm = b0;
        return;
      }
    }
    int ng = g + 1;
    while (ng < p.G && tab.tr(ng + 1) == tab.tr(ng)) ++ng;   // skip empty groups
    if (ng < p.G) set_group(tab, ng);
  }
  __device__ __forceinline__ Tile tile(const Params& p) const {
    Tile T;
    const int64_t m0 = start + (tm << 7);
    const int64_t left = end - m0;
    T.m0 = static_cast<int32_t>(m0);
    T.k0 = static_cast<int32_t>(tk * kTile);
    T.rows = static_cast<int32_t>(left < kTile ? left : kTile);
    T.next_rows = static_cast<int32_t>(left - kTile < kTile ? left - kTile : kTile);
    T.cont = kBands ? ((tm > b0 ? 1 : 0) | (tm + 1 < bend ? 2 : 0))
                    : ((tm > 0 ? 1 : 0) | (tm + 1 < n_tg ? 2 : 0));
    T.s0_dst = p.s0 + ((tr_g + tm) * p.n_kt + tk) * kScaleTile;
    T.s1_dst = p.s1 + static_cast<int64_t>(p.k128) * (tr_g * 4) + (tk * n_tg + tm) * kScaleTile;
    return T;
  }
};

// The tile a role processes at run position t: from the cursor (advanced
// past it) in the grouped mode, from t otherwise.
template <int kMode, typename Cursor>
__device__ __forceinline__ Tile role_tile(const Params& p, const GroupTab& tab, int64_t t,
                                          Cursor& cur) {
  if (is_grouped(kMode)) {
    const Tile T = cur.tile(p);
    cur.next(p, tab);
    return T;
  }
  return get_tile<kMode>(p, tab, t);
}

// ---- compute units ----------------------------------------------------------

// dim0 half-block unit (16 elements), stored straight to q0.  In warp step
// with first row R0 (even), lane l takes row R0 + ((l >> 2) & 1) + 2*(l >> 4),
// 64-column half `box` = (l >> 3) & 1 and half-block hq = l & 3 of that half:
//   - each 8-lane phase of a 16-byte shared load touches two rows of one half
//     whose swizzles differ in the lowest bit, so all 8 bank groups differ;
//   - each warp store writes four whole 128-byte rows of q0;
//   - lanes l and l^1 hold the two halves of one 32-element block and combine
//     their maxima with one shuffle.
// Rows at or beyond `rows` (grouped mode: past the group's end) are neither
// stored nor given a scale (their blocked scale byte is padding, 0).
// kScatter (3D weights with N % 128 != 0): a tile can straddle two experts, so
// each scale byte goes straight to its expert's blocked matrix in global
// memory instead of the tile's staging.
template <bool kScatter>
__device__ __forceinline__ void dim0_half_unit(const uint8_t* in, uint8_t* sc0, uint8_t* q0,
                                               int64_t M, int64_t K, int m0, int k0, int R0,
                                               int lane, int rows, const Params& p) {
  const int row = R0 + ((lane >> 2) & 1) + 2 * (lane >> 4);
  const int box = (lane >> 3) & 1;
  const int hq = lane & 3;
  const int sw = row & 7;
  const uint8_t* src = in + box * kHalfBytes + row * 128;
  const uint4 v0 = *reinterpret_cast<const uint4*>(src + (((2 * hq) ^ sw) << 4));
  const uint4 v1 = *reinterpret_cast<const uint4*>(src + (((2 * hq + 1) ^ sw) << 4));
  uint32_t a = absmax2(absmax2(absmax2(v0.x, v0.y), absmax2(v0.z, v0.w)),
                       absmax2(absmax2(v1.x, v1.y), absmax2(v1.z, v1.w)));
  a = absmax2(a, __shfl_xor_sync(0xffffffffu, a, 1));
  const uint32_t lo = mag_lo(a), hi = mag_hi(a);
  uint32_t sbyte;
  float m;
  mx_scale(lo > hi ? lo : hi, sbyte, m);
  uint4 o;
  o.x = e4m3x4(bf_lo(v0.x), bf_hi(v0.x), bf_lo(v0.y), bf_hi(v0.y), m);
  o.y = e4m3x4(bf_lo(v0.z), bf_hi(v0.z), bf_lo(v0.w), bf_hi(v0.w), m);
  o.z = e4m3x4(bf_lo(v1.x), bf_hi(v1.x), bf_lo(v1.y), bf_hi(v1.y), m);
  o.w = e4m3x4(bf_lo(v1.z), bf_hi(v1.z), bf_lo(v1.w), bf_hi(v1.w), m);
  const int64_t gr = static_cast<int64_t>(m0) + row;
  const int64_t gc = static_cast<int64_t>(k0) + 64 * box + 16 * hq;
  if (row < rows && gr < M && gc < K && in_span(p.sp_q0, q0 + gr * K + gc, 16))
    *reinterpret_cast<uint4*>(q0 + gr * K + gc) = o;
  if ((hq & 1) == 0) {
    if (kScatter) {
      if (gr < M && gc < K) {
        const uint32_t e = static_cast<uint32_t>(gr) / static_cast<uint32_t>(p.N);
        const int64_t n = gr - static_cast<int64_t>(e) * p.N;
        uint8_t* d = p.s0 + e * p.s0_expert_bytes + blocked_offset(n, gc >> 5, p.kb4);
        if (in_span(p.sp_s0, d, 1)) *d = static_cast<uint8_t>(sbyte);
      }
    } else {
      sc0[blocked_in_tile(row, 2 * box + (hq >> 1))] = static_cast<uint8_t>(row < rows ? sbyte : 0u);
    }
  }
}

// Four consecutive rows of one column of a dim1 unit -> four e4m3 bytes.
#define MX_COL4_LO(w, j, m) e4m3x4(bf_lo(w[j]), bf_lo(w[j + 1]), bf_lo(w[j + 2]), bf_lo(w[j + 3]), m)
#define MX_COL4_HI(w, j, m) e4m3x4(bf_hi(w[j]), bf_hi(w[j + 1]), bf_hi(w[j + 2]), bf_hi(w[j + 3]), m)

// dim1 unit: column pair p (columns 2p, 2p+1 of the tile), rows 32*mb ..
// 32*mb+31.  Reads one 4-byte word per row (a warp reads whole 128-byte rows,
// conflict-free under the swizzle), writes 32 e4m3 bytes per column into the
// even / odd halves of the q1 staging tile (row p of each half) and the two
// scale bytes, as one 16-bit store into the plain-order scale staging
// [mb][column] (conflict-free; the store warp transposes it to the blocked
// order).  Rows at or beyond `rows` are treated as zero (grouped mode).
// Returns the two scale bytes (even column in bits 0-7, odd in 8-15).
template <bool kMask>
__device__ __forceinline__ uint32_t dim1_unit(const uint8_t* in, uint8_t* q1s, uint8_t* sc1,
                                              int p, int mb, int rows) {
  const int wd = p & 31;
  const int ch = wd >> 2;
  const uint8_t* src = in + (p >> 5) * kHalfBytes + (mb * 32) * 128 + (wd & 3) * 4;
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 32; ++j)
    w[j] = *reinterpret_cast<const uint32_t*>(src + j * 128 + ((ch ^ (j & 7)) << 4));
  if (kMask) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (mb * 32 + j >= rows) w[j] = 0u;
  }
  uint32_t t[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) t[j] = absmax2(w[2 * j], w[2 * j + 1]);
#pragma unroll
  for (int j = 0; j < 8; ++j) t[j] = absmax2(t[2 * j], t[2 * j + 1]);
#pragma unroll
  for (int j = 0; j < 4; ++j) t[j] = absmax2(t[2 * j], t[2 * j + 1]);
  const uint32_t a = absmax2(absmax2(t[0], t[1]), absmax2(t[2], t[3]));
  uint32_t se, so;
  float me, mo;
  mx_scale(mag_lo(a), se, me);
  mx_scale(mag_hi(a), so, mo);

  uint4 e0, e1, o0, o1;
  e0.x = MX_COL4_LO(w, 0, me);  e0.y = MX_COL4_LO(w, 4, me);
  e0.z = MX_COL4_LO(w, 8, me);  e0.w = MX_COL4_LO(w, 12, me);
  e1.x = MX_COL4_LO(w, 16, me); e1.y = MX_COL4_LO(w, 20, me);
  e1.z = MX_COL4_LO(w, 24, me); e1.w = MX_COL4_LO(w, 28, me);
  o0.x = MX_COL4_HI(w, 0, mo);  o0.y = MX_COL4_HI(w, 4, mo);
  o0.z = MX_COL4_HI(w, 8, mo);  o0.w = MX_COL4_HI(w, 12, mo);
  o1.x = MX_COL4_HI(w, 16, mo); o1.y = MX_COL4_HI(w, 20, mo);
  o1.z = MX_COL4_HI(w, 24, mo); o1.w = MX_COL4_HI(w, 28, mo);
  const int sw = p & 7;
  uint8_t* de = q1s + p * 128;
  uint8_t* dodd = q1s + kQ1Half + p * 128;
  *reinterpret_cast<uint4*>(de + (((2 * mb) ^ sw) << 4)) = e0;
  *reinterpret_cast<uint4*>(de + (((2 * mb + 1) ^ sw) << 4)) = e1;
  *reinterpret_cast<uint4*>(dodd + (((2 * mb) ^ sw) << 4)) = o0;
  *reinterpret_cast<uint4*>(dodd + (((2 * mb + 1) ^ sw) << 4)) = o1;
  const uint32_t pair = se | (so << 8);
  *reinterpret_cast<uint16_t*>(sc1 + mb * 128 + 2 * p) = static_cast<uint16_t>(pair);
  return pair;
}
#undef MX_COL4_LO
#undef MX_COL4_HI

__device__ __forceinline__ uint32_t word_of(const uint4& v, int k) {
  return k < 2 ? (k == 0 ? v.x : v.y) : (k == 2 ? v.z : v.w);
}

// Bytes [lo, hi) of v to the 16-byte aligned address g (+lo ...), as the
// fewest naturally aligned 8 / 4 / 2 / 1-byte stores (at most 7 for a
// partial chunk).
__device__ __forceinline__ void store_partial(uint8_t* g, const uint4& v, int lo, int hi) {
  int i = lo;
#pragma unroll 1
  while (i < hi) {
    if ((i & 7) == 0 && i + 8 <= hi) {
      *reinterpret_cast<uint2*>(g + i) = i == 0 ? make_uint2(v.x, v.y) : make_uint2(v.z, v.w);
      i += 8;
    } else if ((i & 3) == 0 && i + 4 <= hi) {
      *reinterpret_cast<uint32_t*>(g + i) = word_of(v, i >> 2);
      i += 4;
    } else if ((i & 1) == 0 && i + 2 <= hi) {
      *reinterpret_cast<uint16_t*>(g + i) = static_cast<uint16_t>(word_of(v, i >> 2) >> (8 * (i & 3)));
      i += 2;
    } else {
      g[i] = static_cast<uint8_t>(word_of(v, i >> 2) >> (8 * (i & 3)));
      i += 1;
    }
  }
}

// Grouped mode, M % 16 == 0 (every q1 row of a tile starts at the same offset
// delta != 0 inside a 16-byte chunk), a whole tile whose tile above was this
// CTA's previous one: rewrite the staged q1 rows in place onto their aligned
// chunks [m0 - delta, m0 - delta + 128) (chunk 0 completes the previous
// tile's partial last chunk from the carried bytes), so that each row is one
// 16-byte aligned 128-byte TMA box.  The row's raw last 16 bytes become the
// carried chunk of the next tile.  When the tile below is not this CTA's next
// one (`tail`), the row's last delta bytes, which lie past the box, are stored
// here with the fewest aligned narrow stores.  One lane per q1 row: store
// warp sw_idx owns staging rows 16*sw_idx .. +15 of both halves (the rows it
// stores by TMA); each 8-lane phase takes eight consecutive staging rows of
// one half, whose swizzles differ, so the 16-byte accesses are conflict-free.
// The lane loads its extended row [carried chunk | 128 staged bytes], shifts
// it by the uniform byte offset 16 - delta (word offset by two select levels,
// byte offset by funnel shifts) and writes it back; no lane touches another's
// row.
__device__ __forceinline__ void shift_q1_rows(uint8_t* q1s, uint4& carry, int delta, int sw_idx,
                                              int lane, bool tail, uint8_t* q1, int64_t M,
                                              int64_t K, int m0, int k0, const Span& sq1) {
  const int i = lane & 7, ph = lane >> 3;
  const int mrow = (2 * sw_idx + (ph >> 1)) * 8 + i;   // staging row, 16*sw_idx .. +15
  const int h = ph & 1;                                  // even / odd q1 half
  const int c = 2 * mrow + h;                            // q1 row within the tile
  uint8_t* srow = q1s + h * kQ1Half + mrow * 128;
  const int sw = mrow & 7;
  uint32_t e[40];
  e[0] = carry.x; e[1] = carry.y; e[2] = carry.z; e[3] = carry.w;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint4 v = *reinterpret_cast<const uint4*>(srow + ((k ^ sw) << 4));
    e[4 + 4 * k] = v.x; e[5 + 4 * k] = v.y; e[6 + 4 * k] = v.z; e[7 + 4 * k] = v.w;
  }
  e[36] = e[37] = e[38] = e[39] = 0u;
  const int s = 16 - delta;                              // 1 .. 15
  const bool q1b = (s >> 2) & 1, q2b = (s >> 2) & 2;
  const uint32_t r = 8u * static_cast<uint32_t>(s & 3);
  uint32_t f[39], g[37];
#pragma unroll
  for (int t = 0; t < 39; ++t) f[t] = q1b ? e[t + 1] : e[t];
#pragma unroll
  for (int t = 0; t < 37; ++t) g[t] = q2b ? f[t + 2] : f[t];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint4 o;
    o.x = __funnelshift_r(g[4 * k], g[4 * k + 1], r);
    o.y = __funnelshift_r(g[4 * k + 1], g[4 * k + 2], r);
    o.z = __funnelshift_r(g[4 * k + 2], g[4 * k + 3], r);
    o.w = __funnelshift_r(g[4 * k + 3], g[4 * k + 4], r);
    *reinterpret_cast<uint4*>(srow + ((k ^ sw) << 4)) = o;
  }
  carry = make_uint4(e[32], e[33], e[34], e[35]);
  const int64_t kk = static_cast<int64_t>(k0) + c;
  if (tail && kk < K) {
    uint4 o;
    o.x = __funnelshift_r(g[32], g[33], r);
    o.y = __funnelshift_r(g[33], g[34], r);
    o.z = __funnelshift_r(g[34], g[35], r);
    o.w = __funnelshift_r(g[35], g[36], r);
    uint8_t* gp = q1 + (kk * M + m0 - delta + 128);      // 16-byte aligned
    if (in_span(sq1, gp, delta)) store_partial(gp, o, 0, delta);
  }
}

// Grouped mode, M % 16 == 0, a whole tile that starts a CTA's run in a strip
// of a misaligned group (the tile above is another CTA's, or another group's)
// while the tile below is this CTA's next one, with at least 16 - delta rows:
// the rows leave as boxes one chunk later, [m0 - delta + 16, m0 - delta +
// 144), which the first 16 - delta bytes of the tile below complete (its
// staging is in hand).  The rows' first 16 - delta bytes, in the chunk shared
// with the tile above, are stored here with the fewest aligned narrow stores;
// the tile below's own box writes its first chunk, the same bytes as this
// box's last chunk, again.  The raw last 16 bytes of each row become the
// carried chunk of the tile below.  Lane mapping as in shift_q1_rows.
__device__ __forceinline__ void shift_q1_rows_next(uint8_t* q1s, const uint8_t* q1s_next,
                                                   uint4& carry, int delta, int sw_idx,
                                                   int lane, uint8_t* q1, int64_t M, int64_t K,
                                                   int m0, int k0, const Span& sq1) {
  const int i = lane & 7, ph = lane >> 3;
  const int mrow = (2 * sw_idx + (ph >> 1)) * 8 + i;
  const int h = ph & 1;
  const int c = 2 * mrow + h;
  uint8_t* srow = q1s + h * kQ1Half + mrow * 128;
  const int sw = mrow & 7;
  uint32_t e[40];
  e[0] = e[1] = e[2] = e[3] = 0u;                        // no bytes before the tile
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint4 v = *reinterpret_cast<const uint4*>(srow + ((k ^ sw) << 4));
    e[4 + 4 * k] = v.x; e[5 + 4 * k] = v.y; e[6 + 4 * k] = v.z; e[7 + 4 * k] = v.w;
  }
  {
    const uint4 v = *reinterpret_cast<const uint4*>(q1s_next + h * kQ1Half + mrow * 128 +
                                                    ((0 ^ sw) << 4));
    e[36] = v.x; e[37] = v.y; e[38] = v.z; e[39] = v.w;
  }
  const int s = 16 - delta;                              // 1 .. 15
  const bool q1b = (s >> 2) & 1, q2b = (s >> 2) & 2;
  const uint32_t r = 8u * static_cast<uint32_t>(s & 3);
  uint32_t f[39], g[37];
#pragma unroll
  for (int t = 0; t < 39; ++t) f[t] = q1b ? e[t + 1] : e[t];
#pragma unroll
  for (int t = 0; t < 37; ++t) g[t] = q2b ? f[t + 2] : f[t];
  const int64_t kk = static_cast<int64_t>(k0) + c;
  if (kk < K) {                                          // chunk 0: bytes [delta, 16)
    uint4 o;
    o.x = __funnelshift_r(g[0], g[1], r);
    o.y = __funnelshift_r(g[1], g[2], r);
    o.z = __funnelshift_r(g[2], g[3], r);
    o.w = __funnelshift_r(g[3], g[4], r);
    uint8_t* gp = q1 + (kk * M + m0 - delta);            // 16-byte aligned
    if (in_span(sq1, gp + delta, 16 - delta)) store_partial(gp, o, delta, 16);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {                          // chunks 1 .. 8
    uint4 o;
    o.x = __funnelshift_r(g[4 * k + 4], g[4 * k + 5], r);
    o.y = __funnelshift_r(g[4 * k + 5], g[4 * k + 6], r);
    o.z = __funnelshift_r(g[4 * k + 6], g[4 * k + 7], r);
    o.w = __funnelshift_r(g[4 * k + 7], g[4 * k + 8], r);
    *reinterpret_cast<uint4*>(srow + ((k ^ sw) << 4)) = o;
  }
  carry = make_uint4(e[32], e[33], e[34], e[35]);
}

// Grouped mode, other tiles (strip ends, partial tiles, the first tile of a
// CTA's run, odd M): store the staged q1 rows (`len` valid bytes each) to q1
// row k0 + c, columns m0 .. m0 + len - 1, as the aligned chunks they cover.
// One lane per q1 row, the rows and lane mapping of shift_q1_rows: the lane
// loads its extended row [carried chunk | 128 staged bytes], forms all nine
// aligned chunks in registers (the byte offset delta of the row's start in
// its 16-byte chunk is 0..15 and, when M % 16 != 0, differs by row: three
// select levels for the word offset, funnel shifts for the bytes) and
// stores them: whole chunks with one vector store, partial ones (at a strip
// end, or where the tile above was handled by another CTA) with the fewest
// aligned 8 / 4 / 2 / 1-byte stores.  When the tile below follows in this
// CTA, the last chunk is not stored: it is completed there from the carried
// raw last 16 bytes of this row.
__device__ __forceinline__ void copy_out_q1(const uint8_t* q1s, uint4& carry, uint8_t* q1,
                                            int64_t M, int64_t K, int m0, int k0, int len,
                                            bool cont_prev, bool cont_next, int sw_idx, int lane,
                                            const Span& sq1) {
  const int i = lane & 7, ph = lane >> 3;
  const int mrow = (2 * sw_idx + (ph >> 1)) * 8 + i;   // staging row, 16*sw_idx .. +15
  const int h = ph & 1;                                  // even / odd q1 half
  const int c = 2 * mrow + h;                            // q1 row within the tile
  const int64_t kk = static_cast<int64_t>(k0) + c;
  if (kk >= K) return;
  const uint8_t* srow = q1s + h * kQ1Half + mrow * 128;
  const int sw = mrow & 7;
  const int64_t A = kk * M + m0;                         // byte offset of the row segment
  const int delta = static_cast<int>(A & 15);
  uint8_t* g = q1 + (A - delta);                         // its first aligned chunk
  uint32_t e[44];
  if (cont_prev) {
    e[0] = carry.x; e[1] = carry.y; e[2] = carry.z; e[3] = carry.w;
  } else {
    e[0] = e[1] = e[2] = e[3] = 0u;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint4 v = *reinterpret_cast<const uint4*>(srow + ((k ^ sw) << 4));
    e[4 + 4 * k] = v.x; e[5 + 4 * k] = v.y; e[6 + 4 * k] = v.z; e[7 + 4 * k] = v.w;
  }
#pragma unroll
  for (int t = 36; t < 44; ++t) e[t] = 0u;
  // aligned chunk j = bytes [16j + s, 16j + s + 16) of the extended row
  const int s = 16 - delta;                              // 1 .. 16
  const int q = s >> 2;                                  // word offset 0 .. 4
  const uint32_t r = 8u * static_cast<uint32_t>(s & 3);
  uint32_t f[43], gg[41], w[37];
#pragma unroll
  for (int t = 0; t < 43; ++t) f[t] = (q & 1) ? e[t + 1] : e[t];
#pragma unroll
  for (int t = 0; t < 41; ++t) gg[t] = (q & 2) ? f[t + 2] : f[t];
#pragma unroll
  for (int t = 0; t < 37; ++t) w[t] = (q & 4) ? gg[t + 4] : gg[t];
#pragma unroll
  for (int j = 0; j < 9; ++j) {
    const int o = 16 * j - delta;                        // segment offset of the chunk start
    int b_lo = o < 0 ? -o : 0;
    if (j == 0 && cont_prev) b_lo = 0;                   // the carried bytes complete it
    const int b_hi = (len - o) < 16 ? (len - o) : 16;
    if (j == 8 && cont_next) continue;                   // completed by the tile below
    if (b_lo < b_hi) {
      uint4 v;
      v.x = __funnelshift_r(w[4 * j], w[4 * j + 1], r);
      v.y = __funnelshift_r(w[4 * j + 1], w[4 * j + 2], r);
      v.z = __funnelshift_r(w[4 * j + 2], w[4 * j + 3], r);
      v.w = __funnelshift_r(w[4 * j + 3], w[4 * j + 4], r);
      if (!in_span(sq1, g + 16 * j + b_lo, b_hi - b_lo)) continue;
      if (b_lo == 0 && b_hi == 16) *reinterpret_cast<uint4*>(g + 16 * j) = v;
      else store_partial(g + 16 * j, v, b_lo, b_hi);
    }
  }
  if (cont_next) carry = make_uint4(e[32], e[33], e[34], e[35]);
}

// One warp builds the grouped mode's group table from the offsets: it
// validates them, counts ceil(m_g / 128) tile-rows per group and scans the
// counts into tr_s[0..G]; ends_s[g] = offs[g].  Returns the padded tile-rows
// of all groups, or -1 when the offsets are invalid.  kSpeculative: read
// before the previous grid has finished, so the offsets may not be final
// (the table then only picks prefetch addresses); they are read at L2, so
// that no copy of them stays in L1 for the reads after the wait.
template <bool kSpeculative>
__device__ __forceinline__ int64_t warp_group_table(const Params& p, int32_t* tr_s, int32_t* ends_s,
                                                    int lane) {
  int64_t carry = 0;
  int64_t prev_end = 0;                       // offs[base - 1]
  bool bad = false;
  for (int base = 0; base < p.G; base += 32) {
    const int g = base + lane;
    int64_t hi = 0;
    if (g < p.G) hi = kSpeculative ? __ldcg(p.offs + g) : p.offs[g];
    const int64_t below = __shfl_up_sync(0xffffffffu, hi, 1);
    const int64_t lo = lane == 0 ? prev_end : below;
    prev_end = __shfl_sync(0xffffffffu, hi, 31);
    int64_t tiles = 0;
    if (g < p.G) {
      ends_s[g] = static_cast<int32_t>(hi);
      const bool b = hi < lo || hi < 0 || hi > p.M || (g == p.G - 1 && hi != p.M);
      bad = bad || b;
      tiles = b ? 0 : (hi - lo + 127) >> 7;
    }
    int64_t incl = tiles;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t n = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += n;
    }
    if (g < p.G) tr_s[g + 1] = static_cast<int32_t>(carry + incl);
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) tr_s[0] = 0;
  __syncwarp();
  return __any_sync(0xffffffffu, bad) ? -1 : carry;
}

// ---- the kernel -------------------------------------------------------------

// kClaim (2D / 3D modes, launches of kClaimMinRounds rounds or more): the
// last kClaimRounds rounds of tiles are not dealt out in advance but claimed
// from a counter, one tile ahead, so that the CTAs that run fast take more of
// them and all finish close together.  Every CTA makes exactly one claim that
// finds no tile, so a launch makes a known number of claims, and the CTA that
// makes the last one resets the counter: nothing runs after the final
// barrier, and the next launch on the stream (which claims only after this
// one has completed) finds it at zero.
template <int kMode, bool kClaim>
__global__ void __launch_bounds__(threads_of(kMode), 1)
    mx_cast_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_q1e,
                   const __grid_constant__ CUtensorMap tm_q1o, const Params p) {
  static_assert(!(kClaim && is_grouped(kMode)), "the grouped schedule is static");
  constexpr bool kDim0 = has_dim0(kMode);
  constexpr bool kDim1 = has_dim1(kMode);
  constexpr bool kTmaQ1 = kDim1 && !is_grouped(kMode);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bars;                      // [kStages] TMA landed
  uint64_t* empty = bars + kStages;           // [kStages] compute done reading
  uint64_t* sfull = bars + 2 * kStages;       // [kStaging] staging written
  uint64_t* sempty = sfull + kStaging;        // [kStaging] staging drained
  uint64_t* stall_bar = sempty + kStaging;    // diagnostic: never completed
  int64_t* ids_in = reinterpret_cast<int64_t*>(smem + kOffIds);   // claim schedule: [kStages]
  int64_t* ids_st = ids_in + kStages;                                // [kStaging]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffFlag);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Programmatic dependent launch: let the next launch in the stream start
  // its set-up now (it cannot share an SM with this CTA, so it only takes SMs
  // this grid has left), and wait for every earlier grid to finish, with its
  // memory visible, before reading any input into the SM or writing any
  // output (the L2 prefetch hints below are issued before the wait).
  asm volatile("griddepcontrol.launch_dependents;");
  GroupTab tab = {nullptr, nullptr, p.row_offs, p.offs};
  if (!is_grouped(kMode) && threadIdx.x == kProducerWarp * 32) {
    // While the previous grid's last CTAs finish (this CTA got an SM that
    // one of its CTAs left), ask L2 for the tiles the input ring will load
    // first.  Only a hint: nothing is read into the SM before the wait, and
    // the loads after it see the previous grid's writes (L2 is where global
    // memory is coherent).  It puts the DRAM that the previous grid's tail
    // leaves idle to use: 16384^2 167.7 -> 166.0 us, 4096^2 15.4 -> 14.1
    // us; prefetching 6 or 10 tiles measured slower than 3.
    for (int i = 0; i < kStages; ++i) {
      const int64_t t = blockIdx.x + static_cast<int64_t>(gridDim.x) * i;
      if (t >= p.n_tiles) break;
      const Tile T = get_tile<kMode>(p, tab, t);
      tma_prefetch_2d(&tm_x, T.k0, T.m0);
      tma_prefetch_2d(&tm_x, T.k0 + 64, T.m0);
    }
  }
  if (is_grouped(kMode) && p.G <= kMaxSmemGroups && warp == kProducerWarp) {
    // The same hint in the grouped mode, from a group table built now from
    // the offsets as they stand (a stale or invalid table costs a useless
    // prefetch, nothing else).  It lives in the q1 staging, which nothing
    // uses before the first tile has landed.
    int32_t* tr_x = reinterpret_cast<int32_t*>(smem + kOffQ1);
    int32_t* ends_x = tr_x + kMaxSmemGroups + 1;
    const int64_t total = warp_group_table<true>(p, tr_x, ends_x, lane);
    if (total > 0 && lane == 0) {
      const GroupTab st = {tr_x, ends_x, nullptr, nullptr};
      const int64_t n = total * p.n_kt;
      const int64_t f = n * blockIdx.x / gridDim.x;
      const int64_t e = n * (blockIdx.x + 1) / gridDim.x;
      GroupCursor<kMode == kModeGroupedBands> c;
      c.init(p, st, f, (n + gridDim.x - 1) / gridDim.x);
      for (int64_t t = f; t < e && t < f + kStages; ++t) {
        const Tile T = c.tile(p);
        c.next(p, st);
        tma_prefetch_2d(&tm_x, T.k0, T.m0);
        tma_prefetch_2d(&tm_x, T.k0 + 64, T.m0);
      }
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  int64_t first, end, step;
  int64_t run_len = 1;                        // grouped: tiles per CTA run (rounded up)
  if (is_grouped(kMode)) {
    int64_t total_tr;                         // padded tile-rows of all groups
    if (p.G <= kMaxSmemGroups) {
      // Up to kMaxSmemGroups groups every CTA builds the group table itself
      // from the offsets (no separate offsets kernel on the critical path).
      // CTA 0 also writes the padded-offset outputs and the status word.
      int32_t* tr_s = reinterpret_cast<int32_t*>(smem + kOffGTab);
      int32_t* ends_s = tr_s + kMaxSmemGroups + 1;
      volatile int* bad_s = reinterpret_cast<volatile int*>(smem + kOffFlag + 4);
      if (warp == 0) {
        const int64_t total = warp_group_table<false>(p, tr_s, ends_s, lane);
        if (lane == 0) *bad_s = total < 0 ? 1 : 0;
      }
      __syncthreads();
      if (*bad_s) {                           // invalid group offsets: write nothing
        if (blockIdx.x == 0 && threadIdx.x == 0 && in_span(p.sp_st, p.status_out, 4))
          *p.status_out = kStatusBadGroups;
        return;
      }
      if (blockIdx.x == 0) {
        for (int g = threadIdx.x; g <= p.G; g += blockDim.x) {
          if (in_span(p.sp_ro, p.row_offs_out + g, 8))
            p.row_offs_out[g] = static_cast<int64_t>(tr_s[g]) * 128;
          if (in_span(p.sp_co, p.col_offs_out + g, 8))
            p.col_offs_out[g] = static_cast<int64_t>(tr_s[g]) * 4;
        }
        if (threadIdx.x == 0 && in_span(p.sp_st, p.status_out, 4)) *p.status_out = 0;
      }
      tab.tr_s = tr_s;
      tab.ends_s = ends_s;
      total_tr = tr_s[p.G];
    } else {
      // The offsets come from the preceding group_offsets_kernel (waited for
      // above, like every earlier grid).
      if (*p.status != 0) return;             // invalid group offsets: write nothing
      total_tr = p.row_offs[p.G] >> 7;
    }
    const int64_t n_tiles = total_tr * p.n_kt;
    // contiguous, balanced runs of tiles per CTA (32-bit divisions where
    // they fit: three 64-bit ones took 0.3 us here, on every launch's
    // critical path)
    int64_t rem;
    first = div_tiles(n_tiles * blockIdx.x, gridDim.x, rem);
    end = div_tiles(n_tiles * (blockIdx.x + 1), gridDim.x, rem);
    step = 1;
    run_len = div_tiles(n_tiles + gridDim.x - 1, gridDim.x, rem);
  } else {
    first = blockIdx.x;
    end = p.n_tiles;
    step = gridDim.x;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kComputeWarps);
    }
    for (int o = 0; o < kStaging; ++o) {
      mbar_init(&sfull[o], kComputeWarps);
      mbar_init(&sempty[o], store_warps(kMode));
    }
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();


  int64_t issued = 0;                         // producer lane: TMA loads issued
  if (warp == kProducerWarp) {
    if (lane == 0) {
      prefetch_tmap(&tm_x);
      typename ItType<kMode>::T it = 0;
      GroupCursor<kMode == kModeGroupedBands> cur;
      if (is_grouped(kMode)) cur.init(p, tab, first, run_len);
      if (kClaim) {
        const int64_t g = gridDim.x;
        const int64_t n_static = p.n_tiles / g - kClaimRounds;   // whole rounds dealt out
        const int64_t n_claims = p.n_tiles - n_static * g + g;
        int64_t next = blockIdx.x;
        for (;; ++it) {
          const int s = static_cast<int>(it % kStages);
          const uint32_t ph = static_cast<uint32_t>((it / kStages) & 1);
          if (kDiagStall && static_cast<int64_t>(it) == p.stall_at && blockIdx.x == 0) {
            mbar_wait(stall_bar, 0u, abort_flag, p.stall_ns);   // as in the static loop
            break;
          }
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) break;
          const int64_t t = next;
          if (t >= p.n_tiles) {                   // tell the other roles: no more tiles
            ids_in[s] = -1;
            mbar_arrive(&full[s]);
            break;
          }
          ids_in[s] = t;
          const Tile T = get_tile<kMode>(p, tab, t);
          uint8_t* dst = smem + kOffIn + s * kInBytes;
          mbar_arrive_expect_tx(&full[s], kInBytes);
          tma_load_2d(dst, &tm_x, T.k0, T.m0, &full[s]);
          tma_load_2d(dst + kHalfBytes, &tm_x, T.k0 + 64, T.m0, &full[s]);
          issued = static_cast<int64_t>(it) + 1;
          // the next tile: dealt out, or claimed (after this tile's loads are
          // on their way, so that the claim's latency overlaps them)
          if (static_cast<int64_t>(it) + 1 < n_static) {
            next = blockIdx.x + g * (static_cast<int64_t>(it) + 1);
          } else {
            const unsigned int v = atomicAdd(p.claims, 1u);
            if (static_cast<int64_t>(v) == n_claims - 1) atomicExch(p.claims, 0u);
            next = n_static * g + static_cast<int64_t>(v);
          }
        }
      } else
      for (int64_t t = first; t < end; t += step, ++it) {
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = static_cast<uint32_t>((it / kStages) & 1);
        if (kDiagStall && static_cast<int64_t>(it) == p.stall_at && blockIdx.x == 0) {
          // Diagnostic (checked builds, armed from the host): instead of loading this
          // tile, wait on a barrier that nothing completes.  The wait runs
          // out and raises the abort flag; the compute warps, waiting for
          // this tile, and the store warp stop on it.
          mbar_wait(stall_bar, 0u, abort_flag, p.stall_ns);
          break;
        }
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) break;
        const Tile T = role_tile<kMode>(p, tab, t, cur);
        uint8_t* dst = smem + kOffIn + s * kInBytes;
        mbar_arrive_expect_tx(&full[s], kInBytes);
        tma_load_2d(dst, &tm_x, T.k0, T.m0, &full[s]);
        tma_load_2d(dst + kHalfBytes, &tm_x, T.k0 + 64, T.m0, &full[s]);
        issued = static_cast<int64_t>(it) + 1;
      }
    }
    __syncwarp();
  } else if (warp >= kFirstStoreWarp) {
    const int sw = warp - kFirstStoreWarp;
    if (sw == 0 && lane == 0 && (kTmaQ1 || p.q1_tma)) {
      prefetch_tmap(&tm_q1e);
      prefetch_tmap(&tm_q1o);
    }
    typename ItType<kMode>::T it = 0;
    GroupCursor<kMode == kModeGroupedBands> cur;
    if (is_grouped(kMode)) cur.init(p, tab, first, run_len);
    // grouped: the raw last 16 bytes of this lane's q1 row of the previous
    // tile (a lane keeps the same row of every tile)
    uint4 carry = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t t0 = first; kClaim || t0 < end; t0 += step, ++it) {
      const int o = static_cast<int>(it % kStaging);
      const uint32_t ph = static_cast<uint32_t>((it / kStaging) & 1);
      const bool ok = mbar_wait(&sfull[o], ph, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int64_t t = kClaim ? ids_st[o] : t0;
      if (kClaim && t < 0) break;
      const Tile T = role_tile<kMode>(p, tab, t, cur);
      uint8_t* q1s = smem + kOffQ1 + o * kQBytes;
      if (is_grouped(kMode)) {
        // Grouped: store warp sw owns rows 16*sw .. 16*sw+15 of each q1 half.
        // A whole 128-row tile whose q1 rows are 16-byte aligned at a common
        // offset leaves by TMA (one 16-row box per half and warp), shifted
        // onto the aligned chunks when that offset is not 0:
        //   - the tile above was this CTA's: boxes from its carried chunk (the
        //     row's last bytes are carried on, or stored narrow at a run end);
        //   - a run's first tile in the strip: boxes one chunk later, completed
        //     by the first bytes of the tile below (this CTA's next one), and
        //     the row's first bytes stored narrow.
        // Other tiles (partial tiles, a lone tile, odd M) are stored piecewise.
        // Measured at 16640 x 5120, G = 4 (three misaligned groups): the
        // run's first and last tiles as boxes cut the piecewise tiles from 3.2
        // to 1.1 per CTA, 62.9 -> 62.5 us (65536 x 5120, G = 16: 256 -> 245).
        const bool cont_prev = (T.cont & 1) && t > first;
        const bool cont_next = (T.cont & 2) && t + 1 < end;
        const int delta = T.m0 & 15;
        const bool full = p.q1_tma && T.rows == kTile;
        // a run's first tile in a misaligned strip: boxes one chunk later
        const bool box_next = full && delta != 0 && !cont_prev && cont_next &&
                              T.next_rows >= 16 - delta;
        if (box_next || (full && (delta == 0 || cont_prev))) {
          int x = T.m0 - delta;
          if (box_next) {
            // the tile below is this CTA's next one: wait for its staging
            const int o2 = static_cast<int>((it + 1) % kStaging);
            const uint32_t ph2 = static_cast<uint32_t>(((it + 1) / kStaging) & 1);
            const bool ok2 = mbar_wait(&sfull[o2], ph2, abort_flag);
            if (!__all_sync(0xffffffffu, ok2)) break;
            shift_q1_rows_next(q1s, smem + kOffQ1 + o2 * kQBytes, carry, delta, sw,
                               lane, p.q1, p.M, p.K, T.m0, T.k0, p.sp_q1);
            x += 16;
          } else if (delta != 0) {
            shift_q1_rows(q1s, carry, delta, sw, lane, !cont_next, p.q1, p.M, p.K,
                          T.m0, T.k0, p.sp_q1);
          }
          fence_proxy_async_smem();
          __syncwarp();
          const int y = (T.k0 >> 1) + kQ1GroupBoxRows * sw;
          if (lane == 0 && 2 * static_cast<int64_t>(y) < p.K) {
            tma_store_2d(&tm_q1e, x, y, q1s + sw * kQ1GroupBoxRows * 128);
            tma_store_2d(&tm_q1o, x, y, q1s + kQ1Half + sw * kQ1GroupBoxRows * 128);
          }
        } else {
          copy_out_q1(q1s, carry, p.q1, p.M, p.K, T.m0, T.k0, T.rows, cont_prev,
                      cont_next, sw, lane, p.sp_q1);
        }
      } else if (kDim1 && lane == 0) {
        tma_store_2d(&tm_q1e, T.m0, T.k0 >> 1, q1s);
        tma_store_2d(&tm_q1o, T.m0, T.k0 >> 1, q1s + kQ1Half);
      }
      if (sw == 0) {
        if (lane == 0 && kDim0 && T.s0_dst && in_span(p.sp_s0, T.s0_dst, kScaleTile))
          bulk_store(T.s0_dst, smem + kOffS0 + o * kScaleTile, kScaleTile);
        if (T.s1_dst) {
          // dim1 scales are staged as [M-block][column]; storage row `lane` of
          // the blocked tile holds columns lane, lane+32, lane+64, lane+96,
          // four M-blocks each.
          const uint8_t* nat = smem + kOffS1 + o * kScaleTile;
          uint4 w;
          uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const int c = lane + 32 * a;
            wp[a] = static_cast<uint32_t>(nat[c]) | (static_cast<uint32_t>(nat[128 + c]) << 8) |
                    (static_cast<uint32_t>(nat[256 + c]) << 16) |
                    (static_cast<uint32_t>(nat[384 + c]) << 24);
          }
          if (in_span(p.sp_s1, T.s1_dst + lane * 16, 16))
            *reinterpret_cast<uint4*>(T.s1_dst + lane * 16) = w;
        }
      }
      __syncwarp();
      if (lane == 0) {
        // Keep the newest bulk group in flight: the buffer of the previous
        // tile is released once its own group has been read.
        bulk_commit();
        bulk_wait_read<1>();
        if (it > 0) mbar_arrive(&sempty[static_cast<int>((it - 1) % kStaging)]);
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  } else {
    // compute warps
    typename ItType<kMode>::T it = 0;
    GroupCursor<kMode == kModeGroupedBands> cur;
    if (is_grouped(kMode)) cur.init(p, tab, first, run_len);
    for (int64_t t0 = first; kClaim || t0 < end; t0 += step, ++it) {
      const int s = static_cast<int>(it % kStages);
      const uint32_t ph = static_cast<uint32_t>((it / kStages) & 1);
      const int o = static_cast<int>(it % kStaging);
      const uint32_t oph = static_cast<uint32_t>((it / kStaging) & 1);
      bool ok = mbar_wait(&full[s], ph, abort_flag);
      ok = ok && mbar_wait(&sempty[o], oph ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int64_t t = kClaim ? ids_in[s] : t0;
      if (kClaim && t < 0) {                   // no more tiles: pass it on to the store warp
        if (lane == 0) {
          ids_st[o] = -1;
          mbar_arrive(&sfull[o]);
        }
        break;
      }
      if (kClaim && lane == 0 && warp == 0) ids_st[o] = t;

      const Tile T = role_tile<kMode>(p, tab, t, cur);
      const uint8_t* in = smem + kOffIn + s * kInBytes;
      uint8_t* q1s = smem + kOffQ1 + o * kQBytes;
      uint8_t* sc1 = smem + kOffS1 + o * kScaleTile;
      if (kDim0) {
        uint8_t* sc0 = smem + kOffS0 + o * kScaleTile;
        if (per_expert(kMode) && p.s0_scatter) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dim0_half_unit<true>(in, sc0, p.q0, p.M, p.K, T.m0, T.k0, (4 * warp + u) * 4, lane,
                                 T.rows, p);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dim0_half_unit<false>(in, sc0, p.q0, p.M, p.K, T.m0, T.k0, (4 * warp + u) * 4, lane,
                                  T.rows, p);
        }
      }
      const int mb = warp >> 1;
      const int pcol = (warp & 1) * 32 + lane;
      uint32_t sb = 0;
      if (!kDim1)
        ;
      else if (is_grouped(kMode) && T.rows < kTile)
        sb = dim1_unit<true>(in, q1s, sc1, pcol, mb, T.rows);
      else
        sb = dim1_unit<false>(in, q1s, sc1, pcol, mb, T.rows);

      if (kDim1 && per_expert(kMode) && T.s1_dst == nullptr) {
        // 3D weights with N % 128 != 0: a tile can straddle two experts, so
        // each scale byte goes straight to its expert's blocked matrix.
        const int64_t mbg = (static_cast<int64_t>(T.m0) >> 5) + mb;
        if ((mbg << 5) < p.M) {
          const int64_t e = (mbg << 5) / p.N;
          const int64_t col = mbg - e * (p.N >> 5);
          uint8_t* base = p.s1 + e * p.s1_expert_bytes;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int64_t kk = T.k0 + 2 * pcol + h;
            uint8_t* d = base + blocked_offset(kk, col, p.nb4);
            if (kk < p.K && in_span(p.sp_s1, d, 1)) *d = static_cast<uint8_t>(sb >> (8 * h));
          }
        }
      }

      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);     // input stage may be refilled

      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfull[o]);
    }

    if (is_grouped(kMode)) {
      // Zero the scale buffers' tails beyond the last group's padded end.
      const int64_t kb4 = static_cast<int64_t>(p.n_kt) * 4;
      const int64_t s0_beg = tab.tr(p.G) * 128 * kb4;
      const int64_t s0_end = (p.M + 128 * static_cast<int64_t>(p.G)) * kb4;
      const int64_t s1_beg = static_cast<int64_t>(p.k128) * (tab.tr(p.G) * 4);
      const int64_t s1_end = static_cast<int64_t>(p.k128) * (((p.M + 31) >> 5) + 4 * p.G);
      const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kComputeThreads + threadIdx.x;
      const int64_t gstride = static_cast<int64_t>(gridDim.x) * kComputeThreads;
      for (int64_t i = s0_beg / 4 + gtid; i < s0_end / 4; i += gstride)
        if (in_span(p.sp_s0, reinterpret_cast<uint32_t*>(p.s0) + i, 4))
          reinterpret_cast<uint32_t*>(p.s0)[i] = 0u;
      for (int64_t i = s1_beg / 4 + gtid; i < s1_end / 4; i += gstride)
        if (in_span(p.sp_s1, reinterpret_cast<uint32_t*>(p.s1) + i, 4))
          reinterpret_cast<uint32_t*>(p.s1)[i] = 0u;
    }
  }

  __syncthreads();
  if (*abort_flag && warp == kProducerWarp && lane == 0) {
    // A role gave up: TMA loads issued into the input ring may never have
    // been consumed.  Let each stage's last one land (bounded) before the CTA
    // exits and its shared memory is reused, then report.
    for (int s = 0; s < kStages; ++s) {
      if (issued <= s) break;
      const int64_t last = s + (issued - 1 - s) / kStages * kStages;   // last load into s
      mbar_drain(&full[s], static_cast<uint32_t>((last / kStages) & 1));
    }
    atomicOr(&g_watchdog, 1);
  }
}

}  // namespace

// ---- host launchers -----------------------------------------------------------

namespace {

int set_smem(const void* fn) {
  // Set once per device and kernel (DeviceCache); cheap to repeat but avoided.
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  return e == cudaSuccess ? 0 : static_cast<int>(e);
}

template <int kMode, bool kClaim = false>
int launch(const CastMaps& maps, const Params& prm, int grid, cudaStream_t stream) {
  static DeviceCache smem_attr;
  const int attr_rc = smem_attr.get(
      [] { return set_smem(reinterpret_cast<const void*>(&mx_cast_kernel<kMode, kClaim>)); });
  if (attr_rc != 0) return attr_rc;
  // Launched as a programmatic dependent of the previous work in the stream:
  // when that is a cast kernel (which triggers its dependents early), this
  // grid's launch and set-up overlap its tail; the kernel waits for it to
  // complete before any memory access (griddepcontrol.wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads_of(kMode));
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, mx_cast_kernel<kMode, kClaim>, maps.x, maps.q1e,
                                             maps.q1o, prm));
}

}  // namespace

// The claim counter for a launch on `stream` of the current device, or null
// for the static schedule.  Each (device, stream) in use keeps one word of
// g_claims: launches on one stream run one after another (each claims only
// after the previous grid has completed), while launches on different streams
// may overlap and so must not share a counter.  Null when the stream is being
// captured into a graph (a graph may be launched on any stream, so its
// counter could be shared), for cudaStreamPerThread (one handle for many
// streams), when the slots are all taken, or when the symbol cannot be found.
// A stream destroyed while a cast is still running on it must not be replaced
// by a new stream that launches casts before that cast has finished (the new
// stream could get the same handle and counter).
unsigned int* claim_counter(cudaStream_t stream) {
  if (stream == cudaStreamPerThread) return nullptr;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (cs != cudaStreamCaptureStatusNone) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= DeviceCache::kMaxDevices) {
    (void)cudaGetLastError();
    return nullptr;
  }
  struct Slots {
    unsigned int* base = nullptr;
    cudaStream_t stream[kClaimSlots] = {};
    int n = 0;
  };
  static Slots slots[DeviceCache::kMaxDevices];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  Slots& d = slots[dev];
  if (!d.base) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_claims) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    d.base = static_cast<unsigned int*>(a);
  }
  for (int i = 0; i < d.n; ++i)
    if (d.stream[i] == stream) return d.base + i;
  if (d.n == kClaimSlots) return nullptr;
  d.stream[d.n] = stream;
  return d.base + d.n++;
}

// Launch a 2D / 3D mode with the claim schedule when the launch is long
// enough and a counter is free, else with the static one.
template <int kMode>
int launch_tiles(const CastMaps& maps, Params prm, int grid, cudaStream_t stream) {
  if (prm.n_tiles / grid >= kClaimMinRounds) {
    prm.claims = claim_counter(stream);
    if (prm.claims) return launch<kMode, true>(maps, prm, grid, stream);
  }
  prm.claims = nullptr;
  return launch<kMode, false>(maps, prm, grid, stream);
}

// Bytes of a blocked scale matrix (R x C scales).
uint64_t blk_bytes(int64_t R, int64_t C) {
  return static_cast<uint64_t>((R + 127) / 128 * 128) * static_cast<uint64_t>((C + 3) / 4 * 4);
}

int smem_bytes_cast() { return kSmemBytes; }
int threads_cast() { return threads_of(kModeFused2D); }

int launch_cast_2d(const CastMaps& maps, int64_t M, int64_t K, void* q0, void* s0, void* s1,
                   int num_sms, cudaStream_t stream) {
  const bool dim0 = q0 != nullptr;
  const bool dim1 = s1 != nullptr;
  Params prm = {};
  const Stall stall = take_stall();
  prm.stall_at = stall.at;
  prm.stall_ns = stall.ns;
  prm.q0 = static_cast<uint8_t*>(q0);
  prm.M = M;
  prm.K = K;
  prm.n_mt = static_cast<int32_t>((M + kTile - 1) / kTile);
  prm.n_kt = static_cast<int32_t>((K + kTile - 1) / kTile);
  prm.n_tiles = static_cast<int64_t>(prm.n_mt) * prm.n_kt;
  prm.s0 = static_cast<uint8_t*>(s0);
  prm.s1 = static_cast<uint8_t*>(s1);
  prm.sp_q0 = make_span(q0, static_cast<uint64_t>(M) * K);
  prm.sp_s0 = make_span(s0, blk_bytes(M, K / 32));
  prm.sp_s1 = make_span(s1, blk_bytes(K, M / 32));
  const int grid = static_cast<int>(prm.n_tiles < num_sms ? prm.n_tiles : num_sms);
  if (grid <= 0) return 0;
  if (dim0 && dim1) return launch_tiles<kModeFused2D>(maps, prm, grid, stream);
  return dim0 ? launch_tiles<kModeDim0>(maps, prm, grid, stream)
              : launch_tiles<kModeDim1>(maps, prm, grid, stream);
}

// ---- the fused cast with a fixed scratch array (mx_cast_dim0_dim1_noalloc) ----
//
// Scratch of mx_cast_dim0_dim1_noalloc: its tile-claim counter lives here,
// in memory that exists from the moment the library is loaded on a GPU until
// the process exits, so a call allocates nothing.  64 words (256 bytes)
// are reserved; a call uses one.  The host cannot use the name of this array
// as a device address: noalloc_scratch() asks the runtime for that address,
// once per device, with the device current.
constexpr int kNoAllocScratchWords = 64;
static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoAllocScratchWords];

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call for that device; null (and *rc set) if the lookup failed.
unsigned int* noalloc_scratch(int* rc) {
  static std::mutex mu;
  static unsigned int* addr[DeviceCache::kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *rc = static_cast<int>(e);
    return nullptr;
  }
  if (dev < 0 || dev >= DeviceCache::kMaxDevices) {
    *rc = static_cast<int>(cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *rc = static_cast<int>(e);
      return nullptr;
    }
    addr[dev] = static_cast<unsigned int*>(ptr);
  }
  *rc = 0;
  return addr[dev];
}

int launch_cast_2d_noalloc(const CastMaps& maps, int64_t M, int64_t K, void* q0, void* s0,
                           void* q1, void* s1, int num_sms, cudaStream_t stream,
                           int64_t* scratch_words) {
  (void)q1;   // written through maps.q1e / maps.q1o
  Params prm = {};
  const Stall stall = take_stall();
  prm.stall_at = stall.at;
  prm.stall_ns = stall.ns;
  prm.q0 = static_cast<uint8_t*>(q0);
  prm.M = M;
  prm.K = K;
  prm.n_mt = static_cast<int32_t>((M + kTile - 1) / kTile);
  prm.n_kt = static_cast<int32_t>((K + kTile - 1) / kTile);
  prm.n_tiles = static_cast<int64_t>(prm.n_mt) * prm.n_kt;
  prm.s0 = static_cast<uint8_t*>(s0);
  prm.s1 = static_cast<uint8_t*>(s1);
  prm.sp_q0 = make_span(q0, static_cast<uint64_t>(M) * K);
  prm.sp_s0 = make_span(s0, blk_bytes(M, K / 32));
  prm.sp_s1 = make_span(s1, blk_bytes(K, M / 32));
  const int grid = static_cast<int>(prm.n_tiles < num_sms ? prm.n_tiles : num_sms);
  if (grid <= 0) return 0;
  // Scratch this call needs: one counter when it claims tiles, else none.
  const bool claim = prm.n_tiles / grid >= kClaimMinRounds;
  *scratch_words = claim ? 1 : 0;
  if (*scratch_words > kNoAllocScratchWords) return static_cast<int>(cudaErrorInvalidValue);
  if (!claim) return launch<kModeFused2D, false>(maps, prm, grid, stream);
  int rc = 0;
  prm.claims = noalloc_scratch(&rc);
  if (!prm.claims) return rc;
  // The counter must start at zero; a call that gave up may have left it
  // short of its reset, so clear it on the stream first.
  cudaError_t e = cudaMemsetAsync(prm.claims, 0, sizeof(unsigned int), stream);
  if (e != cudaSuccess) return static_cast<int>(e);
  return launch<kModeFused2D, true>(maps, prm, grid, stream);
}

int noalloc_scratch_words() { return kNoAllocScratchWords; }

int launch_cast_experts(const CastMaps& maps, int64_t E, int64_t N, int64_t K, void* q0,
                        void* s0, void* s1, int num_sms, cudaStream_t stream) {
  const bool dim0 = q0 != nullptr;
  const bool dim1 = s1 != nullptr;
  Params prm = {};
  const Stall stall = take_stall();
  prm.stall_at = stall.at;
  prm.stall_ns = stall.ns;
  prm.q0 = static_cast<uint8_t*>(q0);
  prm.s0 = static_cast<uint8_t*>(s0);
  prm.kb4 = static_cast<int32_t>(((K / 32) + 3) / 4 * 4);
  prm.s0_expert_bytes = (N + 127) / 128 * 128 * prm.kb4;
  prm.s0_scatter = (N % 128) != 0;
  prm.M = E * N;
  prm.K = K;
  prm.n_mt = static_cast<int32_t>((prm.M + kTile - 1) / kTile);
  prm.n_kt = static_cast<int32_t>((K + kTile - 1) / kTile);
  prm.n_tiles = static_cast<int64_t>(prm.n_mt) * prm.n_kt;
  prm.s1 = static_cast<uint8_t*>(s1);
  prm.N = N;
  prm.nb4 = static_cast<int32_t>(((N / 32) + 3) / 4 * 4);
  prm.s1_expert_bytes = ((K + 127) / 128) * 128 * prm.nb4;
  prm.s1_scatter = (N % 128) != 0;
  prm.sp_q0 = make_span(q0, static_cast<uint64_t>(prm.M) * K);
  prm.sp_s0 = make_span(s0, static_cast<uint64_t>(E) * prm.s0_expert_bytes);
  prm.sp_s1 = make_span(s1, static_cast<uint64_t>(E) * prm.s1_expert_bytes);
  const int grid = static_cast<int>(prm.n_tiles < num_sms ? prm.n_tiles : num_sms);
  if (grid <= 0) return 0;
  if (dim0 && dim1) return launch_tiles<kModeExperts01>(maps, prm, grid, stream);
  return dim0 ? launch_tiles<kModeExperts0>(maps, prm, grid, stream)
              : launch_tiles<kModeExperts>(maps, prm, grid, stream);
}

int launch_cast_grouped(const CastMaps& maps, int64_t M, int64_t K, const int32_t* offs, int G,
                        void* q0, void* q1, void* s0, int64_t* row_offs, int64_t* col_offs,
                        void* s1, int32_t* status, int num_sms, cudaStream_t stream) {
  Params prm = {};
  const Stall stall = take_stall();
  prm.stall_at = stall.at;
  prm.stall_ns = stall.ns;
  prm.q0 = static_cast<uint8_t*>(q0);
  prm.M = M;
  prm.K = K;
  prm.n_kt = static_cast<int32_t>((K + kTile - 1) / kTile);
  prm.n_mt = static_cast<int32_t>((M + kTile - 1) / kTile + G);   // upper bound
  prm.s0 = static_cast<uint8_t*>(s0);
  prm.s1 = static_cast<uint8_t*>(s1);
  prm.q1 = static_cast<uint8_t*>(q1);
  prm.offs = offs;
  prm.row_offs = row_offs;
  prm.status = status;
  prm.row_offs_out = row_offs;
  prm.col_offs_out = col_offs;
  prm.status_out = status;
  prm.G = G;
  prm.k128 = static_cast<int32_t>((K + 127) / 128 * 128);
  prm.q1_tma = (M % 16) == 0;
  prm.sp_q0 = make_span(q0, static_cast<uint64_t>(M) * K);
  prm.sp_q1 = make_span(q1, static_cast<uint64_t>(M) * K);
  prm.sp_s0 = make_span(s0, static_cast<uint64_t>(M + 128 * static_cast<int64_t>(G)) *
                                static_cast<uint64_t>(prm.n_kt) * 4);
  prm.sp_s1 = make_span(s1, static_cast<uint64_t>(prm.k128) *
                                static_cast<uint64_t>((M + 31) / 32 + 4 * static_cast<int64_t>(G)));
  prm.sp_ro = make_span(row_offs, 8 * static_cast<uint64_t>(G + 1));
  prm.sp_co = make_span(col_offs, 8 * static_cast<uint64_t>(G + 1));
  prm.sp_st = make_span(status, 4);
  if (G > kMaxSmemGroups) {
    // Large group counts: the padded offsets come from a separate kernel.
    if (int rc = launch_group_offsets(offs, G, M, row_offs, col_offs, status, stream)) return rc;
  }
  const int64_t bound = static_cast<int64_t>(prm.n_mt) * prm.n_kt;
  const int grid = static_cast<int>(bound < num_sms ? (bound > 0 ? bound : 1) : num_sms);
  // A CTA's run is at most ceil(bound / grid) tiles: below kBandMinRun no
  // group can be banded, and the plain cursor is taken.
  if ((bound + grid - 1) / grid < kBandMinRun) return launch<kModeGrouped>(maps, prm, grid, stream);
  return launch<kModeGroupedBands>(maps, prm, grid, stream);
}

// Watchdog self-test: one warp waits on an mbarrier that nothing arrives at,
// with a short limit.  The wait must give up, set the device watchdog word and
// let the kernel return normally (no trap, no fault, context stays usable).
__global__ void __launch_bounds__(32) watchdog_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0u, &abort_flag, limit_ns);
  __syncwarp();
  if (threadIdx.x == 0 && !ok) atomicOr(&g_watchdog, 1);
}

int launch_watchdog_selftest(uint64_t limit_ns, cudaStream_t stream) {
  watchdog_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return static_cast<int>(cudaGetLastError());
}

int out_of_bounds_cast(bool clear) { return read_out_of_bounds(clear); }

int read_watchdog(int* out, bool clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_watchdog, sizeof(int));
  if (e != cudaSuccess) return static_cast<int>(e);
  if (clear && v) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_watchdog, &z, sizeof(int));
    if (e != cudaSuccess) return static_cast<int>(e);
    // A launch that gave up may have left its claim counter short of its
    // reset: clear them all (the caller clears the watchdog with no cast in
    // flight).
    static const unsigned int zeros[kClaimSlots] = {};
    e = cudaMemcpyToSymbol(g_claims, zeros, sizeof(zeros));
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  *out = v;
  return 0;
}

}  // namespace mx
