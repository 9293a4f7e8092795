// mx_dequant.cu -- MX-FP8 dequantisation for sm_103a: e4m3 elements with e8m0
// scales in the 128x4 blocked layout -> bf16.
//
// The value of an MX element is its scale times its element value (OCP
// Microscaling Formats (MX) v1.0, MX block definition): out = e4m3(q) *
// 2^(s - 127), rounded once to bf16.  This is the step a consumer of the
// cast's outputs takes back to high precision; applied to the dim1 copy
// (K x M) it gives X's transpose.
//
// Exactness: e4m3 -> f16 -> f32 is exact, and the product of a 4-significant-
// bit value with a power of two in [2^-127, 2^127] is exact in f32 (products
// reach down to 2^-136, well above f32's smallest subnormal 2^-149, and any
// product of 2^128 or more overflows to infinity, where bf16 would too).  The
// single rounding is the final f32 -> bf16 conversion, to nearest even, with
// subnormals kept.  Scale byte 0xFF (NaN) makes the product NaN.
//
// HBM-bound: 1 byte read + 2 bytes written per element, plus 1/32 byte of
// scale.  Each thread converts 8 consecutive elements per step (an 8-byte
// load, one 16-byte store; a warp moves 256 contiguous bytes in and 512 out
// per instruction).  A CTA of 256 threads covers a "tile" of 256 such
// chunks: part of one row when rows are long, several whole rows when they
// are short.  One wave of resident CTAs strides over the tiles together (all
// CTAs work on neighbouring tiles at any time, which keeps DRAM accesses
// local), two tiles' loads in flight per thread.  Measured on GB300 at
// 16384^2: with 16-byte thread stores this read-1 / write-2 mix tops out near
// 5.9 TB/s even for a plain zero-extending copy, which this kernel matches;
// four tiles per thread, 16 elements per thread, or contiguous per-CTA runs
// of tiles were 4-20% slower.  Staging 8192-element tiles in shared memory
// and writing each with one bulk async copy was byte-identical but no faster
// (slower for rows of 12288 values, faster only for rows of about 1024).
#include <cuda_runtime.h>

#include "mx_common.cuh"
#include "mx_kernels.h"

namespace mx {
namespace {

constexpr int kDqThreads = 256;
constexpr int kDqUnroll = 2;

struct DqParams {
  const uint8_t* q;
  const uint8_t* s;
  uint16_t* out;
  int64_t R, C;
  int64_t cpr;        // 8-element chunks per row (C / 8)
  int64_t n_ct;       // tiles per row band (ceil(cpr / 256), or 1)
  int64_t n_tiles;
  int32_t rpt;        // rows per tile band (256 / cpr when cpr < 256, else 1)
  int32_t cb4;        // ceil4(C / 32): padded scale columns
  Span sp_out;        // for the bounds-checked build
};

// Four e4m3 bytes -> four f32 values (exact).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float f[4]) {
  uint32_t h01, h23;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(h01), "=r"(h23)
      : "r"(w));
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.f32.f16 %0, a;\n\t"
      "cvt.f32.f16 %1, b;\n\t}"
      : "=f"(f[0]), "=f"(f[1])
      : "r"(h01));
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.f32.f16 %0, a;\n\t"
      "cvt.f32.f16 %1, b;\n\t}"
      : "=f"(f[2]), "=f"(f[3])
      : "r"(h23));
}

// Two f32 -> bf16x2 (lo = a), round to nearest even, subnormals kept.
__device__ __forceinline__ uint32_t bf16x2_rn(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// 2^(s - 127) as an f32 (s = 0: the subnormal 2^-127; s = 255: NaN).
__device__ __forceinline__ float e8m0_value(uint32_t s) {
  const uint32_t bits = s == 0xFFu ? 0x7FC00000u : (s == 0u ? 0x00400000u : (s << 23));
  return __uint_as_float(bits);
}

__device__ __forceinline__ uint4 dequant8(uint2 v, float m) {
  float f[8];
  e4m3x4_to_f32(v.x, f);
  e4m3x4_to_f32(v.y, f + 4);
  uint4 o;
  o.x = bf16x2_rn(mul_rn(f[0], m), mul_rn(f[1], m));
  o.y = bf16x2_rn(mul_rn(f[2], m), mul_rn(f[3], m));
  o.z = bf16x2_rn(mul_rn(f[4], m), mul_rn(f[5], m));
  o.w = bf16x2_rn(mul_rn(f[6], m), mul_rn(f[7], m));
  return o;
}

__global__ void __launch_bounds__(kDqThreads) dequant_blocked_kernel(const DqParams p) {
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    // While earlier grids finish, ask L2 for this CTA's first tiles of q (a
    // hint only; every access waits below): whole rows of a band, or 2 KB
    // of one row.
    for (int u = 0; u < kDqUnroll; ++u) {
      const int64_t t = blockIdx.x + static_cast<int64_t>(u) * gridDim.x;
      if (t >= p.n_tiles) break;
      const int64_t band = t / p.n_ct, ct = t - band * p.n_ct;
      int64_t off, bytes;
      if (p.rpt > 1 || p.cpr < kDqThreads) {
        const int64_t r0 = band * p.rpt;
        off = r0 * p.C;
        bytes = (p.R - r0 < p.rpt ? p.R - r0 : p.rpt) * p.C;
      } else {
        off = band * p.C + ct * (8 * kDqThreads);
        bytes = p.C - ct * (8 * kDqThreads);
        if (bytes > 8 * kDqThreads) bytes = 8 * kDqThreads;
      }
      bulk_prefetch_l2(p.q + off, static_cast<uint32_t>(bytes));
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // This thread's place inside a tile: row offset within the band and chunk.
  int32_t row_off = 0;
  int64_t chunk_in = threadIdx.x;
  bool active = true;
  if (p.rpt > 1 || p.cpr < kDqThreads) {
    row_off = static_cast<int32_t>(threadIdx.x / static_cast<uint32_t>(p.cpr));
    chunk_in = threadIdx.x - static_cast<int64_t>(row_off) * p.cpr;
    active = row_off < p.rpt;
  }
  const uint32_t n_tiles = static_cast<uint32_t>(p.n_tiles);   // < 2^32 (checked on the host)
  const uint32_t n_ct = static_cast<uint32_t>(p.n_ct);
  for (uint32_t t0 = blockIdx.x; t0 < n_tiles; t0 += gridDim.x * kDqUnroll) {
    uint2 v[kDqUnroll];
    uint32_t sc[kDqUnroll];
    int64_t off[kDqUnroll];
    bool ok[kDqUnroll];
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
      const uint32_t t = t0 + u * gridDim.x;
      const uint32_t band = n_ct == 1 ? t : t / n_ct;
      const uint32_t ct = t - band * n_ct;
      const int64_t row = static_cast<int64_t>(band) * p.rpt + row_off;
      const int64_t chunk = static_cast<int64_t>(ct) * kDqThreads + chunk_in;
      ok[u] = active && t < n_tiles && row < p.R && chunk < p.cpr;
      off[u] = row * p.C + chunk * 8;
      if (ok[u]) {
        v[u] = __ldg(reinterpret_cast<const uint2*>(p.q + off[u]));
        sc[u] = __ldg(p.s + blocked_offset(row, chunk >> 2, p.cb4));
      }
    }
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
      if (ok[u] && in_span(p.sp_out, p.out + off[u], 16))
        *reinterpret_cast<uint4*>(p.out + off[u]) = dequant8(v[u], e8m0_value(sc[u]));
    }
  }
}

// ---- tiled kernel (rows of 128 values or more) --------------------------------
//
// Persistent, one CTA per SM, warp-specialised like the cast kernels: a
// producer warp brings each 128 x 128 tile of q (16 KB, TMA, 128B swizzle)
// and the one 512-byte blocked scale tile that covers it (a 128 x 128 tile of
// q has exactly one: 128 rows x 4 scale columns) into a ring of stages; eight
// compute warps convert the tile into a bf16 staging tile (two 64-column
// halves, 128B swizzle); a store warp writes each staging tile out with two
// TMA tensor stores.  Tiles past the matrix's edge are zero-filled on load and
// clipped on store by the tensor maps, so any R and any C % 32 == 0 works.
// Every wait is bounded; on time-out the CTA stops, lets its copies in flight
// land and reports through g_dequant_watchdog.
constexpr int kDqTile = 128;
constexpr int kDqInBytes = kDqTile * kDqTile;       // e4m3 tile
constexpr int kDqScaleBytes = 512;                  // one blocked scale tile
constexpr int kDqOutHalf = kDqTile * 128;           // 64 bf16 columns x 128 rows
constexpr int kDqOutBytes = 2 * kDqOutHalf;
constexpr int kDqStages = 4;                        // input ring depth
constexpr int kDqStaging = 4;                       // output staging buffers
constexpr int kDqComputeWarps = 8;
constexpr int kDqProducerWarp = kDqComputeWarps;
constexpr int kDqStoreWarp = kDqComputeWarps + 1;
constexpr int kDqTmaThreads = (kDqComputeWarps + 2) * 32;
constexpr int kDqOffIn = 0;
constexpr int kDqOffOut = kDqOffIn + kDqStages * kDqInBytes;
constexpr int kDqOffScale = kDqOffOut + kDqStaging * kDqOutBytes;
constexpr int kDqOffBar = kDqOffScale + kDqStages * kDqScaleBytes;
constexpr int kDqNumBars = 2 * kDqStages + 2 * kDqStaging + 1;   // + the diagnostic stall
constexpr int kDqOffFlag = kDqOffBar + kDqNumBars * 8;
constexpr int kDqSmemBytes = kDqOffFlag + 16 + 1024;             // + alignment slack
static_assert(kDqSmemBytes <= 227 * 1024, "shared memory budget");

__device__ int g_dequant_watchdog = 0;

struct DqTmaParams {
  const uint8_t* s;      // blocked scales
  int64_t C;             // columns
  int64_t n_tc;          // tile columns, ceil(C / 128)
  int64_t n_tiles;
  int64_t s_tiles_row;   // blocked scale tiles per 128-row band, ceil4(C / 32) / 4
  int64_t stall_at;      // diagnostic stall (mx_kernels.h), -1 in normal use
  uint64_t stall_ns;
};

__global__ void __launch_bounds__(kDqTmaThreads, 1)
    dequant_tma_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_out, const DqTmaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDqOffBar);   // [kDqStages] tile landed
  uint64_t* empty = full + kDqStages;                                // [kDqStages] tile read
  uint64_t* sfull = empty + kDqStages;                               // [kDqStaging] staged
  uint64_t* sempty = sfull + kDqStaging;                             // [kDqStaging] drained
  uint64_t* stall_bar = sempty + kDqStaging;                         // never completed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kDqOffFlag);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDqStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDqComputeWarps);
    }
    for (int o = 0; o < kDqStaging; ++o) {
      mbar_init(&sfull[o], kDqComputeWarps);
      mbar_init(&sempty[o], 1);
    }
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Programmatic dependent launch: the barriers above touch no global memory;
  // every global access waits for the earlier grids.  Meanwhile the producer
  // asks L2 for the tiles its ring loads first (a hint only: nothing reaches
  // the SM before the wait, and the loads after it see the earlier grids'
  // writes, L2 being where global memory is coherent).
  asm volatile("griddepcontrol.launch_dependents;");
  if (warp == kDqProducerWarp && lane == 0) {
    for (int i = 0; i < kDqStages; ++i) {
      const int64_t t = blockIdx.x + static_cast<int64_t>(gridDim.x) * i;
      if (t >= p.n_tiles) break;
      const int64_t tr = t / p.n_tc, tc = t - tr * p.n_tc;
      tma_prefetch_2d(&tm_q, static_cast<int32_t>(tc * kDqTile), static_cast<int32_t>(tr * kDqTile));
      bulk_prefetch_l2(p.s + (tr * p.s_tiles_row + tc) * kDqScaleBytes, kDqScaleBytes);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();

  int64_t issued = 0;   // producer lane: tiles whose loads were issued
  if (warp == kDqProducerWarp) {
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      int64_t it = 0;
      for (int64_t t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++it) {
        const int s = static_cast<int>(it % kDqStages);
        if (kDiagStall && it == p.stall_at && blockIdx.x == 0) {
          // Diagnostic (checked builds, armed from the host): a wait that runs out in
          // place of this tile's loads; every role stops on the abort flag.
          mbar_wait(stall_bar, 0u, abort_flag, p.stall_ns);
          break;
        }
        if (!mbar_wait(&empty[s], static_cast<uint32_t>(((it / kDqStages) & 1) ^ 1), abort_flag))
          break;
        const int64_t tr = t / p.n_tc, tc = t - tr * p.n_tc;
        mbar_arrive_expect_tx(&full[s], kDqInBytes + kDqScaleBytes);
        tma_load_2d(smem + kDqOffIn + s * kDqInBytes, &tm_q, static_cast<int32_t>(tc * kDqTile),
                    static_cast<int32_t>(tr * kDqTile), &full[s]);
        bulk_load(smem + kDqOffScale + s * kDqScaleBytes,
                  p.s + (tr * p.s_tiles_row + tc) * kDqScaleBytes, kDqScaleBytes, &full[s]);
        issued = it + 1;
      }
    }
    __syncwarp();
  } else if (warp == kDqStoreWarp) {
    if (lane == 0) {
      prefetch_tmap(&tm_out);
      int64_t it = 0;
      for (int64_t t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++it) {
        const int o = static_cast<int>(it % kDqStaging);
        if (!mbar_wait(&sfull[o], static_cast<uint32_t>((it / kDqStaging) & 1), abort_flag)) break;
        const int64_t tr = t / p.n_tc, tc = t - tr * p.n_tc;
        const uint8_t* stg = smem + kDqOffOut + o * kDqOutBytes;
        const int32_t x0 = static_cast<int32_t>(tc * kDqTile), y0 = static_cast<int32_t>(tr * kDqTile);
        tma_store_2d(&tm_out, x0, y0, stg);
        // (the right half of the last tile column may lie wholly past the
        // matrix when C % 128 != 0: no store starts outside it)
        if (x0 + 64 < p.C) tma_store_2d(&tm_out, x0 + 64, y0, stg + kDqOutHalf);
        // Keep the newest bulk group in flight: the previous tile's staging
        // buffer is released once its own group has been read.
        bulk_commit();
        bulk_wait_read<1>();
        if (it > 0) mbar_arrive(&sempty[static_cast<int>((it - 1) % kDqStaging)]);
      }
      bulk_wait<0>();
    }
    __syncwarp();
  } else {
    // Compute warp w converts rows 16w .. 16w + 15, two per step: lane l takes
    // row 16w + 2k + (l >> 4), 64-column half h = (l >> 3) & 1 and the eight
    // values of output chunk j = l & 7 of that half.  Its 8 input bytes lie in
    // input chunk 4h + (j >> 1); each half-warp reads one whole 128-byte row of
    // q and each 8-lane phase writes eight distinct chunks of one staging row
    // (both conflict-free under the swizzle).
    const int h = (lane >> 3) & 1;
    const int j = lane & 7;
    const int cin = 4 * h + (j >> 1);
    const int c4 = 2 * h + (j >> 2);                 // scale column within the tile
    int64_t it = 0;
    for (int64_t t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++it) {
      const int s = static_cast<int>(it % kDqStages);
      const int o = static_cast<int>(it % kDqStaging);
      bool ok = mbar_wait(&full[s], static_cast<uint32_t>((it / kDqStages) & 1), abort_flag);
      ok = ok && mbar_wait(&sempty[o], static_cast<uint32_t>(((it / kDqStaging) & 1) ^ 1),
                           abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint8_t* in = smem + kDqOffIn + s * kDqInBytes;
      const uint8_t* sc = smem + kDqOffScale + s * kDqScaleBytes;
      uint8_t* stg = smem + kDqOffOut + o * kDqOutBytes + h * kDqOutHalf;
#pragma unroll 4
      for (int k = 0; k < 8; ++k) {
        const int r = 16 * warp + 2 * k + (lane >> 4);
        const int sw = r & 7;
        const uint2 v =
            *reinterpret_cast<const uint2*>(in + r * 128 + ((cin ^ sw) << 4) + 8 * (j & 1));
        const uint32_t sb = sc[blocked_in_tile(r, c4)];
        *reinterpret_cast<uint4*>(stg + r * 128 + ((j ^ sw) << 4)) = dequant8(v, e8m0_value(sb));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      fence_proxy_async_smem();                      // staging writes -> TMA store reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfull[o]);
    }
  }

  __syncthreads();
  if (*abort_flag && warp == kDqProducerWarp && lane == 0) {
    // A role gave up: let each stage's last issued load land (bounded) before
    // the CTA exits, then report.
    for (int s = 0; s < kDqStages; ++s) {
      if (issued <= s) break;
      const int64_t last = s + (issued - 1 - s) / kDqStages * kDqStages;
      mbar_drain(&full[s], static_cast<uint32_t>((last / kDqStages) & 1));
    }
    atomicOr(&g_dequant_watchdog, 1);
  }
}

}  // namespace

int launch_dequant_blocked(const DqMaps* maps, const uint8_t* q, int64_t R, int64_t C,
                           const uint8_t* s_blk, uint16_t* out, int num_sms, cudaStream_t stream) {
  if (C >= kDqTmaMinCols) {
    DqTmaParams p = {};
    p.s = s_blk;
    p.C = C;
    p.n_tc = (C + kDqTile - 1) / kDqTile;
    p.n_tiles = (R + kDqTile - 1) / kDqTile * p.n_tc;
    p.s_tiles_row = ((C / 32) + 3) / 4;
    const Stall stall = take_stall();
    p.stall_at = stall.at;
    p.stall_ns = stall.ns;
    static DeviceCache attr_cache;
    const int attr = attr_cache.get([] {
      return static_cast<int>(cudaFuncSetAttribute(
          dequant_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmemBytes));
    });
    if (attr != 0) return attr;
    const int grid = static_cast<int>(p.n_tiles < num_sms ? p.n_tiles : num_sms);
    if (grid <= 0) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDqTmaThreads);
    cfg.dynamicSmemBytes = kDqSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr_pdl[1];
    attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr_pdl;
    cfg.numAttrs = 1;
    return static_cast<int>(cudaLaunchKernelEx(&cfg, dequant_tma_kernel, maps->q, maps->out, p));
  }
  DqParams p = {};
  p.q = q;
  p.s = s_blk;
  p.out = out;
  p.R = R;
  p.C = C;
  p.cpr = C / 8;
  if (p.cpr >= kDqThreads) {
    p.rpt = 1;
    p.n_ct = (p.cpr + kDqThreads - 1) / kDqThreads;
    p.n_tiles = R * p.n_ct;
  } else {
    p.rpt = static_cast<int32_t>(kDqThreads / p.cpr);
    p.n_ct = 1;
    p.n_tiles = (R + p.rpt - 1) / p.rpt;
  }
  p.cb4 = static_cast<int32_t>(((C / 32) + 3) / 4 * 4);
  p.sp_out = make_span(out, 2 * static_cast<uint64_t>(R) * static_cast<uint64_t>(C));
  if (p.n_tiles > 0xFFFFFFFFll - 2ll * 65536 * 1024) return static_cast<int>(cudaErrorInvalidValue);
  // One wave of resident CTAs (as many per SM as registers allow) striding
  // over the tiles together.
  static DeviceCache occ;
  const int per_sm = occ.get([] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dequant_blocked_kernel, kDqThreads, 0) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    return n;
  });
  const int64_t want = static_cast<int64_t>(num_sms) * per_sm;
  const int grid = static_cast<int>(p.n_tiles < want ? p.n_tiles : want);
  if (grid <= 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDqThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, dequant_blocked_kernel, p));
}

int out_of_bounds_dequant(bool clear) { return read_out_of_bounds(clear); }

int read_dequant_watchdog(int* out, bool clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_dequant_watchdog, sizeof(int));
  if (e != cudaSuccess) return static_cast<int>(e);
  if (clear && v) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_dequant_watchdog, &z, sizeof(int));
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  *out = v;
  return 0;
}

}  // namespace mx
