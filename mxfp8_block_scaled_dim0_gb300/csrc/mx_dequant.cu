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

}  // namespace

int launch_dequant_blocked(const uint8_t* q, int64_t R, int64_t C, const uint8_t* s_blk,
                           uint16_t* out, int num_sms, cudaStream_t stream) {
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

}  // namespace mx
