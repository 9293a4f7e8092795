// mx_common.cuh -- inline-PTX building blocks for the sm_103a MX-FP8 kernels:
// mbarriers with bounded waits, TMA tile loads/stores, bulk copies, and the
// per-block scale / element conversion of the MX rule.
//
// The rule (per 32-element block; OCP MX v1.0 conversion with E4M3 elements
// and an E8M0 scale, blocks of 32 along either dimension as in pytorch/ao PR
// #1869 "triton kernel to cast to mx across dim0 and dim1", summary):
//   E     = biased exponent field of the block's largest |x| (bf16 bits)
//   s     = max(E - 8, 0)          e8m0 byte; floor(log2 amax) - 8, clamped
//   mult  = 2^(127 - s)            exact float built from bits
//   q_i   = e4m3 of x_i * mult, round to nearest even, saturate to +-448
// The exponent comes from integer bit fields (no float log, as the review of
// that PR asks).  E == 255 (Inf or NaN in the block) gives s = 0xFF and a
// NaN multiplier; the product of any element with it is the positive
// canonical NaN, which the e4m3 conversion writes as 0x7F, so every element
// of such a block is 0x7F whatever the sign or payload of its NaN (the GPU
// tests check these bytes).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mx {

// ---- shared-memory addressing ---------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarriers -------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Upper bound on any single wait.  Legitimate waits here last microseconds;
// after this long the CTA gives up, raises its abort flag and winds down.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Wait for the phase of parity `parity` to complete.  Returns false if the
// CTA-wide abort flag is (or becomes) set or the time limit passes; in the
// latter case the flag is raised so that every other role stops too.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      return false;
    }
  }
}

// Wait, regardless of the abort flag, for the phase of parity `parity` to
// complete, giving up after limit_ns.  Used on the way out of a CTA that gave
// up: asynchronous copies it issued into its own shared memory must land
// before the CTA exits.  Returns false if the limit passed.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity,
                                           uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// ---- TMA (tensor) and bulk copies -------------------------------------------

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* m, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Hint: bring the tile at (x, y) of the tensor into L2.  No data reaches the
// SM and nothing waits for it.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* m, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::
                   "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y)
               : "memory");
}

// Hint: bring `bytes` bytes at g into L2 (g 16-byte aligned, bytes a
// multiple of 16).  No data reaches the SM and nothing waits for it.
__device__ __forceinline__ void bulk_prefetch_l2(const void* g, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(g)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, int32_t x, int32_t y,
                                             const void* smem_src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::
                   "l"(reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y), "r"(smem_u32(smem_src))
               : "memory");
}

// Plain bulk copy global -> smem completing on `bar` (bytes counted as
// transaction bytes); both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Plain bulk copy smem -> global; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ---- the MX rule -----------------------------------------------------------

// Running |max| of packed bf16 pairs.  max.xorsign.abs takes the larger
// magnitude of each half (with .NaN, a NaN wins); the sign bit it leaves is
// meaningless and is masked off at the end.
__device__ __forceinline__ uint32_t absmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Magnitude bits (15 bits) of the low and high halves of an absmax2 result.
__device__ __forceinline__ uint32_t mag_lo(uint32_t a) { return a & 0x7FFFu; }
__device__ __forceinline__ uint32_t mag_hi(uint32_t a) { return (a >> 16) & 0x7FFFu; }

// Scale byte and multiplier from a block's largest magnitude (bf16 bits).
__device__ __forceinline__ void mx_scale(uint32_t amax_bits, uint32_t& sbyte, float& mult) {
  const int E = static_cast<int>(amax_bits >> 7);           // 0..255
  const int s = E > 8 ? E - 8 : 0;                           // 0..247
  uint32_t mbits = static_cast<uint32_t>(254 - s) << 23;     // 2^(127 - s)
  uint32_t b = static_cast<uint32_t>(s);
  if (E == 255) {                                            // Inf / NaN block
    b = 0xFFu;
    mbits = 0x7FC00000u;                                     // NaN multiplier
  }
  sbyte = b;
  mult = __uint_as_float(mbits);
}

// bf16 halves of a packed word as exact floats.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round-to-nearest product without flush-to-zero: subnormal bf16 inputs must
// survive the multiply (a block of subnormals scales them up to e4m3 normals).
__device__ __forceinline__ float mul_rn(float a, float b) {
  float d;
  asm("mul.rn.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Four floats (f0 at the lowest address) times mult -> four e4m3 bytes packed
// little-endian.  cvt puts its first source in the high byte of each pair.
__device__ __forceinline__ uint32_t e4m3x4(float f0, float f1, float f2, float f3, float m) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(mul_rn(f0, m)), "f"(mul_rn(f1, m)), "f"(mul_rn(f2, m)), "f"(mul_rn(f3, m)));
  return r;
}

// Byte offset of scale (r, c) inside the 128x4 blocked tile that holds it:
// 32 storage rows of 16 bytes; storage row r % 32 holds rows r, r+32, r+64,
// r+96 (4 columns each).
__device__ __forceinline__ int blocked_in_tile(int r, int c) {
  return (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

// Byte offset of scale (r, c) in the blocked layout of a matrix whose padded
// column count is c4 (a multiple of 4): tiles of 128 x 4, row-major.
__device__ __forceinline__ int64_t blocked_offset(int64_t r, int64_t c, int64_t c4) {
  return ((r >> 7) * (c4 >> 2) + (c >> 2)) * 512 + blocked_in_tile(static_cast<int>(r & 127),
                                                                    static_cast<int>(c & 3));
}

// ---- bounds-checked builds ------------------------------------------------
//
// Built with -DMX_DEBUG_BOUNDS, every global store a kernel issues from its
// threads is checked against the buffer it belongs to: a store that would
// leave the buffer is skipped and counted in a device word of the translation
// unit (read through mx_bounds_check()), never trapped.  The stand-in for a
// memory checker on machines where none may run.  Release builds compile the
// checks away.  (TMA tensor stores are bounded by their tensor map's extents
// in hardware.)

// One output buffer: [base, base + size).
struct Span {
  uint8_t* base;
  uint64_t size;
};

#ifdef MX_DEBUG_BOUNDS
static __device__ unsigned int g_out_of_bounds = 0;
#endif

// Checked builds also carry the diagnostic stall hook (mx_selftest_arm_stall:
// a wait that runs out on purpose, to drive a kernel's abort path).  Release
// builds compile it away: even a never-taken check where loads are issued
// measured 0.2-0.7% on the cast kernels and 4% on the rowwise kernel.
#ifdef MX_DEBUG_BOUNDS
constexpr bool kDiagStall = true;
#else
constexpr bool kDiagStall = false;
#endif

__device__ __forceinline__ bool in_span(const Span& s, const void* p, uint64_t n) {
#ifdef MX_DEBUG_BOUNDS
  const uint64_t a = reinterpret_cast<uint64_t>(p);
  const uint64_t b = reinterpret_cast<uint64_t>(s.base);
  if (s.base != nullptr && a >= b && a - b + n <= s.size) return true;
  atomicAdd(&g_out_of_bounds, 1u);
  return false;
#else
  (void)s;
  (void)p;
  (void)n;
  return true;
#endif
}

inline Span make_span(void* base, uint64_t size) {
  return Span{static_cast<uint8_t*>(base), size};
}

// Host: this translation unit's count of refused stores (cleared on request),
// or -1 in a release build.
static inline int read_out_of_bounds(bool clear) {
#ifdef MX_DEBUG_BOUNDS
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_out_of_bounds, sizeof(v)) != cudaSuccess) return -2;
  if (clear && v) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_out_of_bounds, &z, sizeof(z)) != cudaSuccess) return -2;
  }
  return static_cast<int>(v);
#else
  (void)clear;
  return -1;
#endif
}

}  // namespace mx
