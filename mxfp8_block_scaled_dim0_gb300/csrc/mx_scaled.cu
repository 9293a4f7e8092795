// mx_scaled.cu -- the non-MX fp8 casts for sm_103a: one scale per tensor
// (tensorwise) or per row (rowwise), the contrast cases to the MX block cast.
//
// Tensorwise (pytorch/ao PR #1445 "[float8nocompile] Triton kernels for
// conversion to float8 dtypes": local amaxes in parallel, one global amax,
// then the conversion; the scale computed locally by every block of the
// conversion kernel, as that discussion proposes):
//   amax  = max |x|; scale = fp32(448 / amax) (amax = 0 -> 1, overflow ->
//   the largest finite fp32); q = e4m3(fp32(x * scale)), nearest even,
//   saturated.
//   tensor_amax_kernel  one wave of CTAs, 16-byte loads, a running bf16x2
//                       magnitude maximum (max.NaN.xorsign.abs, so a NaN
//                       anywhere makes the amax NaN), one integer atomicMax
//                       per CTA on the fp32 bits into the caller's amax word
//                       (cleared first; non-negative floats order like their
//                       bit patterns)
//   tensorwise_kernel   programmatic dependent of the amax kernel; walks the
//                       tensor from the end, so the part of x still in L2 from
//                       the amax pass is read first
// Rowwise ("FP8 linear triton with row-wise scaling" gist,
// quantize_fp8_rowwise): scale_r = bf16(amax_r / 448), q = e4m3(fp32(x /
// scale_r)); a zero scale gives signed zeros.  A group of T threads (32 to
// 256, by K) owns a row.  The rows of each step (one to eight) arrive in
// shared memory by one bulk async copy issued steps ahead (rowwise_bulk_kernel;
// rows longer than 24576 values are read from global memory twice instead);
// the group reduces the row's amax, then divides and converts.  The division
// is a reciprocal product with one residual correction, exact for these
// operands (row_quot_fast).
//
// Exactness against a single rounding: the fp32 product of a bf16 value and
// an fp32 scale is rounded once by mul.rn and once more by the e4m3
// conversion, as the pages' fp32 arithmetic does; the fp32 quotients (div.rn,
// IEEE) likewise.  448 / amax and amax / 448 are rounded to fp32 and then (row
// scale) to bf16; double rounding of a quotient through a format with at least
// 2p + 2 bits is harmless, so the bf16 scale equals the nearest bf16 to the
// exact quotient.
#include <cuda_runtime.h>
#include <float.h>

#include "mx_common.cuh"
#include "mx_kernels.h"

namespace mx {
namespace {

constexpr int kThreads = 256;
// Bulk-staged rowwise: ring bytes per CTA (2 to 8 stages), and the largest
// stage (rows of one step) it takes.  The launch shape (threads per row, ring
// depth) follows a sweep on GB300 over K = 1024 ... 16384, every variant
// byte-identical: e.g. 16640 x 5120 took 70.5 us with 256 threads per row and
// 41.7 us with 64; 16384^2 took 135.2 us with two 32 KB stages per CTA and
// 122.6 us with three.
constexpr int64_t kRowRing = 48 * 1024;
constexpr int64_t kMaxRowStage = 48 * 1024;

__device__ __forceinline__ float div_rn(float a, float b) {
  float r;
  asm("div.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Two fp32 values -> two e4m3 bytes (lo = a), nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// Running bf16x2 magnitude maximum: acc takes the larger |value| of the eight
// values of a 16-byte chunk in each half (max.NaN.xorsign.abs.bf16x2: a NaN
// anywhere propagates; the sign bit of the result is not used).
__device__ __forceinline__ uint32_t absmax8(uint32_t acc, uint4 v) {
  return absmax2(acc, absmax2(absmax2(v.x, v.y), absmax2(v.z, v.w)));
}

// Largest bf16 magnitude (bits, 15 of them) held in a bf16x2 accumulator.
__device__ __forceinline__ uint32_t mag_of(uint32_t acc) {
  return max(acc & 0x7FFFu, (acc >> 16) & 0x7FFFu);
}

__device__ __forceinline__ uint32_t block_max(uint32_t v, uint32_t* red) {
  v = __reduce_max_sync(0xffffffffu, v);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  uint32_t m = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) m = max(m, red[w]);
  return m;
}

__global__ void __launch_bounds__(kThreads) tensor_amax_kernel(const uint16_t* x, int64_t n,
                                                               uint32_t* amax_bits, Span sp_amax) {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ uint32_t red[kThreads / 32];
  const int64_t chunks = n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  // Eight 16-byte loads in flight per thread: a probe of this read-only pass
  // at 16384^2 ran 75.8 us with eight, 78.6 us with two or four.
  constexpr int kU = 8;
  uint32_t m = 0;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; c < chunks;
       c += kU * stride) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      v[u] = c + u * stride < chunks ? __ldg(reinterpret_cast<const uint4*>(x) + c + u * stride)
                                     : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < kU; ++u) m = absmax8(m, v[u]);
  }
  m = mag_of(m);
  if (blockIdx.x == 0 && threadIdx.x == 0)
    for (int64_t i = chunks << 3; i < n; ++i) m = max(m, static_cast<uint32_t>(x[i] & 0x7FFFu));
  m = block_max(m, red);
  if (threadIdx.x == 0 && m != 0 && in_span(sp_amax, amax_bits, 4)) atomicMax(amax_bits, m << 16);
}

__device__ __forceinline__ float tensor_scale(uint32_t amax_bits) {
  const float a = __uint_as_float(amax_bits);
  if (a == 0.0f) return 1.0f;
  const float s = div_rn(448.0f, a);
  return s > FLT_MAX ? FLT_MAX : s;   // NaN stays NaN
}

__global__ void __launch_bounds__(kThreads) tensorwise_kernel(const uint16_t* x, int64_t n,
                                                              const uint32_t* amax_bits,
                                                              uint8_t* q, float* scale_out,
                                                              Span sp_q, Span sp_scale) {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float s = tensor_scale(*amax_bits);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (in_span(sp_scale, scale_out, 4)) *scale_out = s;
    for (int64_t i = (n >> 3) << 3; i < n; ++i) {
      const float v = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
      if (in_span(sp_q, q + i, 1)) q[i] = static_cast<uint8_t>(e4m3x2(mul_rn(v, s), 0.0f) & 0xFFu);
    }
  }
  const int64_t chunks = n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  // From the last chunk backwards.
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; k < chunks;
       k += 2 * stride) {
    const int64_t c0 = chunks - 1 - k;
    const int64_t c1 = c0 - stride;
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(x) + c0);
    uint4 b = make_uint4(0, 0, 0, 0);
    if (c1 >= 0) b = __ldg(reinterpret_cast<const uint4*>(x) + c1);
    uint2 oa, ob;
    oa.x = e4m3x4(bf_lo(a.x), bf_hi(a.x), bf_lo(a.y), bf_hi(a.y), s);
    oa.y = e4m3x4(bf_lo(a.z), bf_hi(a.z), bf_lo(a.w), bf_hi(a.w), s);
    if (in_span(sp_q, q + 8 * c0, 8)) reinterpret_cast<uint2*>(q)[c0] = oa;
    if (c1 >= 0) {
      ob.x = e4m3x4(bf_lo(b.x), bf_hi(b.x), bf_lo(b.y), bf_hi(b.y), s);
      ob.y = e4m3x4(bf_lo(b.z), bf_hi(b.z), bf_lo(b.w), bf_hi(b.w), s);
      if (in_span(sp_q, q + 8 * c1, 8)) reinterpret_cast<uint2*>(q)[c1] = ob;
    }
  }
}

// x / s for one bf16 value; a zero scale gives a signed zero.
__device__ __forceinline__ float row_quot(float v, float s) {
  return s == 0.0f ? __uint_as_float(__float_as_uint(v) & 0x80000000u) : div_rn(v, s);
}

// x / s for a normal, finite scale s with r = 1/s rounded to nearest: one
// product and one residual correction (Markstein's division step).  Both
// operands carry 8-bit significands, so an inexact quotient lies at least
// 2^-33 (relative) from every fp32 rounding boundary, far outside the ~2^-46
// error of the corrected quotient: the result is the correctly rounded fp32
// quotient, exact ones included.  The residual is formed as q1*s - v and
// negated inside the second FMA, so that a zero keeps its sign: for v = -0,
// q1 = -0, q1*s - v = +0 and -(+0)*r + (-0) = -0 (for v = +0 the same steps
// give +0), with no separate sign fix-up.
__device__ __forceinline__ float row_quot_fast(float v, float s, float r) {
  const float q1 = mul_rn(v, r);
  float rem, q2;
  asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(rem) : "f"(q1), "f"(s), "f"(-v));
  asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(q2) : "f"(-rem), "f"(r), "f"(q1));
  return q2;
}

template <bool kFast>
__device__ __forceinline__ uint32_t row_e4m3x2(uint32_t w, float s, float r) {
  const float a = bf_lo(w), b = bf_hi(w);
  return kFast ? e4m3x2(row_quot_fast(a, s, r), row_quot_fast(b, s, r))
               : e4m3x2(row_quot(a, s), row_quot(b, s));
}

template <bool kFast>
__device__ __forceinline__ void row_pass2(const uint4* xr, uint2* qr, int64_t chunks, int tid,
                                          int T, float s, float r, const Span& sq) {
  for (int64_t c = tid; c < chunks; c += T) {
    const uint4 a = __ldg(xr + c);
    uint2 o;
    o.x = row_e4m3x2<kFast>(a.x, s, r) | (row_e4m3x2<kFast>(a.y, s, r) << 16);
    o.y = row_e4m3x2<kFast>(a.z, s, r) | (row_e4m3x2<kFast>(a.w, s, r) << 16);
    if (in_span(sq, qr + c, 8)) qr[c] = o;
  }
}

// Row reduction shared by both rowwise variants: the group's amax -> the
// bf16 scale bits.
__device__ __forceinline__ uint16_t row_scale(uint32_t m, uint32_t* red, int g, int t_log2) {
  m = __reduce_max_sync(0xffffffffu, m);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = m;
  __syncthreads();
  const int w0 = (g << t_log2) >> 5;
  for (int w = 0; w < (1 << (t_log2 - 5)); ++w) m = max(m, red[w0 + w]);
  __syncthreads();                            // red is reused by the next row step
  uint16_t sb;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(sb) : "f"(div_rn(__uint_as_float(m << 16), 448.0f)));
  return sb;
}

// Rows too long for the bulk-staged kernel (stage over kMaxRowStage): the
// group reads its row twice, the second time from L2.
__global__ void __launch_bounds__(kThreads) rowwise_kernel(const uint16_t* x, int64_t M,
                                                           int64_t K, int t_log2, uint8_t* q,
                                                           uint16_t* scale, Span sp_q,
                                                           Span sp_scale) {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ uint32_t red[kThreads / 32];
  const int T = 1 << t_log2;                 // threads per row, 32..256
  const int groups = kThreads >> t_log2;     // rows per CTA step
  const int g = threadIdx.x >> t_log2;
  const int tid = threadIdx.x & (T - 1);
  const int64_t chunks = K >> 3;
  for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * groups; r0 < M;
       r0 += static_cast<int64_t>(gridDim.x) * groups) {
    const int64_t r = r0 + g;
    const bool live = r < M;
    const uint4* xr = reinterpret_cast<const uint4*>(x + r * K);
    uint2* qr = reinterpret_cast<uint2*>(q + r * K);
    uint32_t m = 0;
    if (live) {
      for (int64_t c = tid; c < chunks; c += 2 * T) {
        const uint4 a = __ldg(xr + c);
        uint4 b = make_uint4(0, 0, 0, 0);
        if (c + T < chunks) b = __ldg(xr + c + T);
        m = absmax8(absmax8(m, a), b);
      }
    }
    const uint16_t sb = row_scale(mag_of(m), red, g, t_log2);
    if (!live) continue;
    const float s = __uint_as_float(static_cast<uint32_t>(sb) << 16);
    if (tid == 0 && in_span(sp_scale, scale + r, 2)) scale[r] = sb;
    // Normal finite scales take the reciprocal path; zero, subnormal, Inf
    // and NaN scales the IEEE division.
    if (s >= FLT_MIN && s <= FLT_MAX)
      row_pass2<true>(xr, qr, chunks, tid, T, s, div_rn(1.0f, s), sp_q);
    else
      row_pass2<false>(xr, qr, chunks, tid, T, s, 0.0f, sp_q);
  }
}

// Bulk-staged rowwise variant: each step's rows (R = 256 / T consecutive rows,
// contiguous in memory) arrive in shared memory by one 1D bulk async copy,
// kS steps ahead, completing on an mbarrier; the threads reduce and convert
// from shared memory and store q directly.  DRAM latency is hidden by the
// copies in flight instead of by registers.  Every wait is bounded; on time-out
// the CTA raises its abort flag, stops, and reports through g_scaled_watchdog.
__device__ int g_scaled_watchdog = 0;

__global__ void __launch_bounds__(kThreads) rowwise_bulk_kernel(const uint16_t* x, int64_t M,
                                                                int64_t K, int t_log2, int stages,
                                                                uint8_t* q, uint16_t* scale,
                                                                Span sp_q, Span sp_scale,
                                                                int64_t stall_at, uint64_t stall_ns) {
  asm volatile("griddepcontrol.launch_dependents;");
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint32_t red[kThreads / 32];
  __shared__ __align__(8) uint64_t full[8];
  __shared__ __align__(8) uint64_t stall_bar;   // diagnostic: never completed
  __shared__ int abort_flag;
  const int T = 1 << t_log2;
  const int groups = kThreads >> t_log2;
  const int g = threadIdx.x >> t_log2;
  const int tid = threadIdx.x & (T - 1);
  const int64_t chunks = K >> 3;
  const int64_t row_bytes = K * 2;
  const int64_t stage_bytes = row_bytes * groups;
  const int64_t step_rows = static_cast<int64_t>(gridDim.x) * groups;
  const int64_t n_steps = (M - static_cast<int64_t>(blockIdx.x) * groups + step_rows - 1) / step_rows;
  if (threadIdx.x == 0) {
    // While earlier grids finish, ask L2 for the rows of this CTA's first
    // steps (a hint only: nothing reaches the SM before the wait, and the
    // copies after it see the earlier grids' writes).
    for (int64_t i = 0; i < stages && i < n_steps; ++i) {
      const int64_t r0 = static_cast<int64_t>(blockIdx.x) * groups + i * step_rows;
      const int64_t rows = M - r0 < groups ? M - r0 : groups;
      bulk_prefetch_l2(x + r0 * K, static_cast<uint32_t>(rows * row_bytes));
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  auto issue = [&](int64_t i) {             // thread 0: step i into its stage
    const int st = static_cast<int>(i % stages);
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * groups + i * step_rows;
    const int64_t rows = M - r0 < groups ? M - r0 : groups;
    const uint32_t bytes = static_cast<uint32_t>(rows * row_bytes);
    mbar_arrive_expect_tx(&full[st], bytes);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(ring + st * stage_bytes)),
        "l"(reinterpret_cast<uint64_t>(x + r0 * K)), "r"(bytes), "r"(smem_u32(&full[st]))
        : "memory");
  };

  if (threadIdx.x == 0) {
    for (int st = 0; st < stages; ++st) mbar_init(&full[st], 1);
    mbar_init(&stall_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Diagnostic stall (checked builds, armed from the host): in CTA 0, thread
  // 0 waits, in place of issuing step stall_at's copy, on a barrier that
  // nothing completes; the wait runs out and raises the abort flag, and every
  // thread waiting for that step stops on it.
  const int64_t stall_i = kDiagStall && blockIdx.x == 0 ? stall_at : -1;
  int64_t issued = 0;                        // meaningful in thread 0
  if (threadIdx.x == 0)
    for (; issued < stages && issued < n_steps; ++issued) {
      if (kDiagStall && issued == stall_i) {
        mbar_wait(&stall_bar, 0u, &abort_flag, stall_ns);
        break;
      }
      issue(issued);
    }

  int64_t i = 0;
  for (; i < n_steps; ++i) {
    const int st = static_cast<int>(i % stages);
    const bool ok = mbar_wait(&full[st], static_cast<uint32_t>((i / stages) & 1), &abort_flag);
    if (!__syncthreads_and(ok)) break;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * groups + i * step_rows + g;
    const bool live = r < M;
    const uint4* xs = reinterpret_cast<const uint4*>(ring + st * stage_bytes + g * row_bytes);
    uint32_t m = 0;
    if (live)
      for (int64_t c = tid; c < chunks; c += T) m = absmax8(m, xs[c]);
    const uint16_t sb = row_scale(mag_of(m), red, g, t_log2);
    const float sv = __uint_as_float(static_cast<uint32_t>(sb) << 16);
    if (live) {
      if (tid == 0 && in_span(sp_scale, scale + r, 2)) scale[r] = sb;
      uint2* qr = reinterpret_cast<uint2*>(q + r * K);
      if (sv >= FLT_MIN && sv <= FLT_MAX) {
        const float rcp = div_rn(1.0f, sv);
        for (int64_t c = tid; c < chunks; c += T) {
          const uint4 a = xs[c];
          uint2 o;
          o.x = row_e4m3x2<true>(a.x, sv, rcp) | (row_e4m3x2<true>(a.y, sv, rcp) << 16);
          o.y = row_e4m3x2<true>(a.z, sv, rcp) | (row_e4m3x2<true>(a.w, sv, rcp) << 16);
          if (in_span(sp_q, qr + c, 8)) qr[c] = o;
        }
      } else {
        for (int64_t c = tid; c < chunks; c += T) {
          const uint4 a = xs[c];
          uint2 o;
          o.x = row_e4m3x2<false>(a.x, sv, 0.0f) | (row_e4m3x2<false>(a.y, sv, 0.0f) << 16);
          o.y = row_e4m3x2<false>(a.z, sv, 0.0f) | (row_e4m3x2<false>(a.w, sv, 0.0f) << 16);
          if (in_span(sp_q, qr + c, 8)) qr[c] = o;
        }
      }
    }
    __syncthreads();                          // every thread is done with this stage
    if (threadIdx.x == 0 && i + stages < n_steps) {
      if (kDiagStall && issued == stall_i)
        mbar_wait(&stall_bar, 0u, &abort_flag, stall_ns);
      else
        issue(issued++);
    }
  }
  if (threadIdx.x == 0 && abort_flag) {
    // Gave up waiting: let the copies still in flight land (bounded) before
    // the CTA's shared memory is released, then report.
    for (int64_t j = i; j < issued; ++j) {
      const int st = static_cast<int>(j % stages);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&full[st], static_cast<uint32_t>((j / stages) & 1)) &&
             globaltimer_ns() - t0 < 100000000ull) {
      }
    }
    atomicOr(&g_scaled_watchdog, 1);
  }
}

template <typename... Args>
int launch_pdl(void (*kernel)(Args...), int grid, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, kernel, args...));
}

template <typename K>
int wave(K kernel, int num_sms) {
  int per = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, kThreads, 0) != cudaSuccess ||
      per < 1)
    per = 1;
  return num_sms * per;
}

}  // namespace

int launch_cast_tensorwise(const uint16_t* x, int64_t n, uint8_t* q, float* scale, float* amax,
                           int num_sms, cudaStream_t stream) {
  static DeviceCache occ_amax, occ_cast;
  const int per_amax = occ_amax.get([] { return wave(tensor_amax_kernel, 1); });
  const int per_cast = occ_cast.get([] { return wave(tensorwise_kernel, 1); });
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), stream);
  if (e != cudaSuccess) return static_cast<int>(e);
  const int64_t chunks = (n >> 3) > 0 ? (n >> 3) : 1;
  const int64_t want_a = static_cast<int64_t>(num_sms) * per_amax;
  const int64_t want_c = static_cast<int64_t>(num_sms) * per_cast;
  const int ga = static_cast<int>(chunks < want_a ? chunks : want_a);
  const int gc = static_cast<int>(chunks < want_c ? chunks : want_c);
  uint32_t* bits = reinterpret_cast<uint32_t*>(amax);
  if (int rc = launch_pdl(tensor_amax_kernel, ga, stream, x, n, bits, make_span(amax, 4)))
    return rc;
  return launch_pdl(tensorwise_kernel, gc, stream, x, n, static_cast<const uint32_t*>(bits), q,
                    scale, make_span(q, static_cast<uint64_t>(n)), make_span(scale, 4));
}

int launch_cast_rowwise(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint16_t* scale,
                        int num_sms, cudaStream_t stream) {
  const Span sp_q = make_span(q, static_cast<uint64_t>(M) * static_cast<uint64_t>(K));
  const Span sp_scale = make_span(scale, 2 * static_cast<uint64_t>(M));
  // Threads per row T = 2^t_log2: the power of two nearest to K / 64 (in the
  // log domain), 32 to 256, so that each thread converts about eight 16-byte
  // chunks of its row and the per-step barriers and reduction are amortised.
  // t_log2 grows while K / 64 >= 2^(t_log2 + 1/2), i.e. K^2 >= 2^(2 t_log2 + 13).
  int t_log2 = 5;
  const uint64_t k_sq = static_cast<uint64_t>(K) * static_cast<uint64_t>(K);
  while (t_log2 < 8 && k_sq >= (uint64_t{1} << (2 * t_log2 + 13))) ++t_log2;
  const int64_t groups = kThreads >> t_log2;
  const int64_t steps = (M + groups - 1) / groups;
  const int64_t stage_bytes = groups * K * 2;
  if (stage_bytes <= kMaxRowStage) {
    // Bulk-staged: as many stages (2..8) as fit in kRowRing bytes; three
    // stages of 32 KB or more (96 KB, two CTAs per SM) where every CTA of such
    // a grid runs at least 16 steps, so that the deeper ring pays for its
    // fill.
    int stages = static_cast<int>(kRowRing / stage_bytes);
    stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
    if (stages == 2 && stage_bytes >= 32 * 1024 && 3 * stage_bytes <= 2 * kMaxRowStage &&
        steps >= int64_t{32} * num_sms)
      stages = 3;
    const int smem = static_cast<int>(stages * stage_bytes);
    static DeviceCache attr_cache;
    const int attr = attr_cache.get([] {
      return static_cast<int>(cudaFuncSetAttribute(
          rowwise_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
          static_cast<int>(kRowRing > 2 * kMaxRowStage ? kRowRing : 2 * kMaxRowStage)));
    });
    if (attr != 0) return attr;
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, rowwise_bulk_kernel, kThreads, smem) !=
            cudaSuccess ||
        per < 1)
      per = 1;
    const int64_t want = static_cast<int64_t>(num_sms) * per;
    const int grid = static_cast<int>(steps < want ? steps : want);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr_pdl[1];
    attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr_pdl;
    cfg.numAttrs = 1;
    const Stall stall = take_stall();
    return static_cast<int>(cudaLaunchKernelEx(&cfg, rowwise_bulk_kernel, x, M, K, t_log2, stages, q,
                                               scale, sp_q, sp_scale, stall.at, stall.ns));
  }
  static DeviceCache occ;
  const int per = occ.get([] { return wave(rowwise_kernel, 1); });
  const int64_t want = static_cast<int64_t>(num_sms) * per;
  const int grid = static_cast<int>(steps < want ? steps : want);
  return launch_pdl(rowwise_kernel, grid, stream, x, M, K, t_log2, q, scale, sp_q, sp_scale);
}

int out_of_bounds_scaled(bool clear) { return read_out_of_bounds(clear); }

int read_scaled_watchdog(int* out, bool clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_scaled_watchdog, sizeof(int));
  if (e != cudaSuccess) return static_cast<int>(e);
  if (clear && v) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_scaled_watchdog, &z, sizeof(int));
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  *out = v;
  return 0;
}

}  // namespace mx
