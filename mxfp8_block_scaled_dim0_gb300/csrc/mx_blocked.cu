// mx_blocked.cu -- small kernels around the casts:
//   * scale matrix -> 128x4 blocked layout (standalone), the conversion of
//     e8m0 scales to the layout grouped / block-scaled GEMMs read, as in
//     pytorch/ao PR #3416 "[mxfp8 moe training] parallelize along col blocks
//     in scale blocked format kernel for groups along K" (Changes list;
//     128x4 is the minimum granularity of the swizzle);
//   * per-group padded scale offsets computed on the device, the sync-free
//     replacement for reading the padded row count on the host described in
//     pytorch/ao PR #2990 "[mxfp8 moe training] add compile support".
#include <cuda_runtime.h>

#include "mx_common.cuh"
#include "mx_kernels.h"

namespace mx {
namespace {

constexpr int kErrGroups = -5;   // MX_ERR_GROUPS

// One CTA computes, for groups given by cumulative ends offs[0..G-1]:
//   row_offs[g] = sum_{h<g} ceil(m_h / 128) * 128
//   col_offs[g] = sum_{h<g} ceil(m_h / 128) * 4
// and status = 0, or MX_ERR_GROUPS if an offset is negative, decreases,
// exceeds M, or the last one is not M.
__global__ void __launch_bounds__(256) group_offsets_kernel(const int32_t* __restrict__ offs,
                                                            int G, int64_t M,
                                                            int64_t* __restrict__ row_offs,
                                                            int64_t* __restrict__ col_offs,
                                                            int32_t* __restrict__ status,
                                                            Span sp_ro, Span sp_co, Span sp_st) {
  __shared__ int64_t warp_sum[32];
  __shared__ int64_t carry_sh;
  __shared__ int bad_sh;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  // The cast kernel that follows is launched as a programmatic dependent of
  // this one; let it start its set-up now (it waits for this grid's results).
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    carry_sh = 0;
    bad_sh = 0;
    if (in_span(sp_ro, row_offs, 8)) row_offs[0] = 0;
    if (in_span(sp_co, col_offs, 8)) col_offs[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < G; base += blockDim.x) {
    const int64_t carry = carry_sh;
    const int g = base + threadIdx.x;
    int64_t tiles = 0;
    if (g < G) {
      const int64_t hi = offs[g];
      const int64_t lo = g ? static_cast<int64_t>(offs[g - 1]) : 0;
      bool bad = hi < lo || hi < 0 || hi > M || (g == G - 1 && hi != M);
      if (bad) atomicOr(&bad_sh, 1);
      else tiles = (hi - lo + 127) >> 7;
    }
    int64_t v = tiles;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t n = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += n;
    }
    if (lane == 31) warp_sum[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int64_t w = lane < nwarps ? warp_sum[lane] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int64_t n = __shfl_up_sync(0xffffffffu, w, d);
        if (lane >= d) w += n;
      }
      warp_sum[lane] = w;
    }
    __syncthreads();
    const int64_t incl = carry + v + (warp ? warp_sum[warp - 1] : 0);
    if (g < G) {
      if (in_span(sp_ro, row_offs + g + 1, 8)) row_offs[g + 1] = incl * 128;
      if (in_span(sp_co, col_offs + g + 1, 8)) col_offs[g + 1] = incl * 4;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry_sh = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0 && in_span(sp_st, status, 4)) *status = bad_sh ? kErrGroups : 0;
}

// Scale matrix s (R x C bytes, row-major) -> blocked layout.  One CTA takes
// one 128-row band and up to 32 column tiles (128 scale columns, 16 KB):
//   - load: 16-byte global loads when C % 16 == 0 and s is 16-byte aligned
//     (eight lanes per 128-byte row), else byte loads; each lane stores its 16
//     bytes as four words into shared memory rows of 33 words, so that both
//     the stores (row r + 4k + m distinct over a warp) and the transposed
//     reads below hit 32 distinct banks;
//   - store: the 32 tiles are 16 KB contiguous in the output; lane i of a
//     warp builds storage row i of one tile (rows i, i+32, i+64, i+96, four
//     columns each) and writes it with one 16-byte store.
// Out-of-range rows / columns are written as zero padding.
constexpr int kBlkCols = 128;                       // scale columns per CTA
constexpr int kBlkPitch = kBlkCols / 4 + 1;         // words per shared row

__global__ void __launch_bounds__(256) to_blocked_kernel(const uint8_t* __restrict__ s, int64_t R,
                                                        int64_t C, uint8_t* __restrict__ out,
                                                        int64_t n_ct, int vec16, Span sp_out) {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ uint32_t tile[128 * kBlkPitch];
  const int64_t rb = blockIdx.y;
  const int64_t ct0 = static_cast<int64_t>(blockIdx.x) * (kBlkCols / 4);   // first column tile
  const int64_t c0 = ct0 * 4;
  // 128 rows x 8 chunks of 16 bytes
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
    const int r = i >> 3, k = i & 7;
    const int64_t row = rb * 128 + r;
    const int64_t col = c0 + 16 * k;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < R && col < C) {
      const uint8_t* src = s + row * C + col;
      if (vec16) {
        v = *reinterpret_cast<const uint4*>(src);
      } else {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int b = 0; b < 16; ++b)
          if (col + b < C) w[b >> 2] |= static_cast<uint32_t>(src[b]) << (8 * (b & 3));
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    uint32_t* dst = tile + r * kBlkPitch + 4 * k;
    dst[0] = v.x;
    dst[1] = v.y;
    dst[2] = v.z;
    dst[3] = v.w;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < (kBlkCols / 4) * 32; k += blockDim.x) {
    const int j = k >> 5, i = k & 31;
    const int64_t ct = ct0 + j;
    if (ct >= n_ct) break;
    uint4 o;
    o.x = tile[i * kBlkPitch + j];
    o.y = tile[(32 + i) * kBlkPitch + j];
    o.z = tile[(64 + i) * kBlkPitch + j];
    o.w = tile[(96 + i) * kBlkPitch + j];
    uint8_t* d = out + (rb * n_ct + ct) * 512 + i * 16;
    if (in_span(sp_out, d, 16)) *reinterpret_cast<uint4*>(d) = o;
  }
}

}  // namespace

int launch_group_offsets(const int32_t* offs, int G, int64_t M, int64_t* row_offs,
                         int64_t* col_offs, int32_t* status, cudaStream_t stream) {
  // 256 threads: small enough (in registers) to share an SM with a CTA of
  // the cast kernel that follows it as a programmatic dependent.
  const uint64_t n = 8 * static_cast<uint64_t>(G + 1);
  group_offsets_kernel<<<1, 256, 0, stream>>>(offs, G, M, row_offs, col_offs, status,
                                              make_span(row_offs, n), make_span(col_offs, n),
                                              make_span(status, 4));
  return static_cast<int>(cudaGetLastError());
}

int launch_scales_to_blocked(const uint8_t* s, int64_t R, int64_t C, uint8_t* out,
                             cudaStream_t stream) {
  const int64_t n_ct = (C + 3) / 4;
  const int64_t n_rb = (R + 127) / 128;
  if (n_rb > 65535) return static_cast<int>(cudaErrorInvalidConfiguration);
  dim3 grid(static_cast<unsigned>((n_ct + kBlkCols / 4 - 1) / (kBlkCols / 4)),
            static_cast<unsigned>(n_rb));
  const int vec16 = (C % 16 == 0) && ((reinterpret_cast<uintptr_t>(s) & 15) == 0);
  // Programmatic dependent of the previous work in the stream (waits for it
  // before any memory access), so its launch overlaps the previous tail.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const Span sp_out =
      make_span(out, static_cast<uint64_t>(n_rb) * 128 * static_cast<uint64_t>(n_ct) * 4);
  return static_cast<int>(
      cudaLaunchKernelEx(&cfg, to_blocked_kernel, s, R, C, out, n_ct, vec16, sp_out));
}

int out_of_bounds_blocked(bool clear) { return read_out_of_bounds(clear); }

#ifdef MX_DEBUG_BOUNDS
namespace {
// One thread tries a 4-byte store just past an 8-byte span over the caller's
// 16-byte buffer: the check must refuse and count it.
__global__ void bounds_selftest_kernel(uint8_t* buf) {
  const Span sp = {buf, 8};
  if (in_span(sp, buf + 8, 4)) *reinterpret_cast<uint32_t*>(buf + 8) = 0xDEADBEEFu;
}
}  // namespace
#endif

int launch_bounds_selftest(void* buf, cudaStream_t stream) {
#ifdef MX_DEBUG_BOUNDS
  bounds_selftest_kernel<<<1, 1, 0, stream>>>(static_cast<uint8_t*>(buf));
  return static_cast<int>(cudaGetLastError());
#else
  (void)buf;
  (void)stream;
  return -1;
#endif
}

}  // namespace mx
