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

#include "mx_kernels.h"

namespace mx {
namespace {

constexpr int kErrGroups = -5;   // MX_ERR_GROUPS

// One CTA computes, for groups given by cumulative ends offs[0..G-1]:
//   row_offs[g] = sum_{h<g} ceil(m_h / 128) * 128
//   col_offs[g] = sum_{h<g} ceil(m_h / 128) * 4
// and status = 0, or MX_ERR_GROUPS if an offset is negative, decreases,
// exceeds M, or the last one is not M.
__global__ void __launch_bounds__(1024) group_offsets_kernel(const int32_t* __restrict__ offs,
                                                            int G, int64_t M,
                                                            int64_t* __restrict__ row_offs,
                                                            int64_t* __restrict__ col_offs,
                                                            int32_t* __restrict__ status) {
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
    row_offs[0] = 0;
    col_offs[0] = 0;
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
      row_offs[g + 1] = incl * 128;
      col_offs[g + 1] = incl * 4;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry_sh = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) *status = bad_sh ? kErrGroups : 0;
}

// Scale matrix s (R x C bytes, row-major) -> blocked layout.  One CTA takes
// one 128-row band and up to 16 column tiles (64 scale columns): it reads the
// 128 x 64 bytes with coalesced row loads into shared memory, then writes the
// 16 tiles (8 KB contiguous in the output) as 16-byte chunks.  Storage row i
// of a tile is rows i, i+32, i+64, i+96, four columns each.  Out-of-range
// rows / columns are written as zero padding.
__global__ void __launch_bounds__(256) to_blocked_kernel(const uint8_t* __restrict__ s, int64_t R,
                                                        int64_t C, uint8_t* __restrict__ out,
                                                        int64_t n_ct, int vec4) {
  __shared__ uint32_t tile[128][17];
  const int64_t rb = blockIdx.y;
  const int64_t ct0 = static_cast<int64_t>(blockIdx.x) * 16;  // first column tile
  const int64_t c0 = ct0 * 4;
  for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
    const int r = i >> 4, wi = i & 15;
    const int64_t row = rb * 128 + r;
    const int64_t col = c0 + wi * 4;
    uint32_t v = 0u;
    if (row < R && col < C) {
      const uint8_t* src = s + row * C + col;
      if (vec4) {
        v = *reinterpret_cast<const uint32_t*>(src);
      } else {
#pragma unroll
        for (int b = 0; b < 4; ++b)
          if (col + b < C) v |= static_cast<uint32_t>(src[b]) << (8 * b);
      }
    }
    tile[r][wi] = v;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < 16 * 32; k += blockDim.x) {
    const int j = k >> 5, i = k & 31;
    const int64_t ct = ct0 + j;
    if (ct >= n_ct) break;
    uint4 o;
    o.x = tile[i][j];
    o.y = tile[32 + i][j];
    o.z = tile[64 + i][j];
    o.w = tile[96 + i][j];
    *reinterpret_cast<uint4*>(out + (rb * n_ct + ct) * 512 + i * 16) = o;
  }
}

}  // namespace

int launch_group_offsets(const int32_t* offs, int G, int64_t M, int64_t* row_offs,
                         int64_t* col_offs, int32_t* status, cudaStream_t stream) {
  group_offsets_kernel<<<1, 1024, 0, stream>>>(offs, G, M, row_offs, col_offs, status);
  return static_cast<int>(cudaGetLastError());
}

int launch_scales_to_blocked(const uint8_t* s, int64_t R, int64_t C, uint8_t* out,
                             cudaStream_t stream) {
  const int64_t n_ct = (C + 3) / 4;
  const int64_t n_rb = (R + 127) / 128;
  if (n_rb > 65535) return static_cast<int>(cudaErrorInvalidConfiguration);
  dim3 grid(static_cast<unsigned>((n_ct + 15) / 16), static_cast<unsigned>(n_rb));
  const int vec4 = (C % 4 == 0) && ((reinterpret_cast<uintptr_t>(s) & 3) == 0);
  to_blocked_kernel<<<grid, 256, 0, stream>>>(s, R, C, out, n_ct, vec4);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace mx
