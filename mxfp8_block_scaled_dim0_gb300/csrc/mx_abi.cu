// mx_abi.cu -- the C ABI (include/mxfp8_cast.h): argument checks, TMA
// descriptor encoding and kernel launches.  No device allocation, no device
// synchronisation, no host reads of device memory on any cast path.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>
#include <mutex>

#include "mx_kernels.h"
#include "mxfp8_cast.h"

namespace {

thread_local int t_last_cuda = 0;

// Diagnostic stall armed by mx_selftest_arm_stall for this thread's next
// launch of a kernel with bounded waits (at < 0: none).
thread_local mx::Stall t_stall = {-1, 0};

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 256;   // TMA coordinates are int32

int cuda_fail(int code) {
  t_last_cuda = code;
  return MX_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// cuTensorMapEncodeTiled through the runtime's driver entry point, so that the
// library needs no link-time dependency on libcuda.
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// A tensor map depends only on these values, so maps are cached per thread
// (encoding costs microseconds of host time per call).
struct MapKey {
  const void* base;
  uint64_t inner, outer, stride;
  uint32_t bin, bout;
  int dt, l2;
  bool operator==(const MapKey& o) const {
    return base == o.base && inner == o.inner && outer == o.outer && stride == o.stride &&
           bin == o.bin && bout == o.bout && dt == o.dt && l2 == o.l2;
  }
};

struct MapCache {
  static constexpr int kEntries = 16;
  MapKey key[kEntries];
  CUtensorMap map[kEntries];
  bool used[kEntries] = {};
  int next = 0;
};

thread_local MapCache t_maps;

// 2D tiled map: inner dimension `inner` (elements), `outer` rows `stride`
// bytes apart, box `bin` x `bout`, 128-byte swizzle.
int encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
              uint64_t outer, uint64_t stride, uint32_t bin, uint32_t bout,
              CUtensorMapL2promotion l2) {
  const MapKey k = {base, inner, outer, stride, bin, bout, static_cast<int>(dt), static_cast<int>(l2)};
  for (int i = 0; i < MapCache::kEntries; ++i) {
    if (t_maps.used[i] && t_maps.key[i] == k) {
      *m = t_maps.map[i];
      return MX_OK;
    }
  }
  EncodeFn fn = encode_fn();
  if (!fn) return cuda_fail(static_cast<int>(cudaErrorNotSupported));
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {stride};
  const cuuint32_t box[2] = {bin, bout};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(static_cast<int>(cudaErrorInvalidValue));
  const int slot = t_maps.next;
  t_maps.next = (slot + 1) % MapCache::kEntries;
  t_maps.key[slot] = k;
  t_maps.map[slot] = *m;
  t_maps.used[slot] = true;
  return MX_OK;
}

// Descriptors for X (M x K bf16) and q1 (K x M bytes, as its even and odd
// rows, boxes of 128 bytes x q1_rows).  q1 may be null (not written by TMA in
// this call).
int encode_cast_maps(mx::CastMaps* maps, const void* x, int64_t M, int64_t K, const void* q1,
                     unsigned q1_rows = mx::kQ1BoxRowsFused) {
  int rc = encode_2d(&maps->x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, K * 2, 64, 128,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (rc) return rc;
  if (q1) {
    rc = encode_2d(&maps->q1e, CU_TENSOR_MAP_DATA_TYPE_UINT8, q1, M, K / 2, 2 * M, 128, q1_rows,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE);
    if (rc) return rc;
    rc = encode_2d(&maps->q1o, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<const uint8_t*>(q1) + M,
                   M, K / 2, 2 * M, 128, q1_rows, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    if (rc) return rc;
  } else {
    maps->q1e = maps->x;
    maps->q1o = maps->x;
  }
  return MX_OK;
}

int current_sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(static_cast<int>(e));
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(static_cast<int>(e));
  return MX_OK;
}

// Every non-null pointer must be memory that the current device's kernels
// may read and write: device memory of that device, or managed memory.  A
// host pointer or another device's pointer would otherwise reach a kernel
// (and its TMA descriptors) and fault there.
int check_device(std::initializer_list<const void*> ptrs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(static_cast<int>(e));
  for (const void* p : ptrs) {
    if (!p) continue;
    cudaPointerAttributes a;
    e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();   // leave no error behind for the caller's next check
      return MX_ERR_DEVICE;
    }
    if (a.type == cudaMemoryTypeManaged) continue;
    if (a.type != cudaMemoryTypeDevice || a.device != dev) return MX_ERR_DEVICE;
  }
  return MX_OK;
}

int check_2d_shape(int64_t M, int64_t K) {
  if (M < 32 || K < 32 || M > kMaxDim || K > kMaxDim) return MX_ERR_SHAPE;
  if (M % 32 != 0 || K % 32 != 0) return MX_ERR_SHAPE;
  return MX_OK;
}

int launch_rc(int rc) { return rc ? cuda_fail(rc) : MX_OK; }

}  // namespace

mx::Stall mx::take_stall() {
  const Stall s = t_stall;
  t_stall = Stall{-1, 0};
  return s;
}

namespace {

// Shared body of the 3D casts: q0 / s0_blk null for dim1 only, q1 / s1_blk
// null for dim0 only.
int cast_3d(const void* w, int64_t E, int64_t N, int64_t K, void* q0, void* s0_blk, void* q1,
            void* s1_blk, void* stream) {
  const bool dim1 = q1 != nullptr;
  if (E < 1 || N < 1 || K < 32 || K % 32 != 0) return MX_ERR_SHAPE;
  if (dim1 && (N < 32 || N % 32 != 0)) return MX_ERR_SHAPE;
  if (N > kMaxDim || E > kMaxDim / N || K > kMaxDim) return MX_ERR_SHAPE;
  if (!aligned(w, 16) || !aligned(q0, 16) || !aligned(s0_blk, 16) || !aligned(q1, 16) ||
      !aligned(s1_blk, 16))
    return MX_ERR_ALIGN;
  if (int rc = check_device({w, q0, s0_blk, q1, s1_blk})) return rc;
  const int64_t M = E * N;
  mx::CastMaps maps;
  if (int rc = encode_cast_maps(&maps, w, M, K, q1)) return rc;
  int sms = 0;
  if (int rc = current_sm_count(&sms)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (N % 128 != 0) {
    // Scales are scattered byte by byte in this case; the padding of each
    // expert's blocked matrices is cleared first.
    if (s0_blk) {
      cudaError_t e =
          cudaMemsetAsync(s0_blk, 0, static_cast<size_t>(mx_3d_dim0_scale_bytes(E, N, K)), st);
      if (e != cudaSuccess) return cuda_fail(static_cast<int>(e));
    }
    if (s1_blk) {
      cudaError_t e =
          cudaMemsetAsync(s1_blk, 0, static_cast<size_t>(mx_3d_scale_bytes(E, N, K)), st);
      if (e != cudaSuccess) return cuda_fail(static_cast<int>(e));
    }
  }
  return launch_rc(mx::launch_cast_experts(maps, E, N, K, q0, s0_blk, s1_blk, sms, st));
}

}  // namespace

extern "C" {

int64_t mx_blocked_bytes(int64_t R, int64_t C) {
  if (R < 0 || C < 0) return -1;
  return cdiv(R, 128) * 128 * cdiv(C, 4) * 4;
}

int64_t mx_grouped_m_scale_bytes(int64_t M, int64_t K, int32_t G, int32_t dim) {
  if (M < 0 || K < 0 || G < 1 || (dim != 0 && dim != 1)) return -1;
  if (dim == 0) return (M + 128 * static_cast<int64_t>(G)) * cdiv(K / 32, 4) * 4;
  return cdiv(K, 128) * 128 * (cdiv(M, 32) + 4 * static_cast<int64_t>(G));
}

int64_t mx_3d_scale_bytes(int64_t E, int64_t N, int64_t K) {
  if (E < 0 || N < 0 || K < 0) return -1;
  return E * mx_blocked_bytes(K, N / 32);
}

int64_t mx_3d_dim0_scale_bytes(int64_t E, int64_t N, int64_t K) {
  if (E < 0 || N < 0 || K < 0) return -1;
  return E * mx_blocked_bytes(N, K / 32);
}

const char* mx_strerror(int code) {
  switch (code) {
    case MX_OK: return "ok";
    case MX_ERR_NULL: return "null pointer argument";
    case MX_ERR_SHAPE: return "invalid shape (zero, too large, or not a multiple of 32)";
    case MX_ERR_ALIGN: return "misaligned pointer (16-byte alignment required)";
    case MX_ERR_CUDA: return "CUDA call failed (see mx_last_cuda_error)";
    case MX_ERR_GROUPS: return "invalid group count or group offsets";
    case MX_ERR_DEVICE: return "pointer is not device memory of the current CUDA device";
    default: return "unknown error";
  }
}

int mx_last_cuda_error(void) { return t_last_cuda; }

int mx_watchdog(int clear) {
  int v = 0, w = 0;
  int rc = mx::read_watchdog(&v, clear != 0);
  if (rc) return cuda_fail(rc);
  rc = mx::read_scaled_watchdog(&w, clear != 0);
  if (rc) return cuda_fail(rc);
  int d = 0;
  rc = mx::read_dequant_watchdog(&d, clear != 0);
  if (rc) return cuda_fail(rc);
  return v | w | d;
}

int mx_bounds_check(int clear) {
  const int parts[4] = {mx::out_of_bounds_cast(clear != 0), mx::out_of_bounds_blocked(clear != 0),
                        mx::out_of_bounds_dequant(clear != 0), mx::out_of_bounds_scaled(clear != 0)};
  int sum = 0;
  for (int v : parts) {
    if (v == -1) return -1;                     // release build: no checks compiled in
    if (v < 0) return cuda_fail(static_cast<int>(cudaErrorUnknown));
    sum += v;
  }
  return sum;
}

int mx_selftest_bounds(void* buf16, void* stream) {
  if (!buf16) return MX_ERR_NULL;
  if (!aligned(buf16, 16)) return MX_ERR_ALIGN;
#ifndef MX_DEBUG_BOUNDS
  (void)stream;
  return -1;   // release build: no checks compiled in, nothing to launch
#else
  if (int rc = check_device({buf16})) return rc;
  return launch_rc(mx::launch_bounds_selftest(buf16, static_cast<cudaStream_t>(stream)));
#endif
}

int mx_selftest_watchdog(int64_t wait_ns, void* stream) {
  if (wait_ns < 1000 || wait_ns > int64_t{10} * 1000 * 1000 * 1000) return MX_ERR_SHAPE;
  return launch_rc(mx::launch_watchdog_selftest(static_cast<uint64_t>(wait_ns),
                                                static_cast<cudaStream_t>(stream)));
}

int mx_selftest_arm_stall(int64_t at, int64_t wait_ns) {
  if (at < 0 || wait_ns < 1000 || wait_ns > int64_t{10} * 1000 * 1000 * 1000) return MX_ERR_SHAPE;
#ifndef MX_DEBUG_BOUNDS
  return -1;   // release build: the kernels carry no stall hook, nothing is armed
#else
  t_stall = mx::Stall{at, static_cast<uint64_t>(wait_ns)};
  return MX_OK;
#endif
}

int mx_cast_dim0_dim1(const void* x, int64_t M, int64_t K, void* q0, void* s0_blk, void* q1,
                      void* s1_blk, void* stream) {
  if (!x || !q0 || !s0_blk || !q1 || !s1_blk) return MX_ERR_NULL;
  if (int rc = check_2d_shape(M, K)) return rc;
  if (!aligned(x, 16) || !aligned(q0, 16) || !aligned(s0_blk, 16) || !aligned(q1, 16) ||
      !aligned(s1_blk, 16))
    return MX_ERR_ALIGN;
  if (int rc = check_device({x, q0, s0_blk, q1, s1_blk})) return rc;
  mx::CastMaps maps;
  if (int rc = encode_cast_maps(&maps, x, M, K, q1)) return rc;
  int sms = 0;
  if (int rc = current_sm_count(&sms)) return rc;
  return launch_rc(mx::launch_cast_2d(maps, M, K, q0, s0_blk, s1_blk, sms,
                                      static_cast<cudaStream_t>(stream)));
}

int mx_cast_dim0_dim1_noalloc(const void* x, int64_t M, int64_t K, void* q0, void* s0_blk,
                              void* q1, void* s1_blk, void* stream) {
  if (!x || !q0 || !s0_blk || !q1 || !s1_blk) return MX_ERR_NULL;
  if (int rc = check_2d_shape(M, K)) return rc;
  if (!aligned(x, 16) || !aligned(q0, 16) || !aligned(s0_blk, 16) || !aligned(q1, 16) ||
      !aligned(s1_blk, 16))
    return MX_ERR_ALIGN;
  if (int rc = check_device({x, q0, s0_blk, q1, s1_blk})) return rc;
  mx::CastMaps maps;
  if (int rc = encode_cast_maps(&maps, x, M, K, q1)) return rc;
  int sms = 0;
  if (int rc = current_sm_count(&sms)) return rc;
  int64_t words = 0;
  const int rc = mx::launch_cast_2d_noalloc(maps, M, K, q0, s0_blk, q1, s1_blk, sms,
                                            static_cast<cudaStream_t>(stream), &words);
  if (words > mx::noalloc_scratch_words()) return MX_ERR_SHAPE;   // more scratch than reserved
  return launch_rc(rc);
}

int mx_cast_dim1(const void* x, int64_t M, int64_t K, void* q1, void* s1_blk, void* stream) {
  if (!x || !q1 || !s1_blk) return MX_ERR_NULL;
  if (int rc = check_2d_shape(M, K)) return rc;
  if (!aligned(x, 16) || !aligned(q1, 16) || !aligned(s1_blk, 16)) return MX_ERR_ALIGN;
  if (int rc = check_device({x, q1, s1_blk})) return rc;
  mx::CastMaps maps;
  if (int rc = encode_cast_maps(&maps, x, M, K, q1)) return rc;
  int sms = 0;
  if (int rc = current_sm_count(&sms)) return rc;
  return launch_rc(mx::launch_cast_2d(maps, M, K, nullptr, nullptr, s1_blk, sms,
                                      static_cast<cudaStream_t>(stream)));
}

int mx_cast_dim0(const void* x, int64_t M, int64_t K, void* q0, void* s0_blk, void* stream) {
  if (!x || !q0 || !s0_blk) return MX_ERR_NULL;
  if (M < 1 || K < 32 || M > kMaxDim || K > kMaxDim || K % 32 != 0) return MX_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(q0, 16) || !aligned(s0_blk, 16)) return MX_ERR_ALIGN;
  if (int rc = check_device({x, q0, s0_blk})) return rc;
  mx::CastMaps maps;
  if (int rc = encode_cast_maps(&maps, x, M, K, nullptr)) return rc;
  int sms = 0;
  if (int rc = current_sm_count(&sms)) return rc;
  return launch_rc(mx::launch_cast_2d(maps, M, K, q0, s0_blk, nullptr, sms,
                                      static_cast<cudaStream_t>(stream)));
}

int mx_dequant_blocked(const void* q, int64_t R, int64_t C, const void* s_blk, void* out,
                       void* stream) {
  if (!q || !s_blk || !out) return MX_ERR_NULL;
  if (R < 1 || C < 32 || R > kMaxDim || C > kMaxDim || C % 32 != 0) return MX_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(s_blk, 16) || !aligned(out, 16)) return MX_ERR_ALIGN;
  if (int rc = check_device({q, s_blk, out})) return rc;
  int sms = 0;
  if (int rc = current_sm_count(&sms)) return rc;
  mx::DqMaps maps;
  if (C >= mx::kDqTmaMinCols) {
    if (int rc = encode_2d(&maps.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, C, R, C, 128, 128,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
      return rc;
    if (int rc = encode_2d(&maps.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, C, R, 2 * C, 64, 128,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE))
      return rc;
  }
  return launch_rc(mx::launch_dequant_blocked(&maps, static_cast<const uint8_t*>(q), R, C,
                                              static_cast<const uint8_t*>(s_blk),
                                              static_cast<uint16_t*>(out), sms,
                                              static_cast<cudaStream_t>(stream)));
}

int mx_cast_tensorwise(const void* x, int64_t n, void* q, float* scale, float* amax,
                       void* stream) {
  if (!x || !q || !scale || !amax) return MX_ERR_NULL;
  if (n < 1 || n > (int64_t{1} << 40)) return MX_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4) || !aligned(amax, 4))
    return MX_ERR_ALIGN;
  if (int rc = check_device({x, q, scale, amax})) return rc;
  int sms = 0;
  if (int rc = current_sm_count(&sms)) return rc;
  return launch_rc(mx::launch_cast_tensorwise(static_cast<const uint16_t*>(x), n,
                                              static_cast<uint8_t*>(q), scale, amax, sms,
                                              static_cast<cudaStream_t>(stream)));
}

int mx_cast_rowwise(const void* x, int64_t M, int64_t K, void* q, void* scale, void* stream) {
  if (!x || !q || !scale) return MX_ERR_NULL;
  if (M < 1 || K < 8 || K % 8 != 0 || M > kMaxDim || K > kMaxDim) return MX_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 2)) return MX_ERR_ALIGN;
  if (int rc = check_device({x, q, scale})) return rc;
  int sms = 0;
  if (int rc = current_sm_count(&sms)) return rc;
  return launch_rc(mx::launch_cast_rowwise(static_cast<const uint16_t*>(x), M, K,
                                           static_cast<uint8_t*>(q), static_cast<uint16_t*>(scale),
                                           sms, static_cast<cudaStream_t>(stream)));
}

int mx_scales_to_blocked(const void* s, int64_t R, int64_t C, void* out, void* stream) {
  if (!s || !out) return MX_ERR_NULL;
  if (R < 1 || C < 1 || R > int64_t{65535} * 128 || C > kMaxDim) return MX_ERR_SHAPE;
  if (!aligned(out, 16)) return MX_ERR_ALIGN;
  if (int rc = check_device({s, out})) return rc;
  return launch_rc(mx::launch_scales_to_blocked(static_cast<const uint8_t*>(s), R, C,
                                                static_cast<uint8_t*>(out),
                                                static_cast<cudaStream_t>(stream)));
}

int mx_cast_grouped_m(const void* x, int64_t M, int64_t K, const int32_t* offs, int32_t G,
                      void* q0, void* s0_blk, int64_t* s0_row_offs, void* q1, void* s1_blk,
                      int64_t* s1_col_offs, int32_t* status, void* stream) {
  if (!x || !offs || !q0 || !s0_blk || !s0_row_offs || !q1 || !s1_blk || !s1_col_offs || !status)
    return MX_ERR_NULL;
  if (G < 1) return MX_ERR_GROUPS;
  if (M < 1 || K < 32 || M > kMaxDim || K > kMaxDim || K % 32 != 0) return MX_ERR_SHAPE;
  if (M + 128 * static_cast<int64_t>(G) > kMaxDim) return MX_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(q0, 16) || !aligned(s0_blk, 16) || !aligned(q1, 16) ||
      !aligned(s1_blk, 16) || !aligned(offs, 4) || !aligned(s0_row_offs, 8) ||
      !aligned(s1_col_offs, 8) || !aligned(status, 4))
    return MX_ERR_ALIGN;
  if (int rc = check_device({x, offs, q0, s0_blk, s0_row_offs, q1, s1_blk, s1_col_offs, status}))
    return rc;
  mx::CastMaps maps;
  // q1 rows are 16-byte aligned only when M % 16 == 0; then whole tiles may
  // leave by TMA (see the grouped kernel), otherwise all of q1 is written with
  // plain stores.
  if (int rc = encode_cast_maps(&maps, x, M, K, M % 16 == 0 ? q1 : nullptr, mx::kQ1BoxRowsGrouped))
    return rc;
  int sms = 0;
  if (int rc = current_sm_count(&sms)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return launch_rc(mx::launch_cast_grouped(maps, M, K, offs, G, q0, q1, s0_blk, s0_row_offs,
                                           s1_col_offs, s1_blk, status, sms, st));
}

int mx_cast_3d_dim1(const void* w, int64_t E, int64_t N, int64_t K, void* q1, void* s1_blk,
                    void* stream) {
  if (!w || !q1 || !s1_blk) return MX_ERR_NULL;
  return cast_3d(w, E, N, K, nullptr, nullptr, q1, s1_blk, stream);
}

int mx_cast_3d_dim0(const void* w, int64_t E, int64_t N, int64_t K, void* q0, void* s0_blk,
                    void* stream) {
  if (!w || !q0 || !s0_blk) return MX_ERR_NULL;
  return cast_3d(w, E, N, K, q0, s0_blk, nullptr, nullptr, stream);
}

int mx_cast_3d_dim0_dim1(const void* w, int64_t E, int64_t N, int64_t K, void* q0, void* s0_blk,
                         void* q1, void* s1_blk, void* stream) {
  if (!w || !q0 || !s0_blk || !q1 || !s1_blk) return MX_ERR_NULL;
  return cast_3d(w, E, N, K, q0, s0_blk, q1, s1_blk, stream);
}

}  // extern "C"
