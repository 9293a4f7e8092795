// mx_kernels.h -- internal launchers behind the C ABI (not part of the public
// interface; the public declarations are in include/mxfp8_cast.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace mx {

// Host-side value computed once per device and kept for the process: kernel
// attributes (cudaFuncSetAttribute acts on the current device) and occupancy.
// Two threads that race on the first call both compute the same value.
class DeviceCache {
 public:
  static constexpr int kMaxDevices = 64;
  static constexpr int kUnset = -2147483647 - 1;
  DeviceCache() {
    for (auto& x : v_) x.store(kUnset, std::memory_order_relaxed);
  }
  template <typename F>
  int get(F f) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return f();
    int x = v_[d].load(std::memory_order_acquire);
    if (x == kUnset) {
      x = f();
      v_[d].store(x, std::memory_order_release);
    }
    return x;
  }

 private:
  std::atomic<int> v_[kMaxDevices];
};

// TMA descriptors of one cast call: x (bf16, two 64-column halves per tile,
// 128B swizzle) and the even / odd rows of q1 (boxes of 128 bytes x 64 rows,
// or x 16 rows for the grouped kernel's per-warp stores).
struct CastMaps {
  CUtensorMap x;
  CUtensorMap q1e;
  CUtensorMap q1o;
};

// Diagnostic stall, armed from the host (mx_selftest_arm_stall) for the next
// cast, tiled dequantisation or bulk-staged rowwise launch of the arming
// thread: in CTA 0, the thread that issues the loads waits, at its `at`-th
// tile (or step), on a barrier that nothing completes, for at most `ns`
// nanoseconds, so that the wait runs out and the CTA winds down through its
// abort path.  at < 0: none (normal use).
struct Stall {
  int64_t at;
  uint64_t ns;
};
// The armed stall, disarmed by the call (mx_abi.cu).
Stall take_stall();

constexpr unsigned kQ1BoxRowsFused = 64;
constexpr unsigned kQ1BoxRowsGrouped = 16;

int smem_bytes_cast();
int threads_cast();

// All launchers return 0 or a cudaError_t value.
// q0 == nullptr: dim1 only; s1 == nullptr: dim0 only.
int launch_cast_2d(const CastMaps& maps, int64_t M, int64_t K, void* q0, void* s0, void* s1,
                   int num_sms, cudaStream_t stream);
// The fused cast with its tile-claim counter in a fixed device array instead
// of a per-stream counter (mx_cast_dim0_dim1_noalloc); *scratch_words is set
// to the words of that array the call needs (0 or 1).
int launch_cast_2d_noalloc(const CastMaps& maps, int64_t M, int64_t K, void* q0, void* s0,
                           void* q1, void* s1, int num_sms, cudaStream_t stream,
                           int64_t* scratch_words);
int noalloc_scratch_words();
// 3D weights (E, N, K) as the (E*N, K) matrix, scales blocked per expert;
// same null conventions.  With N % 128 != 0 the scales are scattered byte by
// byte and the caller clears the scale buffers first.
int launch_cast_experts(const CastMaps& maps, int64_t E, int64_t N, int64_t K, void* q0,
                        void* s0, void* s1, int num_sms, cudaStream_t stream);
// Tensorwise / rowwise fp8 (mx_scaled.cu).  Tensorwise clears *amax, reduces
// into it, then casts (amax kernel, then the cast as its programmatic
// dependent).
int launch_cast_tensorwise(const uint16_t* x, int64_t n, uint8_t* q, float* scale, float* amax,
                           int num_sms, cudaStream_t stream);
int launch_cast_rowwise(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint16_t* scale,
                        int num_sms, cudaStream_t stream);
// MX dequantisation (mx_dequant.cu).  Rows of at least kDqTmaMinCols values
// take the tiled kernel, which needs the two TMA descriptors (q: e4m3 bytes,
// boxes of 128 x 128, 128B swizzle; out: bf16, boxes of 64 x 128, 128B
// swizzle); shorter rows take the thread-store kernel, which needs none.
struct DqMaps {
  CUtensorMap q;
  CUtensorMap out;
};
constexpr int64_t kDqTmaMinCols = 1024;
int launch_dequant_blocked(const DqMaps* maps, const uint8_t* q, int64_t R, int64_t C,
                           const uint8_t* s_blk, uint16_t* out, int num_sms, cudaStream_t stream);
int read_dequant_watchdog(int* out, bool clear);
// G <= kMaxSmemGroups: one kernel builds the group table itself; larger G:
// group_offsets_kernel first, then the cast kernel as its programmatic
// dependent.
constexpr int kMaxSmemGroups = 1024;
int launch_cast_grouped(const CastMaps& maps, int64_t M, int64_t K, const int32_t* offs, int G,
                        void* q0, void* q1, void* s0, int64_t* row_offs, int64_t* col_offs,
                        void* s1, int32_t* status, int num_sms, cudaStream_t stream);
int launch_group_offsets(const int32_t* offs, int G, int64_t M, int64_t* row_offs,
                         int64_t* col_offs, int32_t* status, cudaStream_t stream);
int launch_scales_to_blocked(const uint8_t* s, int64_t R, int64_t C, uint8_t* out,
                             cudaStream_t stream);
int read_watchdog(int* out, bool clear);
// Stores refused by the bounds-checked build, per translation unit (cleared
// on request); -1 in a release build.
int out_of_bounds_cast(bool clear);
int out_of_bounds_blocked(bool clear);
int out_of_bounds_dequant(bool clear);
int out_of_bounds_scaled(bool clear);
// -1 in a release build (nothing launched), else 0 or a cudaError_t value.
int launch_bounds_selftest(void* buf, cudaStream_t stream);
int read_scaled_watchdog(int* out, bool clear);   // the rowwise kernel's word (mx_scaled.cu)
int launch_watchdog_selftest(uint64_t limit_ns, cudaStream_t stream);

}  // namespace mx
