// Shared definitions for the attention kernels (device side).
#pragma once
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fa {

// Bits of the device status word (read and cleared by fa_device_status).
constexpr unsigned kDevTimeout = 1u;      // a bounded wait inside a kernel ran out
constexpr unsigned kDevLayout = 2u;       // a kernel refused to run: shared-memory window misaligned

// Tile geometry shared by every kernel: 128 query rows x 128 keys, the
// tcgen05 M=128 shape, and 128-byte swizzled shared-memory rows.
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBoxBytes = 128 * 128;   // one TMA box: 128 rows x 128 bytes

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// After a timed-out wait: keep the CTA alive for a grace period so that TMA
// copies and tensor-core operations already in flight land before shared
// memory and TMEM are released.
__device__ __forceinline__ void abort_grace_period() {
  uint64_t until = global_timer_ns() + 2000000ull;   // 2 ms
  while (global_timer_ns() < until) __nanosleep(10000);
}

// SM clock of a launch, measured by the kernel itself: one thread per CTA
// notes the SM cycle counter and the global nanosecond timer when the CTA
// starts (clock_mark, into two words of shared memory, so that no register
// is held across the kernel) and adds both differences into acc[0] (cycles)
// and acc[1] (ns) when it exits, so acc[0] / acc[1] is the mean SM clock over
// the CTAs' lifetimes.
__device__ __forceinline__ void clock_mark(unsigned long long* start) {
  start[0] = static_cast<unsigned long long>(clock64());
  start[1] = global_timer_ns();
}
__device__ __forceinline__ void clock_record(unsigned long long* acc, const unsigned long long* start) {
  if (acc == nullptr) return;
  atomicAdd(acc, static_cast<unsigned long long>(clock64()) - start[0]);
  atomicAdd(acc + 1, global_timer_ns() - start[1]);
}

// Byte address, inside a 128-byte-swizzled box, of 16-byte unit `u` (0..7)
// of row `r`: the unit index is XORed with the row's position in its 8-row
// (1024-byte) group. This is the layout TMA writes with 128-byte swizzle and
// the layout the UMMA descriptors below describe.
__device__ __forceinline__ uint32_t swz128(uint32_t box_base, int r, int u) {
  return box_base + r * 128 + ((u ^ (r & 7)) << 4);
}

// Host side: a kernel's dynamic shared-memory limit is an attribute of each
// device's copy of the kernel, so it is set once per device (and per launcher,
// each holding its own PerDeviceOnce), safely from several host threads.
struct PerDeviceOnce {
  static constexpr int kMaxDevices = 64;
  std::once_flag flag[kMaxDevices];
  cudaError_t result[kMaxDevices] = {};
  template <typename Fn>
  cudaError_t run(Fn fn) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(flag[dev], [&] { result[dev] = fn(); });
    return result[dev];
  }
};

}  // namespace fa
