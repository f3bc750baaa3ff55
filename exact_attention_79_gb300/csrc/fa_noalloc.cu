// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory when they call it.
//
// fa_bwd needs a scratch workspace that the caller allocates. Some callers
// cannot do that at call time: a plugin running inside another framework's
// executor that only receives fixed input and output buffers, a component
// whose host owns the whole device memory pool, or a latency-critical loop
// that must not pay for cudaMalloc's implicit device synchronisation. For
// them this file keeps the scratch in a fixed-size array of device memory
// that belongs to the library itself. Every GPU that loads the library holds
// that array until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"

namespace {

// Largest backward workspace this entry point can serve: 32 MiB (for d = 128
// that is about 64K query rows summed over batch and heads, e.g. 31 heads of
// N = 2048 or 3 heads of N = 8192).
constexpr size_t kScratchBytes = 32u << 20;

__device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  std::mutex mu;
  void* ptr = nullptr;     // set once a lookup on this device has succeeded
};
ScratchSlot g_slots[kMaxDevices];

// Device address of the array on the current device. In host code the
// array's name only stands in for it; the real address comes from
// cudaGetSymbolAddress, looked up with that device current. Only a
// successful lookup is kept: a failed one (for example during stream
// capture, where the lookup may not run) is retried on the next call.
fa_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  ScratchSlot& s = g_slots[dev];
  std::lock_guard<std::mutex> lock(s.mu);
  if (s.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    s.ptr = p;
  }
  *out = s.ptr;
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                                    int d, int causal, float scale, void* stream) {
  const size_t need = fa_bwd_workspace_bytes(B, Hq, Hkv, N, d);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > kScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const fa_status st = scratch_for_current_device(&scratch);
  if (st != FA_OK) return st;
  // The backward's first phase rewrites every part of the workspace it later
  // reads (D, the base-2 LSE copy) and zeroes the dQ accumulator, so what an
  // earlier call left in the array does not leak into this one.
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, kScratchBytes, B, Hq, Hkv, N, d, causal, scale, stream);
}
