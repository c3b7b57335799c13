// noalloc.cu -- fgemm_unfused_bias_relu_noalloc: the unfused bias + ReLU chain for callers that
// cannot allocate device memory.
//
// The chain needs an M x N intermediate.  Here it lives in a fixed array that the library
// reserves in device memory (g_noalloc_scratch, FGEMM_NOALLOC_SCRATCH_BYTES bytes, 256-byte
// aligned) instead of a buffer the caller passes in.  Every device that loads the library keeps
// that array until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it names a shadow
// variable, not device memory), so on the first call on each device, with that device current,
// the address is looked up with cudaGetSymbolAddress and cached; later calls on that device
// reuse it.  That first call may load the library's device code; make it before any stream
// capture.  A failed lookup is not cached: the next call on that device tries again.
//
// All calls share the one array and it keeps whatever the previous call left in it.  Nothing in
// it has to start at zero: the GEMM step writes every intermediate element before the bias and
// ReLU passes read it.  Calls whose work overlaps on the GPU (on different streams, or from
// different host threads without ordering) race on the array.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fgemm.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FGEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchSlot {
  std::mutex mu;
  void* ptr = nullptr;  // set once the lookup has succeeded; never changes afterwards
};
ScratchSlot g_scratch[kMaxDevices];

// Device address of the array on the current device.  Only a successful lookup is kept: if it
// fails (for example when a first call is made while a stream is being captured, where loading
// the library's device code is not allowed), the call reports FGEMM_ERR_NO_DEVICE and the next
// call on that device tries again.
int scratch_on_current_device(void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FGEMM_ERR_NO_DEVICE;
  }
  ScratchSlot& s = g_scratch[dev];
  std::lock_guard<std::mutex> lock(s.mu);
  if (s.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FGEMM_ERR_NO_DEVICE;
    }
    s.ptr = p;
  }
  *ptr = s.ptr;
  return FGEMM_OK;
}

}  // namespace

extern "C" int fgemm_unfused_bias_relu_noalloc(const void* A, const void* B, const void* bias,
                                               void* out, int64_t M, int64_t N, int64_t K,
                                               int dtype, int inter_f32, void* stream) {
  const size_t need = fgemm_unfused_workspace_bytes(M, N, dtype, inter_f32);
  if (need == 0)  // empty problem or invalid arguments: the chain's own checks answer
    return fgemm_unfused_bias_relu(A, B, bias, out, M, N, K, dtype, nullptr, 0, inter_f32, stream);
  if (need > FGEMM_NOALLOC_SCRATCH_BYTES) return FGEMM_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_on_current_device(&scratch);
  if (st != FGEMM_OK) return st;
  return fgemm_unfused_bias_relu(A, B, bias, out, M, N, K, dtype, scratch,
                                 FGEMM_NOALLOC_SCRATCH_BYTES, inter_f32, stream);
}
