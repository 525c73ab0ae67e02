// noalloc.cu -- retention_chunkwise_noalloc: the chunkwise forward for callers
// that must not allocate device memory.
//
// Some callers cannot allocate at call time: serving runtimes that plan every
// device buffer once at start-up and keep a fixed memory budget (an allocation
// on the request path can fail under memory pressure, stall on the pool, or
// fragment it), and embedders whose host code may not call into the CUDA
// allocator at all.  For them this entry point runs the same chunkwise kernels
// as retention_chunkwise, but the float32 segment-state scratch those kernels
// use lives in a file-scope device array of fixed size, reserved when the
// library is loaded and held by every GPU that loads it until the process
// exits.  No call here allocates or frees memory.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "internal.h"
#include "retention.h"

namespace {

// Fixed scratch for the segment states: 8 MiB per device.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock[kMaxDevices];
void* g_scratch[kMaxDevices];  // written under g_lock[dev], only with a successful lookup

// Device address of g_static_scratch on device `dev`, which must be current.
// The host-side symbol is only a stand-in and is never handed to a kernel.
// Only a successful lookup is kept: a failed one (for instance an error left
// pending by an earlier call) is tried again on the device's next call.
cudaError_t static_scratch(int dev, void** ptr) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> hold(g_lock[dev]);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch[dev] = p;
  }
  *ptr = g_scratch[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int retention_chunkwise_noalloc(const void* q, const void* k, const void* v,
                                           const float* gamma, void* out, float* state_out, int B,
                                           int H, int N, int dk, int dv, int chunk, void* stream) {
  // the plan that fits the static scratch (a call with more units than SMs
  // then leaves its last wave whole rather than need more)
  size_t need = 0;
  int st = ret::chunkwise_workspace_within(B, H, N, dk, dv, chunk, kStaticScratchBytes, &need);
  if (st != RET_OK) return st;
  if (need > kStaticScratchBytes) return RET_ERR_UNSUPPORTED;  // beyond the static scratch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RET_ERR_CUDA;
  void* scratch = nullptr;
  if (static_scratch(dev, &scratch) != cudaSuccess || scratch == nullptr) return RET_ERR_CUDA;
  return retention_chunkwise_ws(q, k, v, gamma, out, state_out, B, H, N, dk, dv, chunk, scratch,
                                kStaticScratchBytes, stream);
}
