// fmlp_geglu_noalloc: the GeGLU block for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc or any allocating routine: a plugin inside a serving
// process whose memory pool owns the whole device and forbids allocations after start-up, or
// a real-time loop that may not risk an allocation stall or failure. fmlp_geglu needs a
// workspace for the intermediate m between its stages; this entry point takes that workspace
// from a fixed array in the library's own device memory instead, so it allocates nothing.
//
// The array lives at file scope as a static __device__ object, so every GPU that loads the
// library holds it until the process exits. In host code its name is only a host-side stand-
// in, never a device address: the address kernels use is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached. The first call on a device does
// that look-up; make it before any stream capture on that device. A device reset
// (cudaDeviceReset) while the library is loaded leaves the cached address stale and is not
// supported.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fmlp.h"
#include "internal.h"

namespace fmlp {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

// Holds m (T x H bf16) between the GeGLU block's stages; shared by every call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

}  // namespace
}  // namespace fmlp

using namespace fmlp;

extern "C" fmlp_status fmlp_geglu_noalloc(const void* x, const void* Wg, const void* Wu,
                                          const void* Wd, void* y, int64_t T, int64_t D,
                                          int64_t H, fmlp_stream_t s) {
  // the shape checks come first, so a bad size reports FMLP_ERR_SHAPE, not a scratch overflow
  const int shape = validate_block_dims(T, D, H);
  if (shape != FMLP_OK) return static_cast<fmlp_status>(shape);
  const size_t need = fmlp_geglu_workspace_size(T, D, H);
  if (need > kNoAllocScratchBytes) {
    record_error("fmlp_geglu_noalloc: T*H*2 = %zu bytes of intermediate exceed the fixed "
                 "%zu-byte device scratch; use fmlp_geglu with a workspace",
                 need, kNoAllocScratchBytes);
    return FMLP_ERR_WORKSPACE;
  }
  // Nothing to hold (T == 0, or the single-kernel plan keeps m on chip): no scratch needed,
  // and fmlp_geglu allocates nothing for these sizes.
  if (need == 0) return fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, nullptr, 0, s);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    record_error("fmlp_geglu_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    return FMLP_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) {
    record_error("fmlp_geglu_noalloc: device ordinal %d out of range", dev);
    return FMLP_ERR_DEVICE;
  }
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      e = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_noalloc_scratch);
      if (e != cudaSuccess) {
        g_scratch_ptr[dev] = nullptr;
        record_error("fmlp_geglu_noalloc: cudaGetSymbolAddress(scratch): %s",
                     cudaGetErrorString(e));
        return FMLP_ERR_CUDA;
      }
    }
    ptr = g_scratch_ptr[dev];
  }
  return fmlp_geglu(x, Wg, Wu, Wd, y, T, D, H, ptr, kNoAllocScratchBytes, s);
}
