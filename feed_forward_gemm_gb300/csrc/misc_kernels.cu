// Small utility kernels: the device GELU check and the bounded-wait test.
#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

__global__ void gelu_eval_kernel(const float* __restrict__ in, float* __restrict__ out,
                                 int64_t n, int mode) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride)
    out[i] = gelu_f(in[i], mode);
}

cudaError_t gelu_eval_launch(const float* in, float* out, int64_t n, int mode,
                             cudaStream_t stream) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  gelu_eval_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(in, out, n, mode);
  return cudaGetLastError();
}

// One thread waits on an mbarrier that expects one arrival nobody makes. The bounded wait
// gives up after timeout_ns, records the timeout and the kernel returns normally.
__global__ void wait_timeout_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, status, SITE_TEST, timeout_ns);
}

cudaError_t wait_timeout_launch(uint64_t timeout_ns, int* status, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fmlp
