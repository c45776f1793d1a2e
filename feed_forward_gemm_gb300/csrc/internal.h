// Declarations shared between the host C-ABI translation unit and the kernel translation
// units. Host-only; no device code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fmlp {

// Epilogue kinds of the tcgen05 GEMM.
enum Epi : int {
  EPI_BIAS = 0,       // y = acc (+ bias)
  EPI_BIAS_GELU = 1,  // h = gelu(acc (+ bias))
  EPI_GEGLU = 2,      // m = gelu_tanh(acc_gate) * acc_up   (two B operands)
};

// One launch of the persistent tcgen05 GEMM: D[M, N] = A[M, K] B[N, K]^T with an epilogue.
struct GemmLaunch {
  CUtensorMap tmA;    // A  [M, K] bf16, box {64, 128}, 128B swizzle
  CUtensorMap tmB0;   // B  [N, K] bf16 (Wg for GeGLU), box {64, bn or bn/2}, 128B swizzle
  CUtensorMap tmB1;   // Wu for GeGLU (unused otherwise), box {64, bn/2}
  CUtensorMap tmY;    // output [M, N_out] bf16, box {64, 32}, 128B swizzle
  const void* bias;   // [N_out] bf16 or nullptr
  int M, N_out, K;
  int gelu_mode;      // 0 tanh, 1 erf
  int epi;            // Epi
  int bn;             // MMA N: 64, 128 or 256 (GeGLU: gate bn/2 + up bn/2)
  int grid;           // persistent CTAs
  bool pdl;           // launch as a programmatic dependent of the previous kernel
  cudaStream_t stream;
  int* status;        // device status word
  uint64_t timeout_ns;
};

cudaError_t gemm_tc_launch(const GemmLaunch& L);
// Dynamic shared memory a GEMM configuration needs (0 if the configuration does not exist).
int gemm_tc_smem_bytes(int epi, int bn);

// Device GELU check kernel.
cudaError_t gelu_eval_launch(const float* in, float* out, int64_t n, int mode,
                             cudaStream_t stream);

// Bounded-wait test kernel.
cudaError_t wait_timeout_launch(uint64_t timeout_ns, int* status, cudaStream_t stream);

}  // namespace fmlp
