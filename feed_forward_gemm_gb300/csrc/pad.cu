// Zero-padded copies for inner dimensions that are not multiples of 8.
//
// TMA moves rows whose byte stride is a multiple of 16, so a bf16 matrix with a row of `cols`
// elements packed back to back needs cols % 8 == 0. A call with other sizes runs on copies
// padded with zeros to the next multiple of 8 in every inner dimension, which changes no
// result: a zero column of x and W adds nothing to a dot product; a zero row of W (or of b)
// gives an output that is dropped; in the blocks, a zero gate/up row gives
// m = gelu_tanh(0) * 0 = 0 and a zero first-layer row with a zero bias gives h = act(0) = 0
// (GELU and ReLU of 0 are 0), which the zero columns of the second layer then multiply.
// ("Profiling in PyTorch (Part 2)", section "What's the transpose doing?": a tensor is a flat
// buffer plus shape and strides; the copy only changes the strides the kernels see.)
#include "internal.h"

namespace fmlp {

namespace {

constexpr int kPadThreads = 256;

// dst[r][c] = src[r * ld + c] for r < rows and c < cols, 0 elsewhere, over dst's
// dst_rows x dst_cols (dst_cols a multiple of 8; each thread writes 8 elements).
__global__ void __launch_bounds__(kPadThreads) pad2d_kernel(const uint16_t* __restrict__ src,
                                                            int64_t ld, int64_t rows,
                                                            int64_t cols, uint16_t* __restrict__ dst,
                                                            int64_t dst_rows, int64_t dst_cols) {
  const int64_t vec_per_row = dst_cols / 8;
  const int64_t n = dst_rows * vec_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / vec_per_row, c0 = (i - r * vec_per_row) * 8;
    uint16_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      v[e] = (r < rows && c0 + e < cols) ? src[r * ld + c0 + e] : static_cast<uint16_t>(0);
    uint4 o;
    o.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
    o.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
    o.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
    o.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
    reinterpret_cast<uint4*>(dst)[i] = o;
  }
}

// dst[r * ld_dst + c] = src[r * ld_src + c] for r < rows, c < cols.
__global__ void __launch_bounds__(kPadThreads) copy2d_kernel(const uint16_t* __restrict__ src,
                                                             int64_t ld_src,
                                                             uint16_t* __restrict__ dst,
                                                             int64_t ld_dst, int64_t rows,
                                                             int64_t cols) {
  const int64_t n = rows * cols;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / cols, c = i - r * cols;
    dst[r * ld_dst + c] = src[r * ld_src + c];
  }
}

int grid_for(int64_t work) {
  const int64_t g = (work + kPadThreads - 1) / kPadThreads;
  return static_cast<int>(g < 1 ? 1 : (g > 4096 ? 4096 : g));
}

}  // namespace

cudaError_t pad2d_launch(const void* src, int64_t ld, int64_t rows, int64_t cols, void* dst,
                         int64_t dst_rows, int64_t dst_cols, cudaStream_t s) {
  if (dst_cols % 8 != 0 || rows > dst_rows || cols > dst_cols || ld < cols)
    return cudaErrorInvalidValue;
  pad2d_kernel<<<grid_for(dst_rows * dst_cols / 8), kPadThreads, 0, s>>>(
      static_cast<const uint16_t*>(src), ld, rows, cols, static_cast<uint16_t*>(dst), dst_rows,
      dst_cols);
  return cudaGetLastError();
}

cudaError_t copy2d_launch(const void* src, int64_t ld_src, void* dst, int64_t ld_dst,
                          int64_t rows, int64_t cols, cudaStream_t s) {
  if (ld_src < cols || ld_dst < cols) return cudaErrorInvalidValue;
  copy2d_kernel<<<grid_for(rows * cols), kPadThreads, 0, s>>>(
      static_cast<const uint16_t*>(src), ld_src, static_cast<uint16_t*>(dst), ld_dst, rows, cols);
  return cudaGetLastError();
}

}  // namespace fmlp
