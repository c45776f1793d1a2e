// Weight-streaming GEMV for a few tokens (decode): y[t, n] = epi(sum_k x[t, k] W[n, k] (+ b[n])).
//
// At one token the feed-forward block reads every weight once and does two flops per weight
// byte pair, so it is bound by HBM bandwidth and by launch latency (ainews.cool fused-MLP
// article, technical deep-dive: batch-1 decode pays one launch per layer). The kernel is
// built for that:
//   - each CTA owns a contiguous block of weight rows [r0, r1) (balanced to +-1 row), so the
//     bytes it streams are one contiguous range of W;
//   - a row is cut into 512-byte segments (256 bf16, one 16-byte load per lane); warp w of
//     the CTA takes segments w, w+16, w+32, ... and keeps 8 of them (4 KB) in flight per
//     batch with non-allocating 128-bit loads;
//   - x (T x K bf16) sits in shared memory; each segment's dot product is reduced with warp
//     shuffles in fp32, the per-segment partials go to shared memory, and one thread per
//     (row, token) adds them in segment order (deterministic) and applies the epilogue;
//   - with two weight matrices (GeGLU gate and up) both are streamed and the epilogue forms
//     gelu_tanh(g) * u;
//   - programmatic dependent launch: the kernel lets the next kernel launch at once, prefetches
//     its own weight range into L2 and only then waits for the previous kernel, so one layer's
//     weight stream overlaps the previous layer's tail and launch.
#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

constexpr int kGemvThreads = 512;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kGemvBatch = 8;
constexpr int kSeg = 256;  // elements per segment

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float dot8(uint4 w, uint4 x) {
  float s = bf16_lo(w.x) * bf16_lo(x.x);
  s = fmaf(bf16_hi(w.x), bf16_hi(x.x), s);
  s = fmaf(bf16_lo(w.y), bf16_lo(x.y), s);
  s = fmaf(bf16_hi(w.y), bf16_hi(x.y), s);
  s = fmaf(bf16_lo(w.z), bf16_lo(x.z), s);
  s = fmaf(bf16_hi(w.z), bf16_hi(x.z), s);
  s = fmaf(bf16_lo(w.w), bf16_lo(x.w), s);
  s = fmaf(bf16_hi(w.w), bf16_hi(x.w), s);
  return s;
}

template <int EPI, int NMAT, int TMAX>
__global__ void __launch_bounds__(kGemvThreads, 2)
    gemv_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ W0,
                const __nv_bfloat16* __restrict__ W1, const __nv_bfloat16* __restrict__ bias,
                __nv_bfloat16* __restrict__ y, int T, int K, int N, int gelu_mode) {
  extern __shared__ __align__(16) uint8_t gsm[];
  const int rows_total = N;
  const int r0 = static_cast<int>((static_cast<int64_t>(blockIdx.x) * rows_total) / gridDim.x);
  const int r1 =
      static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * rows_total) / gridDim.x);
  const int rows = r1 - r0;
  const int segs = K / kSeg;
  const int per_mat = rows * segs;
  const int ntask = NMAT * per_mat;

  uint4* xs = reinterpret_cast<uint4*>(gsm);                        // [T][K/8]
  float* part = reinterpret_cast<float*>(gsm + static_cast<size_t>(T) * K * 2);  // [task][T]

  if (threadIdx.x == 0) pdl_launch_dependents();
  // Warm L2 with this CTA's weight rows; they do not depend on the previous kernel.
  if (threadIdx.x < NMAT) {
    const __nv_bfloat16* Wm = threadIdx.x == 0 ? W0 : W1;
    const char* base = reinterpret_cast<const char*>(Wm + static_cast<size_t>(r0) * K);
    size_t bytes = static_cast<size_t>(rows) * K * 2;
    for (size_t off = 0; off < bytes; off += 65536) {
      const size_t n = bytes - off < 65536 ? bytes - off : 65536;
      prefetch_l2_bulk(base + off, static_cast<uint32_t>(n));
    }
  }
  pdl_wait_primary();

  // x -> shared memory
  const int xvec = T * (K / 8);
  for (int i = threadIdx.x; i < xvec; i += kGemvThreads)
    xs[i] = __ldg(reinterpret_cast<const uint4*>(x) + i);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int base = warp; base < ntask; base += kGemvWarps * kGemvBatch) {
    uint4 wv[kGemvBatch];
#pragma unroll
    for (int u = 0; u < kGemvBatch; ++u) {
      const int q = base + u * kGemvWarps;
      if (q < ntask) {
        const int mat = NMAT == 2 ? (q >= per_mat ? 1 : 0) : 0;
        const int rem = q - mat * per_mat;
        const int row = rem / segs, seg = rem - row * segs;
        const __nv_bfloat16* Wm = mat ? W1 : W0;
        wv[u] = ld_stream_v4(Wm + static_cast<size_t>(r0 + row) * K + seg * kSeg + lane * 8);
      } else {
        wv[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < kGemvBatch; ++u) {
      const int q = base + u * kGemvWarps;
      if (q >= ntask) break;  // warp-uniform
      const int mat = NMAT == 2 ? (q >= per_mat ? 1 : 0) : 0;
      const int rem = q - mat * per_mat;
      const int seg = rem % segs;
      float p[TMAX];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        p[t] = 0.f;
        if (t < T) p[t] = dot8(wv[u], xs[t * (K / 8) + seg * (kSeg / 8) + lane]);
      }
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) p[t] += __shfl_xor_sync(0xffffffffu, p[t], o);
      }
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < TMAX; ++t)
          if (t < T) part[static_cast<size_t>(q) * T + t] = p[t];
      }
    }
  }
  __syncthreads();

  // one thread per (row, token): add the segments in order, then the epilogue
  for (int i = threadIdx.x; i < rows * T; i += kGemvThreads) {
    const int row = i / T, t = i - row * T;
    float s0 = 0.f, s1 = 0.f;
    for (int sg = 0; sg < segs; ++sg) s0 += part[static_cast<size_t>(row * segs + sg) * T + t];
    if (NMAT == 2)
      for (int sg = 0; sg < segs; ++sg)
        s1 += part[static_cast<size_t>(per_mat + row * segs + sg) * T + t];
    const int n = r0 + row;
    float v;
    if (EPI == EPI_GEGLU) {
      v = gelu_tanh_f(s0) * s1;
    } else {
      const float z = s0 + (bias != nullptr ? __bfloat162float(bias[n]) : 0.f);
      v = EPI == EPI_BIAS_GELU ? gelu_f(z, gelu_mode) : z;
    }
    y[static_cast<size_t>(t) * N + n] = __float2bfloat16_rn(v);
  }
}

size_t gemv_smem_bytes(int T, int K, int N, int nmat, int grid) {
  const int64_t rows_max = (static_cast<int64_t>(N) + grid - 1) / grid;
  return static_cast<size_t>(T) * K * 2 +
         static_cast<size_t>(nmat) * rows_max * (K / kSeg) * T * 4;
}

template <int EPI, int NMAT, int TMAX>
static cudaError_t gemv_launch_t(const GemvLaunch& L, size_t smem) {
  auto kern = gemv_kernel<EPI, NMAT, TMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const __nv_bfloat16*>(L.x),
                            static_cast<const __nv_bfloat16*>(L.W0),
                            static_cast<const __nv_bfloat16*>(L.W1),
                            static_cast<const __nv_bfloat16*>(L.bias),
                            static_cast<__nv_bfloat16*>(L.y), L.T, L.K, L.N, L.gelu_mode);
}

cudaError_t gemv_launch(const GemvLaunch& L) {
  const int nmat = L.epi == EPI_GEGLU ? 2 : 1;
  const size_t smem = gemv_smem_bytes(L.T, L.K, L.N, nmat, L.grid);
  if (L.T < 1 || L.T > kGemvMaxT || L.K % kSeg != 0 || smem > kGemvMaxSmem)
    return cudaErrorInvalidValue;
  if (L.T == 1) {
    switch (L.epi) {
      case EPI_BIAS: return gemv_launch_t<EPI_BIAS, 1, 1>(L, smem);
      case EPI_BIAS_GELU: return gemv_launch_t<EPI_BIAS_GELU, 1, 1>(L, smem);
      case EPI_GEGLU: return gemv_launch_t<EPI_GEGLU, 2, 1>(L, smem);
    }
  } else {
    switch (L.epi) {
      case EPI_BIAS: return gemv_launch_t<EPI_BIAS, 1, kGemvMaxT>(L, smem);
      case EPI_BIAS_GELU: return gemv_launch_t<EPI_BIAS_GELU, 1, kGemvMaxT>(L, smem);
      case EPI_GEGLU: return gemv_launch_t<EPI_GEGLU, 2, kGemvMaxT>(L, smem);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace fmlp
