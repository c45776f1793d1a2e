// Weight-streaming GEMV for one to four tokens (decode):
//   y[t, n] = epi(sum_k x[t, k] W[n, k] (+ b[n])).
// The host uses it for one token, and for two when the call's weights are small; the
// few-token tcgen05 kernel (gemm_skinny.cu) is faster from there on.
//
// At one token the feed-forward block reads every weight once and does one multiply-add per
// weight, so it is bound by HBM bandwidth and by launch latency (ainews.cool fused-MLP
// article, technical deep-dive: batch-1 decode pays one launch per layer and is limited by
// memory traffic). The kernel is built to keep HBM busy:
//   - each CTA owns a contiguous block of weight rows [r0, r1) (balanced to +-1 row), two
//     CTAs of 16 warps per SM;
//   - the CTA's rows are cut into 512-byte segments (256 weights, one 16-byte vector per
//     lane) and each warp takes one contiguous run of segments, so every warp streams its own
//     contiguous range of W with 8 non-allocating 128-bit loads per lane in flight;
//   - programmatic dependent launch: the kernel lets the next kernel launch at once; after
//     waiting for the previous kernel, the first batch of weight loads is issued before x is
//     staged, so the x load hides under them. (L2 prefetches of the CTA's own rows, or of the
//     next layer's weights, were measured to slow the decode forward down: they queue ahead
//     of the loads the warps need first.)
//   - x (T x K bf16) sits in shared memory; each lane accumulates its dot products in fp32
//     across the consecutive segments of one row and the warp reduces with shuffles only when
//     its run crosses a row boundary. The reduced sum of a run piece is stored as the partial
//     of the piece's first segment (the piece's other segments get 0), and one thread per
//     (row, token) adds a row's partials in segment order: deterministic for a given shape;
//   - with two weight matrices (GeGLU gate and up) both blocks are streamed and the epilogue
//     forms gelu_tanh(g) * u.
#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

constexpr int kGemvThreads = 512;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kSeg = 256;                  // weights per segment (512 bytes)
constexpr int kGemvCtasPerSm = 2;
constexpr int kGemvBatch = 8;              // 16-byte loads in flight per lane

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float dot8(uint4 w, uint4 x, float s) {
  s = fmaf(bf16_lo(w.x), bf16_lo(x.x), s);
  s = fmaf(bf16_hi(w.x), bf16_hi(x.x), s);
  s = fmaf(bf16_lo(w.y), bf16_lo(x.y), s);
  s = fmaf(bf16_hi(w.y), bf16_hi(x.y), s);
  s = fmaf(bf16_lo(w.z), bf16_lo(x.z), s);
  s = fmaf(bf16_hi(w.z), bf16_hi(x.z), s);
  s = fmaf(bf16_lo(w.w), bf16_lo(x.w), s);
  s = fmaf(bf16_hi(w.w), bf16_hi(x.w), s);
  return s;
}

// Reduce a warp's per-lane sums (one per token), store them at part[pi .. pi+T), and clear
// the accumulators.
template <int TMAX>
__device__ __forceinline__ void flush_piece(float (&acc)[TMAX], float* part, size_t pi, int T,
                                            int lane) {
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
  }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < TMAX; ++t)
      if (t < T) part[pi + t] = acc[t];
  }
#pragma unroll
  for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
}

__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// One layer for this CTA's rows [r0, r1) of W (NMAT matrices): y[t, n] for n in [r0, r1).
// All threads of the CTA take part (it synchronises internally). x, which the kernel this one
// waited for may have written, is read through L2 (never a possibly stale L1 line).
template <int EPI, int NMAT, int TMAX>
__device__ __forceinline__ void gemv_rows(uint8_t* gsm, const __nv_bfloat16* __restrict__ x,
                                          const __nv_bfloat16* __restrict__ W0,
                                          const __nv_bfloat16* __restrict__ W1,
                                          const __nv_bfloat16* __restrict__ bias,
                                          __nv_bfloat16* __restrict__ y, int T, int K, int N,
                                          int ldx, int ldy, int gelu_mode, int r0, int r1) {
  const int rows = r1 - r0;
  const int segs = K / kSeg;
  const int per_mat = rows * segs;
  const int total = NMAT * per_mat;          // segments this CTA streams
  uint4* xs = reinterpret_cast<uint4*>(gsm);                                     // [T][K/8]
  float* part = reinterpret_cast<float*>(gsm + static_cast<size_t>(T) * K * 2);  // [seg][T]

  // warp w streams segments [g0, g1) of the CTA's list (matrix-major, then row, then segment)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g0 = static_cast<int>((static_cast<int64_t>(warp) * total) / kGemvWarps);
  const int g1 = static_cast<int>((static_cast<int64_t>(warp + 1) * total) / kGemvWarps);
  uint4 wv[kGemvBatch];
  auto load_batch = [&](int base) {
#pragma unroll
    for (int u = 0; u < kGemvBatch; ++u) {
      const int g = base + u;
      if (g < g1) {
        const int mat = NMAT == 2 ? (g >= per_mat ? 1 : 0) : 0;
        const int gm = g - mat * per_mat;
        const __nv_bfloat16* Wm = mat ? W1 : W0;
        // consecutive segments of a matrix block are consecutive 512-byte pieces of memory
        wv[u] = ld_stream_v4(Wm + static_cast<size_t>(r0) * K + static_cast<size_t>(gm) * kSeg +
                             lane * 8);
      } else {
        wv[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  load_batch(g0);   // in flight while x is staged

  // x rows are ldx elements apart (a multiple of 8); xs packs them
  const int kvec = K / 8, xvec = T * kvec;
  for (int i = threadIdx.x; i < xvec; i += kGemvThreads) {
    const int t = i / kvec;
    xs[i] = ld_cg_v4(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * ldx) + (i - t * kvec));
  }
  __syncthreads();

  float acc[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
  int piece_row = -1;   // (matrix, row) id of the run piece being accumulated
  size_t piece_pi = 0;  // its partial index
  for (int base = g0; base < g1; base += kGemvBatch) {
    if (base != g0) load_batch(base);
#pragma unroll
    for (int u = 0; u < kGemvBatch; ++u) {
      const int g = base + u;
      if (g >= g1) break;  // warp-uniform
      const int mat = NMAT == 2 ? (g >= per_mat ? 1 : 0) : 0;
      const int gm = g - mat * per_mat;
      const int row = gm / segs, seg = gm - row * segs;
      const int rid = mat * rows + row;
      const size_t pi = static_cast<size_t>(g) * T;
      if (rid != piece_row) {
        if (piece_row >= 0) flush_piece<TMAX>(acc, part, piece_pi, T, lane);
        piece_row = rid;
        piece_pi = pi;
      } else if (lane == 0) {
#pragma unroll
        for (int t = 0; t < TMAX; ++t)
          if (t < T) part[pi + t] = 0.f;
      }
#pragma unroll
      for (int t = 0; t < TMAX; ++t)
        if (t < T) acc[t] = dot8(wv[u], xs[t * (K / 8) + seg * (kSeg / 8) + lane], acc[t]);
    }
  }
  if (piece_row >= 0) flush_piece<TMAX>(acc, part, piece_pi, T, lane);
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
    y[static_cast<size_t>(t) * ldy + n] = __float2bfloat16_rn(v);
  }
  __syncthreads();   // the shared memory may be reused by the caller
}

__device__ __forceinline__ int split_row(int i, int N) {
  return static_cast<int>((static_cast<int64_t>(i) * N) / gridDim.x);
}

template <int EPI, int NMAT, int TMAX>
__global__ void __launch_bounds__(kGemvThreads, kGemvCtasPerSm)
    gemv_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ W0,
                const __nv_bfloat16* __restrict__ W1, const __nv_bfloat16* __restrict__ bias,
                __nv_bfloat16* __restrict__ y, int T, int K, int N, int ldx, int ldy,
                int gelu_mode) {
  extern __shared__ __align__(16) uint8_t gsm[];
  const int r0 = split_row(blockIdx.x, N), r1 = split_row(blockIdx.x + 1, N);
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait_primary();
  gemv_rows<EPI, NMAT, TMAX>(gsm, x, W0, W1, bias, y, T, K, N, ldx, ldy, gelu_mode, r0, r1);
}

size_t gemv_smem_bytes(int T, int K, int N, int nmat, int grid) {
  const int64_t rows_max = (static_cast<int64_t>(N) + grid - 1) / grid;
  return static_cast<size_t>(T) * K * 2 +
         static_cast<size_t>(nmat) * rows_max * (K / kSeg) * T * 4;
}

// Two CTAs per SM (each at most half of an SM's registers and threads).
int gemv_grid(int T, int K, int N, int nmat, int sms) {
  (void)T;
  (void)K;
  (void)nmat;
  const int g = sms * kGemvCtasPerSm;
  return g < N ? g : N;
}

template <int EPI, int NMAT, int TMAX>
static cudaError_t gemv_launch_t(const GemvLaunch& L, size_t smem) {
  auto kern = gemv_kernel<EPI, NMAT, TMAX>;
  static SmemAttrCache cache;
  cudaError_t e =
      set_smem_limit(reinterpret_cast<const void*>(kern), static_cast<int>(smem), cache);
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
                            static_cast<__nv_bfloat16*>(L.y), L.T, L.K, L.N, L.ldx, L.ldy,
                            L.gelu_mode);
}

cudaError_t gemv_launch(const GemvLaunch& L) {
  const int nmat = L.epi == EPI_GEGLU ? 2 : 1;
  const size_t smem = gemv_smem_bytes(L.T, L.K, L.N, nmat, L.grid);
  if (L.T < 1 || L.T > kGemvMaxT || L.K % kSeg != 0 || L.grid < 1 || smem > kGemvMaxSmem)
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
