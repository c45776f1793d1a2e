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
//     contiguous range of W with 8 non-allocating 128-bit loads per lane in flight; each
//     register, once its segment is summed, takes the load 8 segments ahead, so the
//     arithmetic overlaps the stream instead of alternating with it;
//   - programmatic dependent launch: the kernel lets the next kernel launch at once; after
//     waiting for the previous kernel, the first batch of weight loads is issued before x is
//     staged, so the x load hides under them. (Requesting x first, L2 prefetches of the CTA's
//     own rows, of the next layer's weights, or before the dependency wait, and one CTA per SM
//     so the next kernel can be resident early, were all measured slower.)
//   - x (T x K) sits in shared memory, widened to fp32 when that still leaves room for two
//     CTAs per SM; each lane accumulates its dot products in fp32 (packed f32x2
//     multiply-adds) across the consecutive segments of one row and the warp reduces with
//     shuffles only when its run crosses a row boundary, storing the piece's sum as the
//     partial of (row, warp). A row's 16 partials are then added by a butterfly in a fixed
//     order: deterministic for a given shape. The (matrix, row, segment) cursor advances by
//     additions: a division by the run-time segment count per segment cost more instructions
//     than the multiply-adds;
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

__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// acc (packed even, odd element sums) += the 8 products of weight chunk w and the x chunk
// given as four packed fp32 pairs.
__device__ __forceinline__ void dot8p(uint64_t& acc, uint4 w, uint64_t x01, uint64_t x23,
                                      uint64_t x45, uint64_t x67) {
  ffma2p(acc, bf16x2_to_f2(w.x), x01);
  ffma2p(acc, bf16x2_to_f2(w.y), x23);
  ffma2p(acc, bf16x2_to_f2(w.z), x45);
  ffma2p(acc, bf16x2_to_f2(w.w), x67);
}

// One layer for this CTA's rows [r0, r1) of W (NMAT matrices): y[t, n] for n in [r0, r1).
// All threads of the CTA take part (it synchronises internally). x, which the kernel this one
// waited for may have written, is read through L2 (never a possibly stale L1 line).
//
// x sits in shared memory widened to fp32 (XF32) or as bf16 (when fp32 would not leave room
// for two CTAs per SM). The fp32 copy is split by halves of each 16-byte chunk: token t's
// chunk c is lo = elements 8c..8c+3 at float4 index t * 2C + c and hi = 8c+4..8c+7 at
// t * 2C + C + c (C = K / 8), so a warp's lanes, on consecutive chunks, read consecutive
// 16-byte words. The streaming loop walks (matrix, row, segment) with a cursor advanced by
// additions only: a division by the run-time segment count per segment used to cost more
// instructions than the multiply-adds.
template <int EPI, int NMAT, int TMAX, bool XF32>
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
  const int C = K / 8;
  const size_t xbytes = static_cast<size_t>(T) * K * (XF32 ? 4 : 2);
  // partial sums, one per (matrix, row, warp, token): a warp's run of segments covers at most
  // one contiguous piece of each row
  float* part = reinterpret_cast<float*>(gsm + xbytes);
  const uint32_t xs = smem_u32(gsm);

  // warp w streams segments [g0, g1) of the CTA's list (matrix-major, then row, then segment)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g0 = static_cast<int>((static_cast<int64_t>(warp) * total) / kGemvWarps);
  const int g1 = static_cast<int>((static_cast<int64_t>(warp + 1) * total) / kGemvWarps);
  // this lane's 16 bytes of segment g (consecutive segments of a matrix block are consecutive
  // 512-byte pieces of memory)
  auto load_seg = [&](int g) {
    const int mat = NMAT == 2 ? (g >= per_mat ? 1 : 0) : 0;
    const int gm = g - mat * per_mat;
    const __nv_bfloat16* Wm = mat ? W1 : W0;
    return ld_stream_v4(Wm + static_cast<size_t>(r0) * K + static_cast<size_t>(gm) * kSeg +
                        lane * 8);
  };
  auto stage_x = [&](int i, uint4 v) {
    if (XF32) {
      const int t = i / C, c = i - t * C;
      float4* xf = reinterpret_cast<float4*>(gsm);
      xf[t * 2 * C + c] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
      xf[t * 2 * C + C + c] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
    } else {
      reinterpret_cast<uint4*>(gsm)[i] = v;
    }
  };
  auto x_at = [&](int i) {   // x rows are ldx elements apart (a multiple of 8)
    const int t = i / C, c = i - t * C;
    return ld_cg_v4(x + static_cast<size_t>(t) * ldx + static_cast<size_t>(c) * 8);
  };
  // the first weights go out before x is requested (x first was measured slower: it holds
  // back the weight stream)
  uint4 wv[kGemvBatch];
#pragma unroll
  for (int u = 0; u < kGemvBatch; ++u)
    wv[u] = g0 + u < g1 ? load_seg(g0 + u) : make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < T * C; i += kGemvThreads) stage_x(i, x_at(i));
  for (int i = threadIdx.x; i < NMAT * rows * kGemvWarps * T; i += kGemvThreads) part[i] = 0.f;
  __syncthreads();

  // cursor of the segment being summed: matrix, row, segment within the row
  int cmat = NMAT == 2 ? (g0 >= per_mat ? 1 : 0) : 0;
  int crow = 0, cseg = 0;
  if (g1 > g0) {
    const int gm = g0 - cmat * per_mat;
    crow = gm / segs;
    cseg = gm - crow * segs;
  }
  // accumulator pairs per token (two at one token, alternating between segments, so the
  // multiply-add chains are shorter; one at more tokens, where the tokens already interleave)
  constexpr int NA = TMAX == 1 ? 2 : 1;
  uint64_t acc[TMAX][NA];   // packed fp32 pairs; all-zero bits are (+0, +0)
#pragma unroll
  for (int t = 0; t < TMAX; ++t)
#pragma unroll
    for (int k = 0; k < NA; ++k) acc[t][k] = 0ull;
  int piece_row = -1;   // (matrix, row) id of the run piece being accumulated
  auto flush = [&]() {
    float v[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      const float2 a0 = unpack_f2(acc[t][0]);
      v[t] = a0.x + a0.y;
      if (NA == 2) {
        const float2 a1 = unpack_f2(acc[t][NA - 1]);
        v[t] += a1.x + a1.y;
      }
#pragma unroll
      for (int k = 0; k < NA; ++k) acc[t][k] = 0ull;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v[t] += __shfl_xor_sync(0xffffffffu, v[t], o);
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < TMAX; ++t)
        if (t < T) part[(piece_row * kGemvWarps + warp) * T + t] = v[t];
    }
  };
  for (int base = g0; base < g1; base += kGemvBatch) {
#pragma unroll
    for (int u = 0; u < kGemvBatch; ++u) {
      const int g = base + u;
      if (g >= g1) break;  // warp-uniform
      const int rid = cmat * rows + crow;
      if (rid != piece_row) {
        if (piece_row >= 0) flush();
        piece_row = rid;
      }
      const uint32_t chunk = static_cast<uint32_t>(cseg * (kSeg / 8) + lane);
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          uint64_t x01, x23, x45, x67;
          if (XF32) {
            const uint32_t xt = xs + static_cast<uint32_t>(t) * static_cast<uint32_t>(C) * 32u;
            lds_f2x2(xt + chunk * 16u, x01, x23);
            lds_f2x2(xt + static_cast<uint32_t>(C) * 16u + chunk * 16u, x45, x67);
          } else {
            const uint4 xv = lds_v4(xs + (static_cast<uint32_t>(t) * static_cast<uint32_t>(C) +
                                          chunk) * 16u);
            x01 = bf16x2_to_f2(xv.x);
            x23 = bf16x2_to_f2(xv.y);
            x45 = bf16x2_to_f2(xv.z);
            x67 = bf16x2_to_f2(xv.w);
          }
          dot8p(acc[t][u % NA], wv[u], x01, x23, x45, x67);
        }
      }
      // the register just used takes the load kGemvBatch segments ahead, so that the
      // arithmetic overlaps the stream (about kGemvBatch loads per lane stay in flight)
      if (g + kGemvBatch < g1) wv[u] = load_seg(g + kGemvBatch);
      // advance the cursor
      if (++cseg == segs) {
        cseg = 0;
        if (++crow == rows) {
          crow = 0;
          ++cmat;
        }
      }
    }
  }
  if (piece_row >= 0) flush();
  __syncthreads();

  // one warp per (row, token): lanes 0..15 take the 16 warps' partials of the row, summed by
  // a butterfly (a fixed order: deterministic), then the epilogue
  for (int i = warp; i < rows * T; i += kGemvWarps) {
    const int row = i / T, t = i - row * T;
    float s0 = lane < kGemvWarps ? part[(row * kGemvWarps + lane) * T + t] : 0.f;
    float s1 = 0.f;
    if (NMAT == 2 && lane < kGemvWarps) s1 = part[((rows + row) * kGemvWarps + lane) * T + t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, o);
      if (NMAT == 2) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    }
    if (lane == 0) {
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
  }
  __syncthreads();   // the shared memory may be reused by the caller
}

__device__ __forceinline__ int split_row(int i, int N) {
  return static_cast<int>((static_cast<int64_t>(i) * N) / gridDim.x);
}

template <int EPI, int NMAT, int TMAX, bool XF32>
__global__ void __launch_bounds__(kGemvThreads, kGemvCtasPerSm)
    gemv_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ W0,
                const __nv_bfloat16* __restrict__ W1, const __nv_bfloat16* __restrict__ bias,
                __nv_bfloat16* __restrict__ y, int T, int K, int N, int ldx, int ldy,
                int gelu_mode) {
  extern __shared__ __align__(16) uint8_t gsm[];
  const int r0 = split_row(blockIdx.x, N), r1 = split_row(blockIdx.x + 1, N);
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait_primary();
  gemv_rows<EPI, NMAT, TMAX, XF32>(gsm, x, W0, W1, bias, y, T, K, N, ldx, ldy, gelu_mode, r0,
                                   r1);
}

// Row partials of the CTA (its rows x 16 warps x tokens, fp32).
static size_t gemv_part_bytes(int T, int K, int N, int nmat, int grid) {
  (void)K;
  const int64_t rows_max = (static_cast<int64_t>(N) + grid - 1) / grid;
  return static_cast<size_t>(nmat) * rows_max * kGemvWarps * T * 4;
}

// x is kept as fp32 while the CTA's shared memory stays within this (two CTAs per SM fit).
constexpr size_t kGemvTwoCtaSmem = 100 * 1024;

static bool gemv_x_f32(int T, int K, int N, int nmat, int grid) {
  return static_cast<size_t>(T) * K * 4 + gemv_part_bytes(T, K, N, nmat, grid) <= kGemvTwoCtaSmem;
}

size_t gemv_smem_bytes(int T, int K, int N, int nmat, int grid) {
  const size_t xb = static_cast<size_t>(T) * K * (gemv_x_f32(T, K, N, nmat, grid) ? 4 : 2);
  return xb + gemv_part_bytes(T, K, N, nmat, grid);
}

// Two CTAs per SM (each at most half of an SM's registers and threads).
int gemv_grid(int T, int K, int N, int nmat, int sms) {
  (void)T;
  (void)K;
  (void)nmat;
  const int g = sms * kGemvCtasPerSm;
  return g < N ? g : N;
}

template <int EPI, int NMAT, int TMAX, bool XF32>
static cudaError_t gemv_launch_t(const GemvLaunch& L, size_t smem) {
  auto kern = gemv_kernel<EPI, NMAT, TMAX, XF32>;
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

template <bool XF32>
static cudaError_t gemv_dispatch(const GemvLaunch& L, size_t smem) {
  if (L.T == 1) {
    switch (L.epi) {
      case EPI_BIAS: return gemv_launch_t<EPI_BIAS, 1, 1, XF32>(L, smem);
      case EPI_BIAS_GELU: return gemv_launch_t<EPI_BIAS_GELU, 1, 1, XF32>(L, smem);
      case EPI_GEGLU: return gemv_launch_t<EPI_GEGLU, 2, 1, XF32>(L, smem);
    }
  } else {
    switch (L.epi) {
      case EPI_BIAS: return gemv_launch_t<EPI_BIAS, 1, kGemvMaxT, XF32>(L, smem);
      case EPI_BIAS_GELU: return gemv_launch_t<EPI_BIAS_GELU, 1, kGemvMaxT, XF32>(L, smem);
      case EPI_GEGLU: return gemv_launch_t<EPI_GEGLU, 2, kGemvMaxT, XF32>(L, smem);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t gemv_launch(const GemvLaunch& L) {
  const int nmat = L.epi == EPI_GEGLU ? 2 : 1;
  if (L.T < 1 || L.T > kGemvMaxT || L.K % kSeg != 0 || L.grid < 1) return cudaErrorInvalidValue;
  const size_t smem = gemv_smem_bytes(L.T, L.K, L.N, nmat, L.grid);
  if (smem > kGemvMaxSmem) return cudaErrorInvalidValue;
  return gemv_x_f32(L.T, L.K, L.N, nmat, L.grid) ? gemv_dispatch<true>(L, smem)
                                                 : gemv_dispatch<false>(L, smem);
}

}  // namespace fmlp
