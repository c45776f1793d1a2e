// Weight-streaming GEMV for a few tokens (decode): y[t, n] = epi(sum_k x[t, k] W[n, k] (+ b[n])).
//
// At one token the feed-forward block reads every weight once and does one multiply-add per
// weight, so it is bound by HBM bandwidth and by launch latency (ainews.cool fused-MLP
// article, technical deep-dive: batch-1 decode pays one launch per layer and is limited by
// memory traffic). The kernel is built for that:
//   - each CTA owns a contiguous block of weight rows [r0, r1) (balanced to +-1 row), so the
//     bytes it streams form one contiguous range per weight matrix;
//   - one producer warp streams that range through a ring of 16 KB shared-memory slots with
//     1-D bulk async copies (cp.async.bulk, completion counted on an mbarrier), keeping up to
//     eight slots - 128 KB per SM - in flight; no register file is spent on loads in flight;
//   - a slot is 32 segments of 512 bytes (one 16-byte vector per lane, 256 weights of one
//     row); eight compute warps take four segments each, form the dot product with x (held
//     in shared memory) in fp32, reduce it with warp shuffles and store one partial per
//     (row, segment); one thread per (row, token) then adds a row's partials in segment
//     order (deterministic) and applies the epilogue;
//   - with two weight matrices (GeGLU gate and up) both ranges are streamed and the epilogue
//     forms gelu_tanh(g) * u;
//   - programmatic dependent launch: the kernel lets the next kernel launch at once and
//     prefetches its whole weight range into L2 before waiting for the previous kernel, so a
//     layer's weights stream in while the previous layer finishes.
// Every wait is bounded.
#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

constexpr int kGemvComputeWarps = 8;
constexpr int kGemvThreads = (kGemvComputeWarps + 1) * 32;  // + one producer warp
constexpr int kSeg = 256;                                    // weights per segment
constexpr int kSegBytes = kSeg * 2;
constexpr int kSlotSegs = 32;
constexpr int kSlotBytes = kSlotSegs * kSegBytes;            // 16 KB
constexpr int kMaxSlots = 8;
constexpr int kMinSlots = 2;

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
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

struct GemvSmem {
  size_t x_off, part_off, ring_off, bar_off, total;
  int slots;
};

__host__ __device__ inline GemvSmem gemv_layout(int T, int K, int rows_max, int nmat,
                                                size_t budget) {
  GemvSmem L;
  L.x_off = 0;
  const size_t xb = static_cast<size_t>(T) * K * 2;
  L.part_off = (xb + 15) & ~size_t(15);
  const size_t pb = static_cast<size_t>(nmat) * rows_max * (K / kSeg) * T * 4;
  L.ring_off = (L.part_off + pb + 1023) & ~size_t(1023);
  const size_t fixed = L.ring_off + 2 * kMaxSlots * 8 + 1024;
  int slots = kMinSlots;
  if (budget > fixed) {
    const size_t s = (budget - fixed) / kSlotBytes;
    slots = s > kMaxSlots ? kMaxSlots : (s < kMinSlots ? kMinSlots : static_cast<int>(s));
  }
  L.slots = slots;
  L.bar_off = L.ring_off + static_cast<size_t>(slots) * kSlotBytes;
  L.total = L.bar_off + 2 * kMaxSlots * 8 + 1024;  // + alignment slack for the base
  return L;
}

template <int EPI, int NMAT, int TMAX>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ W0,
                const __nv_bfloat16* __restrict__ W1, const __nv_bfloat16* __restrict__ bias,
                __nv_bfloat16* __restrict__ y, int T, int K, int N, int gelu_mode,
                int rows_max, int slots, int* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t gsm_raw[];
  uint8_t* gsm = gsm_raw + ((1024u - (smem_u32(gsm_raw) & 1023u)) & 1023u);
  const GemvSmem Ly = gemv_layout(T, K, rows_max, NMAT, 0);  // offsets only (slots from host)
  const int r0 = static_cast<int>((static_cast<int64_t>(blockIdx.x) * N) / gridDim.x);
  const int r1 = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * N) / gridDim.x);
  const int rows = r1 - r0;
  const int segs = K / kSeg;
  const int per_mat = rows * segs;                                   // segments per matrix
  const int chunks_per_mat = (per_mat + kSlotSegs - 1) / kSlotSegs;
  const int nchunks = NMAT * chunks_per_mat;

  uint4* xs = reinterpret_cast<uint4*>(gsm + Ly.x_off);              // [T][K/8]
  float* part = reinterpret_cast<float*>(gsm + Ly.part_off);         // [mat][row][seg][T]
  uint8_t* ring = gsm + Ly.ring_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(slots) * kSlotBytes);
  uint64_t* empty = full + kMaxSlots;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < slots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGemvComputeWarps);
    }
    fence_mbarrier_init();
    pdl_launch_dependents();
  }
  // Warm L2 with this CTA's weight rows; they are not produced by the previous kernel.
  if (warp == kGemvComputeWarps && lane < NMAT) {
    const __nv_bfloat16* Wm = lane == 0 ? W0 : W1;
    const char* base = reinterpret_cast<const char*>(Wm + static_cast<size_t>(r0) * K);
    const size_t bytes = static_cast<size_t>(rows) * K * 2;
    for (size_t off = 0; off < bytes; off += 65536) {
      const size_t n = bytes - off < 65536 ? bytes - off : 65536;
      prefetch_l2_bulk(base + off, static_cast<uint32_t>(n));
    }
  }
  __syncthreads();
  pdl_wait_primary();

  if (warp == kGemvComputeWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t issued = 0, last_par = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % slots;
        const uint32_t par = static_cast<uint32_t>(c / slots) & 1u;
        if (!mbar_wait(&empty[s], par ^ 1u, status, SITE_GEMV, timeout_ns)) break;
        const int mat = NMAT == 2 ? c / chunks_per_mat : 0;
        const int cm = c - mat * chunks_per_mat;
        const int seg0 = cm * kSlotSegs;
        const int nseg = per_mat - seg0 < kSlotSegs ? per_mat - seg0 : kSlotSegs;
        const __nv_bfloat16* Wm = mat ? W1 : W0;
        const char* src = reinterpret_cast<const char*>(Wm + static_cast<size_t>(r0) * K) +
                          static_cast<size_t>(seg0) * kSegBytes;
        const uint32_t bytes = static_cast<uint32_t>(nseg) * kSegBytes;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load(ring + static_cast<size_t>(s) * kSlotBytes, src, bytes, &full[s]);
        issued |= 1u << s;
        last_par = (last_par & ~(1u << s)) | (par << s);
      }
      // every copy issued must land before the CTA can exit (normally consumed already)
      for (int s = 0; s < slots; ++s)
        if (issued & (1u << s))
          mbar_wait(&full[s], (last_par >> s) & 1u, status, SITE_DRAIN, timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps
    const int xvec = T * (K / 8);
    for (int i = threadIdx.x; i < xvec; i += kGemvComputeWarps * 32)
      xs[i] = __ldg(reinterpret_cast<const uint4*>(x) + i);
    asm volatile("bar.sync 1, %0;" ::"n"(kGemvComputeWarps * 32) : "memory");
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % slots;
      const uint32_t par = static_cast<uint32_t>(c / slots) & 1u;
      const bool ok = mbar_wait(&full[s], par, status, SITE_GEMV, timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int mat = NMAT == 2 ? c / chunks_per_mat : 0;
      const int cm = c - mat * chunks_per_mat;
      const int seg0 = cm * kSlotSegs;
      const uint8_t* slot = ring + static_cast<size_t>(s) * kSlotBytes;
#pragma unroll
      for (int j = warp; j < kSlotSegs; j += kGemvComputeWarps) {
        const int g = seg0 + j;   // segment index within this matrix block
        if (g < per_mat) {        // warp-uniform
          const int row = g / segs, seg = g - row * segs;
          const uint4 wv = *reinterpret_cast<const uint4*>(slot + j * kSegBytes + lane * 16);
          float p[TMAX];
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            p[t] = 0.f;
            if (t < T) p[t] = dot8(wv, xs[t * (K / 8) + seg * (kSeg / 8) + lane]);
          }
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) p[t] += __shfl_xor_sync(0xffffffffu, p[t], o);
          }
          if (lane == 0) {
            const size_t pi = (static_cast<size_t>(mat) * per_mat + row * segs + seg) * T;
#pragma unroll
            for (int t = 0; t < TMAX; ++t)
              if (t < T) part[pi + t] = p[t];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
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
  const int rows_max = static_cast<int>((static_cast<int64_t>(N) + grid - 1) / grid);
  return gemv_layout(T, K, rows_max, nmat, kGemvPreferSmem).total;
}

template <int EPI, int NMAT, int TMAX>
static cudaError_t gemv_launch_t(const GemvLaunch& L, const GemvSmem& lay, int rows_max) {
  auto kern = gemv_kernel<EPI, NMAT, TMAX>;
  static SmemAttrCache cache;
  cudaError_t e =
      set_smem_limit(reinterpret_cast<const void*>(kern), static_cast<int>(lay.total), cache);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = lay.total;
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
                            static_cast<__nv_bfloat16*>(L.y), L.T, L.K, L.N, L.gelu_mode,
                            rows_max, lay.slots, L.status, L.timeout_ns);
}

cudaError_t gemv_launch(const GemvLaunch& L) {
  const int nmat = L.epi == EPI_GEGLU ? 2 : 1;
  if (L.T < 1 || L.T > kGemvMaxT || L.K % kSeg != 0 || L.grid < 1) return cudaErrorInvalidValue;
  const int rows_max = static_cast<int>((static_cast<int64_t>(L.N) + L.grid - 1) / L.grid);
  const GemvSmem lay = gemv_layout(L.T, L.K, rows_max, nmat, kGemvPreferSmem);
  if (lay.total > kGemvMaxSmem) return cudaErrorInvalidValue;
  if (L.T == 1) {
    switch (L.epi) {
      case EPI_BIAS: return gemv_launch_t<EPI_BIAS, 1, 1>(L, lay, rows_max);
      case EPI_BIAS_GELU: return gemv_launch_t<EPI_BIAS_GELU, 1, 1>(L, lay, rows_max);
      case EPI_GEGLU: return gemv_launch_t<EPI_GEGLU, 2, 1>(L, lay, rows_max);
    }
  } else {
    switch (L.epi) {
      case EPI_BIAS: return gemv_launch_t<EPI_BIAS, 1, kGemvMaxT>(L, lay, rows_max);
      case EPI_BIAS_GELU: return gemv_launch_t<EPI_BIAS_GELU, 1, kGemvMaxT>(L, lay, rows_max);
      case EPI_GEGLU: return gemv_launch_t<EPI_GEGLU, 2, kGemvMaxT>(L, lay, rows_max);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace fmlp
