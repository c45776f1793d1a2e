// The whole feed-forward block in one kernel, for small model widths (D, Dout <= 256).
//
// One CTA owns 128 tokens. Their x tile stays in shared memory for the whole block; the
// hidden dimension is walked in chunks of 64. GeGLU block:
//   g|u  = x Wg[c]^T | x Wu[c]^T          one tcgen05.mma with N = 128 (gate rows, up rows)
//   m[c] = bf16(gelu_tanh(g) * u)           epilogue warps, written straight into shared
//                                           memory in the 128B-swizzled K-major layout the
//                                           next MMA reads as its A operand
//   y   += m[c] Wd[:, c]^T                  tcgen05.mma with N = D, accumulated in TMEM
// Linear -> activation -> Linear with biases:
//   z    = x W1[c]^T                        one tcgen05.mma with N = 64
//   h[c] = bf16(act(z + b1[c]))             the same epilogue path, GELU (tanh or erf) or ReLU
//   y   += h[c] W2[:, c]^T                  N = Dout; y = bf16(y + b2) at the end
// and only y is written to HBM: the intermediate never leaves the chip. This is the single-
// launch form of the feed-forward block (ainews.cool fused-MLP article, technical deep-dive:
// load x once, W1 x + b1, the activation and W2 h + b2 in one kernel, write only the output),
// also applied to the GeGLU block of "Profiling in PyTorch (Part 2): From nn.Linear to a Fused
// MLP", section "Stacking three Linears: the MLP".
//
// Warps 0-3 run the epilogues (each its own 32 TMEM lanes); warp 4 owns TMEM and one of its
// threads issues every TMA load and MMA. Weight loads of the next chunk overlap the current
// chunk's epilogue. Every wait is bounded.
#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

constexpr int kSmallThreads = 160;
constexpr int kPanel = 128 * 128;  // 128 rows x 64 bf16

int ffn_small_smem_bytes(int D, int Dout) {
  const int P = (D + 63) / 64;
  const int wd = ((Dout * 128 + 1023) / 1024) * 1024;
  return 1024 + P * kPanel /*x*/ + P * kPanel /*gate|up weights*/ + wd + kPanel /*m*/ +
         4 * 4096 /*staging*/ + 128 /*barriers*/;
}

// MLP = false: the GeGLU block (tmWg, tmWu gate and up, tmWd down, no biases);
// MLP = true: Linear -> act -> Linear (tmWg = W1, tmWu unused, tmWd = W2, biases b1, b2).
template <bool MLP>
__global__ void __launch_bounds__(kSmallThreads, 1)
    ffn_small_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmWg,
                     const __grid_constant__ CUtensorMap tmWu,
                     const __grid_constant__ CUtensorMap tmWd,
                     const __grid_constant__ CUtensorMap tmY, const __nv_bfloat16* __restrict__ b1,
                     const __nv_bfloat16* __restrict__ b2, int T, int D, int H, int Dout,
                     int gelu_mode, int* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int P = (D + 63) / 64;
  const int wd_bytes = ((Dout * 128 + 1023) / 1024) * 1024;
  uint8_t* x_s = smem;
  uint8_t* gu_s = x_s + P * kPanel;
  uint8_t* wd_s = gu_s + P * kPanel;
  uint8_t* m_s = wd_s + wd_bytes;
  uint8_t* stg_all = m_s + kPanel;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg_all + 4 * 4096);
  uint64_t* bx = bars + 0;     // x tile landed
  uint64_t* bgw = bars + 1;    // gate/up weight chunk landed
  uint64_t* bwd = bars + 2;    // down weight chunk landed
  uint64_t* bgu = bars + 3;    // gate/up MMAs done
  uint64_t* bdn = bars + 4;    // down MMAs done
  uint64_t* bm = bars + 5;     // m chunk written by the epilogue warps
  uint64_t* bdr = bars + 6;    // drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128;
  const int nch = (H + 63) / 64;
  constexpr uint32_t kGuCol = 0, kYCol = 256;

  if (threadIdx.x == 128) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmWg);
    if (!MLP) prefetch_tmap(&tmWu);
    prefetch_tmap(&tmWd);
    prefetch_tmap(&tmY);
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
    mbar_init(bm, 128);
    mbar_init(bdr, 1);
    fence_mbarrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_primary();
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == 4) {
    if (lane == 0) {
      auto load_gu = [&](int c) {
        mbar_arrive_expect_tx(bgw, P * (MLP ? kPanel / 2 : kPanel));
        for (int p = 0; p < P; ++p) {
          tma_load_2d(gu_s + p * kPanel, &tmWg, bgw, p * 64, c * 64);
          if (!MLP) tma_load_2d(gu_s + p * kPanel + kPanel / 2, &tmWu, bgw, p * 64, c * 64);
        }
      };
      auto load_wd = [&](int c) {
        mbar_arrive_expect_tx(bwd, Dout * 128);
        tma_load_2d(wd_s, &tmWd, bwd, c * 64, 0);
      };
      mbar_arrive_expect_tx(bx, P * kPanel);
      for (int p = 0; p < P; ++p) tma_load_2d(x_s + p * kPanel, &tmX, bx, p * 64, m0);
      load_gu(0);
      load_wd(0);
      bool ok = mbar_wait(bx, 0, status, SITE_SMALL, timeout_ns);
      // loads issued but not yet observed complete (for the drain on an early exit)
      int gw_pending = 1, wd_pending = 1;
      uint32_t gw_par = 0, wd_par = 0;
      const uint32_t idesc_gu = idesc_bf16_f32(128, MLP ? 64 : 128);
      const uint32_t idesc_dn = idesc_bf16_f32(128, static_cast<uint32_t>(Dout));
      const int ksteps = (D + 15) / 16;
      for (int c = 0; c < nch && ok; ++c) {
        const uint32_t par = c & 1;
        if (!(ok = mbar_wait(bgw, par, status, SITE_SMALL, timeout_ns))) break;
        gw_pending = 0;
        tc_fence_after();
        for (int s = 0; s < ksteps; ++s) {
          const int p = s >> 2, kk = s & 3;
          const uint64_t a = sdesc_kmajor_sw128(smem_u32(x_s + p * kPanel)) + 2u * kk;
          const uint64_t b = sdesc_kmajor_sw128(smem_u32(gu_s + p * kPanel)) + 2u * kk;
          tc_mma_bf16(tmem + kGuCol, a, b, idesc_gu, s > 0 ? 1u : 0u);
        }
        tc_commit(bgu);
        if (!(ok = mbar_wait(bgu, par, status, SITE_SMALL, timeout_ns))) break;
        if (c + 1 < nch) {
          load_gu(c + 1);
          gw_pending = 1;
          gw_par = (c + 1) & 1;
        }
        if (!(ok = mbar_wait(bm, par, status, SITE_SMALL, timeout_ns))) break;
        if (!(ok = mbar_wait(bwd, par, status, SITE_SMALL, timeout_ns))) break;
        wd_pending = 0;
        tc_fence_after();
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t a = sdesc_kmajor_sw128(smem_u32(m_s)) + 2u * kk;
          const uint64_t b = sdesc_kmajor_sw128(smem_u32(wd_s)) + 2u * kk;
          tc_mma_bf16(tmem + kYCol, a, b, idesc_dn, (c | kk) != 0 ? 1u : 0u);
        }
        tc_commit(bdn);
        if (!(ok = mbar_wait(bdn, par, status, SITE_SMALL, timeout_ns))) break;
        if (c + 1 < nch) {
          load_wd(c + 1);
          wd_pending = 1;
          wd_par = (c + 1) & 1;
        }
      }
      // drain: outstanding MMAs and loads must finish before the CTA releases its memory
      tc_commit(bdr);
      mbar_wait(bdr, 0, status, SITE_DRAIN, timeout_ns);
      if (gw_pending) mbar_wait(bgw, gw_par, status, SITE_DRAIN, timeout_ns);
      if (wd_pending) mbar_wait(bwd, wd_par, status, SITE_DRAIN, timeout_ns);
    }
    __syncwarp();
  } else {
    // epilogue warps 0..3: warp q owns TMEM lanes / tile rows [32q, 32q+32)
    const int row = warp * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = true;
    for (int c = 0; c < nch; ++c) {
      ok = mbar_wait(bgu, c & 1, status, SITE_SMALL, timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t g[32], u[32];
        tmem_ld_32x32b_x32(t_lane + kGuCol + h * 32, g);
        if (!MLP) tmem_ld_32x32b_x32(t_lane + kGuCol + 64 + h * 32, u);
        tmem_ld_wait();
        if (MLP) {
          // h = act(z + b1): the bias of each of these 32 hidden units (0 past H, where W1's
          // rows read as zeros, so the unit's output is act(0) = 0)
          const int n0 = c * 64 + h * 32;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float bias = (b1 != nullptr && n0 + i < H) ? __bfloat162float(b1[n0 + i]) : 0.f;
            g[i] = __float_as_uint(gelu_f(__uint_as_float(g[i]) + bias, gelu_mode));
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = q * 8 + e * 2;
            if (MLP)
              pk[e] = pack_bf16x2(__uint_as_float(g[i]), __uint_as_float(g[i + 1]));
            else
              pk[e] = pack_bf16x2(gelu_tanh_f(__uint_as_float(g[i])) * __uint_as_float(u[i]),
                                  gelu_tanh_f(__uint_as_float(g[i + 1])) * __uint_as_float(u[i + 1]));
          }
          const int j = h * 4 + q;
          const uint32_t addr = smem_u32(m_s) + static_cast<uint32_t>(row * 128) +
                                static_cast<uint32_t>((j ^ (row & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[0]),
                       "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                       : "memory");
        }
      }
      fence_proxy_async_smem();   // m is read next by the tensor core (async proxy)
      tc_fence_before();
      mbar_arrive(bm);
    }
    if (ok) {
      ok = mbar_wait(bdn, (nch - 1) & 1, status, SITE_SMALL, timeout_ns);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        uint8_t* stg = stg_all + warp * 4096;
        const int row0 = m0 + warp * 32;
        const int PO = (Dout + 63) / 64;
        for (int ch = 0; ch < PO; ++ch) {
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t a[32];
            tmem_ld_32x32b_x32(t_lane + kYCol + ch * 64 + h * 32, a);
            tmem_ld_wait();
            if (MLP && b2 != nullptr) {
              const int n0 = ch * 64 + h * 32;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (n0 + i < Dout)
                  a[i] = __float_as_uint(__uint_as_float(a[i]) + __bfloat162float(b2[n0 + i]));
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t p0 = pack_bf16x2(__uint_as_float(a[q * 8 + 0]), __uint_as_float(a[q * 8 + 1]));
              const uint32_t p1 = pack_bf16x2(__uint_as_float(a[q * 8 + 2]), __uint_as_float(a[q * 8 + 3]));
              const uint32_t p2 = pack_bf16x2(__uint_as_float(a[q * 8 + 4]), __uint_as_float(a[q * 8 + 5]));
              const uint32_t p3 = pack_bf16x2(__uint_as_float(a[q * 8 + 6]), __uint_as_float(a[q * 8 + 7]));
              const int j = h * 4 + q;
              const uint32_t addr = smem_u32(stg) + static_cast<uint32_t>(lane * 128) +
                                    static_cast<uint32_t>((j ^ (lane & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(p0),
                           "r"(p1), "r"(p2), "r"(p3)
                           : "memory");
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (row0 < T) tma_store_2d(&tmY, stg, ch * 64, row0);
            bulk_commit_group();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool MLP>
static cudaError_t ffn_small_launch_t(const SmallLaunch& L) {
  const int smem = ffn_small_smem_bytes(L.D, L.Dout);
  static SmemAttrCache cache;
  auto kern = ffn_small_kernel<MLP>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem, cache);
  if (e != cudaSuccess) return e;
  const int grid = (L.T + 127) / 128;
  kern<<<grid, kSmallThreads, smem, L.stream>>>(
      L.tmX, L.tmWg, L.tmWu, L.tmWd, L.tmY, static_cast<const __nv_bfloat16*>(L.b1),
      static_cast<const __nv_bfloat16*>(L.b2), L.T, L.D, L.H, L.Dout, L.gelu_mode, L.status,
      L.timeout_ns);
  return cudaGetLastError();
}

cudaError_t ffn_small_launch(const SmallLaunch& L) {
  if (L.D < 8 || L.D > kSmallMaxD || L.Dout < 16 || L.Dout > kSmallMaxD || L.Dout % 16 != 0 ||
      L.H < 1 || L.T < 1)
    return cudaErrorInvalidValue;
  return L.mlp ? ffn_small_launch_t<true>(L) : ffn_small_launch_t<false>(L);
}

}  // namespace fmlp
