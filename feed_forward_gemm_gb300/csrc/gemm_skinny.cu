// tcgen05 GEMM for few tokens (2..128): y[T, N] = epi(x[T, K] W[N, K]^T), weights as the M side.
//
// With T <= 128 the usual tiling (128 token rows per tile) leaves most of the MMA's M rows
// padding and, worse, has only N / BN tiles to spread over the SMs, so a few dozen SMs stream
// all the weights. At these sizes the block is bound by reading the weights once ("ainews.cool
// fused-MLP article", technical deep-dive: small-batch inference is limited by memory
// traffic and launches), so this kernel turns the product around and splits it along K:
//   - the MMA computes D[n, t] = sum_k W[n, k] x[t, k]: A = 128 weight rows (K-major, the
//     nn.Linear layout as stored), B = the T tokens padded to Tpad (a multiple of 32, rows past
//     T read as zeros by TMA), M = 128, N = Tpad, K = 16 per instruction; every byte of each
//     16 KB A stage is a weight;
//   - a weight tile of R rows (R <= 128, a multiple of 4) is cut into S K slices (S = 1, 2, 4
//     or 8) computed by the S CTAs of one thread-block cluster, so tiles * S CTAs stream the
//     weights at once. R is chosen so that tiles * S fills the SMs: a 4096-row layer takes 38
//     tiles of 108 rows x 4 slices = 152 CTAs, where 128-row tiles left 24 of 152 SMs idle.
//     TMA loads R rows; the MMA still runs M = 128, and its rows past R (whatever shared
//     memory follows the tile) are never read back;
//   - CTA r owns rows [r rr, (r+1) rr) of the tile's R (rr = R / S rounded up to 4). Once
//     every CTA of the cluster has finished its MMAs (a cluster barrier: every stage ring is
//     free), each CTA reads its fp32 slice D_s out of TMEM and pushes each row's T token
//     values straight into the owning CTA's ring with distributed-shared-memory stores
//     (fire-and-forget; only the T real tokens, not the padding); after a second cluster
//     barrier the owner adds the S slices of its rows from its own shared memory in slice
//     order s = 0..S-1 (the same order on every run), applies the epilogue (bias, GELU/ReLU,
//     or gelu_tanh(g)*u for the GeGLU gate/up pair, whose two accumulators share the B tile)
//     and writes y[t, n]. (Copying the slice to the CTA's own shared memory and pulling the S
//     slices with remote loads instead took 1 us at 4 tokens and 3.5 us at 128: those loads
//     wait a full round trip each.)
// No global scratch, no atomics, no CTA waiting on another outside the cluster barrier,
// which the hardware provides (the CTAs of a cluster are co-scheduled).
//
// Warp roles (one CTA per SM, 6 warps): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer (one thread), warps 2-5 move the accumulator from TMEM to shared memory; all six
// warps share the cluster reduction. All mbarrier waits are bounded; every thread reaches both
// cluster barriers whatever happens, so a timeout unwinds without a hang.
#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

namespace {

constexpr int kSkThreads = 192;
constexpr int kSkBK = 64;                   // K per stage: one 128-byte swizzle row
constexpr int kSkRows = 128;                // weight rows per tile (MMA M)
constexpr int kSkA = kSkRows * kSkBK * 2;   // 16 KB of weights per matrix per stage

__device__ __forceinline__ void st_dsmem_f32(uint32_t cluster_addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}

__device__ __forceinline__ float4 lds_f4_local(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

template <int EPI>
__device__ __forceinline__ float skinny_out(float a0, float a1, float b, int gelu_mode) {
  if (EPI == EPI_GEGLU) return gelu_tanh_f(a0) * a1;
  const float z = a0 + b;
  return EPI == EPI_BIAS_GELU ? gelu_f(z, gelu_mode) : z;
}

}  // namespace

// NMAT = 2: GeGLU gate/up (W0 = Wg, W1 = Wu), two accumulators of Tpad columns each.
template <int EPI, int NMAT>
__global__ void __launch_bounds__(kSkThreads, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW0,
                       const __grid_constant__ CUtensorMap tmW1,
                       const __grid_constant__ CUtensorMap tmX,
                       const __nv_bfloat16* __restrict__ bias, __nv_bfloat16* __restrict__ y,
                       int T, int N, int K, int ldy, int Tpad, int R, int stages, int gelu_mode,
                       int* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int b_bytes = Tpad * kSkBK * 2;
  const int stage_bytes = NMAT * kSkA + b_bytes;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + stages * stage_bytes);
  uint64_t* empty = full + stages;
  uint64_t* tfull = empty + stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  // this CTA's rows of the bias (at most 128), fetched while the weights stream
  float* bias_s = reinterpret_cast<float*>(tmem_slot + 4);
  // after the main loop the ring receives the slices of this CTA's rows: [S][mat][Tpad][rr] fp32
  float* part = reinterpret_cast<float*>(ring);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = static_cast<int>(cluster_nctarank());   // K slices of the tile
  const int s = static_cast<int>(cluster_ctarank());
  const int tile = blockIdx.x / S;
  const int n0 = tile * R;
  // bytes one stage receives: R rows of each weight matrix and the Tpad token rows
  const uint32_t tx_bytes = static_cast<uint32_t>(NMAT * R * kSkBK * 2 + b_bytes);
  const int num_kb = (K + kSkBK - 1) / kSkBK;
  const int kb0 = s * num_kb / S, kb1 = (s + 1) * num_kb / S;
  const uint32_t tmem_cols = NMAT * Tpad <= 32 ? 32u : (NMAT * Tpad <= 64 ? 64u
                             : (NMAT * Tpad <= 128 ? 128u : 256u));

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmW0);
    if (NMAT == 2) prefetch_tmap(&tmW1);
    prefetch_tmap(&tmX);
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  pdl_wait_primary();
  if (threadIdx.x == 0) pdl_launch_dependents();

  bool tfull_ok = true;   // the epilogue warps' wait for the accumulators
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int kb = kb0;
      for (; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, status, SITE_PRODUCER_EMPTY, timeout_ns)) break;
        uint8_t* st = ring + stage * stage_bytes;
        mbar_arrive_expect_tx(&full[stage], tx_bytes);
        tma_load_2d(st, &tmW0, &full[stage], kb * kSkBK, n0);
        if (NMAT == 2) tma_load_2d(st + kSkA, &tmW1, &full[stage], kb * kSkBK, n0);
        tma_load_2d(st + NMAT * kSkA, &tmX, &full[stage], kb * kSkBK, 0);
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kSkRows, static_cast<uint32_t>(Tpad));
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, status, SITE_MMA_FULL, timeout_ns)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + stage * stage_bytes);
        const uint64_t b_desc = sdesc_kmajor_sw128(a_addr + NMAT * kSkA);
#pragma unroll
        for (int mat = 0; mat < NMAT; ++mat) {
          const uint64_t a_desc = sdesc_kmajor_sw128(a_addr + mat * kSkA);
#pragma unroll
          for (int kk = 0; kk < kSkBK / 16; ++kk)
            tc_mma_bf16(tmem_base + static_cast<uint32_t>(mat * Tpad), a_desc + 2u * kk,
                        b_desc + 2u * kk, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
        }
        tc_commit(&empty[stage]);
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      tc_commit(tfull);   // fires once every MMA issued above has completed
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue warps
    // the bias of the rows this CTA finishes, while the weights stream (read in the tail it
    // cost a full memory round trip per output)
    if (EPI != EPI_GEGLU) {
      const int rr = (R + 4 * S - 1) / (4 * S) * 4;
      for (int i = threadIdx.x - 64; i < rr; i += kSkThreads - 64) {
        const int n = n0 + s * rr + i;
        bias_s[i] = (bias != nullptr && s * rr + i < R && n < N) ? __bfloat162float(bias[n]) : 0.f;
      }
    }
    tfull_ok = mbar_wait(tfull, 0, status, SITE_EPI_TMEM_FULL, timeout_ns);
    __syncwarp();
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // every CTA's MMAs are done: every stage ring may take the slices

  // ------------------------------------------------------------------ push the slices
  // Slice s of row `row` goes to the owner of the row, into its ring at
  // recv[s][mat][t][lr] (lr = row - owner rr): [S][NMAT][Tpad][rr] fp32. Rows are contiguous,
  // so a warp's 32 rows go out as 128 contiguous bytes per token (16-byte vectors per thread,
  // tokens contiguous, were slower: a warp's lanes then hit one shared-memory bank).
  const int rr = (R + 4 * S - 1) / (4 * S) * 4;
  const uint32_t recv_addr = smem_u32(part);
  if (warp >= 2 && __all_sync(0xffffffffu, tfull_ok)) {
    const int wq = warp & 3;   // this warp may read TMEM lanes [32 wq, 32 wq + 32)
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(wq * 32) << 16);
    const int row = wq * 32 + lane;
    const int owner = row < R ? row / rr : 0;
    const int lr = row - owner * rr;
    const uint32_t dst0 = mapa_shared(recv_addr, static_cast<uint32_t>(owner));
    for (int mat = 0; mat < NMAT; ++mat) {
      for (int c = 0; c < T; c += 32) {
        uint32_t a[32];
        tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(mat * Tpad + c), a);
        tmem_ld_wait();
        if (row < R) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c + j < T) {
              const int idx = ((s * NMAT + mat) * Tpad + c + j) * rr + lr;
              st_dsmem_f32(dst0 + static_cast<uint32_t>(idx) * 4u, __uint_as_float(a[j]));
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  cluster_sync();   // every slice is in its owner's shared memory

  // ------------------------------------------------------------------ owner reduction
  // CTA s finishes its rows for every token, four consecutive rows per thread: the S slices
  // of the four rows (16-byte loads from this CTA's own shared memory) are added in slice
  // order q = 0..S-1, the same order for every element and every run. Consecutive threads
  // take consecutive row groups, so the writes of y[t, n0 + row .. + 3] are contiguous
  // 8-byte stores.
  {
    const int r_lo = s * rr < R ? s * rr : R;
    const int r_hi = r_lo + rr < R ? r_lo + rr : R;
    const int rg = (r_hi - r_lo) / 4;   // R is a multiple of 4
    for (int e = threadIdx.x; e < rg * T; e += kSkThreads) {
      const int t = e / rg;
      const int lr = (e - t * rg) * 4;
      const int n = n0 + r_lo + lr;
      if (n >= N) continue;
      float4 acc[NMAT];
#pragma unroll
      for (int mat = 0; mat < NMAT; ++mat) {
        acc[mat] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (q < S) {
            const int idx = ((q * NMAT + mat) * Tpad + t) * rr + lr;
            const float4 v = lds_f4_local(recv_addr + static_cast<uint32_t>(idx) * 4u);
            acc[mat].x += v.x;
            acc[mat].y += v.y;
            acc[mat].z += v.z;
            acc[mat].w += v.w;
          }
        }
      }
      const bool epb = EPI != EPI_GEGLU;
      const float o0 = skinny_out<EPI>(acc[0].x, acc[NMAT - 1].x, epb ? bias_s[lr] : 0.f, gelu_mode);
      const float o1 = skinny_out<EPI>(acc[0].y, acc[NMAT - 1].y, epb ? bias_s[lr + 1] : 0.f, gelu_mode);
      const float o2 = skinny_out<EPI>(acc[0].z, acc[NMAT - 1].z, epb ? bias_s[lr + 2] : 0.f, gelu_mode);
      const float o3 = skinny_out<EPI>(acc[0].w, acc[NMAT - 1].w, epb ? bias_s[lr + 3] : 0.f, gelu_mode);
      __nv_bfloat16* yr = y + static_cast<size_t>(t) * ldy + n;
      if (n + 3 < N) {
        uint2 pk;
        pk.x = pack_bf16x2(o0, o1);
        pk.y = pack_bf16x2(o2, o3);
        *reinterpret_cast<uint2*>(yr) = pk;
      } else {
        yr[0] = __float2bfloat16_rn(o0);
        if (n + 1 < N) yr[1] = __float2bfloat16_rn(o1);
        if (n + 2 < N) yr[2] = __float2bfloat16_rn(o2);
      }
    }
  }
  // no other CTA touches this one's shared memory after the second barrier: no third one
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// Shared memory of one CTA: the stage ring (also the slice buffer afterwards), the mbarriers,
// the TMEM address slot and the bias of up to 128 rows, plus 1 KB for the 1024-byte alignment
// of the ring.
static int skinny_smem(int nmat, int tpad, int stages) {
  const int stage_bytes = nmat * kSkA + tpad * kSkBK * 2;
  return 1024 + stages * stage_bytes + (2 * stages + 1) * 8 + 16 + 128 * 4;
}

// Pipeline stages for nmat weight matrices and tpad token rows (0: does not fit): up to 192 KB
// of ring. (A ring of about 100 KB, which leaves room for the next kernel's CTA on the SM so
// that it can fetch its weights before the dependency wait, measured slower: 24.2 and 29.5 us
// against 23.3 and 26.6 for the 4096-wide MLP at 64 and 128 tokens; fetching the weights
// early with the full ring was slower too.) The ring must also take the slices of a CTA's
// rows, [S][nmat][tpad][rr] fp32 with S rr <= 128.
static int gemm_skinny_stages(int nmat, int tpad) {
  const int stage_bytes = nmat * kSkA + tpad * kSkBK * 2;
  int stages = (192 * 1024) / stage_bytes;
  if (stages > 8) stages = 8;
  while (stages * stage_bytes < nmat * tpad * kSkRows * 4) ++stages;
  return skinny_smem(nmat, tpad, stages) <= 232448 ? stages : 0;
}

template <int EPI, int NMAT>
static cudaError_t launch_skinny_t(const SkinnyLaunch& L) {
  auto kern = gemm_skinny_kernel<EPI, NMAT>;
  const int stages = gemm_skinny_stages(NMAT, L.tpad);
  if (stages == 0) return cudaErrorInvalidValue;
  const int smem = skinny_smem(NMAT, L.tpad, stages);
  static SmemAttrCache cache;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem, cache);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.tiles * L.split, 1, 1);
  cfg.blockDim = dim3(kSkThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = L.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = L.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, L.tmW0, L.tmW1, L.tmX,
                            static_cast<const __nv_bfloat16*>(L.bias),
                            static_cast<__nv_bfloat16*>(L.y), L.T, L.N, L.K, L.ldy, L.tpad, L.rows,
                            stages, L.gelu_mode, L.status, L.timeout_ns);
}

cudaError_t gemm_skinny_max_clusters(int split, int* clusters) {
  auto kern = gemm_skinny_kernel<EPI_BIAS, 1>;
  // one CTA per SM (a launch never uses more: the second CTA slot is for the next kernel)
  const int smem = 200 * 1024;
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, 1, 1);
  cfg.blockDim = dim3(kSkThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, kern, &cfg);
}

cudaError_t gemm_skinny_launch(const SkinnyLaunch& L) {
  const int num_kb = (L.K + kSkBK - 1) / kSkBK;
  if (L.T < 1 || L.T > kSkinnyMaxT || L.tpad < L.T || L.tpad % 32 != 0 || L.tpad > kSkinnyMaxT ||
      L.rows < 4 || L.rows > kSkRows || L.rows % 4 != 0 ||
      L.tiles < 1 || static_cast<int64_t>(L.tiles) * L.rows < L.N ||
      (L.split != 1 && L.split != 2 && L.split != 4 && L.split != 8) || L.split > num_kb)
    return cudaErrorInvalidValue;
  switch (L.epi) {
    case EPI_BIAS: return launch_skinny_t<EPI_BIAS, 1>(L);
    case EPI_BIAS_GELU: return launch_skinny_t<EPI_BIAS_GELU, 1>(L);
    case EPI_GEGLU: return launch_skinny_t<EPI_GEGLU, 2>(L);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fmlp
