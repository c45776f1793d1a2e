// Persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
//   D[M, N] = A[M, K] * B[N, K]^T     A = activations (x or the intermediate), row-major
//                                     B = weights in nn.Linear layout [out, in], row-major
//
// Both operands are K-major, which is exactly how nn.Linear stores its weight: the
// transpose in y = x @ W^T is never materialised ("Profiling in PyTorch (Part 2): From
// nn.Linear to a Fused MLP", section "Where did the transpose go? Kernel layouts and
// pre-ops": the GEMM reads the weight in transposed order, the `tn` layout). The epilogue
// runs on the fp32 accumulator before the single write to HBM (section "Why are there no
// separate mul and add kernels?"):
//   EPI_BIAS       y = bf16(acc + b)                 (b optional)
//   EPI_BIAS_GELU  h = bf16(gelu(acc + b))           (first Linear of Linear->GELU->Linear)
//   EPI_GEGLU      m = bf16(gelu_tanh(acc_g) * acc_u) (gate and up of section "Stacking
//                  three Linears: the MLP", computed together for one token block)
//
// Structure (one CTA per SM, 6 warps):
//   warp 0     TMA producer: A tile 128x64 and B tile BNx64 per stage into a ring of
//              128B-swizzled shared-memory stages (mbarrier full/empty pairs).
//   warp 1     TMEM owner and MMA issuer: one thread issues tcgen05.mma (M=128, N=BN,
//              K=16) x4 per stage into one of two TMEM accumulators (double buffer), and
//              tcgen05.commit releases the stage / signals the epilogue.
//   warps 2-5  epilogue: tcgen05.ld the accumulator (each warp its 32 TMEM lanes), apply the
//              epilogue in fp32, round once to bf16, stage 32x64 tiles in swizzled shared
//              memory and write them with TMA stores, then release the accumulator.
// For GeGLU the B stage holds the Wg rows of the tile followed by the matching Wu rows, so
// one MMA with N = BN produces gate in accumulator columns [0, BN/2) and up in [BN/2, BN):
// both share the A tile and the same instruction.
// All waits are bounded; on expiry the kernel records a status code and unwinds.
//
// GROUPED (the mixture-of-experts block): the rows of A are grouped by expert, rows
// [offsets[e], offsets[e+1]) belonging to expert e, whose weights are slice e of a 3-D tensor
// [E, N, K]. One launch serves every expert: each CTA reads the offsets after the dependency
// wait (a router kernel may have written them just before), counts each group's 128-row
// tiles, and walks each group's tiles row tile fastest, so the CTAs in flight share one
// weight panel of the expert and its few token rows in L2. A loads start at the group's
// row; B loads take the expert's slice through a 3-D tensor map; the epilogue stores rows
// directly and skips the rows past the group's end, which the 128-row tile computed
// from the next group's tokens.
#include "activation.cuh"
#include "gemm_epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

constexpr int kBM = 128;
constexpr int kBK = 64;                 // 64 bf16 = 128 bytes = one swizzle row
constexpr int kThreads = 32 * (2 + kEpiWarps);   // producer, MMA issuer, epilogue warps
constexpr int kRasterGroup = 16;        // M tiles per raster group (L2 reuse of weights)

template <int BN, int EPI>
struct Cfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE_BYTES;
  static constexpr int BN_OUT = EPI == EPI_GEGLU ? BN / 2 : BN;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8 + 16;
  static constexpr int SMEM_BYTES =
      1024 + STAGES * STAGE_BYTES + kEpiWarps * kStgPerWarp * kStgBytes + BAR_BYTES;
  static_assert(BN == 64 || BN == 128 || BN == 256, "MMA N");
  static_assert(EPI != EPI_GEGLU || BN >= 128, "GeGLU needs 64-column output chunks");
  static_assert(BN_OUT % 64 == 0, "output chunks are 64 columns");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "1024-byte aligned tiles");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int& tm, int& tn) {
  const int per_group = kRasterGroup * num_n;
  const int g = t / per_group;
  const int first_m = g * kRasterGroup;
  const int gm = min(num_m - first_m, kRasterGroup);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

// Tile t of a GROUPED launch (s_tp: prefix of the groups' tile counts) -> expert e, first row,
// rows in the tile, N tile; within a group the row tile runs fastest.
__device__ __forceinline__ void group_tile(int t, const int* s_off, const int* s_tp, int& e,
                                           int& row0, int& rows, int& tn) {
  e = 0;
  while (s_tp[e + 1] <= t) ++e;
  const int local = t - s_tp[e];
  const int mt_e = (s_off[e + 1] - s_off[e] + kBM - 1) / kBM;
  tn = local / mt_e;
  row0 = s_off[e] + (local - tn * mt_e) * kBM;
  rows = min(kBM, s_off[e + 1] - row0);
}

// B_MN: the weights come as Wt [K, N_out] (N contiguous, the transposed `nn` layout), loaded
// as BN / 64 boxes of 64 N columns x 64 K rows and read by the MMA as an MN-major operand;
// no transposed copy is made ("Profiling in PyTorch (Part 2)", section "Where did the
// transpose go? Kernel layouts and pre-ops": the layout is the kernel's choice of operand
// major-ness).
template <int BN, int EPI, bool GROUPED, bool B_MN = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmY, const __nv_bfloat16* __restrict__ bias,
                   int M, int N_out, int K, int gelu_mode, int* status, uint64_t timeout_ns,
                   const int* __restrict__ offsets, int E, __nv_bfloat16* __restrict__ ydir,
                   int ldy) {
  using C = Cfg<BN, EPI>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  uint8_t* stg_all = smem + STAGES * C::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(stg_all + kEpiWarps * kStgPerWarp * kStgBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (EPI == EPI_GEGLU) prefetch_tmap(&tmB1);
    prefetch_tmap(&tmY);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps * 32);
    }
    mbar_init(drain, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Inputs may be produced by the previous kernel on the stream (programmatic launch).
  pdl_wait_primary();
  if (threadIdx.x == 0) pdl_launch_dependents();

  const int num_m = (M + kBM - 1) / kBM;
  const int num_n = (N_out + C::BN_OUT - 1) / C::BN_OUT;
  const int num_kb = (K + kBK - 1) / kBK;
  // GROUPED: token offsets and the prefix of the groups' tile counts, in the (unused) staging
  // area
  int* s_off = reinterpret_cast<int*>(stg_all);
  int* s_tp = s_off + (kMoeMaxExperts + 1);
  int grouped_tiles = 0;
  if constexpr (GROUPED) {
    for (int i = threadIdx.x; i <= E; i += kThreads) s_off[i] = min(max(__ldcg(offsets + i), 0), M);
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0;
      s_tp[0] = 0;
      for (int g = 0; g < E; ++g) {
        s_off[g + 1] = max(s_off[g + 1], s_off[g]);   // a falling offset makes the group empty
        acc += (s_off[g + 1] - s_off[g] + kBM - 1) / kBM * num_n;
        s_tp[g + 1] = acc;
      }
    }
    __syncthreads();
    grouped_tiles = s_tp[E];
  }
  const int num_tiles = GROUPED ? grouped_tiles : num_m * num_n;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_phase_mask = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int tm = 0, tn, ge = 0, grow = 0, grows = 0;
        if constexpr (GROUPED)
          group_tile(t, s_off, s_tp, ge, grow, grows, tn);
        else
          tile_coords(t, num_m, num_n, tm, tn);
        const int a_row = GROUPED ? grow : tm * kBM;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, status, SITE_PRODUCER_EMPTY, timeout_ns)) {
            ok = false;
            break;
          }
          uint8_t* sA = stages + stage * C::STAGE_BYTES;
          uint8_t* sB = sA + C::A_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(sA, &tmA, &full[stage], kb * kBK, a_row);
          if constexpr (GROUPED) {
            if (EPI == EPI_GEGLU) {
              tma_load_3d(sB, &tmB0, &full[stage], kb * kBK, tn * (BN / 2), ge);
              tma_load_3d(sB + (BN / 2) * 128, &tmB1, &full[stage], kb * kBK, tn * (BN / 2), ge);
            } else {
              tma_load_3d(sB, &tmB0, &full[stage], kb * kBK, tn * BN, ge);
            }
          } else if (B_MN) {
            // Wt [K, N]: box j holds N columns [tn BN + 64 j, + 64) of K rows [kb 64, + 64)
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(sB + j * (64 * kBK * 2), &tmB0, &full[stage], tn * BN + 64 * j,
                          kb * kBK);
          } else if (EPI == EPI_GEGLU) {
            tma_load_2d(sB, &tmB0, &full[stage], kb * kBK, tn * (BN / 2));
            tma_load_2d(sB + (BN / 2) * 128, &tmB1, &full[stage], kb * kBK, tn * (BN / 2));
          } else {
            tma_load_2d(sB, &tmB0, &full[stage], kb * kBK, tn * BN);
          }
          issued_mask |= 1u << stage;
          last_phase_mask = (last_phase_mask & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load issued must land before the CTA can exit (normally already consumed).
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s))
          mbar_wait(&full[s], (last_phase_mask >> s) & 1u, status, SITE_DRAIN, timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = B_MN ? idesc_bf16_f32_bmn(kBM, BN) : idesc_bf16_f32(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t use = (it >> 1) & 1;
        if (!mbar_wait(&tempty[buf], use ^ 1u, status, SITE_MMA_TMEM_EMPTY, timeout_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, status, SITE_MMA_FULL, timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + stage * C::STAGE_BYTES);
          const uint64_t a_desc = sdesc_kmajor_sw128(a_addr);
          const uint64_t b_desc = B_MN ? sdesc_mnmajor_sw128(a_addr + C::A_BYTES, 64 * kBK * 2)
                                       : sdesc_kmajor_sw128(a_addr + C::A_BYTES);
          // advancing K by 16: 32 bytes along a K-major 128-byte row, or 16 rows (2048 bytes)
          // of an MN-major tile
          constexpr uint64_t b_step = B_MN ? (2048u >> 4) : 2u;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            tc_mma_bf16(d_tmem, a_desc + 2u * kk, b_desc + b_step * kk, idesc,
                        (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[buf]);
      }
      // All MMAs issued by this thread must finish before TMEM is released.
      tc_commit(drain);
      mbar_wait(drain, 0, status, SITE_DRAIN, timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* stg = stg_all + (warp - 2) * kStgPerWarp * kStgBytes;
    int sb = 0;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      int tm = 0, tn, ge = 0, grow = 0, grows = 0;
      if constexpr (GROUPED)
        group_tile(t, s_off, s_tp, ge, grow, grows, tn);
      else
        tile_coords(t, num_m, num_n, tm, tn);
      const int buf = it & 1;
      const uint32_t use = (it >> 1) & 1;
      // all lanes wait; the warp proceeds only if every lane saw the phase complete, so the
      // warp-wide tcgen05.ld below never runs with part of the warp gone
      const bool ok = mbar_wait(&tfull[buf], use, status, SITE_EPI_TMEM_FULL, timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(wq * 32) << 16) +
                             static_cast<uint32_t>(buf * BN);
      if constexpr (GROUPED) {
        const int r = wq * 32 + lane;
        epilogue_rows_direct<BN, C::BN_OUT, EPI>(t_row, lane, r < grows,
                                                 ydir + static_cast<size_t>(grow + r) * ldy,
                                                 tn * C::BN_OUT, N_out, bias, gelu_mode);
      } else {
        const int row0 = tm * kBM + wq * 32;
        epilogue_cols<BN, C::BN_OUT, EPI>(t_row, stg, sb, lane, row0, tn * C::BN_OUT, M, N_out,
                                          &tmY, bias, gelu_mode);
      }
      // this warp is done reading the accumulator buffer
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------- host side

template <int BN, int EPI, bool GROUPED = false, bool B_MN = false>
static cudaError_t launch_one(const GemmLaunch& L) {
  using C = Cfg<BN, EPI>;
  auto kern = gemm_tc_kernel<BN, EPI, GROUPED, B_MN>;
  static SmemAttrCache cache;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, cache);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = L.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB0, L.tmB1, L.tmY,
                            static_cast<const __nv_bfloat16*>(L.bias), L.M, L.N_out, L.K,
                            L.gelu_mode, L.status, L.timeout_ns, L.offsets, L.groups,
                            static_cast<__nv_bfloat16*>(L.ydir), L.ldy);
}

cudaError_t gemm_tc_launch(const GemmLaunch& L) {
  switch (L.epi * 1000 + L.bn) {
    case EPI_BIAS * 1000 + 64: return launch_one<64, EPI_BIAS>(L);
    case EPI_BIAS * 1000 + 128: return launch_one<128, EPI_BIAS>(L);
    case EPI_BIAS * 1000 + 256: return launch_one<256, EPI_BIAS>(L);
    case EPI_BIAS_GELU * 1000 + 64: return launch_one<64, EPI_BIAS_GELU>(L);
    case EPI_BIAS_GELU * 1000 + 128: return launch_one<128, EPI_BIAS_GELU>(L);
    case EPI_BIAS_GELU * 1000 + 256: return launch_one<256, EPI_BIAS_GELU>(L);
    case EPI_GEGLU * 1000 + 128: return launch_one<128, EPI_GEGLU>(L);
    case EPI_GEGLU * 1000 + 256: return launch_one<256, EPI_GEGLU>(L);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_tc_wt_launch(const GemmLaunch& L) {
  switch (L.epi * 1000 + L.bn) {
    case EPI_BIAS * 1000 + 128: return launch_one<128, EPI_BIAS, false, true>(L);
    case EPI_BIAS * 1000 + 256: return launch_one<256, EPI_BIAS, false, true>(L);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_tc_grouped_launch(const GemmLaunch& L) {
  if (L.groups < 1 || L.groups > kMoeMaxExperts || !L.offsets || !L.ydir || L.bn != 256)
    return cudaErrorInvalidValue;
  switch (L.epi) {
    case EPI_BIAS: return launch_one<256, EPI_BIAS, true>(L);
    case EPI_GEGLU: return launch_one<256, EPI_GEGLU, true>(L);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fmlp
