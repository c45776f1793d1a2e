// CTA-pair (cta_group::2) variant of the persistent tcgen05 GEMM, for large problems.
//
// A cluster of two CTAs on two SMs computes a 256 x 256 accumulator tile with one MMA stream:
// the even CTA issues tcgen05.mma.cta_group::2 with M = 256, N = 256, K = 16, whose A operand
// is 128 rows from each CTA's shared memory and whose B operand is 128 rows from each CTA's
// shared memory; each CTA's TMEM receives its own 128 rows of D (all 256 columns). Per SM
// and per 64-wide K step that is 16 KB of A plus 16 KB of B instead of 16 KB plus 32 KB for a
// single-SM 128 x 256 tile: a third less shared-memory and L2 traffic for the same MMA work.
//
// For GeGLU the even CTA loads the gate weight rows and the odd CTA the matching up weight
// rows, so D columns [0, 128) are g and [128, 256) are u for all 256 tokens, and each CTA's
// epilogue forms m = bf16(gelu_tanh(g) * u) for its 128 tokens.
//
// Synchronisation:
//   full[s]    (even CTA) one arrive.expect_tx for both CTAs' bytes; both CTAs' TMA loads
//              complete on it (.cta_group::2 lets a load signal the peer's barrier).
//   empty[s]   (both CTAs) the even CTA's tcgen05.commit multicasts to both.
//   tfull[b]   (both CTAs) accumulator b ready, multicast commit.
//   tempty[b]  (even CTA) 256 arrivals: every epilogue thread of both CTAs.
// Cluster barriers bracket the kernel so neither CTA leaves while the other may still touch
// its shared memory or TMEM. Every mbarrier wait is bounded: a wait that runs out records the
// site and ends its role's loop; the MMA thread drains its commits, the even CTA's producer
// waits (bounded) for the loads it issued, and every thread reaches the final cluster barrier.
//
// TWO (a whole GeGLU or MLP block in one persistent launch): the pairs work through a list of
// items, the first stage's tiles (gate/up with the GeGLU epilogue, or up with bias and
// activation) and the second stage's (down, with bias), which the host assigns to pairs by
// list scheduling so that no pair is left idle while others finish a partial wave of long
// down tiles. A down tile reads a 256-row band of the intermediate, so it waits (bounded)
// until every first-stage tile of that band has been stored: each epilogue warp, once the TMA
// stores of its rows of a first-stage tile have completed, adds 1 to the band's counter with
// release semantics; the producers of a down tile poll the counter with acquire semantics and
// fence the async proxy before their TMA loads of the intermediate. The counters are zero when
// the module loads and the last CTA of each launch puts them back to zero. A pair's items only
// wait on items assigned before them, and every pair is resident (the grid is at most the
// co-resident pairs), so the waits cannot form a cycle.
//
// GROUPED (mixture of experts): as in the single-SM kernel, the rows of A are grouped by expert
// with the E + 1 offsets read on the device, each group's tiles walk 256-row tile fastest, each CTA
// loading its 128 rows from the group's first row and the expert's weight slice through a
// 3-D map, and the epilogue stores rows directly, skipping those past the group.
#include "activation.cuh"
#include "gemm_epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

namespace {

constexpr int kPairBK = 64;
constexpr int kPairThreads = 32 * (2 + kEpiWarps);
constexpr int kPairA = 128 * 128;        // this CTA's 128 A rows x 64 bf16

// BN: MMA N of the pair (both CTAs' B rows together). Only 256 is instantiated: a 256x128
// pair tile was measured 1.6-1.8x slower per unit of work on GB300.
template <int BN>
struct PairCfg {
  static constexpr int B_BYTES = (BN / 2) * 128;   // this CTA's BN/2 B rows x 64 bf16
  static constexpr int STAGE = kPairA + B_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE;
  static constexpr int BAR = (2 * STAGES + 5) * 8 + 16;
  static constexpr int SMEM = 1024 + STAGES * STAGE + kEpiWarps * kStgPerWarp * kStgBytes + BAR;
  static constexpr int TMEM_COLS = 2 * BN;
  static_assert(BN == 128 || BN == 256, "pair tile width");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(B_BYTES % 1024 == 0, "1024-byte aligned B tiles");
};

// Tiles are walked in groups of `group` M tiles (256 rows each) across all N tiles, M fastest,
// so the pairs in flight share a band of x rows and a few weight panels in L2.
__device__ __forceinline__ void pair_tile_coords(int t, int num_m, int num_n, int group, int& tm,
                                                 int& tn) {
  const int per_group = group * num_n;
  const int g = t / per_group;
  const int first_m = g * group;
  const int gm = min(num_m - first_m, group);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

// Tile t of a GROUPED launch (s_tp: prefix of the groups' tile counts) -> expert e, first row
// of the 256-row tile, rows in it, N tile; within a group the row tile runs fastest, so the
// pairs in flight share one weight panel of the expert.
__device__ __forceinline__ void pair_group_tile(int t, const int* s_off, const int* s_tp, int& e,
                                                int& row0, int& rows, int& tn) {
  e = 0;
  while (s_tp[e + 1] <= t) ++e;
  const int local = t - s_tp[e];
  const int mt_e = (s_off[e + 1] - s_off[e] + 255) / 256;
  tn = local / mt_e;
  row0 = s_off[e] + (local - tn * mt_e) * 256;
  rows = min(256, s_off[e + 1] - row0);
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add_u32(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's generic-proxy accesses with its async-proxy (TMA) ones on global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

}  // namespace

// Arguments of the second stage (TWO) and the pairs' item lists; a single int otherwise, so
// the one-stage launches pass no more parameter bytes than before.
template <bool TWO>
struct TwoArgs {
  int unused;
};

template <>
struct TwoArgs<true> {
  CUtensorMap tmA2;                   // second-stage A: the intermediate [M, K2], 128-row box
  CUtensorMap tmB2;                   // second-stage weights [N2, K2], 128-row box
  CUtensorMap tmY2;                   // output [M, N2], 32-row box
  const __nv_bfloat16* bias2;         // [N2] or nullptr
  unsigned int* band;                 // [num_m] counters, zero at launch
  int N2, K2, n1, band_target;        // n1: first-stage items; target: 8 x first-stage N tiles
  uint16_t start[kTwoMaxPairs + 1];   // pair p's items: item[start[p] .. start[p + 1])
  uint16_t item[kTwoMaxItems];        // < n1: first-stage tile (raster order); else down tile
};

__device__ __forceinline__ int two_n1(const TwoArgs<true>& a) { return a.n1; }
__device__ __forceinline__ int two_n1(const TwoArgs<false>&) { return 1 << 30; }

// Item t of a two-stage list -> stage, 256-row band, N tile. First-stage items are numbered
// band-major (t = band * num_n1 + n tile; the host orders them), second-stage items follow
// (n1 + band * num_n2 + n tile).
__device__ __forceinline__ void two_tile(int t, int n1, int num_n1, int num_n2, bool& second,
                                         int& tm, int& tn) {
  second = t >= n1;
  const int u = second ? t - n1 : t;
  const int per = second ? num_n2 : num_n1;
  tm = u / per;
  tn = u - tm * per;
}

// Band counters of the two-stage launches, one row of kTwoBandRow words per stream slot (the
// bands, then the count of CTAs that have finished); zero when the module loads, and put back
// to zero by the last CTA of each launch.
constexpr int kTwoBandRow = 128;
static_assert(kTwoMaxBands < kTwoBandRow, "band row holds the bands and the finished count");
__device__ unsigned int g_two_band[kDecodeSlots * kTwoBandRow];

template <int BN, int EPI, bool GROUPED, bool TWO>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmY,
                    const __nv_bfloat16* __restrict__ bias, int M, int N_out, int K,
                    int gelu_mode, int group, int* status, uint64_t timeout_ns,
                    const int* __restrict__ offsets, int E, __nv_bfloat16* __restrict__ ydir,
                    int ldy, int skip_first_load, const __grid_constant__ TwoArgs<TWO> two) {
  using C = PairCfg<BN>;
  constexpr int kPairStages = C::STAGES;
  constexpr int kPairStage = C::STAGE;
  constexpr int BN_OUT = EPI == EPI_GEGLU ? BN / 2 : BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  uint8_t* stg_all = smem + kPairStages * kPairStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(stg_all + kEpiWarps * kStgPerWarp * kStgBytes);
  uint64_t* empty = full + kPairStages;
  uint64_t* tfull = empty + kPairStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: issues the MMAs, 1: its peer
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    prefetch_tmap(&tmB1);
    prefetch_tmap(&tmY);
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * kEpiWarps * 32);
    }
    mbar_init(drain, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // barriers of both CTAs initialised before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  pdl_wait_primary();
  if (threadIdx.x == 0) pdl_launch_dependents();

  const int num_m = (M + 2 * 128 - 1) / (2 * 128);
  const int num_n = (N_out + BN_OUT - 1) / BN_OUT;
  const int num_kb = (K + kPairBK - 1) / kPairBK;
  // GROUPED: token offsets and the prefix of the groups' tile counts, in the (unused) staging
  // area
  int* s_off = reinterpret_cast<int*>(stg_all);
  int* s_tp = s_off + (kMoeMaxExperts + 1);
  int grouped_tiles = 0;
  if constexpr (GROUPED) {
    for (int i = threadIdx.x; i <= E; i += kPairThreads) s_off[i] = min(max(__ldcg(offsets + i), 0), M);
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0;
      s_tp[0] = 0;
      for (int g = 0; g < E; ++g) {
        s_off[g + 1] = max(s_off[g + 1], s_off[g]);   // a falling offset makes the group empty
        acc += (s_off[g + 1] - s_off[g] + 255) / 256 * num_n;
        s_tp[g + 1] = acc;
      }
    }
    __syncthreads();
    grouped_tiles = s_tp[E];
  }
  const int num_tiles = GROUPED ? grouped_tiles : num_m * num_n;
  // This pair's items: t = pair, pair + npairs, ... below num_tiles, or (TWO) its list.
  int n_items = 0;
  if constexpr (TWO)
    n_items = two.start[pair + 1] - two.start[pair];
  else
    n_items = pair < num_tiles ? (num_tiles - pair + npairs - 1) / npairs : 0;
  auto item_at = [&](int k) -> int {
    if constexpr (TWO) return two.item[two.start[pair] + k];
    return pair + k * npairs;
  };
  // second-stage geometry (TWO)
  int num_n2 = 1, num_kb2 = 0;
  if constexpr (TWO) {
    num_n2 = (two.N2 + BN - 1) / BN;
    num_kb2 = (two.K2 + kPairBK - 1) / kPairBK;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(smem_u32(full), 0);   // even CTA's full[0]
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_phase_mask = 0;
      bool ok = true;
      for (int k = 0; k < n_items && ok; ++k) {
        const int t = item_at(k);
        int tm = 0, tn, ge = 0, grow = 0, grows = 0;
        bool second = false;
        if constexpr (GROUPED) {
          pair_group_tile(t, s_off, s_tp, ge, grow, grows, tn);
        } else if (TWO) {
          two_tile(t, two_n1(two), num_n, num_n2, second, tm, tn);
        } else {
          pair_tile_coords(t, num_m, num_n, group, tm, tn);
        }
        const int a_row = (GROUPED ? grow : tm * 256) + static_cast<int>(rank) * 128;
        const CUtensorMap* amap = &tmA;
        const CUtensorMap* bmap = &tmB0;
        int b_row;
        int item_kb = num_kb;
        if constexpr (TWO) {
          if (second) {
            // the band of the intermediate this down tile reads must be stored completely
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_u32(two.band + tm) < static_cast<unsigned>(two.band_target)) {
              if (globaltimer_ns() - t0 > timeout_ns) {
                atomicCAS(status, 0, (SITE_BAND << 8) | kDeviceTimeoutCode);
                ok = false;
                break;
              }
              __nanosleep(64);
            }
            if (!ok) break;
            fence_proxy_async_global();   // the TMA loads below come after the acquire
            amap = &two.tmA2;
            bmap = &two.tmB2;
            item_kb = num_kb2;
          }
        }
        if (second) {
          b_row = tn * BN + static_cast<int>(rank) * (BN / 2);
        } else if (EPI == EPI_GEGLU) {
          bmap = rank == 0 ? &tmB0 : &tmB1;   // gate rows on the even CTA, up rows on the odd
          b_row = tn * (BN / 2);
        } else {
          b_row = tn * BN + static_cast<int>(rank) * (BN / 2);
        }
        for (int kb = 0; kb < item_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, status, SITE_PRODUCER_EMPTY, timeout_ns)) {
            ok = false;
            break;
          }
          uint8_t* sA = stages + stage * kPairStage;
          uint8_t* sB = sA + kPairA;
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * kPairStage);
          // test hook: the first K step of the pair's first tile expects its bytes but no load
          // brings them, so the MMA's bounded wait on this stage runs out
          if (skip_first_load && t == pair && kb == 0) {
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          const uint32_t fb = full0 + static_cast<uint32_t>(stage * 8);
          tma_load_2d_pair(sA, amap, fb, kb * kPairBK, a_row);
          if constexpr (GROUPED)
            tma_load_3d_pair(sB, bmap, fb, kb * kPairBK, b_row, ge);
          else
            tma_load_2d_pair(sB, bmap, fb, kb * kPairBK, b_row);
          issued_mask |= 1u << stage;
          last_phase_mask = (last_phase_mask & ~(1u << stage)) | (phase << stage);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // loads land on the even CTA's barriers; it waits for all of them before exiting
      if (rank == 0)
        for (int s = 0; s < kPairStages; ++s)
          if (issued_mask & (1u << s))
            mbar_wait(&full[s], (last_phase_mask >> s) & 1u, status, SITE_DRAIN, timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(256, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int k = 0; k < n_items && ok; ++k, ++it) {
        const int item_kb = item_at(k) >= two_n1(two) ? num_kb2 : num_kb;
        const int buf = it & 1;
        const uint32_t use = (it >> 1) & 1;
        if (!mbar_wait(&tempty[buf], use ^ 1u, status, SITE_MMA_TMEM_EMPTY, timeout_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < item_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, status, SITE_MMA_FULL, timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + stage * kPairStage);
          const uint64_t a_desc = sdesc_kmajor_sw128(a_addr);
          const uint64_t b_desc = sdesc_kmajor_sw128(a_addr + kPairA);
#pragma unroll
          for (int kk = 0; kk < kPairBK / 16; ++kk)
            tc_mma_bf16_pair(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc,
                             (kb | kk) != 0 ? 1u : 0u);
          tc_commit_pair_mc(&empty[stage], 0x3);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&tfull[buf], 0x3);
      }
      tc_commit_pair(drain);
      mbar_wait(drain, 0, status, SITE_DRAIN, timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int wq = warp & 3;
    uint8_t* stg = stg_all + (warp - 2) * kStgPerWarp * kStgBytes;
    const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);
    int sb = 0;
    int it = 0;
    for (int k = 0; k < n_items; ++k, ++it) {
      const int t = item_at(k);
      int tm = 0, tn, ge = 0, grow = 0, grows = 0;
      bool second = false;
      if constexpr (GROUPED) {
        pair_group_tile(t, s_off, s_tp, ge, grow, grows, tn);
      } else if (TWO) {
        two_tile(t, two_n1(two), num_n, num_n2, second, tm, tn);
      } else {
        pair_tile_coords(t, num_m, num_n, group, tm, tn);
      }
      const int buf = it & 1;
      const uint32_t use = (it >> 1) & 1;
      const bool ok = mbar_wait(&tfull[buf], use, status, SITE_EPI_TMEM_FULL, timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(wq * 32) << 16) +
                             static_cast<uint32_t>(buf * BN);
      if constexpr (GROUPED) {
        const int r = static_cast<int>(rank) * 128 + wq * 32 + lane;
        epilogue_rows_direct<BN, BN_OUT, EPI>(t_row, lane, r < grows,
                                              ydir + static_cast<size_t>(grow + r) * ldy,
                                              tn * BN_OUT, N_out, bias, gelu_mode);
      } else {
        const int row0 = tm * 256 + static_cast<int>(rank) * 128 + wq * 32;
        if constexpr (TWO) {
          if (second) {
            epilogue_cols<BN, BN, EPI_BIAS>(t_row, stg, sb, lane, row0, tn * BN, M, two.N2,
                                            &two.tmY2, two.bias2, 0);
          } else {
            epilogue_cols<BN, BN_OUT, EPI>(t_row, stg, sb, lane, row0, tn * BN_OUT, M, N_out,
                                           &tmY, bias, gelu_mode);
            // this warp's rows of the band are stored: count them for the down tiles
            if (lane == 0) {
              bulk_wait_group<0>();
              fence_proxy_async_global();
              red_release_add_u32(two.band + tm, 1u);
            }
            __syncwarp();
          }
        } else {
          epilogue_cols<BN, BN_OUT, EPI>(t_row, stg, sb, lane, row0, tn * BN_OUT, M, N_out,
                                         &tmY, bias, gelu_mode);
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(buf * 8));
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's MMAs, loads and arrivals are finished
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
  if constexpr (TWO) {
    // Every thread of this CTA is past its last band access. The last CTA to get here puts
    // the counters back to zero for the next launch on this slot (which reads them only after
    // this grid has completed: stream order, or its griddepcontrol.wait).
    int* s_last = reinterpret_cast<int*>(stg_all);
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned done = atomicAdd(two.band + kTwoBandRow - 1, 1u);
      *s_last = done == gridDim.x - 1u;
    }
    __syncthreads();
    if (*s_last) {
      __threadfence();
      for (int i = threadIdx.x; i < num_m; i += kPairThreads) two.band[i] = 0u;
      if (threadIdx.x == 0) two.band[kTwoBandRow - 1] = 0u;
    }
  }
}

int gemm_tc2_group(int K) {
  // Raster group: as many 256-row bands of A as fit in about 64 MB of L2 (at least 2, at most
  // 16; 16 measured best for the 8192-wide, K = 8192 gate/up GEMM).
  int group = static_cast<int>((64ll << 20) / (256ll * K * 2));
  return group < 2 ? 2 : (group > 16 ? 16 : group);
}

template <int BN, int EPI, bool GROUPED = false, bool TWO = false>
static cudaError_t launch_pair(const GemmLaunch& L, const TwoArgs<TWO>& two) {
  using C = PairCfg<BN>;
  auto kern = gemm_tc2_kernel<BN, EPI, GROUPED, TWO>;
  static SmemAttrCache cache;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), C::SMEM, cache);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = L.pdl ? 1 : 0;
  const int group = gemm_tc2_group(L.K);
  return cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB0, L.tmB1, L.tmY,
                            static_cast<const __nv_bfloat16*>(L.bias), L.M, L.N_out, L.K,
                            L.gelu_mode, group, L.status, L.timeout_ns, L.offsets, L.groups,
                            static_cast<__nv_bfloat16*>(L.ydir), L.ldy, L.skip_first_load ? 1 : 0,
                            two);
}

cudaError_t gemm_tc2_launch(const GemmLaunch& L) {
  if (L.grid < 2 || (L.grid & 1)) return cudaErrorInvalidValue;
  const TwoArgs<false> none{0};
  switch (L.epi * 1000 + L.bn) {
    case EPI_BIAS * 1000 + 256: return launch_pair<256, EPI_BIAS>(L, none);
    case EPI_BIAS_GELU * 1000 + 256: return launch_pair<256, EPI_BIAS_GELU>(L, none);
    case EPI_GEGLU * 1000 + 256: return launch_pair<256, EPI_GEGLU>(L, none);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_tc2_two_launch(const GemmLaunch& L, const TwoStageLaunch& T2) {
  const int pairs = L.grid / 2;
  const int num_m = (L.M + 255) / 256;
  if (L.grid < 2 || (L.grid & 1) || L.bn != 256 || pairs > kTwoMaxPairs || num_m > kTwoMaxBands ||
      T2.n_items > kTwoMaxItems || T2.n_items < T2.n1 || !T2.start || !T2.item ||
      T2.slot < 0 || T2.slot >= kDecodeSlots || (L.epi != EPI_GEGLU && L.epi != EPI_BIAS_GELU))
    return cudaErrorInvalidValue;
  unsigned int* band = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&band), g_two_band);
  if (e != cudaSuccess) return e;
  // the launch copies the parameter block, so a stack copy is enough
  static thread_local TwoArgs<true> a;
  a.tmA2 = T2.tmA2;
  a.tmB2 = T2.tmB2;
  a.tmY2 = T2.tmY2;
  a.bias2 = static_cast<const __nv_bfloat16*>(T2.bias2);
  a.band = band + static_cast<size_t>(T2.slot) * kTwoBandRow;
  a.N2 = T2.N2;
  a.K2 = T2.K2;
  a.n1 = T2.n1;
  // each first-stage tile adds one per epilogue warp of the pair to its band
  const int bn_out = L.epi == EPI_GEGLU ? 128 : 256;
  a.band_target = 2 * kEpiWarps * ((L.N_out + bn_out - 1) / bn_out) + T2.band_extra;
  for (int p = 0; p <= pairs; ++p) a.start[p] = T2.start[p];
  for (int i = 0; i < T2.n_items; ++i) a.item[i] = T2.item[i];
  return L.epi == EPI_GEGLU ? launch_pair<256, EPI_GEGLU, false, true>(L, a)
                            : launch_pair<256, EPI_BIAS_GELU, false, true>(L, a);
}

cudaError_t gemm_tc2_grouped_launch(const GemmLaunch& L) {
  if (L.grid < 2 || (L.grid & 1) || L.groups < 1 || L.groups > kMoeMaxExperts || !L.offsets ||
      !L.ydir || L.bn != 256)
    return cudaErrorInvalidValue;
  switch (L.epi) {
    case EPI_BIAS: return launch_pair<256, EPI_BIAS, true>(L, TwoArgs<false>{0});
    case EPI_GEGLU: return launch_pair<256, EPI_GEGLU, true>(L, TwoArgs<false>{0});
    default: return cudaErrorInvalidValue;
  }
}

// Largest number of co-resident CTA pairs (queried once per device by the host).
cudaError_t gemm_tc2_max_pairs(int* pairs) {
  auto kern = gemm_tc2_kernel<256, EPI_BIAS, false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PairCfg<256>::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfg<256>::SMEM;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
  if (e != cudaSuccess) return e;
  *pairs = n;
  return cudaSuccess;
}

}  // namespace fmlp
