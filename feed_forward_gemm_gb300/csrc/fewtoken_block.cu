// Both layers of a few-token block (2..64 tokens, the biased MLP up to 128) in one launch.
//
// The few-token GEMM (gemm_skinny.cu) streams each layer's weights once as the MMA's M side,
// a weight tile of R rows split along K over the S CTAs of a cluster, the slices added in the
// owners' shared memory. Run as two launches, the second layer's weight stream starts only
// once the first layer's last CTA has exchanged its slices, stored h and exited, and the
// second kernel has set up. Here one persistent launch runs both ("ainews.cool fused-MLP
// article", technical deep-dive: a single launch for the whole MLP, only the output written;
// at few tokens the block is bound by reading the weights once):
//   - layer 1 as in the few-token GEMM, its slices exchanged through a region of shared
//     memory of their own, h rows written to the caller's workspace;
//   - as soon as the producer has issued its layer-1 loads, it fills the ring's free stages
//     with this CTA's first layer-2 weight tiles (they do not depend on h), so the layer-2
//     stream runs under layer 1's slice exchange, epilogue and the grid barrier;
//   - a grid barrier (a counter in device memory, one atomic per CTA, a bounded poll; the
//     weighted-arrival scheme of the one-kernel decode, so the counter needs no reset) makes
//     every h row visible; the producer then loads the h tiles of the prefetched stages and
//     streams the rest of layer 2; the layer-2 slices go through the freed ring.
// Every CTA must be resident at once: the grid is at most the clusters that fit (one CTA per
// SM). Every wait is bounded; a wait that runs out records its site and every thread still
// reaches the four cluster barriers, so a timeout unwinds without a hang.
//
// Warp roles (6 warps): warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps 2-5 the
// TMEM reads, slice exchange, reductions, epilogues and the grid-barrier arrival.
#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

namespace {

constexpr int kFbThreads = 192;
constexpr int kFbEpi = 128;                 // epilogue threads (warps 2-5)
constexpr int kFbBK = 64;                   // K per stage
constexpr int kFbA = 128 * kFbBK * 2;       // 16 KB: 128 weight rows x 64
constexpr unsigned long long kFbBarrierUnit = 1ull << 20;

struct FbArgs {
  CUtensorMap tmW1a;   // layer 1 weights (Wg for GeGLU), box {64, R1}
  CUtensorMap tmW1b;   // Wu for GeGLU (else a copy of tmW1a)
  CUtensorMap tmX;     // x [T, D], box {64, Tpad}
  CUtensorMap tmW2;    // layer 2 weights [Dout, H], box {64, R2}
  CUtensorMap tmH;     // h [T, H] as layer 2's token operand, box {64, Tpad}
  const __nv_bfloat16* b1;   // [H] or nullptr
  const __nv_bfloat16* b2;   // [Dout] or nullptr
  __nv_bfloat16* h;          // [T, H]
  __nv_bfloat16* y;          // [T, Dout], row stride ldy
  unsigned long long* barrier;
  int* status;
  uint64_t timeout_ns;
  int T, D, H, Dout, ldy, Tpad, R1, R2, stages, gelu_mode, xbytes;
};

__device__ __forceinline__ void st_dsmem_f32(uint32_t cluster_addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long atom_add_acq_rel_u64(unsigned long long* p,
                                                                   unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global_fb() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Named barrier of the four epilogue warps (the producer and MMA warps never take part).
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kFbEpi) : "memory");
}

template <int EPI>
__device__ __forceinline__ float fb_out(float a0, float a1, float b, int gelu_mode) {
  if (EPI == EPI_GEGLU) return gelu_tanh_f(a0) * a1;
  const float z = a0 + b;
  return EPI == EPI_BIAS_GELU ? gelu_f(z, gelu_mode) : z;
}

// Each epilogue thread's TMEM lane (one weight row of the tile) goes, for every token, to the
// row's owner: recv[s][mat][t][lr] fp32 in the owner's region, rows contiguous.
template <int NMAT>
__device__ __forceinline__ void push_slices(uint32_t recv_addr, uint32_t tmem_base, int warp,
                                            int lane, int T, int Tpad, int R, int rr, int s) {
  const int wq = warp & 3;   // TMEM lanes [32 wq, 32 wq + 32)
  const uint32_t t_row = tmem_base + (static_cast<uint32_t>(wq * 32) << 16);
  const int row = wq * 32 + lane;
  const int owner = row < R ? row / rr : 0;
  const int lr = row - owner * rr;
  const uint32_t dst0 = mapa_shared(recv_addr, static_cast<uint32_t>(owner));
  for (int mat = 0; mat < NMAT; ++mat) {
    for (int c = 0; c < T; c += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(mat * Tpad + c), v);
      tmem_ld_wait();
      if (row < R) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c + j < T)
            st_dsmem_f32(dst0 + static_cast<uint32_t>(((s * NMAT + mat) * Tpad + c + j) * rr + lr) * 4u,
                         __uint_as_float(v[j]));
      }
    }
  }
}

// The owner CTA s adds the S slices of its rows [s rr, s rr + rr) in slice order (the same
// order on every run), applies the epilogue and writes out[t, n0 + row] (row stride ld), four
// rows per thread.
template <int EPI, int NMAT>
__device__ __forceinline__ void reduce_rows(uint32_t recv_addr, int tid, int S, int s, int T,
                                            int Tpad, int R, int rr, int n0, int N,
                                            const float* bias_s, int gelu_mode,
                                            __nv_bfloat16* out, int ld) {
  const int r_lo = s * rr < R ? s * rr : R;
  const int r_hi = r_lo + rr < R ? r_lo + rr : R;
  const int rg = (r_hi - r_lo) / 4;   // R is a multiple of 4
  for (int e = tid; e < rg * T; e += kFbEpi) {
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
          const float4 v = lds_f4(recv_addr +
                                  static_cast<uint32_t>(((q * NMAT + mat) * Tpad + t) * rr + lr) * 4u);
          acc[mat].x += v.x;
          acc[mat].y += v.y;
          acc[mat].z += v.z;
          acc[mat].w += v.w;
        }
      }
    }
    const bool epb = EPI != EPI_GEGLU;
    const float o0 = fb_out<EPI>(acc[0].x, acc[NMAT - 1].x, epb ? bias_s[lr] : 0.f, gelu_mode);
    const float o1 = fb_out<EPI>(acc[0].y, acc[NMAT - 1].y, epb ? bias_s[lr + 1] : 0.f, gelu_mode);
    const float o2 = fb_out<EPI>(acc[0].z, acc[NMAT - 1].z, epb ? bias_s[lr + 2] : 0.f, gelu_mode);
    const float o3 = fb_out<EPI>(acc[0].w, acc[NMAT - 1].w, epb ? bias_s[lr + 3] : 0.f, gelu_mode);
    __nv_bfloat16* o = out + static_cast<size_t>(t) * ld + n;
    if (n + 3 < N) {
      uint2 pk;
      pk.x = pack_bf16x2(o0, o1);
      pk.y = pack_bf16x2(o2, o3);
      *reinterpret_cast<uint2*>(o) = pk;
    } else {
      o[0] = __float2bfloat16_rn(o0);
      if (n + 1 < N) o[1] = __float2bfloat16_rn(o1);
      if (n + 2 < N) o[2] = __float2bfloat16_rn(o2);
    }
  }
}

}  // namespace

template <int EPI1, int NMAT1>
__global__ void __launch_bounds__(kFbThreads, 1)
    fewtoken_block_kernel(const __grid_constant__ FbArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int Tpad = a.Tpad, stages = a.stages, T = a.T;
  const int b_bytes = Tpad * kFbBK * 2;
  const int stage_bytes = NMAT1 * kFbA + b_bytes;
  uint8_t* ring = smem;
  uint8_t* xch = ring + stages * stage_bytes;   // layer 1's slices: [S][NMAT1][Tpad][rr1] fp32
  uint64_t* full = reinterpret_cast<uint64_t*>(xch + a.xbytes);
  uint64_t* empty = full + stages;
  uint64_t* hfull = empty + stages;             // layer 2's h tile of each stage
  uint64_t* tfull = hfull + stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile uint32_t* hflag = tmem_slot + 1;     // 1 once this CTA has arrived at the barrier
  volatile unsigned long long* htarget = reinterpret_cast<unsigned long long*>(tmem_slot + 2);
  float* bias1_s = reinterpret_cast<float*>(tmem_slot + 4);
  float* bias2_s = bias1_s + 128;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = static_cast<int>(cluster_nctarank());
  const int s = static_cast<int>(cluster_ctarank());
  const int tile = blockIdx.x / S;
  const int G = gridDim.x;
  const int n1 = tile * a.R1, n2 = tile * a.R2;
  const int nk1 = (a.D + kFbBK - 1) / kFbBK, nk2 = (a.H + kFbBK - 1) / kFbBK;
  const int k1_0 = s * nk1 / S, k1_1 = (s + 1) * nk1 / S;
  const int k2_0 = s * nk2 / S, k2_1 = (s + 1) * nk2 / S;
  const int rr1 = (a.R1 + 4 * S - 1) / (4 * S) * 4, rr2 = (a.R2 + 4 * S - 1) / (4 * S) * 4;
  const uint32_t tx1 = static_cast<uint32_t>(NMAT1 * a.R1 * kFbBK * 2 + b_bytes);
  const uint32_t txA2 = static_cast<uint32_t>(a.R2 * kFbBK * 2);
  const uint32_t txB = static_cast<uint32_t>(b_bytes);
  const uint32_t tmem_cols = NMAT1 * Tpad <= 32 ? 32u : (NMAT1 * Tpad <= 64 ? 64u
                             : (NMAT1 * Tpad <= 128 ? 128u : 256u));

  if (threadIdx.x == 0) {
    prefetch_tmap(&a.tmW1a);
    if (NMAT1 == 2) prefetch_tmap(&a.tmW1b);
    prefetch_tmap(&a.tmX);
    prefetch_tmap(&a.tmW2);
    prefetch_tmap(&a.tmH);
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&hfull[i], 1);
    }
    mbar_init(tfull, 1);
    *hflag = 0u;
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

  // ring positions, kept across the phases by the producer and the MMA thread
  int pstage = 0, mstage = 0;
  uint32_t pphase = 0, mphase = 0;
  int l2_stage0 = 0, npre = 0;
  bool pok = true, tfull_ok = true;

  // ==================================================================== phase A: layer 1
  if (warp == 0) {
    if (lane == 0) {
      for (int kb = k1_0; kb < k1_1; ++kb) {
        if (!mbar_wait(&empty[pstage], pphase ^ 1u, a.status, SITE_PRODUCER_EMPTY, a.timeout_ns)) {
          pok = false;
          break;
        }
        uint8_t* st = ring + pstage * stage_bytes;
        mbar_arrive_expect_tx(&full[pstage], tx1);
        tma_load_2d(st, &a.tmW1a, &full[pstage], kb * kFbBK, n1);
        if (NMAT1 == 2) tma_load_2d(st + kFbA, &a.tmW1b, &full[pstage], kb * kFbBK, n1);
        tma_load_2d(st + NMAT1 * kFbA, &a.tmX, &full[pstage], kb * kFbBK, 0);
        if (++pstage == stages) {
          pstage = 0;
          pphase ^= 1u;
        }
      }
      // layer 2's first weight tiles, as far as the ring reaches: they do not depend on h
      l2_stage0 = pstage;
      const int npre_max = stages < k2_1 - k2_0 ? stages : k2_1 - k2_0;
      for (; pok && npre < npre_max; ++npre) {
        if (!mbar_wait(&empty[pstage], pphase ^ 1u, a.status, SITE_PRODUCER_EMPTY, a.timeout_ns)) {
          pok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[pstage], txA2);
        tma_load_2d(ring + pstage * stage_bytes, &a.tmW2, &full[pstage], (k2_0 + npre) * kFbBK,
                    n2);
        if (++pstage == stages) {
          pstage = 0;
          pphase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(Tpad));
      for (int kb = k1_0; kb < k1_1; ++kb) {
        if (!mbar_wait(&full[mstage], mphase, a.status, SITE_MMA_FULL, a.timeout_ns)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + mstage * stage_bytes);
        const uint64_t b_desc = sdesc_kmajor_sw128(a_addr + NMAT1 * kFbA);
#pragma unroll
        for (int mat = 0; mat < NMAT1; ++mat) {
          const uint64_t a_desc = sdesc_kmajor_sw128(a_addr + mat * kFbA);
#pragma unroll
          for (int kk = 0; kk < kFbBK / 16; ++kk)
            tc_mma_bf16(tmem_base + static_cast<uint32_t>(mat * Tpad), a_desc + 2u * kk,
                        b_desc + 2u * kk, idesc, (kb != k1_0 || kk != 0) ? 1u : 0u);
        }
        tc_commit(&empty[mstage]);
        if (++mstage == stages) {
          mstage = 0;
          mphase ^= 1u;
        }
      }
      tc_commit(tfull);   // phase 0: every layer-1 MMA issued above has completed
    }
    __syncwarp();
  } else {
    // the biases of the rows this CTA finishes in both layers, while the weights stream
    const int tid = threadIdx.x - 64;
    for (int i = tid; i < rr1; i += kFbEpi) {
      const int r = s * rr1 + i, n = n1 + r;
      bias1_s[i] = (EPI1 != EPI_GEGLU && a.b1 != nullptr && r < a.R1 && n < a.H)
                       ? __bfloat162float(a.b1[n]) : 0.f;
    }
    for (int i = tid; i < rr2; i += kFbEpi) {
      const int r = s * rr2 + i, n = n2 + r;
      bias2_s[i] = (a.b2 != nullptr && r < a.R2 && n < a.Dout) ? __bfloat162float(a.b2[n]) : 0.f;
    }
    tfull_ok = mbar_wait(tfull, 0, a.status, SITE_EPI_TMEM_FULL, a.timeout_ns);
    __syncwarp();
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // #1: every CTA's layer-1 MMAs are done
  const uint32_t xch_addr = smem_u32(xch);
  if (warp >= 2 && __all_sync(0xffffffffu, tfull_ok))
    push_slices<NMAT1>(xch_addr, tmem_base, warp, lane, T, Tpad, a.R1, rr1, s);
  tc_fence_before();
  cluster_sync();   // #2: every layer-1 slice is in its owner's exchange region

  // ==================================================================== phase B: h, layer 2
  if (warp >= 2) {
    const int tid = threadIdx.x - 64;
    reduce_rows<EPI1, NMAT1>(xch_addr, tid, S, s, T, Tpad, a.R1, rr1, n1, a.H, bias1_s,
                             a.gelu_mode, a.h, a.H);
    __threadfence();
    epi_sync();   // this CTA's h rows are written
    if (tid == 0) {
      // the release of the atomic, after the barrier above, publishes this CTA's h rows
      const unsigned long long mine =
          (static_cast<unsigned long long>(blockIdx.x + 1) * kFbBarrierUnit) / G -
          (static_cast<unsigned long long>(blockIdx.x) * kFbBarrierUnit) / G;
      const unsigned long long old = atom_add_acq_rel_u64(a.barrier, mine);
      *htarget = (old / kFbBarrierUnit + 1ull) * kFbBarrierUnit;
      __threadfence_block();
      *hflag = 1u;
    }
    tfull_ok = mbar_wait(tfull, 1, a.status, SITE_EPI_TMEM_FULL, a.timeout_ns);
    __syncwarp();
    tc_fence_after();
  } else if (warp == 0) {
    if (lane == 0 && pok) {
      // every CTA's h rows must be written before their TMA loads: this CTA's own arrival
      // gives the target, the counter reaching it means every CTA has arrived
      const uint64_t t0 = globaltimer_ns();
      while (*hflag == 0u) {
        if (globaltimer_ns() - t0 > a.timeout_ns) {
          atomicCAS(a.status, 0, (SITE_FEWBLOCK_BARRIER << 8) | kDeviceTimeoutCode);
          pok = false;
          break;
        }
        __nanosleep(32);
      }
      if (pok) {
        __threadfence_block();
        const unsigned long long target = *htarget;
        while (ld_acquire_u64(a.barrier) < target) {
          if (globaltimer_ns() - t0 > a.timeout_ns) {
            atomicCAS(a.status, 0, (SITE_FEWBLOCK_BARRIER << 8) | kDeviceTimeoutCode);
            pok = false;
            break;
          }
          __nanosleep(32);
        }
      }
      if (pok) {
        fence_proxy_async_global_fb();   // the TMA loads of h below come after the acquire
        for (int i = 0; i < npre; ++i) {
          const int st = (l2_stage0 + i) % stages;
          mbar_arrive_expect_tx(&hfull[st], txB);
          tma_load_2d(ring + st * stage_bytes + NMAT1 * kFbA, &a.tmH, &hfull[st],
                      (k2_0 + i) * kFbBK, 0);
        }
        for (int kb = k2_0 + npre; kb < k2_1; ++kb) {
          if (!mbar_wait(&empty[pstage], pphase ^ 1u, a.status, SITE_PRODUCER_EMPTY,
                         a.timeout_ns))
            break;
          uint8_t* stp = ring + pstage * stage_bytes;
          mbar_arrive_expect_tx(&full[pstage], txA2);
          tma_load_2d(stp, &a.tmW2, &full[pstage], kb * kFbBK, n2);
          mbar_arrive_expect_tx(&hfull[pstage], txB);
          tma_load_2d(stp + NMAT1 * kFbA, &a.tmH, &hfull[pstage], kb * kFbBK, 0);
          if (++pstage == stages) {
            pstage = 0;
            pphase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(Tpad));
      uint32_t hphase = 0;   // bit i: parity of stage i's next h fill
      for (int kb = k2_0; kb < k2_1; ++kb) {
        if (!mbar_wait(&full[mstage], mphase, a.status, SITE_MMA_FULL, a.timeout_ns)) break;
        // the first h tile comes only after the grid barrier: that wait gets the barrier's
        // limit on top of its own, so a barrier that runs out is the site recorded
        if (!mbar_wait(&hfull[mstage], (hphase >> mstage) & 1u, a.status, SITE_MMA_FULL,
                       kb == k2_0 ? 2 * a.timeout_ns : a.timeout_ns))
          break;
        hphase ^= 1u << mstage;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + mstage * stage_bytes);
        const uint64_t a_desc = sdesc_kmajor_sw128(a_addr);
        const uint64_t b_desc = sdesc_kmajor_sw128(a_addr + NMAT1 * kFbA);
#pragma unroll
        for (int kk = 0; kk < kFbBK / 16; ++kk)
          tc_mma_bf16(tmem_base, a_desc + 2u * kk, b_desc + 2u * kk, idesc,
                      (kb != k2_0 || kk != 0) ? 1u : 0u);
        tc_commit(&empty[mstage]);
        if (++mstage == stages) {
          mstage = 0;
          mphase ^= 1u;
        }
      }
      tc_commit(tfull);   // phase 1: every layer-2 MMA issued above has completed
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // #3: every CTA's layer-2 MMAs are done: the rings take the slices
  const uint32_t ring_addr = smem_u32(ring);
  if (warp >= 2 && __all_sync(0xffffffffu, tfull_ok))
    push_slices<1>(ring_addr, tmem_base, warp, lane, T, Tpad, a.R2, rr2, s);
  tc_fence_before();
  cluster_sync();   // #4: every layer-2 slice is in its owner's ring
  if (warp >= 2)
    reduce_rows<EPI_BIAS, 1>(ring_addr, threadIdx.x - 64, S, s, T, Tpad, a.R2, rr2, n2, a.Dout,
                             bias2_s, 0, a.y, a.ldy);
  // no other CTA touches this one's shared memory after the fourth barrier
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

namespace {

int fb_smem(int stages, int stage_bytes, int xbytes) {
  return 1024 + stages * stage_bytes + xbytes + (3 * stages + 1) * 8 + 16 + 256 * 4;
}

template <int EPI1, int NMAT1>
cudaError_t launch_fb(const FewBlockLaunch& L, int stages, int smem, int xbytes) {
  auto kern = fewtoken_block_kernel<EPI1, NMAT1>;
  static SmemAttrCache cache;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem, cache);
  if (e != cudaSuccess) return e;
  FbArgs a;
  memset(&a, 0, sizeof a);
  a.tmW1a = L.tmW1a;
  a.tmW1b = L.tmW1b;
  a.tmX = L.tmX;
  a.tmW2 = L.tmW2;
  a.tmH = L.tmH;
  a.b1 = static_cast<const __nv_bfloat16*>(L.b1);
  a.b2 = static_cast<const __nv_bfloat16*>(L.b2);
  a.h = static_cast<__nv_bfloat16*>(L.h);
  a.y = static_cast<__nv_bfloat16*>(L.y);
  a.barrier = L.barrier;
  a.status = L.status;
  a.timeout_ns = L.timeout_ns;
  a.T = L.T;
  a.D = L.D;
  a.H = L.H;
  a.Dout = L.Dout;
  a.ldy = L.ldy;
  a.Tpad = L.tpad;
  a.R1 = L.rows1;
  a.R2 = L.rows2;
  a.stages = stages;
  a.gelu_mode = L.gelu_mode;
  a.xbytes = xbytes;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.tiles * L.split, 1, 1);
  cfg.blockDim = dim3(kFbThreads, 1, 1);
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
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

int fewtoken_block_stages(int nmat1, int tpad, int split, int rows1, int rows2, int* smem_out,
                          int* xbytes_out) {
  const int stage_bytes = nmat1 * kFbA + tpad * kFbBK * 2;
  const int rr1 = (rows1 + 4 * split - 1) / (4 * split) * 4;
  const int rr2 = (rows2 + 4 * split - 1) / (4 * split) * 4;
  const int xbytes = split * nmat1 * tpad * rr1 * 4;
  int stages = 8;
  while (stages >= 2 && fb_smem(stages, stage_bytes, xbytes) > 232448) --stages;
  // the ring also takes layer 2's slices: [S][1][tpad][rr2] fp32
  if (stages < 2 || stages * stage_bytes < split * tpad * rr2 * 4) return 0;
  if (smem_out) *smem_out = fb_smem(stages, stage_bytes, xbytes);
  if (xbytes_out) *xbytes_out = xbytes;
  return stages;
}

cudaError_t fewtoken_block_max_clusters(int split, int* clusters) {
  // the largest shared memory any shape takes: one CTA per SM
  auto kern = fewtoken_block_kernel<EPI_BIAS_GELU, 1>;
  const int smem = 232448;
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, 1, 1);
  cfg.blockDim = dim3(kFbThreads, 1, 1);
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

cudaError_t fewtoken_block_launch(const FewBlockLaunch& L) {
  const int nmat1 = L.epi1 == EPI_GEGLU ? 2 : 1;
  const int nk1 = (L.D + kFbBK - 1) / kFbBK, nk2 = (L.H + kFbBK - 1) / kFbBK;
  if (L.T < 1 || L.tpad < L.T || L.tpad % 32 != 0 || L.tpad > kSkinnyMaxT || !L.barrier ||
      L.rows1 < 4 || L.rows1 > 128 || L.rows1 % 4 != 0 || L.rows2 < 4 || L.rows2 > 128 ||
      L.rows2 % 4 != 0 || L.tiles < 1 || static_cast<int64_t>(L.tiles) * L.rows1 < L.H ||
      static_cast<int64_t>(L.tiles) * L.rows2 < L.Dout ||
      (L.split != 1 && L.split != 2 && L.split != 4 && L.split != 8) || L.split > nk1 ||
      L.split > nk2 || (L.epi1 != EPI_GEGLU && L.epi1 != EPI_BIAS_GELU))
    return cudaErrorInvalidValue;
  int smem = 0, xbytes = 0;
  const int stages = fewtoken_block_stages(nmat1, L.tpad, L.split, L.rows1, L.rows2, &smem,
                                           &xbytes);
  if (stages == 0) return cudaErrorInvalidValue;
  return L.epi1 == EPI_GEGLU ? launch_fb<EPI_GEGLU, 2>(L, stages, smem, xbytes)
                             : launch_fb<EPI_BIAS_GELU, 1>(L, stages, smem, xbytes);
}

}  // namespace fmlp
