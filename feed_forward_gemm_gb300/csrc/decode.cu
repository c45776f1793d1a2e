// The whole feed-forward block for one to four tokens (decode) in one kernel:
//   layer 1  h = bf16(act(x W1^T + b1))              (Linear -> GELU/ReLU -> Linear)
//         or h = bf16(gelu_tanh(x Wg^T) * (x Wu^T))   (GeGLU)
//   layer 2  y = bf16(h W2^T + b2)
//
// At a few tokens the block reads every weight once and does one multiply-add per weight, so
// its time is the weight bytes over HBM bandwidth plus whatever the launches and the
// dependency between the layers add (ainews.cool fused-MLP article, technical deep-dive:
// batch-1 decode pays a launch per layer and is bound by memory traffic; its single-launch
// MLP writes only the output). This kernel keeps one stream of weight bytes flowing through
// both layers:
//   - one CTA per SM, every CTA resident at once (grid <= co-resident CTAs); CTA b owns a
//     contiguous block of layer-1 rows and a contiguous block of layer-2 rows;
//   - each thread covers fixed 16-byte chunks of a row (a group of threads covers the row)
//     and streams batches of 8 rows (4 per matrix for GeGLU) with 16-byte non-allocating
//     loads, two batches always in flight (the next is issued before the current is used);
//     the token vectors sit in shared memory and each chunk of them is unpacked once per
//     batch; a batch's row sums are reduced over the warp by recursive halving (about one
//     shuffle per row) and over the group's warps in a fixed order (deterministic);
//   - the x loads go out before the first weight loads, so x is not queued behind them;
//   - layer-1 outputs h go to the caller's workspace; a grid barrier (a counter in device
//     memory, one atomic per CTA, waited on with a bounded poll) makes every h row visible;
//     the first batch of layer-2 weight loads is issued before the barrier (it does not
//     depend on h), so HBM stays busy while the CTAs meet.
// Every input, weights included, is read only after the dependency wait, so a kernel queued
// just before may have written any of them.
//
// Failure handling: the barrier wait is bounded; a wait that runs out records the site in
// the device status word and the CTA skips the rest of its work; nothing spins without a
// limit. The barrier counter needs no reset: CTA b adds w_b = floor((b+1) 2^20 / G) -
// floor(b 2^20 / G) (the G weights sum to 2^20), so the counter is a multiple of 2^20
// between launches and each launch waits for the next multiple. Every CTA adds its weight
// exactly once, even one whose wait runs out, so the counter stays consistent.
#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

// Grid-barrier counters, kDecodeSlots of them 128 bytes apart, zero when the module loads.
__device__ unsigned long long g_decode_barrier[kDecodeSlots * 16];

namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecRegs = 65536 / kDecThreads;   // registers per thread, one CTA per SM
constexpr unsigned long long kBarrierUnit = 1ull << 20;
constexpr int kXRegs = kDecRegs >= 128 ? 4 : 1;   // x chunks held while the weight loads go out

// Rows per load group (two groups in flight per thread): 8 when a thread may use 128
// registers; 4 (2 at four tokens) within 64.
template <int TT>
constexpr int decode_rb() { return kDecRegs >= 128 ? 8 : (TT == 4 ? 2 : 4); }

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Through L2 only: data another CTA of this grid, or the previous kernel, may have written.
__device__ __forceinline__ uint4 ldg_cg(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned long long atom_add_acq_rel(unsigned long long* p,
                                                               unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], %2;"
               : "=l"(old)
               : "l"(p), "l"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Eight bf16 (one 16-byte chunk) widened to fp32.
__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
  f[0] = bf16_lo(v.x);
  f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y);
  f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z);
  f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w);
  f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ float dot8f(uint4 w, const float (&x)[8], float s) {
  s = fmaf(bf16_lo(w.x), x[0], s);
  s = fmaf(bf16_hi(w.x), x[1], s);
  s = fmaf(bf16_lo(w.y), x[2], s);
  s = fmaf(bf16_hi(w.y), x[3], s);
  s = fmaf(bf16_lo(w.z), x[4], s);
  s = fmaf(bf16_hi(w.z), x[5], s);
  s = fmaf(bf16_lo(w.w), x[6], s);
  s = fmaf(bf16_hi(w.w), x[7], s);
  return s;
}

// Warp sums of N values per lane (N a power of two, 2..32) by recursive halving: at the
// exchange with lane ^ o (o = 16, 8, ...) each lane keeps half of its live values, sends the
// other half and adds what its partner sent, so N values cost N - 1 + (5 - log2 N) shuffles
// instead of 5 N. Afterwards lane L holds, in v[0], the warp sum of value L >> (5 - log2 N)
// (each sum held by 32 / N neighbouring lanes). The order of the additions is fixed.
template <int N>
__device__ __forceinline__ void warp_sum_many(float (&v)[N], int lane) {
  int live = N;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (live > 1) {
      const int half = live / 2;
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float keep = up ? v[i + half] : v[i];
          const float give = up ? v[i] : v[i + half];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
        }
      }
      live = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
}

constexpr int log2_const(int n) { return n <= 1 ? 0 : 1 + log2_const(n / 2); }

// How a CTA's threads cover rows of length K: groups of `gt` threads, each group on its own
// rows; thread q of a group sums 16-byte chunks q, q + gt, ... of the row.
struct KSplit {
  int C;       // 16-byte chunks per row (K / 8)
  int gt;      // threads per group (a multiple of 32)
  int groups;  // groups per CTA
  int nch;     // chunks per thread (the last may be past C for some threads)
};

__host__ __device__ inline KSplit make_ksplit(int K) {
  KSplit s;
  s.C = K / 8;
  if (s.C >= kDecThreads) {
    s.gt = kDecThreads;
    s.groups = 1;
    s.nch = (s.C + kDecThreads - 1) / kDecThreads;
  } else {
    const int wg = (s.C + 31) / 32;
    s.gt = wg * 32;
    s.groups = kDecWarps / wg;
    s.nch = 1;
  }
  return s;
}

struct DecodeArgs {
  const __nv_bfloat16* x;    // [T, D], row stride ldx
  const __nv_bfloat16* W1a;  // [H, D]  (W1, or Wg)
  const __nv_bfloat16* W1b;  // [H, D]  (Wu; GeGLU only)
  const __nv_bfloat16* b1;   // [H] or nullptr (MLP only)
  const __nv_bfloat16* W2;   // [Dout, H]
  const __nv_bfloat16* b2;   // [Dout] or nullptr
  __nv_bfloat16* h;          // [T, H] workspace
  __nv_bfloat16* y;          // [T, Dout], row stride ldy
  unsigned long long* barrier;
  int* status;
  unsigned long long timeout_ns;
  int T, D, H, Dout, ldx, ldy;
  int gelu_mode;
  int slots;                 // rows per warp in the reduction buffer
  int vec_bytes;             // shared bytes of the token vectors (T * max(D, H) * 2)
};

// Shared-memory state of one CTA (offsets into the dynamic shared memory).
struct Smem {
  uint4* vec;        // [T][K] bf16: x for layer 1, then h for layer 2
  float* red;        // [warps][slots][NMAT][TT] per-warp row sums
  int* flag;         // 1 while every wait of this CTA succeeded
};

// Per-thread partial dot products of `nrows` rows of NMAT weight matrices (row j of matrix m
// at W_m + j * K) with the T token vectors in s.vec, reduced over each warp into s.red.
// The loads come in groups of RB 16-byte chunks (one chunk of RB / NMAT rows per matrix);
// two groups are always in flight: the next group's loads are issued before the current one
// is used. `hook` runs once, by every thread, after the first two groups have been issued:
// it makes the token vectors ready in s.vec (and synchronises the CTA). The caller
// synchronises before reading s.red.
template <int NMAT, int TT, int RB, typename Hook>
__device__ __forceinline__ void rows_dot(const Smem& s, const KSplit& ks, int K,
                                         const __nv_bfloat16* W0, const __nv_bfloat16* W1,
                                         int nrows, int T, int slots, Hook hook) {
  constexpr int RR = RB / NMAT;  // rows per group
  constexpr int NV = RB * TT;    // values reduced per batch of rows (a power of two, <= 32)
  constexpr int SH = 5 - log2_const(NV);
  static_assert(NV >= 2 && NV <= 32 && (NV & (NV - 1)) == 0, "RB * TT must be 2..32, a power of 2");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wg = ks.gt >> 5;
  const int g = warp / wg;
  const int q = (warp - g * wg) * 32 + lane;
  const bool active = g < ks.groups;
  const int kvec = K / 8;
  // this group's rows j = k * groups + g, k = 0 .. mine - 1; batches of RR of them, each
  // batch read in nch chunk steps: load group u = batch * nch + chunk step
  const int mine = active && g < nrows ? (nrows - g + ks.groups - 1) / ks.groups : 0;
  const int total = (mine + RR - 1) / RR * ks.nch;

  auto issue = [&](int u, uint4 (&w)[RB]) {
    const int kb = (u / ks.nch) * RR, c = u - (u / ks.nch) * ks.nch;
    const int chunk = q + c * ks.gt;
    const bool cok = chunk < ks.C;
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int j = (kb + i / NMAT) * ks.groups + g;
      w[i] = make_uint4(0u, 0u, 0u, 0u);
      if (cok && j < nrows) {
        const __nv_bfloat16* Wm = (NMAT == 2 && (i % NMAT) == 1) ? W1 : W0;
        w[i] = ldg_stream(Wm + static_cast<size_t>(j) * K + static_cast<size_t>(chunk) * 8);
      }
    }
  };
  float acc[NV];
#pragma unroll
  for (int f = 0; f < NV; ++f) acc[f] = 0.f;
  auto consume = [&](int u, const uint4 (&w)[RB]) {
    const int kb = (u / ks.nch) * RR, c = u - (u / ks.nch) * ks.nch;
    const int chunk = q + c * ks.gt;
    if (chunk < ks.C) {
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        if (t < T) {
          float xf[8];
          unpack8(s.vec[t * kvec + chunk], xf);
#pragma unroll
          for (int i = 0; i < RB; ++i) acc[i * TT + t] = dot8f(w[i], xf, acc[i * TT + t]);
        }
      }
    }
    if (c == ks.nch - 1) {   // the batch's last chunk step: reduce and store its row sums
      warp_sum_many<NV>(acc, lane);
      if ((lane & ((1 << SH) - 1)) == 0) {
        const int f = lane >> SH;
        const int i = f / TT, t = f - i * TT;
        const int k = kb + i / NMAT;
        if (t < T && k * ks.groups + g < nrows)
          s.red[((warp * slots + k) * NMAT + (i % NMAT)) * TT + t] = acc[0];
      }
#pragma unroll
      for (int f = 0; f < NV; ++f) acc[f] = 0.f;
    }
  };

  uint4 wa[RB], wb[RB];
  if (total > 0) issue(0, wa);
  if (total > 1) issue(1, wb);
  hook();
  for (int u = 0; u < total; u += 2) {
    consume(u, wa);
    if (u + 2 < total) issue(u + 2, wa);
    if (u + 1 < total) {
      consume(u + 1, wb);
      if (u + 3 < total) issue(u + 3, wb);
    }
  }
}

// Sum of row j (matrix m, token t) over the warps of its group, in warp order.
template <int NMAT, int TT>
__device__ __forceinline__ float row_sum(const Smem& s, const KSplit& ks, int slots, int j,
                                         int m, int t) {
  const int wg = ks.gt >> 5;
  const int g = j % ks.groups, k = j / ks.groups;
  float v = 0.f;
  for (int w = g * wg; w < (g + 1) * wg; ++w) v += s.red[((w * slots + k) * NMAT + m) * TT + t];
  return v;
}

__device__ __forceinline__ int split_at(int i, int n) {
  return static_cast<int>((static_cast<int64_t>(i) * n) / gridDim.x);
}

template <int NMAT, int TT>
__global__ void __launch_bounds__(kDecThreads, 1) ffn_decode_kernel(const DecodeArgs a) {
  constexpr int RB1 = decode_rb<TT>();
  constexpr int RB2 = decode_rb<TT>() >= 2 * NMAT ? decode_rb<TT>() : 2 * NMAT;
  extern __shared__ __align__(16) uint8_t dsm[];
  const int T = a.T, D = a.D, H = a.H;
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  // this CTA's rows of each layer
  const int r0 = split_at(b, H), nr1 = split_at(b + 1, H) - r0;
  const int c0 = split_at(b, a.Dout), nr2 = split_at(b + 1, a.Dout) - c0;

  Smem s;
  s.vec = reinterpret_cast<uint4*>(dsm);
  s.red = reinterpret_cast<float*>(dsm + a.vec_bytes);
  s.flag = reinterpret_cast<int*>(s.red + kDecWarps * a.slots * NMAT * TT);
  if (threadIdx.x == 0) *s.flag = 1;
  // every input (x, all weights and biases) may come from the kernel queued before this one
  pdl_wait_primary();
  // every CTA of this grid is resident once all of them got here: the next kernel may launch
  if (threadIdx.x == 0) pdl_launch_dependents();

  // ---------------------------------------------------------------- layer 1
  const KSplit k1 = make_ksplit(D);
  const int kv1 = D / 8, nx = T * kv1;
  uint4 xr[kXRegs];
#pragma unroll
  for (int u = 0; u < kXRegs; ++u) {
    const int i = threadIdx.x + u * kDecThreads;
    if (i < nx) {
      const int t = i / kv1;
      xr[u] = ldg_cg(a.x + static_cast<size_t>(t) * a.ldx + static_cast<size_t>(i - t * kv1) * 8);
    }
  }
  auto stage_x = [&]() {
#pragma unroll
    for (int u = 0; u < kXRegs; ++u) {
      const int i = threadIdx.x + u * kDecThreads;
      if (i < nx) s.vec[i] = xr[u];
    }
    for (int i = threadIdx.x + kXRegs * kDecThreads; i < nx; i += kDecThreads) {
      const int t = i / kv1;
      s.vec[i] = ldg_cg(a.x + static_cast<size_t>(t) * a.ldx + static_cast<size_t>(i - t * kv1) * 8);
    }
    __syncthreads();
  };
  rows_dot<NMAT, TT, RB1>(s, k1, D, a.W1a + static_cast<size_t>(r0) * D,
                          NMAT == 2 ? a.W1b + static_cast<size_t>(r0) * D : nullptr, nr1, T,
                          a.slots, stage_x);
  __syncthreads();
  for (int e = threadIdx.x; e < nr1 * T; e += kDecThreads) {
    const int t = e / nr1, j = e - t * nr1;
    const int n = r0 + j;
    float v;
    if (NMAT == 2) {
      v = gelu_tanh_f(row_sum<NMAT, TT>(s, k1, a.slots, j, 0, t)) *
          row_sum<NMAT, TT>(s, k1, a.slots, j, 1, t);
    } else {
      const float z = row_sum<NMAT, TT>(s, k1, a.slots, j, 0, t) +
                      (a.b1 != nullptr ? __bfloat162float(a.b1[n]) : 0.f);
      v = gelu_f(z, a.gelu_mode);
    }
    a.h[static_cast<size_t>(t) * H + n] = __float2bfloat16_rn(v);
  }

  // ---------------------------------------------------------------- grid barrier, layer 2
  const KSplit k2 = make_ksplit(H);
  auto barrier_then_stage_h = [&]() {
    __syncthreads();   // this CTA's h stores are issued; the reduction buffer is free
    if (threadIdx.x == 0) {
      // the release of the atomic, after the CTA barrier above, publishes this CTA's h
      const unsigned long long mine =
          (static_cast<unsigned long long>(b + 1) * kBarrierUnit) / G -
          (static_cast<unsigned long long>(b) * kBarrierUnit) / G;
      const unsigned long long old = atom_add_acq_rel(a.barrier, mine);
      const unsigned long long target = (old / kBarrierUnit + 1ull) * kBarrierUnit;
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire(a.barrier) < target) {
        if (globaltimer_ns() - t0 > a.timeout_ns) {
          atomicCAS(a.status, 0, (SITE_DECODE_BARRIER << 8) | kDeviceTimeoutCode);
          *s.flag = 0;
          break;
        }
        __nanosleep(20);
      }
    }
    __syncthreads();
    if (*s.flag) {
      const int kv = H / 8;
      for (int i = threadIdx.x; i < T * kv; i += kDecThreads)
        s.vec[i] = ldg_cg(a.h + static_cast<size_t>(i) * 8);
    }
    __syncthreads();
  };
  rows_dot<1, TT, RB2>(s, k2, H, a.W2 + static_cast<size_t>(c0) * H, nullptr, nr2, T, a.slots,
                       barrier_then_stage_h);
  __syncthreads();
  if (*s.flag) {
    for (int e = threadIdx.x; e < nr2 * T; e += kDecThreads) {
      const int t = e / nr2, j = e - t * nr2;
      const int n = c0 + j;
      const float z = row_sum<1, TT>(s, k2, a.slots, j, 0, t) +
                      (a.b2 != nullptr ? __bfloat162float(a.b2[n]) : 0.f);
      a.y[static_cast<size_t>(t) * a.ldy + n] = __float2bfloat16_rn(z);
    }
  }
}

int decode_slots(int D, int H, int Dout, int grid) {
  const int rows1 = (H + grid - 1) / grid, rows2 = (Dout + grid - 1) / grid;
  const int g1 = make_ksplit(D).groups, g2 = make_ksplit(H).groups;
  const int s1 = (rows1 + g1 - 1) / g1, s2 = (rows2 + g2 - 1) / g2;
  return s1 > s2 ? s1 : s2;
}

int tt_of(int T) { return T <= 1 ? 1 : (T <= 2 ? 2 : 4); }

}  // namespace

size_t decode_smem_bytes(int T, int D, int H, int Dout, int nmat, int grid) {
  const size_t vec = static_cast<size_t>(T) * (D > H ? D : H) * 2;
  const size_t red = static_cast<size_t>(kDecWarps) * decode_slots(D, H, Dout, grid) * nmat *
                     tt_of(T) * 4;
  return vec + red + 16;
}

template <int NMAT, int TT>
static cudaError_t decode_launch_t(const DecodeLaunch& L, const DecodeArgs& a, size_t smem) {
  auto kern = ffn_decode_kernel<NMAT, TT>;
  static SmemAttrCache cache;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), static_cast<int>(smem), cache);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(kDecThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t decode_launch(const DecodeLaunch& L) {
  const int nmat = L.geglu ? 2 : 1;
  if (L.T < 1 || L.T > kDecodeMaxT || L.D < 8 || L.D % 8 != 0 || L.H < 8 || L.H % 8 != 0 ||
      L.Dout < 1 || L.grid < 1 || !L.barrier)
    return cudaErrorInvalidValue;
  const size_t smem = decode_smem_bytes(L.T, L.D, L.H, L.Dout, nmat, L.grid);
  if (smem > kDecodeMaxSmem) return cudaErrorInvalidValue;
  DecodeArgs a;
  a.x = static_cast<const __nv_bfloat16*>(L.x);
  a.W1a = static_cast<const __nv_bfloat16*>(L.W1a);
  a.W1b = static_cast<const __nv_bfloat16*>(L.W1b);
  a.b1 = static_cast<const __nv_bfloat16*>(L.b1);
  a.W2 = static_cast<const __nv_bfloat16*>(L.W2);
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
  a.ldx = L.ldx;
  a.ldy = L.ldy;
  a.gelu_mode = L.gelu_mode;
  a.slots = decode_slots(L.D, L.H, L.Dout, L.grid);
  a.vec_bytes = L.T * (L.D > L.H ? L.D : L.H) * 2;
  const int tt = tt_of(L.T);
  if (L.geglu) {
    switch (tt) {
      case 1: return decode_launch_t<2, 1>(L, a, smem);
      case 2: return decode_launch_t<2, 2>(L, a, smem);
      default: return decode_launch_t<2, 4>(L, a, smem);
    }
  }
  switch (tt) {
    case 1: return decode_launch_t<1, 1>(L, a, smem);
    case 2: return decode_launch_t<1, 2>(L, a, smem);
    default: return decode_launch_t<1, 4>(L, a, smem);
  }
}

cudaError_t decode_barrier_base(unsigned long long** p) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_decode_barrier);
}

// The smallest residency over the kernel's instantiations at the largest shared memory.
cudaError_t decode_occupancy(int* per_sm) {
  const void* kerns[6] = {
      reinterpret_cast<const void*>(ffn_decode_kernel<1, 1>),
      reinterpret_cast<const void*>(ffn_decode_kernel<1, 2>),
      reinterpret_cast<const void*>(ffn_decode_kernel<1, 4>),
      reinterpret_cast<const void*>(ffn_decode_kernel<2, 1>),
      reinterpret_cast<const void*>(ffn_decode_kernel<2, 2>),
      reinterpret_cast<const void*>(ffn_decode_kernel<2, 4>)};
  int best = 1 << 30;
  for (const void* k : kerns) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kDecodeMaxSmem));
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kDecThreads, kDecodeMaxSmem);
    if (e != cudaSuccess) return e;
    if (n < best) best = n;
  }
  *per_sm = best;
  return cudaSuccess;
}

}  // namespace fmlp
