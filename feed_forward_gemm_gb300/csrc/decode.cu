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
//   - one producer thread streams the CTA's weight rows, layer 1 then layer 2, with 1-D bulk
//     copies (cp.async.bulk) into a ring of shared-memory stages of about 8 KB (whole rows;
//     for GeGLU the same rows of Wg and Wu share a stage), each stage completing on its own
//     mbarrier. The ring takes nearly all of the CTA's shared memory (216 KB for the 4096-wide
//     MLP at one token: a CTA's whole share of a layer), so the whole of layer 1 is requested
//     at once without holding a single register; as the consumers free stages the producer
//     refills them with layer-2 rows, which stream in while the CTAs meet at the grid barrier;
//   - 16 consumer warps in groups (a row's 16-byte chunks spread over a group's lanes: the
//     whole CTA for 4096-wide rows); ring slot i belongs to group i mod groups. A group takes
//     its rows in batches (rows x matrices x tokens = 8 sums): it waits for the batch's
//     stages, sums its chunks of all the batch's rows with packed f32x2 multiply-adds (x, held
//     in shared memory as fp32, read once per batch), reduces the batch over the warp by
//     recursive halving and frees the stages; the warps' partial sums meet in a fixed order
//     once the layer is done (deterministic). Spreading each row over many warps keeps the
//     rows that land last from waiting on one warp's long dependency chain;
//   - layer-1 outputs h go to the caller's workspace; a grid barrier (a counter in device
//     memory, one atomic per CTA, waited on with a bounded poll) makes every h row visible
//     before the token vectors are reloaded with h for layer 2.
// Every input, weights included, is read only after the dependency wait, so a kernel queued
// just before may have written any of them.
//
// Failure handling: every wait is bounded (the stage mbarriers and the grid barrier). A wait
// that runs out records the site in the device status word and the CTA's output is undefined.
// The producer issues nothing after a wait of its own runs out, and a consumer hands a stage
// back only once its copy has landed, so no stage is reused under a copy in flight; the
// consumers still wait (bounded) for every stage, so no copy issued can still be writing into
// the CTA's shared memory when it exits; nothing spins without a limit. The barrier counter
// needs no reset: CTA b adds w_b = floor((b+1) 2^20 / G) - floor(b 2^20 / G) (the G weights
// sum to 2^20), so the counter is a multiple of 2^20 between launches and each launch waits
// for the next multiple; every CTA adds its weight exactly once, even one whose wait runs out.
#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

// Grid-barrier counters, kDecodeSlots of them 128 bytes apart, zero when the module loads.
__device__ unsigned long long g_decode_barrier[kDecodeSlots * 16];

namespace {

constexpr int kDecConsumers = 512;                 // 16 consumer warps
constexpr int kDecWarps = kDecConsumers / 32;
constexpr int kDecThreads = kDecConsumers + 32;    // + the producer warp
constexpr unsigned long long kBarrierUnit = 1ull << 20;
constexpr int kMaxStages = 64;      // ring stages (each a whole number of rows, about 8 KB)
constexpr int kStageTarget = 8192;

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

// 1-D bulk copy global -> this CTA's shared memory, completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Named barrier of the 512 consumer threads (the producer warp never takes part).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecConsumers) : "memory");
}

// Arrive on `bar` with `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Warp sums of N values per lane (N a power of two, 1..32) by recursive halving: at the
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
      for (int i = 0; i < (N > 1 ? N / 2 : 1); ++i) {
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

// How the consumer warps cover rows of K elements (C = K / 8 chunks of 16 bytes): groups of
// wg warps (wg the smallest power of two with 32 wg >= C, at most 16), each group on its own
// ring slots; thread q of a group (q < 32 wg) sums chunks q, q + 32 wg, ... of every row of
// the group's stages, so a row is spread over all the group's warps.
struct KSplit {
  int C, wg, gt, groups, nch;
};

__host__ __device__ inline KSplit make_ksplit(int K) {
  KSplit s;
  s.C = K / 8;
  s.wg = 1;
  while (s.wg < kDecWarps && s.wg * 32 < s.C) s.wg <<= 1;
  s.gt = s.wg * 32;
  s.groups = kDecWarps / s.wg;
  s.nch = (s.C + s.gt - 1) / s.gt;
  return s;
}

// Rows of a reduction batch: the batch's rows x NMAT x TT sums make 8 values.
template <int NMAT, int TT>
constexpr int batch_rows() { return 8 / (NMAT * TT) > 0 ? 8 / (NMAT * TT) : 1; }

// Token vectors in shared memory as fp32, split by halves of the 16-byte chunks: for a row of
// K elements (C = K / 8 chunks), token t's chunk c is lo[t][c] = elements 8c..8c+3 and
// hi[t][c] = 8c+4..8c+7, at float4 index t * 2C + c and t * 2C + C + c, so that the lanes of
// a warp, on consecutive chunks, read consecutive 16-byte words (no bank conflicts). Widening
// once here spares every row the conversion of x.
__device__ __forceinline__ void stage_vectors(float4* vec, const __nv_bfloat16* src, int T, int K,
                                              int ld) {
  const int C = K / 8;
  for (int i = threadIdx.x; i < T * C; i += kDecConsumers) {
    const int t = i / C, c = i - t * C;
    const uint4 v = ldg_cg(src + static_cast<size_t>(t) * ld + static_cast<size_t>(c) * 8);
    vec[t * 2 * C + c] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    vec[t * 2 * C + C + c] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
  }
}

// Rows a stage of `stage_bytes` holds for rows of K elements of NMAT matrices (the stage is
// split evenly between the matrices).
__host__ __device__ inline int stage_rows(int K, int nmat, int stage_bytes) {
  return stage_bytes / (nmat * K * 2);
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
  int stages;                // ring stages
  int stage_bytes;           // bytes per stage (whole rows of either layer)
  int rows_max;              // rows per CTA in either layer (size of the row-sum buffer)
  int vec_bytes;             // shared bytes of the token vectors (T * max(D, H) * 4)
};

// One layer's share of the ring traffic for a CTA: rows [0, nrows) of NMAT matrices (row j of
// matrix m at Wm + j * K), `rps` rows per stage; row j is output row0 + j of the layer.
struct LayerPlan {
  const __nv_bfloat16* W0;
  const __nv_bfloat16* W1;
  int K, nrows, rps, nstages, row0;
};

__device__ __forceinline__ LayerPlan make_layer(const __nv_bfloat16* W0, const __nv_bfloat16* W1,
                                                int K, int nrows, int row0, int nmat,
                                                int stage_bytes) {
  LayerPlan L;
  L.W0 = W0;
  L.W1 = W1;
  L.K = K;
  L.nrows = nrows;
  L.row0 = row0;
  L.rps = stage_rows(K, nmat, stage_bytes);
  L.nstages = nrows > 0 ? (nrows + L.rps - 1) / L.rps : 0;
  return L;
}

// The producer: every stage of both layers, in order, into the ring. Waits are bounded; once
// one runs out nothing more is issued (the consumers' bounded waits for the stages never
// issued run out in turn), so no stage is re-armed before its previous copy was consumed.
__device__ __forceinline__ void produce(uint8_t* ring, uint64_t* full, uint64_t* empty,
                                        int nstage_ring, const LayerPlan& L1, int nmat1,
                                        const LayerPlan& L2, const DecodeArgs& a) {
  int slot = 0;
  uint32_t phase = 0;
  bool ok = true;
  auto run = [&](const LayerPlan& L, int nmat) {
    for (int s = 0; s < L.nstages && ok; ++s) {
      if (!mbar_wait_sleep(&empty[slot], phase ^ 1u, a.status, SITE_DECODE_W2, a.timeout_ns)) {
        ok = false;
        break;
      }
      const int j0 = s * L.rps;
      const int n = L.nrows - j0 < L.rps ? L.nrows - j0 : L.rps;
      const uint32_t bytes = static_cast<uint32_t>(n) * static_cast<uint32_t>(L.K) * 2u;
      const uint32_t dst = smem_u32(ring + static_cast<size_t>(slot) * a.stage_bytes);
      mbar_arrive_expect_tx(&full[slot], bytes * static_cast<uint32_t>(nmat));
      bulk_g2s(dst, L.W0 + static_cast<size_t>(j0) * L.K, bytes, &full[slot]);
      if (nmat == 2)
        bulk_g2s(dst + a.stage_bytes / 2, L.W1 + static_cast<size_t>(j0) * L.K, bytes,
                 &full[slot]);
      if (++slot == nstage_ring) {
        slot = 0;
        phase ^= 1u;
      }
    }
  };
  run(L1, nmat1);
  run(L2, 1);
}

// Layer epilogues: the value stored for output row n of token t from its row sums.
template <int NMAT>
__device__ __forceinline__ float layer1_out(const DecodeArgs& a, int n, float s0, float s1) {
  if (NMAT == 2) return gelu_tanh_f(s0) * s1;
  return gelu_f(s0 + (a.b1 != nullptr ? __bfloat162float(a.b1[n]) : 0.f), a.gelu_mode);
}

// One layer on the consumer side. Ring slot i belongs to warp group i mod groups (the ring
// length is a multiple of every layer's group count), so every fill of a slot is consumed by
// the same warps, in order: an mbarrier phase parity tells only the phase right after the last
// one its waiter saw, so a warp must never wait for fill k of a slot before fill k - 1 of it
// has completed. A group walks the rows of its stages (stage s_k = s_first + k groups, rows
// p = k rps + r) in batches of R rows: it waits for the batch's stages, each thread sums its
// chunks of the batch's rows (the chunk of x is read once for all R rows; the R NMAT weight
// chunks are loaded before any arithmetic; packed f32x2 multiply-adds), one recursive-halving
// reduction per batch leaves the warp's partial sums in red[((warp * rows_max + j) * NMAT +
// m) * TT + t] for layer row j, and the stages whose rows are all done go back to the
// producer (each of the wg warps arrives with 16 / wg, so a stage's release always counts 16).
// A row is thus spread over all the group's warps: the rows that land last are summed by
// many warps at once. Returns false if one of the warp's waits ran out.
template <int NMAT, int TT>
__device__ __forceinline__ bool consume(const uint8_t* ring, uint64_t* full, uint64_t* empty,
                                        int nstage_ring, int g0, const LayerPlan& L,
                                        const float4* vec, float* red, const DecodeArgs& a) {
  constexpr int R = batch_rows<NMAT, TT>();
  constexpr int NV = R * NMAT * TT;
  constexpr int SH = 5 - log2_const(NV);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const KSplit ks = make_ksplit(L.K);
  const int G = ks.groups, S = nstage_ring;
  const int g = warp / ks.wg;
  const int q = (warp - g * ks.wg) * 32 + lane;
  const int s_first = ((g - g0 % G) % G + G) % G;
  const int nk = s_first < L.nstages ? (L.nstages - s_first + G - 1) / G : 0;
  // rows per batch: R, or fewer when the group owns few slots. A batch waits for all its
  // stages before freeing any, and the producer refills a slot only once it is freed, so a
  // batch may span at most the group's own slots (S / G of them); with Rb at most
  // rps (owned - 1) + 1 rows it spans at most owned stages.
  const int owned = S / G;
  const int Rb = R < L.rps * (owned - 1) + 1 ? R : L.rps * (owned - 1) + 1;
  const uint32_t half = NMAT == 2 ? a.stage_bytes / 2 : 0;
  const uint32_t row_bytes = static_cast<uint32_t>(L.K) * 2u;
  const uint32_t ring0 = smem_u32(ring);
  const uint32_t xlo = smem_u32(vec), xhi = xlo + static_cast<uint32_t>(ks.C) * 16u;
  const uint32_t xtok = static_cast<uint32_t>(ks.C) * 32u;   // bytes per token
  const uint32_t rel = static_cast<uint32_t>(kDecWarps / ks.wg);
  // Cursors, advanced by additions only (a division by a run-time value costs tens of
  // instructions; in the inner loops it cost more than the arithmetic). The group's k-th stage
  // is layer stage s_first + k G, ring stage g0 + s_first + k G, in slot (that) mod S; the slot
  // advances by G and wraps at S (S is a multiple of G), the fill parity flipping on a wrap.
  const int gfirst = g0 + s_first;
  int w_slot = gfirst % S;
  uint32_t w_par = static_cast<uint32_t>(gfirst / S) & 1u;
  int r_slot = w_slot;
  int k_wait = 0, k_rel = 0;
  // batch cursor: stage k, row r within it, layer stage s, slot
  int bk = 0, br = 0, bs = s_first, bslot = w_slot;
  bool ok = true;
  while (bk < nk) {
    // the batch's rows: base address in shared memory (0: no row) and layer row index
    uint32_t rb[R];
    int jr[R];
    int k_last = bk;
    {
      int k = bk, r = br, st = bs, sl = bslot;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int rows_left = L.nrows - st * L.rps;
        const int n = k < nk ? (rows_left < L.rps ? rows_left : L.rps) : 0;
        const bool valid = i < Rb && r < n;
        rb[i] = valid ? ring0 + static_cast<uint32_t>(sl) * static_cast<uint32_t>(a.stage_bytes) +
                            static_cast<uint32_t>(r) * row_bytes
                      : 0u;
        jr[i] = valid ? st * L.rps + r : -1;
        if (valid) k_last = k;
        if (i < Rb) {
          if (++r == L.rps) {
            r = 0;
            ++k;
            st += G;
            sl += G;
            if (sl >= S) sl -= S;
          }
        }
      }
      bk = k;
      br = r;
      bs = st;
      bslot = sl;
    }
    // bounded; after a failure the later waits still run, so every copy issued has landed
    // before the CTA exits, and no stage goes back to the producer after a failed wait
    for (; k_wait <= k_last && k_wait < nk; ++k_wait) {
      if (!mbar_wait_sleep(&full[w_slot], w_par, a.status, SITE_DECODE_W2, a.timeout_ns))
        ok = false;
      w_slot += G;
      if (w_slot >= S) {
        w_slot -= S;
        w_par ^= 1u;
      }
    }
    float2 acc[NV];
#pragma unroll
    for (int f = 0; f < NV; ++f) acc[f] = make_float2(0.f, 0.f);
    for (int c = 0; c < ks.nch; ++c) {
      const int chunk = q + c * ks.gt;
      if (chunk >= ks.C) break;
      // x first (per token), then each row's weight chunks (the loads of all rows are free to
      // run ahead: they depend on nothing computed here)
      float4 xa[TT], xb[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        if (t < a.T) {
          xa[t] = lds_f4(xlo + t * xtok + static_cast<uint32_t>(chunk) * 16u);
          xb[t] = lds_f4(xhi + t * xtok + static_cast<uint32_t>(chunk) * 16u);
        } else {
          xa[t] = xb[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < R; ++i) {
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const uint4 w = rb[i] != 0u ? lds_v4(rb[i] + m * half + static_cast<uint32_t>(chunk) * 16u)
                                      : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int t = 0; t < TT; ++t) {
            if (t < a.T) {
              float2& d = acc[(i * NMAT + m) * TT + t];
              ffma2(d, bf16_lo(w.x), bf16_hi(w.x), xa[t].x, xa[t].y);
              ffma2(d, bf16_lo(w.y), bf16_hi(w.y), xa[t].z, xa[t].w);
              ffma2(d, bf16_lo(w.z), bf16_hi(w.z), xb[t].x, xb[t].y);
              ffma2(d, bf16_lo(w.w), bf16_hi(w.w), xb[t].z, xb[t].w);
            }
          }
        }
      }
    }
    float v[NV];
#pragma unroll
    for (int f = 0; f < NV; ++f) v[f] = acc[f].x + acc[f].y;
    warp_sum_many<NV>(v, lane);
    if ((lane & ((1 << SH) - 1)) == 0) {
      const int f = lane >> SH;
      const int t = f % TT, m = (f / TT) % NMAT, i = f / (TT * NMAT);   // compile-time divisors
      int j = -1;
#pragma unroll
      for (int ii = 0; ii < R; ++ii)
        if (ii == i) j = jr[ii];
      if (t < a.T && j >= 0) red[((warp * a.rows_max + j) * NMAT + m) * TT + t] = v[0];
    }
    // stages all of whose rows are done (those before the cursor) go back to the producer
    const bool all_ok = __all_sync(0xffffffffu, ok);
    for (; k_rel < bk && k_rel < k_wait; ++k_rel) {
      if (lane == 0 && all_ok) mbar_arrive_cnt(&empty[r_slot], rel);
      r_slot += G;
      if (r_slot >= S) r_slot -= S;
    }
  }
  const bool all_ok = __all_sync(0xffffffffu, ok);
  for (; k_rel < k_wait; ++k_rel) {
    if (lane == 0 && all_ok) mbar_arrive_cnt(&empty[r_slot], rel);
    r_slot += G;
    if (r_slot >= S) r_slot -= S;
  }
  return ok;
}

// Sum of layer row j (matrix m, token t) over the warps of the group that owns its stage, in
// warp order (deterministic).
template <int NMAT, int TT>
__device__ __forceinline__ float row_sum(const float* red, const LayerPlan& L, int g0,
                                         int rows_max, int j, int m, int t) {
  const KSplit ks = make_ksplit(L.K);
  const int g = (g0 + j / L.rps) % ks.groups;
  float v = 0.f;
  for (int w = g * ks.wg; w < (g + 1) * ks.wg; ++w)
    v += red[((w * rows_max + j) * NMAT + m) * TT + t];
  return v;
}

__device__ __forceinline__ int split_at(int i, int n) {
  return static_cast<int>((static_cast<int64_t>(i) * n) / gridDim.x);
}

template <int NMAT, int TT>
__global__ void __launch_bounds__(kDecThreads, 1) ffn_decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  const int T = a.T, D = a.D, H = a.H;
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  // this CTA's rows of each layer
  const int r0 = split_at(b, H), nr1 = split_at(b + 1, H) - r0;
  const int c0 = split_at(b, a.Dout), nr2 = split_at(b + 1, a.Dout) - c0;
  const LayerPlan L1 = make_layer(a.W1a + static_cast<size_t>(r0) * D,
                                  NMAT == 2 ? a.W1b + static_cast<size_t>(r0) * D : nullptr, D,
                                  nr1, r0, NMAT, a.stage_bytes);
  const LayerPlan L2 = make_layer(a.W2 + static_cast<size_t>(c0) * H, nullptr, H, nr2, c0, 1,
                                  a.stage_bytes);

  uint8_t* ring = dsm;
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + static_cast<size_t>(a.stages) * a.stage_bytes);
  uint64_t* empty = full + a.stages;
  float4* vec = reinterpret_cast<float4*>(empty + a.stages);
  float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(vec) + a.vec_bytes);
  int* flag = reinterpret_cast<int*>(red + kDecWarps * a.rows_max * NMAT * TT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecWarps);
    }
    *flag = 1;
    fence_mbarrier_init();
  }
  __syncthreads();
  // every input (x, all weights and biases) may come from the kernel queued before this one
  pdl_wait_primary();
  // every CTA of this grid is resident once all of them got here: the next kernel may launch
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (threadIdx.x >= kDecConsumers) {
    // ------------------------------------------------------------------ producer warp
    if (threadIdx.x == kDecConsumers) produce(ring, full, empty, a.stages, L1, NMAT, L2, a);
    return;
  }

  // -------------------------------------------------------------------- consumers
  stage_vectors(vec, a.x, T, D, a.ldx);
  consumers_sync();
  bool ok = consume<NMAT, TT>(ring, full, empty, a.stages, 0, L1, vec, red, a);
  consumers_sync();
  for (int e = threadIdx.x; e < nr1 * T; e += kDecConsumers) {
    const int t = e / nr1, j = e - t * nr1;
    const float v = layer1_out<NMAT>(a, r0 + j, row_sum<NMAT, TT>(red, L1, 0, a.rows_max, j, 0, t),
                                     row_sum<NMAT, TT>(red, L1, 0, a.rows_max, j, NMAT - 1, t));
    a.h[static_cast<size_t>(t) * H + r0 + j] = __float2bfloat16_rn(v);
  }
  // ------------------------------------------------------------------ grid barrier
  consumers_sync();   // this CTA's h stores are issued; the vectors and row sums are free
  if (threadIdx.x == 0) {
    // the release of the atomic, after the CTA barrier above, publishes this CTA's h
    const unsigned long long mine = (static_cast<unsigned long long>(b + 1) * kBarrierUnit) / G -
                                    (static_cast<unsigned long long>(b) * kBarrierUnit) / G;
    const unsigned long long old = atom_add_acq_rel(a.barrier, mine);
    const unsigned long long target = (old / kBarrierUnit + 1ull) * kBarrierUnit;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire(a.barrier) < target) {
      if (globaltimer_ns() - t0 > a.timeout_ns) {
        atomicCAS(a.status, 0, (SITE_DECODE_BARRIER << 8) | kDeviceTimeoutCode);
        *flag = 0;
        break;
      }
      __nanosleep(20);
    }
  }
  consumers_sync();
  if (*flag) stage_vectors(vec, a.h, T, H, H);
  consumers_sync();
  // ------------------------------------------------------------------ layer 2
  // after a barrier timeout the vectors still hold x: y is then undefined (the status word
  // says so), but every read stays inside the vectors' T * max(D, H) elements
  ok = consume<1, TT>(ring, full, empty, a.stages, L1.nstages, L2, vec, red, a) && ok;
  if (!ok) atomicExch(flag, 0);
  consumers_sync();
  if (*flag) {
    for (int e = threadIdx.x; e < nr2 * T; e += kDecConsumers) {
      const int t = e / nr2, j = e - t * nr2;
      const float z = row_sum<1, TT>(red, L2, L1.nstages, a.rows_max, j, 0, t) +
                      (a.b2 != nullptr ? __bfloat162float(a.b2[c0 + j]) : 0.f);
      a.y[static_cast<size_t>(t) * a.ldy + c0 + j] = __float2bfloat16_rn(z);
    }
  }
  (void)ok;
}

int tt_of(int T) { return T <= 1 ? 1 : (T <= 2 ? 2 : 4); }

}  // namespace

// Shared memory of the decode kernel besides its ring: the token vectors (fp32), the per-warp
// row sums and the flag.
size_t decode_smem_bytes(int T, int D, int H, int Dout, int nmat, int grid) {
  const int rows_max = ((H > Dout ? H : Dout) + grid - 1) / grid;
  const size_t vec = static_cast<size_t>(T) * (D > H ? D : H) * 4;
  const size_t red = static_cast<size_t>(kDecWarps) * rows_max * nmat * tt_of(T) * 4;
  return vec + red + 16;
}

// Bytes per ring stage: a whole number of rows of either layer (NMAT matrices for layer 1),
// about 8 KB, so that the ring holds as many rows as shared memory allows.
// The row is rounded up to 32 bytes so that a GeGLU stage's second half (the Wu rows) starts
// on the 16-byte boundary a bulk copy needs.
int decode_stage_bytes(int D, int H, int nmat) {
  int row = nmat * D * 2 > H * 2 ? nmat * D * 2 : H * 2;
  row = (row + 31) / 32 * 32;
  return row * (kStageTarget / row > 1 ? kStageTarget / row : 1);
}

// Ring stages that fit beside the rest (at most kMaxStages), a multiple of both layers' warp
// group counts (each slot must belong to one group in either layer); 0 when fewer than two.
int decode_ring_stages(int T, int D, int H, int Dout, int nmat, int grid) {
  const size_t sb = static_cast<size_t>(decode_stage_bytes(D, H, nmat));
  const size_t base = decode_smem_bytes(T, D, H, Dout, nmat, grid);
  if (base + 2 * (sb + 16) > kDecodeMaxSmem) return 0;
  size_t st = (kDecodeMaxSmem - base) / (sb + 16);
  if (st > kMaxStages) st = kMaxStages;
  const int g1 = make_ksplit(D).groups, g2 = make_ksplit(H).groups;
  const size_t gmax = static_cast<size_t>(g1 > g2 ? g1 : g2);
  st -= st % gmax;
  return st >= 2 ? static_cast<int>(st) : 0;
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
  const int stages = decode_ring_stages(L.T, L.D, L.H, L.Dout, nmat, L.grid);
  if (stages < 2) return cudaErrorInvalidValue;
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
  a.stages = stages;
  a.stage_bytes = decode_stage_bytes(L.D, L.H, nmat);
  a.rows_max = ((L.H > L.Dout ? L.H : L.Dout) + L.grid - 1) / L.grid;
  a.vec_bytes = L.T * (L.D > L.H ? L.D : L.H) * 4;
  const size_t smem = static_cast<size_t>(stages) * (a.stage_bytes + 16) +
                      decode_smem_bytes(L.T, L.D, L.H, L.Dout, nmat, L.grid);
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

// The smallest residency over the kernel's instantiations (registers and threads decide it;
// each launch raises the kernel's shared-memory limit to what it needs).
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
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kDecThreads, 0);
    if (e != cudaSuccess) return e;
    if (n < best) best = n;
  }
  *per_sm = best;
  return cudaSuccess;
}

}  // namespace fmlp
