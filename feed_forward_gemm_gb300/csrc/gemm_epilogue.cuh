// Epilogue of the tcgen05 GEMM kernels: one warp turns its 32 TMEM lanes (32 output rows) of a
// finished accumulator into bf16 output tiles.
//
// Four epilogue warps share a tile: warp w reads TMEM lanes [32(w%4), 32(w%4)+32) (the quarter
// its position in the CTA allows) and all of the tile's output columns. (Eight warps with half
// the columns each were measured slower: they take issue slots from the single thread that
// issues the MMAs.)
//
// For each 64-column output chunk the warp loads the fp32 accumulator 32 columns at a time
// (tcgen05.ld 32x32b.x32: lane i holds row i), applies the epilogue in place, rounds once to
// bf16, writes the row into a 32x128-byte staging tile in the 128-byte swizzled layout
// (16-byte chunk j of row r goes to slot j ^ (r & 7), so eight consecutive lanes hit eight
// different bank groups) and lane 0 stores the tile with one TMA store. Two staging tiles
// alternate so the store of one chunk overlaps the math of the next.
//   EPI_BIAS       v = acc + b
//   EPI_BIAS_GELU  v = act(acc + b), act = GELU (tanh or erf) or ReLU
//   EPI_GEGLU      v = gelu_tanh(acc[c]) * acc[c + BN/2]  (gate columns, then up columns)
#pragma once

#include "activation.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fmlp {

constexpr int kStgBytes = 32 * 128;  // one staging tile: 32 rows x 64 bf16
constexpr int kEpiWarps = 4;
constexpr int kStgPerWarp = 2;       // staging tiles per epilogue warp (double buffer)

// a[i] += b[n0 + i] for 32 columns (b = 0 past N_out or without a bias: the +0 still turns an
// accumulator of -0 into +0, as a sum that starts from zero does), two at a time.
__device__ __forceinline__ void bias_pairs(uint32_t (&a)[32], const __nv_bfloat16* __restrict__ bias,
                                           int n0, int N_out) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (bias != nullptr && n0 + q * 8 < N_out)
      w = __ldg(reinterpret_cast<const uint4*>(bias + n0 + q * 8));
    const uint32_t wb[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = q * 8 + e * 2;
      float s0, s1;
      f2_unpack(f2_add(f2_pack(__uint_as_float(a[i]), __uint_as_float(a[i + 1])),
                       f2_pack(bf16_lo(wb[e]), bf16_hi(wb[e]))),
                s0, s1);
      a[i] = __float_as_uint(s0);
      a[i + 1] = __float_as_uint(s1);
    }
  }
}

// a[i] = gelu_tanh(a[i]) * u[i] for 32 values, two at a time (f32x2 arithmetic).
__device__ __forceinline__ void geglu_pairs(uint32_t (&a)[32], const uint32_t (&u)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint64_t g = f2_pack(__uint_as_float(a[i]), __uint_as_float(a[i + 1]));
    const uint64_t m =
        f2_mul(gelu_tanh_f2(g), f2_pack(__uint_as_float(u[i]), __uint_as_float(u[i + 1])));
    float m0, m1;
    f2_unpack(m, m0, m1);
    a[i] = __float_as_uint(m0);
    a[i + 1] = __float_as_uint(m1);
  }
}

// a[i] = act(a[i]) for 32 values (mode 0 GELU tanh, 1 GELU erf, 2 ReLU), the GELUs two at a
// time. The mode is chosen once per 32 values, so the evaluations are independent
// straight-line code the scheduler can overlap.
__device__ __forceinline__ void act_pairs(uint32_t (&a)[32], int mode) {
  if (mode == 2) {
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] = __float_as_uint(relu_f(__uint_as_float(a[i])));
    return;
  }
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint64_t v = f2_pack(__uint_as_float(a[i]), __uint_as_float(a[i + 1]));
    float y0, y1;
    f2_unpack(mode == 1 ? gelu_erf_f2(v) : gelu_tanh_f2(v), y0, y1);
    a[i] = __float_as_uint(y0);
    a[i + 1] = __float_as_uint(y1);
  }
}

// stg: this warp's kStgPerWarp staging tiles; sb: which one is next (kept across tiles).
template <int BN, int BN_OUT, int EPI>
__device__ __forceinline__ void epilogue_cols(uint32_t t_row, uint8_t* stg_base, int& sb,
                                              int lane, int row0, int n_tile0, int M,
                                              int N_out, const CUtensorMap* tmY,
                                              const __nv_bfloat16* __restrict__ bias,
                                              int gelu_mode) {
#pragma unroll 1
  for (int ch = 0; ch < BN_OUT; ch += 64) {
    const int n_chunk = n_tile0 + ch;
    uint8_t* stg = stg_base + sb * kStgBytes;
    // the TMA store that last read this staging tile must be done reading it
    if (lane == 0) bulk_wait_group_read<kStgPerWarp - 1>();
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = ch + h * 32;
      uint32_t a[32];
      tmem_ld_32x32b_x32(t_row + c, a);
      if (EPI == EPI_GEGLU) {
        uint32_t u[32];
        tmem_ld_32x32b_x32(t_row + BN / 2 + c, u);
        tmem_ld_wait();
        geglu_pairs(a, u);
      } else {
        tmem_ld_wait();
        bias_pairs(a, bias, n_chunk + h * 32, N_out);
        // the activation is chosen once per 32 columns, so the 32 evaluations are
        // independent straight-line code the scheduler can overlap
        if (EPI == EPI_BIAS_GELU) act_pairs(a, gelu_mode);
      }
      // 32 values = 4 x 16 bytes; 16-byte chunk j of this row goes to slot j ^ (row & 7)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = h * 4 + q;
        const uint32_t addr = smem_u32(stg) + static_cast<uint32_t>(lane * 128) +
                              static_cast<uint32_t>(((j ^ (lane & 7)) << 4));
        const uint32_t p0 = pack_bf16x2(__uint_as_float(a[q * 8 + 0]), __uint_as_float(a[q * 8 + 1]));
        const uint32_t p1 = pack_bf16x2(__uint_as_float(a[q * 8 + 2]), __uint_as_float(a[q * 8 + 3]));
        const uint32_t p2 = pack_bf16x2(__uint_as_float(a[q * 8 + 4]), __uint_as_float(a[q * 8 + 5]));
        const uint32_t p3 = pack_bf16x2(__uint_as_float(a[q * 8 + 6]), __uint_as_float(a[q * 8 + 7]));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(p0), "r"(p1),
                     "r"(p2), "r"(p3)
                     : "memory");
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (row0 < M && n_chunk < N_out) tma_store_2d(tmY, stg, n_chunk, row0);
      bulk_commit_group();
    }
    sb = (sb + 1) % kStgPerWarp;
  }
}

// The same epilogue for a grouped GEMM whose tiles may end inside the tile (the last rows of
// an expert's token group): each lane holds one output row and, when row_ok, stores its
// columns [n_tile0, n_tile0 + BN_OUT) straight to yrow (16-byte stores, columns past N_out
// skipped); rows past the group are computed but never written.
template <int BN, int BN_OUT, int EPI>
__device__ __forceinline__ void epilogue_rows_direct(uint32_t t_row, int lane, bool row_ok,
                                                     __nv_bfloat16* yrow, int n_tile0, int N_out,
                                                     const __nv_bfloat16* __restrict__ bias,
                                                     int gelu_mode) {
  (void)lane;
#pragma unroll 1
  for (int c = 0; c < BN_OUT; c += 32) {
    uint32_t a[32];
    tmem_ld_32x32b_x32(t_row + c, a);
    if (EPI == EPI_GEGLU) {
      uint32_t u[32];
      tmem_ld_32x32b_x32(t_row + BN / 2 + c, u);
      tmem_ld_wait();
      geglu_pairs(a, u);
    } else {
      tmem_ld_wait();
      bias_pairs(a, bias, n_tile0 + c, N_out);
      if (EPI == EPI_BIAS_GELU) act_pairs(a, gelu_mode);
    }
    if (row_ok) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = n_tile0 + c + q * 8;
        if (n < N_out) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(a[q * 8 + 0]), __uint_as_float(a[q * 8 + 1]));
          v.y = pack_bf16x2(__uint_as_float(a[q * 8 + 2]), __uint_as_float(a[q * 8 + 3]));
          v.z = pack_bf16x2(__uint_as_float(a[q * 8 + 4]), __uint_as_float(a[q * 8 + 5]));
          v.w = pack_bf16x2(__uint_as_float(a[q * 8 + 6]), __uint_as_float(a[q * 8 + 7]));
          *reinterpret_cast<uint4*>(yrow + n) = v;
        }
      }
    }
  }
}

}  // namespace fmlp
