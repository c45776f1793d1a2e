// Declarations shared between the host C-ABI translation unit and the kernel translation
// units. Host-only; no device code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace fmlp {

// Raises a kernel's dynamic shared-memory limit on the current device only when a call needs
// more than was set before (one cudaFuncSetAttribute per kernel and device in practice).
// Each launch site keeps its own cache object.
struct SmemAttrCache {
  std::atomic<int> bytes[64] = {};
};

inline cudaError_t set_smem_limit(const void* kern, int bytes, SmemAttrCache& cache) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < 64;
  if (cached && cache.bytes[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) {
    int cur = cache.bytes[dev].load(std::memory_order_relaxed);
    while (cur < bytes && !cache.bytes[dev].compare_exchange_weak(cur, bytes)) {
    }
  }
  return e;
}

// Epilogue kinds of the tcgen05 GEMM.
enum Epi : int {
  EPI_BIAS = 0,       // y = acc (+ bias)
  EPI_BIAS_GELU = 1,  // h = gelu(acc (+ bias))
  EPI_GEGLU = 2,      // m = gelu_tanh(acc_gate) * acc_up   (two B operands)
};

// One launch of the persistent tcgen05 GEMM: D[M, N] = A[M, K] B[N, K]^T with an epilogue.
struct GemmLaunch {
  CUtensorMap tmA;    // A  [M, K] bf16, box {64, 128}, 128B swizzle
  CUtensorMap tmB0;   // B  [N, K] bf16 (Wg for GeGLU), box {64, bn or bn/2}, 128B swizzle
  CUtensorMap tmB1;   // Wu for GeGLU (unused otherwise), box {64, bn/2}
  CUtensorMap tmY;    // output [M, N_out] bf16, box {64, 32}, 128B swizzle
  const void* bias;   // [N_out] bf16 or nullptr
  int M, N_out, K;
  int gelu_mode;      // 0 tanh, 1 erf
  int epi;            // Epi
  int bn;             // MMA N: 64, 128 or 256 (GeGLU: gate bn/2 + up bn/2)
  int grid;           // persistent CTAs
  bool pdl;           // launch as a programmatic dependent of the previous kernel
  cudaStream_t stream;
  int* status;        // device status word
  uint64_t timeout_ns;
  // Grouped (mixture-of-experts) launches only: A rows grouped by expert, [groups + 1]
  // device offsets; B maps are 3-D [groups, N, K]; the output goes to ydir (row stride ldy)
  // with direct stores.
  const int* offsets;
  int groups;
  void* ydir;
  int ldy;
  // Test hook (CTA-pair kernel): skip the loads of the first K step (see fmlp_test_inject).
  bool skip_first_load;
};
constexpr int kMoeMaxExperts = 256;

// A whole two-layer block in one persistent CTA-pair launch (gemm_tc2.cu, TWO): the first
// stage as a GemmLaunch (x, W1 or Wg+Wu, the intermediate as output), the second stage's maps,
// and the pairs' item lists.
constexpr int kTwoMaxItems = 2048;
constexpr int kTwoMaxPairs = 128;
constexpr int kTwoMaxBands = 64;            // 256-row bands: T up to 16384
struct TwoStageLaunch {
  CUtensorMap tmA2;   // the intermediate [M, K2] as A, box {64, 128}
  CUtensorMap tmB2;   // second-stage weights [N2, K2], box {64, 128}
  CUtensorMap tmY2;   // output [M, N2], box {64, 32}
  const void* bias2;  // [N2] or nullptr
  int slot;           // band-counter row (per stream; launches in one row must not overlap)
  int band_extra;     // test hook: added to the complete band count (1: never reached)
  int N2, K2;
  int n_items;        // items in `item` (first-stage tiles + second-stage tiles)
  int n1;             // first-stage tiles (band-major numbering), second-stage ones follow
  const uint16_t* start;   // [pairs + 1]: pair p runs item[start[p] .. start[p + 1])
  const uint16_t* item;    // [n_items]
};
cudaError_t gemm_tc2_two_launch(const GemmLaunch& L, const TwoStageLaunch& T2);

// Few-token tcgen05 GEMM (weights as the MMA's M side, K split over a cluster; gemm_skinny.cu).
constexpr int kSkinnyMaxT = 128;
struct SkinnyLaunch {
  CUtensorMap tmW0;   // weights [N, K] bf16, box {64, rows}, 128B swizzle (Wg for GeGLU)
  CUtensorMap tmW1;   // Wu for GeGLU (else a copy of tmW0)
  CUtensorMap tmX;    // x [T, K] bf16, box {64, tpad}, 128B swizzle
  const void* bias;   // [N] or nullptr
  void* y;            // [T, N] bf16
  int T, N, K;
  int ldy;            // row stride of y in elements
  int tpad;           // T rounded up to a multiple of 32 (the MMA's N)
  int rows;           // weight rows per tile: a multiple of 4, at most 128 (the MMA's M)
  int tiles;          // ceil(N / rows)
  int split;          // K slices per tile = cluster size: 1, 2, 4 or 8
  int epi, gelu_mode;
  bool pdl;           // programmatic dependent launch (second kernel of a block call)
  cudaStream_t stream;
  int* status;
  uint64_t timeout_ns;
};
cudaError_t gemm_skinny_launch(const SkinnyLaunch& L);

// Both layers of a few-token block in one launch (fewtoken_block.cu): layer 1 (x, W1 or
// Wg+Wu, bias1 + activation, or the GeGLU product) to h, a grid barrier, layer 2 (h, W2,
// bias2) to y, with the tiling of the few-token kernel shared by both layers (the same tiles
// and K split: rows1 and rows2 weight rows per tile).
struct FewBlockLaunch {
  CUtensorMap tmW1a, tmW1b;   // layer 1 weights [H, D], box {64, rows1}
  CUtensorMap tmX;            // x [T, D], box {64, tpad}
  CUtensorMap tmW2;           // layer 2 weights [Dout, H], box {64, rows2}
  CUtensorMap tmH;            // h [T, H], box {64, tpad}
  const void* b1;             // [H] or nullptr (GeGLU: unused)
  const void* b2;             // [Dout] or nullptr
  void* h;                    // [T, H] bf16 (the caller's workspace)
  void* y;                    // [T, Dout] bf16, row stride ldy
  unsigned long long* barrier;   // grid-barrier counter (shared with the decode plan's row)
  int T, D, H, Dout, ldy, tpad, rows1, rows2, tiles, split, epi1, gelu_mode;
  bool pdl;
  cudaStream_t stream;
  int* status;
  uint64_t timeout_ns;
};
cudaError_t fewtoken_block_launch(const FewBlockLaunch& L);
// Clusters of `split` CTAs of the few-token block kernel that can be resident at once.
cudaError_t fewtoken_block_max_clusters(int split, int* clusters);
// Ring stages of the launch (0: it does not fit), its shared memory and exchange-region bytes.
int fewtoken_block_stages(int nmat1, int tpad, int split, int rows1, int rows2, int* smem_out,
                          int* xbytes_out);

// Zero-padded copies (pad.cu): dst [dst_rows, dst_cols] (dst_cols a multiple of 8) takes
// src [rows, cols] (row stride ld) and zeros elsewhere; copy2d copies rows x cols between
// row strides.
cudaError_t pad2d_launch(const void* src, int64_t ld, int64_t rows, int64_t cols, void* dst,
                         int64_t dst_rows, int64_t dst_cols, cudaStream_t s);
cudaError_t copy2d_launch(const void* src, int64_t ld_src, void* dst, int64_t ld_dst,
                          int64_t rows, int64_t cols, cudaStream_t s);
// Clusters of `split` few-token CTAs that can be resident at once (the GPCs decide how many
// clusters of a size fit, not just the SM count).
cudaError_t gemm_skinny_max_clusters(int split, int* clusters);

cudaError_t gemm_tc_launch(const GemmLaunch& L);
// The single-SM kernel with the weights given as Wt [K, N_out] (N contiguous; tmB0 a map of
// Wt with a {64, 64} box), read as an MN-major operand; EPI_BIAS, bn 128 or 256.
cudaError_t gemm_tc_wt_launch(const GemmLaunch& L);
// The single-SM kernel over expert groups (bn 256; EPI_GEGLU or EPI_BIAS).
cudaError_t gemm_tc_grouped_launch(const GemmLaunch& L);
// CTA-pair (cta_group::2) kernel: 256 x 256 tiles over clusters of two CTAs; bn is 256;
// grid = 2 x pairs.
cudaError_t gemm_tc2_launch(const GemmLaunch& L);
cudaError_t gemm_tc2_max_pairs(int* pairs);
// The CTA-pair kernel over expert groups (bn 256; EPI_GEGLU or EPI_BIAS).
cudaError_t gemm_tc2_grouped_launch(const GemmLaunch& L);

// Weight-streaming GEMV for T <= kGemvMaxT tokens (decode; the plans use it for one or two).
constexpr int kGemvMaxT = 4;
// Shared memory holds x and the per-segment partial sums.
constexpr size_t kGemvMaxSmem = 200 * 1024;
struct GemvLaunch {
  const void* x;      // [T, K]
  const void* W0;     // [N, K]  (Wg for GeGLU)
  const void* W1;     // [N, K]  Wu for GeGLU, else unused
  const void* bias;   // [N] or nullptr
  void* y;            // [T, N]
  int T, K, N;
  int ldx, ldy;       // row strides of x and y in elements
  int epi;
  int gelu_mode;
  int grid;
  cudaStream_t stream;
};
// CTAs of the GEMV (nmat weight matrices of [N, K], T tokens) on a device with `sms` SMs.
int gemv_grid(int T, int K, int N, int nmat, int sms);
size_t gemv_smem_bytes(int T, int K, int N, int nmat, int grid);
cudaError_t gemv_launch(const GemvLaunch& L);

// The whole block (both layers) in one weight-streaming kernel for 1..kDecodeMaxT tokens
// (decode.cu): one CTA per SM, every CTA resident, weights streamed by bulk copies through a
// shared-memory ring, a bounded grid barrier between the layers.
constexpr int kDecodeMaxT = 4;
constexpr int kDecodeSlots = 1024;           // grid-barrier counters per device
constexpr size_t kDecodeMaxSmem = 227 * 1024;   // the opt-in shared memory of one CTA
struct DecodeLaunch {
  const void* x;      // [T, D], row stride ldx
  const void* W1a;    // [H, D]  W1 (MLP) or Wg (GeGLU)
  const void* W1b;    // [H, D]  Wu (GeGLU), else nullptr
  const void* b1;     // [H] or nullptr (MLP)
  const void* W2;     // [Dout, H]
  const void* b2;     // [Dout] or nullptr
  void* h;            // [T, H] workspace (the layer-1 output)
  void* y;            // [T, Dout], row stride ldy
  int T, D, H, Dout;
  int ldx, ldy;
  bool geglu;
  int gelu_mode;
  int grid;           // CTAs; all must be resident at once
  unsigned long long* barrier;   // this launch's grid-barrier counter
  int* status;
  uint64_t timeout_ns;
  cudaStream_t stream;
};
// Dynamic shared memory the decode kernel needs besides its ring (the token vectors and the
// per-warp row sums), and the ring stages (whole rows, about 8 KB each) that fit beside it
// within kDecodeMaxSmem (0: fewer than two; the plan then does not take the kernel).
size_t decode_smem_bytes(int T, int D, int H, int Dout, int nmat, int grid);
int decode_ring_stages(int T, int D, int H, int Dout, int nmat, int grid);
cudaError_t decode_launch(const DecodeLaunch& L);
// Device address of the first grid-barrier counter (slot i is at + 16 * i).
cudaError_t decode_barrier_base(unsigned long long** p);
// Resident CTAs per SM of the decode kernel (0: it cannot run on this device).
cudaError_t decode_occupancy(int* per_sm);

// Whole block in one kernel for small D and Dout (fused plan): the GeGLU block, or
// Linear -> act -> Linear with biases.
constexpr int kSmallMaxD = 256;
constexpr int kSmallMaxH = 2048;
struct SmallLaunch {
  CUtensorMap tmX;    // x  [T, D], box {64, 128}
  CUtensorMap tmWg;   // Wg or W1 [H, D], box {64, 64}
  CUtensorMap tmWu;   // Wu [H, D], box {64, 64} (GeGLU only)
  CUtensorMap tmWd;   // Wd or W2 [Dout, H], box {64, Dout}
  CUtensorMap tmY;    // y  [T, Dout], box {64, 32}
  const void* b1;     // [H] or nullptr (MLP only)
  const void* b2;     // [Dout] or nullptr (MLP only)
  int T, D, H, Dout;
  bool mlp;           // Linear -> act -> Linear (else GeGLU, Dout == D)
  int gelu_mode;
  int* status;
  uint64_t timeout_ns;
  cudaStream_t stream;
};
int ffn_small_smem_bytes(int D, int Dout);
cudaError_t ffn_small_launch(const SmallLaunch& L);

// Records the calling thread's fmlp_last_error() text (printf-style).
void record_error(const char* fmt, ...);

// The shape checks every block call starts with (T, then D, then H), as an fmlp_status value.
int validate_block_dims(int64_t T, int64_t D, int64_t H);

// Device GELU check kernel.
cudaError_t gelu_eval_launch(const float* in, float* out, int64_t n, int mode,
                             cudaStream_t stream);

// Bounded-wait test kernel.
cudaError_t wait_timeout_launch(uint64_t timeout_ns, int* status, cudaStream_t stream);

}  // namespace fmlp
