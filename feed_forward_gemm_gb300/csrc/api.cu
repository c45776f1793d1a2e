// Host side of the C ABI declared in include/fmlp.h: argument validation, plan choice,
// tensor-map encoding and launches on the caller's stream.
//
// Dispatch follows the lesson of "Profiling in PyTorch (Part 2): From nn.Linear to a Fused
// MLP" (sections "Stacking three Linears: the MLP" and "Why tuned kernels are better"): no
// per-call occupancy query (the SM count is cached once per device), one shape-generic binary
// whose tile shape is picked at run time from a small cost model, no recompilation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/fmlp.h"
#include "internal.h"

namespace fmlp {

// Per-device status word written by kernels that give up on a bounded wait.
__device__ int g_device_status;

namespace {

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s per wait

bool act_mode_ok(int mode) {
  return mode == FMLP_GELU_TANH || mode == FMLP_GELU_ERF || mode == FMLP_RELU;
}
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = 2147483647;

thread_local std::string t_last_error;

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
}

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int major = 0, minor = 0;
  int max_pairs = 0;   // co-resident CTA pairs of the pair GEMM (0: pair kernel unavailable)
  // co-resident clusters of 1, 2, 4, 8 few-token CTAs (0: unknown, assume sms / size)
  int skinny_clusters[4] = {0, 0, 0, 0};
  // co-resident clusters of 1, 2, 4, 8 CTAs of the few-token block kernel (0: unknown: the
  // one-launch block is not taken)
  int fewblock_clusters[4] = {0, 0, 0, 0};
  int* status = nullptr;
  int decode_occ = 0;  // resident decode CTAs per SM (0: the one-kernel decode cannot run)
  unsigned long long* decode_bar = nullptr;  // grid-barrier counters (kDecodeSlots)
  // Stream i of this table uses counter i (a fixed table: assigning one allocates nothing).
  cudaStream_t decode_stream[kDecodeSlots] = {};
  int decode_streams = 0;
};

// Test hook of the one-kernel decode: extra CTAs beyond the resident ones, and the wait limit.
std::atomic<int> g_decode_extra_ctas{0};
// Whether blocks of 1..4 tokens take the one-kernel decode when it accepts the shape (off:
// the two-launch plans, measured faster on GB300; see fmlp_test_prefer_decode).
std::atomic<int> g_prefer_decode{0};
std::atomic<unsigned long long> g_decode_timeout_ns{0};

// Failure-injection test hooks (fmlp_test_inject): launches left to fail on the host, CTA-pair
// GEMM launches left to skip their first loads, and the wait limit of those launches.
std::atomic<int> g_inject_launch{0};
std::atomic<int> g_inject_skip{0};
std::atomic<unsigned long long> g_inject_timeout_ns{0};

// Takes one unit of an injection counter (true if one was left).
bool take_injection(std::atomic<int>& n) {
  int v = n.load(std::memory_order_relaxed);
  while (v > 0 && !n.compare_exchange_weak(v, v - 1)) {
  }
  return v > 0;
}

std::atomic<int> g_tile_policy{FMLP_TILES_AUTO};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

fmlp_status cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return FMLP_ERR_CUDA;
}

// Every kernel launch goes through here first: an injected failure (test hook) stands in for
// a launch that the runtime refused, and nothing is launched.
#define FMLP_LAUNCH_GUARD(what)                                                   \
  do {                                                                            \
    if (take_injection(g_inject_launch)) {                                        \
      set_error("%s: injected launch failure (fmlp_test_inject)", what);         \
      return FMLP_ERR_CUDA;                                                       \
    }                                                                             \
  } while (0)

// Current device's cached state; checks the architecture once.
fmlp_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal %d out of range", dev);
    return FMLP_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) !=
        cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(major)");
    if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
        cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
    if (d.major != 10 || d.minor != 3) {
      set_error("device %d is compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                dev, d.major, d.minor);
      return FMLP_ERR_DEVICE;
    }
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(status)");
    d.status = static_cast<int*>(p);
    if (gemm_tc2_max_pairs(&d.max_pairs) != cudaSuccess) {
      d.max_pairs = 0;
      (void)cudaGetLastError();
    }
    for (int i = 0; i < 4; ++i) {
      if (gemm_skinny_max_clusters(1 << i, &d.skinny_clusters[i]) != cudaSuccess) {
        d.skinny_clusters[i] = 0;
        (void)cudaGetLastError();
      }
      if (fewtoken_block_max_clusters(1 << i, &d.fewblock_clusters[i]) != cudaSuccess) {
        d.fewblock_clusters[i] = 0;
        (void)cudaGetLastError();
      }
    }
    if (decode_occupancy(&d.decode_occ) != cudaSuccess ||
        decode_barrier_base(&d.decode_bar) != cudaSuccess) {
      d.decode_occ = 0;
      d.decode_bar = nullptr;
      (void)cudaGetLastError();
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        set_error("cuTensorMapEncodeTiled unavailable from the driver");
        return FMLP_ERR_CUDA;
      }
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return FMLP_OK;
}

// Encoded tensor maps, process-wide. A map is a pure function of (address, sizes, strides,
// box), all of which are in the key, so an entry never goes stale: a buffer freed and
// reallocated at the same address with the same sizes gets the same, still correct, map.
// Direct-mapped, kMapCacheSlots entries; a colliding key simply re-encodes and replaces.
constexpr int kMapCacheSlots = 1024;
struct MapKey {
  uintptr_t ptr;
  uint64_t depth, rows, cols, ld;
  uint32_t box_rows;
  uint32_t rank;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && depth == o.depth && rows == o.rows && cols == o.cols && ld == o.ld &&
           box_rows == o.box_rows && rank == o.rank;
  }
};
struct MapEntry {
  bool valid = false;
  MapKey key{};
  CUtensorMap map;
};
std::mutex g_map_mu;
MapEntry g_maps[kMapCacheSlots];

size_t map_slot(const MapKey& k) {
  uint64_t h = static_cast<uint64_t>(k.ptr) * 0x9E3779B97F4A7C15ull;
  for (uint64_t v : {k.depth, k.rows, k.cols, k.ld, static_cast<uint64_t>(k.box_rows) << 8 | k.rank})
    h = (h ^ v) * 0xBF58476D1CE4E5B9ull;
  return static_cast<size_t>(h >> 40) % kMapCacheSlots;
}

bool map_lookup(const MapKey& k, CUtensorMap* m) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  const MapEntry& e = g_maps[map_slot(k)];
  if (!e.valid || !(e.key == k)) return false;
  *m = e.map;
  return true;
}

void map_store(const MapKey& k, const CUtensorMap& m) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry& e = g_maps[map_slot(k)];
  e.valid = true;
  e.key = k;
  e.map = m;
}

// Row-major bf16 matrix [rows, cols] -> 2-D tensor map with a {64, box_rows} box, 128B swizzle.
// ld: row stride in elements (0: rows are packed, ld = cols).
fmlp_status make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols,
                     uint32_t box_rows, const char* name, int64_t ld = 0) {
  const MapKey key{reinterpret_cast<uintptr_t>(ptr), 1, static_cast<uint64_t>(rows),
                   static_cast<uint64_t>(cols), static_cast<uint64_t>(ld > 0 ? ld : cols),
                   box_rows, 2};
  if (map_lookup(key, m)) return FMLP_OK;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld > 0 ? ld : cols) * 2u};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t es[2] = {1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled(%s [%lld x %lld], box %u rows) failed with CUresult %d",
              name, static_cast<long long>(rows), static_cast<long long>(cols), box_rows,
              static_cast<int>(r));
    return FMLP_ERR_CUDA;
  }
  map_store(key, *m);
  return FMLP_OK;
}

// A 3-D map over [depth, rows, cols] bf16 (packed), box {64, box_rows, 1}, 128-byte swizzle.
fmlp_status make_map3(CUtensorMap* m, const void* ptr, int64_t depth, int64_t rows, int64_t cols,
                      uint32_t box_rows, const char* name) {
  const MapKey key{reinterpret_cast<uintptr_t>(ptr), static_cast<uint64_t>(depth),
                   static_cast<uint64_t>(rows), static_cast<uint64_t>(cols),
                   static_cast<uint64_t>(cols), box_rows, 3};
  if (map_lookup(key, m)) return FMLP_OK;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(depth)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2u,
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(cols) * 2u};
  cuuint32_t box[3] = {64u, box_rows, 1u};
  cuuint32_t es[3] = {1u, 1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled(%s [%lld x %lld x %lld]) failed with CUresult %d", name,
              static_cast<long long>(depth), static_cast<long long>(rows),
              static_cast<long long>(cols), static_cast<int>(r));
    return FMLP_ERR_CUDA;
  }
  map_store(key, *m);
  return FMLP_OK;
}

// ------------------------------------------------------------------------- validation

// A region of device memory: `rows` rows of `bytes` bytes, `ld` bytes apart (rows == 1: one
// contiguous run of `bytes`).
struct Range {
  const void* p;
  size_t bytes;
  const char* name;
  int64_t rows = 1;
  size_t ld = 0;
};

size_t span(const Range& r) { return r.rows > 1 ? (r.rows - 1) * r.ld + r.bytes : r.bytes; }

int64_t floor_div(int64_t a, int64_t b) { return a / b - ((a % b != 0) && ((a < 0) != (b < 0))); }

bool overlaps(const Range& a, const Range& b) {
  if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  if (!(a0 < b0 + span(b) && b0 < a0 + span(a))) return false;
  // Two row-strided regions with the same stride (views of one buffer, such as two column
  // blocks): row i of a is [a0 + i ld, + wa) and row j of b is [b0 + j ld, + wb); they meet
  // iff some k = j - i in [-(rows_a - 1), rows_b - 1] has -wb < (b0 - a0) + k ld < wa.
  if (a.rows > 1 && b.rows > 1 && a.ld == b.ld && a.bytes <= a.ld && b.bytes <= b.ld) {
    const int64_t ld = static_cast<int64_t>(a.ld);
    const int64_t d = static_cast<int64_t>(b0) - static_cast<int64_t>(a0);
    const int64_t wa = static_cast<int64_t>(a.bytes), wb = static_cast<int64_t>(b.bytes);
    const int64_t klo = std::max<int64_t>(floor_div(-wb - d, ld) + 1, -(a.rows - 1));
    const int64_t khi = std::min<int64_t>(-floor_div(-(wa - d), ld) - 1, b.rows - 1);
    return klo <= khi;
  }
  return true;   // spans meet: treat as overlapping
}

fmlp_status check_T(int64_t T) {
  if (T < 0 || T > kMaxDim) {
    set_error("T = %lld is out of range [0, 2^31-1]", static_cast<long long>(T));
    return FMLP_ERR_SHAPE;
  }
  return FMLP_OK;
}

fmlp_status check_inner(int64_t v, const char* name) {
  if (v < 1 || v > kMaxDim || (v % 8) != 0) {
    set_error("%s = %lld must be in [8, 2^31-1] and a multiple of 8", name,
              static_cast<long long>(v));
    return FMLP_ERR_SHAPE;
  }
  return FMLP_OK;
}

fmlp_status check_ptrs(const Range* r, int n, bool nullable_mask_last = false) {
  (void)nullable_mask_last;
  for (int i = 0; i < n; ++i) {
    if (!r[i].p) continue;
    if (reinterpret_cast<uintptr_t>(r[i].p) % 16 != 0) {
      set_error("%s is not 16-byte aligned", r[i].name);
      return FMLP_ERR_ALIGN;
    }
  }
  return FMLP_OK;
}

fmlp_status check_alias(const Range& out, const Range* in, int n) {
  for (int i = 0; i < n; ++i) {
    if (overlaps(out, in[i])) {
      set_error("%s overlaps %s", out.name, in[i].name);
      return FMLP_ERR_ALIAS;
    }
  }
  return FMLP_OK;
}

#define FMLP_TRY(expr)                 \
  do {                                 \
    fmlp_status _st = (expr);          \
    if (_st != FMLP_OK) return _st;    \
  } while (0)

#define FMLP_NONNULL(p, name)                         \
  do {                                                \
    if (!(p)) {                                       \
      set_error("%s is NULL", name);                  \
      return FMLP_ERR_NULL;                           \
    }                                                 \
  } while (0)

size_t mat_bytes(int64_t r, int64_t c) { return static_cast<size_t>(r) * static_cast<size_t>(c) * 2u; }

// ------------------------------------------------------------------------- ragged dims
// Inner dimensions that are not multiples of 8 run on zero-padded copies (pad.cu says why
// that changes no result): the operands are copied into one stream-ordered scratch with every
// inner dimension rounded up to 8, the normal plan runs on the padded shape, and the output's
// first columns are copied back. Packed rows only (a strided call keeps the multiple-of-8
// rule); it costs a copy of the weights per call.
int64_t up8(int64_t v) { return (v + 7) / 8 * 8; }

fmlp_status check_ragged(int64_t v, const char* name) {
  if (v < 1 || v > kMaxDim - 7) {
    set_error("%s = %lld must be in [1, 2^31-8]", name, static_cast<long long>(v));
    return FMLP_ERR_SHAPE;
  }
  return FMLP_OK;
}

// Regions of one scratch allocation, each 256-byte aligned.
struct PadScratch {
  size_t sizes[8];
  int n = 0;
  void* base = nullptr;
  size_t add(size_t bytes) {
    sizes[n++] = (bytes + 255) / 256 * 256;
    return static_cast<size_t>(n - 1);
  }
  size_t total() const {
    size_t t = 0;
    for (int i = 0; i < n; ++i) t += sizes[i];
    return t;
  }
  void* at(size_t i) const {
    size_t o = 0;
    for (size_t k = 0; k < i; ++k) o += sizes[k];
    return static_cast<char*>(base) + o;
  }
};

fmlp_status pad_alloc(PadScratch* p, cudaStream_t st) {
  cudaError_t e = cudaMallocAsync(&p->base, p->total(), st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(padded operands)");
  return FMLP_OK;
}

fmlp_status pad_free(PadScratch* p, cudaStream_t st, fmlp_status r) {
  cudaError_t e = cudaFreeAsync(p->base, st);
  if (e != cudaSuccess && r == FMLP_OK) return cuda_fail(e, "cudaFreeAsync(padded operands)");
  return r;
}

fmlp_status pad_copy(const void* src, int64_t rows, int64_t cols, void* dst, int64_t dst_rows,
                     int64_t dst_cols, cudaStream_t st) {
  cudaError_t e = pad2d_launch(src, cols, rows, cols, dst, dst_rows, dst_cols, st);
  if (e != cudaSuccess) return cuda_fail(e, "zero-padding copy");
  return FMLP_OK;
}

// ------------------------------------------------------------------------- tile choice

// Persistent grid: each CTA takes tiles round-robin, so the critical path is
// ceil(tiles / SMs) tiles of work proportional to bn. Narrow tiles cost extra shared-memory
// bandwidth per FLOP; the efficiency factors reflect that.
int pick_bn(int64_t M, int64_t N_out, int sms, bool geglu, double* cost_out) {
  const int cands[3] = {64, 128, 256};
  const double eff[3] = {0.60, 0.85, 1.0};
  int best = 0;
  double best_cost = 1e300;
  for (int i = 0; i < 3; ++i) {
    const int bn = cands[i];
    if (geglu && bn < 128) continue;
    const int bn_out = geglu ? bn / 2 : bn;
    const int64_t tiles = ((M + 127) / 128) * ((N_out + bn_out - 1) / bn_out);
    const int64_t waves = (tiles + sms - 1) / sms;
    const double cost = static_cast<double>(waves) * bn / eff[i];
    // candidates come in increasing bn; a (near) tie goes to the wider tile
    if (best == 0 || cost <= best_cost * 1.001) {
      best = bn;
      best_cost = std::min(best_cost, cost);
    }
  }
  *cost_out = best_cost;
  return best;
}

// Per-clock efficiency of the CTA-pair kernel relative to the single-SM 128x256 tile, from ncu
// durations on GB300 (it moves a third less operand data per SM).
constexpr double kPairEff = 1.3;

struct GemmChoice {
  bool pair;   // CTA-pair kernel (256-row tiles) instead of the single-SM kernel
  int bn;      // MMA N: 64/128/256 (single SM) or 256 (pair)
  int grid;    // CTAs launched
};

GemmChoice choose_gemm(const DeviceState& d, int epi, int64_t M, int64_t N_out) {
  GemmChoice c;
  const bool geglu = epi == EPI_GEGLU;
  double cost1 = 0;
  const int bn1 = pick_bn(M, N_out, d.sms, geglu, &cost1);
  c.pair = false;
  c.bn = bn1;
  const int policy = g_tile_policy.load(std::memory_order_relaxed);
  double best = (policy == FMLP_TILES_AUTO || policy == FMLP_TILES_SINGLE) ? cost1 : 1e300;
  int pairs_best = 0;
  if (d.max_pairs >= 1 && M > 128 && policy != FMLP_TILES_SINGLE) {
    const int bn = 256;
    const int bn_out = geglu ? bn / 2 : bn;
    const int64_t tiles2 = ((M + 255) / 256) * ((N_out + bn_out - 1) / bn_out);
    const int pairs = static_cast<int>(std::min<int64_t>(tiles2, d.max_pairs));
    const int64_t waves2 = (tiles2 + pairs - 1) / pairs;
    const double cost = static_cast<double>(waves2) * bn / kPairEff;
    if (cost < best || policy == FMLP_TILES_PAIR) {
      best = cost;
      c.pair = true;
      c.bn = bn;
      pairs_best = pairs;
    }
  }
  if (c.pair) {
    c.grid = 2 * pairs_best;
  } else {
    c.bn = bn1;
    const int bn_out = geglu ? c.bn / 2 : c.bn;
    const int64_t tiles = ((M + 127) / 128) * ((N_out + bn_out - 1) / bn_out);
    c.grid = static_cast<int>(std::min<int64_t>(tiles, d.sms));
  }
  return c;
}

// The few-token kernel (weights as the MMA's M side, K split over a cluster) serves M <= 128
// under the automatic tile policy.
bool use_skinny(int64_t M) {
  return M >= 1 && M <= kSkinnyMaxT &&
         g_tile_policy.load(std::memory_order_relaxed) == FMLP_TILES_AUTO;
}

// Tiling of the few-token kernel: K slices S (a power of two <= 8, every slice at least one
// 64-deep K step) and weight rows per tile R (a multiple of 4, at most 128), all tiles * S
// CTAs in one wave (one CTA per SM; the tiles may not outnumber the clusters of S CTAs that
// fit at once, which the GPCs decide, not just the SM count). Each CTA moves (R + Tpad) rows
// of K / S elements through its TMA (its weight rows and the tokens, which every tile reads
// again), so the choice minimises (R + Tpad) / S: more, shorter tiles put more SMs to work
// but re-read x more often (56-row tiles on 148 SMs ran slower than 128-row ones on 128).
struct SkinnyShape {
  int rows, tiles, split;
};

SkinnyShape skinny_shape(const DeviceState& d, int64_t N_out, int64_t K, int64_t tpad) {
  const int64_t num_kb = (K + 63) / 64;
  SkinnyShape best{128, static_cast<int>((N_out + 127) / 128), 1};
  double best_cost = -1.0;
  for (int S = 1, i = 0; S <= 8 && S <= num_kb; S *= 2, ++i) {
    const int64_t tiles_max = d.skinny_clusters[i] > 0 ? d.skinny_clusters[i] : d.sms / S;
    if (tiles_max < 1) break;
    int64_t R = (N_out + tiles_max - 1) / tiles_max;
    R = (R + 3) / 4 * 4;
    if (R > 128) continue;              // 128-row tiles would not fit in one wave
    const int64_t tiles = (N_out + R - 1) / R;
    const double cost = static_cast<double>(R + tpad) / S;
    if (best_cost < 0.0 || cost < best_cost) {
      best = SkinnyShape{static_cast<int>(R), static_cast<int>(tiles), S};
      best_cost = cost;
    }
  }
  return best;                          // no fit: 128-row tiles, no K split
}

fmlp_status launch_skinny(const DeviceState& d, int epi, const void* A, const void* B0,
                          const void* B1, const void* bias, void* Y, int64_t M, int64_t N_out,
                          int64_t K, int gelu_mode, bool pdl, cudaStream_t s, int64_t lda,
                          int64_t ldy) {
  FMLP_LAUNCH_GUARD("gemm_skinny launch");
  SkinnyLaunch L;
  memset(&L, 0, sizeof L);
  L.tpad = static_cast<int>((M + 31) / 32 * 32);
  const SkinnyShape sh = skinny_shape(d, N_out, K, L.tpad);
  FMLP_TRY(make_map(&L.tmW0, B0, N_out, K, static_cast<uint32_t>(sh.rows), "W"));
  if (epi == EPI_GEGLU) {
    FMLP_TRY(make_map(&L.tmW1, B1, N_out, K, static_cast<uint32_t>(sh.rows), "W_up"));
  } else {
    L.tmW1 = L.tmW0;
  }
  FMLP_TRY(make_map(&L.tmX, A, M, K, static_cast<uint32_t>(L.tpad), "x", lda));
  L.bias = bias;
  L.y = Y;
  L.T = static_cast<int>(M);
  L.N = static_cast<int>(N_out);
  L.K = static_cast<int>(K);
  L.ldy = static_cast<int>(ldy > 0 ? ldy : N_out);
  L.rows = sh.rows;
  L.tiles = sh.tiles;
  L.split = sh.split;
  L.epi = epi;
  L.gelu_mode = gelu_mode;
  L.pdl = pdl;
  L.stream = s;
  L.status = d.status;
  L.timeout_ns = kWaitTimeoutNs;
  const cudaError_t e = gemm_skinny_launch(L);
  if (e != cudaSuccess) return cuda_fail(e, "gemm_skinny launch");
  return FMLP_OK;
}

// lda, ldy: row strides of A and Y in elements (0: packed rows).
fmlp_status launch_gemm(const DeviceState& d, int epi, const void* A, const void* B0,
                        const void* B1, const void* bias, void* Y, int64_t M, int64_t N_out,
                        int64_t K, int gelu_mode, bool pdl, cudaStream_t s, int64_t lda = 0,
                        int64_t ldy = 0) {
  if (use_skinny(M))
    return launch_skinny(d, epi, A, B0, B1, bias, Y, M, N_out, K, gelu_mode, pdl, s, lda, ldy);
  FMLP_LAUNCH_GUARD("gemm launch");
  GemmLaunch L;
  memset(&L, 0, sizeof L);
  const bool geglu = epi == EPI_GEGLU;
  const GemmChoice ch = choose_gemm(d, epi, M, N_out);
  const bool pair = ch.pair;
  L.bn = ch.bn;
  const uint32_t b_rows = static_cast<uint32_t>(pair || geglu ? L.bn / 2 : L.bn);
  FMLP_TRY(make_map(&L.tmA, A, M, K, 128, "A", lda));
  FMLP_TRY(make_map(&L.tmB0, B0, N_out, K, b_rows, "B"));
  if (geglu) {
    FMLP_TRY(make_map(&L.tmB1, B1, N_out, K, b_rows, "B_up"));
  } else {
    L.tmB1 = L.tmB0;
  }
  FMLP_TRY(make_map(&L.tmY, Y, M, N_out, 32, "Y", ldy));
  L.bias = bias;
  L.M = static_cast<int>(M);
  L.N_out = static_cast<int>(N_out);
  L.K = static_cast<int>(K);
  L.gelu_mode = gelu_mode;
  L.epi = epi;
  L.pdl = pdl;
  L.stream = s;
  L.status = d.status;
  L.timeout_ns = kWaitTimeoutNs;
  L.grid = ch.grid;
  if (pair && take_injection(g_inject_skip)) {
    L.skip_first_load = true;
    const unsigned long long tmo = g_inject_timeout_ns.load(std::memory_order_relaxed);
    if (tmo) L.timeout_ns = tmo;
  }
  const cudaError_t e = pair ? gemm_tc2_launch(L) : gemm_tc_launch(L);
  if (e != cudaSuccess) return cuda_fail(e, pair ? "gemm_tc2 launch" : "gemm_tc launch");
  return FMLP_OK;
}

// ------------------------------------------------------------------------- plans

// SM count for the host-only plan queries: the current device's (no context is created), or
// GB300's 152 when no device is visible. The workspace a plan needs never depends on it.
int plan_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
    {
      std::lock_guard<std::mutex> lock(g_mu);
      if (g_dev[dev].ready) return g_dev[dev].sms;
    }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      return n;
  }
  (void)cudaGetLastError();
  return 152;
}

// The one-kernel decode (both layers, one CTA per SM) serves 1..kDecodeMaxT tokens when its
// token vectors and reduction buffers fit in shared memory.
bool decode_ok(int64_t T, int64_t D, int64_t H, int64_t Dout, int nmat, int sms) {
  return T >= 1 && T <= kDecodeMaxT && D >= 8 && D % 8 == 0 && H >= 8 && H % 8 == 0 &&
         D <= kMaxDim && H <= kMaxDim && Dout >= 1 && Dout <= kMaxDim &&
         decode_ring_stages(static_cast<int>(T), static_cast<int>(D), static_cast<int>(H),
                            static_cast<int>(Dout), nmat, sms) >= 2;
}

// Decode crossover, measured on GB300 (CUDA graphs of 20 calls over 5 weight sets): the GEMV
// wins at one token, and at two when the call's weights are small (16 MiB or less: 9.3 vs
// 10.1 us for the GPT-2-small-shaped GeGLU); otherwise the few-token tcgen05 kernel wins
// (4096-wide MLP at 2-4 tokens: 20.3 us against 25.9-33.9 us for the GEMV).
constexpr int64_t kGemvSmallWeights = int64_t(16) << 20;
// Below this many weight bytes a few-token GeGLU stays on the single-CTA fused kernel.
constexpr size_t kSmallDecodeBytes = size_t(1) << 20;
bool gemv_preferred(int64_t T, int64_t weight_bytes) {
  return T == 1 || (T == 2 && weight_bytes <= kGemvSmallWeights);
}

bool gemv_ok(int64_t T, int64_t K, int64_t N, int nmat, int sms) {
  if (T < 1 || T > kGemvMaxT || K % 256 != 0) return false;
  const int grid = gemv_grid(static_cast<int>(T), static_cast<int>(K), static_cast<int>(N), nmat,
                             sms);
  return gemv_smem_bytes(static_cast<int>(T), static_cast<int>(K), static_cast<int>(N), nmat,
                         grid) <= kGemvMaxSmem;
}

int plan_linear(int64_t T, int64_t in, int64_t out, int sms) {
  if (T <= 0) return FMLP_PLAN_NONE;
  return gemv_ok(T, in, out, 1, sms) && gemv_preferred(T, mat_bytes(out, in)) ? FMLP_PLAN_GEMV
                                                                              : FMLP_PLAN_TC;
}

// Whether the single-kernel fused plan takes a block of these sizes. It depends on the shape
// alone (never on the SM count), so the workspace query and the call agree on whether the
// intermediate needs a workspace. At decode sizes (1..kDecodeMaxT tokens) the one-kernel
// decode spreads the weights over every SM; the single-CTA fused kernel only takes tiny ones.
bool fused_small(int64_t T, int64_t D, int64_t H, int64_t Dout, bool mlp) {
  const bool shape = mlp ? (D <= kSmallMaxD && Dout <= kSmallMaxD && Dout % 16 == 0 &&
                            H <= kSmallMaxH)
                         : (D <= kSmallMaxD && D % 16 == 0 && H <= kSmallMaxH);
  const size_t wbytes = mlp ? mat_bytes(H, D) + mat_bytes(Dout, H) : 3 * mat_bytes(H, D);
  return T >= 1 && shape && (T > kDecodeMaxT || wbytes <= kSmallDecodeBytes);
}

int plan_mlp(int64_t T, int64_t D, int64_t H, int64_t Dout, int sms) {
  if (T <= 0) return FMLP_PLAN_NONE;
  if (fused_small(T, D, H, Dout, true)) return FMLP_PLAN_FUSED_SMALL;
  if (g_prefer_decode.load(std::memory_order_relaxed) && decode_ok(T, D, H, Dout, 1, sms))
    return FMLP_PLAN_DECODE;
  if (gemv_ok(T, D, H, 1, sms) && gemv_ok(T, H, Dout, 1, sms) &&
      gemv_preferred(T, mat_bytes(H, D) + mat_bytes(Dout, H)))
    return FMLP_PLAN_GEMV;
  return FMLP_PLAN_TC;
}

int plan_geglu(int64_t T, int64_t D, int64_t H, int sms) {
  if (T <= 0) return FMLP_PLAN_NONE;
  if (fused_small(T, D, H, D, false)) return FMLP_PLAN_FUSED_SMALL;
  if (g_prefer_decode.load(std::memory_order_relaxed) && decode_ok(T, D, H, D, 2, sms))
    return FMLP_PLAN_DECODE;
  if (T <= kGemvMaxT && D % 256 == 0 && H % 256 == 0 && gemv_ok(T, D, H, 2, sms) &&
      gemv_ok(T, H, D, 1, sms) && gemv_preferred(T, 3 * mat_bytes(H, D)))
    return FMLP_PLAN_GEMV;
  return FMLP_PLAN_TC;
}

// ldx, ldy: row strides of x and y in elements (0: packed rows).
fmlp_status launch_gemv(const DeviceState& d, int epi, const void* x, const void* W0,
                        const void* W1, const void* bias, void* y, int64_t T, int64_t K,
                        int64_t N, int gelu_mode, cudaStream_t s, int64_t ldx = 0,
                        int64_t ldy = 0) {
  FMLP_LAUNCH_GUARD("gemv launch");
  GemvLaunch L;
  L.x = x;
  L.W0 = W0;
  L.W1 = W1;
  L.bias = bias;
  L.y = y;
  L.T = static_cast<int>(T);
  L.K = static_cast<int>(K);
  L.N = static_cast<int>(N);
  L.epi = epi;
  L.gelu_mode = gelu_mode;
  L.ldx = static_cast<int>(ldx > 0 ? ldx : K);
  L.ldy = static_cast<int>(ldy > 0 ? ldy : N);
  L.grid = gemv_grid(static_cast<int>(T), static_cast<int>(K), static_cast<int>(N),
                     epi == EPI_GEGLU ? 2 : 1, d.sms);
  L.stream = s;
  cudaError_t e = gemv_launch(L);
  if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
  return FMLP_OK;
}

// The whole block in one kernel (small D and Dout). GeGLU: W1 = Wg, Wu, W2 = Wd, Dout = D,
// no biases. MLP: W1, W2 with nullable biases b1, b2 and the activation `mode`.
fmlp_status launch_small(const DeviceState& d, bool mlp, const void* x, const void* W1,
                         const void* Wu, const void* W2, const void* b1, const void* b2, void* y,
                         int64_t T, int64_t D, int64_t H, int64_t Dout, int mode,
                         cudaStream_t s, int64_t ldx = 0, int64_t ldy = 0) {
  FMLP_LAUNCH_GUARD("fused small launch");
  SmallLaunch L;
  memset(&L, 0, sizeof L);
  FMLP_TRY(make_map(&L.tmX, x, T, D, 128, "x", ldx));
  FMLP_TRY(make_map(&L.tmWg, W1, H, D, 64, mlp ? "W1" : "Wg"));
  if (mlp) {
    L.tmWu = L.tmWg;
  } else {
    FMLP_TRY(make_map(&L.tmWu, Wu, H, D, 64, "Wu"));
  }
  FMLP_TRY(make_map(&L.tmWd, W2, Dout, H, static_cast<uint32_t>(Dout), mlp ? "W2" : "Wd"));
  FMLP_TRY(make_map(&L.tmY, y, T, Dout, 32, "y", ldy));
  L.b1 = b1;
  L.b2 = b2;
  L.T = static_cast<int>(T);
  L.D = static_cast<int>(D);
  L.H = static_cast<int>(H);
  L.Dout = static_cast<int>(Dout);
  L.mlp = mlp;
  L.gelu_mode = mode;
  L.status = d.status;
  L.timeout_ns = kWaitTimeoutNs;
  L.stream = s;
  cudaError_t e = ffn_small_launch(L);
  if (e != cudaSuccess) return cuda_fail(e, "fused small launch");
  return FMLP_OK;
}

// Row of per-stream device counters (decode grid barrier, two-stage band counters) that
// launches on stream s use, or -1 when every row is taken. Launches on one stream run in
// order, so they can share a row; launches on different streams get different rows.
int stream_slot(DeviceState& d, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < d.decode_streams; ++i)
    if (d.decode_stream[i] == s) return i;
  if (d.decode_streams < kDecodeSlots) {
    d.decode_stream[d.decode_streams] = s;
    return d.decode_streams++;
  }
  return -1;
}

// ------------------------------------------------------------------ two-stage block launch

// Both layers of a block in one persistent CTA-pair launch: the pairs work through lists of
// first-stage tiles and second-stage (down) tiles, so the long down tiles of early bands run
// while other pairs still compute first-stage tiles, and no pair waits through a partial wave
// of down tiles at the end, nor for a second launch. Taken when both stages would use the
// pair kernel and both layers' weights fit in L2 together (the first stage then runs band by
// band, each band's tiles reading weights that stay resident).
constexpr double kTwoTileOverhead = 3.0;   // per tile, in 64-deep K steps (prologue, epilogue)
// Bands per group of the first stage's order (GPT-2-small block, groups of 1/2/4/8/16/32:
// 81.9/79.7/78.8/78.1/79.9/84.0 us).
constexpr int kTwoGroup = 8;
constexpr int64_t kTwoMaxWeightBytes = 64ll << 20;

struct TwoSchedule {
  // the key: bands, first-stage N tiles, down N tiles, K steps of each stage, pairs
  int num_m = 0, num_n1 = 0, num_n2 = 0, kb1 = 0, kb2 = 0, pairs = 0;
  std::vector<uint16_t> start, item;
  double makespan = 0.0;     // estimated, in 64-deep K steps of one pair
  double two_launch = 0.0;   // the same estimate for two round-robin launches
};

// List scheduling of the items over the pairs (each pair runs its list in order), in units
// of one 64-deep K step. The pair that frees up first takes a down tile whose band is complete
// while fewer than `early` down tiles have been placed ahead of the last first-stage tile, else
// the next first-stage tile, else the down tile whose band completes first (waiting for it).
// A down tile is only placed once every first-stage tile of its band has been, so every wait
// in the lists is on an item placed earlier: with all pairs resident, the waits end. Returns
// the estimated makespan. Items: first-stage u = band * num_n1 + j, taken in groups of
// kTwoGroup bands with the band running fastest; then down items n1 + band * num_n2 + n.
double list_schedule(const TwoSchedule& sc, int early, std::vector<std::vector<uint16_t>>* lists) {
  const int num_m = sc.num_m, P = sc.pairs, per1 = sc.num_n1;
  const int n1 = num_m * per1, n2 = num_m * sc.num_n2;
  const double c1 = sc.kb1 + kTwoTileOverhead, c2 = sc.kb2 + kTwoTileOverhead;
  lists->assign(P, {});
  std::vector<double> free_at(P, 0.0), band_ready(num_m, 0.0);
  std::vector<int> band_left(num_m, per1);
  std::vector<int> pending;   // down items of complete bands, not yet placed
  int next1 = 0, taken_early = 0;
  auto band_of = [&](int t) { return (t - n1) / sc.num_n2; };
  for (int placed = 0; placed < n1 + n2; ++placed) {
    int p = 0;
    for (int q = 1; q < P; ++q)
      if (free_at[q] < free_at[p]) p = q;
    int best = -1;
    for (int i = 0; i < static_cast<int>(pending.size()); ++i)
      if (best < 0 || band_ready[band_of(pending[i])] < band_ready[band_of(pending[best])])
        best = i;
    const bool down_now =
        best >= 0 && taken_early < early && band_ready[band_of(pending[best])] <= free_at[p];
    if (!down_now && next1 < n1) {
      // first-stage items in groups of kTwoGroup bands, the band running fastest, so the
      // pairs in flight read each weight tile at about the same time from L2
      const int k = next1++, per_group = kTwoGroup * per1, kg = k / per_group;
      const int r = k - kg * per_group, gb = std::min(kTwoGroup, num_m - kg * kTwoGroup);
      const int t = (kg * kTwoGroup + r % gb) * per1 + r / gb;
      const int b = t / per1;
      (*lists)[p].push_back(static_cast<uint16_t>(t));
      free_at[p] += c1;
      band_ready[b] = std::max(band_ready[b], free_at[p]);
      if (--band_left[b] == 0)
        for (int j = 0; j < sc.num_n2; ++j) pending.push_back(n1 + b * sc.num_n2 + j);
    } else {
      if (next1 < n1) ++taken_early;
      const int t = pending[best];
      pending.erase(pending.begin() + best);
      (*lists)[p].push_back(static_cast<uint16_t>(t));
      free_at[p] = std::max(free_at[p], band_ready[band_of(t)]) + c2;
    }
  }
  return *std::max_element(free_at.begin(), free_at.end());
}

// The schedule with the shortest estimated makespan over a sweep of `early` (the down tiles
// that do not fill whole waves at the end are the ones worth running early).
void build_two_schedule(TwoSchedule* sc) {
  const int n2 = sc->num_m * sc->num_n2;
  std::vector<std::vector<uint16_t>> lists, best_lists;
  double best = -1.0;
  const int step = std::max(1, n2 / 16);
  for (int e = -1; e <= n2; e += (e < 0 ? 1 : step)) {
    const int early = e < 0 ? n2 % sc->pairs : e;
    const double ms = list_schedule(*sc, early, &lists);
    if (best < 0.0 || ms < best) {
      best = ms;
      best_lists.swap(lists);
    }
  }
  sc->start.assign(sc->pairs + 1, 0);
  sc->item.clear();
  for (int p = 0; p < sc->pairs; ++p) {
    sc->item.insert(sc->item.end(), best_lists[p].begin(), best_lists[p].end());
    sc->start[p + 1] = static_cast<uint16_t>(sc->item.size());
  }
  sc->makespan = best;
  // the same tiles as two round-robin launches over as many pairs, for the automatic choice
  const int n1 = sc->num_m * sc->num_n1;
  const double waves1 = (n1 + sc->pairs - 1) / sc->pairs, waves2 = (n2 + sc->pairs - 1) / sc->pairs;
  sc->two_launch = waves1 * (sc->kb1 + kTwoTileOverhead) + waves2 * (sc->kb2 + kTwoTileOverhead);
}

// Schedules are a pure function of the key; a few are kept (a model has few block shapes).
constexpr int kTwoCache = 8;
std::mutex g_two_mu;
TwoSchedule g_two_cache[kTwoCache];
int g_two_next = 0;

// A copy: the cached entry may be replaced by another thread once the lock is released.
TwoSchedule two_schedule(int num_m, int num_n1, int num_n2, int kb1, int kb2, int pairs) {
  std::lock_guard<std::mutex> lock(g_two_mu);
  for (const TwoSchedule& c : g_two_cache)
    if (c.pairs == pairs && c.num_m == num_m && c.num_n1 == num_n1 && c.num_n2 == num_n2 &&
        c.kb1 == kb1 && c.kb2 == kb2)
      return c;
  TwoSchedule& c = g_two_cache[g_two_next];
  g_two_next = (g_two_next + 1) % kTwoCache;
  c.num_m = num_m;
  c.num_n1 = num_n1;
  c.num_n2 = num_n2;
  c.kb1 = kb1;
  c.kb2 = kb2;
  c.pairs = pairs;
  build_two_schedule(&c);
  return c;
}

// Test hook (fmlp_test_two_stage): 0 automatic, -1 never, 1 whenever the shape is accepted.
std::atomic<int> g_two_stage{0};

// Pairs of a two-stage launch of this block, or 0 when it does not take one.
struct TwoPlan {
  int pairs = 0;
  int num_m = 0, num_n1 = 0, num_n2 = 0, kb1 = 0, kb2 = 0;
};

TwoPlan plan_two(const DeviceState& d, int epi1, int64_t T, int64_t D, int64_t H, int64_t Dout) {
  TwoPlan tp;
  const int mode = g_two_stage.load(std::memory_order_relaxed);
  if (mode < 0 || d.max_pairs < 1 || use_skinny(T) || T <= 128 ||
      g_tile_policy.load(std::memory_order_relaxed) == FMLP_TILES_SINGLE)
    return tp;
  const bool geglu = epi1 == EPI_GEGLU;
  const int64_t w_bytes = static_cast<int64_t>((geglu ? 2 : 1) * mat_bytes(H, D) + mat_bytes(Dout, H));
  const int64_t num_m = (T + 255) / 256;
  const int64_t num_n1 = (H + (geglu ? 127 : 255)) / (geglu ? 128 : 256);
  const int64_t num_n2 = (Dout + 255) / 256;
  const int64_t items = num_m * (num_n1 + num_n2);
  if (w_bytes > kTwoMaxWeightBytes || num_m > kTwoMaxBands || items > kTwoMaxItems) return tp;
  if (mode == 0 && !(choose_gemm(d, epi1, T, H).pair && choose_gemm(d, EPI_BIAS, T, Dout).pair))
    return tp;
  const int pairs = std::min(std::min(d.max_pairs, kTwoMaxPairs), static_cast<int>(items));
  const int kb1 = static_cast<int>((D + 63) / 64), kb2 = static_cast<int>((H + 63) / 64);
  if (mode == 0) {
    // only where the list schedule is estimated clearly shorter than two launches (at 0.92
    // of their estimate a 8192x1024x4096 GeGLU block measured 2.6 % slower in one launch)
    const TwoSchedule sc = two_schedule(static_cast<int>(num_m), static_cast<int>(num_n1),
                                        static_cast<int>(num_n2), kb1, kb2, pairs);
    if (sc.makespan > 0.9 * sc.two_launch) return tp;
  }
  tp.pairs = pairs;
  tp.num_m = static_cast<int>(num_m);
  tp.num_n1 = static_cast<int>(num_n1);
  tp.num_n2 = static_cast<int>(num_n2);
  tp.kb1 = kb1;
  tp.kb2 = kb2;
  return tp;
}

// One launch for both layers when plan_two accepts the block (*ran = true); otherwise nothing
// is launched and the caller runs the two GEMMs.
fmlp_status launch_two(DeviceState& d, int epi1, const void* x, const void* W1a, const void* W1b,
                       const void* b1, const void* W2, const void* b2, void* h, void* y,
                       int64_t T, int64_t D, int64_t H, int64_t Dout, int gelu_mode,
                       cudaStream_t s, int64_t ldx, int64_t ldy, bool* ran) {
  *ran = false;
  const TwoPlan tp = plan_two(d, epi1, T, D, H, Dout);
  if (tp.pairs < 1) return FMLP_OK;
  const int slot = stream_slot(d, s);
  if (slot < 0) return FMLP_OK;
  FMLP_LAUNCH_GUARD("two-stage launch");
  // test hook: a band count one above what the first stage adds, so every down tile's wait
  // runs out
  const bool starve = take_injection(g_inject_skip);
  const TwoSchedule sc = two_schedule(tp.num_m, tp.num_n1, tp.num_n2, tp.kb1, tp.kb2, tp.pairs);
  const bool geglu = epi1 == EPI_GEGLU;
  GemmLaunch L;
  memset(&L, 0, sizeof L);
  L.bn = 256;
  FMLP_TRY(make_map(&L.tmA, x, T, D, 128, "x", ldx));
  FMLP_TRY(make_map(&L.tmB0, W1a, H, D, 128, geglu ? "Wg" : "W1"));
  if (geglu) {
    FMLP_TRY(make_map(&L.tmB1, W1b, H, D, 128, "Wu"));
  } else {
    L.tmB1 = L.tmB0;
  }
  FMLP_TRY(make_map(&L.tmY, h, T, H, 32, "intermediate"));
  L.bias = b1;
  L.M = static_cast<int>(T);
  L.N_out = static_cast<int>(H);
  L.K = static_cast<int>(D);
  L.gelu_mode = gelu_mode;
  L.epi = epi1;
  L.pdl = false;
  L.stream = s;
  L.status = d.status;
  L.timeout_ns = kWaitTimeoutNs;
  if (starve) {
    const unsigned long long tmo = g_inject_timeout_ns.load(std::memory_order_relaxed);
    if (tmo) L.timeout_ns = tmo;
  }
  L.grid = 2 * tp.pairs;
  TwoStageLaunch T2;
  memset(&T2, 0, sizeof T2);
  FMLP_TRY(make_map(&T2.tmA2, h, T, H, 128, "intermediate"));
  FMLP_TRY(make_map(&T2.tmB2, W2, Dout, H, 128, geglu ? "Wd" : "W2"));
  FMLP_TRY(make_map(&T2.tmY2, y, T, Dout, 32, "y", ldy));
  T2.bias2 = b2;
  T2.slot = slot;
  T2.band_extra = starve ? 1 : 0;
  T2.N2 = static_cast<int>(Dout);
  T2.K2 = static_cast<int>(H);
  T2.n1 = tp.num_m * tp.num_n1;
  T2.n_items = static_cast<int>(sc.item.size());
  T2.start = sc.start.data();
  T2.item = sc.item.data();
  const cudaError_t e = gemm_tc2_two_launch(L, T2);
  if (e != cudaSuccess) return cuda_fail(e, "two-stage launch");
  *ran = true;
  return FMLP_OK;
}

// ------------------------------------------------------------ few-token block launch

// Test hook (fmlp_test_fewtoken_block): 0 automatic, 1 whenever the shape is accepted, -1 never.
std::atomic<int> g_fewblock{0};

struct FewBlockPlan {
  bool ok = false;
  int rows1 = 0, rows2 = 0, tiles = 0, split = 0, tpad = 0;
};

// Both layers of a few-token block in one launch: the few-token kernel's tiling of layer 1,
// the same tiles and K split for layer 2, every CTA resident at once, the ring and the
// exchange region within one CTA's shared memory.
FewBlockPlan plan_fewblock(const DeviceState& d, int epi1, int64_t T, int64_t D, int64_t H,
                           int64_t Dout) {
  FewBlockPlan p;
  const int mode = g_fewblock.load(std::memory_order_relaxed);
  if (mode < 0 || !use_skinny(T) || !d.decode_bar) return p;
  const int nmat1 = epi1 == EPI_GEGLU ? 2 : 1;
  const int64_t tpad = (T + 31) / 32 * 32;
  if (tpad > (nmat1 == 2 ? 64 : 128)) return p;
  const SkinnyShape sh = skinny_shape(d, H, D, tpad);
  const int64_t rows2 = ((Dout + sh.tiles - 1) / sh.tiles + 3) / 4 * 4;
  if (sh.rows > 128 || rows2 > 128 || sh.split > (D + 63) / 64 || sh.split > (H + 63) / 64)
    return p;
  int si = 0;
  while ((1 << si) < sh.split) ++si;
  if (sh.tiles > d.fewblock_clusters[si]) return p;   // every CTA must be resident at once
  if (fewtoken_block_stages(nmat1, static_cast<int>(tpad), sh.split, sh.rows,
                            static_cast<int>(rows2), nullptr, nullptr) == 0)
    return p;
  // Automatically only where it measured faster (CUDA graphs of 20 forwards, rotating weights):
  // layer 2's tiles at least half as tall as layer 1's and at most 64 tokens. The 4096-wide MLP
  // at 2/16/64 tokens took 19.7/19.7/22.5 us in one launch against 20.7/21.1/23.1 in two; at
  // 128 tokens 26.6 against 26.0; the GPT-2-small GeGLU block (layer-2 tiles of 24 rows against
  // 88) 13.7 against 11.8 at 16 tokens.
  if (mode == 0 && (tpad > 64 || 2 * rows2 < sh.rows)) return p;
  p.ok = true;
  p.rows1 = sh.rows;
  p.rows2 = static_cast<int>(rows2);
  p.tiles = sh.tiles;
  p.split = sh.split;
  p.tpad = static_cast<int>(tpad);
  return p;
}

fmlp_status launch_fewblock(DeviceState& d, int epi1, const void* x, const void* W1a,
                            const void* W1b, const void* b1, const void* W2, const void* b2,
                            void* h, void* y, int64_t T, int64_t D, int64_t H, int64_t Dout,
                            int gelu_mode, cudaStream_t s, int64_t ldx, int64_t ldy, bool* ran) {
  *ran = false;
  const FewBlockPlan p = plan_fewblock(d, epi1, T, D, H, Dout);
  if (!p.ok) return FMLP_OK;
  const int slot = stream_slot(d, s);
  if (slot < 0) return FMLP_OK;
  FMLP_LAUNCH_GUARD("few-token block launch");
  const bool geglu = epi1 == EPI_GEGLU;
  FewBlockLaunch L;
  memset(&L, 0, sizeof L);
  FMLP_TRY(make_map(&L.tmW1a, W1a, H, D, static_cast<uint32_t>(p.rows1), geglu ? "Wg" : "W1"));
  if (geglu) {
    FMLP_TRY(make_map(&L.tmW1b, W1b, H, D, static_cast<uint32_t>(p.rows1), "Wu"));
  } else {
    L.tmW1b = L.tmW1a;
  }
  FMLP_TRY(make_map(&L.tmX, x, T, D, static_cast<uint32_t>(p.tpad), "x", ldx));
  FMLP_TRY(make_map(&L.tmW2, W2, Dout, H, static_cast<uint32_t>(p.rows2), geglu ? "Wd" : "W2"));
  FMLP_TRY(make_map(&L.tmH, h, T, H, static_cast<uint32_t>(p.tpad), "intermediate"));
  L.b1 = b1;
  L.b2 = b2;
  L.h = h;
  L.y = y;
  L.barrier = d.decode_bar + 16 * slot;
  L.T = static_cast<int>(T);
  L.D = static_cast<int>(D);
  L.H = static_cast<int>(H);
  L.Dout = static_cast<int>(Dout);
  L.ldy = static_cast<int>(ldy > 0 ? ldy : Dout);
  L.tpad = p.tpad;
  L.rows1 = p.rows1;
  L.rows2 = p.rows2;
  // test hook (fmlp_test_decode_overload): clusters beyond the resident ones, whose tiles lie
  // past the last weight row (zero-filled loads, no stores), so the barrier's wait runs out
  const int extra = g_decode_extra_ctas.load(std::memory_order_relaxed);
  L.tiles = p.tiles + (extra + p.split - 1) / p.split;
  L.split = p.split;
  L.epi1 = epi1;
  L.gelu_mode = gelu_mode;
  L.pdl = true;
  L.stream = s;
  L.status = d.status;
  const unsigned long long tmo = g_decode_timeout_ns.load(std::memory_order_relaxed);
  L.timeout_ns = tmo ? tmo : kWaitTimeoutNs;
  const cudaError_t e = fewtoken_block_launch(L);
  if (e != cudaSuccess) return cuda_fail(e, "few-token block launch");
  *ran = true;
  return FMLP_OK;
}

// One-kernel decode of the whole block. Falls back (returns FMLP_PLAN_NONE in *ran = false)
// when this device cannot run it or every grid-barrier counter is taken.
fmlp_status launch_decode(DeviceState& d, bool geglu, const void* x, const void* W1a,
                          const void* W1b, const void* b1, const void* W2, const void* b2,
                          void* h, void* y, int64_t T, int64_t D, int64_t H, int64_t Dout,
                          int gelu_mode, cudaStream_t s, bool* ran, int64_t ldx, int64_t ldy) {
  *ran = false;
  if (d.decode_occ < 1 || !d.decode_bar) return FMLP_OK;
  const int slot = stream_slot(d, s);
  if (slot < 0) return FMLP_OK;
  FMLP_LAUNCH_GUARD("decode launch");
  DecodeLaunch L;
  memset(&L, 0, sizeof L);
  L.x = x;
  L.W1a = W1a;
  L.W1b = W1b;
  L.b1 = b1;
  L.W2 = W2;
  L.b2 = b2;
  L.h = h;
  L.y = y;
  L.T = static_cast<int>(T);
  L.D = static_cast<int>(D);
  L.H = static_cast<int>(H);
  L.Dout = static_cast<int>(Dout);
  L.ldx = static_cast<int>(ldx);
  L.ldy = static_cast<int>(ldy);
  L.geglu = geglu;
  L.gelu_mode = gelu_mode;
  L.grid = d.sms * std::min(d.decode_occ, 1) + g_decode_extra_ctas.load(std::memory_order_relaxed);
  L.barrier = d.decode_bar + 16 * slot;
  L.status = d.status;
  const unsigned long long tmo = g_decode_timeout_ns.load(std::memory_order_relaxed);
  L.timeout_ns = tmo ? tmo : kWaitTimeoutNs;
  L.stream = s;
  const cudaError_t e = decode_launch(L);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  *ran = true;
  return FMLP_OK;
}

}  // namespace

int validate_block_dims(int64_t T, int64_t D, int64_t H) {
  FMLP_TRY(check_T(T));
  FMLP_TRY(check_inner(D, "D"));
  FMLP_TRY(check_inner(H, "H"));
  return FMLP_OK;
}

void record_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
}

}  // namespace fmlp

using namespace fmlp;

extern "C" {

int fmlp_version(void) { return 100; }

const char* fmlp_status_string(fmlp_status st) {
  switch (st) {
    case FMLP_OK: return "FMLP_OK";
    case FMLP_ERR_NULL: return "FMLP_ERR_NULL: a required pointer is NULL";
    case FMLP_ERR_SHAPE: return "FMLP_ERR_SHAPE: invalid dimension";
    case FMLP_ERR_ALIGN: return "FMLP_ERR_ALIGN: pointer not 16-byte aligned";
    case FMLP_ERR_ALIAS: return "FMLP_ERR_ALIAS: output overlaps an input";
    case FMLP_ERR_WORKSPACE: return "FMLP_ERR_WORKSPACE: workspace too small";
    case FMLP_ERR_CUDA: return "FMLP_ERR_CUDA: CUDA call failed";
    case FMLP_ERR_DEVICE_TIMEOUT: return "FMLP_ERR_DEVICE_TIMEOUT: a device wait ran out";
    case FMLP_ERR_DEVICE: return "FMLP_ERR_DEVICE: unsupported device";
    default: return "unknown fmlp_status";
  }
}

const char* fmlp_last_error(void) { return t_last_error.c_str(); }

// Every plan but the single-kernel small GeGLU keeps the intermediate (T x H bf16) in the
// workspace, so the size depends on the shape alone.
// With an inner dimension that is not a multiple of 8 the zero-padded path takes its own
// scratch (intermediate included): no caller workspace.
size_t fmlp_geglu_workspace_size(int64_t T, int64_t D, int64_t H) {
  if (T <= 0 || H <= 0) return 0;
  if (D % 8 != 0 || H % 8 != 0) return 0;
  return plan_geglu(T, D, H, plan_sms()) == FMLP_PLAN_FUSED_SMALL ? 0 : mat_bytes(T, H);
}

size_t fmlp_mlp_gelu_workspace_size(int64_t T, int64_t D, int64_t H, int64_t Dout) {
  if (T <= 0 || H <= 0) return 0;
  if (D % 8 != 0 || H % 8 != 0 || Dout % 8 != 0) return 0;
  return plan_mlp(T, D, H, Dout, plan_sms()) == FMLP_PLAN_FUSED_SMALL ? 0 : mat_bytes(T, H);
}

// Plans of ragged sizes are those of the zero-padded shape.
int fmlp_geglu_plan(int64_t T, int64_t D, int64_t H) {
  return plan_geglu(T, up8(D), up8(H), plan_sms());
}

int fmlp_mlp_gelu_plan(int64_t T, int64_t D, int64_t H, int64_t Dout) {
  return plan_mlp(T, up8(D), up8(H), up8(Dout), plan_sms());
}

int fmlp_linear_plan(int64_t T, int64_t in, int64_t out) {
  return plan_linear(T, up8(in), up8(out), plan_sms());
}

// Row strides of x [T, in] and y [T, out] in elements: 0 means packed rows (the stride is
// the row length); otherwise at least the row length (else FMLP_ERR_SHAPE) and a multiple of
// 8, the 16-byte row rule of the TMA loads and stores (else FMLP_ERR_ALIGN).
static fmlp_status resolve_strides(int64_t* ldx, int64_t* ldy, int64_t in, int64_t out) {
  if (*ldx == 0) *ldx = in;
  if (*ldy == 0) *ldy = out;
  if (*ldx < in || *ldy < out || *ldx > kMaxDim || *ldy > kMaxDim) {
    set_error("row strides ldx = %lld, ldy = %lld must be at least the rows' lengths %lld, %lld",
              static_cast<long long>(*ldx), static_cast<long long>(*ldy),
              static_cast<long long>(in), static_cast<long long>(out));
    return FMLP_ERR_SHAPE;
  }
  if (*ldx % 8 != 0 || *ldy % 8 != 0) {
    set_error("row strides ldx = %lld, ldy = %lld are not multiples of 8 elements (16 bytes)",
              static_cast<long long>(*ldx), static_cast<long long>(*ldy));
    return FMLP_ERR_ALIGN;
  }
  return FMLP_OK;
}

// ldx, ldy: row strides of x and y in elements (0: packed rows).
static fmlp_status linear_common(const void* x, const void* W, const void* b, void* y,
                                 int64_t T, int64_t in, int64_t out, int epi, int mode,
                                 fmlp_stream_t s, int64_t ldx = 0, int64_t ldy = 0);

// A Linear (or Linear + activation) whose in or out is not a multiple of 8.
static fmlp_status linear_padded(const void* x, const void* W, const void* b, void* y,
                                 int64_t T, int64_t in, int64_t out, int epi, int mode,
                                 fmlp_stream_t s) {
  FMLP_TRY(check_ragged(in, "in"));
  FMLP_TRY(check_ragged(out, "out"));
  if (epi == EPI_BIAS_GELU && !act_mode_ok(mode)) {
    set_error("activation mode %d is not FMLP_GELU_TANH, FMLP_GELU_ERF or FMLP_RELU", mode);
    return FMLP_ERR_SHAPE;
  }
  if (T == 0) return FMLP_OK;
  FMLP_NONNULL(x, "x");
  FMLP_NONNULL(W, "W");
  FMLP_NONNULL(y, "y");
  const Range rx{x, mat_bytes(T, in), "x"}, rw{W, mat_bytes(out, in), "W"},
      rb{b, b ? mat_bytes(1, out) : 0, "b"}, ry{y, mat_bytes(T, out), "y"};
  const Range ins[3] = {rx, rw, rb};
  const Range all[4] = {rx, rw, rb, ry};
  FMLP_TRY(check_ptrs(all, 4));
  FMLP_TRY(check_alias(ry, ins, 3));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  const int64_t Kp = up8(in), Np = up8(out);
  PadScratch p;
  const size_t ix = p.add(mat_bytes(T, Kp)), iw = p.add(mat_bytes(Np, Kp)),
               ib = p.add(b ? mat_bytes(1, Np) : 0), iy = p.add(mat_bytes(T, Np));
  FMLP_TRY(pad_alloc(&p, st));
  fmlp_status r = pad_copy(x, T, in, p.at(ix), T, Kp, st);
  if (r == FMLP_OK) r = pad_copy(W, out, in, p.at(iw), Np, Kp, st);
  if (r == FMLP_OK && b) r = pad_copy(b, 1, out, p.at(ib), 1, Np, st);
  if (r == FMLP_OK)
    r = linear_common(p.at(ix), p.at(iw), b ? p.at(ib) : nullptr, p.at(iy), T, Kp, Np, epi,
                      mode, s);
  if (r == FMLP_OK) {
    cudaError_t e = copy2d_launch(p.at(iy), Np, y, out, T, out, st);
    if (e != cudaSuccess) r = cuda_fail(e, "unpadding copy");
  }
  return pad_free(&p, st, r);
}

static fmlp_status linear_common(const void* x, const void* W, const void* b, void* y,
                                 int64_t T, int64_t in, int64_t out, int epi, int mode,
                                 fmlp_stream_t s, int64_t ldx, int64_t ldy) {
  t_last_error.clear();
  FMLP_TRY(check_T(T));
  if ((in % 8 != 0 || out % 8 != 0) && ldx == 0 && ldy == 0)
    return linear_padded(x, W, b, y, T, in, out, epi, mode, s);
  FMLP_TRY(check_inner(in, "in"));
  FMLP_TRY(check_inner(out, "out"));
  FMLP_TRY(resolve_strides(&ldx, &ldy, in, out));
  if (epi == EPI_BIAS_GELU && !act_mode_ok(mode)) {
    set_error("activation mode %d is not FMLP_GELU_TANH, FMLP_GELU_ERF or FMLP_RELU", mode);
    return FMLP_ERR_SHAPE;
  }
  if (T == 0) return FMLP_OK;
  FMLP_NONNULL(x, "x");
  FMLP_NONNULL(W, "W");
  FMLP_NONNULL(y, "y");
  const Range rx{x, mat_bytes(1, in), "x", T, mat_bytes(1, ldx)},
      rw{W, mat_bytes(out, in), "W"}, rb{b, b ? mat_bytes(1, out) : 0, "b"},
      ry{y, mat_bytes(1, out), "y", T, mat_bytes(1, ldy)};
  const Range ins[3] = {rx, rw, rb};
  const Range all[4] = {rx, rw, rb, ry};
  FMLP_TRY(check_ptrs(all, 4));
  FMLP_TRY(check_alias(ry, ins, 3));
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  if (plan_linear(T, in, out, d->sms) == FMLP_PLAN_GEMV)
    return launch_gemv(*d, epi, x, W, nullptr, b, y, T, in, out, mode, st, ldx, ldy);
  return launch_gemm(*d, epi, x, W, nullptr, b, y, T, out, in, mode, false, st, ldx, ldy);
}

fmlp_status fmlp_linear_bias(const void* x, const void* W, const void* b, void* y, int64_t T,
                             int64_t in, int64_t out, fmlp_stream_t s) {
  return linear_common(x, W, b, y, T, in, out, EPI_BIAS, 0, s);
}

fmlp_status fmlp_linear_bias_strided(const void* x, int64_t ldx, const void* W, const void* b,
                                     void* y, int64_t ldy, int64_t T, int64_t in, int64_t out,
                                     fmlp_stream_t s) {
  return linear_common(x, W, b, y, T, in, out, EPI_BIAS, 0, s, ldx, ldy);
}

fmlp_status fmlp_linear_bias_wt(const void* x, const void* Wt, const void* b, void* y,
                                int64_t T, int64_t in, int64_t out, fmlp_stream_t s) {
  t_last_error.clear();
  FMLP_TRY(check_T(T));
  FMLP_TRY(check_inner(in, "in"));
  FMLP_TRY(check_inner(out, "out"));
  if (T == 0) return FMLP_OK;
  FMLP_NONNULL(x, "x");
  FMLP_NONNULL(Wt, "Wt");
  FMLP_NONNULL(y, "y");
  const Range rx{x, mat_bytes(T, in), "x"}, rw{Wt, mat_bytes(in, out), "Wt"},
      rb{b, b ? mat_bytes(1, out) : 0, "b"}, ry{y, mat_bytes(T, out), "y"};
  const Range ins[3] = {rx, rw, rb};
  const Range all[4] = {rx, rw, rb, ry};
  FMLP_TRY(check_ptrs(all, 4));
  FMLP_TRY(check_alias(ry, ins, 3));
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  FMLP_LAUNCH_GUARD("gemm_tc (transposed weights) launch");
  GemmLaunch L;
  memset(&L, 0, sizeof L);
  double cost = 0;
  L.bn = pick_bn(T, out, d->sms, false, &cost) >= 256 ? 256 : 128;
  FMLP_TRY(make_map(&L.tmA, x, T, in, 128, "x"));
  FMLP_TRY(make_map(&L.tmB0, Wt, in, out, 64, "Wt"));   // [in, out]: boxes of 64 out x 64 in
  L.tmB1 = L.tmB0;
  FMLP_TRY(make_map(&L.tmY, y, T, out, 32, "y"));
  L.bias = b;
  L.M = static_cast<int>(T);
  L.N_out = static_cast<int>(out);
  L.K = static_cast<int>(in);
  L.epi = EPI_BIAS;
  L.stream = reinterpret_cast<cudaStream_t>(s);
  L.status = d->status;
  L.timeout_ns = kWaitTimeoutNs;
  const int64_t tiles = ((T + 127) / 128) * ((out + L.bn - 1) / L.bn);
  L.grid = static_cast<int>(std::min<int64_t>(tiles, d->sms));
  const cudaError_t e = gemm_tc_wt_launch(L);
  if (e != cudaSuccess) return cuda_fail(e, "gemm_tc (transposed weights) launch");
  return FMLP_OK;
}

fmlp_status fmlp_linear_bias_gelu(const void* x, const void* W, const void* b, void* h,
                                  int64_t T, int64_t in, int64_t out, fmlp_gelu_mode mode,
                                  fmlp_stream_t s) {
  return linear_common(x, W, b, h, T, in, out, EPI_BIAS_GELU, static_cast<int>(mode), s);
}

fmlp_status fmlp_geglu_gate_up(const void* x, const void* Wg, const void* Wu, void* m, int64_t T,
                               int64_t D, int64_t H, fmlp_stream_t s) {
  t_last_error.clear();
  FMLP_TRY(check_T(T));
  if (D % 8 != 0 || H % 8 != 0) {
    // zero-padded copies of x, Wg, Wu; m's first H columns copied back
    FMLP_TRY(check_ragged(D, "D"));
    FMLP_TRY(check_ragged(H, "H"));
    if (T == 0) return FMLP_OK;
    FMLP_NONNULL(x, "x");
    FMLP_NONNULL(Wg, "Wg");
    FMLP_NONNULL(Wu, "Wu");
    FMLP_NONNULL(m, "m");
    const Range rx{x, mat_bytes(T, D), "x"}, rg{Wg, mat_bytes(H, D), "Wg"},
        ru{Wu, mat_bytes(H, D), "Wu"}, rm{m, mat_bytes(T, H), "m"};
    const Range ins[3] = {rx, rg, ru};
    const Range all[4] = {rx, rg, ru, rm};
    FMLP_TRY(check_ptrs(all, 4));
    FMLP_TRY(check_alias(rm, ins, 3));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
    const int64_t Dp = up8(D), Hp = up8(H);
    PadScratch p;
    const size_t ix = p.add(mat_bytes(T, Dp)), ig = p.add(mat_bytes(Hp, Dp)),
                 iu = p.add(mat_bytes(Hp, Dp)), im = p.add(mat_bytes(T, Hp));
    FMLP_TRY(pad_alloc(&p, st));
    fmlp_status r = pad_copy(x, T, D, p.at(ix), T, Dp, st);
    if (r == FMLP_OK) r = pad_copy(Wg, H, D, p.at(ig), Hp, Dp, st);
    if (r == FMLP_OK) r = pad_copy(Wu, H, D, p.at(iu), Hp, Dp, st);
    if (r == FMLP_OK) r = fmlp_geglu_gate_up(p.at(ix), p.at(ig), p.at(iu), p.at(im), T, Dp, Hp, s);
    if (r == FMLP_OK) {
      cudaError_t e = copy2d_launch(p.at(im), Hp, m, H, T, H, st);
      if (e != cudaSuccess) r = cuda_fail(e, "unpadding copy");
    }
    return pad_free(&p, st, r);
  }
  FMLP_TRY(check_inner(D, "D"));
  FMLP_TRY(check_inner(H, "H"));
  if (T == 0) return FMLP_OK;
  FMLP_NONNULL(x, "x");
  FMLP_NONNULL(Wg, "Wg");
  FMLP_NONNULL(Wu, "Wu");
  FMLP_NONNULL(m, "m");
  const Range rx{x, mat_bytes(T, D), "x"}, rg{Wg, mat_bytes(H, D), "Wg"},
      ru{Wu, mat_bytes(H, D), "Wu"}, rm{m, mat_bytes(T, H), "m"};
  const Range ins[3] = {rx, rg, ru};
  const Range all[4] = {rx, rg, ru, rm};
  FMLP_TRY(check_ptrs(all, 4));
  FMLP_TRY(check_alias(rm, ins, 3));
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  if (gemv_ok(T, D, H, 2, d->sms) && gemv_preferred(T, 2 * mat_bytes(H, D)))
    return launch_gemv(*d, EPI_GEGLU, x, Wg, Wu, nullptr, m, T, D, H, 0, st);
  return launch_gemm(*d, EPI_GEGLU, x, Wg, Wu, nullptr, m, T, H, D, 0, false, st);
}

// ldx, ldy: row strides of x and y in elements (0: packed rows).
static fmlp_status geglu_common(const void* x, int64_t ldx, const void* Wg, const void* Wu,
                                const void* Wd, void* y, int64_t ldy, int64_t T, int64_t D,
                                int64_t H, void* ws, size_t ws_bytes, fmlp_stream_t s);

// The GeGLU block with D or H not a multiple of 8 (the caller's workspace is not used).
static fmlp_status geglu_padded(const void* x, const void* Wg, const void* Wu, const void* Wd,
                                void* y, int64_t T, int64_t D, int64_t H, fmlp_stream_t s) {
  FMLP_TRY(check_ragged(D, "D"));
  FMLP_TRY(check_ragged(H, "H"));
  if (T == 0) return FMLP_OK;
  FMLP_NONNULL(x, "x");
  FMLP_NONNULL(Wg, "Wg");
  FMLP_NONNULL(Wu, "Wu");
  FMLP_NONNULL(Wd, "Wd");
  FMLP_NONNULL(y, "y");
  const Range rx{x, mat_bytes(T, D), "x"}, rg{Wg, mat_bytes(H, D), "Wg"},
      ru{Wu, mat_bytes(H, D), "Wu"}, rd{Wd, mat_bytes(D, H), "Wd"}, ry{y, mat_bytes(T, D), "y"};
  const Range ins[4] = {rx, rg, ru, rd};
  const Range all[5] = {rx, rg, ru, rd, ry};
  FMLP_TRY(check_ptrs(all, 5));
  FMLP_TRY(check_alias(ry, ins, 4));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  const int64_t Dp = up8(D), Hp = up8(H);
  PadScratch p;
  const size_t ix = p.add(mat_bytes(T, Dp)), ig = p.add(mat_bytes(Hp, Dp)),
               iu = p.add(mat_bytes(Hp, Dp)), id = p.add(mat_bytes(Dp, Hp)),
               iy = p.add(mat_bytes(T, Dp));
  FMLP_TRY(pad_alloc(&p, st));
  fmlp_status r = pad_copy(x, T, D, p.at(ix), T, Dp, st);
  if (r == FMLP_OK) r = pad_copy(Wg, H, D, p.at(ig), Hp, Dp, st);
  if (r == FMLP_OK) r = pad_copy(Wu, H, D, p.at(iu), Hp, Dp, st);
  if (r == FMLP_OK) r = pad_copy(Wd, D, H, p.at(id), Dp, Hp, st);
  if (r == FMLP_OK)
    r = geglu_common(p.at(ix), 0, p.at(ig), p.at(iu), p.at(id), p.at(iy), 0, T, Dp, Hp, nullptr,
                     0, s);
  if (r == FMLP_OK) {
    cudaError_t e = copy2d_launch(p.at(iy), Dp, y, D, T, D, st);
    if (e != cudaSuccess) r = cuda_fail(e, "unpadding copy");
  }
  return pad_free(&p, st, r);
}

static fmlp_status geglu_common(const void* x, int64_t ldx, const void* Wg, const void* Wu,
                                const void* Wd, void* y, int64_t ldy, int64_t T, int64_t D,
                                int64_t H, void* ws, size_t ws_bytes, fmlp_stream_t s) {
  t_last_error.clear();
  FMLP_TRY(check_T(T));
  if ((D % 8 != 0 || H % 8 != 0) && ldx == 0 && ldy == 0)
    return geglu_padded(x, Wg, Wu, Wd, y, T, D, H, s);
  FMLP_TRY(check_inner(D, "D"));
  FMLP_TRY(check_inner(H, "H"));
  FMLP_TRY(resolve_strides(&ldx, &ldy, D, D));
  if (T == 0) return FMLP_OK;
  FMLP_NONNULL(x, "x");
  FMLP_NONNULL(Wg, "Wg");
  FMLP_NONNULL(Wu, "Wu");
  FMLP_NONNULL(Wd, "Wd");
  FMLP_NONNULL(y, "y");
  const size_t need = fmlp_geglu_workspace_size(T, D, H);
  if (ws && ws_bytes < need) {
    set_error("workspace has %zu bytes, needs %zu", ws_bytes, need);
    return FMLP_ERR_WORKSPACE;
  }
  const Range rx{x, mat_bytes(1, D), "x", T, mat_bytes(1, ldx)}, rg{Wg, mat_bytes(H, D), "Wg"},
      ru{Wu, mat_bytes(H, D), "Wu"}, rd{Wd, mat_bytes(D, H), "Wd"},
      ry{y, mat_bytes(1, D), "y", T, mat_bytes(1, ldy)}, rw{ws, ws ? need : 0, "workspace"};
  const Range all[6] = {rx, rg, ru, rd, ry, rw};
  FMLP_TRY(check_ptrs(all, 6));
  const Range ins_y[5] = {rx, rg, ru, rd, rw};
  FMLP_TRY(check_alias(ry, ins_y, 5));
  const Range ins_w[4] = {rx, rg, ru, rd};
  FMLP_TRY(check_alias(rw, ins_w, 4));
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  const int plan = plan_geglu(T, D, H, d->sms);
  if (plan == FMLP_PLAN_FUSED_SMALL)
    return launch_small(*d, false, x, Wg, Wu, Wd, nullptr, nullptr, y, T, D, H, D, 0, st, ldx,
                        ldy);
  void* m = ws;
  if (!m) {
    cudaError_t e = cudaMallocAsync(&m, need, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
  }
  fmlp_status r = FMLP_OK;
  bool ran = false;
  if (plan == FMLP_PLAN_DECODE)
    r = launch_decode(*d, true, x, Wg, Wu, nullptr, Wd, nullptr, m, y, T, D, H, D, 0, st, &ran,
                      ldx, ldy);
  if (ran || r != FMLP_OK) {
    // done (or failed) in one kernel
  } else if (plan == FMLP_PLAN_GEMV || (plan == FMLP_PLAN_DECODE && gemv_ok(T, D, H, 2, d->sms) &&
                                        gemv_ok(T, H, D, 1, d->sms))) {
    r = launch_gemv(*d, EPI_GEGLU, x, Wg, Wu, nullptr, m, T, D, H, 0, st, ldx, 0);
    if (r == FMLP_OK)
      r = launch_gemv(*d, EPI_BIAS, m, Wd, nullptr, nullptr, y, T, H, D, 0, st, 0, ldy);
  } else {
    r = launch_fewblock(*d, EPI_GEGLU, x, Wg, Wu, nullptr, Wd, nullptr, m, y, T, D, H, D, 0, st,
                        ldx, ldy, &ran);
    if (r == FMLP_OK && !ran)
      r = launch_two(*d, EPI_GEGLU, x, Wg, Wu, nullptr, Wd, nullptr, m, y, T, D, H, D, 0, st,
                     ldx, ldy, &ran);
    if (r == FMLP_OK && !ran)
      r = launch_gemm(*d, EPI_GEGLU, x, Wg, Wu, nullptr, m, T, H, D, 0, false, st, ldx, 0);
    if (r == FMLP_OK && !ran)
      r = launch_gemm(*d, EPI_BIAS, m, Wd, nullptr, nullptr, y, T, D, H, 0, true, st, 0, ldy);
  }
  if (!ws) {
    cudaError_t e = cudaFreeAsync(m, st);
    if (e != cudaSuccess && r == FMLP_OK) return cuda_fail(e, "cudaFreeAsync(workspace)");
  }
  return r;
}

fmlp_status fmlp_geglu(const void* x, const void* Wg, const void* Wu, const void* Wd, void* y,
                       int64_t T, int64_t D, int64_t H, void* ws, size_t ws_bytes,
                       fmlp_stream_t s) {
  return geglu_common(x, 0, Wg, Wu, Wd, y, 0, T, D, H, ws, ws_bytes, s);
}

fmlp_status fmlp_geglu_strided(const void* x, int64_t ldx, const void* Wg, const void* Wu,
                               const void* Wd, void* y, int64_t ldy, int64_t T, int64_t D,
                               int64_t H, void* ws, size_t ws_bytes, fmlp_stream_t s) {
  return geglu_common(x, ldx, Wg, Wu, Wd, y, ldy, T, D, H, ws, ws_bytes, s);
}

size_t fmlp_moe_geglu_workspace_size(int64_t T, int64_t D, int64_t H) {
  (void)D;
  return T > 0 && H > 0 ? mat_bytes(T, H) : 0;
}

fmlp_status fmlp_moe_geglu(const void* x, const int32_t* offsets, int64_t E, const void* Wg,
                           const void* Wu, const void* Wd, void* y, int64_t T, int64_t D,
                           int64_t H, void* ws, size_t ws_bytes, fmlp_stream_t s) {
  t_last_error.clear();
  FMLP_TRY(check_T(T));
  FMLP_TRY(check_inner(D, "D"));
  FMLP_TRY(check_inner(H, "H"));
  if (E < 1 || E > kMoeMaxExperts) {
    set_error("E = %lld experts is outside [1, %d]", static_cast<long long>(E), kMoeMaxExperts);
    return FMLP_ERR_SHAPE;
  }
  if (T == 0) return FMLP_OK;
  FMLP_NONNULL(x, "x");
  FMLP_NONNULL(offsets, "offsets");
  FMLP_NONNULL(Wg, "Wg");
  FMLP_NONNULL(Wu, "Wu");
  FMLP_NONNULL(Wd, "Wd");
  FMLP_NONNULL(y, "y");
  const size_t need = mat_bytes(T, H);
  if (ws && ws_bytes < need) {
    set_error("workspace has %zu bytes, needs %zu", ws_bytes, need);
    return FMLP_ERR_WORKSPACE;
  }
  if (reinterpret_cast<uintptr_t>(offsets) % 4 != 0) {
    set_error("offsets is not 4-byte aligned");
    return FMLP_ERR_ALIGN;
  }
  const size_t wbytes = static_cast<size_t>(E) * mat_bytes(H, D);
  const Range rx{x, mat_bytes(T, D), "x"}, rg{Wg, wbytes, "Wg"}, ru{Wu, wbytes, "Wu"},
      rd{Wd, wbytes, "Wd"}, ry{y, mat_bytes(T, D), "y"}, rw{ws, ws ? need : 0, "workspace"},
      ro{offsets, static_cast<size_t>(E + 1) * 4u, "offsets"};
  const Range all[6] = {rx, rg, ru, rd, ry, rw};
  FMLP_TRY(check_ptrs(all, 6));
  const Range ins_y[6] = {rx, rg, ru, rd, rw, ro};
  FMLP_TRY(check_alias(ry, ins_y, 6));
  const Range ins_w[5] = {rx, rg, ru, rd, ro};
  FMLP_TRY(check_alias(rw, ins_w, 5));
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  void* m = ws;
  if (!m) {
    cudaError_t e = cudaMallocAsync(&m, need, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
  }
  fmlp_status r = FMLP_OK;
  // CTA pairs (256-row tiles, each CTA loading 128 weight rows) when the device runs them
  const bool pair = d->max_pairs >= 1 &&
                    g_tile_policy.load(std::memory_order_relaxed) != FMLP_TILES_SINGLE;
  for (int stage = 0; stage < 2 && r == FMLP_OK; ++stage) {
    // stage 0: m = gelu_tanh(x Wg[e]^T) * (x Wu[e]^T); stage 1: y = m Wd[e]^T
    GemmLaunch L;
    memset(&L, 0, sizeof L);
    const bool gu = stage == 0;
    const void* A = gu ? x : m;
    const int64_t K = gu ? D : H, N = gu ? H : D;
    if ((r = make_map(&L.tmA, A, T, K, 128, gu ? "x" : "m")) != FMLP_OK) break;
    if (gu) {
      if ((r = make_map3(&L.tmB0, Wg, E, H, D, 128, "Wg")) != FMLP_OK) break;
      if ((r = make_map3(&L.tmB1, Wu, E, H, D, 128, "Wu")) != FMLP_OK) break;
    } else {
      if ((r = make_map3(&L.tmB0, Wd, E, D, H, pair ? 128 : 256, "Wd")) != FMLP_OK) break;
      L.tmB1 = L.tmB0;
    }
    L.tmY = L.tmA;   // unused: the grouped epilogue stores directly
    L.M = static_cast<int>(T);
    L.N_out = static_cast<int>(N);
    L.K = static_cast<int>(K);
    L.epi = gu ? EPI_GEGLU : EPI_BIAS;
    L.bn = 256;
    // persistent: the tile count is only known on the device
    L.grid = pair ? 2 * d->max_pairs : d->sms;
    L.pdl = !gu;
    L.stream = st;
    L.status = d->status;
    L.timeout_ns = kWaitTimeoutNs;
    L.offsets = offsets;
    L.groups = static_cast<int>(E);
    L.ydir = gu ? m : y;
    L.ldy = static_cast<int>(N);
    if (take_injection(g_inject_launch)) {
      set_error("grouped gemm launch: injected launch failure (fmlp_test_inject)");
      r = FMLP_ERR_CUDA;
      break;
    }
    const cudaError_t e = pair ? gemm_tc2_grouped_launch(L) : gemm_tc_grouped_launch(L);
    if (e != cudaSuccess) r = cuda_fail(e, "grouped gemm launch");
  }
  if (!ws) {
    cudaError_t e = cudaFreeAsync(m, st);
    if (e != cudaSuccess && r == FMLP_OK) return cuda_fail(e, "cudaFreeAsync(workspace)");
  }
  return r;
}

// ldx, ldy: row strides of x and y in elements (0: packed rows).
static fmlp_status mlp_common(const void* x, int64_t ldx, const void* W1, const void* b1,
                              const void* W2, const void* b2, void* y, int64_t ldy, int64_t T,
                              int64_t D, int64_t H, int64_t Dout, fmlp_gelu_mode mode, void* ws,
                              size_t ws_bytes, fmlp_stream_t s);

// The MLP block with D, H or Dout not a multiple of 8 (the caller's workspace is not used).
static fmlp_status mlp_padded(const void* x, const void* W1, const void* b1, const void* W2,
                              const void* b2, void* y, int64_t T, int64_t D, int64_t H,
                              int64_t Dout, fmlp_gelu_mode mode, fmlp_stream_t s) {
  FMLP_TRY(check_ragged(D, "D"));
  FMLP_TRY(check_ragged(H, "H"));
  FMLP_TRY(check_ragged(Dout, "Dout"));
  if (!act_mode_ok(mode)) {
    set_error("activation mode %d is not FMLP_GELU_TANH, FMLP_GELU_ERF or FMLP_RELU",
              static_cast<int>(mode));
    return FMLP_ERR_SHAPE;
  }
  if (T == 0) return FMLP_OK;
  FMLP_NONNULL(x, "x");
  FMLP_NONNULL(W1, "W1");
  FMLP_NONNULL(W2, "W2");
  FMLP_NONNULL(y, "y");
  const Range rx{x, mat_bytes(T, D), "x"}, r1{W1, mat_bytes(H, D), "W1"},
      rb1{b1, b1 ? mat_bytes(1, H) : 0, "b1"}, r2{W2, mat_bytes(Dout, H), "W2"},
      rb2{b2, b2 ? mat_bytes(1, Dout) : 0, "b2"}, ry{y, mat_bytes(T, Dout), "y"};
  const Range ins[5] = {rx, r1, rb1, r2, rb2};
  const Range all[6] = {rx, r1, rb1, r2, rb2, ry};
  FMLP_TRY(check_ptrs(all, 6));
  FMLP_TRY(check_alias(ry, ins, 5));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  const int64_t Dp = up8(D), Hp = up8(H), Op = up8(Dout);
  PadScratch p;
  const size_t ix = p.add(mat_bytes(T, Dp)), i1 = p.add(mat_bytes(Hp, Dp)),
               ib1 = p.add(b1 ? mat_bytes(1, Hp) : 0), i2 = p.add(mat_bytes(Op, Hp)),
               ib2 = p.add(b2 ? mat_bytes(1, Op) : 0), iy = p.add(mat_bytes(T, Op));
  FMLP_TRY(pad_alloc(&p, st));
  fmlp_status r = pad_copy(x, T, D, p.at(ix), T, Dp, st);
  if (r == FMLP_OK) r = pad_copy(W1, H, D, p.at(i1), Hp, Dp, st);
  if (r == FMLP_OK && b1) r = pad_copy(b1, 1, H, p.at(ib1), 1, Hp, st);
  if (r == FMLP_OK) r = pad_copy(W2, Dout, H, p.at(i2), Op, Hp, st);
  if (r == FMLP_OK && b2) r = pad_copy(b2, 1, Dout, p.at(ib2), 1, Op, st);
  if (r == FMLP_OK)
    r = mlp_common(p.at(ix), 0, p.at(i1), b1 ? p.at(ib1) : nullptr, p.at(i2),
                   b2 ? p.at(ib2) : nullptr, p.at(iy), 0, T, Dp, Hp, Op, mode, nullptr, 0, s);
  if (r == FMLP_OK) {
    cudaError_t e = copy2d_launch(p.at(iy), Op, y, Dout, T, Dout, st);
    if (e != cudaSuccess) r = cuda_fail(e, "unpadding copy");
  }
  return pad_free(&p, st, r);
}

static fmlp_status mlp_common(const void* x, int64_t ldx, const void* W1, const void* b1,
                              const void* W2, const void* b2, void* y, int64_t ldy, int64_t T,
                              int64_t D, int64_t H, int64_t Dout, fmlp_gelu_mode mode, void* ws,
                              size_t ws_bytes, fmlp_stream_t s) {
  t_last_error.clear();
  FMLP_TRY(check_T(T));
  if ((D % 8 != 0 || H % 8 != 0 || Dout % 8 != 0) && ldx == 0 && ldy == 0)
    return mlp_padded(x, W1, b1, W2, b2, y, T, D, H, Dout, mode, s);
  FMLP_TRY(check_inner(D, "D"));
  FMLP_TRY(check_inner(H, "H"));
  FMLP_TRY(check_inner(Dout, "Dout"));
  FMLP_TRY(resolve_strides(&ldx, &ldy, D, Dout));
  if (!act_mode_ok(mode)) {
    set_error("activation mode %d is not FMLP_GELU_TANH, FMLP_GELU_ERF or FMLP_RELU",
              static_cast<int>(mode));
    return FMLP_ERR_SHAPE;
  }
  if (T == 0) return FMLP_OK;
  FMLP_NONNULL(x, "x");
  FMLP_NONNULL(W1, "W1");
  FMLP_NONNULL(W2, "W2");
  FMLP_NONNULL(y, "y");
  const size_t need = fmlp_mlp_gelu_workspace_size(T, D, H, Dout);
  if (ws && ws_bytes < need) {
    set_error("workspace has %zu bytes, needs %zu", ws_bytes, need);
    return FMLP_ERR_WORKSPACE;
  }
  const Range rx{x, mat_bytes(1, D), "x", T, mat_bytes(1, ldx)}, r1{W1, mat_bytes(H, D), "W1"},
      rb1{b1, b1 ? mat_bytes(1, H) : 0, "b1"}, r2{W2, mat_bytes(Dout, H), "W2"},
      rb2{b2, b2 ? mat_bytes(1, Dout) : 0, "b2"},
      ry{y, mat_bytes(1, Dout), "y", T, mat_bytes(1, ldy)}, rw{ws, ws ? need : 0, "workspace"};
  const Range all[7] = {rx, r1, rb1, r2, rb2, ry, rw};
  FMLP_TRY(check_ptrs(all, 7));
  const Range ins_y[6] = {rx, r1, rb1, r2, rb2, rw};
  FMLP_TRY(check_alias(ry, ins_y, 6));
  const Range ins_w[5] = {rx, r1, rb1, r2, rb2};
  FMLP_TRY(check_alias(rw, ins_w, 5));
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  const int plan = plan_mlp(T, D, H, Dout, d->sms);
  if (plan == FMLP_PLAN_FUSED_SMALL)
    return launch_small(*d, true, x, W1, nullptr, W2, b1, b2, y, T, D, H, Dout,
                        static_cast<int>(mode), st, ldx, ldy);
  void* h = ws;
  if (!h) {
    cudaError_t e = cudaMallocAsync(&h, need, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
  }
  fmlp_status r = FMLP_OK;
  bool ran = false;
  if (plan == FMLP_PLAN_DECODE)
    r = launch_decode(*d, false, x, W1, nullptr, b1, W2, b2, h, y, T, D, H, Dout,
                      static_cast<int>(mode), st, &ran, ldx, ldy);
  if (ran || r != FMLP_OK) {
    // done (or failed) in one kernel
  } else if (plan == FMLP_PLAN_GEMV ||
             (plan == FMLP_PLAN_DECODE && gemv_ok(T, D, H, 1, d->sms) &&
              gemv_ok(T, H, Dout, 1, d->sms))) {
    r = launch_gemv(*d, EPI_BIAS_GELU, x, W1, nullptr, b1, h, T, D, H, static_cast<int>(mode),
                    st, ldx, 0);
    if (r == FMLP_OK)
      r = launch_gemv(*d, EPI_BIAS, h, W2, nullptr, b2, y, T, H, Dout, 0, st, 0, ldy);
  } else {
    r = launch_fewblock(*d, EPI_BIAS_GELU, x, W1, nullptr, b1, W2, b2, h, y, T, D, H, Dout,
                        static_cast<int>(mode), st, ldx, ldy, &ran);
    if (r == FMLP_OK && !ran)
      r = launch_two(*d, EPI_BIAS_GELU, x, W1, nullptr, b1, W2, b2, h, y, T, D, H, Dout,
                     static_cast<int>(mode), st, ldx, ldy, &ran);
    if (r == FMLP_OK && !ran)
      r = launch_gemm(*d, EPI_BIAS_GELU, x, W1, nullptr, b1, h, T, H, D,
                      static_cast<int>(mode), false, st, ldx, 0);
    if (r == FMLP_OK && !ran)
      r = launch_gemm(*d, EPI_BIAS, h, W2, nullptr, b2, y, T, Dout, H, 0, true, st, 0, ldy);
  }
  if (!ws) {
    cudaError_t e = cudaFreeAsync(h, st);
    if (e != cudaSuccess && r == FMLP_OK) return cuda_fail(e, "cudaFreeAsync(workspace)");
  }
  return r;
}

fmlp_status fmlp_mlp_gelu(const void* x, const void* W1, const void* b1, const void* W2,
                          const void* b2, void* y, int64_t T, int64_t D, int64_t H, int64_t Dout,
                          fmlp_gelu_mode mode, void* ws, size_t ws_bytes, fmlp_stream_t s) {
  return mlp_common(x, 0, W1, b1, W2, b2, y, 0, T, D, H, Dout, mode, ws, ws_bytes, s);
}

fmlp_status fmlp_mlp_gelu_strided(const void* x, int64_t ldx, const void* W1, const void* b1,
                                  const void* W2, const void* b2, void* y, int64_t ldy,
                                  int64_t T, int64_t D, int64_t H, int64_t Dout,
                                  fmlp_gelu_mode mode, void* ws, size_t ws_bytes,
                                  fmlp_stream_t s) {
  return mlp_common(x, ldx, W1, b1, W2, b2, y, ldy, T, D, H, Dout, mode, ws, ws_bytes, s);
}

static std::string describe_gemm(const DeviceState& d, const char* name, int epi, int64_t M,
                                 int64_t N, int64_t K) {
  if (use_skinny(M)) {
    const SkinnyShape sh = skinny_shape(d, N, K, (M + 31) / 32 * 32);
    char b[256];
    snprintf(b, sizeof b,
             "%s: tcgen05 few-token kernel, %d weight rows x %lld tokens per tile, K split %d "
             "ways over a cluster, M=%lld N=%lld K=%lld, grid=%lld",
             name, sh.rows, static_cast<long long>((M + 31) / 32 * 32), sh.split,
             static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K),
             static_cast<long long>(sh.tiles) * sh.split);
    return b;
  }
  const GemmChoice c = choose_gemm(d, epi, M, N);
  char b[256];
  if (c.pair)
    snprintf(b, sizeof b, "%s: tcgen05 CTA-pair 256x%d tiles, M=%lld N=%lld K=%lld, grid=%d",
             name, c.bn, static_cast<long long>(M), static_cast<long long>(N),
             static_cast<long long>(K), c.grid);
  else
    snprintf(b, sizeof b, "%s: tcgen05 single-SM 128x%d tiles, M=%lld N=%lld K=%lld, grid=%d",
             name, c.bn, static_cast<long long>(M), static_cast<long long>(N),
             static_cast<long long>(K), c.grid);
  return b;
}

static std::string describe_gemv(const DeviceState& d, const char* name, int64_t T, int64_t K,
                                 int64_t N, int nmat = 1) {
  char b[256];
  snprintf(b, sizeof b, "%s: weight-streaming GEMV, T=%lld K=%lld N=%lld, grid=%lld", name,
           static_cast<long long>(T), static_cast<long long>(K), static_cast<long long>(N),
           static_cast<long long>(gemv_grid(static_cast<int>(T), static_cast<int>(K),
                                            static_cast<int>(N), nmat, d.sms)));
  return b;
}

static std::string describe_decode(const DeviceState& d, const char* name, int64_t T, int64_t D,
                                   int64_t H, int64_t Dout, int nmat) {
  char b[256];
  snprintf(b, sizeof b,
           "%s: one weight-streaming kernel for both layers (grid barrier between them), "
           "T=%lld D=%lld H=%lld Dout=%lld, grid=%d, ring of %d bulk-copy stages of whole rows",
           name, static_cast<long long>(T), static_cast<long long>(D), static_cast<long long>(H),
           static_cast<long long>(Dout), d.sms,
           decode_ring_stages(static_cast<int>(T), static_cast<int>(D), static_cast<int>(H),
                              static_cast<int>(Dout), nmat, d.sms));
  return b;
}

static std::string describe_fewblock(const FewBlockPlan& p, const char* name1, int64_t T,
                                     int64_t D, int64_t H, int64_t Dout) {
  char b[384];
  snprintf(b, sizeof b,
           "%s and down: one few-token tcgen05 launch for both layers (weights as the M side, "
           "%d + %d weight rows x %d tokens per tile, K split %d ways over a cluster, layer 2's "
           "weights prefetched before a grid barrier on h), T=%lld D=%lld H=%lld Dout=%lld, "
           "grid=%d",
           name1, p.rows1, p.rows2, p.tpad, p.split, static_cast<long long>(T),
           static_cast<long long>(D), static_cast<long long>(H), static_cast<long long>(Dout),
           p.tiles * p.split);
  return b;
}

static std::string describe_two(const TwoPlan& tp, const char* name1, int64_t T, int64_t D,
                                int64_t H, int64_t Dout) {
  char b[384];
  snprintf(b, sizeof b,
           "%s and down: one tcgen05 CTA-pair launch for both layers, %d first-stage and %d "
           "down 256-row tiles listed over %d pairs (each band's down tiles after its "
           "first-stage tiles), T=%lld D=%lld H=%lld Dout=%lld, grid=%d",
           name1, tp.num_m * tp.num_n1, tp.num_m * tp.num_n2, tp.pairs,
           static_cast<long long>(T), static_cast<long long>(D), static_cast<long long>(H),
           static_cast<long long>(Dout), 2 * tp.pairs);
  return b;
}

fmlp_status fmlp_describe_plan(int op, int64_t T, int64_t D, int64_t H, int64_t Dout, char* buf,
                               size_t buflen) {
  t_last_error.clear();
  if (!buf || buflen == 0) {
    set_error("buf is NULL or empty");
    return FMLP_ERR_NULL;
  }
  buf[0] = 0;
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  std::string r;
  if (T > 0 && (D % 8 != 0 || H % 8 != 0 || (op == 4 && Dout % 8 != 0))) {
    char b[200];
    snprintf(b, sizeof b, "zero-padded copies (inner dims %lld, %lld%s%s -> multiples of 8), then ",
             static_cast<long long>(D), static_cast<long long>(H), op == 4 ? ", " : "",
             op == 4 ? std::to_string(static_cast<long long>(Dout)).c_str() : "");
    r = b;
    D = up8(D);
    H = up8(H);
    Dout = up8(Dout);
  }
  if (T <= 0) {
    r = "nothing launched (T = 0)";
  } else if (op == 0 || op == 1) {   // linear (+gelu): D -> H
    const int epi = op == 0 ? EPI_BIAS : EPI_BIAS_GELU;
    r += plan_linear(T, D, H, d->sms) == FMLP_PLAN_GEMV ? describe_gemv(*d, "linear", T, D, H)
                                                        : describe_gemm(*d, "linear", epi, T, H, D);
  } else if (op == 2) {              // gate/up
    r += gemv_ok(T, D, H, 2, d->sms) && gemv_preferred(T, 2 * mat_bytes(H, D))
             ? describe_gemv(*d, "gate/up", T, D, H, 2)
             : describe_gemm(*d, "gate/up", EPI_GEGLU, T, H, D);
  } else if (op == 3) {              // geglu block
    const int p = plan_geglu(T, D, H, d->sms);
    if (p == FMLP_PLAN_DECODE) {
      r += describe_decode(*d, "GeGLU block", T, D, H, D, 2);
    } else if (p == FMLP_PLAN_FUSED_SMALL) {
      char b[160];
      snprintf(b, sizeof b, "fused block: one kernel, grid=%lld", static_cast<long long>((T + 127) / 128));
      r += b;
    } else if (p == FMLP_PLAN_GEMV) {
      r += describe_gemv(*d, "gate/up", T, D, H, 2) + "; " + describe_gemv(*d, "down", T, H, D);
    } else if (const FewBlockPlan fp = plan_fewblock(*d, EPI_GEGLU, T, D, H, D); fp.ok) {
      r += describe_fewblock(fp, "gate/up", T, D, H, D);
    } else if (const TwoPlan tp = plan_two(*d, EPI_GEGLU, T, D, H, D); tp.pairs > 0) {
      r += describe_two(tp, "gate/up", T, D, H, D);
    } else {
      r += describe_gemm(*d, "gate/up", EPI_GEGLU, T, H, D) + "; " +
           describe_gemm(*d, "down", EPI_BIAS, T, D, H);
    }
  } else if (op == 4) {              // mlp: D -> H -> Dout
    const int p = plan_mlp(T, D, H, Dout, d->sms);
    if (p == FMLP_PLAN_FUSED_SMALL) {
      char b[160];
      snprintf(b, sizeof b, "fused block: one kernel, grid=%lld",
               static_cast<long long>((T + 127) / 128));
      r += b;
    } else if (p == FMLP_PLAN_DECODE)
      r += describe_decode(*d, "MLP block", T, D, H, Dout, 1);
    else if (p == FMLP_PLAN_GEMV)
      r += describe_gemv(*d, "up", T, D, H) + "; " + describe_gemv(*d, "down", T, H, Dout);
    else if (const FewBlockPlan fp = plan_fewblock(*d, EPI_BIAS_GELU, T, D, H, Dout); fp.ok)
      r += describe_fewblock(fp, "up", T, D, H, Dout);
    else if (const TwoPlan tp = plan_two(*d, EPI_BIAS_GELU, T, D, H, Dout); tp.pairs > 0)
      r += describe_two(tp, "up", T, D, H, Dout);
    else
      r += describe_gemm(*d, "up", EPI_BIAS_GELU, T, H, D) + "; " +
           describe_gemm(*d, "down", EPI_BIAS, T, Dout, H);
  } else {
    set_error("op %d unknown", op);
    return FMLP_ERR_SHAPE;
  }
  snprintf(buf, buflen, "%s", r.c_str());
  return FMLP_OK;
}

fmlp_status fmlp_set_tile_policy(int policy) {
  if (policy != FMLP_TILES_AUTO && policy != FMLP_TILES_SINGLE && policy != FMLP_TILES_PAIR) {
    set_error("tile policy %d unknown", policy);
    return FMLP_ERR_SHAPE;
  }
  g_tile_policy.store(policy, std::memory_order_relaxed);
  return FMLP_OK;
}

fmlp_status fmlp_gelu_eval(const float* in, float* out, int64_t n, fmlp_gelu_mode mode,
                           fmlp_stream_t s) {
  t_last_error.clear();
  if (n < 0) {
    set_error("n = %lld < 0", static_cast<long long>(n));
    return FMLP_ERR_SHAPE;
  }
  if (!act_mode_ok(mode)) {
    set_error("activation mode %d invalid", static_cast<int>(mode));
    return FMLP_ERR_SHAPE;
  }
  if (n == 0) return FMLP_OK;
  FMLP_NONNULL(in, "in");
  FMLP_NONNULL(out, "out");
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  cudaError_t e = gelu_eval_launch(in, out, n, static_cast<int>(mode),
                                   reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return cuda_fail(e, "gelu_eval launch");
  return FMLP_OK;
}

fmlp_status fmlp_device_status(fmlp_stream_t s) {
  t_last_error.clear();
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  if ((e = cudaMemcpy(&v, d->status, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read device status");
  if (v == 0) return FMLP_OK;
  const int zero = 0;
  if ((e = cudaMemcpy(d->status, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail(e, "clear device status");

  static const char* sites[] = {"?",          "test wait",          "producer (empty slot)",
                                "MMA (full slot)", "MMA (free accumulator)", "epilogue (accumulator)",
                                "drain",      "fused kernel", "GEMV",
                                "decode (layer-2 weight copy)", "decode (grid barrier)",
                                "two-stage block (band of the intermediate)",
                                "few-token block (grid barrier)"};
  const int site = v >> 8;
  set_error("a kernel gave up waiting at: %s (code 0x%x)",
            (site >= 0 && site < static_cast<int>(sizeof sites / sizeof sites[0])) ? sites[site]
                                                                                     : "?",
            v);
  return static_cast<fmlp_status>(v & 0xFF);
}

fmlp_status fmlp_test_inject(int kind, int64_t count, int64_t timeout_us) {
  t_last_error.clear();
  if (count < 0 || count > 1000000 || timeout_us < 0 || timeout_us > 2000000) {
    set_error("count = %lld (0..1000000) or timeout_us = %lld (0..2000000) out of range",
              static_cast<long long>(count), static_cast<long long>(timeout_us));
    return FMLP_ERR_SHAPE;
  }
  switch (kind) {
    case FMLP_INJECT_NONE:
      g_inject_launch.store(0);
      g_inject_skip.store(0);
      g_inject_timeout_ns.store(0);
      return FMLP_OK;
    case FMLP_INJECT_LAUNCH:
      g_inject_launch.store(static_cast<int>(count));
      return FMLP_OK;
    case FMLP_INJECT_SKIP_LOAD:
      g_inject_timeout_ns.store(static_cast<unsigned long long>(timeout_us) * 1000ull);
      g_inject_skip.store(static_cast<int>(count));
      return FMLP_OK;
    default:
      set_error("injection kind %d unknown", kind);
      return FMLP_ERR_SHAPE;
  }
}

fmlp_status fmlp_test_decode_overload(int64_t extra_ctas, int64_t timeout_us) {
  t_last_error.clear();
  if (extra_ctas < 0 || extra_ctas > 4096 || timeout_us < 0 || timeout_us > 2000000) {
    set_error("extra_ctas = %lld (0..4096) or timeout_us = %lld (0..2000000) out of range",
              static_cast<long long>(extra_ctas), static_cast<long long>(timeout_us));
    return FMLP_ERR_SHAPE;
  }
  g_decode_extra_ctas.store(static_cast<int>(extra_ctas), std::memory_order_relaxed);
  g_decode_timeout_ns.store(static_cast<unsigned long long>(timeout_us) * 1000ull,
                            std::memory_order_relaxed);
  return FMLP_OK;
}

fmlp_status fmlp_test_prefer_decode(int on) {
  t_last_error.clear();
  if (on != 0 && on != 1) {
    set_error("on = %d, expected 0 or 1", on);
    return FMLP_ERR_SHAPE;
  }
  g_prefer_decode.store(on, std::memory_order_relaxed);
  return FMLP_OK;
}

fmlp_status fmlp_test_two_stage_schedule(int num_m, int num_n1, int num_n2, int kb1, int kb2,
                                         int pairs, uint16_t* start, uint16_t* item,
                                         int64_t* n_items) {
  t_last_error.clear();
  if (!start || !item || !n_items) {
    set_error("start, item and n_items must not be NULL");
    return FMLP_ERR_NULL;
  }
  if (num_m < 1 || num_m > kTwoMaxBands || num_n1 < 1 || num_n2 < 1 || kb1 < 1 || kb2 < 1 ||
      pairs < 1 || pairs > kTwoMaxPairs ||
      static_cast<int64_t>(num_m) * (num_n1 + num_n2) > kTwoMaxItems) {
    set_error("schedule shape out of range");
    return FMLP_ERR_SHAPE;
  }
  const TwoSchedule sc = two_schedule(num_m, num_n1, num_n2, kb1, kb2, pairs);
  for (int i = 0; i <= pairs; ++i) start[i] = sc.start[i];
  for (size_t i = 0; i < sc.item.size(); ++i) item[i] = sc.item[i];
  *n_items = static_cast<int64_t>(sc.item.size());
  return FMLP_OK;
}

fmlp_status fmlp_test_fewtoken_block(int mode) {
  t_last_error.clear();
  if (mode < -1 || mode > 1) {
    set_error("mode = %d, expected -1, 0 or 1", mode);
    return FMLP_ERR_SHAPE;
  }
  g_fewblock.store(mode, std::memory_order_relaxed);
  return FMLP_OK;
}

fmlp_status fmlp_test_two_stage(int mode) {
  t_last_error.clear();
  if (mode < -1 || mode > 1) {
    set_error("mode = %d, expected -1, 0 or 1", mode);
    return FMLP_ERR_SHAPE;
  }
  g_two_stage.store(mode, std::memory_order_relaxed);
  return FMLP_OK;
}

fmlp_status fmlp_test_wait_timeout(int64_t timeout_us, fmlp_stream_t s) {
  t_last_error.clear();
  if (timeout_us < 1 || timeout_us > 2000000) {
    set_error("timeout_us = %lld out of range [1, 2000000]", static_cast<long long>(timeout_us));
    return FMLP_ERR_SHAPE;
  }
  DeviceState* d = nullptr;
  FMLP_TRY(device_state(&d));
  cudaError_t e = wait_timeout_launch(static_cast<uint64_t>(timeout_us) * 1000u, d->status,
                                      reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return cuda_fail(e, "wait_timeout launch");
  return FMLP_OK;
}

}  // extern "C"
