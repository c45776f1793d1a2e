/*
 * fmlp.h - C ABI of the fused transformer feed-forward library for GB300 (sm_103a).
 *
 * Operations (all source citations are to "Profiling in PyTorch (Part 2): From nn.Linear to
 * a Fused MLP" unless another page is named):
 *   fmlp_linear_bias   y = x @ W^T + b with the bias added in the GEMM epilogue
 *                      (sections "From matmul-add to Linear" and "Why are there no separate
 *                      mul and add kernels?"; the weight is read in its stored [out, in]
 *                      layout, the transpose being only a view, section "Where did the
 *                      transpose go? Kernel layouts and pre-ops").
 *   fmlp_geglu         the GeGLU feed-forward block of section "Stacking three Linears: the
 *                      MLP": g = x Wg^T, u = x Wu^T, m = gelu_tanh(g) * u, y = m Wd^T, with
 *                      gelu(g)*u fused into the gate/up GEMM epilogue (sections "The fused
 *                      Triton kernel" and "Why tuned kernels are better" fuse it as a separate
 *                      pointwise pass; here it never leaves the GEMM).
 *   fmlp_mlp_gelu      Linear -> GELU -> Linear with biases, y = W2 GELU(W1 x + b1) + b2
 *                      (ainews.cool fused-MLP article, technical deep-dive and benchmark
 *                      sections: one launch instead of three at batch 1); ReLU may replace
 *                      the GELU (the same article's two-layer ReLU MLP).
 *   fmlp_moe_geglu     a mixture of experts, each a GeGLU block over the tokens routed to it
 *                      (the same article's MoE note), one launch per stage over all experts.
 *   fmlp_*_strided     the calls above on row-strided views of x and y (section "What's the
 *                      transpose doing?").
 *
 * Common conventions
 *   - Tensors are dense, row-major (last index fastest), contiguous (except the x and y views
 *     of the *_strided calls), bfloat16 bit patterns in device memory. x is [T, in]; weights
 *     use the nn.Linear layout [out, in]; biases [out].
 *     T is the token count batch*seq (section "Why are there two kinds of GEMM kernels?").
 *   - Accumulation is fp32. The bias is added in fp32 before the activation. The output and
 *     the one intermediate (m or h) are each rounded to bf16 once, round-to-nearest-even.
 *   - Every call is asynchronous on the caller's stream `s` (NULL = legacy default stream)
 *     and launches only hand-written kernels. Results are valid once `s` has synchronised.
 *     Results are deterministic: no atomics take part in any sum.
 *   - Ownership: all tensor and workspace pointers belong to the caller; the library keeps
 *     none of them after the call returns. The library owns host caches (per device: SM
 *     count, CUDA function attributes, the stream -> counter-row table of the decode plan and
 *     the two-stage block launch; per process: encoded TMA tensor maps, keyed by address,
 *     sizes, strides and box, so an entry is valid for any buffer at that address with those
 *     sizes, and the two-stage launches' item lists, keyed by shape), guarded by mutexes, and
 *     four arrays of its own device memory on every GPU it runs on, held until the process
 *     exits: the status word below, the decode plan's grid-barrier counters (1024 x 128
 *     bytes), the two-stage launches' band counters (1024 x 512 bytes), and the 64 MiB
 *     scratch of fmlp_geglu_noalloc. The calls are thread-safe, with two exceptions stated
 *     where they apply: fmlp_geglu_noalloc calls must not overlap on the GPU, and
 *     FMLP_PLAN_DECODE and the two-stage launch keep one row of counters per stream (a launch
 *     captured in a CUDA graph keeps its stream's row: replays of that graph must not overlap
 *     one another or other launches on that stream).
 *     The library looks up the device addresses of its arrays once per device; a device reset
 *     (cudaDeviceReset) while the library is loaded leaves them stale and is not supported.
 *   - Requirements checked before anything is launched (the status names the first failure):
 *       FMLP_ERR_NULL       a required pointer is NULL
 *       FMLP_ERR_SHAPE      T < 0, or an inner dimension (in/out/D/H/Dout) < 1, or a
 *                           dimension above 2^31 - 8; for the strided calls (with a row
 *                           stride given), fmlp_moe_geglu and fmlp_geglu_noalloc also an
 *                           inner dimension that is not a multiple of 8
 *       FMLP_ERR_ALIGN      a tensor pointer not 16-byte aligned
 *       FMLP_ERR_ALIAS      the output overlaps an input (or the workspace)
 *       FMLP_ERR_WORKSPACE  ws_bytes smaller than the matching *_workspace_size()
 *       FMLP_ERR_DEVICE     the current device is not compute capability 10.3
 *     T == 0 returns FMLP_OK and launches nothing. A failed launch returns FMLP_ERR_CUDA with
 *     the CUDA error text in fmlp_last_error(). The library never aborts the process.
 *   - Device-side waits are bounded (about one second). A wait that runs out makes the kernel
 *     record the fault in a per-device status word and return early; the output is then
 *     undefined and fmlp_device_status() reports FMLP_ERR_DEVICE_TIMEOUT.
 */
#ifndef FMLP_H_
#define FMLP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FMLP_API __attribute__((visibility("default")))
#else
#define FMLP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
struct CUstream_st;
typedef struct CUstream_st* fmlp_stream_t;

typedef enum {
    FMLP_OK = 0,
    FMLP_ERR_NULL = 1,
    FMLP_ERR_SHAPE = 2,
    FMLP_ERR_ALIGN = 3,
    FMLP_ERR_ALIAS = 4,
    FMLP_ERR_WORKSPACE = 5,
    FMLP_ERR_CUDA = 6,
    FMLP_ERR_DEVICE_TIMEOUT = 7,
    FMLP_ERR_DEVICE = 8
} fmlp_status;

/* Hidden activation of the MLP calls. GELU_TANH: 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))),
 * the approximate="tanh" form of section "Stacking three Linears: the MLP". GELU_ERF: the exact
 * 0.5 x (1 + erf(x / sqrt 2)), nn.GELU's default. RELU: max(x, 0) (NaN passed through, -0
 * giving +0), the activation of the ainews.cool article's two-layer MLP. */
typedef enum { FMLP_GELU_TANH = 0, FMLP_GELU_ERF = 1, FMLP_RELU = 2 } fmlp_gelu_mode;

/* Which kernel sequence a call with these sizes runs (reported by the *_plan queries). */
typedef enum {
    FMLP_PLAN_NONE = 0,         /* T == 0: nothing launched */
    FMLP_PLAN_TC = 1,           /* tcgen05 GEMM kernel(s) (the few-token kernel for 2..128
                                   tokens, the batched ones above); GeGLU/MLP: 2 kernels, or
                                   1 two-stage launch (fmlp_test_two_stage), m/h in ws */
    FMLP_PLAN_FUSED_SMALL = 2,  /* GeGLU: whole block in 1 kernel, m kept on chip */
    FMLP_PLAN_GEMV = 3,         /* one token (two when the call's weights are <= 16 MiB):
                                   weight-streaming GEMV kernel(s) */
    FMLP_PLAN_DECODE = 4        /* GeGLU/MLP, 1..4 tokens: both layers in one weight-streaming
                                   kernel (one CTA per SM, a grid barrier between the layers),
                                   h/m in ws; taken only after fmlp_test_prefer_decode(1) */
} fmlp_plan;

/* y[T, out] = bf16(x[T, in] @ W[out, in]^T + b[out]).
 * b may be NULL (no bias). One kernel. Section "Why are there no separate mul and add
 * kernels?": the bias add is the GEMM's epilogue, done before the write to HBM. */
FMLP_API fmlp_status fmlp_linear_bias(const void* x, const void* W, const void* b, void* y,
                             int64_t T, int64_t in, int64_t out, fmlp_stream_t s);

/* fmlp_linear_bias on row-strided views: row t of x starts at x + t * ldx and row t of y at
 * y + t * ldy (in elements), as with a slice x[:, a:a+in] of a wider tensor (section "What's
 * the transpose doing?": strides describe a view without moving data). ldx >= in and ldy >= out
 * (else FMLP_ERR_SHAPE), both multiples of 8 (the 16-byte TMA row rule; else FMLP_ERR_ALIGN);
 * 0 means packed rows. y must not share an element with x, W or b; two views of one buffer
 * with the same stride are compared element-exactly (column blocks that interleave row by
 * row do not overlap), other pairs by the bytes they span. W and b stay packed. Same kernels
 * and plans as fmlp_linear_bias. */
FMLP_API fmlp_status fmlp_linear_bias_strided(const void* x, int64_t ldx, const void* W,
                                              const void* b, void* y, int64_t ldy, int64_t T,
                                              int64_t in, int64_t out, fmlp_stream_t s);

/* y[T, out] = bf16(x[T, in] @ Wt[in, out] + b[out]): the Linear with the weight given
 * transposed, [in, out] row-major (out contiguous; W.t() of an nn.Linear weight made
 * contiguous, the `nn` layout of "Profiling in PyTorch (Part 2)", section "Where did the
 * transpose go? Kernel layouts and pre-ops"). No transposed copy is made: the tcgen05 GEMM
 * reads Wt tiles as an MN-major operand. b may be NULL. in and out multiples of 8 (else
 * FMLP_ERR_SHAPE), pointers 16-byte aligned, y overlapping no input; one single-SM tcgen05
 * kernel for every T (no GEMV or few-token variant for this layout). */
FMLP_API fmlp_status fmlp_linear_bias_wt(const void* x, const void* Wt, const void* b, void* y,
                                         int64_t T, int64_t in, int64_t out, fmlp_stream_t s);

/* h[T, out] = bf16(act(x[T, in] @ W[out, in]^T + b[out])), act = GELU or ReLU per `mode`, b
 * nullable. The first half of fmlp_mlp_gelu as its own call (bias+activation epilogue). */
FMLP_API fmlp_status fmlp_linear_bias_gelu(const void* x, const void* W, const void* b, void* h,
                                  int64_t T, int64_t in, int64_t out, fmlp_gelu_mode mode,
                                  fmlp_stream_t s);

/* m[T, H] = bf16(gelu_tanh(x[T, D] Wg[H, D]^T) * (x Wu[H, D]^T)).
 * The gate and up GEMMs of one token block run together in one kernel and share the x tile;
 * gelu(g)*u is the epilogue, so m is written to HBM exactly once. */
FMLP_API fmlp_status fmlp_geglu_gate_up(const void* x, const void* Wg, const void* Wu, void* m,
                               int64_t T, int64_t D, int64_t H, fmlp_stream_t s);

/* y[T, D] = bf16(m Wd[D, H]^T) with m = bf16(gelu_tanh(x Wg^T) * (x Wu^T)); bias-free, as in
 * the page's SimpleGeGLUMLP. ws: device workspace of at least
 * fmlp_geglu_workspace_size(T, D, H) bytes, 256-byte aligned, that holds m between the
 * stages (every plan but FMLP_PLAN_FUSED_SMALL); NULL with ws_bytes == 0 lets the library
 * take it from the stream-ordered allocator (cudaMallocAsync/cudaFreeAsync on `s`).
 *
 * Decode plan (1..4 tokens, FMLP_PLAN_DECODE; also fmlp_mlp_gelu; only while
 * fmlp_test_prefer_decode(1) is in effect, since the two-launch plans measure faster on
 * GB300): one kernel whose thread blocks, one per SM and all resident at once, meet at a
 * grid barrier between the layers.
 * The barrier is a counter in the library's device memory that belongs to the calling
 * stream (the first 1024 streams that call it on a device get one each; later streams take
 * the two-kernel plans). Calls on one stream are ordered and share the counter safely; calls
 * on different streams use different counters. Work captured into a CUDA graph keeps the
 * counter of the stream it was captured on, so two graphs captured on one stream must not run
 * at the same time as each other or as calls on that stream. The barrier wait is bounded
 * like every device wait: if other work keeps some of the kernel's thread blocks from
 * becoming resident for about a second, the call reports FMLP_ERR_DEVICE_TIMEOUT through
 * fmlp_device_status() and its output is undefined. */
FMLP_API fmlp_status fmlp_geglu(const void* x, const void* Wg, const void* Wu, const void* Wd, void* y,
                       int64_t T, int64_t D, int64_t H, void* ws, size_t ws_bytes,
                       fmlp_stream_t s);

/* y[T, Dout] = bf16(h W2[Dout, H]^T + b2) with h = bf16(act(x[T, D] W1[H, D]^T + b1)), act =
 * GELU (tanh or erf) or ReLU per `mode`.
 * b1, b2 nullable. ws as for fmlp_geglu, sized by fmlp_mlp_gelu_workspace_size(). */
FMLP_API fmlp_status fmlp_mlp_gelu(const void* x, const void* W1, const void* b1, const void* W2,
                          const void* b2, void* y, int64_t T, int64_t D, int64_t H,
                          int64_t Dout, fmlp_gelu_mode mode, void* ws, size_t ws_bytes,
                          fmlp_stream_t s);

/* fmlp_geglu and fmlp_mlp_gelu on row-strided views of x and y: row t of x starts at
 * x + t * ldx and row t of y at y + t * ldy (in elements), as with slices of wider tensors
 * (section "What's the transpose doing?": strides describe a view without moving data). The
 * same rules as fmlp_linear_bias_strided: ldx >= D and ldy >= D (Dout for the MLP), else
 * FMLP_ERR_SHAPE; multiples of 8, else FMLP_ERR_ALIGN; 0 means packed rows; y must not share
 * an element with any input or the workspace. Weights, biases and the workspace stay packed.
 * Same plans and kernels as the packed calls. */
FMLP_API fmlp_status fmlp_geglu_strided(const void* x, int64_t ldx, const void* Wg,
                                        const void* Wu, const void* Wd, void* y, int64_t ldy,
                                        int64_t T, int64_t D, int64_t H, void* ws,
                                        size_t ws_bytes, fmlp_stream_t s);
FMLP_API fmlp_status fmlp_mlp_gelu_strided(const void* x, int64_t ldx, const void* W1,
                                           const void* b1, const void* W2, const void* b2,
                                           void* y, int64_t ldy, int64_t T, int64_t D, int64_t H,
                                           int64_t Dout, fmlp_gelu_mode mode, void* ws,
                                           size_t ws_bytes, fmlp_stream_t s);

/* Mixture-of-experts feed-forward: E experts, each a GeGLU block (the ainews.cool article's MoE
 * note: every expert is an MLP, and fusing them cuts per-expert overhead). The tokens are
 * already grouped by expert: rows [offsets[e], offsets[e+1]) of x [T, D] go through expert e,
 *   m = bf16(gelu_tanh(x Wg[e]^T) * (x Wu[e]^T)),  y = bf16(m Wd[e]^T),
 * with Wg, Wu [E, H, D] and Wd [E, D, H] packed. offsets: E + 1 int32 in device memory
 * (4-byte aligned), rising from 0 to T; the kernels read them after waiting for the previous
 * kernel on `s`, so a routing kernel may write them just before, and the host never reads
 * them. Offsets outside [0, T] are clamped and a falling one empties that expert's group
 * (rows no group covers are left as they were); nothing faults. 1 <= E <= 256. ws: T*H*2
 * bytes (m), or NULL to take it from the stream-ordered allocator. Two kernels, each one
 * launch over all experts. No routing, gather or scatter is done here. */
FMLP_API fmlp_status fmlp_moe_geglu(const void* x, const int32_t* offsets, int64_t E,
                                    const void* Wg, const void* Wu, const void* Wd, void* y,
                                    int64_t T, int64_t D, int64_t H, void* ws, size_t ws_bytes,
                                    fmlp_stream_t s);
FMLP_API size_t fmlp_moe_geglu_workspace_size(int64_t T, int64_t D, int64_t H);

/* fmlp_geglu for callers that cannot allocate device memory (no counterpart in the pages).
 *
 * Who needs it: code that may not call cudaMalloc or any allocating routine - a plugin in a
 * serving process whose memory pool owns the device and forbids allocations after start-up,
 * or a real-time loop that must not risk an allocation stall or failure. fmlp_geglu keeps
 * the intermediate m in a caller workspace (or allocates one); this call keeps it in a fixed
 * 64 MiB array of device memory that belongs to the library, and allocates nothing: it
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Same arguments, layouts and results as fmlp_geglu without ws/ws_bytes. The shape checks
 * come first (FMLP_ERR_SHAPE as for fmlp_geglu). Limit: fmlp_geglu_workspace_size(T, D, H)
 * <= 64 MiB (e.g. T*H <= 32M); larger sizes return FMLP_ERR_WORKSPACE without launching
 * anything. Every GPU that loads the library holds the
 * 64 MiB array until the process exits. All calls share the array (it keeps the last call's
 * m; every call overwrites all of m it reads, so nothing needs clearing): calls whose kernels
 * can overlap on the GPU - on different streams, or from different threads without ordering -
 * race on it and must be serialised by the caller. The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture on the device. */
FMLP_API fmlp_status fmlp_geglu_noalloc(const void* x, const void* Wg, const void* Wu,
                                        const void* Wd, void* y, int64_t T, int64_t D, int64_t H,
                                        fmlp_stream_t s);

/* Inner dimensions that are not multiples of 8 (packed rows). The TMA loads and stores move
 * rows whose byte stride is a multiple of 16, so such a call copies its operands, zero-padded
 * to the next multiple of 8 in every inner dimension, into one scratch taken from the
 * stream-ordered allocator (cudaMallocAsync/cudaFreeAsync on the call's stream), runs the plan
 * of the padded shape, and copies the output's columns back: exact (zero columns add nothing,
 * padded outputs are dropped, a zero gate/up or first-layer row gives gelu(0) or act(0) = 0),
 * at the cost of one extra read and write of every operand. The caller's workspace is not
 * used (the workspace queries return 0 for such sizes); the plan queries report the padded
 * shape's plan. "Profiling in PyTorch (Part 2)", section "What's the transpose doing?": the
 * copy changes only the strides the kernels see. */

/* Workspace bytes the calls above need (T*H*2 for the 2-kernel plans, else 0; 0 for inner
 * dimensions that are not multiples of 8). Pure host functions; they touch no device. */
FMLP_API size_t fmlp_geglu_workspace_size(int64_t T, int64_t D, int64_t H);
FMLP_API size_t fmlp_mlp_gelu_workspace_size(int64_t T, int64_t D, int64_t H, int64_t Dout);

/* The plan a call with these sizes takes (an fmlp_plan value). Pure host functions. */
FMLP_API int fmlp_geglu_plan(int64_t T, int64_t D, int64_t H);
FMLP_API int fmlp_mlp_gelu_plan(int64_t T, int64_t D, int64_t H, int64_t Dout);
FMLP_API int fmlp_linear_plan(int64_t T, int64_t in, int64_t out);

/* Tile-kernel policy for the tensor-core plans, process-wide (default FMLP_TILES_AUTO):
 * AUTO picks per call from the shape; SINGLE forces one-SM 128-row tiles; PAIR forces two-SM
 * (CTA pair, 256-row) tiles wherever the shape has more than 128 rows. Results are identical
 * up to fp32 summation order. Returns FMLP_ERR_SHAPE for an unknown value. */
typedef enum { FMLP_TILES_AUTO = 0, FMLP_TILES_SINGLE = 1, FMLP_TILES_PAIR = 2 } fmlp_tile_policy;
FMLP_API fmlp_status fmlp_set_tile_policy(int policy);

/* Writes a one-line description of the kernels a call with these sizes would launch on the
 * current device (tile kernel, tile shape, grid) into buf (NUL-terminated, truncated to
 * buflen). op: 0 fmlp_linear_bias (in = D, out = H), 1 fmlp_linear_bias_gelu (same),
 * 2 fmlp_geglu_gate_up, 3 fmlp_geglu, 4 fmlp_mlp_gelu. Launches nothing. */
FMLP_API fmlp_status fmlp_describe_plan(int op, int64_t T, int64_t D, int64_t H, int64_t Dout,
                                        char* buf, size_t buflen);

/* Device activation check: out[i] = act(in[i]) (GELU or ReLU per mode) in fp32 with the exact
 * device code the epilogues use. in/out: n floats in device memory. One kernel. */
FMLP_API fmlp_status fmlp_gelu_eval(const float* in, float* out, int64_t n, fmlp_gelu_mode mode,
                           fmlp_stream_t s);

/* Synchronises `s`, then returns and clears the current device's status word:
 * FMLP_OK, or FMLP_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded wait since the last
 * call (which wait is named in fmlp_last_error()). */
FMLP_API fmlp_status fmlp_device_status(fmlp_stream_t s);

/* Failure-injection test hooks, process-wide, all off by default. Neither faults nor hangs a
 * GPU: the failures are made on the host, or by a bounded device wait that runs out.
 *   FMLP_INJECT_NONE       clear every injection (count and timeout_us ignored).
 *   FMLP_INJECT_LAUNCH     the next `count` kernel launches of the library fail on the host as
 *                          a refused launch would: nothing is launched, the call returns
 *                          FMLP_ERR_CUDA and fmlp_last_error() says "injected". A block call
 *                          whose second kernel is refused has launched its first.
 *   FMLP_INJECT_SKIP_LOAD  the next `count` launches of the CTA-pair tcgen05 GEMM (the batched
 *                          tile kernel) expect the bytes of their first K step but issue no
 *                          load for it, with every device wait of those launches bounded by
 *                          timeout_us (0: about one second): the MMA's wait on that stage runs
 *                          out, the producer's and the epilogue's waits follow, the kernel
 *                          records FMLP_ERR_DEVICE_TIMEOUT (read by fmlp_device_status()) and
 *                          returns with its output undefined.
 * count in [0, 1000000], timeout_us in [0, 2000000], kind known; else FMLP_ERR_SHAPE. */
typedef enum {
    FMLP_INJECT_NONE = 0,
    FMLP_INJECT_LAUNCH = 1,
    FMLP_INJECT_SKIP_LOAD = 2
} fmlp_inject_kind;
FMLP_API fmlp_status fmlp_test_inject(int kind, int64_t count, int64_t timeout_us);

/* Test hook for the launches with a grid barrier, process-wide: later one-kernel decode
 * launches (FMLP_PLAN_DECODE) and few-token block launches (fmlp_test_fewtoken_block) add
 * extra_ctas CTAs (the latter: rounded up to whole clusters, their tiles past the last weight
 * row) beyond the ones that can be resident at once, so the resident
 * CTAs wait at the grid barrier for CTAs that cannot start until they leave, and every device
 * wait of those launches is bounded by timeout_us (0: the default of about one second). The
 * waits run out, the kernel records FMLP_ERR_DEVICE_TIMEOUT and returns; the output is then
 * undefined; nothing faults or hangs. (0, 0) restores normal launches. extra_ctas in
 * [0, 4096], timeout_us in [0, 2000000], else FMLP_ERR_SHAPE. */
FMLP_API fmlp_status fmlp_test_decode_overload(int64_t extra_ctas, int64_t timeout_us);

/* Plan switch for the one-kernel decode, process-wide: with on = 1, GeGLU and MLP blocks of
 * 1..4 tokens whose shapes the decode kernel accepts run as FMLP_PLAN_DECODE (plan queries
 * report it; the workspace size is the same T * H * 2 bytes); with on = 0 (the default) they
 * take the GEMV or the few-token tcgen05 kernels, which measure faster on GB300 (the 4096-wide
 * MLP at one token: 19.1 us against 25.4 us). Switch it only while no other thread queries
 * plans or launches. on not 0 or 1: FMLP_ERR_SHAPE. */
FMLP_API fmlp_status fmlp_test_prefer_decode(int on);

/* Plan switch for the two-stage block launch, process-wide. Under FMLP_PLAN_TC a GeGLU or MLP
 * block of more than 128 tokens whose weights (both layers) take at most 64 MiB, with at most
 * 64 bands of 256 tokens and 2048 tiles in all, can run as ONE persistent CTA-pair launch:
 * the first layer's 256-row tiles and the down tiles share one list per pair, a down tile
 * waiting (bounded) until every first-layer tile of its 256 rows has been stored. mode 0 (the
 * default) takes it when both layers would run on the CTA-pair kernel anyway; mode 1 takes it
 * for every block it accepts (also the FMLP_TILES_PAIR policy's); mode -1 never (two
 * launches). The results are bit-identical either way: the same tiles, the same K order, the
 * same roundings. The launch keeps one row of counters per stream, like FMLP_PLAN_DECODE, and
 * expects every one of its CTA pairs to be resident at once (a concurrent kernel on another
 * stream that holds SMs until this launch ends makes its waits run out with
 * FMLP_ERR_DEVICE_TIMEOUT). Under FMLP_INJECT_SKIP_LOAD, a two-stage launch takes the
 * injection instead as a band count that is never reached, so its down tiles' waits run out.
 * Switch it only while no other thread queries plans or launches. mode not in {-1, 0, 1}:
 * FMLP_ERR_SHAPE. */
FMLP_API fmlp_status fmlp_test_two_stage(int mode);

/* The item lists of a two-stage launch (host only, no device needed), for checking the
 * schedule: num_m bands of 256 rows, num_n1 first-stage and num_n2 down N tiles, kb1 and kb2
 * K steps of 64 per tile, `pairs` CTA pairs. First-stage items are u = band * num_n1 + j; down
 * items follow, n1 + band * num_n2 + n. Writes start[0 .. pairs] (pair p runs
 * item[start[p] .. start[p + 1])) and the items (at most 2048), and their count to *n_items.
 * Shape out of range: FMLP_ERR_SHAPE; a NULL pointer: FMLP_ERR_NULL. */
FMLP_API fmlp_status fmlp_test_two_stage_schedule(int num_m, int num_n1, int num_n2, int kb1,
                                                  int kb2, int pairs, uint16_t* start,
                                                  uint16_t* item, int64_t* n_items);

/* Plan switch for the few-token block launch, process-wide. Under FMLP_PLAN_TC a GeGLU block
 * of 2..64 tokens, or an MLP block of 2..128, can run both layers in ONE launch of the
 * few-token kernel's design (weights as the MMA's M side, K split over a cluster): layer 1 to
 * h in the workspace, layer 2's first weight tiles prefetched into shared memory meanwhile, a
 * bounded grid barrier (a counter of the stream's decode-plan row) before h is read, layer 2
 * to y. It needs every CTA resident at once (a concurrent kernel on another stream that holds
 * SMs until this launch ends makes its barrier run out with FMLP_ERR_DEVICE_TIMEOUT). mode 0
 * (the default) takes it for blocks of at most 64 tokens whose second layer's weight tiles
 * are at least half as tall as the first's (e.g. the 4096-wide MLP; measured faster there,
 * slower otherwise); 1 takes it for every block it accepts; -1 never (two few-token launches). Results agree with the two launches within rounding (the same tiles,
 * K slices and slice order). Switch it only while no other thread queries plans or launches.
 * mode not in {-1, 0, 1}: FMLP_ERR_SHAPE. */
FMLP_API fmlp_status fmlp_test_fewtoken_block(int mode);

/* Test hook for the bounded-wait machinery: launches one CTA whose thread waits on an
 * mbarrier that nothing completes, with a limit of timeout_us microseconds (1..2,000,000).
 * The kernel then records FMLP_ERR_DEVICE_TIMEOUT and exits; nothing faults or hangs. */
FMLP_API fmlp_status fmlp_test_wait_timeout(int64_t timeout_us, fmlp_stream_t s);

/* Static text for a status code. */
FMLP_API const char* fmlp_status_string(fmlp_status st);

/* Detail of the last failure on the calling thread ("" if none). */
FMLP_API const char* fmlp_last_error(void);

/* Library ABI version (major*10000 + minor*100 + patch). */
FMLP_API int fmlp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FMLP_H_ */
