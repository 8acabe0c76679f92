/*
 * fp8w8a8.h — C ABI of the FP8 (e4m3fn) W8A8 linear layer with dynamic
 * per-tensor activation quantization, for NVIDIA sm_103a (GB300).
 *
 * The layer (source pages: "Prototype FP8Linear W8A8 runtime quantization",
 * "[WIP] FP8 support", "[Kernel] Implement fallback for FP8 channelwise using
 * torch._scaled_mm", "Fp8 Quantization Support"):
 *
 *   s_w      = amax(W) / 448              (per tensor, or per output row n)
 *   qW       = e4m3(W / s_w)              once, when weights are loaded
 *   s_a      = amax(A) / 448              every call, on the device
 *   qA       = e4m3(A / s_a)
 *   Y[m, n]  = bf16( s_a * s_w[n] * sum_k qA[m, k] qW[n, k]  (+ bias[n]) )
 *
 * e4m3(x): IEEE fp32 quotient, then round-to-nearest-even to float8_e4m3fn,
 * saturating to +-448; the sign of zero is kept. A zero amax gives scale 1.
 * The product accumulates in fp32 on tensor cores.
 *
 * Conventions for every call:
 *  - Matrices are row-major. A bf16 [M, K] with row stride lda >= K elements;
 *    W bf16 [N, K] (out_features x in_features, as in nn.Linear) with stride
 *    ldw >= K; Y bf16 [M, N] with stride ldy >= N. bf16 strides may be any
 *    value: no padding of the logical dimensions is required ("[WIP] FP8
 *    support": dimensions that are not multiples of 16 must work).
 *  - The library's own FP8 matrices (qA, qW) are u8 [rows, ld] with ld a
 *    multiple of 16 and ld >= K (fp8_min_ld(K) is the smallest). The
 *    quantizers write bytes [K, ld) of every row as zero; consumers rely on
 *    that. The base address of an FP8 matrix must be 16-byte aligned.
 *  - Scales (s_a, s_w) are fp32 in DEVICE memory, so dynamic quantization
 *    never needs a host round trip.
 *  - Every pointer is a device pointer owned by the caller. The library
 *    allocates nothing, never synchronizes (except fp8_last_device_status),
 *    and enqueues all work on `stream` (NULL = the legacy default stream).
 *  - Argument errors are returned synchronously before anything is enqueued.
 *    FP8_ERR_CUDA reports a failed launch. Kernel-side errors (a bounded wait
 *    that expired) are reported later by fp8_last_device_status().
 *  - M == 0 or N == 0 is a no-op returning FP8_OK. K == 0 gives Y = bias (or 0).
 *  - A workspace may be used by one call at a time; calls are otherwise
 *    reentrant and thread-safe.
 *  - Launch ordering: kernels use programmatic dependent launch. The weight
 *    operands (qW, s_w, bias) of a linear call may be read before the kernel
 *    enqueued just before it has finished, so they must not be written by the
 *    immediately preceding kernel unless that kernel is fp8_quantize_weight or
 *    a kernel that does not trigger programmatic launch early (any ordinary
 *    CUDA or PyTorch kernel). Activations, workspace and Y are always ordered.
 */
#ifndef FP8W8A8_H
#define FP8W8A8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* fp8_stream_t;

typedef enum fp8_status {
  FP8_OK = 0,
  FP8_ERR_INVALID_ARG = 1,        /* null pointer, negative size, ld too small, bad flag */
  FP8_ERR_MISALIGNED = 2,         /* FP8 ld not a multiple of 16, or a base address not aligned */
  FP8_ERR_WORKSPACE = 3,          /* workspace too small or not 256-byte aligned */
  FP8_ERR_CUDA = 4,               /* a CUDA runtime/driver call or kernel launch failed */
  FP8_ERR_TIMEOUT = 5,            /* a device-side bounded wait expired (see fp8_last_device_status) */
  FP8_ERR_UNSUPPORTED_DEVICE = 6  /* current device is not sm_103 */
} fp8_status;

/* FP8 storage formats. float8_e4m3fn is the pages' format ("Fp8 Quantization
 * Support": fp8 is assumed to be torch.float8_e4m3fn); float8_e5m2 is the one that
 * page names as the later extension. Every call without an _ex suffix uses e4m3. */
typedef enum fp8_format {
  FP8_E4M3 = 0, /* 1 sign, 4 exponent (bias 7), 3 mantissa bits; max 448; no infinity */
  FP8_E5M2 = 1  /* 1 sign, 5 exponent (bias 15), 2 mantissa bits; max 57344 */
} fp8_format;

#define FP8_E4M3_MAX 448.0f
#define FP8_E5M2_MAX 57344.0f
#define FP8_LD_ALIGN 16
/* Workspace needed by fp8_quantize_weight / fp8_quantize_act (partial amax values). */
#define FP8_QUANT_WORKSPACE_BYTES 4352

/* Smallest valid leading dimension (bytes) of an FP8 matrix with K columns: K rounded up to 16 (16 for K == 0). */
int64_t fp8_min_ld(int64_t K);

/* Bytes of workspace fp8_linear / fp8_linear_channelwise use for this shape.
 * 0 for decode shapes of up to 16 tokens (fp8_uses_gemv): the GEMV quantizes A
 * itself. Every other shape (the GEMV at 17..32 tokens, the GEMM) needs at
 * least FP8_QUANT_WORKSPACE_BYTES (partial amax values, s_a) plus the
 * quantized activations qA [M, fp8_min_ld(K)]. GEMM shapes with too few
 * output tiles to fill the GPU (small M) split K across CTAs when the
 * workspace also holds, from the next 256-byte boundary, fp32 partials
 * [splits, M, N rounded up to 4]; the value returned includes that space for
 * the split a GB300 (152 SMs) takes. A workspace between the two sizes works
 * too, with a smaller split or none. 0 when M or K is 0. Host-only, never
 * touches the device. */
size_t fp8_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* 1 when fp8_linear takes the decode GEMV path for this shape, 0 for the GEMM path:
 * M <= the crossover (32 by default, see fp8_set_gemv_max_m) and K <= 32768. Host-only. */
int fp8_uses_gemv(int64_t M, int64_t K, int64_t N);

/* Sets the decode crossover: calls with M <= m (and K <= 32768) run the GEMV,
 * larger M the GEMM. m is clamped to [0, 32] (32 is the GEMV's largest M; 0
 * sends every shape to the GEMM); m < 0 only queries. Returns the previous
 * value. The start-up value is 32, or FP8W8A8_GEMV_MAX_M from the environment.
 * Process-wide; it changes which kernels later calls enqueue (and so
 * fp8_workspace_bytes), never their results beyond the stated tolerance.
 * ("[WIP] FP8 support": decode runs at sequence length < 16 and wants its own
 * GEMV; where exactly to switch is a tuning choice.) Host-only. */
int fp8_set_gemv_max_m(int m);

/*
 * Quantize bf16 weights W [N, K] (stride ldw) to qW u8 [N, ldq] and scales s_w.
 * per_channel == 0: one scale, s_w[0] = amax(W)/448 ("Fp8 Quantization
 * Support", recipe strategy "tensor"). per_channel == 1: s_w[n] = amax(W[n,:])/448
 * for each output channel ("[Kernel] Implement fallback for FP8 channelwise
 * using torch._scaled_mm"). Bytes [K, ldq) of each row are written as zero.
 * ws: device workspace of >= FP8_QUANT_WORKSPACE_BYTES bytes, 256-byte aligned
 * (unused when per_channel == 1; may then be NULL).
 */
fp8_status fp8_quantize_weight(const void* w_bf16, int64_t N, int64_t K, int64_t ldw,
                               int per_channel, uint8_t* qw, int64_t ldq, float* s_w,
                               void* ws, size_t ws_bytes, fp8_stream_t stream);

/*
 * Dynamic per-tensor activation quantization ("Prototype FP8Linear W8A8
 * runtime quantization": activations are quantized at run time):
 * s_a[0] = amax(A)/448, qA = e4m3(A / s_a) as u8 [M, ldq], tail bytes zero.
 * ws: >= FP8_QUANT_WORKSPACE_BYTES bytes, 256-byte aligned.
 */
fp8_status fp8_quantize_act(const void* a_bf16, int64_t M, int64_t K, int64_t lda,
                            uint8_t* qa, int64_t ldq, float* s_a,
                            void* ws, size_t ws_bytes, fp8_stream_t stream);

/*
 * Scaled FP8 GEMM on already-quantized operands — the step the pages run with
 * torch._scaled_mm ("Prototype FP8Linear W8A8 runtime quantization";
 * "[Kernel] Implement fallback for FP8 channelwise using torch._scaled_mm"):
 *   Y[m, n] = bf16( s_a[0] * s_w[n or 0] * sum_k qA[m,k] qW[n,k] (+ bias[n]) ).
 * qa u8 [M, ldqa], qw u8 [N, ldqw] (both ld multiples of 16, tails zero);
 * s_a device fp32 [1]; s_w device fp32 [1] (per_channel == 0) or [N]
 * (per_channel == 1); bias bf16 [N] or NULL; y bf16 [M, ldy].
 * Uses no workspace.
 */
fp8_status fp8_scaled_mm(const uint8_t* qa, int64_t M, int64_t K, int64_t ldqa, const float* s_a,
                         const uint8_t* qw, int64_t N, int64_t ldqw, const float* s_w,
                         int per_channel, const void* bias_bf16, void* y_bf16, int64_t ldy,
                         fp8_stream_t stream);

/*
 * The W8A8 linear with dynamic per-tensor activation quantization and a
 * per-tensor weight scale s_w[0]: amax(A) -> s_a -> e4m3(A/s_a) -> FP8 GEMM
 * (fp32 accumulate) -> s_a*s_w (+bias) epilogue -> bf16 Y.
 * Decode shapes (fp8_uses_gemv) run one persistent split-K GEMV kernel that
 * quantizes A itself and streams qW once ("[WIP] FP8 support": LLM decode runs
 * at sequence length < 16 and wants a custom gemv); larger M runs amax + cast
 * + the tcgen05 GEMM. No padding or repacking of A, W or Y happens on any path.
 * ws: >= fp8_workspace_bytes(M, K, N) bytes, 256-byte aligned (may be NULL
 * when that is 0).
 */
fp8_status fp8_linear(const void* a_bf16, int64_t M, int64_t K, int64_t lda,
                      const uint8_t* qw, int64_t N, int64_t ldqw, const float* s_w,
                      const void* bias_bf16, void* y_bf16, int64_t ldy,
                      void* ws, size_t ws_bytes, fp8_stream_t stream);

/*
 * Same as fp8_linear with one weight scale per output channel, s_w[N]; the
 * channel scale is applied to column n after the product, using
 * (s_a A)(s_w,n W_n)^T = s_a s_w,n (A W_n^T) ("[Kernel] Implement fallback for
 * FP8 channelwise using torch._scaled_mm"), fused into the epilogue.
 */
fp8_status fp8_linear_channelwise(const void* a_bf16, int64_t M, int64_t K, int64_t lda,
                                  const uint8_t* qw, int64_t N, int64_t ldqw, const float* s_w,
                                  const void* bias_bf16, void* y_bf16, int64_t ldy,
                                  void* ws, size_t ws_bytes, fp8_stream_t stream);

/*
 * fp8_linear (per_channel == 0) or fp8_linear_channelwise (per_channel == 1)
 * without a workspace argument, for callers that cannot allocate device memory:
 * for example code that runs inside a host application which owns the whole
 * device-memory budget and hands a kernel only its input and output buffers,
 * or a latency-critical path that must not call cudaMalloc, which can block
 * until other work on the device has finished. The source pages have no
 * counterpart of this call; it exists only for such callers.
 *
 * The scratch lives in one fixed array inside the library of
 * FP8_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the library holds
 * until the process exits. A call needs the least workspace fp8_linear
 * accepts: nothing for decode shapes, and for GEMM shapes M * fp8_min_ld(K)
 * may be at most FP8_NOALLOC_SCRATCH_BYTES - 4352. Larger shapes are refused
 * with FP8_ERR_WORKSPACE before anything is enqueued. The rest of the array
 * serves a K split where one fits (the same launches fp8_linear makes with a
 * workspace of FP8_NOALLOC_SCRATCH_BYTES). The call allocates nothing.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. After a device reset (cudaDeviceReset) the
 * address is looked up again on the next call, which then also belongs
 * outside any capture. All calls share the one array and it keeps the
 * previous call's contents: nothing in it has to start at zero (each call
 * writes every scratch byte it reads before reading it), but two calls whose
 * kernels overlap on the GPU — on different streams or from different host
 * threads — race on it and give wrong results. Order such calls on one stream.
 * Arguments and every other rule are those of fp8_linear.
 */
#define FP8_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
fp8_status fp8_linear_noalloc(const void* a_bf16, int64_t M, int64_t K, int64_t lda,
                              const uint8_t* qw, int64_t N, int64_t ldqw, const float* s_w,
                              int per_channel, const void* bias_bf16, void* y_bf16, int64_t ldy,
                              fp8_stream_t stream);

/*
 * ---------------------------------------------------------------------------
 * Wider calls: the format of each FP8 operand, and a static activation scale.
 * In all of them, for format F: max(F) = 448 (FP8_E4M3) or 57344 (FP8_E5M2),
 * dynamic scale = amax / max(F), q = F(x / scale) with the rounding and
 * saturation rules above (saturation to +-max(F), never infinity).
 * Invalid format values return FP8_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------------
 */

/* fp8_quantize_weight with the weight format `fmt`. */
fp8_status fp8_quantize_weight_ex(const void* w_bf16, int64_t N, int64_t K, int64_t ldw,
                                  int per_channel, fp8_format fmt, uint8_t* qw, int64_t ldq,
                                  float* s_w, void* ws, size_t ws_bytes, fp8_stream_t stream);

/*
 * fp8_quantize_act with the activation format `fmt` and an optional static
 * scale. s_static == NULL: dynamic, s_a[0] = amax(A) / max(fmt); ws as for
 * fp8_quantize_act. s_static != NULL (device fp32 [1], 4-byte aligned): the
 * calibrated scale is used as given ("Fp8 Quantization Support": the recipe
 * quantizes input activations per tensor with scales from the calibration
 * run), no amax pass runs, s_a[0] receives a copy of it and ws may be NULL.
 * Elements beyond s * max(fmt) saturate. The scale must be positive and finite.
 */
fp8_status fp8_quantize_act_ex(const void* a_bf16, int64_t M, int64_t K, int64_t lda,
                               fp8_format fmt, const float* s_static, uint8_t* qa, int64_t ldq,
                               float* s_a, void* ws, size_t ws_bytes, fp8_stream_t stream);

/* fp8_scaled_mm with the formats of qA (fmt_a) and qW (fmt_w); any pairing. */
fp8_status fp8_scaled_mm_ex(const uint8_t* qa, fp8_format fmt_a, int64_t M, int64_t K, int64_t ldqa,
                            const float* s_a, const uint8_t* qw, fp8_format fmt_w, int64_t N,
                            int64_t ldqw, const float* s_w, int per_channel, const void* bias_bf16,
                            void* y_bf16, int64_t ldy, fp8_stream_t stream);

/*
 * The W8A8 linear with a static (calibrated) per-tensor activation scale s_a
 * (device fp32 [1]) instead of the dynamic one: qA = e4m3(A / s_a), then the
 * same product and epilogue as fp8_linear (per_channel == 0) or
 * fp8_linear_channelwise (per_channel == 1). No amax is computed. Workspace as
 * for fp8_linear (fp8_workspace_bytes).
 */
fp8_status fp8_linear_static(const void* a_bf16, int64_t M, int64_t K, int64_t lda,
                             const float* s_a, const uint8_t* qw, int64_t N, int64_t ldqw,
                             const float* s_w, int per_channel, const void* bias_bf16,
                             void* y_bf16, int64_t ldy, void* ws, size_t ws_bytes,
                             fp8_stream_t stream);

/*
 * The general linear: activation format fmt_a, weight format fmt_w (qW as
 * written by fp8_quantize_weight_ex with that format), dynamic activation
 * scale when s_static is NULL, else the static one; per_channel selects the
 * weight-scale mode. Workspace as for fp8_linear.
 */
fp8_status fp8_linear_ex(const void* a_bf16, int64_t M, int64_t K, int64_t lda, fp8_format fmt_a,
                         const float* s_static, const uint8_t* qw, fp8_format fmt_w, int64_t N,
                         int64_t ldqw, const float* s_w, int per_channel, const void* bias_bf16,
                         void* y_bf16, int64_t ldy, void* ws, size_t ws_bytes, fp8_stream_t stream);

/*
 * ---------------------------------------------------------------------------
 * Weight-only FP8: the FP8 weights are kept for memory and up-converted to the
 * original dtype for the product ("Prototype FP8Linear W8A8 runtime
 * quantization": the path below compute capability 9.0, where weights are
 * dequantized into higher precision with no compute savings). A stays bf16:
 *   Y[m, n] = bf16( s_w[n or 0] * sum_k A[m, k] * decode(qW[n, k]) (+ bias[n]) ).
 * Every e4m3 / e5m2 value is a bf16 value, so the up-conversion is exact; the
 * weight scale multiplies the fp32 accumulator in the epilogue, as in the
 * channelwise identity (s_w,n W_n) A = s_w,n (W_n A).
 * Decode shapes (M <= the crossover, K <= 32768) run the split-K GEMV, which up-converts
 * each weight tile in registers and needs no workspace; larger shapes
 * up-convert W into the workspace once per call and run a bf16 tcgen05 GEMM.
 * ---------------------------------------------------------------------------
 */

/* Workspace fp8_linear_weight_only needs: 0 for decode shapes; otherwise the
 * up-converted weights (N * round_up(K, 8) bf16, rounded up to 256 bytes) plus
 * M * round_up(K, 8) bf16 for an aligned copy of A, used only when A's row
 * stride or base address is not a multiple of 16 bytes. Host-only. */
size_t fp8_weight_only_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* qw, s_w from fp8_quantize_weight(_ex) with format fmt_w; per_channel as
 * there; other arguments and rules as for fp8_linear. */
fp8_status fp8_linear_weight_only(const void* a_bf16, int64_t M, int64_t K, int64_t lda,
                                  const uint8_t* qw, fp8_format fmt_w, int64_t N, int64_t ldqw,
                                  const float* s_w, int per_channel, const void* bias_bf16,
                                  void* y_bf16, int64_t ldy, void* ws, size_t ws_bytes,
                                  fp8_stream_t stream);

/*
 * Diagnostics (no counterpart on the source pages): the launch the GEMM path of
 * fp8_linear (and fp8_scaled_mm, which never splits K) would use for FP8
 * operands qa [M, ldqa] and qw [N, ldqw] (ld in bytes), K columns, and a
 * linear workspace of ws_bytes, on the current device. *two_sm = 1 when CTA
 * pairs run the two-SM MMA (tcgen05 cta_group::2), which needs at least two
 * 128-row blocks and both operands in the current device's own memory
 * (cudaMalloc'd on it); any other memory (pinned or managed host memory,
 * another GPU's memory) takes one CTA per tile, *two_sm = 0. *grid = CTAs
 * launched; *group_n = column tiles per raster group; *splits = CTAs that
 * share each output tile's K (1: no split; more when there are too few tiles
 * to fill the GPU and ws_bytes holds the fp32 partials); *tail_split = column
 * units each tile of the last, partial wave is divided into (1: none; 2 or 4
 * when that many units per left-over tile still fit one wave, each computing
 * 256 / tail_split columns over all of K). Output pointers may be NULL.
 * Enqueues nothing; FP8_ERR_INVALID_ARG for non-positive sizes,
 * FP8_ERR_CUDA or FP8_ERR_UNSUPPORTED_DEVICE when the device cannot be queried.
 */
fp8_status fp8_gemm_config(const uint8_t* qa, int64_t M, int64_t ldqa, const uint8_t* qw, int64_t N,
                           int64_t ldqw, int64_t K, size_t ws_bytes, int* two_sm, int* grid, int* group_n,
                           int* splits, int* tail_split);

/* The same plan as fp8_gemm_config, computed on the host without a device for a GPU with
 * num_sms SMs and pair_slots co-resident CTA pairs (0: no pair mode), with both operands in
 * that GPU's own memory and gap-free (leading dimension fp8_min_ld(K)). Outputs as above
 * (NULL allowed). FP8_ERR_INVALID_ARG for non-positive sizes or num_sms, negative pair_slots.
 * Host-only, never touches the device. */
fp8_status fp8_gemm_plan_model(int64_t M, int64_t N, int64_t K, int num_sms, int pair_slots, size_t ws_bytes,
                               int* two_sm, int* grid, int* group_n, int* splits, int* tail_split);

/* The decode GEMV's launch configuration, computed on the host without a device ("[WIP] FP8
 * support": the decode GEMV). mode: 0 activations already quantized (fp8_scaled_mm, and
 * fp8_linear from 17 tokens on), 1 quantized inside the kernel (fp8_linear up to 16 tokens;
 * static_scale != 0 for fp8_linear_static), 2 bf16 activations (weight-only). smem_limit:
 * dynamic shared memory a CTA may use; clusters_of_size[s - 1]: co-resident clusters of s CTAs
 * at that shared memory, s = 1..8 (host memory, 8 ints). Outputs (NULL allowed): *cluster = CTAs
 * per cluster sharing K, *clusters = clusters launched, *stages = weight-ring depth, *kslice =
 * bytes of K per CTA, *scratch_a = how A reaches shared memory in mode 1 (0 per-thread loads,
 * 1 all of A bulk-copied, 2 the CTA's slice), *cluster_amax = 1 when the dynamic maximum is
 * exchanged over the cluster, *tcgen05 = 1 when the main loop runs on tcgen05. A's rows are
 * taken as 16-byte aligned. FP8_ERR_INVALID_ARG for M outside 1..32, K outside 1..32768, other
 * bad sizes or mode; FP8_ERR_CUDA when no configuration fits (the launch would fail the same
 * way). Host-only, never touches the device. */
fp8_status fp8_gemv_plan_model(int64_t M, int64_t N, int64_t K, int mode, int static_scale, int smem_limit,
                               const int* clusters_of_size, int* cluster, int* clusters, int* stages, int* kslice,
                               int* scratch_a, int* cluster_amax, int* tcgen05);

/*
 * Synchronizes `stream`, then reports and clears device-side errors recorded
 * by the library's kernels on the current device since the last query
 * (FP8_ERR_TIMEOUT when a bounded wait expired), or FP8_ERR_CUDA when the
 * stream itself reports an error. FP8_OK otherwise.
 */
fp8_status fp8_last_device_status(fp8_stream_t stream);

/*
 * Failure-path self-test: enqueues a small kernel whose bounded device wait is
 * made to run out (its producer withholds one item), using the same wait
 * primitive and error word as the library's GEMV. The wait gives up after
 * limit_ns (1e3 .. 1e10 nanoseconds, else FP8_ERR_INVALID_ARG), the kernel
 * returns normally and the context stays usable; the next
 * fp8_last_device_status reports FP8_ERR_TIMEOUT once. Nothing faults or hangs.
 * The pages have no counterpart; it exists so the error path can be tested.
 */
fp8_status fp8_selftest_timeout(int64_t limit_ns, fp8_stream_t stream);

/* Static, human-readable name of a status code. Never NULL. */
const char* fp8_status_string(fp8_status status);

#ifdef __cplusplus
}
#endif

#endif /* FP8W8A8_H */
