/*
 * swiglu.h -- C ABI of the GB300 (sm_103a) fused SwiGLU up-projection library.
 *
 * The operation ("Tile-Level Activation Overlap for Efficient LLM Inference",
 * technical summary, section "Enonce du probleme"; "1 . Anatomie d'un
 * transformeur sur GPU", section 1.1, "Wgate, Wup -> SwiGLU"):
 *
 *     h[i, j] = silu(g[i, j]) * u[i, j],   silu(z) = z / (1 + e^-z)
 *     g = x . W_gate,  u = x . W_up
 *
 *     x      [M, d]     row-major, contiguous (activations, one row per token)
 *     W_gate [d, d_ff]  row-major, contiguous (element (k, j) at k*d_ff + j, the
 *     W_up   [d, d_ff]  weight layout of "Ou part le temps d'un token", section
 *                       "Un kernel pour les matrices etroites")
 *     h      [M, d_ff]  row-major, contiguous
 *
 * Arithmetic: products and sums in f32 (bf16 operands are widened exactly);
 * g and u are never rounded to the operand type; only h is rounded, to
 * nearest even, to `dtype`.  Partial sums are combined in a fixed order, so a
 * given call on a given device returns the same bits every time (the
 * reproducibility argument of "Un kernel pour les matrices etroites").
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never frees or retains them past the call's stream work.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work; they return before it runs.  Faults inside enqueued work
 *     surface at the caller's next synchronisation, as for any CUDA library.
 *   - Argument validation is synchronous and enqueues nothing on failure.
 *   - The return value is a swiglu_status; swiglu_last_error_string() gives a
 *     human-readable detail for the calling thread's last failure.
 *   - h must not overlap x, W_gate, W_up or the workspace.
 *   - Requirements checked on every call: sizes M, d, d_ff >= 0 (M == 0 or
 *     d_ff == 0 is a no-op; d == 0 gives h = 0); pointers 16-byte aligned;
 *     d and d_ff multiples of 8 (bf16) or 4 (f32), so that every row starts on
 *     a 16-byte boundary for vector loads and TMA; the current device must be
 *     compute capability 10.3 (sm_103).
 */
#ifndef SWIGLU_GB300_H
#define SWIGLU_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SWIGLU_API __attribute__((visibility("default")))
#else
#define SWIGLU_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SWIGLU_F32 = 0, SWIGLU_BF16 = 1 } swiglu_dtype;

typedef enum {
  SWIGLU_OK = 0,
  SWIGLU_ERR_INVALID_ARG = 1,   /* null pointer, negative size, unknown dtype/path */
  SWIGLU_ERR_UNSUPPORTED = 2,   /* valid arguments the library does not serve  */
  SWIGLU_ERR_ALIGNMENT = 3,     /* pointer or row stride not 16-byte aligned    */
  SWIGLU_ERR_OOM = 4,           /* workspace allocation failed                  */
  SWIGLU_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed            */
  SWIGLU_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up           */
  SWIGLU_ERR_ARCH = 7,          /* current device is not sm_103                 */
  SWIGLU_ERR_WORKSPACE = 8      /* caller workspace too small or misaligned     */
} swiglu_status;

/* Which kernels serve a call.  AUTO is the dispatcher (M-based, see below);
 * the others force one path (tests compare paths against each other). */
typedef enum {
  SWIGLU_PATH_AUTO = 0,
  SWIGLU_PATH_SIMT = 1,     /* split-K CUDA-core GEMV + reduction (f32 and bf16) */
  SWIGLU_PATH_SKINNY = 2,   /* split-K tcgen05 swap-AB partials + reduction (bf16) */
  SWIGLU_PATH_TC = 3        /* tcgen05 tile GEMM with the SwiGLU epilogue (bf16)  */
} swiglu_path;

/*
 * h = silu(x . W_gate) (.) (x . W_up).
 *
 * Dispatch (AUTO): f32 -> SIMT path; bf16 with M <= the skinny limit
 * (swiglu_plan reports it) -> SKINNY; larger bf16 M -> TC.  One row on
 * weights of 32 MB or less with d <= 2048 (f32) or d <= 1024 (bf16) takes
 * the SIMT path's cluster form (one launch, no workspace).  The split-K
 * paths, and the TC path where it splits its last wave of tiles along K
 * (stream-K), need a workspace for their partial sums; this entry point takes it
 * from a library-owned, stream-ordered pool (cudaMallocFromPoolAsync /
 * cudaFreeAsync on `stream`), so calls on different streams never share it.
 * The buffer is cached per stream (up to 256 streams, 256 MB of partial sums
 * each) and reused by the stream's later calls; swiglu_release_stream_workspace
 * and swiglu_release_workspaces give it back.
 * A call captured into a CUDA graph takes its workspace from memory the
 * library allocates outside the graph. It switches the calling thread to
 * relaxed capture mode for a cudaMalloc and a clearing memset on a private
 * stream, then restores the mode. There is one zeroed slice per capture
 * sequence and capturing stream, shared by that capture's calls on that
 * stream, which run one after another.
 *   - These slices are kept until the process exits, because the graph may be
 *     replayed at any time; the release calls do not free them.
 *   - Two instances (graph execs) of one captured graph must not run at the
 *     same time.
 *   - Past 8 GB of slices on a device, captures allocate inside the graph
 *     instead (allocation and free nodes), taking their arrival counters from
 *     a 4 MB zeroed region.  The first call on a device that uses arrival
 *     counters outside a capture creates that region, and waits for `stream`
 *     once to do so.
 * Errors: SWIGLU_ERR_INVALID_ARG, _ALIGNMENT, _ARCH, _OOM, _CUDA.
 */
SWIGLU_API int swiglu_up(const void* x, const void* w_gate, const void* w_up, void* h,
              int64_t M, int64_t d, int64_t d_ff, int dtype, void* stream);

/*
 * As swiglu_up, with an explicit path and an optional caller workspace.
 *   path       a swiglu_path; a forced path that cannot serve the call (e.g.
 *              SKINNY or TC for f32) returns SWIGLU_ERR_UNSUPPORTED.
 *   workspace  device buffer, 256-byte aligned, of at least
 *              swiglu_workspace_bytes(M, d, d_ff, dtype, path) bytes, or NULL
 *              to use the library pool.  Used only by the enqueued work; the
 *              caller must keep it alive until that work completes and must
 *              not share it between calls that may run concurrently.
 */
SWIGLU_API int swiglu_up_ex(const void* x, const void* w_gate, const void* w_up, void* h,
                 int64_t M, int64_t d, int64_t d_ff, int dtype, int path,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Down projection y = h . W_down (+ residual): the MLP's second GEMM and its
 * residual addition ("1 . Anatomie d'un transformeur sur GPU", section 1.6,
 * kernels #10 "GEMM down" and #11 the residual).
 *
 *     h        [M, d_ff]  row-major (typically swiglu_up's output)
 *     w_down   [d_ff, d]  row-major (element (k, j) at k*d + j)
 *     residual [M, d]     row-major, or NULL for none; it may be y itself
 *                         (in-place residual update) but must not partially
 *                         overlap y
 *     y        [M, d]     row-major output; must not overlap h or w_down
 *
 * Sums in f32 over k, the residual added to the f32 sum, one rounding to the
 * output type.  bf16 only (f32 returns SWIGLU_ERR_UNSUPPORTED), on the
 * tensor-core paths: M up to the skinny limit that swiglu_down_plan reports
 * (256) -> split-K skinny kernel, larger M -> tile kernel (SWIGLU_PATH_SIMT
 * is rejected).  Above 32 MB of weights the skinny kernel's stream-K form
 * enqueues two kernels: one writes partial sums, the second adds them (in
 * k order, the same bits as one kernel would give) and the residual.
 * d_ff == 0 gives y = residual (or 0).
 * Workspace, streams, determinism and errors as for swiglu_up.
 */
SWIGLU_API int swiglu_down(const void* h, const void* w_down, const void* residual, void* y,
                           int64_t M, int64_t d_ff, int64_t d, int dtype, void* stream);

/* As swiglu_down, with an explicit path and optional caller workspace (see
 * swiglu_up_ex; size from swiglu_down_workspace_bytes). */
SWIGLU_API int swiglu_down_ex(const void* h, const void* w_down, const void* residual, void* y,
                              int64_t M, int64_t d_ff, int64_t d, int dtype, int path,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of swiglu_down_ex on the current device (0 when invalid). */
SWIGLU_API size_t swiglu_down_workspace_bytes(int64_t M, int64_t d_ff, int64_t d, int dtype,
                                              int path);

/*
 * As swiglu_up_ex and swiglu_down_ex, for weights stored with the shared
 * dimension contiguous -- the layout of torch.nn.Linear.weight:
 *     w_gate_nk, w_up_nk [d_ff, d]   (element (j, k) at j*d + k)
 *     w_down_nk          [d, d_ff]   (element (j, k) at j*d_ff + k)
 * No copy or transpose is made: the kernels read these weights directly
 * (the decode article's "TransposedMatmul" point, "Deux operations de trop":
 * a . b^T without copying b).  bf16 on the tensor-core paths only;
 * SWIGLU_PATH_SIMT and f32 return SWIGLU_ERR_UNSUPPORTED.  Workspace sizes
 * are those of the [K, N] entry points.
 */
SWIGLU_API int swiglu_up_nk(const void* x, const void* w_gate_nk, const void* w_up_nk, void* h,
                            int64_t M, int64_t d, int64_t d_ff, int dtype, int path,
                            void* workspace, size_t workspace_bytes, void* stream);
SWIGLU_API int swiglu_down_nk(const void* h, const void* w_down_nk, const void* residual, void* y,
                              int64_t M, int64_t d_ff, int64_t d, int dtype, int path,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * Weight packing (step a0).  "Tile-Level Activation Overlap for Efficient
 * LLM Inference", Kernel-2, interleaves the gate and up weight columns once,
 * before any GEMM, so that one tile of the packed matrix holds matching gate
 * and up columns.  Here the interleave unit is a block of 64 columns:
 *
 *     w_packed [d, 2P], P = ceil(d_ff / 64) * 64, row k =
 *         W_gate[k, 0:64] | W_up[k, 0:64] | W_gate[k, 64:128] | W_up[k, 64:128] | ...
 *
 * with zeros where a column index reaches d_ff.  The packing copies element
 * bits (nothing is rounded) and is done once per weight set, off the
 * per-call path.
 *
 * swiglu_packed_weight_bytes: size of w_packed (d * 2P * element size), or 0
 *   for invalid sizes.  Host-only.
 * swiglu_pack_weights: writes w_packed from w_gate and w_up (both [d, d_ff]
 *   row-major), asynchronously on `stream`.  w_packed is caller-owned device
 *   memory of swiglu_packed_weight_bytes bytes, 16-byte aligned, overlapping
 *   neither input.  Errors: SWIGLU_ERR_INVALID_ARG, _ALIGNMENT, _ARCH, _CUDA.
 * swiglu_up_packed: as swiglu_up_ex, reading both weight matrices from
 *   w_packed; every path and dtype of swiglu_up_ex is served, and workspace
 *   sizes are those of swiglu_workspace_bytes.  h [M, d_ff] must not overlap
 *   x or w_packed.
 */
SWIGLU_API size_t swiglu_packed_weight_bytes(int64_t d, int64_t d_ff, int dtype);
SWIGLU_API int swiglu_pack_weights(const void* w_gate, const void* w_up, void* w_packed,
                                   int64_t d, int64_t d_ff, int dtype, void* stream);
SWIGLU_API int swiglu_up_packed(const void* x, const void* w_packed, void* h, int64_t M,
                                int64_t d, int64_t d_ff, int dtype, int path, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * FP8 weights (e4m3) on the tcgen05 kind::f8f6f4 tensor cores.  "Tile-Level
 * Activation Overlap for Efficient LLM Inference" (problem statement)
 * observes that quantization shrinks the GEMM's share of the time and so
 * raises the activation's; this is the up projection with 8-bit operands and
 * the same fused epilogue.
 *
 * Numerical contract.  Weights are quantized once, per output column:
 * amax_j = max_k |W[k, j]|, code = e4m3(f32(W[k, j]) * f32(448 / amax_j)),
 * scale_j = f32(amax_j / 448) (e4m3: 1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits, largest finite value 448; conversion rounds to nearest even
 * and saturates).  Each call quantizes x per row the same way (into the
 * workspace), sums code products in f32 on the tensor cores, multiplies each
 * sum by scale_x[i] * scale_w[j], and applies h = silu(g) * u to the scaled
 * f32 sums; h is bf16.  An all-zero row or column gets scale 0.  The result
 * is the fused definition evaluated on the dequantized operands (code value
 * times scale), within the bf16 tolerance.
 *
 * swiglu_quantize_weights_fp8: w_gate, w_up bf16 [d, d_ff] row-major ->
 *   w8_gate, w8_up: e4m3 codes [d_ff, d] (the shared dimension contiguous,
 *   as tcgen05 reads 8-bit operands), s_gate, s_up: f32 [d_ff].  All
 *   caller-owned device memory, 16-byte aligned; the outputs overlap neither
 *   each other nor the inputs.  Asynchronous on `stream`; uses a short-lived
 *   d_ff * 4-byte allocation from the library's stream-ordered pool.
 * swiglu_up_fp8: x bf16 [M, d], the codes and scales above, h bf16 [M, d_ff].
 *   Paths: AUTO (SKINNY for M <= the skinny limit, else TC), SKINNY, TC;
 *   SIMT returns SWIGLU_ERR_UNSUPPORTED.  Workspace as swiglu_up_ex, sized by
 *   swiglu_fp8_workspace_bytes.  It also holds x's codes and row scales: in
 *   a caller workspace, after the call, bytes [0, M d) are x's e4m3 codes
 *   [M, d] and the M f32 row scales start at byte M d rounded up to 256.
 * Both need d a multiple of 16 and d_ff a multiple of 8
 * (SWIGLU_ERR_ALIGNMENT); other errors as swiglu_up_ex.
 */
SWIGLU_API int swiglu_quantize_weights_fp8(const void* w_gate, const void* w_up, void* w8_gate,
                                           void* w8_up, float* s_gate, float* s_up, int64_t d,
                                           int64_t d_ff, void* stream);
SWIGLU_API int swiglu_up_fp8(const void* x, const void* w8_gate, const void* w8_up,
                             const float* s_gate, const float* s_up, void* h, int64_t M,
                             int64_t d, int64_t d_ff, int path, void* workspace,
                             size_t workspace_bytes, void* stream);
SWIGLU_API size_t swiglu_fp8_workspace_bytes(int64_t M, int64_t d, int64_t d_ff, int path);

/*
 * The same FP8 contract for the down projection y = h . W_down (+ residual)
 * ("1 . Anatomie d'un transformeur sur GPU", section 1.6, kernels #10 and
 * #11): h [M, d_ff] bf16 is quantized per row inside the call, W_down once
 * per output column, and each f32 sum is scaled by scale_h[i] * scale_w[j]
 * before the residual (bf16 [M, d], may be y itself) is added and y [M, d]
 * is rounded to bf16.
 *
 * swiglu_quantize_weight_fp8: one bf16 matrix w [K, N] row-major -> e4m3
 *   codes w8 [N, K] (K contiguous) and f32 column scales s [N]; for the down
 *   projection K = d_ff, N = d.  Needs K a multiple of 16.  As
 *   swiglu_quantize_weights_fp8 otherwise.
 * swiglu_down_fp8: paths AUTO (SKINNY for M <= its skinny limit, else TC),
 *   SKINNY, TC; needs d_ff a multiple of 16.  Workspace sized by
 *   swiglu_down_fp8_workspace_bytes (h's codes and row scales first, as in
 *   swiglu_up_fp8).  Other errors as swiglu_down_ex.
 */
SWIGLU_API int swiglu_quantize_weight_fp8(const void* w, void* w8, float* s, int64_t K,
                                          int64_t N, void* stream);
SWIGLU_API int swiglu_down_fp8(const void* h, const void* w8_down, const float* s_down,
                               const void* residual, void* y, int64_t M, int64_t d_ff,
                               int64_t d, int path, void* workspace, size_t workspace_bytes,
                               void* stream);
SWIGLU_API size_t swiglu_down_fp8_workspace_bytes(int64_t M, int64_t d_ff, int64_t d, int path);

/*
 * The whole MLP of "1 . Anatomie d'un transformeur sur GPU", section 1.1,
 * after its RMSNorm: h = silu(x . W_gate) (.) (x . W_up), then
 * y = h . W_down (+ residual).  Two kernels on `stream`; h [M, d_ff] is the
 * caller's buffer and holds the up projection's (bf16-rounded) output
 * afterwards.  y may be x only when residual is x too.  bf16 only.  All
 * arguments of both steps are validated before anything is enqueued.
 */
SWIGLU_API int swiglu_mlp(const void* x, const void* w_gate, const void* w_up,
                          const void* w_down, const void* residual, void* h, void* y,
                          int64_t M, int64_t d, int64_t d_ff, int dtype, void* stream);

/*
 * As swiglu_up, for callers that cannot allocate device memory.  Some
 * callers may not call cudaMalloc (or any allocator) while they run this
 * operation: a host framework that invokes operators from an enqueue
 * callback in which allocation is forbidden, a process whose device memory is
 * entirely reserved by another allocator, or a latency-critical loop in which
 * an allocation or free could block or synchronise the device.  This entry
 * point allocates nothing: it runs the SIMT split-K path (the per-slice
 * partial-sum kernel and the reduction kernel) with the partial sums in a
 * fixed scratch array that the library holds in device memory, of
 * SWIGLU_NOALLOC_SCRATCH_BYTES bytes on every GPU that loads the library,
 * until the process exits.  The caller still passes x, the weights and h.
 * There is no counterpart of this entry point in the pages.
 *
 *   - Set-up: the first call on a device, with that device current, looks up
 *     the scratch array's device address (cudaGetSymbolAddress) and caches
 *     it; make that first call before any stream capture.
 *   - Limit: a call whose partial sums need more than
 *     SWIGLU_NOALLOC_SCRATCH_BYTES returns SWIGLU_ERR_WORKSPACE and enqueues
 *     nothing.  The need is slices x M x 2 x d_ff x 4 bytes, slices being
 *     the split-K kernel's K slices (swiglu_plan reports them and this
 *     `workspace` for SWIGLU_PATH_SIMT, except for the one-row calls that
 *     swiglu_up serves with the SIMT path's cluster form, which this entry
 *     point does not use); on a 152-SM GB300 the d = 4096, d_ff = 14336
 *     decode calls need at most 7.3 MB (M = 16).
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's contents.  Nothing in it needs to start at zero (each call
 *     writes every partial it later reads), but calls that may overlap on
 *     the GPU (on different streams, or from different threads without
 *     ordering) race on it and must be serialised by the caller.
 *   - Validation and other errors: as swiglu_up.
 */
#define SWIGLU_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
SWIGLU_API int swiglu_up_noalloc(const void* x, const void* w_gate, const void* w_up, void* h,
                                 int64_t M, int64_t d, int64_t d_ff, int dtype, void* stream);

/* Workspace bytes a call with these arguments needs on the current device
 * (0 for TC calls whose tiles fill whole waves of the GPU).  Returns 0 and sets
 * the thread's error string when the arguments are invalid or no device is
 * current. */
SWIGLU_API size_t swiglu_workspace_bytes(int64_t M, int64_t d, int64_t d_ff, int dtype,
                              int path);

/* How a call would be served.
 *   num_sms > 0   for a device with `num_sms` SMs: host-only, needs no GPU,
 *                 a pure function of its arguments (thread-block cluster
 *                 capacities are estimated from the SM count).
 *   num_sms == 0  on the current device, exactly as a call would be: its SM
 *                 count and the cluster capacities it reports
 *                 (cudaOccupancyMaxActiveClusters).  Needs a GPU; without
 *                 one it returns SWIGLU_ERR_CUDA. */
typedef struct {
  int path;              /* resolved swiglu_path                                */
  int64_t slices;        /* K slices of the split-K paths (1 for TC)            */
  int64_t grid;          /* CTAs of the main kernel                              */
  int64_t row_chunk;     /* rows of x per SIMT pass (SIMT path)                  */
  int64_t workspace;     /* bytes of partial sums                                */
  int64_t skinny_max_m;  /* largest bf16 M that AUTO sends to SKINNY at these
                            weight sizes.  Up projection: 32, or 128 for
                            weights of 32 MB or less (where one row may take
                            the SIMT path's cluster form instead).  Down
                            projection: 256                                  */
  int64_t launches;      /* kernel launches one call enqueues                   */
  int64_t cluster;       /* CTAs per thread-block cluster of the main kernel
                            (1: none; 2-8: the skinny kernel's split-K
                            clusters; 4-8: the SIMT path's cluster form, 8
                            unless 8-CTA clusters would not all fit at once
                            on the device; 2: the TC path's CTA pairs)       */
} swiglu_plan_info;

SWIGLU_API int swiglu_plan(int64_t M, int64_t d, int64_t d_ff, int dtype, int path,
                int num_sms, swiglu_plan_info* out);

/* As swiglu_plan, for the down projection y [M, d] = h [M, d_ff] . W_down. */
SWIGLU_API int swiglu_down_plan(int64_t M, int64_t d_ff, int64_t d, int dtype, int path,
                                int num_sms, swiglu_plan_info* out);

/*
 * The K-slice rule of "Ou part le temps d'un token", section "Un kernel pour
 * les matrices etroites": split the shared dimension K so that
 * col_blocks * slices approaches target_blocks, without any slice having
 * fewer than min_k_per_slice indices (and at least one slice).  Host-only.
 * Returns the slice count, or -1 on invalid arguments.
 */
SWIGLU_API int64_t swiglu_split_k_slices(int64_t K, int64_t col_blocks,
                              int64_t target_blocks, int64_t min_k_per_slice);

/*
 * Workspace cache management (the per-stream buffers swiglu_up, swiglu_down
 * and the FP8 entry points keep when they run without a caller workspace).
 * The workspace serves the split-K reductions of "Ou part le temps d'un
 * token", section "Un kernel pour les matrices etroites".
 *
 * swiglu_release_stream_workspace: frees the buffer cached for `stream` on
 *   the current device, stream-ordered (cudaFreeAsync on `stream`, after the
 *   work already enqueued there).  Call it before destroying a stream that
 *   made calls; a later call on the stream allocates a new buffer.  NULL is
 *   the legacy default stream.  Returns SWIGLU_OK (also when nothing was
 *   cached) or SWIGLU_ERR_CUDA.
 * swiglu_release_workspaces: waits for the current device to finish its
 *   work (cudaDeviceSynchronize), frees every buffer cached on it, including
 *   those of streams already destroyed, and returns the library pool's unused
 *   memory to the driver.  Returns SWIGLU_OK or SWIGLU_ERR_CUDA.
 * swiglu_cached_workspace_bytes: bytes the cache holds on the current
 *   device (0 when no device is current); the workspaces of captured calls
 *   (see swiglu_up) are not part of the cache.
 * Neither release call may run while another thread enqueues calls of this
 * library on the same stream (release_stream) or device (release).
 */
SWIGLU_API int swiglu_release_stream_workspace(void* stream);
SWIGLU_API int swiglu_release_workspaces(void);
SWIGLU_API size_t swiglu_cached_workspace_bytes(void);

/* Reads and clears the device-side error word that bounded waits inside the
 * kernels set when they give up.  Synchronises the current device first.
 * Returns SWIGLU_OK, SWIGLU_ERR_TIMEOUT or SWIGLU_ERR_CUDA. */
SWIGLU_API int swiglu_check_device_status(void);

/* Self-test of failure detection: launches one CTA that waits, through the
 * same bounded wait the tensor-core kernels use, on a barrier that nothing
 * ever completes.  After `timeout_ms` (1..10000) the wait gives up, raises
 * the device error word and the kernel returns normally, so the next
 * swiglu_check_device_status() reports SWIGLU_ERR_TIMEOUT and the CUDA
 * context stays usable.  No counterpart in the pages. */
SWIGLU_API int swiglu_selftest_wait_timeout(int timeout_ms, void* stream);

/* Text for a swiglu_status value (static storage). */
SWIGLU_API const char* swiglu_status_string(int status);

/* Detail of the calling thread's most recent failure ("" if none). */
SWIGLU_API const char* swiglu_last_error_string(void);

/* Library version, as MAJOR*10000 + MINOR*100 + PATCH. */
SWIGLU_API int swiglu_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SWIGLU_GB300_H */
