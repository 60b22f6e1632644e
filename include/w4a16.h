/*
 * w4a16.h - C ABI of libw4a16.so: the W4A16 mixed-precision linear layer on one NVIDIA GB300 (sm_103a).
 *
 *     C[M, N] = A[M, K] . dequant(W) (+ bias[N])
 *
 * A is fp16 or bf16. W is stored as unsigned 4-bit values packed eight per int32 along N
 * (b_q[K, N/8]) with one scale per (group of G rows of K, output column) and a zero point that
 * is either the fixed bias zp_bias (8 for the symmetric uint4b8 type) or unpacked from
 * qzeros[K/G, N/8]:   dequant(W)[k, n] = (q[k, n] - zp[k/G, n]) * scales[k/G, n].
 *
 * Sources (the pages describing the method):
 *   - "PR #51453 report: register Triton W4A16 GEMM as custom op" - key source snippets: the facade
 *     triton_w4a16_gemm(a, b_q, scales, qzeros, group_size, zp_bias=8), the fake implementation
 *     (out shape (M, b_q.size(1)*8), dtype and device of a), and the fake-impl test shapes
 *     a(4,256) b_q(256,64) scales(2,512) group_size 128 -> out(4,512).
 *   - "PR #43731 report: TritonW4A16LinearKernel as CUDA fallback" - key source snippets:
 *     can_implement() rejections (fp16/bf16 activations only, N % 8 == 0, no g_idx, supported group
 *     sizes or G == K) and their reason strings; motivation: K or N = 2112 must work.
 *   - "PR #40977 report: ROCm RDNA hybrid W4A16" - key source snippets: the test reference
 *     (dequant in high precision, bias added before the cast to the activation dtype), and the
 *     runtime routing on M between a skinny split-K decode kernel and a tiled prefill kernel.
 *
 * Conventions shared by every entry point:
 *   - Tensor pointers are device pointers owned by the caller, contiguous and row-major. Natural
 *     alignment is required (2 bytes for 16-bit tensors, 4 bytes for int32). Higher alignment
 *     (16 bytes) and N % 32 == 0, K % 8 == 0 unlock the TMA-fed paths; otherwise a generic GPU path runs.
 *   - scales, bias, out and w_out have the dtype of A.
 *   - Calls are stream-ordered on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *     w4a16_gemm, w4a16_pack, w4a16_unpack and w4a16_dequant allocate nothing, do not synchronise and
 *     read nothing back to the host, and keep no pointer after they return.
 *   - w4a16_gemm kernels use programmatic dependent launch: when the previous kernel of the stream
 *     releases its dependents early (as this library's kernels do), a w4a16_gemm kernel may start
 *     fetching b_q, scales and qzeros - model parameters - before that kernel has finished. a and bias
 *     are read, and out is written, only after it has completed. So do not let the kernel that runs
 *     just before w4a16_gemm on the same stream write that call's b_q, scales or qzeros unless it
 *     completes normally (kernels that do not use programmatic launch always do).
 *   - Errors are reported by the returned status; a human-readable reason for the last failure on the
 *     calling thread is available from w4a16_last_error(). Validation happens before any launch, so a
 *     rejected call touches no memory. The library never aborts the process and device code never traps.
 *   - Rows M may be 0 (nothing is launched). There is no g_idx (activation reordering) argument: the
 *     pages' kernel rejects it.
 */
#ifndef W4A16_H_
#define W4A16_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *w4a16_stream_t;

typedef enum { W4A16_F16 = 0, W4A16_BF16 = 1 } w4a16_dtype;

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_INVALID_ARG = 1, /* shapes, null pointers, aliasing, zp_bias range            */
  W4A16_ERR_UNSUPPORTED = 2, /* dtype or group size outside what the layer defines         */
  W4A16_ERR_MISALIGNED = 3,  /* a pointer is not naturally aligned for its element type     */
  W4A16_ERR_CUDA = 4,        /* a CUDA runtime call failed; the message carries its text     */
  W4A16_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (see w4a16_get_device_error) */
} w4a16_status;

/* Kernel paths chosen by the runtime dispatcher (w4a16_plan / w4a16_debug_selected_path). */
typedef enum {
  W4A16_PATH_NONE = 0,    /* M == 0: nothing to do                                            */
  W4A16_PATH_GENERIC = 1, /* any alignment: one thread per (8 output columns, 8 rows), K-sliced   */
  W4A16_PATH_DECODE = 2,  /* M <= 32: split-K skinny GEMM, TMA weight stream, ldmatrix.trans +
                             in-register magic-number dequant, mma.sync, cluster (DSMEM) split-K */
  W4A16_PATH_PREFILL = 3  /* large M: TMA-fed tcgen05/TMEM GEMM, int4 tiles dequantised into
                             shared memory before each UMMA                                     */
} w4a16_path;

/* Launch plan for one w4a16_gemm call. Filled by w4a16_plan; informational. */
typedef struct {
  int32_t path;          /* w4a16_path                                                     */
  int32_t k_blocks_per_stage; /* decode: 64-row K blocks per pipeline stage (1, 2 or 4); else 1 */
  int32_t m_tile;        /* rows of A per CTA                                              */
  int32_t n_tile;        /* output columns per CTA                                         */
  int32_t k_split;       /* CTAs (one cluster) sharing one output tile along K               */
  int32_t warps;         /* warps per CTA                                                  */
  int64_t grid;          /* CTAs launched                                                  */
  int32_t smem_bytes;    /* dynamic shared memory per CTA                                  */
  int32_t stream_k;      /* PREFILL: 1 when persistent CTAs share (tile, K block) units evenly  */
} w4a16_plan_t;

/*
 * w4a16_pack - pack 4-bit values eight per int32 along the last dimension.
 *   q:      device, uint8 [rows, n], each value 0..15 (higher bits are ignored)
 *   packed: device, int32 [rows, n/8]; nibble j (bits 4j..4j+3) of word c receives q[r, 8c+j].
 * The nibble order inside a word is not printed on the pages; sequential little-endian order is
 * the plain reading of "eight values packed along N" (PR #51453 report, implementation breakdown:
 * N = b_q.shape[1] * 8). Used for weights [K, N] -> b_q and zero points [K/G, N] -> qzeros.
 * Errors: INVALID_ARG if rows < 0, n <= 0, n % 8 != 0, a null pointer with rows > 0, or overlap.
 */
w4a16_status w4a16_pack(const uint8_t *q, int32_t *packed, int64_t rows, int64_t n,
                        w4a16_stream_t stream);

/* w4a16_unpack - inverse of w4a16_pack: packed int32 [rows, n/8] -> uint8 [rows, n] (values 0..15). */
w4a16_status w4a16_unpack(const int32_t *packed, uint8_t *q, int64_t rows, int64_t n,
                          w4a16_stream_t stream);

/*
 * w4a16_repack_k_to_n - ingest weights packed along K, int32 [n, k/8] (the "[N, K//8] int32" layout
 * of the PR #40977 report, implementation breakdown and key source snippets), into this library's
 * b_q int32 [k, n/8] layout. The report does not print the order of the nibbles inside a K-packed
 * word; this function reads nibble j (bits 4j..4j+3) of word c of row r as weight [k = 8c+j, n = r],
 * the same sequential little-endian convention as w4a16_pack, applied along K. A load-time step.
 *   k_packed: device, int32 [n, k/8];  b_q: device, int32 [k, n/8].
 * Errors: INVALID_ARG if k or n is not positive or not divisible by 8, a pointer is NULL, or the
 * buffers overlap; MISALIGNED if either is not 4-byte aligned.
 */
w4a16_status w4a16_repack_k_to_n(const int32_t *k_packed, int32_t *b_q, int64_t k, int64_t n,
                                 w4a16_stream_t stream);

/*
 * Prepacked weights: this library's kernel-native layout of b_q (a load-time step; the pages' kernels
 * read b_q as it is). The packed words are regrouped into blocks of 64 K rows x 32 words (the 256
 * output columns of one column tile), stored tile-major and then by K block, each block 8 KB
 * contiguous; K and N are padded with zero words to multiples of 64 and 256. Inside a block row r
 * holds its 32 words with the 16-byte chunk j at position j ^ (r % 8) - the order in which the
 * kernels keep a block in shared memory - so a block reaches shared memory by one plain bulk copy
 * instead of a 64-row tensor copy. Both the decode and the prefill kernels read it; the generic path
 * does not.
 *
 * w4a16_prepack_bytes - bytes of the prepacked form of a [k, n] weight matrix (0 for invalid sizes).
 * w4a16_prepack - b_q int32 [k, n/8] -> b_pp (w4a16_prepack_bytes(k, n) bytes, 16-byte aligned), every
 *   byte written (padding included). Device pointers, stream-ordered, no allocation.
 *   Errors: INVALID_ARG (k or n not positive, n % 8 != 0, NULL, overlap), MISALIGNED (b_q 4 bytes,
 *   b_pp 16 bytes).
 */
size_t w4a16_prepack_bytes(int64_t k, int64_t n);
w4a16_status w4a16_prepack(const int32_t *b_q, int32_t *b_pp, int64_t k, int64_t n, w4a16_stream_t stream);

/*
 * w4a16_dequant - materialise dequant(W) in the activation dtype:
 *   w_out[k, n] = RNE_dtype((q[k, n] - zp[k/G, n]) * scales[k/G, n])
 * i.e. the exact product rounded once to nearest-even (dequantisation rule: PR #40977 report, key
 * source snippets, test reference; zp = qzeros nibble, or zp_bias when qzeros is NULL). The prefill
 * kernel feeds exactly these values to its tensor-core MMA; the decode kernel multiplies the exact
 * integers q - zp and applies the scale in fp32, so a one-hot activation row reproduces them exactly.
 *   b_q [k, n/8] int32, scales [k/G, n] dtype, qzeros [k/G, n/8] int32 or NULL, w_out [k, n] dtype.
 * Errors: as w4a16_gemm's validation (dtype, n % 8, group size, k % G, zp_bias, nulls, overlap).
 */
w4a16_status w4a16_dequant(const int32_t *b_q, const void *scales, const int32_t *qzeros,
                           int64_t k, int64_t n, int group_size, int zp_bias, w4a16_dtype dtype,
                           void *w_out, w4a16_stream_t stream);

/*
 * w4a16_gemm - out[M, N] = cast_dtype( A[M, K] . dequant(W) (+ bias) ), fp32 accumulation.
 *   a       [m, k]    dtype            activations (PR #51453 facade argument a)
 *   b_q     [k, n/8]  int32            packed 4-bit weights
 *   scales  [k/G, n]  dtype            per-group scales
 *   qzeros  [k/G, n/8] int32 or NULL   packed zero points; NULL selects the fixed zp_bias
 *   group_size G in {32, 64, 128} or G == k (per-channel); k % G == 0
 *   zp_bias 0..15 (8 = symmetric uint4b8); ignored when qzeros is given
 *   bias    [n] dtype or NULL          added in fp32 before the cast (PR #40977 test reference)
 *   out     [m, n]    dtype            written; must not overlap any input
 * The kernel and its tile, split-K factor and cluster size are chosen on every call from the runtime
 * M, K, N, G and the device (SM count, shared memory), never frozen between calls - the failure the
 * PR #51453 report describes (prefill tile configuration reused for decode under compilation).
 * Dequantised weights are rounded to the dtype before the product, exactly as w4a16_dequant returns
 * them; the sum is kept in fp32 and rounded once (nearest-even) after the bias.
 * Errors: UNSUPPORTED (dtype, group size), INVALID_ARG (shapes, nulls, zp_bias, overlap),
 *         MISALIGNED (natural alignment), CUDA (launch failure). A kernel that gives up a bounded
 *         device-side wait is reported later by w4a16_get_device_error (no host read happens here).
 */
w4a16_status w4a16_gemm(const void *a, const int32_t *b_q, const void *scales, const int32_t *qzeros,
                        int group_size, int zp_bias, const void *bias, void *out, int64_t m,
                        int64_t k, int64_t n, w4a16_dtype dtype, w4a16_stream_t stream);

/*
 * w4a16_gemm_ws - w4a16_gemm with a caller-owned scratch buffer, which lets large-M calls whose
 * output tiles do not fill the GPU in whole waves use stream-K: persistent CTAs take equal shares of
 * the (tile, K block) work and exchange fp32 partial tiles through the workspace.
 *   workspace       device memory, 256-byte aligned, at least w4a16_gemm_workspace_size(...) bytes
 *                   (a smaller or NULL workspace simply disables stream-K). Its first 4 KiB hold
 *                   per-CTA flags: they must be zero before the first use, and every call that
 *                   completes leaves them zero again; the rest is scratch whose contents between
 *                   calls do not matter (zero-filling the whole buffer once is the simple way to
 *                   satisfy this). A call that gives up a bounded wait (w4a16_get_device_error then
 *                   reports W4A16_ERR_TIMEOUT) may leave flags set: zero the first 4 KiB again before
 *                   the workspace is used by another call.
 *   workspace_bytes its size
 * Calls that may run concurrently (different streams) need different workspaces. Everything else
 * is as for w4a16_gemm (no allocation, no synchronisation, no host read).
 * Errors: as w4a16_gemm, plus INVALID_ARG if the workspace overlaps a tensor argument and
 * MISALIGNED if it is not 256-byte aligned.
 */
w4a16_status w4a16_gemm_ws(const void *a, const int32_t *b_q, const void *scales, const int32_t *qzeros,
                           int group_size, int zp_bias, const void *bias, void *out, int64_t m, int64_t k,
                           int64_t n, w4a16_dtype dtype, void *workspace, size_t workspace_bytes,
                           w4a16_stream_t stream);

/*
 * w4a16_gemm_noalloc - w4a16_gemm_ws without a caller-provided workspace and without allocating:
 * for callers that cannot call cudaMalloc - e.g. code running while a CUDA graph is being captured
 * (allocation is not capturable), allocator-less runtimes and plugins handed only tensor pointers, or
 * hosts that forbid device allocations after start-up. The paper has no counterpart; it is an
 * addition of this library.
 *   The scratch is a static device array inside the library (40 MiB + 4 KiB: stream-K partial tiles
 *   for up to 160 CTAs and their flags). Every GPU that loads the library holds it until the process
 *   exits. The first call on a device looks its address up (cudaGetSymbolAddress) with that device
 *   current; make that first call before any stream capture.
 *   Every call on a device shares the one array, which keeps the previous call's contents: the call
 *   clears the part that must start at zero (the flags) on `stream` first. Calls that overlap on the
 *   GPU (other streams, other threads, graphs replayed concurrently) race on it: serialise them.
 *   A call whose plan needs more scratch than the array holds (stream-K on a device with more than
 *   160 SMs) is rejected with W4A16_ERR_UNSUPPORTED and the sizes in the message, rather than run
 *   with a different plan: a call of this entry point always runs the plan that w4a16_gemm_ws runs
 *   with a large enough workspace, never a slower one in its place. A caller that wants the plan
 *   without scratch calls w4a16_gemm, which needs no workspace and allocates nothing either.
 * It calls no cudaMalloc, cudaFree or allocating library routine. Arguments, results and other
 * errors are those of w4a16_gemm.
 */
w4a16_status w4a16_gemm_noalloc(const void *a, const int32_t *b_q, const void *scales,
                                const int32_t *qzeros, int group_size, int zp_bias, const void *bias,
                                void *out, int64_t m, int64_t k, int64_t n, w4a16_dtype dtype,
                                w4a16_stream_t stream);

/* Bytes of workspace w4a16_gemm_ws can use for these sizes on the current device (0: none). */
size_t w4a16_gemm_workspace_size(int64_t m, int64_t k, int64_t n, int group_size, int dtype);

/*
 * Prepared layer: the weights of one linear layer checked once, and per call shape the dispatcher's
 * plan and the TMA descriptors of the weights kept, so that a call (a model's per-layer, per-step
 * call) checks and encodes only the activations and the output. The handle stores the weight
 * pointers, not copies: the caller keeps b_q, scales, qzeros and bias alive and unchanged while the
 * handle is in use. It is bound to the device current at creation. A handle may be used from
 * several threads (an internal lock guards its cache).
 *
 * w4a16_layer_create - validates the layer configuration as w4a16_gemm does (dtype, n % 8, group
 *   size, k % G, zp_bias, NULL b_q / scales, natural alignment) and returns a handle in *layer.
 *   Host memory only; no device access. Errors: those of the validation.
 * w4a16_layer_gemm - out[m, n] = w4a16_gemm(a, layer weights, ...) with an optional workspace as in
 *   w4a16_gemm_ws (NULL: none). Same results, launches and errors as w4a16_gemm / w4a16_gemm_ws, plus
 *   INVALID_ARG when the current device is not the layer's.
 * w4a16_layer_workspace_size - w4a16_gemm_workspace_size for this layer and m.
 * w4a16_layer_destroy - releases the handle (NULL is allowed); the weights are not touched.
 */
typedef struct w4a16_layer_st *w4a16_layer_t;
w4a16_status w4a16_layer_create(const int32_t *b_q, const void *scales, const int32_t *qzeros, int group_size,
                                int zp_bias, const void *bias, int64_t k, int64_t n, w4a16_dtype dtype,
                                w4a16_layer_t *layer);
/*
 * w4a16_layer_create_prepacked - as w4a16_layer_create, with the weights in the prepacked layout
 *   (b_pp from w4a16_prepack, 16-byte aligned) instead of b_q. Its calls produce exactly the results of
 *   a layer built on b_q. They run on the TMA-fed kernels only: a call that would take the generic
 *   path (a or out not 16-byte aligned, n % 32 != 0, k % 8 != 0, or a forced generic path) returns
 *   W4A16_ERR_UNSUPPORTED.
 */
w4a16_status w4a16_layer_create_prepacked(const int32_t *b_pp, const void *scales, const int32_t *qzeros,
                                          int group_size, int zp_bias, const void *bias, int64_t k, int64_t n,
                                          w4a16_dtype dtype, w4a16_layer_t *layer);
w4a16_status w4a16_layer_gemm(w4a16_layer_t layer, const void *a, void *out, int64_t m, void *workspace,
                              size_t workspace_bytes, w4a16_stream_t stream);
size_t w4a16_layer_workspace_size(w4a16_layer_t layer, int64_t m);
w4a16_status w4a16_layer_destroy(w4a16_layer_t layer);

/*
 * w4a16_can_implement - host-only check of a layer configuration, mirroring
 * TritonW4A16LinearKernel.can_implement (PR #43731 report, key source snippets): returns W4A16_OK or
 * the rejection status, with the reason available from w4a16_last_error(). No device access.
 *   dtype: W4A16_F16 / W4A16_BF16 (other values rejected); has_g_idx != 0 is rejected.
 */
w4a16_status w4a16_can_implement(int64_t k, int64_t n, int group_size, int dtype, int has_g_idx);

/*
 * w4a16_plan - host-only: the launch plan w4a16_gemm (with_workspace == 0) or w4a16_gemm_ws with a
 * large enough workspace (with_workspace != 0) would use for these sizes on a device with `num_sms`
 * SMs (num_sms <= 0: query the current device). Pointer alignment is assumed to be 16 bytes.
 */
w4a16_status w4a16_plan(int64_t m, int64_t k, int64_t n, int group_size, int dtype, int has_zp,
                        int num_sms, int with_workspace, w4a16_plan_t *plan);

/* Thread-local, NUL-terminated reason for the last failing call on this thread ("" if none). */
const char *w4a16_last_error(void);

/*
 * w4a16_get_device_error - reads and clears the device-side error word of the current device:
 * W4A16_ERR_TIMEOUT if a kernel of this library gave up a bounded wait (it then wrote no result and
 * released its resources), W4A16_OK otherwise. Synchronises the current device.
 */
w4a16_status w4a16_get_device_error(void);

/* Path w4a16_gemm would choose for these sizes on the current device (a w4a16_path value), or -1. */
int w4a16_debug_selected_path(int64_t m, int64_t k, int64_t n, int group_size);

/*
 * w4a16_debug_force_path - restricts the dispatcher to one path for tests and benchmarks:
 * W4A16_PATH_GENERIC, W4A16_PATH_DECODE or W4A16_PATH_PREFILL (used when that path supports the call,
 * otherwise the dispatcher chooses as usual), or -1 to lift the restriction. The initial value comes
 * from the environment variable W4A16_FORCE_PATH (generic|decode|prefill), read once at the first
 * call that plans. Process-wide; not meant for concurrent use with calls on other threads.
 * Errors: INVALID_ARG for any other value.
 */
w4a16_status w4a16_debug_force_path(int path);

/*
 * w4a16_debug_decode_override - fixes parts of the decode path's launch plan for tests and tuning:
 * consumer_groups (1: one group of eight consumer warps per CTA and an 8-block ring, so that two CTAs
 * fit on an SM up to 16 rows; 2: two groups and a 16-block ring, up to 16 rows; calls of 17..32 rows
 * always run one group), k_split (the CTAs of a cluster that split K,
 * 1..16; the rank ranges are rounded to whole stages, which may leave fewer ranks) and
 * k_blocks_per_stage (1, 2 or 4). 0 leaves a field to the dispatcher; all zero restores the
 * automatic plan. Process-wide. Errors: INVALID_ARG for values outside those ranges.
 */
w4a16_status w4a16_debug_decode_override(int consumer_groups, int k_split, int k_blocks_per_stage);

/*
 * w4a16_debug_set_wait_limit_ns - sets the limit of every bounded device-side wait (nanoseconds;
 * 0 restores the default of 2 s). A test sets a tiny limit to make a wait give up and checks that
 * the TIMEOUT status is reported without hanging the GPU. Synchronous.
 */
w4a16_status w4a16_debug_set_wait_limit_ns(uint64_t ns);

/*
 * w4a16_debug_inject_stall - test hook for failure detection (on != 0: enable, 0: disable). While
 * enabled, the worker warps of the TMA-fed kernels first wait on a barrier that nothing arrives on,
 * so that wait runs out after the bounded-wait limit: the kernel records W4A16_ERR_TIMEOUT in its
 * device error word, releases its resources and exits without hanging. Synchronous; current device.
 */
w4a16_status w4a16_debug_inject_stall(int on);

/* Number of kernels this library has launched in this process (all devices, all threads). */
uint64_t w4a16_debug_launch_count(void);

/* Library version string. */
const char *w4a16_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H_ */
