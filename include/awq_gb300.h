/*
 * awq_gb300.h -- C ABI of the GB300 (sm_103a) AWQ W4A16 linear-forward library.
 *
 * The operation (Predibase Lorax "AWQ WQLinear" page):
 *   - Overview: a 4-bit weight-quantised linear layer, GEMM with group-wise
 *     scaling.
 *   - I/O Contract: qweight is int32 [in_features, out_features / 8] holding
 *     eight 4-bit values per int32; qzeros are packed zero points; scales are
 *     per-group scale factors; bias is optional; the output has shape
 *     (*input_shape[:-1], out_features).
 *   - Description, __init__: only w_bit = 4; in_features = rows of qweight;
 *     out_features = 8 x its columns; group_size -1 means one group spanning
 *     in_features; in_features % group_size == 0 and out_features % 8 == 0.
 *   - Description, forward: flatten x to 2-D, run the quantised GEMM with a
 *     pack factor of 8, add the optional bias, restore the batch shape.
 *
 * Notation: M = rows of x (tokens), K = in_features, N = out_features,
 * g = group_size (g = -1 is read as g = K), G = K / g.
 *
 *   W[k, n] = fp16_rn( (q[k, n] - z[k / g, n]) * scales[k / g, n] )
 *   y[m, n] = fp16_rn( sum_k x[m, k] * W[k, n]  +  bias[n] )
 *
 * Readings this library fixes where the page is silent:
 *   - packing: nibble i (bits 4i .. 4i+3, lowest first) of int32 j in a row
 *     holds column 8j + i. qzeros uses the same order, shape [G, N / 8].
 *   - scales: fp16 [G, N]; x, bias, y, W: fp16. q and z are unsigned 0..15.
 *   - the dequantised weight is rounded once to fp16 (round to nearest even)
 *     before it enters the product; the sum over k is accumulated in fp32;
 *     the bias is added to the fp32 sum and the result is rounded once.
 *
 * Conventions for every call below:
 *   - All tensors are device pointers to row-major, contiguous arrays, and
 *     every base pointer must be 16-byte aligned (AWQ_ERR_MISALIGNED if not).
 *   - The caller owns every buffer; outputs are caller-allocated.
 *   - Every call works on the current CUDA device (cudaSetDevice): its
 *     pointers and `stream` must belong to that device.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Argument errors are returned before anything is enqueued. A device-side
 *     error (a bounded wait that timed out) is recorded in a per-device status
 *     word that awq_last_device_status() reads.
 *   - The library keeps, per (device, stream), a scratch area for split-K
 *     partial sums (and, on some paths, dequantised weights or reordered
 *     activations), freed by awq_shutdown. Either reserve it up front with
 *     awq_reserve() -- then no call on that stream allocates or synchronises,
 *     and a call that would need more returns AWQ_ERR_TOO_LARGE -- or let it
 *     grow lazily: the first call that needs more than the stream holds
 *     synchronises the stream and replaces the area (cudaFree + cudaMalloc),
 *     which a stream capture does not allow, so make one call of every shape
 *     and path on the stream before capturing it into a CUDA graph.
 *   - Thread safety: calls may come from several host threads on different
 *     streams. Two host threads must not call at the same time on one stream
 *     (a growing scratch area could be freed under the other call).
 */
#ifndef AWQ_GB300_H
#define AWQ_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; declared here so that this header
 * needs no CUDA header. */
typedef struct CUstream_st *awq_stream_t;

typedef enum {
    AWQ_OK = 0,
    AWQ_ERR_INVALID_ARG = 1, /* a shape rule of the WQLinear page, a NULL required pointer, M < 0 */
    AWQ_ERR_MISALIGNED = 2,  /* a base pointer is not 16-byte aligned */
    AWQ_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
    AWQ_ERR_TIMEOUT = 4,     /* a kernel's bounded wait ran out (device status only) */
    AWQ_ERR_TOO_LARGE = 5    /* the shape needs more than the fixed scratch of
                                awq_linear_forward_decode_noalloc, or more than
                                the stream's reservation (awq_reserve) */
} awq_status_t;

/* Which kernel family serves a forward call. */
typedef enum {
    AWQ_PATH_AUTO = 0,    /* pick by shape (M against the measured crossover) */
    AWQ_PATH_GENERIC = 1, /* any valid shape; plain CUDA-core kernel */
    AWQ_PATH_DECODE = 2,  /* small M: split-K streaming GEMV-style kernel */
    AWQ_PATH_PREFILL = 3, /* large M: tcgen05 / TMEM tensor-core kernel, dequantising in
                             shared memory */
    AWQ_PATH_DEQUANT_GEMM = 4 /* very large M: weights dequantised once per window of at
                             most 256 MB of fp16 into a per-stream scratch area, then the
                             same kernel's tcgen05 GEMM core on each window */
} awq_path_t;

/*
 * awq_linear_forward -- the WQLinear forward (Description, forward steps 2-3):
 *   y[M, N] = fp16_rn(x[M, K] . W[K, N] + bias[N]), W dequantised per group.
 *
 *   x          fp16 [M, K]                      (read)
 *   qweight    int32 [K, N / 8]                 (read)
 *   qzeros     int32 [G, N / 8]                 (read)
 *   scales     fp16 [G, N]                      (read)
 *   bias       fp16 [N], or NULL for no bias    (read)
 *   y          fp16 [M, N]                      (written; must not alias inputs)
 *   M          rows of x; M == 0 returns AWQ_OK and enqueues nothing once K, N and
 *              group_size pass their rules (x and y may then be NULL)
 *   K, N       in_features, out_features (N % 8 == 0)
 *   group_size g > 0 with K % g == 0, or -1 for g = K
 *   stream     CUDA stream to enqueue on
 *
 * Kernel family (AWQ_PATH_AUTO, chosen from measurements on GB300): the
 * decode kernel for M <= 32; the fused tcgen05 prefill kernel for larger M;
 * for M >= 6144 with K <= 16384, the weights dequantised once into a
 * per-stream scratch area (windows of at most 256 MB of fp16, allocated on
 * first use) and the same kernel's tcgen05 GEMM core; the generic kernel
 * for shapes the others do not take.
 *
 * Returns AWQ_ERR_INVALID_ARG for N % 8 != 0, K % g != 0, g == 0, g < -1,
 * M < 0, K <= 0, N <= 0 or a NULL required pointer; AWQ_ERR_MISALIGNED for a
 * pointer that is not 16-byte aligned; AWQ_ERR_CUDA if a launch failed.
 */
awq_status_t awq_linear_forward(const void *x, const int32_t *qweight,
                                const int32_t *qzeros, const void *scales,
                                const void *bias, void *y, int64_t M, int64_t K,
                                int64_t N, int64_t group_size, awq_stream_t stream);

/*
 * awq_linear_forward_path -- awq_linear_forward with the kernel family
 * chosen by the caller (benchmarks and tests use it to time or check one
 * path at every M). Same arguments, same result within the same tolerance.
 * Returns AWQ_ERR_INVALID_ARG if `path` cannot serve this shape
 * (awq_path_supported tells beforehand).
 */
awq_status_t awq_linear_forward_path(const void *x, const int32_t *qweight,
                                     const int32_t *qzeros, const void *scales,
                                     const void *bias, void *y, int64_t M, int64_t K,
                                     int64_t N, int64_t group_size, awq_stream_t stream,
                                     awq_path_t path);

/* 1 if `path` can serve this (valid) shape, else 0. Host-only, no CUDA call. */
int awq_path_supported(int64_t M, int64_t K, int64_t N, int64_t group_size, awq_path_t path);

/* The path AWQ_PATH_AUTO picks for this shape (AWQ_PATH_GENERIC if only the
 * generic kernel fits). Host-only, no CUDA call. Returns -1 for an invalid shape. */
int awq_select_path(int64_t M, int64_t K, int64_t N, int64_t group_size);

/*
 * awq_forward_launches -- how many kernels one awq_linear_forward_path call
 * (or awq_linear_forward with AWQ_PATH_AUTO) enqueues for this shape on the
 * current device: 1 on the decode and generic paths; on the prefill path the
 * persistent kernel plus, when its last partial wave splits tiles along k, the
 * kernel that sums their pieces; on the dequantise-then-GEMM path, per window,
 * the dequant kernel and the GEMM core (plus that sum kernel). For callers that
 * count or budget launches (CUDA graphs). Host-only: reads the current
 * device's SM count, enqueues nothing. Returns 0 for M == 0 and -1 for an
 * invalid shape, a path that cannot serve it, or no CUDA device.
 */
int awq_forward_launches(int64_t M, int64_t K, int64_t N, int64_t group_size, awq_path_t path);

/*
 * awq_decode_tile_columns -- the output-column width of one tile of the decode
 * kernel (AWQ_PATH_DECODE) for this shape: 512 when N is a multiple of 512 and
 * at least 32768 (rows of 256 bytes of packed weights), else 256. Returns 0 if
 * the decode kernel cannot serve the shape and -1 for an invalid shape.
 * Host-only, no CUDA call. Tests use it to check that a shape reaches the
 * kernel variant they mean to exercise.
 */
int awq_decode_tile_columns(int64_t M, int64_t K, int64_t N, int64_t group_size);

/*
 * awq_dequant -- unpack and dequantise the packed weights (the per-group
 * dequantisation of the WQLinear page, Description, __init__ bullet 3):
 *   W[k, n] = fp16_rn((q[k, n] - z[k / g, n]) * scales[k / g, n])
 *
 *   qweight int32 [K, N / 8], qzeros int32 [G, N / 8], scales fp16 [G, N]  (read)
 *   W       fp16 [K, N]                                                   (written)
 * Same argument rules and statuses as awq_linear_forward (no M).
 */
awq_status_t awq_dequant(const int32_t *qweight, const int32_t *qzeros,
                         const void *scales, void *W, int64_t K, int64_t N,
                         int64_t group_size, awq_stream_t stream);

/*
 * awq_linear_forward_rows / awq_finish_rows -- one piece of a row-parallel
 * (K-sharded) WQLinear and its end (the Tensor Parallel Layers page's
 * RowLinear: every shard holds a group-aligned slice of in_features, and the
 * partial results are summed before the bias is added).
 *   awq_linear_forward_rows: y32[M, N] += x[:, 0:K] . W[K, N] in fp32 -- no
 *     bias, no rounding -- where x has row pitch ldx >= K (a K-slice of a
 *     wider x: pass x + k0 and the full width), W is this shard's qweight /
 *     qzeros / scales (K rows, group_size as awq_linear_forward), y32 fp32
 *     [M, N] is caller-allocated and read and written. ldx % 8 == 0. The
 *     kernel family is chosen as for awq_linear_forward.
 *   awq_finish_rows: y[M, N] = fp16_rn(y32 + bias[N]) (bias may be NULL).
 * On one GPU, zeroing y32, calling awq_linear_forward_rows once per shard
 * on the same stream and then awq_finish_rows gives the unsharded forward
 * up to the order of the fp32 sums; across GPUs the y32 of all shards would
 * be summed (an all-reduce) before awq_finish_rows. Argument errors as
 * awq_linear_forward (AWQ_ERR_INVALID_ARG also for ldx < K or ldx % 8 != 0).
 */
awq_status_t awq_linear_forward_rows(const void *x, int64_t ldx, const int32_t *qweight,
                                     const int32_t *qzeros, const void *scales, float *y32,
                                     int64_t M, int64_t K, int64_t N, int64_t group_size,
                                     awq_stream_t stream);
awq_status_t awq_finish_rows(const float *y32, const void *bias, void *y, int64_t M, int64_t N,
                             awq_stream_t stream);

/*
 * awq_dequant_gidx / awq_linear_forward_gidx -- the "g_idx" grouping variant
 * (act-order, as in the GPTQ quantisation tuple the Linear Layer Factory page
 * lists): the group of input row k is read from a table instead of being
 * k / group_size.
 *   W[k, n] = fp16_rn((q[k, n] - z[g_idx[k], n]) * scales[g_idx[k], n])
 *   y[m, n] = fp16_rn(sum_k x[m, k] * W[k, n] + bias[n])
 *   g_idx   int32 [K], every entry in [0, G)       (read)
 *   qzeros  int32 [G, N / 8], scales fp16 [G, N]   (read)
 * Other arguments and layouts as awq_dequant / awq_linear_forward, with the
 * number of groups G in place of group_size. Requires K > 0, N % 8 == 0,
 * G > 0 (AWQ_ERR_INVALID_ARG otherwise); the forward also needs K % 16 == 0
 * and N % 32 == 0. A table entry outside [0, G) cannot be seen before the
 * kernel runs: that row of W is written as zeros and the next
 * awq_last_device_status() returns AWQ_ERR_INVALID_ARG.
 * The forward dequantises W into a per-(device, stream) scratch area of
 * K x N fp16 (allocated on first use, like the split-K scratch) and runs the
 * prefill kernel's tcgen05 core on it (as awq_gemm_f16): it reads and writes
 * W once more than the grouped forward, so it is meant for prefill-sized M.
 */
awq_status_t awq_dequant_gidx(const int32_t *qweight, const int32_t *qzeros, const void *scales,
                              const int32_t *g_idx, void *W, int64_t K, int64_t N, int64_t G,
                              awq_stream_t stream);
awq_status_t awq_linear_forward_gidx(const void *x, const int32_t *qweight, const int32_t *qzeros,
                                     const void *scales, const int32_t *g_idx, const void *bias,
                                     void *y, int64_t M, int64_t K, int64_t N, int64_t G,
                                     awq_stream_t stream);

/*
 * Act-order g_idx layers on the grouped kernels. When every group of a g_idx
 * table holds the same number of rows g = K / G (the act-order tables of the
 * GPTQ tuple the Linear Layer Factory page lists), sorting the rows by group
 * turns the layer into an ordinary grouped one with group_size g and the same
 * qzeros and scales; the forward then reads x's columns in that order:
 *   y[m, n] = fp16_rn(sum_i x[m, perm[i]] * W[perm[i], n] + bias[n]),
 * the g_idx forward's sum with its terms reordered.
 *
 * awq_gidx_sort -- HOST pointers, no CUDA call: perm[i] = the original row of
 *   sorted row i, rows of each group in their original order (stable).
 *   g_idx int32 [K] (read), perm int32 [K] (written). Returns
 *   AWQ_ERR_INVALID_ARG unless K > 0, G > 0, K % G == 0, every entry lies in
 *   [0, G) and every group holds exactly K / G rows.
 * awq_permute_rows -- qweight_sorted[i, :] = qweight[perm[i], :], on the
 *   device (once, when the layer is loaded). qweight, qweight_sorted int32
 *   [K, N / 8], perm int32 [K]; N % 32 == 0. A perm entry outside [0, K)
 *   writes a zero row and makes the next awq_last_device_status() return
 *   AWQ_ERR_INVALID_ARG.
 * awq_linear_forward_sorted -- the forward of such a layer: x's columns are
 *   gathered in perm order into a per-(device, stream) scratch area of M x K
 *   fp16 (allocated on first use), then awq_linear_forward runs on the sorted
 *   weights with group_size = K / G. Arguments as awq_linear_forward, plus
 *   perm (device, int32 [K]); K % 8 == 0. A perm entry outside [0, K) reads
 *   as a zero activation and is reported as above.
 */
awq_status_t awq_gidx_sort(const int32_t *g_idx, int64_t K, int64_t G, int32_t *perm);
awq_status_t awq_permute_rows(const int32_t *qweight, const int32_t *perm, int32_t *qweight_sorted,
                              int64_t K, int64_t N, awq_stream_t stream);
awq_status_t awq_linear_forward_sorted(const void *x, const int32_t *perm, const int32_t *qweight_sorted,
                                       const int32_t *qzeros, const void *scales, const void *bias,
                                       void *y, int64_t M, int64_t K, int64_t N, int64_t group_size,
                                       awq_stream_t stream);

/*
 * awq_pack -- packs 4-bit codes into the layer's int32 format, the inverse of
 * the unpacking every forward call does (I/O Contract of the WQLinear page:
 * eight 4-bit values per int32; the order is this library's reading):
 *   packed[r, j] = sum_i (codes[r, 8 j + i] & 0xF) << (4 i),   i = 0..7.
 *   codes   uint8 [rows, cols], one code per byte (read; only the low 4 bits
 *           of each byte are used)
 *   packed  int32 [rows, cols / 8]                     (written)
 * Serves qweight (rows = K, cols = N) and qzeros (rows = G). Requires
 * rows >= 0, cols > 0 and cols % 8 == 0 (AWQ_ERR_INVALID_ARG otherwise);
 * rows == 0 is a no-op (pointers may be NULL then); both base pointers
 * 16-byte aligned (AWQ_ERR_MISALIGNED).
 */
awq_status_t awq_pack(const uint8_t *codes, int32_t *packed, int64_t rows, int64_t cols,
                      awq_stream_t stream);

/*
 * awq_quantize_rtn -- round-to-nearest quantisation of an fp16 weight with
 * given per-group scales and zero points, packed; the inverse of the
 * dequantisation W = (q - z) * s (Overview of the WQLinear page: group-wise
 * scaling):
 *   q[k, n] = clamp(round_half_even(W[k, n] / s[k / g, n]) + z[k / g, n], 0, 15)
 *   W       fp16 [K, N]                   (read)
 *   scales  fp16 [G, N], qzeros int32 [G, N / 8]   (read)
 *   qweight int32 [K, N / 8]              (written)
 * The quotient of two fp16 values is rounded as if exact (it is formed in
 * fp32, which decides every rounding the same way); a NaN quotient (0 / 0)
 * counts as 0, an infinite one clamps. For any normal nonzero scale,
 * awq_quantize_rtn(awq_dequant(q)) returns q. Shape and pointer rules as
 * awq_dequant.
 */
awq_status_t awq_quantize_rtn(const void *W, const void *scales, const int32_t *qzeros,
                              int32_t *qweight, int64_t K, int64_t N, int64_t group_size,
                              awq_stream_t stream);

/*
 * awq_gemm_f16 -- y[M, N] = fp16_rn(x[M, K] . W[K, N] + bias[N]) for an
 * already dequantised fp16 W (row-major [K, N], e.g. from awq_dequant), on the
 * same tcgen05 tensor-core pipeline as the prefill path of awq_linear_forward
 * but without its dequant stage. It checks that pipeline on its own (against
 * a library GEMM) and serves callers that keep W in fp16.
 *   x fp16 [M, K], W fp16 [K, N], bias fp16 [N] or NULL, y fp16 [M, N].
 * Requires K % 16 == 0 and N % 32 == 0 (AWQ_ERR_INVALID_ARG otherwise);
 * pointer and M rules as awq_linear_forward.
 */
awq_status_t awq_gemm_f16(const void *x, const void *W, const void *bias, void *y, int64_t M,
                          int64_t K, int64_t N, awq_stream_t stream);

/*
 * awq_linear_forward_decode_noalloc -- the same forward as awq_linear_forward,
 * computed by the same decode kernel, for callers that must not have device
 * memory allocated on their behalf. (The page has no counterpart of this
 * call: it exists for how the library is embedded, not for the method.)
 *
 * Who needs it: a serving process that plans all of its device memory up
 * front and may not allocate on the request path (a cudaMalloc there can
 * stall the device and fragment memory that was budgeted to the last byte),
 * and frameworks whose own caching allocator owns the GPU, where a hidden
 * allocation is not accounted for and can fail once the framework has
 * reserved nearly all of HBM. awq_linear_forward allocates a split-K scratch
 * area on first use; this call never allocates. Its scratch is one array
 * compiled into the library (5,275,648 bytes on every GPU that loads the
 * library, held until the process exits).
 *
 * Arguments, layouts and result: as awq_linear_forward. It serves only
 * shapes the decode kernel takes with at most 16 rows of x (1 <= M <= 16,
 * K % 64 == 0, N % 32 == 0, group_size % 16 == 0 after the -1 rule; else
 * AWQ_ERR_INVALID_ARG) and at
 * most 8192 column tiles of 256 (N <= 2,097,152; else AWQ_ERR_TOO_LARGE,
 * returned before anything is enqueued). It uses at most 160 CTAs.
 *
 * The first call on a device looks up the array's device address and sets
 * the kernel's launch attributes for that device; make that first call
 * before any stream capture. Every call shares the one array and finds it as
 * the previous call left it: each call clears the counters it needs
 * (cudaMemsetAsync on `stream`), so calls ordered on the GPU are safe, and
 * calls that overlap on the GPU (different streams, no ordering) race and
 * give wrong results. No cudaMalloc, cudaFree or allocating library routine
 * is called.
 */
awq_status_t awq_linear_forward_decode_noalloc(const void *x, const int32_t *qweight,
                                               const int32_t *qzeros, const void *scales,
                                               const void *bias, void *y, int64_t M,
                                               int64_t K, int64_t N, int64_t group_size,
                                               awq_stream_t stream);

/*
 * awq_reserve -- sizes, once, every scratch area the library keeps for
 * `stream` on the current device, so that later calls on that stream never
 * allocate and never synchronise. Without it the areas are created and grown
 * lazily: a call that needs more than its stream holds synchronises the
 * stream, frees the old area and allocates a larger one.
 *
 *   max_M, max_K, max_N  the largest M, K and N the stream's calls will use
 *                        (max_M >= 0, max_K > 0, max_N > 0)
 *   flags                0, or-ed with AWQ_RESERVE_SORTED (room for x's
 *                        columns in sorted order, max_M x max_K fp16:
 *                        awq_linear_forward_sorted) and AWQ_RESERVE_GIDX
 *                        (room for a whole dequantised layer, max_K x max_N
 *                        fp16: awq_linear_forward_gidx)
 *
 * It reserves the split-K partials of the decode and prefill kernels (sized
 * for the GPU's SM count, whatever the shape), the arrival counters of up to
 * ceil(max_N / 256) column tiles and, when max_M reaches the
 * dequantise-then-GEMM crossover (M >= 6144), that path's fp16 weight window.
 * This call itself allocates and synchronises `stream`: make it at set-up,
 * before any stream capture. Afterwards the stream's areas are fixed: a
 * forward call (any path) that would need more returns AWQ_ERR_TOO_LARGE
 * before launching anything, instead of growing them. Calling awq_reserve
 * again with larger bounds grows the areas; awq_shutdown() drops every
 * reservation. Returns AWQ_ERR_INVALID_ARG for invalid bounds or flags,
 * AWQ_ERR_CUDA if an allocation failed.
 */
#define AWQ_RESERVE_SORTED 1u
#define AWQ_RESERVE_GIDX 2u
awq_status_t awq_reserve(int64_t max_M, int64_t max_K, int64_t max_N, unsigned flags,
                         awq_stream_t stream);

/* Static description of a status code. Never NULL. */
const char *awq_status_string(awq_status_t status);

/*
 * awq_last_device_status -- synchronises `stream`, then reads and clears the
 * current device's status word. Returns AWQ_OK, AWQ_ERR_TIMEOUT if a kernel's
 * bounded wait ran out since the last read, AWQ_ERR_INVALID_ARG if a g_idx
 * entry was outside [0, G), or AWQ_ERR_CUDA if a synchronisation or reset
 * failed.
 *
 * After a timeout: the kernel that gave up wrote no result, and it may have
 * left split-K arrival counters of its stream non-zero. Results of later
 * decode-path calls on that device are not to be trusted until this call
 * has returned AWQ_ERR_TIMEOUT: it then synchronises the whole device and
 * zeroes, in place, the counters of every stream's scratch area (the areas
 * stay allocated, so CUDA graphs captured earlier remain valid).
 */
awq_status_t awq_last_device_status(awq_stream_t stream);

/* Frees every scratch area the library allocated, on every device, and drops
 * the per-device values the library caches (symbol addresses, kernel
 * attributes). Call it only when no call of this library is in flight, and
 * after a cudaDeviceReset before the next call. Later calls set up again. */
void awq_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_GB300_H */
