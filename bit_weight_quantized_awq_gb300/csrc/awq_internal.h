// awq_internal.h -- host-side interface between the C-ABI layer (awq_api.cu)
// and the kernel translation units. Not installed; not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace awq {

// One validated forward/dequant problem. g is the resolved group size (the
// page's group_size -1 already replaced by K), G = K / g.
struct Problem {
    const void *x;          // fp16 [M, K]
    const int32_t *qweight; // int32 [K, N / 8]
    const int32_t *qzeros;  // int32 [G, N / 8]
    const void *scales;     // fp16 [G, N]
    const void *bias;       // fp16 [N] or nullptr
    void *y;                // fp16 [M, N]
    int64_t M, K, N, g, G;
    int64_t ldx = 0;        // elements between rows of x (0 = K): a K-slice of a wider x
    float *y32 = nullptr;   // if set: y32[M, N] += x . W in fp32 (no bias, no rounding),
                            // instead of writing y
    const int32_t *row_perm = nullptr;   // dequantise-then-GEMM only: weight row k is
                                         // row row_perm[k] of W (act-order layers)
};

// Per-(device, stream) scratch: fp32 split-K partials plus self-resetting
// per-tile arrival counters (zero between calls).
struct Scratch {
    float *partials;
    size_t partial_floats;
    unsigned int *counters;
    size_t n_counters;
};

// Bumped by awq_shutdown(): per-device values a launcher caches (symbol
// addresses, function attributes set once per device) are looked up again
// when the generation they were cached in is no longer current.
unsigned cache_generation();

#ifdef AWQ_FAULT_TEST
// Fault-test build only: when non-zero, the next decode and prefill launches
// tell CTA 0's TMA producer to issue nothing, so that the waits of that CTA's
// consumers on the stage barriers run out (see awq_gb300_fault_test.h).
int fault_injection();
#endif

// Returns the address of this device's status word (bit flags, see
// kStatusTimeout) for kernels to record device-side errors in.
unsigned int *device_status_word();
constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned int kStatusBadIndex = 2u;   // a group or row index out of range

// Scratch for `stream` on the current device, grown to at least the given
// sizes. Returns false if an allocation failed, or if the stream's scratch
// was reserved (awq_reserve) and is smaller than asked: a reserved area never
// grows (scratch_over_reservation() then reports true on this thread).
bool get_scratch(cudaStream_t stream, size_t partial_floats, size_t n_counters, Scratch *out);
bool scratch_over_reservation();
void clear_scratch_over_reservation();

// Largest split-K partial areas (floats) a decode / prefill launch on a GPU
// with `sms` SMs asks for, whatever the shape.
size_t decode_partial_floats_max(int sms);
size_t prefill_partial_floats_max(int sms);

// A buffer of at least `bytes` for `stream` on the current device (dequantised
// weights of the g_idx forward), grown on demand.
bool get_w16_scratch(cudaStream_t stream, size_t bytes, void **out);

// ---- kernel launchers (each returns the launch's cudaError_t) ----

cudaError_t launch_dequant(const Problem &p, void *W, cudaStream_t stream);

// Dequantisation of output columns c0 .. c0 + nc - 1 (multiples of 8) into a
// [K, nc] fp16 array.
cudaError_t launch_dequant_cols(const Problem &p, int64_t c0, int64_t nc, void *W, cudaStream_t stream);

// Large-M forward: the weights dequantised once per column window into a
// per-stream scratch area, then the tcgen05 fp16 GEMM core on each window.
cudaError_t launch_dequant_gemm(const Problem &p, cudaStream_t stream);

// Dequantisation with the group of row k taken from g_idx[k] (p.G groups);
// an index outside [0, G) writes zeros for that row and sets kStatusBadIndex.
cudaError_t launch_dequant_gidx(const Problem &p, const int32_t *g_idx, void *W, cudaStream_t stream);

// y[M, N] = fp16_rn(y32 + bias): the end of a row-parallel forward.
cudaError_t launch_finish_rows(const float *y32, const void *bias, void *y, int64_t M, int64_t N,
                               cudaStream_t stream);

// Packing of 4-bit codes (uint8, one per byte) into int32 words, and
// round-to-nearest quantisation of an fp16 W with the problem's scales and
// zero points into its qweight.
cudaError_t launch_pack(const uint8_t *codes, int32_t *packed, int64_t rows, int64_t cols,
                        cudaStream_t stream);
cudaError_t launch_quantize(const Problem &p, const void *W, int32_t *qweight, cudaStream_t stream);

cudaError_t launch_generic(const Problem &p, cudaStream_t stream);

// Decode path (small M). supported_* is host-only shape logic.
bool decode_supported(int64_t M, int64_t K, int64_t N, int64_t g);
// columns per decode tile for this shape (0 if the decode kernel cannot serve it)
int decode_tile_columns(int64_t M, int64_t K, int64_t N, int64_t g);
cudaError_t launch_decode(const Problem &p, cudaStream_t stream);

// Prefill path (large M, tcgen05).
bool prefill_supported(int64_t M, int64_t K, int64_t N, int64_t g);
cudaError_t launch_prefill(const Problem &p, cudaStream_t stream);

// The prefill kernel's tensor-core pipeline on an already dequantised fp16
// W [K, N] (no dequant stage): y = x . W + bias. Same shape rules as prefill.
// ldy: elements between rows of y (0 = N), so that a call can write a
// column window of a wider output.
cudaError_t launch_gemm_f16(const Problem &p, const void *w16, cudaStream_t stream, int64_t ldy = 0);
// kernels one prefill / GEMM-core launch enqueues on a GPU with `sms` SMs:
// the persistent kernel, plus sk_fixup_kernel when a tile is split along k
int prefill_launches(int64_t M, int64_t K, int64_t N, int sms);
// act-order layers: rows of packed weights / columns of x in sorted order
cudaError_t launch_gather_rows(const int32_t *src, const int32_t *perm, int32_t *dst, int64_t K,
                               int64_t words, cudaStream_t stream);
cudaError_t launch_gather_cols(const void *x, int64_t ldx, const int32_t *perm, void *xs, int64_t M,
                               int64_t K, cudaStream_t stream);
bool get_xs_scratch(cudaStream_t stream, size_t bytes, void **out);
// fp16 weight columns per window of the dequantise-then-GEMM path
int64_t dequant_gemm_window(int64_t K, int64_t N);

} // namespace awq
