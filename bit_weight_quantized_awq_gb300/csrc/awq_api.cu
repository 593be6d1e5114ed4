// awq_api.cu -- the C ABI (include/awq_gb300.h): argument checks, path
// choice, per-(device, stream) scratch and the device status word.
//
// The argument checks are the WQLinear page's construction rules (Predibase
// Lorax "AWQ WQLinear", Description, __init__ bullets): w_bit is 4 (implicit:
// the ABI has no other width), out_features = 8 x qweight columns so
// N % 8 == 0, group_size -1 means K, and K % group_size == 0. Where the page
// asserts, this layer returns a status instead; nothing aborts.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/awq_gb300.h"
#ifdef AWQ_FAULT_TEST
#include "../../include/awq_gb300_fault_test.h"
#endif
#include "awq_internal.h"

namespace awq {

// ---------------------------------------------------------------------------
// device status word: one per device that loads the library
// ---------------------------------------------------------------------------

__device__ unsigned int g_device_status = 0;

namespace {

std::mutex g_mutex;
// device -> (&g_device_status on it, cache generation it was looked up in)
std::map<int, std::pair<unsigned int *, unsigned>> g_status_addr;

struct ScratchEntry {
    float *partials = nullptr;
    size_t partial_floats = 0;
    unsigned int *counters = nullptr;
    size_t n_counters = 0;
    void *w16 = nullptr;           // dequantised weights of the g_idx forward
    size_t w16_bytes = 0;
    void *xs = nullptr;            // activations in sorted row order (act-order forward)
    size_t xs_bytes = 0;
    bool reserved = false;         // sized by awq_reserve: never grows afterwards
};

// set when a call needed more scratch than its stream's reservation
thread_local bool t_over_reservation = false;
std::map<std::pair<int, cudaStream_t>, ScratchEntry> g_scratch;

} // namespace

unsigned int *device_status_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    const unsigned gen = cache_generation();
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_status_addr.find(dev);
    if (it != g_status_addr.end() && it->second.second == gen) return it->second.first;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return nullptr;
    g_status_addr[dev] = std::make_pair(static_cast<unsigned int *>(addr), gen);
    return static_cast<unsigned int *>(addr);
}

bool get_scratch(cudaStream_t stream, size_t partial_floats, size_t n_counters, Scratch *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchEntry &e = g_scratch[std::make_pair(dev, stream)];
    if (e.reserved && (e.partial_floats < partial_floats || e.n_counters < n_counters)) {
        t_over_reservation = true;
        return false;
    }
    if (e.partial_floats < partial_floats) {
        // the old area may still be read by work queued on this stream
        if (e.partials) {
            cudaStreamSynchronize(stream);
            cudaFree(e.partials);
            e.partials = nullptr;
            e.partial_floats = 0;
        }
        size_t want = partial_floats + partial_floats / 2;
        if (cudaMalloc(&e.partials, want * sizeof(float)) != cudaSuccess) {
            e.partials = nullptr;
            return false;
        }
        e.partial_floats = want;
    }
    if (e.n_counters < n_counters) {
        if (e.counters) {
            cudaStreamSynchronize(stream);
            cudaFree(e.counters);
            e.counters = nullptr;
            e.n_counters = 0;
        }
        size_t want = n_counters + n_counters / 2 + 64;
        if (cudaMalloc(&e.counters, want * sizeof(unsigned int)) != cudaSuccess) {
            e.counters = nullptr;
            return false;
        }
        // counters start at zero; every kernel leaves them at zero again
        if (cudaMemsetAsync(e.counters, 0, want * sizeof(unsigned int), stream) != cudaSuccess)
            return false;
        e.n_counters = want;
    }
    out->partials = e.partials;
    out->partial_floats = e.partial_floats;
    out->counters = e.counters;
    out->n_counters = e.n_counters;
    return true;
}

namespace {

// Grows one byte area of this (device, stream)'s scratch to at least `bytes`.
bool grow_area(cudaStream_t stream, size_t bytes, void *ScratchEntry::*ptr, size_t ScratchEntry::*cap,
               void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchEntry &e = g_scratch[std::make_pair(dev, stream)];
    if (e.reserved && e.*cap < bytes) {
        t_over_reservation = true;
        return false;
    }
    if (e.*cap < bytes) {
        // the old area may still be read by work queued on this stream
        if (e.*ptr) {
            cudaStreamSynchronize(stream);
            cudaFree(e.*ptr);
            e.*ptr = nullptr;
            e.*cap = 0;
        }
        if (cudaMalloc(&(e.*ptr), bytes) != cudaSuccess) {
            e.*ptr = nullptr;
            return false;
        }
        e.*cap = bytes;
    }
    *out = e.*ptr;
    return true;
}

} // namespace

bool scratch_over_reservation() { return t_over_reservation; }
void clear_scratch_over_reservation() { t_over_reservation = false; }

bool get_w16_scratch(cudaStream_t stream, size_t bytes, void **out)
{
    return grow_area(stream, bytes, &ScratchEntry::w16, &ScratchEntry::w16_bytes, out);
}

bool get_xs_scratch(cudaStream_t stream, size_t bytes, void **out)
{
    return grow_area(stream, bytes, &ScratchEntry::xs, &ScratchEntry::xs_bytes, out);
}

// Zeroes, in place, the split-K arrival counters of every scratch area on
// this device (a kernel whose bounded wait ran out leaves some non-zero). The
// caller has synchronised the device, so no queued kernel still uses them.
// The allocations stay where they are: CUDA graphs captured earlier hold
// these pointers and remain valid.
static cudaError_t reset_scratch_counters(int dev)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    cudaError_t first = cudaSuccess;
    for (auto &kv : g_scratch) {
        if (kv.first.first != dev || !kv.second.counters) continue;
        const cudaError_t e = cudaMemset(kv.second.counters, 0, kv.second.n_counters * sizeof(unsigned int));
        if (first == cudaSuccess) first = e;
    }
    const cudaError_t e = cudaDeviceSynchronize();
    return first != cudaSuccess ? first : e;
}

std::atomic<unsigned> g_cache_generation{1};

#ifdef AWQ_FAULT_TEST
std::atomic<int> g_fault_injection{0};
int fault_injection() { return g_fault_injection.load(std::memory_order_acquire); }
#endif

unsigned cache_generation() { return g_cache_generation.load(std::memory_order_acquire); }

} // namespace awq

using awq::Problem;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Status of a call whose launches returned `e`: a scratch need beyond the
// stream's reservation is AWQ_ERR_TOO_LARGE, any other failure AWQ_ERR_CUDA.
awq_status_t launch_status(cudaError_t e)
{
    if (e == cudaSuccess) return AWQ_OK;
    if (awq::scratch_over_reservation()) {
        awq::clear_scratch_over_reservation();
        return AWQ_ERR_TOO_LARGE;
    }
    return AWQ_ERR_CUDA;
}

// The WQLinear page's shape rules; fills the resolved group size.
awq_status_t check_shape(int64_t K, int64_t N, int64_t group_size, int64_t *g_out)
{
    if (K <= 0 || N <= 0) return AWQ_ERR_INVALID_ARG;
    if (N % 8 != 0) return AWQ_ERR_INVALID_ARG;
    if (group_size == 0 || group_size < -1) return AWQ_ERR_INVALID_ARG;
    const int64_t g = (group_size == -1) ? K : group_size;
    if (K % g != 0) return AWQ_ERR_INVALID_ARG;
    *g_out = g;
    return AWQ_OK;
}

bool path_fits(const Problem &p, awq_path_t path)
{
    switch (path) {
    case AWQ_PATH_GENERIC: return true;
    case AWQ_PATH_DECODE: return awq::decode_supported(p.M, p.K, p.N, p.g);
    case AWQ_PATH_PREFILL: return awq::prefill_supported(p.M, p.K, p.N, p.g);
    case AWQ_PATH_DEQUANT_GEMM: return awq::prefill_supported(p.M, p.K, p.N, p.g);
    default: return false;
    }
}

// Largest M served by the decode kernel when both fast paths fit.
constexpr int64_t kDecodeMaxM = 32;
// Dequantising the weights once and running the plain tcgen05 GEMM beats
// the fused kernel (which dequantises every weight tile once per 256-token
// tile) only for long runs of tokens: at M = 8192 by 1.03-1.08x on the 7B
// and 70B shapes with K <= 11008, while at M = 2048 the fused kernel is
// 1.1-1.25x faster, and at K = 28672 it wins at M = 8192 too (the fp16
// weights, 3.6x the packed bytes, no longer stay in L2): measured rule
// M >= 6144 and K <= 16384.
constexpr int64_t kDequantGemmMinM = 6144;
constexpr int64_t kDequantGemmMaxK = 16384;

bool dequant_gemm_pays(const Problem &p) { return p.M >= kDequantGemmMinM && p.K <= kDequantGemmMaxK; }

awq_path_t auto_path(const Problem &p)
{
    if (p.M <= kDecodeMaxM && awq::decode_supported(p.M, p.K, p.N, p.g)) return AWQ_PATH_DECODE;
    if (awq::prefill_supported(p.M, p.K, p.N, p.g))
        return dequant_gemm_pays(p) ? AWQ_PATH_DEQUANT_GEMM : AWQ_PATH_PREFILL;
    if (awq::decode_supported(p.M, p.K, p.N, p.g)) return AWQ_PATH_DECODE;
    return AWQ_PATH_GENERIC;
}

} // namespace

extern "C" {

const char *awq_status_string(awq_status_t status)
{
    switch (status) {
    case AWQ_OK: return "AWQ_OK";
    case AWQ_ERR_INVALID_ARG: return "AWQ_ERR_INVALID_ARG: shape rule violated, NULL pointer or M < 0";
    case AWQ_ERR_MISALIGNED: return "AWQ_ERR_MISALIGNED: a base pointer is not 16-byte aligned";
    case AWQ_ERR_CUDA: return "AWQ_ERR_CUDA: a CUDA call or kernel launch failed";
    case AWQ_ERR_TIMEOUT: return "AWQ_ERR_TIMEOUT: a kernel's bounded wait ran out";
    case AWQ_ERR_TOO_LARGE:
        return "AWQ_ERR_TOO_LARGE: shape exceeds the fixed scratch of the allocation-free entry point";
    default: return "AWQ: unknown status";
    }
}

int awq_path_supported(int64_t M, int64_t K, int64_t N, int64_t group_size, awq_path_t path)
{
    int64_t g = 0;
    if (M < 0 || check_shape(K, N, group_size, &g) != AWQ_OK) return 0;
    Problem p{};
    p.M = M; p.K = K; p.N = N; p.g = g; p.G = K / g;
    return path_fits(p, path) ? 1 : 0;
}

int awq_select_path(int64_t M, int64_t K, int64_t N, int64_t group_size)
{
    int64_t g = 0;
    if (M < 0 || check_shape(K, N, group_size, &g) != AWQ_OK) return -1;
    Problem p{};
    p.M = M; p.K = K; p.N = N; p.g = g; p.G = K / g;
    return (int)auto_path(p);
}

int awq_decode_tile_columns(int64_t M, int64_t K, int64_t N, int64_t group_size)
{
    int64_t g = 0;
    if (M < 0 || check_shape(K, N, group_size, &g) != AWQ_OK) return -1;
    return awq::decode_tile_columns(M, K, N, g);
}

int awq_forward_launches(int64_t M, int64_t K, int64_t N, int64_t group_size, awq_path_t path)
{
    int64_t g = 0;
    if (M < 0 || check_shape(K, N, group_size, &g) != AWQ_OK) return -1;
    if (M == 0) return 0;
    Problem p{};
    p.M = M; p.K = K; p.N = N; p.g = g; p.G = K / g;
    if (path == AWQ_PATH_AUTO) path = auto_path(p);
    else if (!path_fits(p, path)) return -1;
    if (path == AWQ_PATH_DECODE || path == AWQ_PATH_GENERIC) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return -1;
    if (path == AWQ_PATH_PREFILL) return awq::prefill_launches(M, K, N, sms);
    // AWQ_PATH_DEQUANT_GEMM: per window, the dequant kernel and the GEMM core
    const int64_t nc = awq::dequant_gemm_window(K, N);
    int n = 0;
    for (int64_t c0 = 0; c0 < N; c0 += nc)
        n += 1 + awq::prefill_launches(M, K, N - c0 < nc ? N - c0 : nc, sms);
    return n;
}

awq_status_t awq_linear_forward_path(const void *x, const int32_t *qweight, const int32_t *qzeros,
                                     const void *scales, const void *bias, void *y, int64_t M,
                                     int64_t K, int64_t N, int64_t group_size, awq_stream_t stream,
                                     awq_path_t path)
{
    int64_t g = 0;
    if (M < 0) return AWQ_ERR_INVALID_ARG;
    awq_status_t st = check_shape(K, N, group_size, &g);
    if (st != AWQ_OK) return st;
    if (path != AWQ_PATH_AUTO && path != AWQ_PATH_GENERIC && path != AWQ_PATH_DECODE &&
        path != AWQ_PATH_PREFILL && path != AWQ_PATH_DEQUANT_GEMM)
        return AWQ_ERR_INVALID_ARG;
    if (M == 0) return AWQ_OK;   // empty x and y may be NULL; nothing to do
    if (!x || !qweight || !qzeros || !scales || !y) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(qweight) || !aligned16(qzeros) || !aligned16(scales) ||
        !aligned16(y) || (bias && !aligned16(bias)))
        return AWQ_ERR_MISALIGNED;
    Problem p{x, qweight, qzeros, scales, bias, y, M, K, N, g, K / g};
    if (path != AWQ_PATH_AUTO && !path_fits(p, path)) return AWQ_ERR_INVALID_ARG;
    const awq_path_t use = (path == AWQ_PATH_AUTO) ? auto_path(p) : path;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (use) {
    case AWQ_PATH_DECODE: e = awq::launch_decode(p, s); break;
    case AWQ_PATH_PREFILL: e = awq::launch_prefill(p, s); break;
    case AWQ_PATH_DEQUANT_GEMM: e = awq::launch_dequant_gemm(p, s); break;
    default: e = awq::launch_generic(p, s); break;
    }
    return launch_status(e);
}

awq_status_t awq_linear_forward(const void *x, const int32_t *qweight, const int32_t *qzeros,
                                const void *scales, const void *bias, void *y, int64_t M,
                                int64_t K, int64_t N, int64_t group_size, awq_stream_t stream)
{
    return awq_linear_forward_path(x, qweight, qzeros, scales, bias, y, M, K, N, group_size,
                                   stream, AWQ_PATH_AUTO);
}

awq_status_t awq_dequant(const int32_t *qweight, const int32_t *qzeros, const void *scales,
                         void *W, int64_t K, int64_t N, int64_t group_size, awq_stream_t stream)
{
    int64_t g = 0;
    awq_status_t st = check_shape(K, N, group_size, &g);
    if (st != AWQ_OK) return st;
    if (!qweight || !qzeros || !scales || !W) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(qweight) || !aligned16(qzeros) || !aligned16(scales) || !aligned16(W))
        return AWQ_ERR_MISALIGNED;
    Problem p{nullptr, qweight, qzeros, scales, nullptr, nullptr, 0, K, N, g, K / g};
    cudaError_t e = awq::launch_dequant(p, W, reinterpret_cast<cudaStream_t>(stream));
    return launch_status(e);
}

awq_status_t awq_linear_forward_rows(const void *x, int64_t ldx, const int32_t *qweight,
                                     const int32_t *qzeros, const void *scales, float *y32,
                                     int64_t M, int64_t K, int64_t N, int64_t group_size,
                                     awq_stream_t stream)
{
    int64_t g = 0;
    if (M < 0) return AWQ_ERR_INVALID_ARG;
    awq_status_t st = check_shape(K, N, group_size, &g);
    if (st != AWQ_OK) return st;
    if (ldx < K || ldx % 8 != 0) return AWQ_ERR_INVALID_ARG;
    if (M == 0) return AWQ_OK;
    if (!x || !qweight || !qzeros || !scales || !y32) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(qweight) || !aligned16(qzeros) || !aligned16(scales) ||
        !aligned16(y32))
        return AWQ_ERR_MISALIGNED;
    Problem p{x, qweight, qzeros, scales, nullptr, nullptr, M, K, N, g, K / g};
    p.ldx = ldx;
    p.y32 = y32;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (auto_path(p)) {
    case AWQ_PATH_DECODE: e = awq::launch_decode(p, s); break;
    case AWQ_PATH_PREFILL: e = awq::launch_prefill(p, s); break;
    case AWQ_PATH_DEQUANT_GEMM: e = awq::launch_dequant_gemm(p, s); break;
    default: e = awq::launch_generic(p, s); break;
    }
    return launch_status(e);
}

awq_status_t awq_finish_rows(const float *y32, const void *bias, void *y, int64_t M, int64_t N,
                             awq_stream_t stream)
{
    if (M < 0 || N <= 0 || N % 8 != 0) return AWQ_ERR_INVALID_ARG;
    if (M == 0) return AWQ_OK;
    if (!y32 || !y) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(y32) || !aligned16(y) || (bias && !aligned16(bias))) return AWQ_ERR_MISALIGNED;
    cudaError_t e = awq::launch_finish_rows(y32, bias, y, M, N, reinterpret_cast<cudaStream_t>(stream));
    return launch_status(e);
}

awq_status_t awq_dequant_gidx(const int32_t *qweight, const int32_t *qzeros, const void *scales,
                              const int32_t *g_idx, void *W, int64_t K, int64_t N, int64_t G,
                              awq_stream_t stream)
{
    if (K <= 0 || N <= 0 || N % 8 != 0 || G <= 0) return AWQ_ERR_INVALID_ARG;
    if (!qweight || !qzeros || !scales || !g_idx || !W) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(qweight) || !aligned16(qzeros) || !aligned16(scales) || !aligned16(g_idx) ||
        !aligned16(W))
        return AWQ_ERR_MISALIGNED;
    Problem p{nullptr, qweight, qzeros, scales, nullptr, nullptr, 0, K, N, 0, G};
    cudaError_t e = awq::launch_dequant_gidx(p, g_idx, W, reinterpret_cast<cudaStream_t>(stream));
    return launch_status(e);
}

awq_status_t awq_linear_forward_gidx(const void *x, const int32_t *qweight, const int32_t *qzeros,
                                     const void *scales, const int32_t *g_idx, const void *bias,
                                     void *y, int64_t M, int64_t K, int64_t N, int64_t G,
                                     awq_stream_t stream)
{
    if (M < 0 || K <= 0 || N <= 0 || N % 8 != 0 || G <= 0) return AWQ_ERR_INVALID_ARG;
    if (!awq::prefill_supported(M > 0 ? M : 1, K, N, 16)) return AWQ_ERR_INVALID_ARG;
    if (M == 0) return AWQ_OK;
    if (!x || !qweight || !qzeros || !scales || !g_idx || !y) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(qweight) || !aligned16(qzeros) || !aligned16(scales) ||
        !aligned16(g_idx) || !aligned16(y) || (bias && !aligned16(bias)))
        return AWQ_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *w16 = nullptr;
    if (!awq::get_w16_scratch(s, (size_t)K * (size_t)N * 2, &w16)) return launch_status(cudaErrorMemoryAllocation);
    Problem pw{nullptr, qweight, qzeros, scales, nullptr, nullptr, 0, K, N, 0, G};
    cudaError_t e = awq::launch_dequant_gidx(pw, g_idx, w16, s);
    if (e == cudaSuccess) {
        Problem pg{x, nullptr, nullptr, nullptr, bias, y, M, K, N, K, 1};
        e = awq::launch_gemm_f16(pg, w16, s);
    }
    return launch_status(e);
}

awq_status_t awq_gidx_sort(const int32_t *g_idx, int64_t K, int64_t G, int32_t *perm)
{
    if (K <= 0 || G <= 0 || K % G != 0 || K > (int64_t(1) << 30) || !g_idx || !perm)
        return AWQ_ERR_INVALID_ARG;
    const int64_t g = K / G;
    std::vector<int64_t> next((size_t)G, 0);
    for (int64_t k = 0; k < K; ++k) {
        const int64_t gi = g_idx[k];
        if (gi < 0 || gi >= G || next[(size_t)gi] == g) return AWQ_ERR_INVALID_ARG;
        ++next[(size_t)gi];
    }
    // every group holds exactly g rows: sorted row gi * g + j is the j-th
    // row of group gi in the original order (a stable counting sort)
    for (int64_t gi = 0; gi < G; ++gi) next[(size_t)gi] = gi * g;
    for (int64_t k = 0; k < K; ++k) perm[next[(size_t)g_idx[k]]++] = (int32_t)k;
    return AWQ_OK;
}

awq_status_t awq_permute_rows(const int32_t *qweight, const int32_t *perm, int32_t *qweight_sorted,
                              int64_t K, int64_t N, awq_stream_t stream)
{
    if (K <= 0 || N <= 0 || N % 32 != 0 || K > (int64_t(1) << 30)) return AWQ_ERR_INVALID_ARG;
    if (!qweight || !perm || !qweight_sorted) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(qweight) || !aligned16(perm) || !aligned16(qweight_sorted)) return AWQ_ERR_MISALIGNED;
    cudaError_t e = awq::launch_gather_rows(qweight, perm, qweight_sorted, K, N / 8,
                                            reinterpret_cast<cudaStream_t>(stream));
    return launch_status(e);
}

awq_status_t awq_linear_forward_sorted(const void *x, const int32_t *perm, const int32_t *qweight_sorted,
                                       const int32_t *qzeros, const void *scales, const void *bias,
                                       void *y, int64_t M, int64_t K, int64_t N, int64_t group_size,
                                       awq_stream_t stream)
{
    int64_t g = 0;
    if (M < 0) return AWQ_ERR_INVALID_ARG;
    awq_status_t st = check_shape(K, N, group_size, &g);
    if (st != AWQ_OK) return st;
    if (K % 8 != 0) return AWQ_ERR_INVALID_ARG;
    if (M == 0) return AWQ_OK;
    if (!x || !perm || !qweight_sorted || !qzeros || !scales || !y) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(perm) || !aligned16(qweight_sorted) || !aligned16(qzeros) ||
        !aligned16(scales) || !aligned16(y) || (bias && !aligned16(bias)))
        return AWQ_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    Problem p{x, qweight_sorted, qzeros, scales, bias, y, M, K, N, g, K / g};
    if (auto_path(p) == AWQ_PATH_DEQUANT_GEMM) {
        // the weights are dequantised anyway: put their rows back in the
        // original order while doing so, and leave x as it is
        p.row_perm = perm;
        return launch_status(awq::launch_dequant_gemm(p, s));
    }
    void *xs = nullptr;
    if (!awq::get_xs_scratch(s, (size_t)M * (size_t)K * 2, &xs)) return launch_status(cudaErrorMemoryAllocation);
    if (awq::launch_gather_cols(x, K, perm, xs, M, K, s) != cudaSuccess) return AWQ_ERR_CUDA;
    return awq_linear_forward_path(xs, qweight_sorted, qzeros, scales, bias, y, M, K, N, group_size, stream,
                                   AWQ_PATH_AUTO);
}

awq_status_t awq_pack(const uint8_t *codes, int32_t *packed, int64_t rows, int64_t cols,
                      awq_stream_t stream)
{
    if (rows < 0 || cols <= 0 || cols % 8 != 0) return AWQ_ERR_INVALID_ARG;
    if (rows == 0) return AWQ_OK;
    if (!codes || !packed) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(codes) || !aligned16(packed)) return AWQ_ERR_MISALIGNED;
    cudaError_t e = awq::launch_pack(codes, packed, rows, cols, reinterpret_cast<cudaStream_t>(stream));
    return launch_status(e);
}

awq_status_t awq_quantize_rtn(const void *W, const void *scales, const int32_t *qzeros,
                              int32_t *qweight, int64_t K, int64_t N, int64_t group_size,
                              awq_stream_t stream)
{
    int64_t g = 0;
    awq_status_t st = check_shape(K, N, group_size, &g);
    if (st != AWQ_OK) return st;
    if (!W || !scales || !qzeros || !qweight) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(scales) || !aligned16(qzeros) || !aligned16(qweight))
        return AWQ_ERR_MISALIGNED;
    Problem p{nullptr, nullptr, qzeros, scales, nullptr, nullptr, 0, K, N, g, K / g};
    cudaError_t e = awq::launch_quantize(p, W, qweight, reinterpret_cast<cudaStream_t>(stream));
    return launch_status(e);
}

awq_status_t awq_gemm_f16(const void *x, const void *W, const void *bias, void *y, int64_t M,
                          int64_t K, int64_t N, awq_stream_t stream)
{
    if (M < 0 || K <= 0 || N <= 0) return AWQ_ERR_INVALID_ARG;
    if (!awq::prefill_supported(M > 0 ? M : 1, K, N, 16)) return AWQ_ERR_INVALID_ARG;
    if (M == 0) return AWQ_OK;
    if (!x || !W || !y) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W) || !aligned16(y) || (bias && !aligned16(bias)))
        return AWQ_ERR_MISALIGNED;
    Problem p{x, nullptr, nullptr, nullptr, bias, y, M, K, N, K, 1};
    cudaError_t e = awq::launch_gemm_f16(p, W, reinterpret_cast<cudaStream_t>(stream));
    return launch_status(e);
}

awq_status_t awq_reserve(int64_t max_M, int64_t max_K, int64_t max_N, unsigned flags, awq_stream_t stream)
{
    if (max_M < 0 || max_K <= 0 || max_N <= 0 || (flags & ~3u) != 0) return AWQ_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return AWQ_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    {
        // a stream reserved before may be reserved again (larger): lift the
        // lock for the growth below
        std::lock_guard<std::mutex> lock(awq::g_mutex);
        awq::g_scratch[std::make_pair(dev, s)].reserved = false;
    }
    const size_t partials = std::max(awq::decode_partial_floats_max(sms), awq::prefill_partial_floats_max(sms));
    const size_t tiles = (size_t)((max_N + 255) / 256);
    awq::Scratch sc{};
    bool ok = awq::get_scratch(s, partials, tiles, &sc);
    void *area = nullptr;
    if (ok && max_M >= kDequantGemmMinM) {
        // dequantise-then-GEMM windows: K x (a multiple of 256 columns within
        // 256 MiB of fp16, or all of N), for every K up to max_K
        const size_t window = (size_t)max_K * (size_t)awq::dequant_gemm_window(max_K, max_N) * 2;
        const size_t bound = std::min((size_t)max_K * (size_t)max_N * 2,
                                      std::max((size_t)256 << 20, (size_t)512 * (size_t)max_K));
        ok = awq::get_w16_scratch(s, std::max(window, bound), &area);
    }
    if (ok && (flags & AWQ_RESERVE_GIDX)) {
        size_t need = (size_t)max_K * (size_t)max_N * 2;   // the whole layer, dequantised
        size_t have = 0;
        {
            std::lock_guard<std::mutex> lock(awq::g_mutex);
            have = awq::g_scratch[std::make_pair(dev, s)].w16_bytes;
        }
        ok = awq::get_w16_scratch(s, std::max(need, have), &area);
    }
    if (ok && (flags & AWQ_RESERVE_SORTED)) ok = awq::get_xs_scratch(s, (size_t)max_M * (size_t)max_K * 2, &area);
    if (!ok) return AWQ_ERR_CUDA;
    // growth above may have queued zeroing work: let it finish, then pin
    if (cudaStreamSynchronize(s) != cudaSuccess) return AWQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(awq::g_mutex);
    awq::g_scratch[std::make_pair(dev, s)].reserved = true;
    return AWQ_OK;
}

awq_status_t awq_last_device_status(awq_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return AWQ_ERR_CUDA;
    unsigned int *addr = awq::device_status_word();
    if (!addr) return AWQ_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, addr, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return AWQ_ERR_CUDA;
    if (word == 0) return AWQ_OK;
    const unsigned int zero = 0;
    if (cudaMemcpy(addr, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return AWQ_ERR_CUDA;
    if (word & awq::kStatusTimeout) {
        // the kernel that gave up may have run on any stream of this device:
        // wait for all of them, then zero every stream's counters in place
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
            awq::reset_scratch_counters(dev) != cudaSuccess)
            return AWQ_ERR_CUDA;
        return AWQ_ERR_TIMEOUT;
    }
    if (word & awq::kStatusBadIndex) return AWQ_ERR_INVALID_ARG;
    return AWQ_ERR_CUDA;
}

#ifdef AWQ_FAULT_TEST
void awq_test_inject_fault(int on)
{
    awq::g_fault_injection.store(on ? 1 : 0, std::memory_order_release);
}
#endif

void awq_shutdown(void)
{
    std::lock_guard<std::mutex> lock(awq::g_mutex);
    int prev = 0;
    cudaGetDevice(&prev);
    for (auto &kv : awq::g_scratch) {
        cudaSetDevice(kv.first.first);
        if (kv.second.partials) cudaFree(kv.second.partials);
        if (kv.second.counters) cudaFree(kv.second.counters);
        if (kv.second.w16) cudaFree(kv.second.w16);
        if (kv.second.xs) cudaFree(kv.second.xs);
    }
    awq::g_scratch.clear();
    awq::g_status_addr.clear();
    // per-device lookups cached by the kernel launchers (symbol addresses,
    // function attributes) are redone on the next call: after a
    // cudaDeviceReset they would be stale
    awq::g_cache_generation.fetch_add(1, std::memory_order_acq_rel);
    cudaSetDevice(prev);
}

} // extern "C"
