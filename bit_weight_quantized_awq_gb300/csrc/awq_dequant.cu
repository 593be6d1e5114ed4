// awq_dequant.cu -- the awq_dequant kernel: packed int4 weights -> fp16 W.
//
// Predibase Lorax "AWQ WQLinear" page, Description (__init__: per-group
// dequantisation; qweight packs eight 4-bit values per int32):
//   W[k, n] = fp16_rn((q[k, n] - z[k / g, n]) * scales[k / g, n]).
//
// HBM-bound elementwise work: per packed int32 read (4 B) it writes 8 fp16
// (16 B); scales and zero points are re-read by the g rows of a group and stay
// in L2. dequant_vec_kernel (rows of a multiple of four packed words): each
// thread takes four consecutive packed words of one row with one 16-byte
// load, their zero-point words with one 16-byte load and their 32 scales
// with four, converts them two weights per half2 instruction
// (dequant_word_h2), and stores 64 contiguous bytes; two such groups are in
// flight per thread before either is used. dequant_kernel takes one word per
// thread for any other width (N % 32 != 0). The grids are a multiple of the
// SM count and stride over the words.
#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {
namespace {

__global__ void __launch_bounds__(256)
dequant_kernel(const uint32_t *__restrict__ qweight, const uint32_t *__restrict__ qzeros,
               const __half *__restrict__ scales, __half *__restrict__ W,
               int64_t K, int64_t words, int64_t g, int64_t word0, int64_t wwords,
               const int32_t *__restrict__ row_out, unsigned int *status)
{
    // output: words word0 .. word0 + wwords - 1 of every row, as a [K, 8 wwords]
    // array; row k goes to row row_out[k] when a row order is given (the
    // sorted rows of an act-order layer put back in their original order)
    const int64_t total = K * wwords;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t k = idx / wwords;
        const int64_t jw = idx - k * wwords;
        const int64_t j = word0 + jw;
        int64_t dst = idx;
        if (row_out) {
            const int64_t r = __ldg(row_out + k);
            if (r < 0 || r >= K) {
                raise_status(status, kStatusBadIndex);
                continue;
            }
            dst = r * wwords + jw;
        }
        const int64_t gi = k / g;
        const uint32_t qw = __ldg(qweight + k * words + j);
        const uint32_t zw = __ldg(qzeros + gi * words + j);
        // 8 scales of columns 8j .. 8j+7: 16 bytes, 16-byte aligned
        const uint4 sraw = __ldg(reinterpret_cast<const uint4 *>(scales + (gi * words + j) * 8));
        __half s[8], w[8];
        *reinterpret_cast<uint4 *>(s) = sraw;
        dequant_word(qw, zw, s, w);
        *reinterpret_cast<uint4 *>(W + dst * 8) = *reinterpret_cast<const uint4 *>(w);
    }
}

// Four consecutive packed words per thread (window width and start multiples
// of four words): quads q = idx of the [K, wwords / 4] array of word quads.
__global__ void __launch_bounds__(256)
dequant_vec_kernel(const uint32_t *__restrict__ qweight, const uint32_t *__restrict__ qzeros,
                   const __half *__restrict__ scales, __half *__restrict__ W,
                   int64_t K, int64_t words, int64_t g, int64_t word0, int64_t wwords,
                   const int32_t *__restrict__ row_out, unsigned int *status)
{
    const int64_t wq = wwords / 4;        // quads per output row
    const int64_t total = K * wq;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t base = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; base < total; base += 2 * stride) {
        uint4 qv[2], zv[2], sv[2][4];
        int64_t dst[2];
        bool live[2];
        // issue every load of both quads before any arithmetic
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t idx = base + u * stride;
            live[u] = idx < total;
            if (!live[u]) continue;
            const int64_t k = idx / wq;
            const int64_t jq = idx - k * wq;
            const int64_t j = word0 + 4 * jq;     // first packed word of the quad
            dst[u] = idx;
            if (row_out) {
                const int64_t r = __ldg(row_out + k);
                if (r < 0 || r >= K) {
                    raise_status(status, kStatusBadIndex);
                    live[u] = false;
                    continue;
                }
                dst[u] = r * wq + jq;
            }
            const int64_t gi = k / g;
            qv[u] = __ldg(reinterpret_cast<const uint4 *>(qweight + k * words + j));
            zv[u] = __ldg(reinterpret_cast<const uint4 *>(qzeros + gi * words + j));
            const uint4 *sp = reinterpret_cast<const uint4 *>(scales + (gi * words + j) * 8);
#pragma unroll
            for (int w = 0; w < 4; ++w) sv[u][w] = __ldg(sp + w);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (!live[u]) continue;
            uint4 *out = reinterpret_cast<uint4 *>(W + dst[u] * 32);
            out[0] = dequant_word_h2(qv[u].x, zv[u].x, sv[u][0]);
            out[1] = dequant_word_h2(qv[u].y, zv[u].y, sv[u][1]);
            out[2] = dequant_word_h2(qv[u].z, zv[u].z, sv[u][2]);
            out[3] = dequant_word_h2(qv[u].w, zv[u].w, sv[u][3]);
        }
    }
}

// The same with the group of row k read from g_idx[k]: the "g_idx"
// (act-order) grouping, G groups of scales and zero points.
__global__ void __launch_bounds__(256)
dequant_gidx_kernel(const uint32_t *__restrict__ qweight, const uint32_t *__restrict__ qzeros,
                    const __half *__restrict__ scales, const int32_t *__restrict__ g_idx,
                    __half *__restrict__ W, int64_t K, int64_t words, int64_t G,
                    unsigned int *status)
{
    const int64_t total = K * words;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t k = idx / words;
        const int64_t j = idx - k * words;
        const int64_t gi = __ldg(g_idx + k);
        __half w[8];
        if (gi < 0 || gi >= G) {
            raise_status(status, kStatusBadIndex);
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = __ushort_as_half((unsigned short)0);
        } else {
            const uint32_t qw = __ldg(qweight + idx);
            const uint32_t zw = __ldg(qzeros + gi * words + j);
            __half s[8];
            *reinterpret_cast<uint4 *>(s) = __ldg(reinterpret_cast<const uint4 *>(scales + (gi * words + j) * 8));
            dequant_word(qw, zw, s, w);
        }
        *reinterpret_cast<uint4 *>(W + idx * 8) = *reinterpret_cast<const uint4 *>(w);
    }
}

} // namespace

cudaError_t launch_dequant_gidx(const Problem &p, const int32_t *g_idx, void *W, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t words = p.N / 8;
    const int64_t total = p.K * words;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    dequant_gidx_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        reinterpret_cast<const uint32_t *>(p.qweight), reinterpret_cast<const uint32_t *>(p.qzeros),
        static_cast<const __half *>(p.scales), g_idx, static_cast<__half *>(W), p.K, words, p.G,
        device_status_word());
    return cudaGetLastError();
}

cudaError_t launch_dequant_cols(const Problem &p, int64_t c0, int64_t nc, void *W, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t words = p.N / 8;
    const int threads = 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
    if (words % 4 == 0 && (c0 / 8) % 4 == 0 && (nc / 8) % 4 == 0) {
        // 16-byte rows of packed words: four words per thread, two quads in flight
        const int64_t quads = p.K * (nc / 32);
        int64_t blocks = (quads + 2 * threads - 1) / (2 * threads);
        if (blocks > cap) blocks = cap;
        if (blocks < 1) return cudaSuccess;
        dequant_vec_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
            reinterpret_cast<const uint32_t *>(p.qweight), reinterpret_cast<const uint32_t *>(p.qzeros),
            static_cast<const __half *>(p.scales), static_cast<__half *>(W), p.K, words, p.g, c0 / 8,
            nc / 8, p.row_perm, device_status_word());
        return cudaGetLastError();
    }
    const int64_t total = p.K * (nc / 8);
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    dequant_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        reinterpret_cast<const uint32_t *>(p.qweight), reinterpret_cast<const uint32_t *>(p.qzeros),
        static_cast<const __half *>(p.scales), static_cast<__half *>(W), p.K, words, p.g, c0 / 8, nc / 8,
        p.row_perm, device_status_word());
    return cudaGetLastError();
}

cudaError_t launch_dequant(const Problem &p, void *W, cudaStream_t stream)
{
    return launch_dequant_cols(p, 0, p.N, W, stream);
}

// Windows of at most this many bytes of fp16 weights bound the scratch.
constexpr int64_t kW16WindowBytes = 256ll << 20;

int64_t dequant_gemm_window(int64_t K, int64_t N)
{
    // window width: a multiple of 256 columns (one GEMM tile), or all of N
    int64_t nc = (kW16WindowBytes / (2 * K)) / 256 * 256;
    if (nc < 256) nc = 256;
    if (nc > N) nc = N;
    return nc;
}

cudaError_t launch_dequant_gemm(const Problem &p, cudaStream_t stream)
{
    const int64_t nc = dequant_gemm_window(p.K, p.N);
    void *w16 = nullptr;
    if (!get_w16_scratch(stream, (size_t)p.K * (size_t)nc * 2, &w16)) return cudaErrorMemoryAllocation;
    for (int64_t c0 = 0; c0 < p.N; c0 += nc) {
        const int64_t w = (p.N - c0 < nc) ? p.N - c0 : nc;
        cudaError_t e = launch_dequant_cols(p, c0, w, w16, stream);
        if (e != cudaSuccess) return e;
        Problem pg{p.x, nullptr, nullptr, nullptr,
                   p.bias ? static_cast<const __half *>(p.bias) + c0 : nullptr,
                   p.y ? static_cast<__half *>(p.y) + c0 : nullptr, p.M, p.K, w, p.K, 1};
        pg.ldx = p.ldx;
        pg.y32 = p.y32 ? p.y32 + c0 : nullptr;
        e = launch_gemm_f16(pg, w16, stream, p.N);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

__global__ void __launch_bounds__(256)
finish_rows_kernel(const float4 *__restrict__ y32, const __half *__restrict__ bias,
                   uint2 *__restrict__ y, int64_t quads, int64_t n_quads)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < quads;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = __ldg(y32 + i);
        float b[4] = {0.f, 0.f, 0.f, 0.f};
        if (bias) {
            const int64_t c = (i % n_quads) * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e) b[e] = __half2float(bias[c + e]);
        }
        __align__(8) __half out[4] = {__float2half_rn(v.x + b[0]), __float2half_rn(v.y + b[1]),
                                      __float2half_rn(v.z + b[2]), __float2half_rn(v.w + b[3])};
        y[i] = *reinterpret_cast<const uint2 *>(out);
    }
}

cudaError_t launch_finish_rows(const float *y32, const void *bias, void *y, int64_t M, int64_t N,
                               cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t quads = M * N / 4;
    int64_t blocks = (quads + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    finish_rows_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        reinterpret_cast<const float4 *>(y32), static_cast<const __half *>(bias), static_cast<uint2 *>(y),
        quads, N / 4);
    return cudaGetLastError();
}

} // namespace awq
