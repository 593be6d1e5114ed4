// awq_pack.cu -- the step before the WQLinear forward: packing 4-bit codes
// into the layer's int32 format and round-to-nearest quantisation of an fp16
// weight with given per-group scales and zero points.
//
// Predibase Lorax "AWQ WQLinear" page: I/O Contract (qweight int32
// [in_features, out_features / 8] holding eight 4-bit values per int32;
// packed qzeros; per-group scales) and Overview (group-wise scaling). Packing
// is the inverse of the unpacking every forward kernel does (nibble i of
// int32 j of a row holds column 8j + i); quantisation inverts the
// dequantisation W = (q - z) * s:
//   q[k, n] = clamp(round_half_even(W[k, n] / s[k/g, n]) + z[k/g, n], 0, 15).
// The quotient is formed in fp32 as w * rcp(s), rcp correctly rounded, so it
// is within 2^-23 relative (2^-17 absolute up to magnitude 64) of the exact
// quotient. For two fp16 operands the exact quotient lies at least 2^-13 from
// any half-integer of magnitude up to 64 unless it is one (write w and s as
// integer significands times powers of two and bound the numerator of the
// difference), so rounding the fp32 value to the nearest integer decides as
// rounding the exact quotient would, except at exact halves; those are
// recognised exactly (h * s == w for the half-integer h next to the fp32
// value; the product is exact in fp32) and rounded to even. A NaN quotient
// (0 / 0) counts as 0; the quotient is clamped to [-64, 64] before rounding,
// which changes no result because the code is clamped to 0..15 afterwards.
//
// Both kernels are HBM-bound elementwise passes with coalesced 8- or 16-byte
// loads and 4-byte stores, grid a multiple of the SM count striding over the
// words.
#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {
namespace {

__global__ void __launch_bounds__(256)
pack_kernel(const uint2 *__restrict__ codes, uint32_t *__restrict__ packed, int64_t words)
{
    for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < words;
         w += (int64_t)gridDim.x * blockDim.x) {
        const uint2 c = __ldg(codes + w);   // columns 8j .. 8j+3 in c.x, 8j+4 .. 8j+7 in c.y
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v |= ((c.x >> (8 * i)) & 0xFu) << (4 * i);
            v |= ((c.y >> (8 * i)) & 0xFu) << (4 * (i + 4));
        }
        packed[w] = v;
    }
}

// One thread per (packed word, run of kRows consecutive rows). When the run
// lies in one group (always when kRows divides g), the group's eight scales,
// their reciprocals and the zero word are loaded once and the run's kRows
// 16-byte loads of W are all issued before any is used; otherwise the rows
// are taken one at a time, reloading at the group boundary.
constexpr int kRows = 8;

// Code of one weight: round_half_even(w / s) + z, clamped to 0..15, from the
// fp32 quotient w * rcp(s) (see the file comment for why it decides exactly).
__device__ __forceinline__ uint32_t code_of(float wf, float sf, float rcp, uint32_t z)
{
    float t = wf * rcp;
    // exact halves are recognised by h * s == w (exact in fp32: h has at
    // most 8 significant bits, s 11) and kept as they are
    const float h = floorf(t) + 0.5f;
    if (h * sf == wf) t = h;
    if (t != t) t = 0.f;   // NaN (0 / 0)
    t = fminf(fmaxf(t, -64.f), 64.f);
    int c = (int)rintf(t) + (int)z;
    c = c < 0 ? 0 : (c > 15 ? 15 : c);
    return (uint32_t)c;
}

__device__ __forceinline__ void load_group(const __half *scales, const uint32_t *qzeros, int64_t gi,
                                           int64_t words, int64_t j, float (&sf)[8], float (&rcp)[8],
                                           uint32_t &zw)
{
    __half s[8];
    *reinterpret_cast<uint4 *>(s) = __ldg(reinterpret_cast<const uint4 *>(scales + (gi * words + j) * 8));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        sf[i] = __half2float(s[i]);
        rcp[i] = __frcp_rn(sf[i]);
    }
    zw = __ldg(qzeros + gi * words + j);
}

__device__ __forceinline__ uint32_t quantize_word(const uint4 wraw, const float (&sf)[8], const float (&rcp)[8],
                                                  uint32_t zw)
{
    __half w[8];
    *reinterpret_cast<uint4 *>(w) = wraw;
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) v |= code_of(__half2float(w[i]), sf[i], rcp[i], nibble(zw, i)) << (4 * i);
    return v;
}

__global__ void __launch_bounds__(256)
quantize_kernel(const __half *__restrict__ W, const __half *__restrict__ scales,
                const uint32_t *__restrict__ qzeros, uint32_t *__restrict__ qweight,
                int64_t K, int64_t words, int64_t g)
{
    const int64_t runs = (K + kRows - 1) / kRows;
    const int64_t total = runs * words;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t run = idx / words;
        const int64_t j = idx - run * words;
        const int64_t k0 = run * kRows;
        float sf[8], rcp[8];
        uint32_t zw;
        if (k0 + kRows <= K && k0 / g == (k0 + kRows - 1) / g) {
            uint4 wv[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                wv[r] = __ldg(reinterpret_cast<const uint4 *>(W + ((k0 + r) * words + j) * 8));
            load_group(scales, qzeros, k0 / g, words, j, sf, rcp, zw);
#pragma unroll
            for (int r = 0; r < kRows; ++r) qweight[(k0 + r) * words + j] = quantize_word(wv[r], sf, rcp, zw);
            continue;
        }
        int64_t cur = -1;
        for (int r = 0; r < kRows && k0 + r < K; ++r) {
            const int64_t k = k0 + r;
            if (k / g != cur) {
                cur = k / g;
                load_group(scales, qzeros, cur, words, j, sf, rcp, zw);
            }
            const uint4 wraw = __ldg(reinterpret_cast<const uint4 *>(W + (k * words + j) * 8));
            qweight[k * words + j] = quantize_word(wraw, sf, rcp, zw);
        }
    }
}

int grid_for(int64_t items)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (items + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

} // namespace

cudaError_t launch_pack(const uint8_t *codes, int32_t *packed, int64_t rows, int64_t cols,
                        cudaStream_t stream)
{
    const int64_t words = rows * (cols / 8);
    if (words == 0) return cudaSuccess;
    pack_kernel<<<grid_for(words), 256, 0, stream>>>(reinterpret_cast<const uint2 *>(codes),
                                                     reinterpret_cast<uint32_t *>(packed), words);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const Problem &p, const void *W, int32_t *qweight, cudaStream_t stream)
{
    const int64_t words = p.N / 8;
    quantize_kernel<<<grid_for((p.K + kRows - 1) / kRows * words), 256, 0, stream>>>(
        static_cast<const __half *>(W), static_cast<const __half *>(p.scales),
        reinterpret_cast<const uint32_t *>(p.qzeros), reinterpret_cast<uint32_t *>(qweight), p.K,
        words, p.g);
    return cudaGetLastError();
}

} // namespace awq
