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
// The quotient is formed in fp32 with the correctly rounded division. For two
// fp16 operands it lies at least 2^-13 from any half integer of magnitude up
// to 64 unless it is one, while the fp32 rounding error there is at most
// 2^-18, so rounding the fp32 quotient to the nearest integer (ties to even)
// decides exactly as rounding the exact quotient would. A NaN quotient
// (0 / 0) counts as 0; the quotient is clamped to [-64, 64] before rounding,
// which changes no result because the code is clamped to 0..15 afterwards.
//
// Both kernels are HBM-bound elementwise passes: one thread per packed word,
// coalesced 8- or 16-byte loads and a 4-byte store, grid a multiple of the SM
// count striding over the words.
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

__global__ void __launch_bounds__(256)
quantize_kernel(const __half *__restrict__ W, const __half *__restrict__ scales,
                const uint32_t *__restrict__ qzeros, uint32_t *__restrict__ qweight,
                int64_t K, int64_t words, int64_t g)
{
    const int64_t total = K * words;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t k = idx / words;
        const int64_t j = idx - k * words;
        const int64_t gi = k / g;
        __half w[8], s[8];
        *reinterpret_cast<uint4 *>(w) = __ldg(reinterpret_cast<const uint4 *>(W + idx * 8));
        *reinterpret_cast<uint4 *>(s) = __ldg(reinterpret_cast<const uint4 *>(scales + (gi * words + j) * 8));
        const uint32_t zw = __ldg(qzeros + gi * words + j);
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float t = __fdiv_rn(__half2float(w[i]), __half2float(s[i]));
            if (t != t) t = 0.f;   // NaN
            t = fminf(fmaxf(t, -64.f), 64.f);
            int c = (int)rintf(t) + (int)nibble(zw, i);
            c = c < 0 ? 0 : (c > 15 ? 15 : c);
            v |= (uint32_t)c << (4 * i);
        }
        qweight[idx] = v;
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
    quantize_kernel<<<grid_for(p.K * words), 256, 0, stream>>>(
        static_cast<const __half *>(W), static_cast<const __half *>(p.scales),
        reinterpret_cast<const uint32_t *>(p.qzeros), reinterpret_cast<uint32_t *>(qweight), p.K,
        words, p.g);
    return cudaGetLastError();
}

} // namespace awq
