// awq_generic.cu -- the generic forward kernel: serves every shape the
// WQLinear page admits (any N % 8 == 0, any group size dividing K, any
// pointer pitch), including the ones the tensor-core paths do not take
// (N = 8, K not a multiple of 16, odd group sizes).
//
// Predibase Lorax "AWQ WQLinear" page, Description, forward steps 2-3:
//   y[m, n] = fp16_rn( sum_k x[m, k] * W[k, n] + bias[n] ),
//   W[k, n] = fp16_rn((q - z) * s) per group, accumulated in fp32.
//
// With Problem::y32 set it adds the fp32 sums into y32 instead (no bias, no
// rounding): one piece of a row-parallel forward.
//
// One thread owns one packed column word j (8 outputs) for up to kRows rows
// of x: it dequantises each packed word once and feeds kRows x 8 fp32 FMAs.
// Adjacent threads take adjacent words, so the qweight loads are coalesced.
// This is the correctness fallback, not a fast path.
#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kRows = 4;

__global__ void __launch_bounds__(128)
generic_forward_kernel(const __half *__restrict__ x, const uint32_t *__restrict__ qweight,
                       const uint32_t *__restrict__ qzeros, const __half *__restrict__ scales,
                       const __half *__restrict__ bias, __half *__restrict__ y,
                       float *__restrict__ y32, int64_t M, int64_t K, int64_t ldx, int64_t words,
                       int64_t g)
{
    const int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int64_t m0 = (int64_t)blockIdx.y * kRows;
    if (j >= words) return;
    const int64_t N = words * 8;
    float acc[kRows][8];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[r][i] = 0.f;

    __half s[8];
    uint32_t zw = 0;
    int64_t cur_group = -1;
    for (int64_t k = 0; k < K; ++k) {
        const int64_t gi = k / g;
        if (gi != cur_group) {
            cur_group = gi;
            zw = __ldg(qzeros + gi * words + j);
#pragma unroll
            for (int i = 0; i < 8; ++i) s[i] = scales[gi * N + 8 * j + i];
        }
        __half w[8];
        dequant_word(__ldg(qweight + k * words + j), zw, s, w);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            if (m0 + r < M) {
                const float xv = __half2float(x[(m0 + r) * ldx + k]);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[r][i] = fmaf(xv, __half2float(w[i]), acc[r][i]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        if (m0 + r >= M) break;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (y32) {
                y32[(m0 + r) * N + 8 * j + i] += acc[r][i];
            } else {
                const float b = bias ? __half2float(bias[8 * j + i]) : 0.f;
                y[(m0 + r) * N + 8 * j + i] = __float2half_rn(acc[r][i] + b);
            }
        }
    }
}

} // namespace

cudaError_t launch_generic(const Problem &p, cudaStream_t stream)
{
    const int64_t words = p.N / 8;
    const int threads = 128;
    const int64_t gx = (words + threads - 1) / threads;
    const int64_t gy = (p.M + kRows - 1) / kRows;
    if (gy > 65535) {
        // grid.y limit: split the rows into chunks of at most 65535 * kRows
        const int64_t chunk = (int64_t)65535 * kRows;
        for (int64_t m = 0; m < p.M; m += chunk) {
            Problem q = p;
            q.M = (p.M - m < chunk) ? (p.M - m) : chunk;
            q.x = static_cast<const __half *>(p.x) + m * (p.ldx > 0 ? p.ldx : p.K);
            if (p.y32) q.y32 = p.y32 + m * p.N;
            else q.y = static_cast<__half *>(p.y) + m * p.N;
            cudaError_t e = launch_generic(q, stream);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    dim3 grid((unsigned)gx, (unsigned)gy);
    generic_forward_kernel<<<grid, threads, 0, stream>>>(
        static_cast<const __half *>(p.x), reinterpret_cast<const uint32_t *>(p.qweight),
        reinterpret_cast<const uint32_t *>(p.qzeros), static_cast<const __half *>(p.scales),
        static_cast<const __half *>(p.bias), static_cast<__half *>(p.y), p.y32, p.M, p.K,
        p.ldx > 0 ? p.ldx : p.K, words, p.g);
    return cudaGetLastError();
}

} // namespace awq
