// awq_gather.cu -- the act-order form of the g_idx grouping variant run on
// the grouped kernels.
//
// Linear Layer Factory page, Description: the GPTQ quantisation tuple holds a
// g_idx table, the group of every input row. Under act-order that table is a
// permutation of contiguous groups: every group holds the same number of
// rows g = K / G, only not consecutive ones. Sorting the rows by group (a
// fixed permutation perm, taken once when the layer is loaded) gives an
// ordinary grouped layer: row i of the sorted weights is row perm[i] of the
// original and lies in group i / g, so qzeros and scales are unchanged. The
// forward then needs the activations in the same order,
//   y[m, n] = sum_i x[m, perm[i]] * W[perm[i], n],
// which is the original sum with its terms reordered.
//
//   gather_rows_kernel: qweight_sorted[i, :] = qweight[perm[i], :] (once).
//   gather_cols_kernel: x_sorted[m, i] = x[m, perm[i]] (every call; M x K
//                       fp16 read and written, small next to the weights).
// Both check every perm entry: one outside [0, K) writes zeros and records
// kStatusBadIndex in the device status word instead of reading out of bounds.
#include <mutex>
#include <map>
#include <set>

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {
namespace {

__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4 *__restrict__ src, const int32_t *__restrict__ perm, uint4 *__restrict__ dst,
                   int64_t K, int64_t row_vecs, unsigned int *status)
{
    const int64_t total = K * row_vecs;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / row_vecs;
        const int64_t v = idx - i * row_vecs;
        const int64_t k = __ldg(perm + i);
        if (k < 0 || k >= K) {
            raise_status(status, kStatusBadIndex);
            dst[idx] = make_uint4(0u, 0u, 0u, 0u);
        } else {
            dst[idx] = __ldg(src + k * row_vecs + v);
        }
    }
}

// Rows of x up to this many fp16 elements are staged in shared memory.
constexpr int64_t kStagedMaxK = 96 * 1024;

// One CTA per row of x at a time: the row is read into shared memory with
// coalesced 16-byte loads, then every thread takes 8 consecutive sorted
// columns: eight 2-byte reads from shared memory, one 16-byte store. The
// next kernel on the stream (the forward, launched as a programmatic
// dependent) may start streaming its weights meanwhile.
__global__ void __launch_bounds__(256)
gather_cols_staged_kernel(const __half *__restrict__ x, int64_t ldx, const int32_t *__restrict__ perm,
                          __half *__restrict__ xs, int64_t M, int64_t K, unsigned int *status)
{
    extern __shared__ uint4 row_smem[];
    const __half *row = reinterpret_cast<const __half *>(row_smem);
    ptx::launch_dependents();
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + m * ldx);
        for (int64_t v = threadIdx.x; v < K / 8; v += blockDim.x) row_smem[v] = __ldg(src + v);
        __syncthreads();
        for (int64_t i0 = 8 * (int64_t)threadIdx.x; i0 < K; i0 += 8 * (int64_t)blockDim.x) {
            const int4 pa = __ldg(reinterpret_cast<const int4 *>(perm + i0));
            const int4 pb = __ldg(reinterpret_cast<const int4 *>(perm + i0 + 4));
            const int p8[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
            __align__(16) __half out[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int k = p8[e];
                if (k < 0 || k >= K) {
                    raise_status(status, kStatusBadIndex);
                    out[e] = __ushort_as_half((unsigned short)0);
                } else {
                    out[e] = row[k];
                }
            }
            *reinterpret_cast<uint4 *>(xs + m * K + i0) = *reinterpret_cast<const uint4 *>(out);
        }
        __syncthreads();
    }
}

// Longer rows: one thread per (row of x, 8 consecutive sorted columns),
// eight 2-byte gathers from the row in global memory, one 16-byte store.
__global__ void __launch_bounds__(256)
gather_cols_kernel(const __half *__restrict__ x, int64_t ldx, const int32_t *__restrict__ perm,
                   __half *__restrict__ xs, int64_t M, int64_t K, unsigned int *status)
{
    const int64_t per_row = K / 8;
    const int64_t total = M * per_row;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = idx / per_row;
        const int64_t i0 = (idx - m * per_row) * 8;
        const int4 pa = __ldg(reinterpret_cast<const int4 *>(perm + i0));
        const int4 pb = __ldg(reinterpret_cast<const int4 *>(perm + i0 + 4));
        const int p8[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
        __align__(16) __half out[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int k = p8[e];
            if (k < 0 || k >= K) {
                raise_status(status, kStatusBadIndex);
                out[e] = __ushort_as_half((unsigned short)0);
            } else {
                out[e] = x[m * ldx + k];
            }
        }
        *reinterpret_cast<uint4 *>(xs + m * K + i0) = *reinterpret_cast<const uint4 *>(out);
    }
}

int grid_for(int64_t items)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = (items + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

} // namespace

cudaError_t launch_gather_rows(const int32_t *src, const int32_t *perm, int32_t *dst, int64_t K,
                               int64_t words, cudaStream_t stream)
{
    const int64_t row_vecs = words / 4;   // words % 4 == 0: N % 32 == 0
    gather_rows_kernel<<<grid_for(K * row_vecs), 256, 0, stream>>>(
        reinterpret_cast<const uint4 *>(src), perm, reinterpret_cast<uint4 *>(dst), K, row_vecs,
        device_status_word());
    return cudaGetLastError();
}

cudaError_t launch_gather_cols(const void *x, int64_t ldx, const int32_t *perm, void *xs, int64_t M,
                               int64_t K, cudaStream_t stream)
{
    if (K <= kStagedMaxK) {
        const size_t smem = (size_t)K * 2;
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        {
            // the shared-memory limit is a per-device attribute of the function
            static std::mutex mu;
            static std::map<int, unsigned> ready;   // device -> cache generation
            const unsigned gen = cache_generation();
            std::lock_guard<std::mutex> lock(mu);
            auto it = ready.find(dev);
            if (it == ready.end() || it->second != gen) {
                cudaError_t e = cudaFuncSetAttribute(gather_cols_staged_kernel,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     (int)(kStagedMaxK * 2));
                if (e != cudaSuccess) return e;
                ready[dev] = gen;
            }
        }
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 4;
        const unsigned grid = (unsigned)(M < cap ? M : cap);
        gather_cols_staged_kernel<<<grid, 256, smem, stream>>>(
            static_cast<const __half *>(x), ldx, perm, static_cast<__half *>(xs), M, K, device_status_word());
        return cudaGetLastError();
    }
    gather_cols_kernel<<<grid_for(M * (K / 8)), 256, 0, stream>>>(
        static_cast<const __half *>(x), ldx, perm, static_cast<__half *>(xs), M, K, device_status_word());
    return cudaGetLastError();
}

} // namespace awq
