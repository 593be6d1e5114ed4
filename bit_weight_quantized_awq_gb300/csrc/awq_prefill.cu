// awq_prefill.cu -- prefill path of the WQLinear forward (large M), on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Predibase Lorax "AWQ WQLinear" page, Description, forward steps 2-3:
//   y[m, n] = fp16_rn( sum_k x[m, k] * W[k, n] + bias[n] ),
//   W[k, n] = fp16_rn((q[k, n] - z[k/g, n]) * s[k/g, n]), fp32 accumulation.
//
// Output tile: 128 rows of x (tokens) x 256 output columns; one tcgen05 MMA
// is M = 128 (tokens) x N = 256 (columns) x K = 16. A persistent grid (one
// CTA per SM) walks the tiles; inside a CTA, warps are specialised:
//
//   warp 0      TMA producer: per 64-deep k-stage, the x tile (128 x 64 fp16,
//               K-major, 128-byte swizzle) and the packed-weight tile
//               (64 k-rows x 32 words), plus the scale and zero-point rows of
//               the groups the stage touches, into a 3-stage ring.
//   warps 2-5   dequant: packed words -> fp16 W in shared memory, written
//               directly in the MN-major 128-byte-swizzled layout the MMA reads
//               as its B operand (one packed word = 8 consecutive columns =
//               one 16-byte store). Per column pair: one byte permute puts the
//               word's byte p in both halves, one LOP3 masks the low nibble
//               into the fraction of 1024.0 and the high nibble into that of
//               64.0, one half2 subtract removes (1024 + z, 64 + z) exactly,
//               one half2 multiply by the (s, s') pair -- which is simply the
//               scales word -- rounds once: exactly fp16_rn((q - z) s).
//   warp 1      MMA issuer (one thread) and TMEM owner: 4 MMAs per stage into
//               one of two 256-column fp32 accumulators, tcgen05.commit frees
//               the stage and, at the last stage, hands the accumulator over.
//   warps 6-9   epilogue: tcgen05.ld of the accumulator (each warp its 32
//               lanes = 32 tokens), + bias, one rounding to fp16, store. With
//               two accumulators the epilogue of one tile overlaps the
//               main loop of the next.
//
// A second build of the same kernel (kDequant = false) loads an already
// dequantised fp16 W with TMA straight into the B layout; it serves
// awq_gemm_f16, which checks the tensor-core core of this path on its own.
//
// Every wait is bounded; a wait that runs out records AWQ_ERR_TIMEOUT in the
// device status word, the CTA lets issued copies and MMAs finish, frees its
// tensor memory and returns.
//
// Requirements (else another path serves): K % 16 == 0, N % 32 == 0,
// group_size % 16 == 0, base pointers 16-byte aligned.
#include <algorithm>
#include <map>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "awq_device.cuh"
#include "awq_internal.h"
#include "awq_tcgen05.cuh"

namespace awq {
namespace {

constexpr int BM = 128;          // tokens per tile (MMA M)
constexpr int BN = 256;          // output columns per tile (MMA N)
constexpr int BK = 64;           // k per stage (one 128-byte swizzle row of fp16)
constexpr int kStages = 3;
constexpr int kMmaK = 16;
constexpr int kMaxGroupRows = 5;

constexpr int kABytes = BM * BK * 2;            // 16 KB
constexpr int kBBytes = BN * BK * 2;            // 32 KB
constexpr int kPBytes = BK * (BN / 8) * 4;      // 8 KB
constexpr int kSBytes = kMaxGroupRows * BN * 2;
constexpr int kZBytes = kMaxGroupRows * (BN / 8) * 4;
constexpr int kAOff = 0;
constexpr int kBOff = kAOff + kABytes;
constexpr int kPOff = kBOff + kBBytes;
constexpr int kSOff = kPOff + kPBytes;
constexpr int kZOff = kSOff + kSBytes;
constexpr int kStageBytes = 60 * 1024;
static_assert(kZOff + kZBytes <= kStageBytes, "stage layout overflows");
static_assert(kStageBytes % 1024 == 0 && kBOff % 1024 == 0, "swizzled tiles need 1024-byte alignment");
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;

// B tile layout (MN-major, 128-byte swizzle): 4 column atoms of 64 columns,
// each 8 k-groups of (8 k-rows x 128 bytes).
constexpr int kBAtomStride = 8 * 1024;   // between 64-column atoms (leading byte offset)
constexpr int kBKGroupStride = 1024;     // between 8-row k groups (stride byte offset)

constexpr int kWarps = 10;
constexpr int kThreads = kWarps * 32;
constexpr int kDequantWarp0 = 2;
constexpr int kEpilogueWarp0 = 6;
constexpr int kDequantThreads = 128;
constexpr int kEpilogueThreads = 128;
constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators

constexpr uint32_t kIdesc = tc::idesc_f16_f32(BM, BN, true);

struct PrefillParams {
    const __half *bias;
    __half *y;
    unsigned int *status;
    int M, K, N, g;
    int tiles_m, tiles_n, kiters;
    uint32_t stage_tx;
};

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    __half2 r = __hmul2_rn(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

template <bool kDequant>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
               const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
               const PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    // round up to 1024 bytes by offsetting the shared array itself, so that
    // the compiler still knows every derived pointer is a shared address
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kBarOff);
    uint64_t *dqd = full + kStages;        // dequantised B ready
    uint64_t *empty = dqd + kStages;       // MMAs of the stage done
    uint64_t *acc_full = empty + kStages;  // [2]
    uint64_t *acc_empty = acc_full + 2;    // [2]
    uint64_t *drain = acc_empty + 2;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_tiles = p.tiles_m * p.tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(full + s), 1);
            ptx::mbar_init(ptx::smem_addr(dqd + s), kDequantThreads);
            ptx::mbar_init(ptx::smem_addr(empty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_addr(acc_full + b), 1);
            ptx::mbar_init(ptx::smem_addr(acc_empty + b), kEpilogueThreads);
        }
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(ptx::smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tc::tmem_relinquish();
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_x);
            ptx::prefetch_tmap(&tm_w);
            if (kDequant) {
                ptx::prefetch_tmap(&tm_s);
                ptx::prefetch_tmap(&tm_z);
            }
            int it = 0, issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                const int m0 = (tile % p.tiles_m) * BM;
                const int n0 = (tile / p.tiles_m) * BN;
                for (int kb = 0; kb < p.kiters; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!ptx::mbar_wait_bounded(ptx::smem_addr(empty + s), ((it / kStages) & 1) ^ 1,
                                                abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = ptx::smem_addr(full + s);
                    const uint32_t st = ptx::smem_addr(smem + s * kStageBytes);
                    const int k0 = kb * BK;
                    ptx::mbar_arrive_expect_tx(fb, p.stage_tx);
                    ptx::tma_load_2d(st + kAOff, &tm_x, fb, k0, m0);
                    if (kDequant) {
                        ptx::tma_load_2d(st + kPOff, &tm_w, fb, n0 / 8, k0);
                        ptx::tma_load_2d(st + kSOff, &tm_s, fb, n0, k0 / p.g);
                        ptx::tma_load_2d(st + kZOff, &tm_z, fb, n0 / 8, k0 / p.g);
                    } else {
#pragma unroll
                        for (int a = 0; a < BN / 64; ++a)
                            ptx::tma_load_2d(st + kBOff + a * kBAtomStride, &tm_w, fb, n0 + 64 * a, k0);
                    }
                    issued = it + 1;
                }
            }
            if (!ok) {
                // let the copies already in flight land before the CTA exits
                for (int i = std::max(0, issued - kStages); i < issued; ++i)
                    ptx::mbar_wait_bounded(ptx::smem_addr(full + i % kStages), (i / kStages) & 1,
                                           nullptr, nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int it = 0, acc_it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++acc_it) {
                const int abuf = acc_it & 1;
                if (!ptx::mbar_wait_bounded(ptx::smem_addr(acc_empty + abuf), ((acc_it >> 1) & 1) ^ 1,
                                            abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(abuf * BN);
                for (int kb = 0; kb < p.kiters; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t par = (it / kStages) & 1;
                    bool ready = ptx::mbar_wait_bounded(ptx::smem_addr(full + s), par, abort_flag, p.status);
                    if (ready && kDequant)
                        ready = ptx::mbar_wait_bounded(ptx::smem_addr(dqd + s), par, abort_flag, p.status);
                    if (!ready) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t st = ptx::smem_addr(smem + s * kStageBytes);
#pragma unroll
                    for (int kk = 0; kk < BK / kMmaK; ++kk) {
                        const uint64_t ad = tc::smem_desc_sw128(st + kAOff + kk * 32, 16, 1024);
                        const uint64_t bd = tc::smem_desc_sw128(st + kBOff + kk * 2 * kBKGroupStride,
                                                                kBAtomStride, kBKGroupStride);
                        tc::mma_f16(d_tmem, ad, bd, kIdesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc::commit(ptx::smem_addr(empty + s));
                    if (kb == p.kiters - 1) tc::commit(ptx::smem_addr(acc_full + abuf));
                }
            }
            // every MMA this thread issued has completed once `drain` flips
            tc::commit(ptx::smem_addr(drain));
            ptx::mbar_wait_bounded(ptx::smem_addr(drain), 0, nullptr, p.status);
        }
    } else if (warp < kEpilogueWarp0) {
        // ------------------------------------------------------------ dequant
        if (kDequant) {
            const int dt = threadIdx.x - kDequantWarp0 * 32;   // 0..127
            const int dw = dt >> 5;                            // row phase 0..3
            const int j = dt & 31;                             // packed word in the tile row
            const int na = j >> 3, chunk = j & 7;
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                for (int kb = 0; kb < p.kiters; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!ptx::mbar_wait_bounded(ptx::smem_addr(full + s), (it / kStages) & 1,
                                                abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = ptx::smem_addr(smem + s * kStageBytes);
                    const uint32_t pbase = st + kPOff + j * 4;
                    const uint32_t bbase = st + kBOff + na * kBAtomStride;
                    const int k0 = kb * BK;
                    const int grp0 = k0 / p.g;
                    int cur = -1;
                    uint32_t S[4], Z[4];
#pragma unroll 4
                    for (int i = 0; i < BK / 4; ++i) {
                        const int row = dw + 4 * i;
                        const int grp = (k0 + row) / p.g;
                        if (grp != cur) {
                            cur = grp;
                            const int r = grp - grp0;
                            uint32_t sv0, sv1, sv2, sv3, zw;
                            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(sv0), "=r"(sv1), "=r"(sv2), "=r"(sv3)
                                         : "r"(st + kSOff + r * (BN * 2) + j * 16));
                            asm volatile("ld.shared.b32 %0, [%1];"
                                         : "=r"(zw) : "r"(st + kZOff + r * (BN / 8 * 4) + j * 4));
                            S[0] = sv0; S[1] = sv1; S[2] = sv2; S[3] = sv3;
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                Z[q] = (__byte_perm(zw, zw, q | (q << 8)) & 0x00F0000Fu) | 0x54006400u;
                        }
                        uint32_t v;
                        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(pbase + row * 128));
                        uint32_t h[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t w = (__byte_perm(v, v, q | (q << 8)) & 0x00F0000Fu) | 0x54006400u;
                            h[q] = hmul2_u(hsub2_u(w, Z[q]), S[q]);
                        }
                        const int krow = row & 7;
                        const uint32_t dst = bbase + (row >> 3) * kBKGroupStride + krow * 128 +
                                             (((uint32_t)chunk ^ (uint32_t)krow) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                     ::"r"(dst), "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]) : "memory");
                    }
                    // make the generic-proxy stores visible to the tensor core
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(ptx::smem_addr(dqd + s));
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter this warp may read
        int acc_it = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++acc_it) {
            const int abuf = acc_it & 1;
            const bool ok = __all_sync(0xffffffffu,
                                       ptx::mbar_wait_bounded(ptx::smem_addr(acc_full + abuf),
                                                              (acc_it >> 1) & 1, abort_flag, p.status));
            if (!ok) break;
            tc::fence_after_sync();
            const int m0 = (tile % p.tiles_m) * BM;
            const int n0 = (tile / p.tiles_m) * BN;
            const int m = m0 + 32 * q + lane;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tc::ld_32x32b_x32(tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(abuf * BN + 32 * c), r);
                tc::ld_wait();
                const int col = n0 + 32 * c;
                if (col < p.N && m < p.M) {
                    __align__(16) __half out[32];
                    if (p.bias) {
                        __align__(16) __half bh[32];
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            reinterpret_cast<uint4 *>(bh)[v] = __ldg(reinterpret_cast<const uint4 *>(p.bias + col) + v);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            out[e] = __float2half_rn(__uint_as_float(r[e]) + __half2float(bh[e]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) out[e] = __float2half_rn(__uint_as_float(r[e]));
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(p.y + (int64_t)m * p.N + col);
#pragma unroll
                    for (int v = 0; v < 4; ++v) dst[v] = reinterpret_cast<const uint4 *>(out)[v];
                }
            }
            tc::fence_before_sync();
            ptx::mbar_arrive(ptx::smem_addr(acc_empty + abuf));
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
                 uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int group_rows_per_stage(int64_t g)
{
    if (BK % g == 0) return (int)(BK / g);
    if (g % BK == 0) return 1;
    return (int)((BK - 1) / g + 2);
}

struct LaunchInfo {
    int sms = 0;
    cudaError_t err = cudaSuccess;
};

template <bool kDequant>
LaunchInfo launch_info()
{
    static std::mutex mu;
    static std::map<int, LaunchInfo> cache;
    int dev = 0;
    LaunchInfo li;
    li.err = cudaGetDevice(&dev);
    if (li.err != cudaSuccess) return li;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    li.err = cudaFuncSetAttribute(prefill_kernel<kDequant>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSmemBytes);
    if (li.err == cudaSuccess)
        li.err = cudaDeviceGetAttribute(&li.sms, cudaDevAttrMultiProcessorCount, dev);
    if (li.err == cudaSuccess) cache[dev] = li;
    return li;
}

template <bool kDequant>
cudaError_t launch(const Problem &pr, const void *w16, cudaStream_t stream)
{
    const LaunchInfo li = launch_info<kDequant>();
    if (li.err != cudaSuccess) return li.err;
    const int M = (int)pr.M, K = (int)pr.K, N = (int)pr.N, g = (int)pr.g;
    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    const int kiters = (K + BK - 1) / BK;
    const int64_t n_tiles = (int64_t)tiles_m * tiles_n;
    const int ctas = (int)std::min<int64_t>(n_tiles, li.sms);

    CUtensorMap tx, tw, ts, tz;
    bool ok = make_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pr.x, K, M, (uint64_t)K * 2, BK, BM,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    uint32_t tx_bytes = kABytes;
    if (kDequant) {
        const int R = group_rows_per_stage(g);
        ok = ok &&
             make_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_INT32, pr.qweight, N / 8, K, (uint64_t)N / 2,
                         BN / 8, BK, CU_TENSOR_MAP_SWIZZLE_NONE) &&
             make_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pr.scales, N, pr.G, (uint64_t)N * 2, BN, R,
                         CU_TENSOR_MAP_SWIZZLE_NONE) &&
             make_map_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_INT32, pr.qzeros, N / 8, pr.G, (uint64_t)N / 2,
                         BN / 8, R, CU_TENSOR_MAP_SWIZZLE_NONE);
        tx_bytes += kPBytes + R * (BN * 2) + R * (BN / 8 * 4);
    } else {
        ok = ok && make_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w16, N, K, (uint64_t)N * 2, 64, BK,
                               CU_TENSOR_MAP_SWIZZLE_128B);
        ts = tw;
        tz = tw;
        tx_bytes += kBBytes;
    }
    if (!ok) return cudaErrorInvalidValue;

    PrefillParams p{};
    p.bias = static_cast<const __half *>(pr.bias);
    p.y = static_cast<__half *>(pr.y);
    p.status = device_status_word();
    p.M = M; p.K = K; p.N = N; p.g = g;
    p.tiles_m = tiles_m; p.tiles_n = tiles_n; p.kiters = kiters;
    p.stage_tx = tx_bytes;
    prefill_kernel<kDequant><<<ctas, kThreads, kSmemBytes, stream>>>(tx, tw, ts, tz, p);
    return cudaGetLastError();
}

} // namespace

bool prefill_supported(int64_t M, int64_t K, int64_t N, int64_t g)
{
    return M >= 1 && M < (int64_t(1) << 31) && K % 16 == 0 && N % 32 == 0 && g % 16 == 0 &&
           K <= (int64_t(1) << 30) && N <= (int64_t(1) << 30);
}

cudaError_t launch_prefill(const Problem &p, cudaStream_t stream)
{
    if (!prefill_supported(p.M, p.K, p.N, p.g)) return cudaErrorInvalidValue;
    return launch<true>(p, nullptr, stream);
}

cudaError_t launch_gemm_f16(const Problem &p, const void *w16, cudaStream_t stream)
{
    return launch<false>(p, w16, stream);
}

} // namespace awq
