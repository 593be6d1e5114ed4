// awq_decode.cu -- decode path of the WQLinear forward (small M, 1..16 rows).
//
// Predibase Lorax "AWQ WQLinear" page, Description, forward steps 2-3:
//   y[m, n] = fp16_rn( sum_k x[m, k] * W[k, n] + bias[n] ),
//   W[k, n] = fp16_rn((q[k, n] - z[k/g, n]) * s[k/g, n]), fp32 accumulation.
//
// At small M the layer is bound by streaming the packed weights from HBM
// (0.52 bytes per weight at g = 128). The kernel is built around that:
//
//  * Work: the K x N weight matrix is cut into tiles of 256 columns (one
//    128-byte row of packed words) and stages of 256 k-rows. The (tile,
//    stage) iterations, tile-major, are split evenly between the CTAs (one
//    per SM): each CTA streams a contiguous run of them ("stream-K").
//  * Loads: one producer warp issues four TMA boxes per stage -- 256 x 128 B
//    of qweight (32 KB, 128-byte swizzle), the 256 x Mpad activation slice
//    (one 3-D box), and the scale and zero-point rows of the groups the stage
//    touches -- into a 4-stage ring guarded by mbarriers (full: bytes landed;
//    empty: the consumers released the slot). Issuing a TMA instruction costs
//    the producer on the order of a hundred cycles, so each one moves as many
//    bytes as the box limits allow.
//  * Math: 8 consumer warps: two k-groups (group kg takes rows 128 kg ..
//    128 kg + 127 of every stage, eight 16-row chunks) of four warps (each
//    owns 64 columns). Each warp dequantises in registers and runs the legacy-path
//    tensor-core MMA m16n8k16 with W as the A operand (16 output columns x 16
//    k) and the activations as B (16 k x 8 tokens), fp32 accumulators. Two
//    k-adjacent weights of one column form one half2 operand register: a byte
//    permute brings byte b of rows k and k+1 together, one LOP3 masks a nibble
//    into the fraction of 1024.0 or 64.0, an exact half2 subtract removes the
//    zero point and one half2 multiply (round to nearest) applies the scale --
//    exactly fp16_rn((q - z) s).
//  * Reduction: a tile split between CTAs is finished by the CTA that holds
//    its last k-stages, which is the highest-numbered contributor (its range
//    starts inside the tile). Every contributor writes its fp32 partial to
//    scratch; the others count themselves in, and after its own stream the
//    finisher waits (bounded) for them -- only ever for lower-numbered CTAs,
//    which were dispatched before it, so no co-residency is needed -- sums
//    all partials in contributor order, adds the bias and rounds once.
//  * Launch: programmatic dependent launch. The kernel lets the next one be
//    scheduled at once and loads its first stages' weights before waiting
//    for the previous kernel; activations, bias, output and scratch are
//    touched only after that wait.
//
// Requirements (else another path serves): 1 <= M <= 16, K % 64 == 0,
// N % 32 == 0 (TMA row pitch), g % 16 == 0 with at most 8 groups per 256-row
// stage (g >= 32), base pointers 16-byte aligned.
#include <algorithm>
#include <map>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kTileWords = 32;   // packed words per tile row
constexpr int kTileCols = 256;   // output columns per tile
constexpr int kStageRows = 256;  // k-rows per pipeline stage
constexpr int kStages = 4;
constexpr int kKBlocks = kStageRows / 64;   // 64-row blocks of a stage (activation layout)
constexpr int kColWarps = 4;     // warps across a tile's columns, 8 words each

// Warp layout for KG consumer k-groups: k-group kg takes stage rows
// kRowsPerWarp * kg .. + kRowsPerWarp - 1, split in 16-row chunks; each of its
// kColWarps warps owns 64 columns. One producer warp follows the consumers.
template <int KG>
struct Layout {
    static constexpr int kKGroups = KG;
    static constexpr int kRowsPerWarp = kStageRows / KG;
    static constexpr int kChunksPerWarp = kRowsPerWarp / 16;
    static constexpr int kConsumerWarps = kColWarps * KG;
    static constexpr int kConsumerThreads = kConsumerWarps * 32;
    static constexpr int kThreads = kConsumerThreads + 32;
};
constexpr int kMaxTokens = 16;
constexpr int kMaxGroupRows = 8; // group rows one stage may touch (g >= 32)

constexpr int kWBytes = kStageRows * 128;
constexpr int kXBytes = kMaxTokens * kStageRows * 2;
constexpr int kSBytes = kMaxGroupRows * kTileCols * 2;
constexpr int kZBytes = kMaxGroupRows * kTileWords * 4;
constexpr int kXOff = kWBytes;
constexpr int kSOff = kXOff + kXBytes;
constexpr int kZOff = kSOff + kSBytes;
constexpr int kStageBytes = 45 * 1024;
static_assert(kZOff + kZBytes <= kStageBytes, "stage layout overflows");
static_assert(kStageBytes % 1024 == 0 && kXOff % 1024 == 0, "swizzled tiles need 1024-byte alignment");
constexpr int kFoldFloats = kMaxTokens * kTileCols;     // one k-group's sums
constexpr int kRedOff = kStages * kStageBytes;
constexpr int kRedBytes = 2 * kFoldFloats * 4;
constexpr int kBarOff = kRedOff + kRedBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;   // barriers + flags + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

constexpr int kPartialFloats = kMaxTokens * kTileCols;  // one partial slot

struct DecodeParams {
    const __half *bias;
    __half *y;
    float *partials;        // [2 * ctas][16][256]
    unsigned int *arrive;   // [tiles]
    unsigned int *status;
    int M, K, N, g;
    int tiles, kiters, total, ctas;
    uint32_t stage_tx;      // bytes one stage's TMA boxes deliver
};

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    __half2 r = __hmul2_rn(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// The CTA whose iteration range contains iteration `it`.
__device__ __forceinline__ int cta_of(int it, int total, int ctas) {
    return (int)((((int64_t)it + 1) * ctas - 1) / total);
}
__device__ __forceinline__ int range_begin(int c, int total, int ctas) {
    return (int)(((int64_t)c * total) / ctas);
}

template <int MT>
__device__ __forceinline__ void fold_store(float *dst, const float (&acc)[4][MT][4], int ct) {
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[((b * MT + mt) * 4 + e) * 128 + ct] = acc[b][mt][e];
}
template <int MT>
__device__ __forceinline__ void fold_add(const float *src, float (&acc)[4][MT][4], int ct) {
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[b][mt][e] += src[((b * MT + mt) * 4 + e) * 128 + ct];
}

template <int MT, int KG, bool kWholeGroups>
__global__ void __launch_bounds__(Layout<KG>::kThreads, 1)
decode_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
              const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
              const DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    // round up to 1024 bytes by offsetting the shared array itself, so that
    // the compiler still knows every derived pointer is a shared address
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    float *red = reinterpret_cast<float *>(smem + kRedOff);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kBarOff);
    uint64_t *empty = full + kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kStages);
    volatile int *duty_ok = abort_flag + 1;
    volatile uint32_t *consts = reinterpret_cast<volatile uint32_t *>(abort_flag + 2);

    using L = Layout<KG>;
    constexpr int kConsumerWarps = L::kConsumerWarps;
    constexpr int kConsumerThreads = L::kConsumerThreads;
    constexpr int kChunksPerWarp = L::kChunksPerWarp;
    constexpr int kRowsPerWarp = L::kRowsPerWarp;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int begin = range_begin(c, p.total, p.ctas);
    const int end = range_begin(c + 1, p.total, p.ctas);
    const int n_iters = end - begin;
    const int first_tile = begin / p.kiters;
    // This CTA finishes the tile its range starts in when the range starts
    // inside that tile and reaches the tile's last k-stage: the other
    // contributors are then lower-numbered CTAs, which started before it.
    const bool reducer = n_iters > 0 && begin % p.kiters != 0 && end >= (first_tile + 1) * p.kiters;

    // the next kernel on the stream may be scheduled as SMs free up
    ptx::launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(full + s), 1);
            ptx::mbar_init(ptx::smem_addr(empty + s), kConsumerWarps);
        }
        *abort_flag = 0;
        *duty_ok = 0;
        consts[0] = 0x64006400u;   // 1024.0 in both halves
        consts[1] = 0x54005400u;   // 64.0 in both halves
        ptx::fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------------ producer
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_w);
            ptx::prefetch_tmap(&tm_x);
            ptx::prefetch_tmap(&tm_s);
            ptx::prefetch_tmap(&tm_z);
            int tile = first_tile;
            int kb = begin - tile * p.kiters;
            // The weights, scales and zero points of the first stages do not
            // depend on the kernel before this one: load them while it
            // finishes, and the activations once it has.
            const int pre = n_iters < kStages ? n_iters : kStages;
            for (int i = 0; i < pre; ++i) {
                const uint32_t fb = ptx::smem_addr(full + i);
                const uint32_t st = ptx::smem_addr(smem + i * kStageBytes);
                const int k0 = kb * kStageRows;
                const int grp0 = k0 / p.g;
                ptx::mbar_arrive_expect_tx(fb, p.stage_tx);
                ptx::tma_load_2d(st, &tm_w, fb, tile * kTileWords, k0);
                ptx::tma_load_2d(st + kSOff, &tm_s, fb, tile * kTileCols, grp0);
                ptx::tma_load_2d(st + kZOff, &tm_z, fb, tile * kTileWords, grp0);
                if (++kb == p.kiters) { kb = 0; ++tile; }
            }
            ptx::wait_prerequisites();
            for (int i = 0, kx = begin % p.kiters; i < pre; ++i) {
                ptx::tma_load_3d(ptx::smem_addr(smem + i * kStageBytes + kXOff), &tm_x,
                                 ptx::smem_addr(full + i), 0, kx * (kStageRows / 64), 0);
                if (++kx == p.kiters) kx = 0;
            }
            int issued = pre;
            for (int i = pre; i < n_iters; ++i) {
                const int s = i % kStages;
                const uint32_t parity = ((i / kStages) & 1) ^ 1;
                if (!ptx::mbar_wait_bounded(ptx::smem_addr(empty + s), parity, abort_flag, p.status))
                    break;
                const uint32_t fb = ptx::smem_addr(full + s);
                const uint32_t st = ptx::smem_addr(smem + s * kStageBytes);
                const int k0 = kb * kStageRows;
                const int grp0 = k0 / p.g;
                ptx::mbar_arrive_expect_tx(fb, p.stage_tx);
                ptx::tma_load_2d(st, &tm_w, fb, tile * kTileWords, k0);
                ptx::tma_load_3d(st + kXOff, &tm_x, fb, 0, k0 / 64, 0);
                ptx::tma_load_2d(st + kSOff, &tm_s, fb, tile * kTileCols, grp0);
                ptx::tma_load_2d(st + kZOff, &tm_z, fb, tile * kTileWords, grp0);
                issued = i + 1;
                if (++kb == p.kiters) { kb = 0; ++tile; }
            }
            if (*abort_flag) {
                // let the copies already in flight land before the CTA exits
                for (int i = std::max(0, issued - kStages); i < issued; ++i)
                    ptx::mbar_wait_bounded(ptx::smem_addr(full + i % kStages), (i / kStages) & 1,
                                           nullptr, nullptr);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    // everything below reads or writes global memory the kernel before this
    // one may still use (activations come through the producer, which waited)
    ptx::wait_prerequisites();
    const int kg = warp / kColWarps;   // rows kRowsPerWarp * kg .. of every stage
    const int cw = warp % kColWarps;   // which 64-column quarter of the tile
    const int gq = lane >> 2;          // MMA groupID: output column pair / token
    const int tq = lane & 3;           // MMA thread-in-group: k pair / token pair
    const int word = cw * 8 + gq;      // packed word (8 columns) this thread owns
    const int ct = cw * 32 + lane;     // thread index within a k-group

    // Byte offsets inside a stage. Chunk j of this warp is stage rows
    // R0 + 16 j .. +15 (R0 = kRowsPerWarp kg); rows 16ch + 2tq (+1) sit at a
    // fixed 128-byte swizzle phase, rows +8 / +9 one 1024-byte atom further.
    const int R0 = kRowsPerWarp * kg;
    const uint32_t wchunk = (uint32_t)(word >> 2);
    const uint32_t inw = (uint32_t)(word & 3) * 4;
    const uint32_t rA = (uint32_t)(2 * tq), rB = rA + 1;
    const uint32_t offA = (uint32_t)R0 * 128 + rA * 128 + ((wchunk ^ rA) << 4) + inw;
    const uint32_t offB = (uint32_t)R0 * 128 + rB * 128 + ((wchunk ^ rB) << 4) + inw;
    // activation slice: [token m][64-row block][64 halves], 128-byte rows
    // (r = m * 4 + block), 16-byte unit u of row r stored at unit u ^ (r % 8).
    // Chunk j of this warp is block R0 / 64 + j / 4, units 2 (j % 4) and
    // 2 (j % 4) + 1 -- the k 0..7 and 8..15 halves of its B operand. One
    // ldmatrix.x4 fetches the B operands of a chunk pair for eight tokens:
    // lane L addresses token L % 8, unit 4 * pair + L / 8 of the block.
    constexpr int kBlocksPerWarp = (kChunksPerWarp + 3) / 4;
    static_assert(kChunksPerWarp % 2 == 0, "chunks are fetched in pairs");
    uint32_t xoff[MT][kBlocksPerWarp][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int jb = 0; jb < kBlocksPerWarp; ++jb) {
            const uint32_t r = (uint32_t)((8 * mt + (lane & 7)) * kKBlocks + R0 / 64 + jb);
#pragma unroll
            for (int pr = 0; pr < 2; ++pr)
                xoff[mt][jb][pr] = kXOff + r * 128 + (((uint32_t)(4 * pr + (lane >> 3)) ^ (r & 7)) << 4);
        }
    const uint32_t soff = kSOff + (uint32_t)word * 16;
    const uint32_t zoff = kZOff + (uint32_t)word * 4;
    // the fp16 exponent patterns OR-ed into the nibbles, read from shared
    // memory so that they stay in registers instead of being rebuilt before
    // every use (a LOP3 takes only one immediate operand)
    const uint32_t base_lo = consts[0];
    const uint32_t base_hi = consts[1];

    float acc[4][MT][4];
    uint32_t S2[8], Zlo[4], Zhi[4];
    int loaded_grp = -1;
    // group index and offset inside its group of the stage's first row (st_)
    // and of this warp's first row (wg_)
    int st_grp = 0, st_rem = 0, wg_grp = 0, wg_rem = 0;
    int seg_kb0 = 0;
    int tile = first_tile;
    int kb = begin - tile * p.kiters;

    // loads this thread's 8 scales and zero points of group row r of a stage
    auto load_group = [&](const uint8_t *stp, uint32_t r) {
        const uint4 sv = *reinterpret_cast<const uint4 *>(stp + soff + r * (kTileCols * 2));
        const uint32_t zw = *reinterpret_cast<const uint32_t *>(stp + zoff + r * (kTileWords * 4));
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            S2[2 * h] = __byte_perm(sw[h], sw[h], 0x1010);
            S2[2 * h + 1] = __byte_perm(sw[h], sw[h], 0x3232);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t t = __byte_perm(zw, zw, b | ((4 + b) << 8));
            Zlo[b] = (t & 0x000F000Fu) | base_lo;
            Zhi[b] = (t & 0x00F000F0u) | base_hi;
        }
    };

    for (int i = 0; i < n_iters; ++i) {
        const int k0 = kb * kStageRows;
        if (i == 0 || kb == 0) {
            seg_kb0 = kb;
            loaded_grp = -1;
            st_grp = k0 / p.g;
            st_rem = k0 - st_grp * p.g;
            wg_grp = (k0 + R0) / p.g;
            wg_rem = k0 + R0 - wg_grp * p.g;
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[b][mt][e] = 0.f;
        } else {
            st_rem += kStageRows;
            while (st_rem >= p.g) { st_rem -= p.g; ++st_grp; }
            wg_rem += kStageRows;
            while (wg_rem >= p.g) { wg_rem -= p.g; ++wg_grp; }
        }
        const int s = i % kStages;
        // every lane waits (each needs the acquire); the MMA below is
        // warp-wide, so the outcome is made uniform across the warp
        const bool ok = __all_sync(0xffffffffu,
                                   ptx::mbar_wait_bounded(ptx::smem_addr(full + s), (i / kStages) & 1,
                                                          abort_flag, p.status));
        if (ok && k0 + R0 < p.K) {
            const uint8_t *stp = smem + s * kStageBytes;
            if (kWholeGroups) {
                // g % kRowsPerWarp == 0: the warp's rows lie in one group
                if (wg_grp != loaded_grp) {
                    loaded_grp = wg_grp;
                    load_group(stp, (uint32_t)(wg_grp - st_grp));
                }
            }
            int grp = wg_grp, rem = wg_rem;
            const uint32_t sbase = ptx::smem_addr(stp);
            uint32_t xq[MT][4];   // B operands of the current chunk pair
#pragma unroll
            for (int j = 0; j < kChunksPerWarp; ++j) {
                if (!kWholeGroups) {
                    if (j > 0) {
                        rem += 16;
                        if (rem >= p.g) { rem -= p.g; ++grp; }
                    }
                    if (grp != loaded_grp) {
                        loaded_grp = grp;
                        load_group(stp, (uint32_t)(grp - st_grp));
                    }
                }
                const uint8_t *wp = stp + j * (16 * 128);
                const uint32_t v0 = *reinterpret_cast<const uint32_t *>(wp + offA);
                const uint32_t v1 = *reinterpret_cast<const uint32_t *>(wp + offB);
                const uint32_t v8 = *reinterpret_cast<const uint32_t *>(wp + offA + 1024);
                const uint32_t v9 = *reinterpret_cast<const uint32_t *>(wp + offB + 1024);
                if ((j & 1) == 0) {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        ptx::ldmatrix_x4(sbase + xoff[mt][j / 4][(j % 4) / 2], xq[mt]);
                }
                uint32_t bf[MT][2];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    bf[mt][0] = xq[mt][2 * (j & 1)];
                    bf[mt][1] = xq[mt][2 * (j & 1) + 1];
                }
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const uint32_t sel = (uint32_t)(b | ((4 + b) << 8));
                    const uint32_t t01 = __byte_perm(v0, v1, sel);
                    const uint32_t t89 = __byte_perm(v8, v9, sel);
                    uint32_t a[4];
                    a[0] = hmul2_u(hsub2_u((t01 & 0x000F000Fu) | base_lo, Zlo[b]), S2[2 * b]);
                    a[1] = hmul2_u(hsub2_u((t01 & 0x00F000F0u) | base_hi, Zhi[b]), S2[2 * b + 1]);
                    a[2] = hmul2_u(hsub2_u((t89 & 0x000F000Fu) | base_lo, Zlo[b]), S2[2 * b]);
                    a[3] = hmul2_u(hsub2_u((t89 & 0x00F000F0u) | base_hi, Zhi[b]), S2[2 * b + 1]);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) ptx::mma_16816(acc[b][mt], a, bf[mt][0], bf[mt][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(empty + s));

        if (i == n_iters - 1 || kb == p.kiters - 1) {
            // ---- segment end: fold the k-groups into group 0, in the fixed
            //      order (g0 + g2) + (g1 + g3) for four groups
            if (KG == 4) {
                if (kg >= 2) fold_store<MT>(red + (kg - 2) * kFoldFloats, acc, ct);
                ptx::named_barrier(1, kConsumerThreads);
                if (kg < 2) fold_add<MT>(red + kg * kFoldFloats, acc, ct);
                ptx::named_barrier(1, kConsumerThreads);
            }
            if (kg == 1) fold_store<MT>(red, acc, ct);
            ptx::named_barrier(1, kConsumerThreads);
            if (kg == 0) fold_add<MT>(red, acc, ct);
            ptx::named_barrier(1, kConsumerThreads);

            // `whole` is uniform across the CTA; barrier participation never
            // depends on the abort flag, which other warps may set at any time
            const bool whole = (seg_kb0 == 0 && kb == p.kiters - 1);
            if (kg == 0) {
                const bool live = !*abort_flag;
                const int col0 = tile * kTileCols + word * 8;
                if (whole && live) {
                    float bv[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) bv[jj] = 0.f;
                    if (p.bias && col0 < p.N) {
                        const uint4 braw = *reinterpret_cast<const uint4 *>(p.bias + col0);
                        const __half *bh = reinterpret_cast<const __half *>(&braw);
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) bv[jj] = __half2float(bh[jj]);
                    }
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int m = 8 * mt + 2 * tq + e;
                            if (m < p.M && col0 < p.N) {
                                __align__(16) __half out[8];
#pragma unroll
                                for (int b = 0; b < 4; ++b) {
                                    out[2 * b] = __float2half_rn(acc[b][mt][e] + bv[2 * b]);
                                    out[2 * b + 1] = __float2half_rn(acc[b][mt][2 + e] + bv[2 * b + 1]);
                                }
                                *reinterpret_cast<uint4 *>(p.y + (int64_t)m * p.N + col0) =
                                    *reinterpret_cast<const uint4 *>(out);
                            }
                        }
                } else if (!whole && live) {
                    const int which = (tile == first_tile) ? 0 : 1;
                    float *slot = p.partials + (int64_t)(2 * c + which) * kPartialFloats;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int m = 8 * mt + 2 * tq + e;
                            if (m < p.M) {
                                float4 lo = make_float4(acc[0][mt][e], acc[0][mt][2 + e], acc[1][mt][e], acc[1][mt][2 + e]);
                                float4 hi = make_float4(acc[2][mt][e], acc[2][mt][2 + e], acc[3][mt][e], acc[3][mt][2 + e]);
                                float4 *dst = reinterpret_cast<float4 *>(slot + m * kTileCols + word * 8);
                                dst[0] = lo;
                                dst[1] = hi;
                            }
                        }
                    __threadfence();
                }
                if (!whole) {
                    ptx::named_barrier(2, kConsumerThreads / KG);
                    // count in with the tile's finisher (not needed for its own tile)
                    if (ct == 0 && !*abort_flag && !(reducer && tile == first_tile))
                        atomicAdd(p.arrive + tile, 1u);
                }
            }
        }
        if (++kb == p.kiters) { kb = 0; ++tile; }
    }

    // ---- finishing the split tile this range starts in: wait for the other
    //      contributors (lower-numbered CTAs) to count in, then sum every
    //      partial, its own included, in contributor order, so the result
    //      does not depend on timing; add the bias and round once.
    if (!reducer) return;
    const int ctid = threadIdx.x;   // 0 .. kConsumerThreads-1
    const int t = first_tile;
    const int cf = cta_of(t * p.kiters, p.total, p.ctas);
    const int n = c - cf + 1;
    if (ctid == 0) {
        bool ok = !*abort_flag;
        const long long t0 = clock64();
        while (ok && ptx::ld_acquire_gpu(p.arrive + t) < (unsigned)(n - 1)) {
            if (*abort_flag || clock64() - t0 > ptx::kWaitLimitCycles) {
                ok = false;
                *abort_flag = 1;
                atomicOr(p.status, kStatusTimeout);
            } else {
                __nanosleep(32);
            }
        }
        *duty_ok = ok ? 1 : 0;
    }
    ptx::named_barrier(1, kConsumerThreads);
    if (!*duty_ok) return;
    // Each thread owns float4 positions of the tile (pos = ctid + k * threads)
    // and copies them from every contributor's partial into the idle stage
    // ring with asynchronous 16-byte copies -- all in flight at once -- then
    // adds them up in contributor order from its own slots (no barrier: a
    // thread reads only what it copied). The order is fixed, so the result
    // does not depend on timing. Only the first contributor may hold the
    // tile in its second slot.
    const int which_cf = (range_begin(cf, p.total, p.ctas) / p.kiters == t) ? 0 : 1;
    constexpr int kPosPerThread = (kMaxTokens * kTileCols / 4 + kConsumerThreads - 1) / kConsumerThreads;
    const int n4 = p.M * (kTileCols / 4);   // float4 positions of one partial
    const int per_round = (kStages * kStageBytes) / (n4 * 16);
    const uint32_t ring = ptx::smem_addr(smem);
    float4 acc4[kPosPerThread];
#pragma unroll
    for (int k = 0; k < kPosPerThread; ++k) acc4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r0 = 0; r0 < n; r0 += per_round) {
        const int cnt = std::min(per_round, n - r0);
        for (int q = 0; q < cnt; ++q) {
            const int ci = cf + r0 + q;
            const float *slot = p.partials + (int64_t)(2 * ci + (ci == cf ? which_cf : 0)) * kPartialFloats;
#pragma unroll
            for (int k = 0; k < kPosPerThread; ++k) {
                const int pos = ctid + k * kConsumerThreads;
                if (pos < n4)
                    ptx::cp_async_16(ring + (uint32_t)(q * n4 + pos) * 16,
                                     slot + (pos / (kTileCols / 4)) * kTileCols + (pos % (kTileCols / 4)) * 4);
            }
        }
        ptx::cp_async_wait_all();
        for (int q = 0; q < cnt; ++q) {
#pragma unroll
            for (int k = 0; k < kPosPerThread; ++k) {
                const int pos = ctid + k * kConsumerThreads;
                if (pos < n4) {
                    const float4 v = *reinterpret_cast<const float4 *>(smem + (size_t)(q * n4 + pos) * 16);
                    acc4[k].x += v.x; acc4[k].y += v.y; acc4[k].z += v.z; acc4[k].w += v.w;
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < kPosPerThread; ++k) {
        const int pos = ctid + k * kConsumerThreads;
        if (pos >= n4) continue;
        const int m = pos / (kTileCols / 4);
        const int col = t * kTileCols + (pos % (kTileCols / 4)) * 4;
        if (col >= p.N || *abort_flag) continue;
        float b[4] = {0.f, 0.f, 0.f, 0.f};
        if (p.bias) {
            const uint2 braw = *reinterpret_cast<const uint2 *>(p.bias + col);
            const __half *bh = reinterpret_cast<const __half *>(&braw);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) b[jj] = __half2float(bh[jj]);
        }
        __align__(8) __half out[4] = {__float2half_rn(acc4[k].x + b[0]), __float2half_rn(acc4[k].y + b[1]),
                                      __float2half_rn(acc4[k].z + b[2]), __float2half_rn(acc4[k].w + b[3])};
        *reinterpret_cast<uint2 *>(p.y + (int64_t)m * p.N + col) = *reinterpret_cast<const uint2 *>(out);
    }
    // the counter is this CTA's alone now: reset it for the next call
    if (ctid == 0) atomicExch(p.arrive + t, 0u);
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

// rank-2 or rank-3 tiled map; dims/box innermost first, strides in bytes for
// dims 1.. (rank - 1 entries)
bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, int rank,
              const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
              CUtensorMapSwizzle swizzle)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t d[3], st[2];
    cuuint32_t b[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
    return enc(m, dt, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest number of groups one stage can touch.
int group_rows_per_stage(int64_t g)
{
    if (kStageRows % g == 0) return (int)(kStageRows / g);
    if (g % kStageRows == 0) return 1;
    return (int)((kStageRows - 1) / g + 2);
}

// The four tensor maps of a launch and the bytes one stage delivers.
bool build_maps(const Problem &pr, int mpad, CUtensorMap *tw, CUtensorMap *tx, CUtensorMap *ts,
                CUtensorMap *tz, uint32_t *stage_tx)
{
    const uint64_t K = (uint64_t)pr.K, N = (uint64_t)pr.N, M = (uint64_t)pr.M, G = (uint64_t)pr.G;
    const int R = group_rows_per_stage(pr.g);
    const uint64_t wd[2] = {N / 8, K}, ws[1] = {N / 2};
    const uint32_t wb[2] = {kTileWords, kStageRows};
    // x viewed as [M][K / 64][64]: one box covers a stage's 256 k for every token
    const uint64_t xd[3] = {64, K / 64, M}, xs[2] = {128, K * 2};
    const uint32_t xb[3] = {64, kKBlocks, (uint32_t)mpad};
    const uint64_t sd[2] = {N, G}, ss[1] = {N * 2};
    const uint32_t sb[2] = {kTileCols, (uint32_t)R};
    const uint64_t zd[2] = {N / 8, G}, zs[1] = {N / 2};
    const uint32_t zb[2] = {kTileWords, (uint32_t)R};
    *stage_tx = (uint32_t)(kWBytes + mpad * kStageRows * 2 + R * (kTileCols * 2) + R * (kTileWords * 4));
    return make_map(tw, CU_TENSOR_MAP_DATA_TYPE_INT32, pr.qweight, 2, wd, ws, wb, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pr.x, 3, xd, xs, xb, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pr.scales, 2, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           make_map(tz, CU_TENSOR_MAP_DATA_TYPE_INT32, pr.qzeros, 2, zd, zs, zb, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Per (device, kernel variant): dynamic shared memory opted in once, and the
// number of resident CTAs per SM with the SM count.
struct LaunchInfo {
    int occ = 0;
    int sms = 0;
    cudaError_t err = cudaSuccess;
};

template <int MT, int KG, bool WG>
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
    auto kern = decode_kernel<MT, KG, WG>;
    li.err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (li.err == cudaSuccess)
        li.err = cudaDeviceGetAttribute(&li.sms, cudaDevAttrMultiProcessorCount, dev);
    if (li.err == cudaSuccess)
        li.err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&li.occ, kern, Layout<KG>::kThreads, kSmemBytes);
    if (li.err == cudaSuccess && li.occ < 1) li.err = cudaErrorLaunchOutOfResources;
    if (li.err == cudaSuccess) cache[dev] = li;
    return li;
}

// Fills everything but the scratch pointers; the grid size goes to p->ctas.
template <int MT, int KG, bool WG>
cudaError_t prepare(const Problem &pr, int max_ctas, CUtensorMap *maps, DecodeParams *p)
{
    const LaunchInfo li = launch_info<MT, KG, WG>();
    if (li.err != cudaSuccess) return li.err;
    const int tiles = (int)((pr.N + kTileCols - 1) / kTileCols);
    const int kiters = (int)((pr.K + kStageRows - 1) / kStageRows);
    const int64_t total = (int64_t)tiles * kiters;
    const int ctas = (int)std::min<int64_t>(std::min<int64_t>(total, (int64_t)li.occ * li.sms), max_ctas);
    uint32_t stage_tx = 0;
    if (!build_maps(pr, 8 * MT, &maps[0], &maps[1], &maps[2], &maps[3], &stage_tx))
        return cudaErrorInvalidValue;
    *p = DecodeParams{};
    p->bias = static_cast<const __half *>(pr.bias);
    p->y = static_cast<__half *>(pr.y);
    p->status = device_status_word();
    p->M = (int)pr.M; p->K = (int)pr.K; p->N = (int)pr.N; p->g = (int)pr.g;
    p->tiles = tiles; p->kiters = kiters; p->total = (int)total; p->ctas = ctas;
    p->stage_tx = stage_tx;
    return cudaSuccess;
}

template <int MT, int KG, bool WG>
cudaError_t launch_kernel(const CUtensorMap *maps, const DecodeParams &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p.ctas);
    cfg.blockDim = dim3(Layout<KG>::kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    // programmatic dependent launch: the kernel starts streaming weights while
    // the previous kernel on the stream drains (it waits for it before
    // touching activations, bias, output or scratch)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<MT, KG, WG>, maps[0], maps[1], maps[2], maps[3], p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int MT, int KG, bool WG>
cudaError_t launch_decode_t(const Problem &pr, cudaStream_t stream)
{
    CUtensorMap maps[4];
    DecodeParams p;
    cudaError_t e = prepare<MT, KG, WG>(pr, 1 << 30, maps, &p);
    if (e != cudaSuccess) return e;
    Scratch sc{};
    if (!get_scratch(stream, (size_t)2 * p.ctas * kPartialFloats, (size_t)p.tiles, &sc))
        return cudaErrorMemoryAllocation;
    p.partials = sc.partials;
    p.arrive = sc.counters;
    return launch_kernel<MT, KG, WG>(maps, p, stream);
}

// Consumer k-groups. Two (8 consumer warps + the producer, up to 168
// registers a thread) ran a little faster than four (16 + 1 warps, held to
// 96 registers, which spilled at two token tiles) for every decode shape.
template <int MT> struct KGroupsFor { static constexpr int value = 2; };

// whole: g divides the rows each warp takes per stage into one group
template <int MT>
cudaError_t dispatch_decode(const Problem &p, cudaStream_t stream)
{
    constexpr int KG = KGroupsFor<MT>::value;
    const bool whole = p.g % Layout<KG>::kRowsPerWarp == 0;
    return whole ? launch_decode_t<MT, KG, true>(p, stream) : launch_decode_t<MT, KG, false>(p, stream);
}

} // namespace

bool decode_supported(int64_t M, int64_t K, int64_t N, int64_t g)
{
    return M >= 1 && M <= kMaxTokens && K % 64 == 0 && N % 32 == 0 && g % 16 == 0 &&
           group_rows_per_stage(g) <= kMaxGroupRows && K <= (int64_t(1) << 30) &&
           N <= (int64_t(1) << 30) &&
           ((K + kStageRows - 1) / kStageRows) * ((N + kTileCols - 1) / kTileCols) < (int64_t(1) << 31);
}

cudaError_t launch_decode(const Problem &p, cudaStream_t stream)
{
    if (!decode_supported(p.M, p.K, p.N, p.g)) return cudaErrorInvalidValue;
    return p.M <= 8 ? dispatch_decode<1>(p, stream) : dispatch_decode<2>(p, stream);
}

} // namespace awq

// ---------------------------------------------------------------------------
// Allocation-free entry point: the decode kernel above, with its split-K
// scratch taken from a fixed array compiled into this library instead of
// memory the library allocates. The page has no counterpart of this call.
// ---------------------------------------------------------------------------

#include "../../include/awq_gb300.h"

namespace awq {
namespace {

constexpr int kNoAllocMaxCtas = 160;    // grid cap: partial slots for 160 CTAs
constexpr int kNoAllocMaxTiles = 8192;  // 256-column tiles: N up to 2,097,152
constexpr size_t kNoAllocPartialWords = (size_t)2 * kNoAllocMaxCtas * kPartialFloats;
constexpr size_t kNoAllocWords = kNoAllocPartialWords + (size_t)kNoAllocMaxTiles;

// fp32 partials (2 slots per CTA) followed by the arrival counter of every
// tile: 5,242,880 + 32,768 bytes on every GPU that loads this library, for as
// long as the library stays loaded.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocWords];

// Device address of g_noalloc_scratch on the current device. Host code only
// holds a stand-in for the symbol, so the address is looked up once per
// device (with that device current) and cached.
cudaError_t noalloc_scratch_address(uint32_t **out)
{
    static std::mutex mu;
    static std::map<int, uint32_t *> addr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    auto it = addr.find(dev);
    if (it != addr.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    uint32_t *ptr = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = ptr;
    *out = ptr;
    return cudaSuccess;
}

template <int MT, int KG, bool WG>
cudaError_t launch_decode_noalloc_t(const Problem &pr, cudaStream_t stream, uint32_t *scratch)
{
    CUtensorMap maps[4];
    DecodeParams p;
    cudaError_t e = prepare<MT, KG, WG>(pr, kNoAllocMaxCtas, maps, &p);
    if (e != cudaSuccess) return e;
    p.partials = reinterpret_cast<float *>(scratch);
    p.arrive = scratch + kNoAllocPartialWords;
    // the array keeps whatever the previous call left: the counters must
    // start at zero (the partial slots are always written before being read)
    e = cudaMemsetAsync(p.arrive, 0, sizeof(uint32_t) * (size_t)p.tiles, stream);
    if (e != cudaSuccess) return e;
    return launch_kernel<MT, KG, WG>(maps, p, stream);
}

template <int MT>
cudaError_t dispatch_noalloc(const Problem &p, cudaStream_t stream, uint32_t *scratch)
{
    constexpr int KG = KGroupsFor<MT>::value;
    const bool whole = p.g % Layout<KG>::kRowsPerWarp == 0;
    return whole ? launch_decode_noalloc_t<MT, KG, true>(p, stream, scratch)
                 : launch_decode_noalloc_t<MT, KG, false>(p, stream, scratch);
}

bool aligned16_ptr(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

} // namespace
} // namespace awq

extern "C" awq_status_t awq_linear_forward_decode_noalloc(
    const void *x, const int32_t *qweight, const int32_t *qzeros, const void *scales,
    const void *bias, void *y, int64_t M, int64_t K, int64_t N, int64_t group_size,
    awq_stream_t stream)
{
    if (M < 0 || K <= 0 || N <= 0 || N % 8 != 0 || group_size == 0 || group_size < -1)
        return AWQ_ERR_INVALID_ARG;
    const int64_t g = (group_size == -1) ? K : group_size;
    if (K % g != 0) return AWQ_ERR_INVALID_ARG;
    if (M == 0) return AWQ_OK;
    if (!x || !qweight || !qzeros || !scales || !y) return AWQ_ERR_INVALID_ARG;
    if (!awq::aligned16_ptr(x) || !awq::aligned16_ptr(qweight) || !awq::aligned16_ptr(qzeros) ||
        !awq::aligned16_ptr(scales) || !awq::aligned16_ptr(y) || (bias && !awq::aligned16_ptr(bias)))
        return AWQ_ERR_MISALIGNED;
    if (!awq::decode_supported(M, K, N, g)) return AWQ_ERR_INVALID_ARG;
    if ((N + awq::kTileCols - 1) / awq::kTileCols > awq::kNoAllocMaxTiles) return AWQ_ERR_TOO_LARGE;
    uint32_t *scratch = nullptr;
    if (awq::noalloc_scratch_address(&scratch) != cudaSuccess) return AWQ_ERR_CUDA;
    awq::Problem p{x, qweight, qzeros, scales, bias, y, M, K, N, g, K / g};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = (M <= 8) ? awq::dispatch_noalloc<1>(p, s, scratch)
                                   : awq::dispatch_noalloc<2>(p, s, scratch);
    return e == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA;
}
