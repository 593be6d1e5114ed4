// awq_decode.cu -- decode path of the WQLinear forward (small M, 1..32 rows).
//
// Predibase Lorax "AWQ WQLinear" page, Description, forward steps 2-3:
//   y[m, n] = fp16_rn( sum_k x[m, k] * W[k, n] + bias[n] ),
//   W[k, n] = fp16_rn((q[k, n] - z[k/g, n]) * s[k/g, n]), fp32 accumulation.
//
// At small M the layer is bound by streaming the packed weights from HBM
// (0.52 bytes per weight at g = 128). The kernel is built around that:
//
//  * Work: the K x N weight matrix is cut into column tiles of CW 128-byte
//    chunks of packed words (CW = 1: 256 columns; CW = 2: 512 columns, used
//    when N is a multiple of 512 and at least 32768) and stages of 32 KB of
//    packed weights (256 / CW k-rows). The (tile, stage) iterations,
//    tile-major, are split evenly between the CTAs (one per SM): each CTA
//    streams a contiguous run of them ("stream-K"). Rows 256 bytes wide keep
//    HBM reads of large matrices ~20 % closer to the copy bandwidth than
//    128-byte rows; on small N the narrower tile keeps split-K short.
//  * Loads: thread 0 issues four TMA boxes per stage -- the qweight slice
//    (32 KB, 128-byte swizzle), the activation slice (one 3-D box), and the
//    scale and zero-point rows of the groups the stage touches -- into a ring
//    of as many stages as shared memory holds (5-6 at g = 128), guarded by
//    mbarriers (full: bytes landed; empty: every warp released the slot).
//    All but one slot are in flight ahead of the stage being computed; after
//    each stage thread 0 refills the slot released one stage earlier, so it
//    seldom waits. Issuing a TMA instruction costs on the order of a hundred
//    cycles, so each one moves as many bytes as the box limits allow.
//  * Math: 8 warps, each taking 128 rows x 64 columns of every stage (eight
//    16-row chunks): 2 / CW k-groups of 4 CW column warps. Each warp
//    dequantises in registers and runs the legacy-path tensor-core MMA
//    m16n8k16 with W as the A operand (16 output columns x 16 k) and the
//    activations as B (16 k x 8 tokens), fp32 accumulators; M is padded to
//    1, 2 or 4 such token tiles, each costing one MMA per A operand (eight
//    tiles would need more registers than a thread of this 9-warp CTA gets:
//    three warps share one sub-partition, 168 registers each). Two k-adjacent
//    weights of one column form one half2 operand register: a byte permute
//    brings byte b of rows k and k+1 together, one LOP3 masks a nibble into
//    the fraction of 1024.0 or 64.0, an exact half2 subtract removes the zero
//    point and one half2 multiply (round to nearest) applies the scale --
//    exactly fp16_rn((q - z) s). At the end of a tile's run the k-groups are
//    summed in a fixed order through the weight area of the slot just
//    consumed, which is released afterwards.
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
// Requirements (else another path serves): 1 <= M <= 32, K % 64 == 0,
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

constexpr int kMaxTokens = 32;
constexpr int kMaxGroupRows = 8;     // group rows one stage may touch
constexpr int kWBytes = 32768;       // packed weights per stage
constexpr int kMaxStages = 8;
// Warps that dequantise and multiply (plus one TMA producer warp), by the
// number MT of 8-token tiles: more warps per SM sub-partition hide more of
// the load and instruction latencies; a thread of a CTA of W warps gets at
// most 65536 / (32 W) registers.
constexpr int kConsumerWarpsOneTile = 8;
template <int MT>
struct Warps {
    static constexpr int kConsumer = MT == 1 ? kConsumerWarpsOneTile : 8;
    static constexpr int kConsumerThreads = kConsumer * 32;
    static constexpr int kThreads = kConsumerThreads + 32;
};
constexpr int kBarBytes = 2 * kMaxStages * 8 + 64;   // full/empty barriers + flags
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMaxTileCols = 512;
constexpr int kMaxPartialFloats = kMaxTokens * kMaxTileCols;  // one partial slot

// Tile geometry for CW 128-byte chunks of packed words per weight row and
// NW consumer warps.
template <int CW, int NW = 8>
struct Geo {
    static constexpr int kTileWords = 32 * CW;
    static constexpr int kTileCols = 256 * CW;
    static constexpr int kStageRows = kWBytes / (kTileWords * 4);
    static constexpr int kKBlocks = kStageRows / 64;     // 64-row blocks of a stage
    static constexpr int kColWarps = 4 * CW;                      // warps across a tile (64 columns each)
    static constexpr int kKGroups = NW / kColWarps;               // warps down a stage
    static constexpr int kRowsPerWarp = kStageRows / kKGroups;    // 128
    static constexpr int kChunksPerWarp = kRowsPerWarp / 16;
    static_assert(kKGroups * kRowsPerWarp == kStageRows, "warps must cover a stage");
};
// The fp32 sums of every k-group but the first, 16 MT floats per thread,
// fit the weight area (32 KB) of the slot they are folded through.
template <int MT, int CW>
constexpr bool fold_fits()
{
    using G = Geo<CW, Warps<MT>::kConsumer>;
    return (G::kKGroups - 1) * 16 * MT * G::kColWarps * 32 * 4 <= kWBytes;
}
static_assert(fold_fits<1, 1>() && fold_fits<2, 1>() && fold_fits<4, 1>() && fold_fits<1, 2>() &&
                  fold_fits<2, 2>() && fold_fits<4, 2>(), "fold buffer fits a slot");

struct DecodeParams {
    const __half *bias;
    __half *y;
    float *y32;             // if set: y32 += the fp32 sums (no bias, no rounding) instead of y
    float *partials;        // [2 * ctas][8 MT][tile columns]
    unsigned int *arrive;   // [tiles]
    unsigned int *status;
    int M, K, N, g;
    int tiles, kiters, total, ctas;
    int stages;             // ring slots
    uint32_t stage_bytes;   // bytes per slot (multiple of 1024)
    uint32_t x_off, s_off, z_off;  // activation / scale / zero rows inside a slot
    uint32_t stage_tx;      // bytes one stage's TMA boxes deliver
#ifdef AWQ_FAULT_TEST
    int fault;              // CTA 0's producer issues nothing (fault-test build only)
#endif
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

// One k-group's accumulators to / from shared memory; STRIDE = threads of a
// k-group, so that consecutive threads touch consecutive words.
template <int MT, int STRIDE>
__device__ __forceinline__ void fold_store(float *dst, const float (&acc)[4][MT][4], int ct) {
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[((b * MT + mt) * 4 + e) * STRIDE + ct] = acc[b][mt][e];
}
template <int MT, int STRIDE>
__device__ __forceinline__ void fold_add(const float *src, float (&acc)[4][MT][4], int ct) {
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[b][mt][e] += src[((b * MT + mt) * 4 + e) * STRIDE + ct];
}

template <int MT, int CW, bool kWholeGroups>
__global__ void __launch_bounds__(Warps<MT>::kThreads, 1)
decode_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
              const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
              const DecodeParams p)
{
    constexpr int kConsumerWarps = Warps<MT>::kConsumer;
    constexpr int kConsumerThreads = Warps<MT>::kConsumerThreads;
    using G = Geo<CW, kConsumerWarps>;
    constexpr int kTileCols = G::kTileCols;
    constexpr int kTileWords = G::kTileWords;
    constexpr int kStageRows = G::kStageRows;
    constexpr int kKBlocks = G::kKBlocks;
    constexpr int kColWarps = G::kColWarps;
    constexpr int KG = G::kKGroups;
    constexpr int kChunksPerWarp = G::kChunksPerWarp;
    constexpr int kRowsPerWarp = G::kRowsPerWarp;
    constexpr int kKGroupThreads = kColWarps * 32;
    constexpr int kSlotFloats = 8 * MT * kTileCols;   // one partial: 8 MT tokens x the tile

    extern __shared__ uint8_t smem_raw[];
    // round up to 1024 bytes by offsetting the shared array itself, so that
    // the compiler still knows every derived pointer is a shared address
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages;
    const uint32_t SB = p.stage_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (uint32_t)S * SB);
    uint64_t *empty = full + kMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kMaxStages);
    volatile int *duty_ok = abort_flag + 1;
    volatile int *go = abort_flag + 2;
    volatile uint32_t *consts = reinterpret_cast<volatile uint32_t *>(abort_flag + 3);

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
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(ptx::smem_addr(full + s), 1);
            ptx::mbar_init(ptx::smem_addr(empty + s), kConsumerWarps);
        }
        *abort_flag = 0;
        *duty_ok = 0;
        *go = 0;
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
            int slot = 0, round = 0;
            auto issue_weights = [&]() {
                const uint32_t fb = ptx::smem_addr(full + slot);
                const uint32_t st = ptx::smem_addr(smem + (uint32_t)slot * SB);
                const int k0 = kb * kStageRows;
                const int grp0 = k0 / p.g;
                ptx::mbar_arrive_expect_tx(fb, p.stage_tx);
                if (CW == 1) {
                    ptx::tma_load_2d(st, &tm_w, fb, tile * kTileWords, k0);
                    ptx::tma_load_2d(st + p.s_off, &tm_s, fb, tile * kTileCols, grp0);
                    ptx::tma_load_2d(st + p.z_off, &tm_z, fb, tile * kTileWords, grp0);
                } else {
                    ptx::tma_load_3d(st, &tm_w, fb, 0, tile * CW, k0);
                    ptx::tma_load_3d(st + p.s_off, &tm_s, fb, 0, tile * CW, grp0);
                    ptx::tma_load_3d(st + p.z_off, &tm_z, fb, 0, tile * CW, grp0);
                }
            };
            auto issue_x = [&](int sl, int kbx) {
                ptx::tma_load_3d(ptx::smem_addr(smem + (uint32_t)sl * SB + p.x_off), &tm_x,
                                 ptx::smem_addr(full + sl), 0, 0, kbx * kKBlocks);
            };
            auto advance = [&]() {
                if (++kb == p.kiters) { kb = 0; ++tile; }
                if (++slot == S) { slot = 0; ++round; }
            };
            // The weights, scales and zero points of the first S stages do
            // not depend on the kernel before this one: load them while it
            // finishes, and the activations once it has.
            int pre = n_iters < S ? n_iters : S;
#ifdef AWQ_FAULT_TEST
            // injected fault: nothing is loaded, so the consumers' bounded
            // waits on the first stage run out
            if (p.fault && c == 0) {
                ptx::wait_prerequisites();
                return;
            }
#endif
            const int kb_first = kb;
            for (int i = 0; i < pre; ++i) {
                issue_weights();
                advance();
            }
            ptx::wait_prerequisites();
            for (int i = 0, kx = kb_first; i < pre; ++i) {
                issue_x(i, kx);
                if (++kx == p.kiters) kx = 0;
            }
            int issued = pre;
            for (int i = pre; i < n_iters; ++i) {
                if (!ptx::mbar_wait_bounded(ptx::smem_addr(empty + slot), (uint32_t)((round - 1) & 1),
                                            abort_flag, p.status))
                    break;
                issue_weights();
                issue_x(slot, kb);
                advance();
                issued = i + 1;
            }
            if (*abort_flag) {
                // let the copies already in flight land before the CTA's
                // shared memory is released
                for (int i = std::max(0, issued - S); i < issued; ++i)
                    ptx::mbar_wait_bounded(ptx::smem_addr(full + i % S), (uint32_t)((i / S) & 1), nullptr,
                                           nullptr);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    // everything below reads or writes global memory the kernel before this
    // one may still use (activations come through the producer, which waited)
    ptx::wait_prerequisites();
    const int kg = warp / kColWarps;   // rows 128 kg .. 128 kg + 127 of every stage
    const int cw = warp % kColWarps;   // which 64 columns of the tile
    const int gq = lane >> 2;          // MMA groupID: output column pair / token
    const int tq = lane & 3;           // MMA thread-in-group: k pair / token pair
    const int word = cw * 8 + gq;      // packed word (8 columns) of the tile this thread owns
    const int ct = cw * 32 + lane;     // thread index within a k-group

    // Byte offsets of this thread's packed words inside a slot. The weight
    // area is [row][CW chunks][128 bytes]; 128-byte segment q = row * CW +
    // chunk holds its 16-byte unit u at unit u ^ (q % 8). Chunk j of this
    // warp is rows R0 + 16 j .. +15 (R0 = 128 kg); the thread reads rows
    // 2tq, 2tq + 1 and the same + 8 (one 8-row step keeps q % 8).
    const int R0 = kRowsPerWarp * kg;
    const uint32_t chunk = (uint32_t)(word >> 5);
    const uint32_t wic = (uint32_t)(word & 31);
    const uint32_t unit = wic >> 2;
    const uint32_t inw = (wic & 3) * 4;
    const uint32_t qA = (uint32_t)(2 * tq) * CW + chunk, qB = (uint32_t)(2 * tq + 1) * CW + chunk;
    const uint32_t rowbase = (uint32_t)R0 * (CW * 128);
    const uint32_t offA = rowbase + qA * 128 + ((unit ^ (qA & 7)) << 4) + inw;
    const uint32_t offB = rowbase + qB * 128 + ((unit ^ (qB & 7)) << 4) + inw;
    constexpr uint32_t kChunkStride = 16 * CW * 128;   // 16 rows
    constexpr uint32_t kRow8 = 8 * CW * 128;           // 8 rows
    // activation slice: [64-row block][token m][64 halves], 128-byte rows
    // (r = block * 8 MT + m), 16-byte unit u of row r stored at unit
    // u ^ (r % 8). Chunk j of this warp is block R0 / 64 + j / 4, units
    // 2 (j % 4) and 2 (j % 4) + 1 -- the k 0..7 and 8..15 halves of its B
    // operand. One ldmatrix.x4 fetches the B operands of a chunk pair for
    // eight tokens: lane L addresses token L % 8, unit 4 * pair + L / 8. The
    // eight rows of one 8 x 8 matrix are eight consecutive tokens, so r % 8
    // takes every value once and the eight 16-byte reads fall in distinct
    // banks. Token tile mt adds 8 rows, which keeps r % 8.
    constexpr int kBlocksPerWarp = kChunksPerWarp / 4;
    static_assert(kChunksPerWarp % 4 == 0, "whole 64-row activation blocks per warp and stage");
    constexpr uint32_t kXTokenTile = 8 * 128;
    uint32_t xoff[kBlocksPerWarp][2];
#pragma unroll
    for (int jb = 0; jb < kBlocksPerWarp; ++jb) {
        const uint32_t r = (uint32_t)((R0 / 64 + jb) * (8 * MT) + (lane & 7));
#pragma unroll
        for (int pr = 0; pr < 2; ++pr)
            xoff[jb][pr] = p.x_off + r * 128 + (((uint32_t)(4 * pr + (lane >> 3)) ^ (r & 7)) << 4);
    }
    const uint32_t soff = p.s_off + (uint32_t)word * 16;
    const uint32_t zoff = p.z_off + (uint32_t)word * 4;
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
    int slot = 0;
    uint32_t phase = 0;

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
        uint8_t *stp = smem + (uint32_t)slot * SB;
        // every lane waits (each needs the acquire); the MMA below is
        // warp-wide, so the outcome is made uniform across the warp
        const bool ok = __all_sync(0xffffffffu,
                                   ptx::mbar_wait_bounded(ptx::smem_addr(full + slot), phase,
                                                          abort_flag, p.status));
        if (ok && k0 + R0 < p.K) {
            if (kWholeGroups) {
                // g % 128 == 0: the warp's rows lie in one group
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
                const uint8_t *wp = stp + j * kChunkStride;
                const uint32_t v0 = *reinterpret_cast<const uint32_t *>(wp + offA);
                const uint32_t v1 = *reinterpret_cast<const uint32_t *>(wp + offB);
                const uint32_t v8 = *reinterpret_cast<const uint32_t *>(wp + offA + kRow8);
                const uint32_t v9 = *reinterpret_cast<const uint32_t *>(wp + offB + kRow8);
                if ((j & 1) == 0) {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        ptx::ldmatrix_x4(sbase + xoff[j / 4][(j % 4) / 2] + mt * kXTokenTile, xq[mt]);
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
        const bool seg_end = (i == n_iters - 1 || kb == p.kiters - 1);
        if (!seg_end || KG == 1) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(empty + slot));
        }

        if (seg_end) {
            if (KG >= 2) {
                // ---- fold k-groups 1 .. KG - 1 into k-group 0, in that order,
                //      through this slot's weight area (every warp has
                //      finished reading it at the first barrier), then
                //      release the slot
                float *red = reinterpret_cast<float *>(stp);
                constexpr int kRegion = 16 * MT * kKGroupThreads;
                ptx::named_barrier(1, kConsumerThreads);
                if (kg >= 1) fold_store<MT, kKGroupThreads>(red + (kg - 1) * kRegion, acc, ct);
                ptx::named_barrier(1, kConsumerThreads);
                if (kg == 0) {
#pragma unroll
                    for (int q = 1; q < KG; ++q) fold_add<MT, kKGroupThreads>(red + (q - 1) * kRegion, acc, ct);
                }
                // generic-proxy accesses to the slot are ordered before the
                // TMA writes that refill it
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(empty + slot));
            }

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
                                if (p.y32) {
                                    float4 *d = reinterpret_cast<float4 *>(p.y32 + (int64_t)m * p.N + col0);
                                    float4 lo = d[0], hi = d[1];
                                    lo.x += acc[0][mt][e]; lo.y += acc[0][mt][2 + e];
                                    lo.z += acc[1][mt][e]; lo.w += acc[1][mt][2 + e];
                                    hi.x += acc[2][mt][e]; hi.y += acc[2][mt][2 + e];
                                    hi.z += acc[3][mt][e]; hi.w += acc[3][mt][2 + e];
                                    d[0] = lo;
                                    d[1] = hi;
                                    continue;
                                }
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
                    float *pslot = p.partials + (int64_t)(2 * c + which) * kSlotFloats;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int m = 8 * mt + 2 * tq + e;
                            if (m < p.M) {
                                float4 lo = make_float4(acc[0][mt][e], acc[0][mt][2 + e], acc[1][mt][e], acc[1][mt][2 + e]);
                                float4 hi = make_float4(acc[2][mt][e], acc[2][mt][2 + e], acc[3][mt][e], acc[3][mt][2 + e]);
                                float4 *dst = reinterpret_cast<float4 *>(pslot + m * kTileCols + word * 8);
                                dst[0] = lo;
                                dst[1] = hi;
                            }
                        }
                    __threadfence();
                }
                if (!whole) {
                    ptx::named_barrier(2, kKGroupThreads);
                    // count in with the tile's finisher (not needed for its own tile)
                    if (ct == 0 && !*abort_flag && !(reducer && tile == first_tile))
                        atomicAdd(p.arrive + tile, 1u);
                }
            }
        }
        if (++kb == p.kiters) { kb = 0; ++tile; }
        if (++slot == S) { slot = 0; phase ^= 1u; }
    }

    // One consumer thread decides, for all of them, whether the CTA goes on
    // (the producer may still set the abort flag while the others read it).
    const int ctid = threadIdx.x;   // 0 .. kConsumerThreads - 1
    ptx::named_barrier(1, kConsumerThreads);
    if (ctid == 0) *go = *abort_flag ? 0 : 1;
    ptx::named_barrier(1, kConsumerThreads);
    if (!*go) return;

    // ---- finishing the split tile this range starts in: wait for the other
    //      contributors (lower-numbered CTAs) to count in, then sum every
    //      partial, its own included, in contributor order, so the result
    //      does not depend on timing; add the bias and round once.
    if (!reducer) return;
    const int t = first_tile;
    const int cf = cta_of(t * p.kiters, p.total, p.ctas);
    const int n = c - cf + 1;
    if (ctid == 0) {
        bool ok = true;
        const long long t0 = clock64();
        while (ptx::ld_acquire_gpu(p.arrive + t) < (unsigned)(n - 1)) {
            if (clock64() - t0 > ptx::kWaitLimitCycles) {
                ok = false;
                atomicOr(p.status, kStatusTimeout);
                break;
            }
            __nanosleep(32);
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
    constexpr int kPosPerThread = (8 * MT * kTileCols / 4 + kConsumerThreads - 1) / kConsumerThreads;
    const int n4 = p.M * (kTileCols / 4);   // float4 positions of one partial
    const int per_round = (int)(((uint32_t)S * SB) / (uint32_t)(n4 * 16));
    const uint32_t ring = ptx::smem_addr(smem);
    float4 acc4[kPosPerThread];
#pragma unroll
    for (int k = 0; k < kPosPerThread; ++k) acc4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r0 = 0; r0 < n; r0 += per_round) {
        const int cnt = std::min(per_round, n - r0);
        for (int q = 0; q < cnt; ++q) {
            const int ci = cf + r0 + q;
            const float *src = p.partials + (int64_t)(2 * ci + (ci == cf ? which_cf : 0)) * kSlotFloats;
#pragma unroll
            for (int k = 0; k < kPosPerThread; ++k) {
                const int pos = ctid + k * kConsumerThreads;
                if (pos < n4)
                    ptx::cp_async_16(ring + (uint32_t)(q * n4 + pos) * 16,
                                     src + (pos / (kTileCols / 4)) * kTileCols + (pos % (kTileCols / 4)) * 4);
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
        if (col >= p.N) continue;
        if (p.y32) {
            float4 *d = reinterpret_cast<float4 *>(p.y32 + (int64_t)m * p.N + col);
            float4 v = *d;
            v.x += acc4[k].x; v.y += acc4[k].y; v.z += acc4[k].z; v.w += acc4[k].w;
            *d = v;
            continue;
        }
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

// Largest number of groups a stage of `rows` k-rows can touch.
int group_rows_per_stage(int64_t g, int rows)
{
    if (rows % g == 0) return (int)(rows / g);
    if (g % rows == 0) return 1;
    return (int)((rows - 1) / g + 2);
}

// The tensor maps of a launch and the slot layout. CW = 1 uses 2-D maps
// (any N % 32 == 0; the last tile reads past N as zeros); CW = 2 views the
// row-major arrays as [rows][N / 256][256 columns] (N % 512 == 0).
template <int CW>
bool build_maps(const Problem &pr, int mpad, CUtensorMap *tw, CUtensorMap *tx, CUtensorMap *ts,
                CUtensorMap *tz, DecodeParams *p)
{
    using G = Geo<CW>;
    const uint64_t K = (uint64_t)pr.K, N = (uint64_t)pr.N, M = (uint64_t)pr.M, Gn = (uint64_t)pr.G;
    const int R = group_rows_per_stage(pr.g, G::kStageRows);
    // x viewed as [K / 64][M][64] (a 64-column block of every token, block
    // by block): one box covers a stage's k for every token, stored block
    // by block in shared memory
    const uint64_t ldx = pr.ldx > 0 ? (uint64_t)pr.ldx : K;
    const uint64_t xd[3] = {64, M, K / 64}, xs[2] = {ldx * 2, 128};
    const uint32_t xb[3] = {64, (uint32_t)mpad, (uint32_t)G::kKBlocks};
    bool ok = make_map(tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pr.x, 3, xd, xs, xb, CU_TENSOR_MAP_SWIZZLE_128B);
    if (CW == 1) {
        const uint64_t wd[2] = {N / 8, K}, ws[1] = {N / 2};
        const uint32_t wb[2] = {(uint32_t)G::kTileWords, (uint32_t)G::kStageRows};
        const uint64_t sd[2] = {N, Gn}, ss[1] = {N * 2};
        const uint32_t sb[2] = {(uint32_t)G::kTileCols, (uint32_t)R};
        const uint64_t zd[2] = {N / 8, Gn}, zs[1] = {N / 2};
        const uint32_t zb[2] = {(uint32_t)G::kTileWords, (uint32_t)R};
        ok = ok && make_map(tw, CU_TENSOR_MAP_DATA_TYPE_INT32, pr.qweight, 2, wd, ws, wb, CU_TENSOR_MAP_SWIZZLE_128B) &&
             make_map(ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pr.scales, 2, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE) &&
             make_map(tz, CU_TENSOR_MAP_DATA_TYPE_INT32, pr.qzeros, 2, zd, zs, zb, CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
        const uint64_t wd[3] = {32, N / 256, K}, ws[2] = {128, N / 2};
        const uint32_t wb[3] = {32, (uint32_t)CW, (uint32_t)G::kStageRows};
        const uint64_t sd[3] = {256, N / 256, Gn}, ss[2] = {512, N * 2};
        const uint32_t sb[3] = {256, (uint32_t)CW, (uint32_t)R};
        const uint64_t zd[3] = {32, N / 256, Gn}, zs[2] = {128, N / 2};
        const uint32_t zb[3] = {32, (uint32_t)CW, (uint32_t)R};
        ok = ok && make_map(tw, CU_TENSOR_MAP_DATA_TYPE_INT32, pr.qweight, 3, wd, ws, wb, CU_TENSOR_MAP_SWIZZLE_128B) &&
             make_map(ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pr.scales, 3, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE) &&
             make_map(tz, CU_TENSOR_MAP_DATA_TYPE_INT32, pr.qzeros, 3, zd, zs, zb, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    // slot: weights | activations | scale rows | zero rows, 1024-aligned
    const uint32_t xbytes = (uint32_t)(mpad * G::kStageRows * 2);
    const uint32_t sbytes = (uint32_t)(R * G::kTileCols * 2);
    const uint32_t zbytes = (uint32_t)(R * G::kTileWords * 4);
    p->x_off = kWBytes;
    p->s_off = p->x_off + xbytes;
    p->z_off = p->s_off + sbytes;
    p->stage_bytes = (p->z_off + zbytes + 1023u) & ~1023u;
    p->stages = std::min<int>(kMaxStages, (kSmemLimit - kBarBytes - 1024) / (int)p->stage_bytes);
    p->stage_tx = kWBytes + xbytes + sbytes + zbytes;
    return ok && p->stages >= 2;
}

uint32_t smem_bytes(const DecodeParams &p) { return (uint32_t)p.stages * p.stage_bytes + kBarBytes + 1024; }

// Per (device, kernel variant): dynamic shared memory opted in once, and the
// SM count.
struct LaunchInfo {
    int sms = 0;
    cudaError_t err = cudaSuccess;
    unsigned gen = 0;   // cache generation this was set up in
};

template <int MT, int CW, bool WG>
LaunchInfo launch_info()
{
    static std::mutex mu;
    static std::map<int, LaunchInfo> cache;
    int dev = 0;
    LaunchInfo li;
    li.err = cudaGetDevice(&dev);
    if (li.err != cudaSuccess) return li;
    const unsigned gen = cache_generation();
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end() && it->second.gen == gen) return it->second;
    li.gen = gen;
    auto kern = decode_kernel<MT, CW, WG>;
    constexpr int kThreads = Warps<MT>::kThreads;
    li.err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (li.err == cudaSuccess)
        li.err = cudaDeviceGetAttribute(&li.sms, cudaDevAttrMultiProcessorCount, dev);
    int occ = 0;
    if (li.err == cudaSuccess)
        li.err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, kSmemLimit);
    if (li.err == cudaSuccess && occ < 1) li.err = cudaErrorLaunchOutOfResources;
    if (li.err == cudaSuccess) cache[dev] = li;
    return li;
}

// Fills everything but the scratch pointers; the grid size goes to p->ctas
// (one CTA per SM).
template <int MT, int CW, bool WG>
cudaError_t prepare(const Problem &pr, int max_ctas, CUtensorMap *maps, DecodeParams *p)
{
    using G = Geo<CW>;
    const LaunchInfo li = launch_info<MT, CW, WG>();
    if (li.err != cudaSuccess) return li.err;
    const int tiles = (int)((pr.N + G::kTileCols - 1) / G::kTileCols);
    const int kiters = (int)((pr.K + G::kStageRows - 1) / G::kStageRows);
    const int64_t total = (int64_t)tiles * kiters;
    const int ctas = (int)std::min<int64_t>(std::min<int64_t>(total, (int64_t)li.sms), max_ctas);
    *p = DecodeParams{};
    if (!build_maps<CW>(pr, 8 * MT, &maps[0], &maps[1], &maps[2], &maps[3], p))
        return cudaErrorInvalidValue;
    p->bias = static_cast<const __half *>(pr.bias);
    p->y = static_cast<__half *>(pr.y);
    p->y32 = pr.y32;
    p->status = device_status_word();
    p->M = (int)pr.M; p->K = (int)pr.K; p->N = (int)pr.N; p->g = (int)pr.g;
    p->tiles = tiles; p->kiters = kiters; p->total = (int)total; p->ctas = ctas;
#ifdef AWQ_FAULT_TEST
    p->fault = fault_injection();
#endif
    return cudaSuccess;
}

template <int MT, int CW, bool WG>
cudaError_t launch_kernel(const CUtensorMap *maps, const DecodeParams &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p.ctas);
    cfg.blockDim = dim3(Warps<MT>::kThreads);
    cfg.dynamicSmemBytes = smem_bytes(p);
    cfg.stream = stream;
    // programmatic dependent launch: the kernel starts streaming weights while
    // the previous kernel on the stream drains (it waits for it before
    // touching activations, bias, output or scratch)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<MT, CW, WG>, maps[0], maps[1], maps[2], maps[3], p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int MT, int CW, bool WG>
cudaError_t launch_decode_t(const Problem &pr, cudaStream_t stream)
{
    CUtensorMap maps[4];
    DecodeParams p;
    cudaError_t e = prepare<MT, CW, WG>(pr, 1 << 30, maps, &p);
    if (e != cudaSuccess) return e;
    Scratch sc{};
    // sized for the widest tile, so that the area never grows between the
    // first call on a stream and a later graph capture of other shapes
    if (!get_scratch(stream, (size_t)2 * p.ctas * kMaxPartialFloats, (size_t)p.tiles, &sc))
        return cudaErrorMemoryAllocation;
    p.partials = sc.partials;
    p.arrive = sc.counters;
    return launch_kernel<MT, CW, WG>(maps, p, stream);
}

// Tile width: 512 columns for very wide matrices (rows 256 bytes wide read
// HBM closer to its copy bandwidth: 3-5 % faster at N = 57344), 256 otherwise
// (fewer CTAs share a tile, so split-K finishing stays short; 512-column
// tiles measured 2-10 % slower at N = 10240..22016).
bool wide_tiles(int64_t N) { return N % 512 == 0 && N >= 32768; }

// whole: every warp's 128 rows of a stage lie in one group
template <int MT>
cudaError_t dispatch_decode(const Problem &p, cudaStream_t stream)
{
    const bool whole = p.g % 128 == 0;
    if (wide_tiles(p.N))
        return whole ? launch_decode_t<MT, 2, true>(p, stream) : launch_decode_t<MT, 2, false>(p, stream);
    return whole ? launch_decode_t<MT, 1, true>(p, stream) : launch_decode_t<MT, 1, false>(p, stream);
}

} // namespace

bool decode_supported(int64_t M, int64_t K, int64_t N, int64_t g)
{
    return M >= 1 && M <= kMaxTokens && K % 64 == 0 && N % 32 == 0 && g % 16 == 0 &&
           group_rows_per_stage(g, Geo<1>::kStageRows) <= kMaxGroupRows && K <= (int64_t(1) << 30) &&
           N <= (int64_t(1) << 30) &&
           ((K + Geo<1>::kStageRows - 1) / Geo<1>::kStageRows) * ((N + Geo<1>::kTileCols - 1) / Geo<1>::kTileCols) <
               (int64_t(1) << 30);
}

size_t decode_partial_floats_max(int sms) { return (size_t)2 * (size_t)sms * kMaxPartialFloats; }

int decode_tile_columns(int64_t M, int64_t K, int64_t N, int64_t g)
{
    if (!decode_supported(M, K, N, g)) return 0;
    return wide_tiles(N) ? Geo<2>::kTileCols : Geo<1>::kTileCols;
}

cudaError_t launch_decode(const Problem &p, cudaStream_t stream)
{
    if (!decode_supported(p.M, p.K, p.N, p.g)) return cudaErrorInvalidValue;
    // token tiles of 8: one MMA per 16 columns x 16 k and tile
    if (p.M <= 8) return dispatch_decode<1>(p, stream);
    if (p.M <= 16) return dispatch_decode<2>(p, stream);
    return dispatch_decode<4>(p, stream);
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
constexpr int kNoAllocMaxTokens = 16;   // partial slots hold 16 tokens x 256 columns
constexpr size_t kNoAllocPartialWords = (size_t)2 * kNoAllocMaxCtas * kNoAllocMaxTokens * Geo<1>::kTileCols;
constexpr size_t kNoAllocWords = kNoAllocPartialWords + (size_t)kNoAllocMaxTiles;

// fp32 partials (2 slots per CTA) followed by the arrival counter of every
// tile: 5,242,880 + 32,768 bytes on every GPU that loads this library, for as
// long as the library stays loaded.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocWords];

// Device address of g_noalloc_scratch on the current device. Host code only
// holds a stand-in for the symbol, so the address is looked up once per
// device (with that device current) and cached until awq_shutdown().
cudaError_t noalloc_scratch_address(uint32_t **out)
{
    static std::mutex mu;
    static std::map<int, std::pair<uint32_t *, unsigned>> addr;   // device -> (address, generation)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned gen = cache_generation();
    std::lock_guard<std::mutex> lock(mu);
    auto it = addr.find(dev);
    if (it != addr.end() && it->second.second == gen) {
        *out = it->second.first;
        return cudaSuccess;
    }
    uint32_t *ptr = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = std::make_pair(ptr, gen);
    *out = ptr;
    return cudaSuccess;
}

template <int MT, bool WG>
cudaError_t launch_decode_noalloc_t(const Problem &pr, cudaStream_t stream, uint32_t *scratch)
{
    CUtensorMap maps[4];
    DecodeParams p;
    cudaError_t e = prepare<MT, 1, WG>(pr, kNoAllocMaxCtas, maps, &p);
    if (e != cudaSuccess) return e;
    p.partials = reinterpret_cast<float *>(scratch);
    p.arrive = scratch + kNoAllocPartialWords;
    // the array keeps whatever the previous call left: the counters must
    // start at zero (the partial slots are always written before being read)
    e = cudaMemsetAsync(p.arrive, 0, sizeof(uint32_t) * (size_t)p.tiles, stream);
    if (e != cudaSuccess) return e;
    return launch_kernel<MT, 1, WG>(maps, p, stream);
}

template <int MT>
cudaError_t dispatch_noalloc(const Problem &p, cudaStream_t stream, uint32_t *scratch)
{
    // always 256-column tiles: the fixed array holds partials of that width
    const bool whole = p.g % 128 == 0;
    return whole ? launch_decode_noalloc_t<MT, true>(p, stream, scratch)
                 : launch_decode_noalloc_t<MT, false>(p, stream, scratch);
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
    if (M > awq::kNoAllocMaxTokens || !awq::decode_supported(M, K, N, g)) return AWQ_ERR_INVALID_ARG;
    if ((N + awq::Geo<1>::kTileCols - 1) / awq::Geo<1>::kTileCols > awq::kNoAllocMaxTiles) return AWQ_ERR_TOO_LARGE;
    uint32_t *scratch = nullptr;
    if (awq::noalloc_scratch_address(&scratch) != cudaSuccess) return AWQ_ERR_CUDA;
    awq::Problem p{x, qweight, qzeros, scales, bias, y, M, K, N, g, K / g};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = (M <= 8) ? awq::dispatch_noalloc<1>(p, s, scratch)
                                   : awq::dispatch_noalloc<2>(p, s, scratch);
    return e == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA;
}
