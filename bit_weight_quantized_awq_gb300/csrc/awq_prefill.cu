// awq_prefill.cu -- prefill path of the WQLinear forward (large M), on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Predibase Lorax "AWQ WQLinear" page, Description, forward steps 2-3:
//   y[m, n] = fp16_rn( sum_k x[m, k] * W[k, n] + bias[n] ),
//   W[k, n] = fp16_rn((q[k, n] - z[k/g, n]) * s[k/g, n]), fp32 accumulation.
//
// Output tile: 128 rows of x (tokens) x 256 output columns, or for M > 128
// 256 rows in two 128-row halves that share every weight tile (MH = 2: the
// weight tile, and its dequantisation, serve twice the MMA work). One
// tcgen05 MMA is M = 128 (tokens) x N = 256 (columns) x K = 16. A persistent
// grid (one CTA per SM) walks the tiles; inside a CTA, warps are specialised:
//
//   warp 0      TMA producer: per 64-deep k-stage, the x tile (128 or 256
//               x 64 fp16, K-major, 128-byte swizzle) and the packed-weight
//               tile (64 k-rows x 32 words), plus the scale and zero-point
//               rows of the groups the stage touches, into a ring of 5 (MH =
//               1) or 3 (MH = 2) stages (only what comes from global memory
//               sits in the ring, so it can be deep enough to cover the load
//               latency).
//   warps 2-9   dequant: packed words -> fp16 W in one of two B slots,
//               written directly in the MN-major 128-byte-swizzled layout the
//               MMA reads as its B operand (one packed word = 8 columns = one
//               16-byte store). Per column pair (c, c + 4) of a word: one LOP3
//               masks the two nibbles into the fraction of 1024.0 (low nibble
//               of a byte) or 64.0 (high nibble), one half2 subtract removes
//               (1024 + z) or (64 + z) exactly, one half2 multiply by the
//               scales rounds once: exactly fp16_rn((q - z) s). The columns of
//               every group of 8 are therefore stored as 0 4 1 5 2 6 3 7, and
//               the epilogue undoes that order.
//   warp 1      MMA issuer (one thread) and TMEM owner: 4 MMAs per stage and
//               half into a 256-column fp32 accumulator, tcgen05.commit frees
//               the stage and the B slot and, at the last stage, hands the
//               accumulator over. TMEM holds two accumulators: with MH = 1
//               tiles alternate between them, with MH = 2 a tile's halves use
//               one each.
//   warps 10-17 epilogue: tcgen05.ld of the accumulator (each warp its 32
//               lanes = 32 tokens, two warps per lane quarter, each half of
//               the 256 columns), + bias, one rounding to fp16, TMA stores
//               of 32 x 32 boxes. The epilogue of one tile (or half)
//               overlaps the MMAs of the next tile (or of the other half).
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
#include <cstring>
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
constexpr int kMmaK = 16;
constexpr int kMaxGroupRows = 5;

constexpr int kABytes = BM * BK * 2;            // 16 KB
constexpr int kEpiWarpBytes = 32 * 64;          // 32 rows x 32 fp16 columns of output
constexpr int kBBytes = BN * BK * 2;            // 32 KB
constexpr int kPBytes = BK * (BN / 8) * 4;      // 8 KB

// Shared memory. With dequantisation the TMA ring carries only what comes
// from global memory -- the x tile, the packed-weight tile and the scale and
// zero-point rows (28 KB a stage, five stages, enough to cover the load
// latency) -- and the dequantised B tiles the MMA reads live in a separate
// pair of slots that the dequant warps fill. Without dequantisation
// (awq_gemm_f16) a stage is the x tile plus the fp16 B tile, four stages.
// With MH = 2 a tile has 256 rows of x in two 128-row halves that share
// every B tile (two MMAs per B tile, one per half): the x tile doubles and
// three stages fit; per MMA cycle an SM then takes in a third less data, and
// the dequant warps' work per MMA halves.
template <bool kDequant, int MH>
struct Cfg {
    static constexpr int kATile = MH * kABytes;                 // x tile: MH x 128 rows
    static constexpr int kStages = MH == 1 ? (kDequant ? 5 : 4) : 3;
    static constexpr int kAOff = 0;
    static constexpr int kPOff = kATile;                        // packed words (dequant)
    static constexpr int kSOff = kPOff + kPBytes;               // scale rows (dequant)
    static constexpr int kZOff = kSOff + kMaxGroupRows * BN * 2; // zero-point rows (dequant)
    static constexpr int kBOff = kATile;                        // fp16 B tile (no dequant)
    static constexpr int kStageBytes = kDequant ? (MH == 1 ? 28 : 44) * 1024 : kATile + kBBytes;
    static constexpr int kBSlots = kDequant ? 2 : 0;
    static constexpr int kBSlotOff = kStages * kStageBytes;
    static constexpr int kEpiOff = kBSlotOff + kBSlots * kBBytes;   // epilogue staging, 2 KB per warp
    static constexpr int kBarOff = kEpiOff + 8 * kEpiWarpBytes;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;
    static_assert(!kDequant || kZOff + kMaxGroupRows * (BN / 8) * 4 <= kStageBytes, "stage layout overflows");
    static_assert(kStageBytes % 1024 == 0 && kBSlotOff % 1024 == 0 && kEpiOff % 1024 == 0,
                  "swizzled tiles need 1024-byte alignment");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// B tile layout (MN-major, 128-byte swizzle): 4 column atoms of 64 columns,
// each 8 k-groups of (8 k-rows x 128 bytes).
constexpr int kBAtomStride = 8 * 1024;   // between 64-column atoms (leading byte offset)
constexpr int kBKGroupStride = 1024;     // between 8-row k groups (stride byte offset)

// Inside every 8-column group the dequantised tile stores the columns in the
// order 0 4 1 5 2 6 3 7 (one LOP3 yields columns c and c + 4 of a packed word
// without a byte permute); the accumulator columns come out in that order
// and the epilogue puts them back: output column q of a group is accumulator
// column unperm(q).
__host__ __device__ constexpr int unperm(int q) { return q < 4 ? 2 * q : 2 * (q - 4) + 1; }

constexpr int kWarps = 18;
constexpr int kThreads = kWarps * 32;
constexpr int kDequantWarp0 = 2;
constexpr int kEpilogueWarp0 = 10;
constexpr int kDequantThreads = 256;
constexpr int kEpilogueThreads = 256;
constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators

constexpr uint32_t kIdesc = tc::idesc_f16_f32(BM, BN, true);

// Tiles of two 128-row halves from this many rows of x on (see m_halves).
constexpr int64_t kTwoHalvesMinM = 128;

struct PrefillParams {
    const __half *bias;
    __half *y;
    float *y32;             // if set: y32 += the fp32 sums (no bias, no rounding) instead of y
    unsigned int *status;
    float *partials;        // [2 * sk_ctas][MH][kPartialFloats] stream-K partial sums
    int M, K, N, g;
    int64_t ldy;            // elements between rows of y (N, or more for a column window)
    int tiles_m, tiles_n, kiters;
    int group_m;            // row blocks per band of the tile order (see tile_coords)
    int dp_waves;           // full waves of whole tiles, tile = cta + wave * gridDim.x
    int sk_tiles;           // tiles after those, split along k between sk_ctas CTAs
    int sk_ctas;
    uint32_t stage_tx;
#ifdef AWQ_FAULT_TEST
    int fault;              // CTA 0's producer issues nothing (fault-test build only)
#endif
};

// One stream-K partial: 128 rows x 256 accumulator columns, fp32, laid out
// [32-column chunk][4-column group][row][4] so that the 32 epilogue lanes of
// a warp (32 consecutive rows) touch 512 consecutive bytes per access.
constexpr int kPartialFloats = BM * BN;

__device__ __forceinline__ int sk_range_begin(int c, int units, int ctas) {
    return (int)(((int64_t)c * units) / ctas);
}
// The CTA whose stream-K range contains unit u.
__device__ __forceinline__ int sk_cta_of(int u, int units, int ctas) {
    return (int)((((int64_t)u + 1) * ctas - 1) / units);
}

// The work of one CTA as a list of segments (tile, k-stages kb0 .. kb1 - 1):
// first its whole tiles of the data-parallel waves, then the pieces of its
// stream-K range, split at tile boundaries. Every warp role walks the same
// list.
struct Segments {
    int dp;            // whole tiles first
    int ub, ue;        // stream-K units [ub, ue)
    int count;
    __device__ Segments(const PrefillParams &p) {
        dp = p.dp_waves;
        const int units = p.sk_tiles * p.kiters;
        if ((int)blockIdx.x < p.sk_ctas) {
            ub = sk_range_begin(blockIdx.x, units, p.sk_ctas);
            ue = sk_range_begin(blockIdx.x + 1, units, p.sk_ctas);
        } else {
            ub = ue = 0;
        }
        count = dp + (ue > ub ? (ue - 1) / p.kiters - ub / p.kiters + 1 : 0);
    }
    // segment i: tile index (0 .. tiles - 1) and its k-stage range
    __device__ void get(const PrefillParams &p, int i, int &tile, int &kb0, int &kb1) const {
        if (i < dp) {
            tile = blockIdx.x + i * gridDim.x;
            kb0 = 0;
            kb1 = p.kiters;
            return;
        }
        const int t = ub / p.kiters + (i - dp);   // stream-K tile
        kb0 = (i == dp) ? ub % p.kiters : 0;
        kb1 = (t == (ue - 1) / p.kiters) ? (ue - 1) % p.kiters + 1 : p.kiters;
        tile = p.dp_waves * gridDim.x + t;
    }
};

// Tile order: bands of group_m row blocks, the row block fastest inside a
// band, then the column block. A wave of tiles then shares group_m blocks of
// x and a run of weight column blocks, which stay in L2 while the wave runs;
// with group_m = tiles_m this is plain row-fastest order.
__host__ __device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m,
                                                     int &mi, int &ni)
{
    const int band = tile / (group_m * tiles_n);
    const int first = band * group_m;
    const int rows = tiles_m - first < group_m ? tiles_m - first : group_m;
    const int r = tile - band * group_m * tiles_n;
    mi = first + r % rows;
    ni = r / rows;
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    __half2 r = __hmul2_rn(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// Scales and zero points of one group for packed word j, in the register
// order of the dequantised columns: pair q holds columns (q, q + 4).
__device__ __forceinline__ void load_group(uint32_t s_row, uint32_t z_row, uint32_t (&S)[4], uint32_t (&Z)[4])
{
    uint32_t sv0, sv1, sv2, sv3, zw;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(sv0), "=r"(sv1), "=r"(sv2), "=r"(sv3) : "r"(s_row));
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(zw) : "r"(z_row));
    S[0] = __byte_perm(sv0, sv2, 0x5410);   // (s0, s4)
    S[1] = __byte_perm(sv0, sv2, 0x7632);   // (s1, s5)
    S[2] = __byte_perm(sv1, sv3, 0x5410);   // (s2, s6)
    S[3] = __byte_perm(sv1, sv3, 0x7632);   // (s3, s7)
    const uint32_t zh = zw >> 8;
    Z[0] = (zw & 0x000F000Fu) | 0x64006400u;   // 1024 + (z0, z4)
    Z[1] = (zw & 0x00F000F0u) | 0x54005400u;   // 64 + (z1, z5)
    Z[2] = (zh & 0x000F000Fu) | 0x64006400u;   // 1024 + (z2, z6)
    Z[3] = (zh & 0x00F000F0u) | 0x54005400u;   // 64 + (z3, z7)
}

// One packed word (8 columns of one k-row) -> four half2 registers of
// fp16_rn((q - z) s): the nibble ORed into the fraction of 1024.0 (low
// nibble of a byte) or 64.0 (high nibble, one sixteenth per unit), an exact
// subtraction of (1024 + z) or (64 + z), one multiply rounding once.
__device__ __forceinline__ void dequant_word(uint32_t v, const uint32_t (&S)[4], const uint32_t (&Z)[4],
                                             uint32_t (&h)[4])
{
    const uint32_t vh = v >> 8;
    h[0] = hmul2_u(hsub2_u((v & 0x000F000Fu) | 0x64006400u, Z[0]), S[0]);
    h[1] = hmul2_u(hsub2_u((v & 0x00F000F0u) | 0x54005400u, Z[1]), S[1]);
    h[2] = hmul2_u(hsub2_u((vh & 0x000F000Fu) | 0x64006400u, Z[2]), S[2]);
    h[3] = hmul2_u(hsub2_u((vh & 0x00F000F0u) | 0x54005400u, Z[3]), S[3]);
}

template <bool kDequant, bool kWhole, int MH>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
               const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_y, const PrefillParams p)
{
    using C = Cfg<kDequant, MH>;
    constexpr int kStages = C::kStages;
    constexpr int BMT = BM * MH;   // rows of x per tile
    extern __shared__ uint8_t smem_raw[];
    // round up to 1024 bytes by offsetting the shared array itself, so that
    // the compiler still knows every derived pointer is a shared address
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);   // [kStages] TMA bytes landed
    uint64_t *tfree = full + kStages;       // [kStages] MMAs that read the stage are done
    constexpr int kNB = C::kBSlots > 0 ? C::kBSlots : 1;
    uint64_t *bready = tfree + kStages;     // [kNB] dequantised B slot written
    uint64_t *bfree = bready + kNB;         // [kNB] MMAs that read the B slot are done
    uint64_t *acc_full = bfree + kNB;       // [2]
    uint64_t *acc_empty = acc_full + 2;     // [2]
    uint64_t *drain = acc_empty + 2;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Segments sg(p);
    // the stream-K finishing kernel (or the next layer's kernel) may be
    // scheduled now; it waits for this grid to complete before reading
    ptx::launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(full + s), 1);
            ptx::mbar_init(ptx::smem_addr(tfree + s), 1);
        }
        for (int b = 0; b < kNB; ++b) {
            ptx::mbar_init(ptx::smem_addr(bready + b), kDequantThreads);
            ptx::mbar_init(ptx::smem_addr(bfree + b), 1);
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
#ifdef AWQ_FAULT_TEST
            // injected fault: nothing is loaded, so the bounded waits of the
            // MMA, dequant and epilogue warps on the first stage run out
            if (p.fault && blockIdx.x == 0) ok = false;
#endif
            // Programmatic dependent launch: the packed weights, scales and
            // zero points of the first stages (the ring is empty, no wait)
            // are requested before waiting for the previous kernel; x -- and
            // the fp16 weights of the GEMM core, which the kernel before may
            // have written -- only after that wait.
            int pend_k0[kStages], pend_m0[kStages];
            int npend = 0;
            bool waited = !kDequant;
            if (!kDequant) ptx::wait_prerequisites();
            auto flush_x = [&]() {
                ptx::wait_prerequisites();
                for (int i = 0; i < npend; ++i)
                    ptx::tma_load_2d(ptx::smem_addr(smem + i * C::kStageBytes) + C::kAOff, &tm_x,
                                     ptx::smem_addr(full + i), pend_k0[i], pend_m0[i]);
                waited = true;
            };
            for (int si = 0; si < sg.count && ok; ++si) {
                int tile, kb0, kb1;
                sg.get(p, si, tile, kb0, kb1);
                int mi, ni;
                tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, mi, ni);
                const int m0 = mi * BMT;
                const int n0 = ni * BN;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!ptx::mbar_wait_bounded(ptx::smem_addr(tfree + s), ((it / kStages) & 1) ^ 1,
                                                abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = ptx::smem_addr(full + s);
                    const uint32_t st = ptx::smem_addr(smem + s * C::kStageBytes);
                    const int k0 = kb * BK;
                    ptx::mbar_arrive_expect_tx(fb, p.stage_tx);
                    if (waited) {
                        ptx::tma_load_2d(st + C::kAOff, &tm_x, fb, k0, m0);
                    } else {
                        pend_k0[npend] = k0;   // stage npend == it
                        pend_m0[npend] = m0;
                        ++npend;
                    }
                    if (kDequant) {
                        ptx::tma_load_2d(st + C::kPOff, &tm_w, fb, n0 / 8, k0);
                        ptx::tma_load_2d(st + C::kSOff, &tm_s, fb, n0, k0 / p.g);
                        ptx::tma_load_2d(st + C::kZOff, &tm_z, fb, n0 / 8, k0 / p.g);
                    } else {
#pragma unroll
                        for (int a = 0; a < BN / 64; ++a)
                            ptx::tma_load_2d(st + C::kBOff + a * kBAtomStride, &tm_w, fb, n0 + 64 * a, k0);
                    }
                    issued = it + 1;
                    if (!waited && npend == kStages) flush_x();
                }
            }
            if (!waited) flush_x();
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
            for (int si = 0; si < sg.count && ok; ++si, ++acc_it) {
                int tile, kb0, kb1;
                sg.get(p, si, tile, kb0, kb1);
                // accumulator buffers: with MH == 1 tiles alternate between the
                // two 256-column buffers; with MH == 2 a tile's halves use both
                const int ab0 = MH == 1 ? (acc_it & 1) : 0;
                const uint32_t empty_parity = (uint32_t)((MH == 1 ? (acc_it >> 1) : acc_it) & 1) ^ 1u;
                for (int kb = kb0; kb < kb1 && ok; ++kb, ++it) {
                    const int s = it % kStages;
                    const int b = it % kNB;
                    bool ready = ptx::mbar_wait_bounded(ptx::smem_addr(full + s), (it / kStages) & 1,
                                                        abort_flag, p.status);
                    if (ready && kDequant)
                        ready = ptx::mbar_wait_bounded(ptx::smem_addr(bready + b), (it / kNB) & 1,
                                                       abort_flag, p.status);
                    if (!ready) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t st = ptx::smem_addr(smem + s * C::kStageBytes);
                    const uint32_t bt = kDequant ? ptx::smem_addr(smem + C::kBSlotOff + b * kBBytes)
                                                 : st + C::kBOff;
#pragma unroll
                    for (int h = 0; h < MH; ++h) {
                        // the first stage of a tile waits until the epilogue
                        // has drained this half's buffer (the other half's
                        // MMAs may already run)
                        if (kb == kb0) {
                            if (!ptx::mbar_wait_bounded(ptx::smem_addr(acc_empty + ab0 + h), empty_parity,
                                                        abort_flag, p.status)) {
                                ok = false;
                                break;
                            }
                            tc::fence_after_sync();
                        }
                        const uint32_t d_tmem = tmem_base + (uint32_t)((ab0 + h) * BN);
#pragma unroll
                        for (int kk = 0; kk < BK / kMmaK; ++kk) {
                            const uint64_t ad = tc::smem_desc_sw128(st + C::kAOff + h * kABytes + kk * 32, 16, 1024);
                            const uint64_t bd = tc::smem_desc_sw128(bt + kk * 2 * kBKGroupStride,
                                                                    kBAtomStride, kBKGroupStride);
                            tc::mma_f16(d_tmem, ad, bd, kIdesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                        }
                    }
                    if (!ok) break;
                    tc::commit(ptx::smem_addr(tfree + s));
                    if (kDequant) tc::commit(ptx::smem_addr(bfree + b));
                    if (kb == kb1 - 1) {
#pragma unroll
                        for (int h = 0; h < MH; ++h) tc::commit(ptx::smem_addr(acc_full + ab0 + h));
                    }
                }
            }
            // every MMA this thread issued has completed once `drain` flips
            tc::commit(ptx::smem_addr(drain));
            ptx::mbar_wait_bounded(ptx::smem_addr(drain), 0, nullptr, p.status);
        }
    } else if (warp < kEpilogueWarp0) {
        // ------------------------------------------------------------ dequant
        if (kDequant) {
            const int dt = threadIdx.x - kDequantWarp0 * 32;   // 0..255
            const int dw = dt >> 5;            // k-row inside every 8-row group: dw, dw + 8, ...
            const int j = dt & 31;             // packed word (8 columns) in the tile row
            // B slot: 64-column atom j / 8, 16-byte chunk (j % 8) ^ row in the
            // 128-byte swizzle; the k-group adds 1024 bytes
            const uint32_t b_in = (uint32_t)(j >> 3) * kBAtomStride + (uint32_t)dw * 128 +
                                  ((uint32_t)((j & 7) ^ dw) << 4);
            const uint32_t p_in = C::kPOff + (uint32_t)dw * 128 + (uint32_t)j * 4;
            const uint32_t s_in = C::kSOff + (uint32_t)j * 16;
            const uint32_t z_in = C::kZOff + (uint32_t)j * 4;
            int it = 0;
            bool ok = true;
            for (int si = 0; si < sg.count && ok; ++si) {
                int tile, kb0, kb1;
                sg.get(p, si, tile, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    const int b = it % kNB;
                    bool ready = ptx::mbar_wait_bounded(ptx::smem_addr(full + s), (it / kStages) & 1,
                                                        abort_flag, p.status);
                    if (ready)
                        ready = ptx::mbar_wait_bounded(ptx::smem_addr(bfree + b), ((it / kNB) & 1) ^ 1,
                                                       abort_flag, p.status);
                    if (!ready) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = ptx::smem_addr(smem + s * C::kStageBytes);
                    const uint32_t bb = ptx::smem_addr(smem + C::kBSlotOff + b * kBBytes) + b_in;
                    // all of this thread's packed words of the stage are
                    // requested before any is converted, so their latencies
                    // overlap instead of adding up word by word
                    uint32_t v[BK / 8];
#pragma unroll
                    for (int i = 0; i < BK / 8; ++i)
                        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[i]) : "r"(st + p_in + i * 1024));
                    uint32_t S[4], Z[4];
                    int r = 0, rem = 0;
                    if (kWhole) {
                        // g % 64 == 0: the whole stage lies in one group
                        load_group(st + s_in, st + z_in, S, Z);
                    } else {
                        const int k0 = kb * BK;
                        const int grp0 = k0 / p.g;
                        r = (k0 + dw) / p.g - grp0;   // group row of this thread's first k-row
                        rem = (k0 + dw) - (r + grp0) * p.g;
                        load_group(st + s_in + r * (BN * 2), st + z_in + r * (BN / 8 * 4), S, Z);
                    }
#pragma unroll
                    for (int i = 0; i < BK / 8; ++i) {
                        if (!kWhole && i > 0) {
                            rem += 8;   // g >= 16: at most one group boundary per step
                            if (rem >= p.g) {
                                rem -= p.g;
                                ++r;
                                load_group(st + s_in + r * (BN * 2), st + z_in + r * (BN / 8 * 4), S, Z);
                            }
                        }
                        uint32_t h[4];
                        dequant_word(v[i], S, Z, h);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                     ::"r"(bb + i * kBKGroupStride), "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                                     : "memory");
                    }
                    // make the generic-proxy stores visible to the tensor core
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(ptx::smem_addr(bready + b));
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // bias, y and the stream-K scratch may be in use by the previous
        // kernel until it completes
        ptx::wait_prerequisites();
        const int q = warp & 3;                 // TMEM lane quarter this warp may read
        const int ew = warp - kEpilogueWarp0;   // 0..7: two warps per lane quarter
        const int ch = ew >> 2;                 // accumulator columns 128 ch .. 128 ch + 127
        int acc_it = 0;
        bool ok = true;
        for (int si = 0; si < sg.count && ok; ++si, ++acc_it) {
            int tile, kb0, kb1;
            sg.get(p, si, tile, kb0, kb1);
            const int ab0 = MH == 1 ? (acc_it & 1) : 0;
            const uint32_t full_parity = (uint32_t)((MH == 1 ? (acc_it >> 1) : acc_it) & 1);
            int mi, ni;
            tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, mi, ni);
            const int m0 = mi * BMT;
            const int n0 = ni * BN;
            const bool whole = kb0 == 0 && kb1 == p.kiters;
            // a piece of a stream-K tile goes to this CTA's slot: the first
            // piece of its range in slot 0, the last in slot 1
            float *piece = whole ? nullptr
                                 : p.partials + (int64_t)(2 * (int)blockIdx.x + (si == sg.dp ? 0 : 1)) *
                                                    (MH * kPartialFloats);
            for (int h = 0; h < MH; ++h) {
                const int ab = ab0 + h;
                // the decision to go on is taken together by the eight warps,
                // which meet at a named barrier
                ok = ptx::named_barrier_and(
                    1, kEpilogueThreads,
                    ptx::mbar_wait_bounded(ptx::smem_addr(acc_full + ab), full_parity, abort_flag, p.status));
                if (!ok) break;
                tc::fence_after_sync();
                const int m = m0 + h * BM + 32 * q + lane;
                const uint32_t t_acc = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * BN);
                if (whole && p.y32 == nullptr) {
                    // ---- whole tile: + bias, one rounding, staged 32 columns
                    //      at a time in this warp's 2 KB buffer (32 rows x 64
                    //      bytes, 64-byte swizzle) and written by a TMA store,
                    //      which clips rows >= M and columns >= N
                    const uint32_t stg = ptx::smem_addr(smem + C::kEpiOff + ew * kEpiWarpBytes);
                    const int row0 = m0 + h * BM + 32 * q;
#pragma unroll 1
                    for (int c = 4 * ch; c < 4 * ch + 4; ++c) {
                        const int col = n0 + 32 * c;
                        if (col >= p.N) break;
                        // the previous store from the buffer has read it
                        if (lane == 0) ptx::bulk_wait_read_all();
                        __syncwarp();
                        uint32_t raw[32];
                        tc::ld_32x32b_x32(t_acc + (uint32_t)(32 * c), raw);
                        tc::ld_wait();
                        float b[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) b[e] = 0.f;
                        if (p.bias) {
                            __align__(16) __half bh[32];
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                reinterpret_cast<uint4 *>(bh)[v] = __ldg(reinterpret_cast<const uint4 *>(p.bias + col) + v);
#pragma unroll
                            for (int e = 0; e < 32; ++e) b[e] = __half2float(bh[e]);
                        }
                        uint32_t hv[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int e0 = 2 * e, e1 = 2 * e + 1;
                            const float v0 = __uint_as_float(kDequant ? raw[(e0 & ~7) + unperm(e0 & 7)] : raw[e0]);
                            const float v1 = __uint_as_float(kDequant ? raw[(e1 & ~7) + unperm(e1 & 7)] : raw[e1]);
                            const __half2 hh = __halves2half2(__float2half_rn(v0 + b[e0]), __float2half_rn(v1 + b[e1]));
                            hv[e] = *reinterpret_cast<const uint32_t *>(&hh);
                        }
                        // row `lane` of the box: 16-byte chunk u at chunk
                        // u ^ ((row / 2) % 4) of its 64-byte row
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                         ::"r"(stg + (uint32_t)lane * 64 + (((uint32_t)u ^ (((uint32_t)lane >> 1) & 3u)) << 4)),
                                           "r"(hv[4 * u]), "r"(hv[4 * u + 1]), "r"(hv[4 * u + 2]), "r"(hv[4 * u + 3])
                                         : "memory");
                        // the generic-proxy writes are made visible to the TMA
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && row0 < p.M) {
                            ptx::tma_store_2d(&tm_y, stg, col, row0);
                            ptx::bulk_commit_group();
                        }
                    }
                } else if (whole) {
                    // ---- whole tile, row-shard form: y32 += the fp32 sums
#pragma unroll 1
                    for (int c = 4 * ch; c < 4 * ch + 4; ++c) {
                        uint32_t raw[32];
                        tc::ld_32x32b_x32(t_acc + (uint32_t)(32 * c), raw);
                        tc::ld_wait();
                        const int col = n0 + 32 * c;
                        uint32_t r[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = kDequant ? raw[(e & ~7) + unperm(e & 7)] : raw[e];
                        if (col < p.N && m < p.M) {
                            float4 *d = reinterpret_cast<float4 *>(p.y32 + (int64_t)m * p.ldy + col);
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                float4 t = d[v];
                                t.x += __uint_as_float(r[4 * v]);
                                t.y += __uint_as_float(r[4 * v + 1]);
                                t.z += __uint_as_float(r[4 * v + 2]);
                                t.w += __uint_as_float(r[4 * v + 3]);
                                d[v] = t;
                            }
                        }
                    }
                } else {
                    // ---- a piece of a stream-K tile: store the fp32 partial
                    //      of this half; sk_fixup_kernel, launched after this
                    //      grid, sums the pieces of every split tile
                    float *mine = piece + (int64_t)h * kPartialFloats;
#pragma unroll 1
                    for (int c = 4 * ch; c < 4 * ch + 4; ++c) {
                        uint32_t raw[32];
                        tc::ld_32x32b_x32(t_acc + (uint32_t)(32 * c), raw);
                        tc::ld_wait();
                        if (m < p.M) {
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                reinterpret_cast<uint4 *>(mine)[(c * 8 + v) * BM + 32 * q + lane] =
                                    make_uint4(raw[4 * v], raw[4 * v + 1], raw[4 * v + 2], raw[4 * v + 3]);
                        }
                    }
                }
                tc::fence_before_sync();
                ptx::mbar_arrive(ptx::smem_addr(acc_empty + ab));
            }
        }
        // this warp's TMA stores have completed before the CTA exits
        if (lane == 0) ptx::bulk_wait_all();
    }
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Finishing the stream-K tiles: one CTA per (split tile, 128-row half,
// 32-column chunk), one thread per row. Each thread adds the fp32 pieces of its row
// and chunk in contributor order (the same order every call), adds the bias,
// rounds once and stores (or adds the sum into y32). It is launched right
// after prefill_kernel as a programmatic dependent: its CTAs may be scheduled
// while the main grid drains and wait for that grid to complete before they
// read any partial.
struct FixupParams {
    const float *partials;
    const __half *bias;
    __half *y;
    float *y32;
    int M, N;
    int64_t ldy;
    int tiles_m, tiles_n, group_m, kiters;
    int first_tile;         // tile index of stream-K tile 0: dp_waves x the main grid's size
    int sk_tiles, sk_ctas;
};

template <bool kDequant, int MH>
__global__ void __launch_bounds__(BM)
sk_fixup_kernel(const FixupParams p)
{
    // the next kernel may be scheduled now (it waits for this grid, which
    // itself has waited for the main grid)
    ptx::launch_dependents();
    ptx::wait_prerequisites();
    const int t = blockIdx.x / (MH * (BN / 32));
    const int h = (blockIdx.x / (BN / 32)) % MH;
    const int c = blockIdx.x % (BN / 32);
    const int units = p.sk_tiles * p.kiters;
    const int cf = sk_cta_of(t * p.kiters, units, p.sk_ctas);
    const int cl = sk_cta_of(t * p.kiters + p.kiters - 1, units, p.sk_ctas);
    if (cl == cf) return;   // a single contributor took the whole tile and stored it
    const int tile = p.first_tile + t;
    int mi, ni;
    tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, mi, ni);
    const int m = mi * (BM * MH) + h * BM + (int)threadIdx.x;
    const int col0 = ni * BN + 32 * c;
    if (m >= p.M || col0 >= p.N) return;
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
#pragma unroll 2
    for (int ci = cf; ci <= cl; ++ci) {
        const int which = (sk_range_begin(ci, units, p.sk_ctas) / p.kiters == t) ? 0 : 1;
        const float4 *src = reinterpret_cast<const float4 *>(p.partials + ((int64_t)(2 * ci + which) * MH + h) *
                                                                               kPartialFloats) +
                            (c * 8) * BM + threadIdx.x;
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + j * BM);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            acc[4 * j] += v[j].x;
            acc[4 * j + 1] += v[j].y;
            acc[4 * j + 2] += v[j].z;
            acc[4 * j + 3] += v[j].w;
        }
    }
    // accumulator column order -> output column order inside every 8-group
    float o[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = kDequant ? acc[(e & ~7) + unperm(e & 7)] : acc[e];
    if (p.y32) {
        float4 *d = reinterpret_cast<float4 *>(p.y32 + (int64_t)m * p.ldy + col0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 t4 = d[j];
            t4.x += o[4 * j];
            t4.y += o[4 * j + 1];
            t4.z += o[4 * j + 2];
            t4.w += o[4 * j + 3];
            d[j] = t4;
        }
        return;
    }
    if (p.bias) {
        __align__(16) __half bh[32];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            reinterpret_cast<uint4 *>(bh)[j] = __ldg(reinterpret_cast<const uint4 *>(p.bias + col0) + j);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] += __half2float(bh[e]);
    }
    __align__(16) __half out[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) out[e] = __float2half_rn(o[e]);
    uint4 *dst = reinterpret_cast<uint4 *>(p.y + (int64_t)m * p.ldy + col0);
#pragma unroll
    for (int j = 0; j < 4; ++j) dst[j] = reinterpret_cast<const uint4 *>(out)[j];
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

// How a launch covers the tiles. Whole waves of tiles go round-robin over
// one CTA per SM (neighbouring CTAs share weight tiles in L2). The tiles left
// over for a last, partial wave are split along k ("stream-K") between up to
// one CTA per SM, each taking at least kMinUnits k-stages, so that the last
// wave keeps every SM busy instead of a few; sk_fixup_kernel then sums the
// pieces of every tile that was split. Where that wave already fills most
// SMs, it runs whole instead (split_last_wave).
struct Plan {
    int tiles_m, tiles_n, kiters;
    int group_m;
    int dp_waves, sk_tiles, sk_ctas, ctas;
    bool split;             // some tile has more than one contributor
    bool ok;                // sizes within the kernel's index range
};

// Row blocks per band of the tile order. Whole waves in row-fastest order
// sweep all of x once per wave. When x is larger than a share of L2, bands
// of as many row blocks as fit that share are used instead -- and at least
// as many as make a band span a wave of tiles, so that a wave takes all the
// column blocks of a few row blocks: the CTAs of a wave walk k in step, so
// a wave reads each of its blocks of x and of W from DRAM about once, and
// over the whole launch x is read about once and the weights once per
// band. (Row-fastest waves of a tall x instead read all of x in every wave:
// 846 MB for 338 MB of operands at M = 8192, K = 11008, N = 4096.)
constexpr int64_t kL2Share = 32ll << 20;

int group_rows(int tiles_m, int tiles_n, int64_t K, int sms, int mh)
{
    const int64_t x_block = (int64_t)BM * mh * K * 2;      // one row block of x
    if ((int64_t)tiles_m * x_block <= kL2Share) return tiles_m;
    int64_t gm = kL2Share / x_block;
    const int64_t wave_rows = (sms + tiles_n - 1) / tiles_n;   // row blocks that span a wave
    if (gm < wave_rows) gm = wave_rows;
    if (gm >= tiles_m) return tiles_m;
    return (int)gm;
}

Plan plan_tiles(int64_t M, int64_t K, int64_t N, int sms, int mh, bool allow_split)
{
    constexpr int kMinUnits = 8;
    Plan pl{};
    pl.tiles_m = (int)((M + BM * mh - 1) / (BM * mh));
    pl.tiles_n = (int)((N + BN - 1) / BN);
    pl.kiters = (int)((K + BK - 1) / BK);
    pl.group_m = group_rows(pl.tiles_m, pl.tiles_n, K, sms, mh);
    const int64_t n_tiles = (int64_t)pl.tiles_m * pl.tiles_n;
    pl.dp_waves = (int)(n_tiles / sms);
    pl.sk_tiles = (int)(n_tiles - (int64_t)pl.dp_waves * sms);
    const int64_t sk_units = (int64_t)pl.sk_tiles * pl.kiters;
    // without splitting, the last wave's tiles go whole to one CTA each
    pl.sk_ctas = pl.sk_tiles == 0 ? 0
                 : !allow_split ? pl.sk_tiles
                 : (int)std::min<int64_t>(sms, std::max<int64_t>(pl.sk_tiles, sk_units / kMinUnits));
    pl.ctas = pl.dp_waves > 0 ? sms : pl.sk_ctas;
    pl.split = pl.sk_tiles > 0 && pl.sk_ctas > pl.sk_tiles;
    pl.ok = sk_units < (int64_t(1) << 31);
    return pl;
}

// Whether to split the last, partial wave of tiles along k. Splitting
// spreads its k-stages over every SM but costs the sum kernel, which reads
// every piece back (about 0.05 us per 256 KB piece, plus 3 us); leaving the
// wave whole costs one tile's time with SMs idle. Estimates in microseconds,
// from a sweep of both choices over M = 512..8192 and the 7B and 70B
// projection shapes: a 256 x 256 x 64 stage takes about 0.8 us.
bool split_last_wave(int64_t M, int64_t K, int64_t N, int sms, int mh)
{
    const Plan pl = plan_tiles(M, K, N, sms, mh, true);
    if (!pl.split || mh != 2) return true;
    const double kStageUs = 0.8, kPieceUs = 0.052, kSumUs = 3.0;
    const double tile_us = (double)pl.kiters * kStageUs;
    const double split_us = (double)pl.sk_tiles / (double)sms * tile_us +
                            (double)(pl.sk_ctas + pl.sk_tiles) * kPieceUs + kSumUs;
    return split_us <= tile_us;
}

struct LaunchInfo {
    int sms = 0;
    cudaError_t err = cudaSuccess;
    unsigned gen = 0;   // cache generation this was set up in
};

template <bool kDequant, bool kWhole, int MH>
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
    li.err = cudaFuncSetAttribute(prefill_kernel<kDequant, kWhole, MH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  Cfg<kDequant, MH>::kSmemBytes);
    if (li.err == cudaSuccess)
        li.err = cudaDeviceGetAttribute(&li.sms, cudaDevAttrMultiProcessorCount, dev);
    if (li.err == cudaSuccess) cache[dev] = li;
    return li;
}

template <bool kDequant, bool kWhole, int MH>
cudaError_t launch(const Problem &pr, const void *w16, cudaStream_t stream, int64_t ldy)
{
    const LaunchInfo li = launch_info<kDequant, kWhole, MH>();
    if (li.err != cudaSuccess) return li.err;
    const int M = (int)pr.M, K = (int)pr.K, N = (int)pr.N, g = (int)pr.g;
    const Plan pl = plan_tiles(M, K, N, li.sms, MH, split_last_wave(M, K, N, li.sms, MH));
    if (!pl.ok) return cudaErrorInvalidValue;
    const int tiles_m = pl.tiles_m, tiles_n = pl.tiles_n, kiters = pl.kiters;
    const int dp_waves = pl.dp_waves, sk_tiles = pl.sk_tiles, sk_ctas = pl.sk_ctas, ctas = pl.ctas;

    CUtensorMap tx, tw, ts, tz;
    const uint64_t ldx = pr.ldx > 0 ? (uint64_t)pr.ldx : (uint64_t)K;
    bool ok = make_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pr.x, K, M, ldx * 2, BK, BM * MH,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    uint32_t tx_bytes = kABytes * MH;
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

    // y for the TMA stores of whole tiles: [M, N] fp16 with row pitch ldy,
    // boxes of 32 rows x 64 columns (not used when summing into y32)
    CUtensorMap ty;
    memset(&ty, 0, sizeof(ty));
    const uint64_t ldy_eff = ldy > 0 ? (uint64_t)ldy : (uint64_t)N;
    if (pr.y32 == nullptr &&
        !make_map_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pr.y, N, M, ldy_eff * 2, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;

    PrefillParams p{};
    p.bias = static_cast<const __half *>(pr.bias);
    p.y = static_cast<__half *>(pr.y);
    p.y32 = pr.y32;
    p.status = device_status_word();
#ifdef AWQ_FAULT_TEST
    p.fault = fault_injection();
#endif
    p.M = M; p.K = K; p.N = N; p.g = g;
    p.ldy = ldy > 0 ? ldy : N;
    p.tiles_m = tiles_m; p.tiles_n = tiles_n; p.kiters = kiters;
    p.group_m = pl.group_m;
    p.dp_waves = dp_waves; p.sk_tiles = sk_tiles; p.sk_ctas = sk_ctas;
    p.stage_tx = tx_bytes;
    const bool split = pl.split;
    if (split) {
        Scratch sc{};
        if (!get_scratch(stream, (size_t)2 * sk_ctas * MH * kPartialFloats, 0, &sc))
            return cudaErrorMemoryAllocation;
        p.partials = sc.partials;
    }
    // programmatic dependent launch: the CTAs may start while the previous
    // kernel drains (they wait for it before touching what it writes)
    cudaLaunchConfig_t mcfg{};
    mcfg.gridDim = dim3((unsigned)ctas);
    mcfg.blockDim = dim3(kThreads);
    mcfg.dynamicSmemBytes = Cfg<kDequant, MH>::kSmemBytes;
    mcfg.stream = stream;
    cudaLaunchAttribute mattr[1];
    mattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    mattr[0].val.programmaticStreamSerializationAllowed = 1;
    mcfg.attrs = mattr;
    mcfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&mcfg, prefill_kernel<kDequant, kWhole, MH>, tx, tw, ts, tz, ty, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess || !split) return e;

    FixupParams f{};
    f.partials = p.partials;
    f.bias = p.bias;
    f.y = p.y;
    f.y32 = p.y32;
    f.M = M; f.N = N; f.ldy = p.ldy;
    f.tiles_m = tiles_m; f.tiles_n = tiles_n; f.group_m = pl.group_m; f.kiters = kiters;
    f.first_tile = dp_waves * ctas;
    f.sk_tiles = sk_tiles; f.sk_ctas = sk_ctas;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(sk_tiles * MH * (BN / 32)));
    cfg.blockDim = dim3(BM);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, sk_fixup_kernel<kDequant, MH>, f);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

} // namespace

// every stream-K CTA (at most one per SM) keeps two pieces of up to two
// 128-row halves
size_t prefill_partial_floats_max(int sms) { return (size_t)2 * (size_t)sms * 2 * kPartialFloats; }

bool prefill_supported(int64_t M, int64_t K, int64_t N, int64_t g)
{
    return M >= 1 && M < (int64_t(1) << 31) && K % 16 == 0 && N % 32 == 0 && g % 16 == 0 &&
           K <= (int64_t(1) << 30) && N <= (int64_t(1) << 30);
}

// 128-row halves per tile: two (256-row tiles sharing every B tile) once M
// fills them, else one.
int m_halves(int64_t M)
{
    return M > kTwoHalvesMinM ? 2 : 1;
}

cudaError_t launch_prefill(const Problem &p, cudaStream_t stream)
{
    if (!prefill_supported(p.M, p.K, p.N, p.g)) return cudaErrorInvalidValue;
    // g % 64 == 0: every 64-row stage lies in one group
    if (m_halves(p.M) == 2)
        return p.g % BK == 0 ? launch<true, true, 2>(p, nullptr, stream, 0)
                             : launch<true, false, 2>(p, nullptr, stream, 0);
    return p.g % BK == 0 ? launch<true, true, 1>(p, nullptr, stream, 0)
                         : launch<true, false, 1>(p, nullptr, stream, 0);
}

cudaError_t launch_gemm_f16(const Problem &p, const void *w16, cudaStream_t stream, int64_t ldy)
{
    return m_halves(p.M) == 2 ? launch<false, true, 2>(p, w16, stream, ldy)
                              : launch<false, true, 1>(p, w16, stream, ldy);
}

int prefill_launches(int64_t M, int64_t K, int64_t N, int sms)
{
    const int mh = m_halves(M);
    return plan_tiles(M, K, N, sms, mh, split_last_wave(M, K, N, sms, mh)).split ? 2 : 1;
}

} // namespace awq
