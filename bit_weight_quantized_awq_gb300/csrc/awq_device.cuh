// awq_device.cuh -- device-side building blocks shared by the library's
// kernels: int4 -> fp16 dequantisation and small PTX wrappers.
//
// Dequantisation (Predibase Lorax "AWQ WQLinear" page, Overview: group-wise
// scaling; Description, __init__: per-group dequantisation):
//   W = fp16_rn((q - z) * s), q and z unsigned 4-bit codes, s an fp16 scale.
// (q - z) is an integer in [-15, 15], so the product with an fp16 scale has at
// most 15 significant bits and the single fp16 multiply rounds it exactly
// once. The codes become fp16 without a conversion instruction: OR-ing a code
// c into the low fraction bits of 1024.0 (0x6400) gives exactly 1024 + c, and
// into bits 4..7 of 64.0 (0x5400) gives exactly 64 + c (the fraction step of
// 64.0 is 1/16). The difference of two such values is the exact integer
// q - z. This is the IEEE binary16 layout, nothing more.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace awq {

// The nibble order this library fixes: nibble i (bits 4i..4i+3) of an int32
// holds column 8j + i of that row.
__device__ __forceinline__ uint32_t nibble(uint32_t word, int i) {
    return (word >> (4 * i)) & 0xFu;
}

// One weight: fp16_rn((q - z) * s).
__device__ __forceinline__ __half dequant_one(uint32_t q, uint32_t z, __half s) {
    const __half qh = __ushort_as_half(static_cast<unsigned short>(0x6400u | q));
    const __half zh = __ushort_as_half(static_cast<unsigned short>(0x6400u | z));
    return __hmul_rn(__hsub_rn(qh, zh), s);
}

// Eight weights of one packed word, columns 8j .. 8j+7 in order.
__device__ __forceinline__ void dequant_word(uint32_t qword, uint32_t zword,
                                             const __half (&s)[8], __half (&w)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = dequant_one(nibble(qword, i), nibble(zword, i), s[i]);
}

// The same eight weights with half2 arithmetic: two weights per instruction.
// One LOP3 puts the nibbles of columns c and c + 4 (c = 0..3; bytes 0 and 2
// of the word, or of the word shifted right by 8) into the low fraction bits
// of 1024.0 (low nibble of a byte) or bits 4..7 of 64.0 (high nibble: the
// fraction step of 64.0 is 1/16, so the value is 64 + code), the same for the
// zero word, then one exact half2 subtraction and one half2 multiply that
// rounds once -- exactly dequant_one on each lane. Result in column order:
// out[p] holds columns 2p and 2p + 1 (low half first), i.e. the 16 bytes of
// the eight fp16 weights as they lie in memory.
__device__ __forceinline__ uint4 dequant_word_h2(uint32_t v, uint32_t zw, uint4 sraw) {
    const uint32_t vh = v >> 8, zh = zw >> 8;
    // scale pairs (s0, s4) (s1, s5) (s2, s6) (s3, s7)
    const uint32_t s04 = __byte_perm(sraw.x, sraw.z, 0x5410), s15 = __byte_perm(sraw.x, sraw.z, 0x7632);
    const uint32_t s26 = __byte_perm(sraw.y, sraw.w, 0x5410), s37 = __byte_perm(sraw.y, sraw.w, 0x7632);
    const uint32_t lo = 0x64006400u, hi = 0x54005400u;
    __half2 q, z, r04, r15, r26, r37;
    uint32_t t;
    t = (v & 0x000F000Fu) | lo; q = *reinterpret_cast<__half2 *>(&t);
    t = (zw & 0x000F000Fu) | lo; z = *reinterpret_cast<__half2 *>(&t);
    r04 = __hmul2_rn(__hsub2(q, z), *reinterpret_cast<const __half2 *>(&s04));
    t = (v & 0x00F000F0u) | hi; q = *reinterpret_cast<__half2 *>(&t);
    t = (zw & 0x00F000F0u) | hi; z = *reinterpret_cast<__half2 *>(&t);
    r15 = __hmul2_rn(__hsub2(q, z), *reinterpret_cast<const __half2 *>(&s15));
    t = (vh & 0x000F000Fu) | lo; q = *reinterpret_cast<__half2 *>(&t);
    t = (zh & 0x000F000Fu) | lo; z = *reinterpret_cast<__half2 *>(&t);
    r26 = __hmul2_rn(__hsub2(q, z), *reinterpret_cast<const __half2 *>(&s26));
    t = (vh & 0x00F000F0u) | hi; q = *reinterpret_cast<__half2 *>(&t);
    t = (zh & 0x00F000F0u) | hi; z = *reinterpret_cast<__half2 *>(&t);
    r37 = __hmul2_rn(__hsub2(q, z), *reinterpret_cast<const __half2 *>(&s37));
    const uint32_t a = *reinterpret_cast<uint32_t *>(&r04), b = *reinterpret_cast<uint32_t *>(&r15);
    const uint32_t c = *reinterpret_cast<uint32_t *>(&r26), d = *reinterpret_cast<uint32_t *>(&r37);
    // back to column order: (0,1) (2,3) (4,5) (6,7)
    return make_uint4(__byte_perm(a, b, 0x5410), __byte_perm(c, d, 0x5410), __byte_perm(a, b, 0x7632),
                      __byte_perm(c, d, 0x7632));
}

// Record a device-side error in the status word.
__device__ __forceinline__ void raise_status(unsigned int *status, unsigned int bits) {
    if (status) atomicOr(status, bits);
}

} // namespace awq

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, TMA, timers, legacy tensor-core MMA
// ---------------------------------------------------------------------------
namespace awq {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Tests the phase; if it has not completed, the thread is suspended until it
// does or until about `hint_ns` nanoseconds pass, so a waiting thread does
// not spin and take issue slots from the warps doing the work.
constexpr uint32_t kSuspendHintNs = 1000000u;   // 1 ms

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Device-side wait limit: a wait that has not completed after this many SM
// clock cycles (about 2 s at 2 GHz, longer at lower clocks) records
// AWQ_ERR_TIMEOUT in the status word and gives up. The limit is kept with the
// SM-local cycle counter: reading %globaltimer costs far more than a poll.
#ifdef AWQ_FAULT_TEST
// the fault-test build of the library (tests only): about 2 ms, so that a
// test that makes a wait run out finishes quickly
constexpr long long kWaitLimitCycles = 4000000ll;
#else
constexpr long long kWaitLimitCycles = 4000000000ll;
#endif

// Bounded wait on an mbarrier phase. Returns false if the wait gave up,
// either because its own limit ran out or because another thread of the CTA
// already gave up (*abort != 0; abort may be nullptr). Never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort, unsigned int *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            if (abort) *abort = 1;
            if (status) atomicOr(status, 1u);
            return false;
        }
    }
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
// x is the innermost coordinate (elements), y the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// 3-D tiled TMA load global -> shared; coordinates innermost first.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// TMA store of one 2-D box from shared memory (the tensor map's box and
// swizzle), tracked by the issuing thread's bulk groups. The hardware clips
// the parts of the box outside the tensor.
__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t src, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// until the shared-memory sources of this thread's committed bulk groups
// have been read (the buffer may be written again)
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// until this thread's committed bulk groups have completed
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices from shared memory in the mma operand layout: lanes
// 8i..8i+7 give the row addresses (16 bytes each) of matrix i; lane
// (4 g + t) receives elements 2t, 2t+1 of row g of every matrix.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&d)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]) : "r"(addr) : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only, not L1), and the wait
// for every such copy this thread has issued.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0),
// completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Orders this thread's earlier generic-proxy accesses (and what they
// acquired) before its later async-proxy (TMA) accesses, in every state space.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async;" ::: "memory");
}

// Programmatic dependent launch: let the next kernel on the stream be
// scheduled now / wait until the previous kernel has finished and its memory
// is visible. Both are no-ops when the launch has no such dependency.
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const unsigned int *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads:
// every thread gets the same answer, so a decision taken on it is uniform.
__device__ __forceinline__ bool named_barrier_and(int id, int threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %2, 0;\n\t"
        "bar.red.and.pred q, %1, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"((uint32_t)pred), "r"(threads)
        : "memory");
    return r != 0;
}

} // namespace ptx
} // namespace awq
