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

// Record a device-side error in the status word.
__device__ __forceinline__ void raise_status(unsigned int *status, unsigned int bits) {
    if (status) atomicOr(status, bits);
}

} // namespace awq
