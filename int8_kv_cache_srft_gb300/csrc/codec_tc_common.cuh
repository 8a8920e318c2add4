// codec_tc_common.cuh -- helpers shared by the tensor-core dequantize kernels
// (codec_tc.cu at d = 128 and 96, codec_tc_wide.cuh at d = 192 and 256): the
// contraction's K order, exact fp16 pairs of signed codes, swizzled 16-byte
// chunks of TMA-copied rows.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace srftkv {

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 16-byte chunk c of row r of a buffer of RB-byte rows written by TMA with the
// swizzle mode equal to RB (32, 64 or 128; 16 = no swizzle), 1024-aligned
__device__ __forceinline__ int swz16(int rb, int r, int c) {
    return (rb == 32 || rb == 64 || rb == 128) ? c ^ (((r * rb) >> 7) & (rb / 16 - 1)) : c;
}

// K order of the dequantize contraction.  A column c = 4k + j (k: 8-element
// code word, j = 0..3) holds the packed coordinates (8k + j, 8k + j + 4): those
// two codes sit at bit offsets 16 apart in a 4-bit code word, so one logic op
// and one f16x2 op turn them into an exact fp16 pair.  B is built in the same
// K order, so the contraction is unchanged.
__host__ __device__ constexpr int dq_kperm(int q) { return 8 * (q >> 3) + ((q >> 1) & 3) + 4 * (q & 1); }

__device__ __forceinline__ uint32_t h2sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t h2mul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t h2fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
// Exact fp16 pairs of signed codes: XOR with 8 (128) makes a code offset
// binary; under the exponent of 1024 its fp16 value is 1024 + 8 + q
// (1024 + 16 (q + 8) for the high nibble, 1024 + 128 + q for bytes), and one
// f16x2 subtract (or scaled fma) leaves q.
__device__ __forceinline__ uint32_t codes_lo4(uint32_t w) {  // nibbles at bits 0 and 16
    return h2sub((w & 0x000F000Fu) ^ 0x64086408u, 0x64086408u);
}
__device__ __forceinline__ uint32_t codes_hi4(uint32_t w) {  // nibbles at bits 4 and 20
    return h2fma((w & 0x00F000F0u) ^ 0x64806480u, 0x2C002C00u /* 1/16 */, 0xD480D480u /* -72 */);
}
__device__ __forceinline__ uint32_t codes_b8(uint32_t w) {  // bytes 0 and 2
    return h2sub((w & 0x00FF00FFu) ^ 0x64806480u, 0x64806480u);
}
__device__ __forceinline__ uint32_t half2_bcast(__half h) {
    const uint32_t u = __half_as_ushort(h);
    return u | (u << 16);
}

}  // namespace srftkv
