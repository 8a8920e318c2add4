// codec_tc_common.cuh -- helpers shared by the tensor-core codec kernels
// (codec_tc.cu at d = 128, 96 and 80, codec_tc_wide.cuh at d = 192 and 256):
// the dequantize contraction's K order, exact fp16 pairs of signed codes,
// swizzled 16-byte chunks of TMA-copied rows, and the pieces every kernel's
// prologue uses to build its block of R_s in shared memory.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace srftkv {

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// (a, b) as fp16 hi + lo pairs: hi the fp16 rounding of each, lo the fp16
// rounding of the fp32 residual (the same values as converting one entry at a
// time; the even coordinate in the low half, as in memory)
__device__ __forceinline__ void split_pair_h2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 f = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - f.x, b - f.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// The sign vector s as the kernel parameters carry it (word j: bit 15 for
// coordinate 2j, bit 31 for 2j + 1), copied into shared memory before a
// prologue builds R_s = R diag(s): read from the parameters with a per-lane
// index, each lookup serialises over the distinct words a warp asks for (half
// of the d = 128 prologue's time).  The caller synchronises the block.
__device__ __forceinline__ void stage_sign_mask(uint32_t* dst, const uint32_t* mask, int words) {
    for (int i = threadIdx.x; i < words; i += blockDim.x) dst[i] = mask[i];
}
__device__ __forceinline__ bool sign_flip(const uint32_t* smask, int k) {
    return (smask[k >> 1] & ((k & 1) ? 0x80000000u : 0x8000u)) != 0u;
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
