// codec_pair.cuh -- quantize / dequantize kernels for head dimension 256, two
// threads per head vector (quantize instantiated in codec_d256.cu, dequantize
// in codec_d256_dq.cu).
//
// Method: "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
// Apple Silicon", Methodology 1 and 2: the same fused steps as the other head
// dimensions (signs, the 128-point complex transform of z_n = u_{2n} +
// i u_{2n+1}, Hermitian packing, lambda, group absmax, rounding, packing).
//
// GB300 mapping.  One thread holding a whole d = 256 vector needs 128 complex
// values plus their Stockham copy: past the 255-register limit, it spilled
// kilobytes a thread.  Here the two lanes of a pair (lane 2r + t, t = 0, 1)
// share row r of a 16-row warp tile, and lane t loads half t of the row (z_n,
// n in [64t, 64t + 64)).  One decimation-in-frequency step splits the
// transform between them:
//   Z_{2k}   = sum_{n<64} (z_n + z_{n+64}) W_64^{nk}            (lane 0)
//   Z_{2k+1} = sum_{n<64} (z_n - z_{n+64}) W_128^n W_64^{nk}    (lane 1)
// one shuffle per value, then a 64-point FFT in each lane, the register
// footprint of d = 128.  A Hermitian pair (K, 128 - K) keeps the parity of K,
// so each lane packs its own pairs without further exchange: lane t ends with
// the packed coordinates p_{4m+2t}, p_{4m+2t+1} (m < 64) at local 2m, 2m+1.
// A group of 16 coordinates is 8 values in each lane: its absmax takes one
// more shuffle, and the nibbles of the two lanes interleave byte by byte in
// the code row (one shuffle and one byte permute per group).  The SRHT goes
// the same way: a 128-point Walsh-Hadamard transform of each half, then the
// butterfly on index bit 7 across the pair, arranged so that lane t keeps the
// outputs with index bit 1 equal to t (the same layout).  The dequantize
// kernel runs these steps backwards and ends with lane t holding half t of
// the fp16 row, which it writes into the staging tile for a TMA store.
#pragma once
#include "codec_impl.cuh"

namespace srftkv {
namespace {

constexpr int PR_ROWS = 16;                        // rows per warp tile (two lanes a row)
constexpr int PR_HALF = 128 + 8;                   // fp16 elements of one padded half row in shared memory
constexpr int PR_ROW = 2 * PR_HALF;                // fp16 elements of one row in shared memory
constexpr int PR_BUF = PR_ROWS * PR_ROW * 2;       // bytes of one tile buffer (the 5-d TMA box)
constexpr int PR_WARPS = 4;
constexpr int PR_SMEM = 128 + PR_WARPS * 2 * PR_BUF;     // quantize: two input buffers a warp
constexpr int PR_SMEM_DQ = 128 + PR_WARPS * PR_BUF;      // dequantize: one staging buffer a warp
constexpr int PR_MIN_BLOCKS = 3;
constexpr unsigned FULL = 0xffffffffu;
using C256 = SplitConst<256>;

__device__ __forceinline__ float xch(float v) { return __shfl_xor_sync(FULL, v, 1); }
__device__ __forceinline__ uint32_t xch(uint32_t v) { return __shfl_xor_sync(FULL, v, 1); }

// Sign mask word of complex index n of this lane's half (n < 64): the kernel
// parameter words are read at uniform addresses and chosen per lane.
__device__ __forceinline__ uint32_t half_mask(const CodecParams& P, int t, int n) {
    const uint32_t lo = P.sign_mask[n], hi = P.sign_mask[64 + n];
    return t ? hi : lo;
}

// ---------------------------------------------------------------------------
// Forward: the signed row in shared memory (both lanes of a pair read all of
// it, the two halves at offsets 0 and PR_HALF) -> this lane's packed
// coordinates z[2m+e] = p_{4m+2t+e}
// ---------------------------------------------------------------------------
// 16 bytes of the row = complex values z_{4c}..z_{4c+3} (c < 32), signs applied
__device__ __forceinline__ void load_signed4(const CodecParams& P, const uint16_t* row, int c, float (&re)[4],
                                             float (&im)[4]) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + (c >> 4) * PR_HALF + (c & 15) * 8);
    signed_pair(v.x, P.sign_mask[4 * c + 0], re[0], im[0]);
    signed_pair(v.y, P.sign_mask[4 * c + 1], re[1], im[1]);
    signed_pair(v.z, P.sign_mask[4 * c + 2], re[2], im[2]);
    signed_pair(v.w, P.sign_mask[4 * c + 3], re[3], im[3]);
}

__device__ __forceinline__ void pair_srft_forward(const CodecParams& P, const uint16_t* row, int t, float (&z)[128]) {
    const float sgn = t ? -1.f : 1.f;
    float zr[64], zi[64];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        float lr[4], li[4], hr[4], hi[4];
        load_signed4(P, row, c, lr, li);       // z_n, n = 4c..4c+3
        load_signed4(P, row, 16 + c, hr, hi);  // z_{n+64}
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int n = 4 * c + e;
            // lane 0: z_n + z_{n+64}; lane 1: (z_n - z_{n+64}) W_128^n, W_128^n = W_256^{2n}
            const float vr = fmaf_(sgn, hr[e], lr[e]), vi = fmaf_(sgn, hi[e], li[e]);
            if (n == 0) {
                zr[n] = vr;
                zi[n] = vi;
            } else {
                // both lanes form the product (twiddles as constant operands) and lane 0 keeps v: a select
                // between twiddle constants would hold them all in registers
                const float wr = tw_re(2 * n), wi = tw_im(2 * n);
                const float pr = fmaf_(vr, wr, -(vi * wi)), pi = fmaf_(vr, wi, vi * wr);
                zr[n] = t ? pr : vr;
                zi[n] = t ? pi : vi;
            }
        }
    }
    fft<64, false>(zr, zi);  // lane 0: X_k = Z_{2k}; lane 1: X_k = Z_{2k+1}
    // Hermitian pairs: lane 0 (X_k, X_{64-k}) = (Z_{2k}, Z_{128-2k}), k = 1..31, and the two real bins
    // Z_0 = X_0, Z_64 = X_32; lane 1 (X_k, X_{63-k}) = (Z_{2k+1}, Z_{127-2k}), k = 0..31
    float h2r[32], h2i[32];  // the partner-side outputs of pair k
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const int m0 = (64 - k) & 63, m1 = 63 - k;
        const float mr = t ? zr[m1] : zr[m0], mi = t ? zi[m1] : zi[m0];
        const int K0 = 2 * k, K1 = 2 * k + 1;
        const float a1 = t ? sp_re(split_offset(256) + K1) : sp_re(split_offset(256) + K0);
        const float a2 = t ? sp_im(split_offset(256) + K1) : sp_im(split_offset(256) + K0);
        float o0, o1, o2, o3;
        split_pair_fwd(zr[k], zi[k], mr, mi, a1, a2, C256::h, o0, o1, o2, o3);
        if (k == 0) {  // lane 0: the real bins Z_0 -> p_0, p_1 and Z_64 -> p_128, p_129
            const float s0 = (zr[0] + zi[0]) * C256::inv_sqrt_d, s1 = (zr[0] - zi[0]) * C256::inv_sqrt_d;
            const float s2 = C256::c * zr[32], s3 = -C256::c * zi[32];
            o0 = t ? o0 : s0;
            o1 = t ? o1 : s1;
            o2 = t ? o2 : s2;
            o3 = t ? o3 : s3;
        }
        z[2 * k] = o0;
        z[2 * k + 1] = o1;
        h2r[k] = o2;
        h2i[k] = o3;
    }
    // partner outputs: lane 0 puts pair k at local 128 - 2k (k >= 1) and the Z_64 bin at 64; lane 1 puts
    // pair k at 126 - 2k
#pragma unroll
    for (int j = 32; j < 64; ++j) {
        const int k0 = (j == 32) ? 0 : 64 - j, k1 = 63 - j;
        z[2 * j] = t ? h2r[k1] : h2r[k0];
        z[2 * j + 1] = t ? h2i[k1] : h2i[k0];
    }
}

// SRHT forward: d^-1/2 H_256 (signed x), Sylvester order, in the same layout.  The butterfly on index bit 1
// comes first (both of its inputs sit in one 16-byte chunk): lane t keeps output bit 1 = t,
//   v[2m+e] = u_{4m+e} + (-1)^t u_{4m+2+e},
// then a 128-point transform over the local index 2m+e carries out the other bits (0 and 2..7).
__device__ __forceinline__ void pair_srht_forward(const CodecParams& P, const uint16_t* row, int t, float (&z)[128]) {
    const float sgn = t ? -1.f : 1.f;
    float zr[64], zi[64];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        float r4[4], i4[4];
        load_signed4(P, row, c, r4, i4);  // z_{4c+j} = u_{8c+2j} + i u_{8c+2j+1}
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // m = 2c + q: z_{2m} and z_{2m+1}
            zr[2 * c + q] = fmaf_(sgn, r4[2 * q + 1], r4[2 * q]);
            zi[2 * c + q] = fmaf_(sgn, i4[2 * q + 1], i4[2 * q]);
        }
    }
    wht_pairs<64>(zr, zi);
#pragma unroll
    for (int m = 0; m < 64; ++m) {
        z[2 * m] = zr[m] * C256::inv_sqrt_d;
        z[2 * m + 1] = zi[m] * C256::inv_sqrt_d;
    }
}

// ---------------------------------------------------------------------------
// Inverse: packed coordinates (same layout) -> the lane's half of the
// transform before the last step, which pair_store_half does across the pair
// while it writes the fp16 row
// ---------------------------------------------------------------------------
// SRFT: lane 0 a_n, lane 1 W_128^{-n} b_n, where z_n = a_n + W^-n b_n and z_{n+64} = a_n - W^-n b_n
__device__ __forceinline__ void pair_srft_inverse(const float (&p)[128], int t, float (&zr)[64], float (&zi)[64]) {
    float h2r[32], h2i[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        // lane 0 partner coordinates at local 128 - 2k (k >= 1), lane 1 at 126 - 2k
        const int l0 = (k == 0) ? 64 : 128 - 2 * k, l1 = 126 - 2 * k;
        const float pm0 = t ? p[l1] : p[l0], pm1 = t ? p[l1 + 1] : p[l0 + 1];
        const int K0 = 2 * k, K1 = 2 * k + 1;
        const float a1 = t ? sp_re(split_offset(256) + K1) : sp_re(split_offset(256) + K0);
        const float a2 = t ? sp_im(split_offset(256) + K1) : sp_im(split_offset(256) + K0);
        float xr, xi, yr, yi;
        split_pair_inv(p[2 * k], p[2 * k + 1], pm0, pm1, a1, a2, C256::h, xr, xi, yr, yi);
        if (k == 0) {  // lane 0: the real bins from p_0, p_1 and p_128, p_129 (local 64, 65)
            const float s0 = (p[0] + p[1]) * C256::inv_sqrt_d, s1 = (p[0] - p[1]) * C256::inv_sqrt_d;
            const float s2 = C256::c * p[64], s3 = -C256::c * p[65];
            xr = t ? xr : s0;
            xi = t ? xi : s1;
            yr = t ? yr : s2;
            yi = t ? yi : s3;
        }
        zr[k] = xr;
        zi[k] = xi;
        h2r[k] = yr;
        h2i[k] = yi;
    }
    // partner bins: lane 0 X_{64-k} (k >= 1) and X_32 = Z_64 from k = 0; lane 1 X_{63-k}
#pragma unroll
    for (int j = 32; j < 64; ++j) {
        const int k0 = (j == 32) ? 0 : 64 - j, k1 = 63 - j;
        zr[j] = t ? h2r[k1] : h2r[k0];
        zi[j] = t ? h2i[k1] : h2i[k0];
    }
    fft<64, true>(zr, zi);  // lane 0: a_n; lane 1: b_n
#pragma unroll
    for (int n = 1; n < 64; ++n) {  // lane 1: b_n W_128^{-n} (formed in both lanes, kept by lane 1)
        const float wr = tw_re(2 * n), wi = -tw_im(2 * n);
        const float pr = fmaf_(zr[n], wr, -(zi[n] * wi)), pi = fmaf_(zr[n], wi, zi[n] * wr);
        zr[n] = t ? pr : zr[n];
        zi[n] = t ? pi : zi[n];
    }
}

// SRHT: the 128-point transform over the local index 2m+e (index bits 0 and 2..7); the butterfly on bit 1
// is the last step
__device__ __forceinline__ void pair_srht_inverse(const float (&p)[128], float (&zr)[64], float (&zi)[64]) {
#pragma unroll
    for (int m = 0; m < 64; ++m) {
        zr[m] = p[2 * m];
        zi[m] = p[2 * m + 1];
    }
    wht_pairs<64>(zr, zi);
}

// The last step across the pair, signs, fp16, and this lane's half row (half t of `row`) in shared memory
__device__ __forceinline__ void pair_store_half(const CodecParams& P, uint16_t* row, int t, bool srht,
                                                const float (&zr)[64], const float (&zi)[64]) {
    const float sgn = t ? -1.f : 1.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        float o[8];  // u_{128t+8c..128t+8c+7}
        if (!srht) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = 4 * c + j;
                // lane 0: z_n = a_n + W^-n b_n; lane 1: z_{n+64} = a_n - W^-n b_n
                o[2 * j] = fmaf_(sgn, zr[n], xch(zr[n]));
                o[2 * j + 1] = fmaf_(sgn, zi[n], xch(zi[n]));
            }
        } else {
            // output index 128t + 2n + e with n = 2m' + o1: w_0[l] + (-1)^{o1} w_1[l], l = 64t + 2m' + e
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int mq = 2 * c + q;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float lo = e ? zi[mq] : zr[mq], hi = e ? zi[32 + mq] : zr[32 + mq];
                    const float keep = t ? hi : lo, other = xch(t ? lo : hi);
                    o[4 * q + e] = (keep + other) * C256::inv_sqrt_d;
                    o[4 * q + 2 + e] = sgn * (keep - other) * C256::inv_sqrt_d;
                }
            }
        }
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half2 h = __floats2half2_rn(o[2 * j], o[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t*>(&h) ^ half_mask(P, t, 4 * c + j);
        }
        *reinterpret_cast<uint4*>(row + t * PR_HALF + 8 * c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ---------------------------------------------------------------------------
// Quantize this lane's 128 coordinates (z, lambda applied) and store them
// ---------------------------------------------------------------------------
template <int BITS, int SF>
__device__ __forceinline__ void pair_quant_store(float (&z)[128], int group, int t, bool store, uint8_t* __restrict__ crow,
                                                 uint8_t* __restrict__ srow) {
    constexpr float Q = (BITS == 4) ? 7.f : 127.f;
    constexpr float MAG = kMagic + ((BITS == 4) ? 8.f : 128.f);
    float mu[16];  // unit u: coordinates 16u..16u+15, locals 8u..8u+7 of both lanes
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        float a = fabs_(z[8 * u]);
#pragma unroll
        for (int i = 1; i < 8; ++i) a = fmax_(a, fabs_(z[8 * u + i]));
        mu[u] = fmax_(a, xch(a));
    }
#pragma unroll
    for (int s = 1; s < 16; s <<= 1) {
        if (group >= 32 * s) {
#pragma unroll
            for (int u = 0; u < 16; ++u) mu[u] = fmax_(mu[u], mu[u ^ s]);
        }
    }
    // one group unit at a time: scale, rounding, packing and the code store, so the unit's values die early
    // (the stored scales are recomputed from the maxima at the end rather than held)
    const uint32_t sel = t ? 0x3726u : 0x5140u;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        float inv, scu;
        uint32_t rawu;
        group_scale<BITS, SF>(mu[u], scu, rawu, inv);
#pragma unroll
        for (int i = 0; i < 8; ++i) z[8 * u + i] = fmaf_(z[8 * u + i], inv, MAG);
        if constexpr (SF == SRFTKV_SCALE_FP16) {
            if (mu[u] > 65504.f * Q) {  // a saturated scale can push |z/scale| past Q
#pragma unroll
                for (int i = 0; i < 8; ++i) z[8 * u + i] = fminf(fmaxf(z[8 * u + i], MAG - Q), MAG + Q);
            }
        }
        if constexpr (BITS == 4) {
            // this lane's bytes 2m + t (m = 4u..4u+3) of the group's 8 bytes; lane 0 assembles the first
            // word, lane 1 the second
            const uint32_t own = pack8_int4(&z[8 * u]);
            const uint32_t w = __byte_perm(own, xch(own), sel);
            if (store) reinterpret_cast<uint32_t*>(crow)[2 * u + t] = w;
        } else {
            // this lane's 16-bit halves of words 4u..4u+3; lane 0 assembles words 4u, 4u+1, lane 1 4u+2, 4u+3
            const uint32_t w0 = pack4_int8(&z[8 * u]), w1 = pack4_int8(&z[8 * u + 4]);
            const uint32_t other = xch(t ? w0 : w1);
            const uint32_t a = t ? other : w0, b = t ? w1 : other;
            if (store)
                reinterpret_cast<uint2*>(crow)[2 * u + t] = make_uint2(__byte_perm(a, b, 0x5410), __byte_perm(a, b, 0x7632));
        }
    }
    if (!store || t) return;
    float sc[16];
    uint32_t raw[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        float inv;
        group_scale<BITS, SF>(mu[u], sc[u], raw[u], inv);
    }
    const int gu = group >> 4, sh = __ffs(gu) - 1;
    if constexpr (SF == SRFTKV_SCALE_FP32) {
        float* sr = reinterpret_cast<float*>(srow);
        if (group == 16) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                reinterpret_cast<float4*>(sr)[i] = make_float4(sc[4 * i], sc[4 * i + 1], sc[4 * i + 2], sc[4 * i + 3]);
        } else {
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if ((u & (gu - 1)) == 0) sr[u >> sh] = sc[u];
        }
    } else if constexpr (SF == SRFTKV_SCALE_FP16) {
        uint16_t* sr = reinterpret_cast<uint16_t*>(srow);
        if (group == 16) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
                reinterpret_cast<uint4*>(sr)[i] =
                    make_uint4(raw[8 * i] | (raw[8 * i + 1] << 16), raw[8 * i + 2] | (raw[8 * i + 3] << 16),
                               raw[8 * i + 4] | (raw[8 * i + 5] << 16), raw[8 * i + 6] | (raw[8 * i + 7] << 16));
        } else {
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if ((u & (gu - 1)) == 0) sr[u >> sh] = (uint16_t)raw[u];
        }
    } else {
        if (group == 16) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
                reinterpret_cast<uint2*>(srow)[i] =
                    make_uint2(raw[8 * i] | (raw[8 * i + 1] << 8) | (raw[8 * i + 2] << 16) | (raw[8 * i + 3] << 24),
                               raw[8 * i + 4] | (raw[8 * i + 5] << 8) | (raw[8 * i + 6] << 16) | (raw[8 * i + 7] << 24));
        } else {
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if ((u & (gu - 1)) == 0) srow[u >> sh] = (uint8_t)raw[u];
        }
    }
}

// This lane's coordinates of one stored row: p[2m+e] = code * scale of p_{4m+2t+e}
template <int SF>
__device__ __forceinline__ float load_scale_t(const uint8_t* __restrict__ srow, int i) {
    if constexpr (SF == SRFTKV_SCALE_FP32) return __ldg(reinterpret_cast<const float*>(srow) + i);
    if constexpr (SF == SRFTKV_SCALE_FP16)
        return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(srow) + i)));
    return __uint_as_float((uint32_t)__ldg(srow + i) << 23);  // e8m0: the byte is the fp32 exponent field
}

template <int BITS, int SF>
__device__ __forceinline__ void pair_dequant_load(const uint8_t* __restrict__ crow, const uint8_t* __restrict__ srow,
                                                  int group, int t, float (&p)[128]) {
    const int sh = __ffs(group >> 4) - 1;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const float sc = load_scale_t<SF>(srow, u >> sh);
        if constexpr (BITS == 4) {
            // bytes 2m + t (m = 4u..4u+3) of the group's 8 bytes
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(crow) + u);
            const uint32_t own = __byte_perm(v.x, v.y, t ? 0x7531u : 0x6420u);
#pragma unroll
            for (int i = 0; i < 8; ++i) p[8 * u + i] = code_int4(own, i) * sc;
        } else {
            // 16-bit half t of words 4u..4u+3
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(crow) + u);
            const uint32_t s = t ? 0x7632u : 0x5410u;
            const uint32_t o0 = __byte_perm(v.x, v.y, s), o1 = __byte_perm(v.z, v.w, s);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                p[8 * u + i] = code_int8(o0, i) * sc;
                p[8 * u + 4 + i] = code_int8(o1, i) * sc;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// K1': fused quantize, d = 256
// ---------------------------------------------------------------------------
template <int BK, int BV, int SF, bool SRHT>
__device__ __forceinline__ void pair_quantize_tile(const CodecParams& P, const TileId& id, const uint16_t* __restrict__ buf,
                                                   int lane) {
    const int r = lane >> 1, t = lane & 1;
    const CodecSideK& S = P.side[id.side];
    const int tok = id.t0 + r;
    const uint16_t* row = buf + r * PR_ROW;
    float z[128];
    if constexpr (SRHT)
        pair_srht_forward(P, row, t, z);
    else
        pair_srft_forward(P, row, t, z);
    if (S.lambda != nullptr) {
        const float2* lr = reinterpret_cast<const float2*>(S.lambda + (long long)id.o * S.lambda_outer_stride +
                                                           (long long)id.h * 256 + 2 * t);
#pragma unroll
        for (int m = 0; m < 64; ++m) {
            const float2 l = __ldg(lr + 2 * m);  // lambda_{4m+2t}, lambda_{4m+2t+1}
            z[2 * m] *= l.x;
            z[2 * m + 1] *= l.y;
        }
    }
    // rows past n_tokens (zero fill) run along so both lanes of every pair reach the shuffles
    const bool store = tok < P.n_tokens;
    const long long vrow = packed_row(P, id, store ? tok : 0);
    if (BK == BV || id.side == 0)
        pair_quant_store<BK, SF>(z, P.group, t, store, S.codes + vrow * (256 * BK / 8),
                                 S.scales + vrow * (256 / P.group) * S.sbytes);
    else
        pair_quant_store<BV, SF>(z, P.group, t, store, S.codes + vrow * (256 * BV / 8),
                                 S.scales + vrow * (256 / P.group) * S.sbytes);
}

// One kernel per transform and scale format (a call whose sides differ in either runs as two calls), so each
// carries one path: the code of all of them together overflowed the instruction cache.
template <int BK, int BV, int SF, bool SRHT>
__global__ void __launch_bounds__(128, PR_MIN_BLOCKS)
    srft_quantize_pair_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                              const __grid_constant__ CodecParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint8_t* bufs = smem + 128 + warp * 2 * PR_BUF;
    const uint32_t bar0 = ptx::smem_u32(&bars[2 * warp]), bar1 = ptx::smem_u32(&bars[2 * warp + 1]);
    if (lane == 0) {
        ptx::mbar_init(bar0, 1);
        ptx::mbar_init(bar1, 1);
        ptx::fence_barrier_init();
    }
    __syncwarp();
    const int stride = gridDim.x * PR_WARPS;
    int tile = blockIdx.x * PR_WARPS + warp;
    auto issue = [&](int tl, int b) {
        const TileId id = decode_tile<PR_ROWS>(P, tl);
        const CUtensorMap* tm = id.side ? &tm1 : &tm0;
        const uint32_t bar = b ? bar1 : bar0;
        ptx::mbar_arrive_expect_tx(bar, PR_BUF);
        ptx::tma_load_5d(ptx::smem_u32(bufs + b * PR_BUF), tm, bar, 0, 0, id.h, id.t0, id.o);
    };
    if (lane == 0 && tile < P.total_tiles) issue(tile, 0);
    for (int it = 0; tile < P.total_tiles; ++it, tile += stride) {
        const int b = it & 1;
        const bool has_next = tile + stride < P.total_tiles;
        if (lane == 0 && has_next) issue(tile + stride, b ^ 1);
        const bool ok = __all_sync(FULL, ptx::mbar_wait_bounded(b ? bar1 : bar0, (it >> 1) & 1));
        if (!ok) {
            if (lane == 0) {
                atomicOr(P.fault, 1u);
                if (has_next) ptx::mbar_wait_bounded(b ? bar0 : bar1, ((it + 1) >> 1) & 1, 1u << 16);
            }
            return;
        }
        pair_quantize_tile<BK, BV, SF, SRHT>(P, decode_tile<PR_ROWS>(P, tile), reinterpret_cast<const uint16_t*>(bufs + b * PR_BUF),
                                   lane);
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// K2': fused dequantize, d = 256
// ---------------------------------------------------------------------------
// Prefetch the code and scale rows of a later tile into L1, one line a lane (each address inside the rows)
template <int BK, int BV>
__device__ __forceinline__ void prefetch_packed_rows(const CodecParams& P, int tile, int lane) {
    const TileId id = decode_tile<PR_ROWS>(P, tile);
    const CodecSideK& S = P.side[id.side];
    const int rows = min(PR_ROWS, P.n_tokens - id.t0);
    const long long v0 = packed_row(P, id, 0);
    const int cb = (BK == BV || id.side == 0) ? 256 * BK / 8 : 256 * BV / 8, sb = (256 / P.group) * S.sbytes;
    const char* c0 = reinterpret_cast<const char*>(S.codes + v0 * cb);
    const char* s0 = reinterpret_cast<const char*>(S.scales + v0 * sb);
    const int clen = rows * cb, slen = rows * sb;
    for (int i = lane; i <= (clen >> 7); i += 32) {
        const char* a = c0 + min(i << 7, clen - 1);
        asm volatile("prefetch.global.L1 [%0];" ::"l"(a));
    }
    if (lane <= (slen >> 7)) {
        const char* a = s0 + min(lane << 7, slen - 1);
        asm volatile("prefetch.global.L1 [%0];" ::"l"(a));
    }
}

template <int BK, int BV, int SF, bool SRHT>
__global__ void __launch_bounds__(128, PR_MIN_BLOCKS)
    srft_dequantize_pair_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                                const __grid_constant__ CodecParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 1, t = lane & 1;
    uint16_t* buf = reinterpret_cast<uint16_t*>(smem + 128 + warp * PR_BUF);
    const int stride = gridDim.x * PR_WARPS;
    int tile = blockIdx.x * PR_WARPS + warp;
    if (tile < P.total_tiles) prefetch_packed_rows<BK, BV>(P, tile, lane);
    for (; tile < P.total_tiles; tile += stride) {
        // the loads of this tile find their lines in L1; the next tile's are requested now
        if (tile + stride < P.total_tiles) prefetch_packed_rows<BK, BV>(P, tile + stride, lane);
        const TileId id = decode_tile<PR_ROWS>(P, tile);
        const CodecSideK& S = P.side[id.side];
        const int tok = id.t0 + r;
        float p[128];
        if (tok < P.n_tokens) {
            const long long vrow = packed_row(P, id, tok);
            const uint8_t* srow = S.scales + vrow * (256 / P.group) * S.sbytes;
            if (BK == BV || id.side == 0)
                pair_dequant_load<BK, SF>(S.codes + vrow * (256 * BK / 8), srow, P.group, t, p);
            else
                pair_dequant_load<BV, SF>(S.codes + vrow * (256 * BV / 8), srow, P.group, t, p);
            if (S.lambda != nullptr) {
                const float2* lr = reinterpret_cast<const float2*>(S.lambda + (long long)id.o * S.lambda_outer_stride +
                                                                   (long long)id.h * 256 + 2 * t);
#pragma unroll
                for (int m = 0; m < 64; ++m) {
                    const float2 l = __ldg(lr + 2 * m);
                    p[2 * m] *= __frcp_rn(l.x);
                    p[2 * m + 1] *= __frcp_rn(l.y);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 128; ++i) p[i] = 0.f;
        }
        float zr[64], zi[64];
        if constexpr (SRHT)
            pair_srht_inverse(p, zr, zi);
        else
            pair_srft_inverse(p, t, zr, zi);
        // the previous tile's store, issued a whole tile of work ago, must have read the staging buffer
        if (lane == 0) ptx::bulk_wait_read<0>();
        __syncwarp();
        pair_store_half(P, buf + r * PR_ROW, t, SRHT, zr, zi);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const CUtensorMap* tm = id.side ? &tm1 : &tm0;
            ptx::tma_store_5d(tm, ptx::smem_u32(buf), 0, 0, id.h, id.t0, id.o);
            ptx::bulk_commit();
        }
    }
    if (lane == 0) ptx::bulk_wait<0>();
}

template <bool QUANTIZE, int BK, int BV, int SF, bool SRHT>
int launch_pair(const CodecCall& c) {
    if ((long long)c.n_sides * c.n_outer * c.H * ((c.n_tokens + PR_ROWS - 1) / PR_ROWS) > 0x7fffffffll) {
        set_error("sizes too large for 32-bit tile indexing at d = 256");
        return SRFTKV_ERR_INVALID;
    }
    CodecParams P;
    fill_params(c, P);
    P.tiles_per_head = (c.n_tokens + PR_ROWS - 1) / PR_ROWS;
    P.tiles_per_side = c.n_outer * c.H * P.tiles_per_head;
    P.total_tiles = c.n_sides * P.tiles_per_side;
    if (P.total_tiles == 0) return 0;
    CUtensorMap tm[2];
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        if (!encode_x_map(&tm[s], d.x, 256, c.H, c.n_tokens, c.n_outer, PR_ROWS, false)) return SRFTKV_ERR_CUDA;
    }
    P.fault = codec_fault_word();
    if (!P.fault) return SRFTKV_ERR_CUDA;
    auto kern = [] {
        if constexpr (QUANTIZE)
            return srft_quantize_pair_kernel<BK, BV, SF, SRHT>;
        else
            return srft_dequantize_pair_kernel<BK, BV, SF, SRHT>;
    }();
    const int smem_bytes = QUANTIZE ? PR_SMEM : PR_SMEM_DQ;
    static bool attr_done = false;
    if (!attr_done) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        attr_done = true;
    }
    int blocks = (P.total_tiles + PR_WARPS - 1) / PR_WARPS;
    const int cap = device_sm_count() * PR_MIN_BLOCKS;
    if (blocks > cap) blocks = cap;
    kern<<<blocks, PR_WARPS * 32, smem_bytes, c.stream>>>(tm[0], tm[1], P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("codec kernel launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return 0;
}

template <bool Q, int BK, int BV>
int launch_pair_bits(const CodecCall& c) {
    // both sides of one launch share the transform and the scale format
    const bool srht = c.side[0].transform == SRFTKV_TRANSFORM_SRHT;
    switch (c.side[0].scale_format) {
        case SRFTKV_SCALE_FP32:
            return srht ? launch_pair<Q, BK, BV, SRFTKV_SCALE_FP32, true>(c)
                        : launch_pair<Q, BK, BV, SRFTKV_SCALE_FP32, false>(c);
        case SRFTKV_SCALE_FP16:
            return srht ? launch_pair<Q, BK, BV, SRFTKV_SCALE_FP16, true>(c)
                        : launch_pair<Q, BK, BV, SRFTKV_SCALE_FP16, false>(c);
        default:
            return srht ? launch_pair<Q, BK, BV, SRFTKV_SCALE_E8M0, true>(c)
                        : launch_pair<Q, BK, BV, SRFTKV_SCALE_E8M0, false>(c);
    }
}

template <bool Q>
int launch_pair_all(const CodecCall& c) {
    if (c.n_sides == 2 && (c.side[0].transform != c.side[1].transform ||
                           c.side[0].scale_format != c.side[1].scale_format)) {
        set_error("d = 256 launch with sides of different transforms or scale formats");
        return SRFTKV_ERR_INVALID;
    }
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    if (bk == 4 && bv == 4) return launch_pair_bits<Q, 4, 4>(c);
    if (bk == 8 && bv == 8) return launch_pair_bits<Q, 8, 8>(c);
    if (bk == 8 && bv == 4) return launch_pair_bits<Q, 8, 4>(c);
    return launch_pair_bits<Q, 4, 8>(c);
}

}  // namespace

// defined in codec_d256_dq.cu
int pair_dequantize_d256(const CodecCall& c);

}  // namespace srftkv
