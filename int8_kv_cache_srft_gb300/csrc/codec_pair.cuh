// codec_pair.cuh -- quantize / dequantize kernels for head dimensions 192 and
// 256, two threads per head vector (instantiated in codec_d192.cu,
// codec_d192_dq.cu, codec_d256.cu and codec_d256_dq.cu).
//
// Method: "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
// Apple Silicon", Methodology 1 and 2: the same fused steps as the other head
// dimensions (signs, the N = d/2 point complex transform of z_n = u_{2n} +
// i u_{2n+1}, Hermitian packing, lambda, group absmax, rounding, packing).
// Methodology 1 credits the SRFT with dimensions that are not powers of two:
// d = 192 runs the same steps with a mixed-radix (3 x 16) transform.
//
// GB300 mapping.  One thread holding a whole d = 256 vector needs 128 complex
// values plus their Stockham copy: past the 255-register limit, it spilled
// kilobytes a thread.  Here the two lanes of a pair (lane 2r + t, t = 0, 1)
// share row r of a 16-row warp tile, with H = d/4 complex values each.  One
// decimation-in-frequency step splits the transform between them:
//   Z_{2k}   = sum_{n<H} (z_n + z_{n+H}) W_H^{nk}             (lane 0)
//   Z_{2k+1} = sum_{n<H} (z_n - z_{n+H}) W_N^n W_H^{nk}       (lane 1)
// both lanes reading both halves of the row from the TMA tile, then an
// H-point FFT in each lane (radix 2 for H = 64; 3 x 16 for H = 48).  A
// Hermitian pair (K, N - K) keeps the parity of K, so each lane packs its own
// pairs without exchange: lane t ends with the packed coordinates p_{4m+2t},
// p_{4m+2t+1} (m < H) at local 2m, 2m+1.  A group of 16 coordinates is 8
// values in each lane: its absmax takes one shuffle, and the nibbles of the
// two lanes interleave byte by byte in the code row (one shuffle and one byte
// permute per group).  The SRHT (d = 256) does the butterfly on index bit 1
// first, whose two inputs sit in one 16-byte chunk, then a 128-point
// Walsh-Hadamard transform in each lane: the same layout.  The dequantize
// kernel runs the steps backwards and ends with the one exchange across the
// pair, fused with the fp16 stores of half t of the row.
#pragma once
#include "codec_impl.cuh"

namespace srftkv {
namespace {

constexpr int PR_ROWS = 16;  // rows per warp tile (two lanes a row)
constexpr int PR_WARPS = 4;
constexpr int PR_MIN_BLOCKS = 3;
constexpr unsigned FULL = 0xffffffffu;

constexpr double csqrt(double x) {  // Newton's iteration, for compile-time constants
    double r = x > 1.0 ? x : 1.0;
    for (int i = 0; i < 64; ++i) r = 0.5 * (r + x / r);
    return r;
}

template <int D>
struct PairGeo {
    static constexpr int HALF = D / 2;                  // fp16 elements of a half row
    static constexpr int HP = HALF + 8;                 // padded half row in shared memory (the TMA box)
    static constexpr int ROW = 2 * HP;                  // fp16 elements of one row in shared memory
    static constexpr int BUF = PR_ROWS * ROW * 2;       // bytes of one tile buffer
    static constexpr int SMEM = 128 + PR_WARPS * 2 * BUF;   // quantize: two input buffers a warp
    static constexpr int SMEM_DQ = 128 + PR_WARPS * BUF;    // dequantize: one staging buffer a warp
    static constexpr int H = D / 4;                     // complex values per lane
    static constexpr int L = D / 2;                     // packed coordinates per lane
    static constexpr int U = D / 16;                    // 16-coordinate units (groups of 16)
    static constexpr int CH = D / 16;                   // 16-byte chunks of a half row
    static constexpr float isd = float(1.0 / csqrt(D));            // d^-1/2
    static constexpr float c = float(csqrt(2.0 / D));              // sqrt(2/d)
    static constexpr float h = float(1.0 / csqrt(2.0 * D));        // 1/sqrt(2d)
};

// W_192^m (m < 192) and the d = 192 split-step twiddles h W_192^k (k < 48)
struct Tw192 {
    float re[192], im[192];
    float sre[48], sim[48];
};
constexpr Tw192 make_tw192() {
    Tw192 t{};
    const double h = 1.0 / csqrt(384.0);
    for (int m = 0; m < 192; ++m) {
        double cv = 0, sv = 0;
        trig::cos_sin_2pi(m, 192, cv, sv);
        t.re[m] = float(cv);
        t.im[m] = float(-sv);
        if (m < 48) {
            t.sre[m] = float(h * cv);
            t.sim[m] = float(-h * sv);
        }
    }
    return t;
}
static __constant__ Tw192 c_tw192 = make_tw192();

// W_D^m and h W_D^k for the two head dimensions (constant-bank operands: every index is a compile-time constant)
template <int D>
__device__ __forceinline__ float pw_re(int m) {
    if constexpr (D == 256) return tw_re(m); else return c_tw192.re[m];
}
template <int D>
__device__ __forceinline__ float pw_im(int m) {
    if constexpr (D == 256) return tw_im(m); else return c_tw192.im[m];
}
template <int D>
__device__ __forceinline__ float psp_re(int k) {
    if constexpr (D == 256) return sp_re(split_offset(256) + k); else return c_tw192.sre[k];
}
template <int D>
__device__ __forceinline__ float psp_im(int k) {
    if constexpr (D == 256) return sp_im(split_offset(256) + k); else return c_tw192.sim[k];
}

// 48-point DFT, unnormalised (conjugate twiddles for INV), 48 = 3 x 16 (Cooley-Tukey): X_{k+16q} =
// sum_r W_3^{rq} W_48^{rk} Y_r[k], with Y_r the 16-point FFT of x_{3j+r}
template <bool INV>
__device__ __forceinline__ void fft48(float (&re)[48], float (&im)[48]) {
    float ar[3][16], ai[3][16];
#pragma unroll
    for (int r = 0; r < 3; ++r) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            ar[r][j] = re[3 * j + r];
            ai[r][j] = im[3 * j + r];
        }
        fft<16, INV>(ar[r], ai[r]);
    }
#pragma unroll
    for (int r = 1; r < 3; ++r) {
#pragma unroll
        for (int k = 1; k < 16; ++k) {  // W_48^{rk} = W_192^{4rk}
            const float wr = c_tw192.re[4 * r * k], wi = INV ? -c_tw192.im[4 * r * k] : c_tw192.im[4 * r * k];
            const float xr = ar[r][k], xi = ai[r][k];
            ar[r][k] = fmaf_(xr, wr, -(xi * wi));
            ai[r][k] = fmaf_(xr, wi, xi * wr);
        }
    }
    // W_3 = -1/2 + i s3 with s3 = -sqrt(3)/2 (forward) or +sqrt(3)/2 (inverse)
    constexpr float s3 = INV ? 0.866025403784438647f : -0.866025403784438647f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float sr = ar[1][k] + ar[2][k], si = ai[1][k] + ai[2][k];
        const float dr = ar[1][k] - ar[2][k], di = ai[1][k] - ai[2][k];
        const float mr = fmaf_(-0.5f, sr, ar[0][k]), mi = fmaf_(-0.5f, si, ai[0][k]);
        re[k] = ar[0][k] + sr;
        im[k] = ai[0][k] + si;
        re[k + 16] = fmaf_(-s3, di, mr);  // m + i s3 d
        im[k + 16] = fmaf_(s3, dr, mi);
        re[k + 32] = fmaf_(s3, di, mr);   // m - i s3 d
        im[k + 32] = fmaf_(-s3, dr, mi);
    }
}

template <int D, bool INV>
__device__ __forceinline__ void lane_fft(float (&re)[D / 4], float (&im)[D / 4]) {
    if constexpr (D == 256)
        fft<64, INV>(re, im);
    else
        fft48<INV>(re, im);
}

__device__ __forceinline__ float xch(float v) { return __shfl_xor_sync(FULL, v, 1); }
__device__ __forceinline__ uint32_t xch(uint32_t v) { return __shfl_xor_sync(FULL, v, 1); }

// Sign mask word of complex index n of this lane's half (n < H): the kernel
// parameter words are read at uniform addresses and chosen per lane.
template <int D>
__device__ __forceinline__ uint32_t half_mask(const CodecParams& P, int t, int n) {
    const uint32_t lo = P.sign_mask[n], hi = P.sign_mask[D / 4 + n];
    return t ? hi : lo;
}

// ---------------------------------------------------------------------------
// Forward: the signed row in shared memory (both lanes of a pair read all of
// it, the two halves at offsets 0 and HP) -> this lane's packed coordinates
// z[2m+e] = p_{4m+2t+e}
// ---------------------------------------------------------------------------
// 16 bytes of the row = complex values z_{4c}..z_{4c+3} (c < d/8), signs applied
template <int D>
__device__ __forceinline__ void load_signed4(const CodecParams& P, const uint16_t* row, int c, float (&re)[4],
                                             float (&im)[4]) {
    using G = PairGeo<D>;
    const uint4 v = *reinterpret_cast<const uint4*>(row + (c / G::CH) * G::HP + (c % G::CH) * 8);
    signed_pair(v.x, P.sign_mask[4 * c + 0], re[0], im[0]);
    signed_pair(v.y, P.sign_mask[4 * c + 1], re[1], im[1]);
    signed_pair(v.z, P.sign_mask[4 * c + 2], re[2], im[2]);
    signed_pair(v.w, P.sign_mask[4 * c + 3], re[3], im[3]);
}

template <int D>
__device__ __forceinline__ void pair_srft_forward(const CodecParams& P, const uint16_t* row, int t,
                                                  float (&z)[D / 2]) {
    using G = PairGeo<D>;
    constexpr int H = G::H;
    const float sgn = t ? -1.f : 1.f;
    float zr[H], zi[H];
#pragma unroll
    for (int c = 0; c < G::CH; ++c) {
        float lr[4], li[4], hr[4], hi[4];
        load_signed4<D>(P, row, c, lr, li);          // z_n, n = 4c..4c+3
        load_signed4<D>(P, row, G::CH + c, hr, hi);  // z_{n+H}
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int n = 4 * c + e;
            // lane 0: z_n + z_{n+H}; lane 1: (z_n - z_{n+H}) W_N^n, W_N^n = W_D^{2n}
            const float vr = fmaf_(sgn, hr[e], lr[e]), vi = fmaf_(sgn, hi[e], li[e]);
            if (n == 0) {
                zr[n] = vr;
                zi[n] = vi;
            } else {
                // both lanes form the product (twiddles as constant operands) and lane 0 keeps v: a select
                // between twiddle constants would hold them all in registers
                const float wr = pw_re<D>(2 * n), wi = pw_im<D>(2 * n);
                const float pr = fmaf_(vr, wr, -(vi * wi)), pi = fmaf_(vr, wi, vi * wr);
                zr[n] = t ? pr : vr;
                zi[n] = t ? pi : vi;
            }
        }
    }
    lane_fft<D, false>(zr, zi);  // lane 0: X_k = Z_{2k}; lane 1: X_k = Z_{2k+1}
    // Hermitian pairs: lane 0 (X_k, X_{H-k}) = (Z_{2k}, Z_{N-2k}), k = 1..H/2-1, and the two real bins
    // Z_0 = X_0, Z_{N/2} = X_{H/2}; lane 1 (X_k, X_{H-1-k}) = (Z_{2k+1}, Z_{N-1-2k}), k = 0..H/2-1
    float h2r[H / 2], h2i[H / 2];  // the partner-side outputs of pair k
#pragma unroll
    for (int k = 0; k < H / 2; ++k) {
        const int m0 = (k == 0) ? 0 : H - k, m1 = H - 1 - k;
        const float mr = t ? zr[m1] : zr[m0], mi = t ? zi[m1] : zi[m0];
        const int K0 = 2 * k, K1 = 2 * k + 1;
        const float a1 = t ? psp_re<D>(K1) : psp_re<D>(K0);
        const float a2 = t ? psp_im<D>(K1) : psp_im<D>(K0);
        float o0, o1, o2, o3;
        split_pair_fwd(zr[k], zi[k], mr, mi, a1, a2, G::h, o0, o1, o2, o3);
        if (k == 0) {  // lane 0: the real bins Z_0 -> p_0, p_1 and Z_{N/2} -> p_N, p_{N+1}
            const float s0 = (zr[0] + zi[0]) * G::isd, s1 = (zr[0] - zi[0]) * G::isd;
            const float s2 = G::c * zr[H / 2], s3 = -G::c * zi[H / 2];
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
    // partner outputs: lane 0 puts pair k at local 2(H - k) (k >= 1) and the Z_{N/2} bin at H; lane 1 puts
    // pair k at 2(H - 1 - k)
#pragma unroll
    for (int j = H / 2; j < H; ++j) {
        const int k0 = (j == H / 2) ? 0 : H - j, k1 = H - 1 - j;
        z[2 * j] = t ? h2r[k1] : h2r[k0];
        z[2 * j + 1] = t ? h2i[k1] : h2i[k0];
    }
}

// SRHT forward (d = 256): d^-1/2 H_256 (signed x), Sylvester order, in the same layout.  The butterfly on
// index bit 1 comes first (both of its inputs sit in one 16-byte chunk): lane t keeps output bit 1 = t,
//   v[2m+e] = u_{4m+e} + (-1)^t u_{4m+2+e},
// then a 128-point transform over the local index 2m+e carries out the other bits (0 and 2..7).
__device__ __forceinline__ void pair_srht_forward(const CodecParams& P, const uint16_t* row, int t, float (&z)[128]) {
    const float sgn = t ? -1.f : 1.f;
    float zr[64], zi[64];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        float r4[4], i4[4];
        load_signed4<256>(P, row, c, r4, i4);  // z_{4c+j} = u_{8c+2j} + i u_{8c+2j+1}
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // m = 2c + q: z_{2m} and z_{2m+1}
            zr[2 * c + q] = fmaf_(sgn, r4[2 * q + 1], r4[2 * q]);
            zi[2 * c + q] = fmaf_(sgn, i4[2 * q + 1], i4[2 * q]);
        }
    }
    wht_pairs<64>(zr, zi);
#pragma unroll
    for (int m = 0; m < 64; ++m) {
        z[2 * m] = zr[m] * PairGeo<256>::isd;
        z[2 * m + 1] = zi[m] * PairGeo<256>::isd;
    }
}

// ---------------------------------------------------------------------------
// Inverse: packed coordinates (same layout) -> the lane's half of the
// transform before the last step, which pair_store_half does across the pair
// while it writes the fp16 row
// ---------------------------------------------------------------------------
// SRFT: lane 0 a_n, lane 1 W_N^{-n} b_n, where z_n = a_n + W^-n b_n and z_{n+H} = a_n - W^-n b_n
template <int D>
__device__ __forceinline__ void pair_srft_inverse(const float (&p)[D / 2], int t, float (&zr)[D / 4],
                                                  float (&zi)[D / 4]) {
    using G = PairGeo<D>;
    constexpr int H = G::H;
    float h2r[H / 2], h2i[H / 2];
#pragma unroll
    for (int k = 0; k < H / 2; ++k) {
        // lane 0 partner coordinates at local 2(H - k) (k >= 1), lane 1 at 2(H - 1 - k)
        const int l0 = (k == 0) ? H : 2 * (H - k), l1 = 2 * (H - 1 - k);
        const float pm0 = t ? p[l1] : p[l0], pm1 = t ? p[l1 + 1] : p[l0 + 1];
        const int K0 = 2 * k, K1 = 2 * k + 1;
        const float a1 = t ? psp_re<D>(K1) : psp_re<D>(K0);
        const float a2 = t ? psp_im<D>(K1) : psp_im<D>(K0);
        float xr, xi, yr, yi;
        split_pair_inv(p[2 * k], p[2 * k + 1], pm0, pm1, a1, a2, G::h, xr, xi, yr, yi);
        if (k == 0) {  // lane 0: the real bins from p_0, p_1 and p_N, p_{N+1} (local H, H + 1)
            const float s0 = (p[0] + p[1]) * G::isd, s1 = (p[0] - p[1]) * G::isd;
            const float s2 = G::c * p[H], s3 = -G::c * p[H + 1];
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
    // partner bins: lane 0 X_{H-k} (k >= 1) and X_{H/2} = Z_{N/2} from k = 0; lane 1 X_{H-1-k}
#pragma unroll
    for (int j = H / 2; j < H; ++j) {
        const int k0 = (j == H / 2) ? 0 : H - j, k1 = H - 1 - j;
        zr[j] = t ? h2r[k1] : h2r[k0];
        zi[j] = t ? h2i[k1] : h2i[k0];
    }
    lane_fft<D, true>(zr, zi);  // lane 0: a_n; lane 1: b_n
#pragma unroll
    for (int n = 1; n < H; ++n) {  // lane 1: b_n W_N^{-n} (formed in both lanes, kept by lane 1)
        const float wr = pw_re<D>(2 * n), wi = -pw_im<D>(2 * n);
        const float pr = fmaf_(zr[n], wr, -(zi[n] * wi)), pi = fmaf_(zr[n], wi, zi[n] * wr);
        zr[n] = t ? pr : zr[n];
        zi[n] = t ? pi : zi[n];
    }
}

// SRHT (d = 256): the 128-point transform over the local index 2m+e (index bits 0 and 2..7); the
// butterfly on bit 1 is the last step
__device__ __forceinline__ void pair_srht_inverse(const float (&p)[128], float (&zr)[64], float (&zi)[64]) {
#pragma unroll
    for (int m = 0; m < 64; ++m) {
        zr[m] = p[2 * m];
        zi[m] = p[2 * m + 1];
    }
    wht_pairs<64>(zr, zi);
}

// The last step across the pair, signs, fp16, and this lane's half row (half t of `row`) in shared memory
template <int D, bool SRHT>
__device__ __forceinline__ void pair_store_half(const CodecParams& P, uint16_t* row, int t, const float (&zr)[D / 4],
                                                const float (&zi)[D / 4]) {
    using G = PairGeo<D>;
    const float sgn = t ? -1.f : 1.f;
#pragma unroll
    for (int c = 0; c < G::CH; ++c) {
        float o[8];  // u_{D/2 t + 8c .. + 7}
        if constexpr (!SRHT) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = 4 * c + j;
                // lane 0: z_n = a_n + W^-n b_n; lane 1: z_{n+H} = a_n - W^-n b_n
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
                    o[4 * q + e] = (keep + other) * G::isd;
                    o[4 * q + 2 + e] = sgn * (keep - other) * G::isd;
                }
            }
        }
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half2 h = __floats2half2_rn(o[2 * j], o[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t*>(&h) ^ half_mask<D>(P, t, 4 * c + j);
        }
        *reinterpret_cast<uint4*>(row + t * G::HP + 8 * c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ---------------------------------------------------------------------------
// Quantize this lane's D/2 coordinates (z, lambda applied) and store them
// ---------------------------------------------------------------------------
template <int D, int BITS, int SF>
__device__ __forceinline__ void pair_quant_store(float (&z)[D / 2], int group, int t, bool store,
                                                 uint8_t* __restrict__ crow, uint8_t* __restrict__ srow) {
    constexpr int U = PairGeo<D>::U;
    constexpr float Q = (BITS == 4) ? 7.f : 127.f;
    constexpr float MAG = kMagic + ((BITS == 4) ? 8.f : 128.f);
    float mu[U];  // unit u: coordinates 16u..16u+15, locals 8u..8u+7 of both lanes
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float a = fabs_(z[8 * u]);
#pragma unroll
        for (int i = 1; i < 8; ++i) a = fmax_(a, fabs_(z[8 * u + i]));
        mu[u] = fmax_(a, xch(a));
    }
    // widen to the group: U is a multiple of group/16 (a power of two dividing d)
#pragma unroll
    for (int s = 1; s < U; s <<= 1) {
        if (group >= 32 * s) {
#pragma unroll
            for (int u = 0; u < U; ++u)
                if ((u ^ s) < U) mu[u] = fmax_(mu[u], mu[u ^ s]);
        }
    }
    // one group unit at a time: scale, rounding, packing and the code store, so the unit's values die early
    // (the stored scales are recomputed from the maxima at the end rather than held)
    const uint32_t sel = t ? 0x3726u : 0x5140u;
#pragma unroll
    for (int u = 0; u < U; ++u) {
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
    float sc[U];
    uint32_t raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float inv;
        group_scale<BITS, SF>(mu[u], sc[u], raw[u], inv);
    }
    const int gu = group >> 4, sh = __ffs(gu) - 1;
    if (group == 16 && D == 256) {  // 64 / 32 / 16-byte scale rows: vector stores
        if constexpr (SF == SRFTKV_SCALE_FP32) {
#pragma unroll
            for (int i = 0; i < U / 4; ++i)
                reinterpret_cast<float4*>(srow)[i] = make_float4(sc[4 * i], sc[4 * i + 1], sc[4 * i + 2], sc[4 * i + 3]);
        } else if constexpr (SF == SRFTKV_SCALE_FP16) {
#pragma unroll
            for (int i = 0; i < U / 8; ++i)
                reinterpret_cast<uint4*>(srow)[i] =
                    make_uint4(raw[8 * i] | (raw[8 * i + 1] << 16), raw[8 * i + 2] | (raw[8 * i + 3] << 16),
                               raw[8 * i + 4] | (raw[8 * i + 5] << 16), raw[8 * i + 6] | (raw[8 * i + 7] << 16));
        } else {
#pragma unroll
            for (int i = 0; i < U / 8; ++i)
                reinterpret_cast<uint2*>(srow)[i] =
                    make_uint2(raw[8 * i] | (raw[8 * i + 1] << 8) | (raw[8 * i + 2] << 16) | (raw[8 * i + 3] << 24),
                               raw[8 * i + 4] | (raw[8 * i + 5] << 8) | (raw[8 * i + 6] << 16) | (raw[8 * i + 7] << 24));
        }
    } else if (group == 16) {  // d = 192: 48 / 24 / 12-byte rows, 4-byte aligned: one word at a time
        if constexpr (SF == SRFTKV_SCALE_FP32) {
#pragma unroll
            for (int u = 0; u < U; ++u) reinterpret_cast<float*>(srow)[u] = sc[u];
        } else if constexpr (SF == SRFTKV_SCALE_FP16) {
#pragma unroll
            for (int i = 0; i < U / 2; ++i) reinterpret_cast<uint32_t*>(srow)[i] = raw[2 * i] | (raw[2 * i + 1] << 16);
        } else {
#pragma unroll
            for (int i = 0; i < U / 4; ++i)
                reinterpret_cast<uint32_t*>(srow)[i] =
                    raw[4 * i] | (raw[4 * i + 1] << 8) | (raw[4 * i + 2] << 16) | (raw[4 * i + 3] << 24);
        }
    } else {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if ((u & (gu - 1)) != 0) continue;
            if constexpr (SF == SRFTKV_SCALE_FP32)
                reinterpret_cast<float*>(srow)[u >> sh] = sc[u];
            else if constexpr (SF == SRFTKV_SCALE_FP16)
                reinterpret_cast<uint16_t*>(srow)[u >> sh] = (uint16_t)raw[u];
            else
                srow[u >> sh] = (uint8_t)raw[u];
        }
    }
}

template <int SF>
__device__ __forceinline__ float load_scale_t(const uint8_t* __restrict__ srow, int i) {
    if constexpr (SF == SRFTKV_SCALE_FP32) return __ldg(reinterpret_cast<const float*>(srow) + i);
    if constexpr (SF == SRFTKV_SCALE_FP16)
        return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(srow) + i)));
    return __uint_as_float((uint32_t)__ldg(srow + i) << 23);  // e8m0: the byte is the fp32 exponent field
}

// This lane's coordinates of one stored row: p[2m+e] = code * scale of p_{4m+2t+e}
template <int D, int BITS, int SF>
__device__ __forceinline__ void pair_dequant_load(const uint8_t* __restrict__ crow, const uint8_t* __restrict__ srow,
                                                  int group, int t, float (&p)[D / 2]) {
    const int sh = __ffs(group >> 4) - 1;
#pragma unroll
    for (int u = 0; u < PairGeo<D>::U; ++u) {
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
// K1': fused quantize, d = 192 and 256
// ---------------------------------------------------------------------------
template <int D, int BK, int BV, int SF, bool SRHT>
__device__ __forceinline__ void pair_quantize_tile(const CodecParams& P, const TileId& id, const uint16_t* __restrict__ buf,
                                                   int lane) {
    using G = PairGeo<D>;
    const int r = lane >> 1, t = lane & 1;
    const CodecSideK& S = P.side[id.side];
    const int tok = id.t0 + r;
    const uint16_t* row = buf + r * G::ROW;
    float z[G::L];
    if constexpr (SRHT)
        pair_srht_forward(P, row, t, z);
    else
        pair_srft_forward<D>(P, row, t, z);
    if (S.lambda != nullptr) {
        const float2* lr = reinterpret_cast<const float2*>(S.lambda + (long long)id.o * S.lambda_outer_stride +
                                                           (long long)id.h * D + 2 * t);
#pragma unroll
        for (int m = 0; m < G::H; ++m) {
            const float2 l = __ldg(lr + 2 * m);  // lambda_{4m+2t}, lambda_{4m+2t+1}
            z[2 * m] *= l.x;
            z[2 * m + 1] *= l.y;
        }
    }
    // rows past n_tokens (zero fill) run along so both lanes of every pair reach the shuffles
    const bool store = tok < P.n_tokens;
    const long long vrow = packed_row(P, id, store ? tok : 0);
    if (BK == BV || id.side == 0)
        pair_quant_store<D, BK, SF>(z, P.group, t, store, S.codes + vrow * (D * BK / 8),
                                    S.scales + vrow * (D / P.group) * S.sbytes);
    else
        pair_quant_store<D, BV, SF>(z, P.group, t, store, S.codes + vrow * (D * BV / 8),
                                    S.scales + vrow * (D / P.group) * S.sbytes);
}

// One kernel per transform and scale format (a call whose sides differ in either runs as two calls), so each
// carries one path: the code of all of them together overflowed the instruction cache.
template <int D, int BK, int BV, int SF, bool SRHT>
__global__ void __launch_bounds__(128, PR_MIN_BLOCKS)
    srft_quantize_pair_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                              const __grid_constant__ CodecParams P) {
    using G = PairGeo<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint8_t* bufs = smem + 128 + warp * 2 * G::BUF;
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
        ptx::mbar_arrive_expect_tx(bar, G::BUF);
        ptx::tma_load_5d(ptx::smem_u32(bufs + b * G::BUF), tm, bar, 0, 0, id.h, id.t0, id.o);
    };
    if (lane == 0 && tile < P.total_tiles) issue(tile, 0);
    for (int it = 0; tile < P.total_tiles; ++it, tile += stride) {
        const int b = it & 1;
        const bool has_next = tile + stride < P.total_tiles;
        if (lane == 0 && has_next) issue(tile + stride, b ^ 1);
        const bool ok = __all_sync(FULL, ptx::mbar_wait_bounded(b ? bar1 : bar0, (it >> 1) & 1, P.poll_limit));
        if (!ok) {
            if (lane == 0) {
                atomicOr(P.fault, 1u);
                // let this warp's copies in flight land before it leaves: the stage whose wait gave up and the
                // one issued after it (each wait bounded, so the warp still returns)
                ptx::mbar_wait_bounded(b ? bar1 : bar0, (it >> 1) & 1, 1u << 16);
                if (has_next) ptx::mbar_wait_bounded(b ? bar0 : bar1, ((it + 1) >> 1) & 1, 1u << 16);
            }
            return;
        }
        pair_quantize_tile<D, BK, BV, SF, SRHT>(P, decode_tile<PR_ROWS>(P, tile),
                                                reinterpret_cast<const uint16_t*>(bufs + b * G::BUF), lane);
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// K2': fused dequantize, d = 192 and 256
// ---------------------------------------------------------------------------
// Prefetch the code and scale rows of a later tile into L1, one line a lane (each address inside the rows)
template <int D, int BK, int BV>
__device__ __forceinline__ void prefetch_packed_rows(const CodecParams& P, int tile, int lane) {
    const TileId id = decode_tile<PR_ROWS>(P, tile);
    const CodecSideK& S = P.side[id.side];
    const int rows = min(PR_ROWS, P.n_tokens - id.t0);
    const long long v0 = packed_row(P, id, 0);
    const int cb = (BK == BV || id.side == 0) ? D * BK / 8 : D * BV / 8, sb = (D / P.group) * S.sbytes;
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

template <int D, int BK, int BV, int SF, bool SRHT>
__global__ void __launch_bounds__(128, PR_MIN_BLOCKS)
    srft_dequantize_pair_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                                const __grid_constant__ CodecParams P) {
    using G = PairGeo<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 1, t = lane & 1;
    uint16_t* buf = reinterpret_cast<uint16_t*>(smem + 128 + warp * G::BUF);
    const int stride = gridDim.x * PR_WARPS;
    int tile = blockIdx.x * PR_WARPS + warp;
    if (tile < P.total_tiles) prefetch_packed_rows<D, BK, BV>(P, tile, lane);
    for (; tile < P.total_tiles; tile += stride) {
        // the loads of this tile find their lines in L1; the next tile's are requested now
        if (tile + stride < P.total_tiles) prefetch_packed_rows<D, BK, BV>(P, tile + stride, lane);
        const TileId id = decode_tile<PR_ROWS>(P, tile);
        const CodecSideK& S = P.side[id.side];
        const int tok = id.t0 + r;
        float p[G::L];
        if (tok < P.n_tokens) {
            const long long vrow = packed_row(P, id, tok);
            const uint8_t* srow = S.scales + vrow * (D / P.group) * S.sbytes;
            if (BK == BV || id.side == 0)
                pair_dequant_load<D, BK, SF>(S.codes + vrow * (D * BK / 8), srow, P.group, t, p);
            else
                pair_dequant_load<D, BV, SF>(S.codes + vrow * (D * BV / 8), srow, P.group, t, p);
            if (S.lambda != nullptr) {
                const float2* lr = reinterpret_cast<const float2*>(S.lambda + (long long)id.o * S.lambda_outer_stride +
                                                                   (long long)id.h * D + 2 * t);
#pragma unroll
                for (int m = 0; m < G::H; ++m) {
                    const float2 l = __ldg(lr + 2 * m);
                    p[2 * m] *= __frcp_rn(l.x);
                    p[2 * m + 1] *= __frcp_rn(l.y);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < G::L; ++i) p[i] = 0.f;
        }
        float zr[G::H], zi[G::H];
        if constexpr (SRHT)
            pair_srht_inverse(p, zr, zi);
        else
            pair_srft_inverse<D>(p, t, zr, zi);
        // the previous tile's store, issued a whole tile of work ago, must have read the staging buffer
        if (lane == 0) ptx::bulk_wait_read<0>();
        __syncwarp();
        pair_store_half<D, SRHT>(P, buf + r * G::ROW, t, zr, zi);
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

template <int D, bool QUANTIZE, int BK, int BV, int SF, bool SRHT>
int launch_pair(const CodecCall& c) {
    using G = PairGeo<D>;
    if ((long long)c.n_sides * c.n_outer * c.H * ((c.n_tokens + PR_ROWS - 1) / PR_ROWS) > 0x7fffffffll) {
        set_error("sizes too large for 32-bit tile indexing at d = %d", D);
        return SRFTKV_ERR_INVALID;
    }
    CodecParams P;
    fill_params(c, P);
    set_tile_grid(c, P, PR_ROWS);
    if (P.total_tiles == 0) return 0;
    CUtensorMap tm[2];
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        if (!encode_x_map(&tm[s], d.x, D, c.H, c.n_tokens, c.n_outer, PR_ROWS, false)) return SRFTKV_ERR_CUDA;
    }
    P.fault = codec_fault_word();
    if (!P.fault) return SRFTKV_ERR_CUDA;
    auto kern = [] {
        if constexpr (QUANTIZE)
            return srft_quantize_pair_kernel<D, BK, BV, SF, SRHT>;
        else
            return srft_dequantize_pair_kernel<D, BK, BV, SF, SRHT>;
    }();
    const int smem_bytes = QUANTIZE ? G::SMEM : G::SMEM_DQ;
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

template <int D, bool Q, int BK, int BV>
int launch_pair_bits(const CodecCall& c) {
    // both sides of one launch share the transform and the scale format; the Hadamard transform is d = 256 only
    const bool srht = c.side[0].transform == SRFTKV_TRANSFORM_SRHT;
    if constexpr (D == 256) {
        switch (c.side[0].scale_format) {
            case SRFTKV_SCALE_FP32:
                return srht ? launch_pair<D, Q, BK, BV, SRFTKV_SCALE_FP32, true>(c)
                            : launch_pair<D, Q, BK, BV, SRFTKV_SCALE_FP32, false>(c);
            case SRFTKV_SCALE_FP16:
                return srht ? launch_pair<D, Q, BK, BV, SRFTKV_SCALE_FP16, true>(c)
                            : launch_pair<D, Q, BK, BV, SRFTKV_SCALE_FP16, false>(c);
            default:
                return srht ? launch_pair<D, Q, BK, BV, SRFTKV_SCALE_E8M0, true>(c)
                            : launch_pair<D, Q, BK, BV, SRFTKV_SCALE_E8M0, false>(c);
        }
    } else {
        if (srht) {
            set_error("the Hadamard transform needs a power-of-two d");
            return SRFTKV_ERR_INVALID;
        }
        switch (c.side[0].scale_format) {
            case SRFTKV_SCALE_FP32: return launch_pair<D, Q, BK, BV, SRFTKV_SCALE_FP32, false>(c);
            case SRFTKV_SCALE_FP16: return launch_pair<D, Q, BK, BV, SRFTKV_SCALE_FP16, false>(c);
            default: return launch_pair<D, Q, BK, BV, SRFTKV_SCALE_E8M0, false>(c);
        }
    }
}

template <int D, bool Q>
int launch_pair_all(const CodecCall& c) {
    if (c.n_sides == 2 && (c.side[0].transform != c.side[1].transform ||
                           c.side[0].scale_format != c.side[1].scale_format)) {
        set_error("d = %d launch with sides of different transforms or scale formats", D);
        return SRFTKV_ERR_INVALID;
    }
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    if (bk == 4 && bv == 4) return launch_pair_bits<D, Q, 4, 4>(c);
    if (bk == 8 && bv == 8) return launch_pair_bits<D, Q, 8, 8>(c);
    if (bk == 8 && bv == 4) return launch_pair_bits<D, Q, 8, 4>(c);
    return launch_pair_bits<D, Q, 4, 8>(c);
}

}  // namespace

// dequantize entries, each in a translation unit of its own (codec_d192_dq.cu, codec_d256_dq.cu)
int pair_dequantize_d192(const CodecCall& c);
int pair_dequantize_d256(const CodecCall& c);

}  // namespace srftkv
