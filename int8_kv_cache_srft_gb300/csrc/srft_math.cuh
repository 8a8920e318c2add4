// srft_math.cuh -- register-resident SRFT arithmetic shared by the codec and
// attention kernels.
//
// Method: "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
// Apple Silicon", Methodology 1 (SRFT(x) = pack(F diag(s) x)) and 2 (sign
// multiply, log2(d/2) radix-2 Stockham stages on the d/2-point complex
// sequence z_n = u_{2n} + i u_{2n+1}, Hermitian packing, lambda, group
// absmax, rounding, nibble packing).
//
// Everything here is __host__ __device__ so the same arithmetic can be
// compiled for the host; every array index is a compile-time constant after
// unrolling, so the data stays in registers and the twiddles become
// constant-bank operands of the FMAs.
#pragma once

#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#define SRFT_HD __host__ __device__ __forceinline__
#else
#define SRFT_HD inline
#endif

namespace srftkv {

// ---------------------------------------------------------------------------
// Twiddle factors, computed at compile time
// ---------------------------------------------------------------------------
namespace trig {
constexpr double kPi = 3.14159265358979323846264338327950288;
constexpr double kSqrt2 = 1.41421356237309504880168872420969808;

// Taylor series; only called with |x| <= pi/4 where 14 terms are far below
// double rounding.
constexpr double taylor_sin(double x) {
    double t = x, s = x;
    for (int i = 1; i < 14; ++i) {
        t *= -x * x / ((2.0 * i) * (2.0 * i + 1.0));
        s += t;
    }
    return s;
}
constexpr double taylor_cos(double x) {
    double t = 1.0, s = 1.0;
    for (int i = 1; i < 14; ++i) {
        t *= -x * x / ((2.0 * i - 1.0) * (2.0 * i));
        s += t;
    }
    return s;
}
// cos and sin of 2 pi k / n: reduce to a quadrant exactly in integers, then
// to [0, pi/4] by the complementary-angle identity.
constexpr void cos_sin_2pi(long k, long n, double& c, double& s) {
    k %= n;
    if (k < 0) k += n;
    const long q = (4 * k) / n;
    const long a = 4 * k - q * n;  // angle within the quadrant = (pi/2) a / n
    double ca = 0, sa = 0;
    if (2 * a <= n) {
        const double x = (kPi / 2) * double(a) / double(n);
        ca = taylor_cos(x);
        sa = taylor_sin(x);
    } else {
        const double x = (kPi / 2) * double(n - a) / double(n);
        ca = taylor_sin(x);
        sa = taylor_cos(x);
    }
    switch (q) {
        case 0: c = ca; s = sa; break;
        case 1: c = -sa; s = ca; break;
        case 2: c = -ca; s = -sa; break;
        default: c = sa; s = -ca; break;
    }
}
constexpr double inv_sqrt_pow2(int d) {  // 1/sqrt(d) for d a power of two
    double r = 1.0;
    int m = 0;
    while ((1 << m) < d) ++m;
    for (int i = 0; i < m / 2; ++i) r *= 0.5;
    if (m & 1) r *= 0.5 * kSqrt2;
    return r;
}
}  // namespace trig

// W_256^m = exp(-2 pi i m / 256) for m = 0..255: every FFT twiddle of a
// power-of-two length <= 256 is one of these.
struct TwiddleTable {
    float re[256];
    float im[256];
};
// Split-step twiddles pre-multiplied by h_D = 1/sqrt(2 d): for d = 16..256,
// entries k = 1..d/4-1 of h_D * W_d^k live at offset split_offset(d) + k.
struct SplitTable {
    float re[128];
    float im[128];
};
SRFT_HD constexpr int split_offset(int d) { return d / 4 - 4; }

constexpr TwiddleTable make_twiddles() {
    TwiddleTable t{};
    for (int m = 0; m < 256; ++m) {
        double c = 0, s = 0;
        trig::cos_sin_2pi(m, 256, c, s);
        t.re[m] = float(c);
        t.im[m] = float(-s);
    }
    return t;
}
constexpr SplitTable make_split_twiddles() {
    SplitTable t{};
    for (int d = 16; d <= 256; d *= 2) {
        const double h = trig::inv_sqrt_pow2(d) / trig::kSqrt2;
        for (int k = 0; k < d / 4; ++k) {
            double c = 0, s = 0;
            trig::cos_sin_2pi(k, d, c, s);
            t.re[split_offset(d) + k] = float(h * c);
            t.im[split_offset(d) + k] = float(-h * s);
        }
    }
    return t;
}

#if defined(__CUDACC__)
static __constant__ TwiddleTable c_tw = make_twiddles();
static __constant__ SplitTable c_split = make_split_twiddles();
// The same table in global memory, for indices that differ between the lanes
// of a warp: the constant bank serialises those, L1 serves them in a few lines.
static __device__ const TwiddleTable g_tw = make_twiddles();
__device__ __forceinline__ float tw_re_lane(int m) { return __ldg(&g_tw.re[m]); }
__device__ __forceinline__ float tw_im_lane(int m) { return __ldg(&g_tw.im[m]); }
#endif
static constexpr TwiddleTable h_tw = make_twiddles();
static constexpr SplitTable h_split = make_split_twiddles();

SRFT_HD float tw_re(int m) {
#if defined(__CUDA_ARCH__)
    return c_tw.re[m];
#else
    return h_tw.re[m];
#endif
}
SRFT_HD float tw_im(int m) {
#if defined(__CUDA_ARCH__)
    return c_tw.im[m];
#else
    return h_tw.im[m];
#endif
}
SRFT_HD float sp_re(int m) {
#if defined(__CUDA_ARCH__)
    return c_split.re[m];
#else
    return h_split.re[m];
#endif
}
SRFT_HD float sp_im(int m) {
#if defined(__CUDA_ARCH__)
    return c_split.im[m];
#else
    return h_split.im[m];
#endif
}

SRFT_HD float fmaf_(float a, float b, float c) {
#if defined(__CUDA_ARCH__)
    return __fmaf_rn(a, b, c);
#else
    return __builtin_fmaf(a, b, c);
#endif
}

// ---------------------------------------------------------------------------
// Radix-2 Stockham FFT (decimation in time), unnormalised
// ---------------------------------------------------------------------------
// Stage L merges pairs of length-L transforms into length-2L transforms.
// With R = N/(2L), A holds element [k][j] at k*2R + j (k < L: bin, j < 2R:
// residue class of the input index mod 2R) and B holds [k][j] at k*R + j:
//   B[k][j]   = A[k][j] + w A[k][j+R],   B[k+L][j] = A[k][j] - w A[k][j+R],
// w = W_{2L}^k (conjugated for the inverse).  The final stage leaves bin k
// at index k: the sort is automatic, as in Stockham's formulation.
template <int N, int L, bool INV>
SRFT_HD void stockham_stage(const float (&ar)[N], const float (&ai)[N], float (&br)[N], float (&bi)[N]) {
    constexpr int R = N / (2 * L);
    constexpr int TSTEP = 256 / (2 * L);
#pragma unroll
    for (int k = 0; k < L; ++k) {
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int ia = k * 2 * R + j, ib = ia + R;
            const int o0 = k * R + j, o1 = (k + L) * R + j;
            const float are = ar[ia], aim = ai[ia], bre = ar[ib], bim = ai[ib];
            if (k == 0) {
                br[o0] = are + bre;
                bi[o0] = aim + bim;
                br[o1] = are - bre;
                bi[o1] = aim - bim;
            } else if (2 * k == L) {  // w = -i (forward), +i (inverse)
                if (!INV) {
                    br[o0] = are + bim;
                    bi[o0] = aim - bre;
                    br[o1] = are - bim;
                    bi[o1] = aim + bre;
                } else {
                    br[o0] = are - bim;
                    bi[o0] = aim + bre;
                    br[o1] = are + bim;
                    bi[o1] = aim - bre;
                }
            } else {
                const float wr = tw_re(k * TSTEP);
                const float wi = INV ? -tw_im(k * TSTEP) : tw_im(k * TSTEP);
                // a + w b with two FMAs per component; a - w b = 2a - (a + w b)
                const float yr = fmaf_(wr, bre, fmaf_(-wi, bim, are));
                const float yi = fmaf_(wr, bim, fmaf_(wi, bre, aim));
                br[o0] = yr;
                bi[o0] = yi;
                br[o1] = fmaf_(2.f, are, -yr);
                bi[o1] = fmaf_(2.f, aim, -yi);
            }
        }
    }
}

template <int N, int L, bool INV>
SRFT_HD void fft_from(float (&re)[N], float (&im)[N]) {
    if constexpr (L < N) {
        float br[N], bi[N];
        stockham_stage<N, L, INV>(re, im, br, bi);
        fft_from<N, 2 * L, INV>(br, bi);
#pragma unroll
        for (int i = 0; i < N; ++i) {
            re[i] = br[i];
            im[i] = bi[i];
        }
    }
}

// In place: Z_k = sum_n z_n exp(-+2 pi i nk/N) (no normalisation).
template <int N, bool INV>
SRFT_HD void fft(float (&re)[N], float (&im)[N]) {
    fft_from<N, 1, INV>(re, im);
}

// ---------------------------------------------------------------------------
// Real-signal split: N-point complex transform of z_n = u_{2n} + i u_{2n+1}
// <-> packed coordinates p of the unitary d-point real DFT (d = 2N).
// Packing: p0 = y_0, p1 = y_N, p_{2k} = sqrt2 Re y_k, p_{2k+1} = sqrt2 Im y_k.
// ---------------------------------------------------------------------------
// Forward, one conjugate pair (k, m = N-k): from Z_k, Z_m to p_{2k..2k+1},
// p_{2m..2m+1}.  With E = (Z_k + conj Z_m)/2, O = (Z_k - conj Z_m)/(2i),
// U_k = E + W_d^k O and U_m = conj(E - W_d^k O); p = sqrt(2/d) U.
// a1 + i a2 = h W_d^k with h = 1/sqrt(2d) (table), so every output is one FMA.
SRFT_HD void split_pair_fwd(float zkr, float zki, float zmr, float zmi, float a1, float a2, float h,
                            float& pk0, float& pk1, float& pm0, float& pm1) {
    const float s1 = zkr + zmr, s2 = zki - zmi, d1 = zkr - zmr, d2 = zki + zmi;
    const float tr = fmaf_(a1, d2, a2 * d1);
    const float ti = fmaf_(a2, d2, -(a1 * d1));
    pk0 = fmaf_(h, s1, tr);
    pk1 = fmaf_(h, s2, ti);
    pm0 = fmaf_(h, s1, -tr);
    pm1 = fmaf_(-h, s2, ti);
}

// Walsh-Hadamard transform, unnormalised, Sylvester natural order
// (H_ij = (-1)^popcount(i & j)): in-place butterflies over strides 1..N/2.
template <int N>
SRFT_HD void wht(float (&a)[N]) {
#pragma unroll
    for (int h = 1; h < N; h <<= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            if (i & h) continue;
            const float x = a[i], y = a[i + h];
            a[i] = x + y;
            a[i + h] = x - y;
        }
    }
}
// The same transform of the length-2N vector u with u_{2n} = re[n],
// u_{2n+1} = im[n].  H_{2N} = H_N (x) H_2 with the H_2 factor on the low
// index bit: one butterfly per pair, then a length-N transform of each half.
// Its own inverse up to the factor 2N.
template <int N>
SRFT_HD void wht_pairs(float (&re)[N], float (&im)[N]) {
#pragma unroll
    for (int n = 0; n < N; ++n) {
        const float x = re[n], y = im[n];
        re[n] = x + y;
        im[n] = x - y;
    }
    wht<N>(re);
    wht<N>(im);
}

// Inverse of split_pair_fwd, including the 1/N of the inverse transform:
// from packed (p_{2k}, p_{2k+1}), (p_{2m}, p_{2m+1}) to Z'_k, Z'_m such that
// the unnormalised inverse N-point transform of Z' gives z_n = u_{2n} + i u_{2n+1}.
SRFT_HD void split_pair_inv(float pk0, float pk1, float pm0, float pm1, float a1, float a2, float h,
                            float& zkr, float& zki, float& zmr, float& zmi) {
    const float s1 = pk0 + pm0, s2 = pk1 - pm1, d1 = pk0 - pm0, d2 = pk1 + pm1;
    const float vr = fmaf_(a2, d1, -(a1 * d2));
    const float vi = fmaf_(a2, d2, a1 * d1);
    zkr = fmaf_(h, s1, vr);
    zki = fmaf_(h, s2, vi);
    zmr = fmaf_(h, s1, -vr);
    zmi = fmaf_(-h, s2, vi);
}

template <int D>
struct SplitConst {
    static constexpr int N = D / 2;
    static constexpr float inv_sqrt_d = float(trig::inv_sqrt_pow2(D));
    static constexpr float c = float(trig::kSqrt2 * trig::inv_sqrt_pow2(D));   // sqrt(2/d)
    static constexpr float h = float(trig::inv_sqrt_pow2(D) / trig::kSqrt2);   // 1/sqrt(2d)
};

// Full forward split for one thread holding all N bins.
template <int D>
SRFT_HD void split_forward(const float (&zr)[D / 2], const float (&zi)[D / 2], float (&p)[D]) {
    using C = SplitConst<D>;
    constexpr int N = C::N;
    p[0] = (zr[0] + zi[0]) * C::inv_sqrt_d;
    p[1] = (zr[0] - zi[0]) * C::inv_sqrt_d;
    p[N] = C::c * zr[N / 2];
    p[N + 1] = -C::c * zi[N / 2];
#pragma unroll
    for (int k = 1; k < N / 2; ++k) {
        const int m = N - k;
        split_pair_fwd(zr[k], zi[k], zr[m], zi[m], sp_re(split_offset(D) + k), sp_im(split_offset(D) + k), C::h,
                       p[2 * k], p[2 * k + 1], p[2 * m], p[2 * m + 1]);
    }
}

// Full inverse split for one thread holding all d packed coordinates.
template <int D>
SRFT_HD void split_inverse(const float (&p)[D], float (&zr)[D / 2], float (&zi)[D / 2]) {
    using C = SplitConst<D>;
    constexpr int N = C::N;
    zr[0] = (p[0] + p[1]) * C::inv_sqrt_d;
    zi[0] = (p[0] - p[1]) * C::inv_sqrt_d;
    zr[N / 2] = C::c * p[N];
    zi[N / 2] = -C::c * p[N + 1];
#pragma unroll
    for (int k = 1; k < N / 2; ++k) {
        const int m = N - k;
        split_pair_inv(p[2 * k], p[2 * k + 1], p[2 * m], p[2 * m + 1], sp_re(split_offset(D) + k),
                       sp_im(split_offset(D) + k), C::h, zr[k], zi[k], zr[m], zi[m]);
    }
}

// ---------------------------------------------------------------------------
// Bit helpers
// ---------------------------------------------------------------------------
SRFT_HD uint32_t f2u(float f) {
#if defined(__CUDA_ARCH__)
    return __float_as_uint(f);
#else
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
#endif
}
SRFT_HD float u2f(uint32_t u) {
#if defined(__CUDA_ARCH__)
    return __uint_as_float(u);
#else
    float f;
    std::memcpy(&f, &u, 4);
    return f;
#endif
}
// Byte permute: byte i of the result is byte (s >> 4i) & 7 of {hi:lo}.
SRFT_HD uint32_t prmt(uint32_t lo, uint32_t hi, uint32_t s) {
#if defined(__CUDA_ARCH__)
    return __byte_perm(lo, hi, s);
#else
    const uint64_t v = (uint64_t(hi) << 32) | lo;
    uint32_t r = 0;
    for (int i = 0; i < 4; ++i) r |= uint32_t((v >> (8 * ((s >> (4 * i)) & 7))) & 0xFF) << (8 * i);
    return r;
#endif
}
SRFT_HD float fdiv_rn(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fdiv_rn(a, b);
#else
    return a / b;
#endif
}
// |a|: on the device the hardware absolute value (an operand modifier, free);
// the host form is for host-side builds of the same helpers
SRFT_HD float fabs_(float a) {
#if defined(__CUDA_ARCH__)
    return fabsf(a);
#else
    return a < 0.f ? -a : a;
#endif
}
SRFT_HD float fmax_(float a, float b) {
#if defined(__CUDA_ARCH__)
    return fmaxf(a, b);
#else
    return a > b ? a : b;
#endif
}

// fp16 bits <-> float (exact, no rounding involved in the widening)
SRFT_HD float half_bits_to_float(uint32_t h) {
#if defined(__CUDA_ARCH__)
    return __half2float(__ushort_as_half((unsigned short)h));
#else
    const uint32_t sign = (h & 0x8000u) << 16, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    if (e == 0) {
        const float v = float(m) * (1.0f / 16777216.0f);  // m * 2^-24
        return sign ? -v : v;
    }
    if (e == 31) return u2f(sign | 0x7F800000u | (m << 13));
    return u2f(sign | ((e + 112) << 23) | (m << 13));
#endif
}

// ---------------------------------------------------------------------------
// Rounding and packing.  Adding 1.5*2^23 + off to r (|r| <= 2^21) leaves
// rint(r) + off in the low mantissa bits, rounded half-to-even by the FMA's
// single rounding of z*inv + magic.
// ---------------------------------------------------------------------------
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

// int4: offset-binary nibbles (q + 8) from the magic bits, two per byte, eight
// per word, then flipped to two's complement (x ^ 8 per nibble).
SRFT_HD uint32_t pack8_int4(const float* r_magic_bits_as_float) {
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = f2u(r_magic_bits_as_float[i]);
    const uint32_t p0 = b[0] + (b[1] << 4), p1 = b[2] + (b[3] << 4);
    const uint32_t p2 = b[4] + (b[5] << 4), p3 = b[6] + (b[7] << 4);
    const uint32_t q01 = p0 + (p1 << 8), q23 = p2 + (p3 << 8);
    return prmt(q01, q23, 0x5410) ^ 0x88888888u;
}
// int8: offset-binary bytes (q + 128), four per word, flipped to two's complement.
SRFT_HD uint32_t pack4_int8(const float* r_magic_bits_as_float) {
    const uint32_t b0 = f2u(r_magic_bits_as_float[0]), b1 = f2u(r_magic_bits_as_float[1]);
    const uint32_t b2 = f2u(r_magic_bits_as_float[2]), b3 = f2u(r_magic_bits_as_float[3]);
    return prmt(b0 + (b1 << 8), b2 + (b3 << 8), 0x5410) ^ 0x80808080u;
}

// Signed code of element i of a packed word, as a float (exact).
SRFT_HD float code_int4(uint32_t w, int i) {
    return u2f(0x4B400000u | (((w >> (4 * i)) & 0xFu) ^ 0x8u)) - (kMagic + 8.0f);
}
SRFT_HD float code_int8(uint32_t w, int i) {
    return u2f(0x4B400000u | (((w >> (8 * i)) & 0xFFu) ^ 0x80u)) - (kMagic + 128.0f);
}

}  // namespace srftkv
