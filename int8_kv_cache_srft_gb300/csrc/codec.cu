// codec.cu -- host dispatch of the fused SRFT quantize / dequantize kernels
// (codec_impl.cuh, instantiated per head dimension in codec_d*.cu), the bare
// transform kernel used for testing, and the device fault word.
//
// Method: "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
// Apple Silicon", Methodology 1 (SRFT) and 2 (the fused kernel's steps).
#include <cuda_fp16.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "srft_math.cuh"

namespace srftkv {

static __device__ unsigned int g_codec_fault;

template <int D>
int launch_codec_d(const CodecCall& c, bool quantize);
extern template int launch_codec_d<16>(const CodecCall&, bool);
extern template int launch_codec_d<32>(const CodecCall&, bool);
extern template int launch_codec_d<64>(const CodecCall&, bool);
extern template int launch_codec_d<128>(const CodecCall&, bool);

// fp16 pair (x_{2n}, x_{2n+1}) with the SRFT signs applied -> complex z_n
__device__ __forceinline__ void signed_pair_t(uint32_t w, uint32_t mask, float& re, float& im) {
    const uint32_t s = w ^ mask;
    re = __half2float(__ushort_as_half((unsigned short)(s & 0xFFFFu)));
    im = __half2float(__ushort_as_half((unsigned short)(s >> 16)));
}

// ---------------------------------------------------------------------------
// K5: the bare transform (fp16 in, fp32 out), one thread per row
// ---------------------------------------------------------------------------
struct SignParams {
    uint32_t w[128];
};

template <int D, bool INV>
__global__ void __launch_bounds__(128) srft_transform_kernel(const uint16_t* __restrict__ x, float* __restrict__ y, int n,
                                                             const __grid_constant__ SignParams S, int srht) {
    constexpr int N = D / 2;
    constexpr float isd = SplitConst<D>::inv_sqrt_d;
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n) return;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (long long)r * D);
    float4* yr = reinterpret_cast<float4*>(y + (long long)r * D);
    float zr[N], zi[N];
    if (srht) {  // y = d^-1/2 H diag(s) x, or its inverse diag(s) H x / sqrt(d)
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 v = __ldg(xr + c);
            const uint32_t m0 = INV ? 0u : S.w[4 * c + 0], m1 = INV ? 0u : S.w[4 * c + 1];
            const uint32_t m2 = INV ? 0u : S.w[4 * c + 2], m3 = INV ? 0u : S.w[4 * c + 3];
            signed_pair_t(v.x, m0, zr[4 * c + 0], zi[4 * c + 0]);
            signed_pair_t(v.y, m1, zr[4 * c + 1], zi[4 * c + 1]);
            signed_pair_t(v.z, m2, zr[4 * c + 2], zi[4 * c + 2]);
            signed_pair_t(v.w, m3, zr[4 * c + 3], zi[4 * c + 3]);
        }
        wht_pairs<N>(zr, zi);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) {
            const int n0 = 2 * c, n1 = 2 * c + 1;
            float a = zr[n0] * isd, b = zi[n0] * isd, cc = zr[n1] * isd, dd = zi[n1] * isd;
            if (INV) {
                a = u2f(f2u(a) ^ ((S.w[n0] & 0x8000u) << 16));
                b = u2f(f2u(b) ^ (S.w[n0] & 0x80000000u));
                cc = u2f(f2u(cc) ^ ((S.w[n1] & 0x8000u) << 16));
                dd = u2f(f2u(dd) ^ (S.w[n1] & 0x80000000u));
            }
            yr[c] = make_float4(a, b, cc, dd);
        }
        return;
    }
    if constexpr (!INV) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 v = __ldg(xr + c);
            signed_pair_t(v.x, S.w[4 * c + 0], zr[4 * c + 0], zi[4 * c + 0]);
            signed_pair_t(v.y, S.w[4 * c + 1], zr[4 * c + 1], zi[4 * c + 1]);
            signed_pair_t(v.z, S.w[4 * c + 2], zr[4 * c + 2], zi[4 * c + 2]);
            signed_pair_t(v.w, S.w[4 * c + 3], zr[4 * c + 3], zi[4 * c + 3]);
        }
        fft<N, false>(zr, zi);
        float p[D];
        split_forward<D>(zr, zi, p);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) yr[c] = make_float4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
    } else {
        float p[D];
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 v = __ldg(xr + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                p[8 * c + 2 * e] = f.x;
                p[8 * c + 2 * e + 1] = f.y;
            }
        }
        split_inverse<D>(p, zr, zi);
        fft<N, true>(zr, zi);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) {
            const int n0 = 2 * c, n1 = 2 * c + 1;
            const float a = u2f(f2u(zr[n0]) ^ ((S.w[n0] & 0x8000u) << 16));
            const float b = u2f(f2u(zi[n0]) ^ (S.w[n0] & 0x80000000u));
            const float cc = u2f(f2u(zr[n1]) ^ ((S.w[n1] & 0x8000u) << 16));
            const float dd = u2f(f2u(zi[n1]) ^ (S.w[n1] & 0x80000000u));
            yr[c] = make_float4(a, b, cc, dd);
        }
    }
}

static int dispatch_codec(const CodecCall& c, bool quantize) {
    switch (c.d) {
        case 16: return launch_codec_d<16>(c, quantize);
        case 32: return launch_codec_d<32>(c, quantize);
        case 64: return launch_codec_d<64>(c, quantize);
        case 128: return launch_codec_d<128>(c, quantize);
        case 192: return launch_codec_d192(c, quantize);
        case 256: return launch_codec_d256(c, quantize);
        default: set_error("unsupported d = %d", c.d); return -1;
    }
}

// Codec path: the tensor-core contraction (codec_tc.cu) for d = 128 when the
// call is large enough to amortise building R_s in every CTA (measured on
// GB300: from about 150 K vectors a call for the quantize and 65 K for the
// dequantize it beats the register FFT, and is 1.5-1.8x faster at millions); to quantize a small d = 128
// call (a token append), one warp per vector (codec_small.cu), faster than
// one thread per vector up to about 4 K vectors; the register FFT otherwise.
// SRFTKV_QUANT_PATH=fft, =tc or =warp in the environment forces one path (tc
// and warp only where they apply).
static int quant_path_override() {
    const char* e = getenv("SRFTKV_QUANT_PATH");
    if (!e) return 0;
    return !strcmp(e, "fft") ? 1 : !strcmp(e, "tc") ? 2 : !strcmp(e, "warp") ? 3 : 0;
}
constexpr long long kWarpPathMaxRows = 4096;
// d = 128: the tensor-core kernels' fixed cost (about 13 us a launch, some 4 us
// of it the R_s block every CTA builds) against the register FFT: measured crossovers
// about 150 K vectors for the quantize (0.21 M: 0.027 against 0.029 ms) and 65 K
// for the dequantize (0.11 M: 0.019 against 0.021 ms)
constexpr long long kTensorCoreQuantMinRows = 5ll << 15;
constexpr long long kTensorCoreDequantMinRows = 1ll << 16;
// d = 192 / 256: the tensor-core kernels pay a fixed cost (every CTA builds
// its N x d block of R_s: about 20 us a launch at d = 256, 16-19 at d = 192)
// that the two-lane register kernels do not.  Measured crossovers (vectors of
// K and V together, L2 flushed): dequantize about 65 K at d = 256 and 32 K at
// d = 192, quantize about 106 K at both (the Gemma-shaped 0.21 M vectors of
// d = 256: quantize 0.064 against 0.068 ms, dequantize 0.048 against 0.077).
constexpr long long kWideTensorCoreQuantMinRows = 1ll << 17;
constexpr long long kWideTensorCoreDequantMinRows = 1ll << 16;

// A call whose two sides use different transforms or scale formats runs as
// two one-sided calls (the tensor-core kernels hold one transform matrix per
// CTA and are compiled per scale format).
static bool split_mixed(const CodecCall& c, int (*fn)(const CodecCall&), int& rc) {
    if (c.n_sides != 2 ||
        (c.side[0].transform == c.side[1].transform && c.side[0].scale_format == c.side[1].scale_format))
        return false;
    CodecCall one = c;
    one.n_sides = 1;
    rc = fn(one);
    if (rc) return true;
    one.side[0] = c.side[1];
    rc = fn(one);
    return true;
}

// d = 80 and 96 run only as the tensor-core contraction padded to 128 (the
// register FFT is built for powers of two)
static int tc_only(const CodecCall& c, int (*fn)(const CodecCall&), const char* what) {
    const int rc = fn(c);
    if (rc == 1) {
        set_error("%s at d = %d needs groups of 16 or 32 and, for dequantize, t_cap and t_offset such that "
                  "t_cap * (d / group) * scale bytes and t_offset * (d / group) * scale bytes (at d = 80 also "
                  "t_cap and t_offset * d * bits / 8) are multiples of 16",
                  what, c.d);
        return SRFTKV_ERR_INVALID;
    }
    return rc;
}

int codec_quantize(const CodecCall& c) {
    int split_rc = 0;
    if (split_mixed(c, codec_quantize, split_rc)) return split_rc;
    if (c.d == 96 || c.d == 80) return tc_only(c, codec_quantize_tc, "quantize");
    const int ov = quant_path_override();
    const long long rows = (long long)c.n_sides * c.n_outer * c.n_tokens * c.H;
    if ((c.d == 192 || c.d == 256) && c.group <= 32 &&  // a group must fit in one epilogue thread's 32 columns
        (ov == 2 || (ov == 0 && rows >= kWideTensorCoreQuantMinRows)))
        return c.d == 192 ? codec_quantize_tc_wide192(c) : codec_quantize_tc_wide256(c);
    if (ov == 2 || (ov == 0 && rows >= kTensorCoreQuantMinRows)) {
        const int rc = codec_quantize_tc(c);
        if (rc != 1) return rc;
    }
    if (ov == 3 || (ov == 0 && rows <= kWarpPathMaxRows)) {
        const int rc = codec_quantize_warp(c);
        if (rc != 1) return rc;
    }
    return dispatch_codec(c, true);
}
int codec_dequantize(const CodecCall& c) {
    int split_rc = 0;
    if (split_mixed(c, codec_dequantize, split_rc)) return split_rc;
    if (c.d == 96 || c.d == 80) return tc_only(c, codec_dequantize_tc, "dequantize");
    const int ov = quant_path_override();
    const long long rows = (long long)c.n_sides * c.n_outer * c.n_tokens * c.H;
    if ((c.d == 192 || c.d == 256) && (ov == 2 || (ov == 0 && rows >= kWideTensorCoreDequantMinRows))) {
        const int rc = c.d == 192 ? codec_dequantize_tc_wide192(c) : codec_dequantize_tc_wide256(c);
        if (rc != 1) return rc;  // 1: a call the tensor-core kernel does not take (lambda, groups > 32, scale rows)
    }
    if (ov == 2 || (ov == 0 && rows >= kTensorCoreDequantMinRows)) {
        const int rc = codec_dequantize_tc(c);
        if (rc != 1) return rc;
    }
    return dispatch_codec(c, false);
}

template <int D>
static int launch_transform(const void* x, float* y, int n, uint64_t seed, bool inverse, bool srht, cudaStream_t s) {
    SignParams S;
    for (int i = 0; i < 128; ++i) S.w[i] = 0;
    sign_masks(D, seed, S.w);
    const int blocks = (n + 127) / 128;
    if (inverse)
        srft_transform_kernel<D, true><<<blocks, 128, 0, s>>>(static_cast<const uint16_t*>(x), y, n, S, srht ? 1 : 0);
    else
        srft_transform_kernel<D, false><<<blocks, 128, 0, s>>>(static_cast<const uint16_t*>(x), y, n, S, srht ? 1 : 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("transform kernel launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return 0;
}

// ---------------------------------------------------------------------------
// The bare SRFT at a head dimension that is not a power of two (d = 80, 96, 192) as the
// dense real map p = R diag(s) x of the packed unitary DFT: R[0][k] = d^-1/2,
// R[1][k] = (-1)^k d^-1/2, and for 1 <= j < d/2 R[2j][k] = sqrt(2/d) cos(2 pi jk/d),
// R[2j+1][k] = -sqrt(2/d) sin(2 pi jk/d); the inverse is diag(s) R^T.  A block
// takes four rows at a time, one thread per output coordinate, with the
// angles from a table of cos / sin(2 pi m/d) evaluated in double.
// ---------------------------------------------------------------------------
constexpr int DT_ROWS = 4, DT_MAXD = 256;

__global__ void __launch_bounds__(128) srft_dense_transform_kernel(const __half* __restrict__ x, float* __restrict__ y,
                                                                   int n, int d, const __grid_constant__ SignParams S,
                                                                   int inverse) {
    __shared__ float cs[DT_MAXD], sn[DT_MAXD], xs[DT_ROWS][DT_MAXD];
    for (int m = threadIdx.x; m < d; m += blockDim.x) {
        double sv, cv;
        sincospi(2.0 * m / d, &sv, &cv);
        cs[m] = (float)cv;
        sn[m] = (float)sv;
    }
    const float isd = (float)(1.0 / sqrt((double)d)), r2 = (float)sqrt(2.0 / d);
    auto neg = [&](int k) { return (S.w[k >> 1] & ((k & 1) ? 0x80000000u : 0x8000u)) != 0u; };
    auto R = [&](int row, int k) {
        if (row == 0) return isd;
        if (row == 1) return (k & 1) ? -isd : isd;
        const int m = ((row >> 1) * k) % d;
        return (row & 1) ? -r2 * sn[m] : r2 * cs[m];
    };
    for (long long r0 = (long long)blockIdx.x * DT_ROWS; r0 < n; r0 += (long long)gridDim.x * DT_ROWS) {
        __syncthreads();
        for (int i = threadIdx.x; i < DT_ROWS * d; i += blockDim.x) {
            const int v = i / d, k = i % d;
            const long long r = r0 + v;
            float val = r < n ? __half2float(x[r * d + k]) : 0.f;
            if (!inverse && neg(k)) val = -val;
            xs[v][k] = val;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < DT_ROWS * d; i += blockDim.x) {
            const int v = i / d, o = i % d;
            const long long r = r0 + v;
            if (r >= n) continue;
            float acc = 0.f;
            if (!inverse) {
                for (int k = 0; k < d; ++k) acc = fmaf(R(o, k), xs[v][k], acc);
            } else {
                for (int k = 0; k < d; ++k) acc = fmaf(R(k, o), xs[v][k], acc);
                if (neg(o)) acc = -acc;
            }
            y[r * d + o] = acc;
        }
    }
}

static int launch_dense_transform(const void* x, float* y, int n, int d, uint64_t seed, bool inverse, cudaStream_t s) {
    SignParams S;
    for (int i = 0; i < 128; ++i) S.w[i] = 0;
    sign_masks(d, seed, S.w);
    long long blocks = ((long long)n + DT_ROWS - 1) / DT_ROWS;
    if (blocks > 152 * 8) blocks = 152 * 8;
    srft_dense_transform_kernel<<<(int)blocks, 128, 0, s>>>(static_cast<const __half*>(x), y, n, d, S, inverse ? 1 : 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("transform kernel launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return 0;
}

int transform_launch(const void* x, float* y, int n, int d, uint64_t seed, bool inverse, bool srht, cudaStream_t s) {
    if (n == 0) return 0;
    if ((d == 80 || d == 96 || d == 192) && !srht) return launch_dense_transform(x, y, n, d, seed, inverse, s);
    switch (d) {
        case 16: return launch_transform<16>(x, y, n, seed, inverse, srht, s);
        case 32: return launch_transform<32>(x, y, n, seed, inverse, srht, s);
        case 64: return launch_transform<64>(x, y, n, seed, inverse, srht, s);
        case 128: return launch_transform<128>(x, y, n, seed, inverse, srht, s);
        case 256: return launch_transform<256>(x, y, n, seed, inverse, srht, s);
        default: set_error("unsupported d = %d", d); return -1;
    }
}

unsigned int* codec_fault_word() {
    static SymbolCache cache;
    void* p = nullptr;
    return symbol_address(cache, &g_codec_fault, &p, "the codec fault word") == SRFTKV_OK
               ? static_cast<unsigned int*>(p)
               : nullptr;
}

unsigned int codec_take_fault() {
    unsigned int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_codec_fault, sizeof(v));
    cudaMemcpyToSymbol(g_codec_fault, &z, sizeof(z));
    return v;
}

// Polls of a register-path quantize warp's wait for its next tile; -1 = the
// default bound.  Set only by srftkv_set_codec_poll_limit_for_testing.
static std::atomic<int> g_codec_poll_limit{-1};

uint32_t codec_poll_limit() {
    const int lim = g_codec_poll_limit.load();
    return lim < 0 ? (1u << 20) : (uint32_t)lim;
}

}  // namespace srftkv

extern "C" int srftkv_set_codec_poll_limit_for_testing(int polls) {
    srftkv::g_codec_poll_limit.store(polls < 0 ? -1 : polls);
    return SRFTKV_OK;
}
