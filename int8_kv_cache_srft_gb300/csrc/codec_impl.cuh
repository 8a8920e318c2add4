// codec_impl.cuh -- the fused SRFT quantize and dequantize kernels for the
// power-of-two head dimensions up to 128, one thread per head vector; each d is
// instantiated in its own translation unit (codec_d16.cu ... codec_d128.cu).
// d = 192 and 256 use two threads per vector (codec_pair.cuh).  The helpers
// shared with the other codec kernels (group scales, packing, tiles) live here.
//
// Method: "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
// Apple Silicon", Methodology 2: one fused kernel per direction doing the
// sign multiply, the radix-2 Stockham FFT of length d/2, the Hermitian
// packing, the per-channel lambda, the per-group absmax, the rounding to
// signed int4/int8 and the nibble packing.  Methodology 3: lambda per
// coordinate combined with one scale per group of `group` coordinates.
//
// GB300 mapping: one thread owns one head vector for the whole pipeline, so
// the FFT, the group maxima and the packing never leave registers and need
// no shuffles.  Each warp streams tiles of 32 tokens of one (outer, head):
// their packed rows are contiguous in the head-major planes.  A TMA tensor copy
// brings the fp16 rows into shared memory padded by 16 bytes per row (the
// box is 8 elements wider than the tensor; the extra columns are the zero
// fill), which makes the row-per-thread 16-byte reads bank-conflict free.
// Two buffers per warp overlap the next tile's copy with this tile's math.
// The dequantize kernel runs the same pipeline backwards and writes its fp16
// rows through shared memory with a TMA store.
#pragma once
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "srft_math.cuh"

namespace srftkv {

struct CodecSideK {
    void* x;             // fp16 rows [n_outer][n_tokens][H][d] (written directly only by the wide tensor-core dequantize)
    uint8_t* codes;
    uint8_t* scales;     // element type per sfmt
    const float* lambda;
    long long lambda_outer_stride;
    int bits;
    int transform;  // SRFTKV_TRANSFORM_SRFT or SRFTKV_TRANSFORM_SRHT
    int sfmt;       // SRFTKV_SCALE_FP32 / _FP16 / _E8M0
    int sbytes;     // bytes per stored scale
};

// Division by a divisor fixed for a launch, as a multiply and a shift
// (Granlund & Montgomery, "Division by invariant integers using
// multiplication", 1994: the round-up multiplier m = floor(2^32 (2^s - d) / d)
// + 1 with s = ceil(log2 d), q = (mulhi(n, m) + n) >> s), exact for
// 0 <= n < 2^31.  The tile index decode runs in every epilogue unit and
// converter warp; a runtime integer division there is a sequence of some
// twenty instructions.
struct FastDiv {
    uint32_t mul;
    int shift;
};
static inline FastDiv make_fastdiv(uint32_t d) {  // d >= 1
    int s = 0;
    while ((1ull << s) < d) ++s;
    FastDiv f;
    f.mul = (uint32_t)(((1ull << 32) * ((1ull << s) - d)) / d + 1);
    f.shift = s;
    return f;
}
__device__ __forceinline__ uint32_t fastdiv(uint32_t n, FastDiv f) { return (__umulhi(n, f.mul) + n) >> f.shift; }

struct CodecParams {
    CodecSideK side[2];
    int n_outer, H, t_cap, t_offset, group;
    int lg_group;         // log2(group)
    int n_tokens;
    int tiles_per_head;   // ceil(n_tokens / rows per tile)
    int tiles_per_side;   // n_outer * H * tiles_per_head
    int total_tiles;      // n_sides * tiles_per_side
    FastDiv div_side, div_head, div_H;  // by tiles_per_side, tiles_per_head, H
    unsigned int* fault;  // device fault word (bit 0: a bounded wait gave up)
    uint32_t poll_limit;  // polls of a register-path warp's wait for its next tile (a test hook lowers it)
    uint32_t sign_mask[128];
};

template <int D>
struct Geo {
    static constexpr int N = D / 2;
    static constexpr int ROWS = 32;                                       // rows per warp tile
    static constexpr int PAD = 8;                                         // fp16 elements of row padding
    static constexpr int ROW_H = D + PAD;                                 // elements per smem row
    static constexpr int BUF_BYTES = ROWS * ROW_H * 2;
    static constexpr int WARPS = 4;
    static constexpr int SMEM = 128 + WARPS * 2 * BUF_BYTES;
    static constexpr int MIN_BLOCKS = 3;
    static_assert(D <= 128, "one thread per vector covers d <= 128");
    // element offset of 16-byte chunk c inside a padded smem row
    static __device__ __forceinline__ int chunk_off(int c) { return c * 8; }
};

// A tile is a block of ROWS consecutive tokens of one (side, outer, head): its
// fp16 rows are strided by H*d in x, its packed rows are contiguous in the
// head-major planes.
struct TileId {
    int side, o, h, t0;
};
template <int ROWS>
__device__ __forceinline__ TileId decode_tile(const CodecParams& P, int t) {
    TileId id;
    id.side = (int)fastdiv((uint32_t)t, P.div_side);
    const int rem = t - id.side * P.tiles_per_side;
    const int oh = (int)fastdiv((uint32_t)rem, P.div_head);
    id.t0 = (rem - oh * P.tiles_per_head) * ROWS;
    id.o = (int)fastdiv((uint32_t)oh, P.div_H);
    id.h = oh - id.o * P.H;
    return id;
}
// packed row of token t of a tile: [outer][head][t_cap]
__device__ __forceinline__ long long packed_row(const CodecParams& P, const TileId& id, int t) {
    return ((long long)id.o * P.H + id.h) * P.t_cap + P.t_offset + t;
}

// ---------------------------------------------------------------------------
// Quantise one row z (rotated, lambda applied) and store codes and scales.
// The group maxima are built from 16-coordinate units, widened to the
// runtime group size by a butterfly over units, so one code path serves
// every group size; group == 16 (the default) keeps 16-byte scale stores.
// ---------------------------------------------------------------------------
// The stored scale of a group with absmax A, in the side's format, the value
// its codes are rounded against (sc), its stored bits (raw: fp16 bits or the
// e8m0 byte) and the multiplier inv that turns z into z / sc.
template <int BITS, int SF>
__device__ __forceinline__ void group_scale(float A, float& sc, uint32_t& raw, float& inv) {
    constexpr float Q = (BITS == 4) ? 7.f : 127.f;
    if constexpr (SF == SRFTKV_SCALE_FP32) {
        // scale = A/Q to within an ulp; z * (Q * rcp(A)) rounds z/scale to within a few ulp, far inside the
        // 1e-4 band around rounding boundaries
        sc = A * (1.0f / Q);
        raw = 0;
        inv = A > 0.f ? Q * __frcp_rn(A) : 0.f;
    } else if constexpr (SF == SRFTKV_SCALE_FP16) {
        // A * (1/Q) (within an ulp of A/Q) rounded to fp16, saturating at the largest finite fp16; it can
        // differ from rounding A/Q itself only within ~2^-23 of an fp16 midpoint
        const __half h = __float2half_rn(fminf(A * (1.0f / Q), 65504.f));
        sc = __half2float(h);
        raw = __half_as_ushort(h);
        inv = sc > 0.f ? __frcp_rn(sc) : 0.f;
    } else {
        // e8m0: biased exponent of the smallest power of two not below A/Q (normal or subnormal v); A * (1/Q)
        // is within an ulp of A/Q, which matters only within ~2^-23 of a power of two
        const float v = A * (1.0f / Q);
        const uint32_t b = __float_as_uint(v);
        uint32_t e = (b >> 23) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u);
        e = v > 0.f ? min(max(e, 1u), 254u) : 0u;
        raw = e;
        sc = __uint_as_float(e << 23);
        inv = e ? __frcp_rn(sc) : 0.f;
    }
}

// ZLOG2: z holds the coordinates times 2^ZLOG2 (a contraction whose operand
// was scaled by a power of two); the scales stored are those of the true
// coordinates, the codes are unchanged.  NARROW: the code row is only 8-byte
// aligned and the scale row only aligned to one scale (rows of d = 80: 40
// bytes of int4 codes, 5 scales), so codes go out as 8-byte stores and scales
// one at a time.
template <int D, int BITS, int SF, int ZLOG2 = 0, bool NARROW = false>
__device__ __forceinline__ void quant_store_row(float (&z)[D], int group, uint8_t* __restrict__ crow,
                                                uint8_t* __restrict__ srow) {
    constexpr int sfmt = SF;
    static_assert(ZLOG2 >= 0 && ZLOG2 < 30, "z unit");
    constexpr float ZUNIT = 1.f / (float)(1 << ZLOG2);
    constexpr int U = D / 16;
    constexpr float Q = (BITS == 4) ? 7.f : 127.f;
    constexpr float MAG = kMagic + ((BITS == 4) ? 8.f : 128.f);
    float m[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        // a tree (depth 4, max is exact in any order) rather than a chain of 15 dependent maxima
        float t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = fmax_(fabs_(z[16 * u + i]), fabs_(z[16 * u + i + 8]));
#pragma unroll
        for (int i = 0; i < 4; ++i) t[i] = fmax_(t[i], t[i + 4]);
        m[u] = fmax_(fmax_(t[0], t[2]), fmax_(t[1], t[3]));
    }
#pragma unroll
    for (int s = 1; s < U; s <<= 1) {
        if (group >= 32 * s) {
#pragma unroll
            for (int u = 0; u < U; ++u) m[u] = fmax_(m[u], m[u ^ s]);
        }
    }
    float sc[U];
    uint32_t raw[U];  // fp16 bits or the e8m0 byte of the stored scale
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float A = m[u];
        if constexpr (ZLOG2 != 0) A *= ZUNIT;  // the true group absmax (exact: a power of two)
        float inv;
        group_scale<BITS, SF>(A, sc[u], raw[u], inv);
        if constexpr (ZLOG2 != 0) inv *= ZUNIT;  // z / scale for z in units of 2^-ZLOG2
#pragma unroll
        for (int i = 0; i < 16; ++i) z[16 * u + i] = fmaf_(z[16 * u + i], inv, MAG);
        if constexpr (sfmt == SRFTKV_SCALE_FP16) {
            if (A > 65504.f * Q) {  // a saturated scale can push |z/scale| past Q
#pragma unroll
                for (int i = 0; i < 16; ++i) z[16 * u + i] = fminf(fmaxf(z[16 * u + i], MAG - Q), MAG + Q);
            }
        }
    }
    constexpr int WORDS = D * BITS / 32;
    uint32_t w[WORDS];
#pragma unroll
    for (int i = 0; i < WORDS; ++i) w[i] = (BITS == 4) ? pack8_int4(&z[8 * i]) : pack4_int8(&z[4 * i]);
    if constexpr (NARROW) {
        static_assert(WORDS % 2 == 0, "8-byte code stores");
#pragma unroll
        for (int i = 0; i < WORDS / 2; ++i) reinterpret_cast<uint2*>(crow)[i] = make_uint2(w[2 * i], w[2 * i + 1]);
        const int gu = group >> 4, sh = __ffs(gu) - 1;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if ((u & (gu - 1)) != 0) continue;
            if constexpr (sfmt == SRFTKV_SCALE_FP32) reinterpret_cast<float*>(srow)[u >> sh] = sc[u];
            else if constexpr (sfmt == SRFTKV_SCALE_FP16) reinterpret_cast<uint16_t*>(srow)[u >> sh] = (uint16_t)raw[u];
            else srow[u >> sh] = (uint8_t)raw[u];
        }
        return;
    }
    if constexpr (WORDS >= 4) {
#pragma unroll
        for (int i = 0; i < WORDS / 4; ++i)
            reinterpret_cast<uint4*>(crow)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else {
        reinterpret_cast<uint2*>(crow)[0] = make_uint2(w[0], w[1]);
    }
    if constexpr (sfmt == SRFTKV_SCALE_FP32) {
        float* sr = reinterpret_cast<float*>(srow);
        if (group == 16) {
            if constexpr (U >= 4) {
#pragma unroll
                for (int i = 0; i < U / 4; ++i)
                    reinterpret_cast<float4*>(sr)[i] = make_float4(sc[4 * i], sc[4 * i + 1], sc[4 * i + 2], sc[4 * i + 3]);
            } else if constexpr (U == 2) {
                reinterpret_cast<float2*>(sr)[0] = make_float2(sc[0], sc[1]);
            } else {
                sr[0] = sc[0];
            }
        } else {
            const int gu = group >> 4, sh = __ffs(gu) - 1;
#pragma unroll
            for (int u = 0; u < U; ++u)
                if ((u & (gu - 1)) == 0) sr[u >> sh] = sc[u];
        }
    } else if constexpr (sfmt == SRFTKV_SCALE_FP16) {
        uint16_t* sr = reinterpret_cast<uint16_t*>(srow);
        if (group == 16) {
            if constexpr (U >= 8) {
#pragma unroll
                for (int i = 0; i < U / 8; ++i)
                    reinterpret_cast<uint4*>(sr)[i] =
                        make_uint4(raw[8 * i] | (raw[8 * i + 1] << 16), raw[8 * i + 2] | (raw[8 * i + 3] << 16),
                                   raw[8 * i + 4] | (raw[8 * i + 5] << 16), raw[8 * i + 6] | (raw[8 * i + 7] << 16));
            } else if constexpr (U == 4) {
                reinterpret_cast<uint2*>(sr)[0] = make_uint2(raw[0] | (raw[1] << 16), raw[2] | (raw[3] << 16));
            } else if constexpr (U == 2) {
                reinterpret_cast<uint32_t*>(sr)[0] = raw[0] | (raw[1] << 16);
            } else {
                sr[0] = (uint16_t)raw[0];
            }
        } else {
            const int gu = group >> 4, sh = __ffs(gu) - 1;
#pragma unroll
            for (int u = 0; u < U; ++u)
                if ((u & (gu - 1)) == 0) sr[u >> sh] = (uint16_t)raw[u];
        }
    } else {
        if (group == 16) {
            if constexpr (U >= 8) {
#pragma unroll
                for (int i = 0; i < U / 8; ++i)
                    reinterpret_cast<uint2*>(srow)[i] =
                        make_uint2(raw[8 * i] | (raw[8 * i + 1] << 8) | (raw[8 * i + 2] << 16) | (raw[8 * i + 3] << 24),
                                   raw[8 * i + 4] | (raw[8 * i + 5] << 8) | (raw[8 * i + 6] << 16) |
                                       (raw[8 * i + 7] << 24));
            } else if constexpr (U == 4) {
                reinterpret_cast<uint32_t*>(srow)[0] = raw[0] | (raw[1] << 8) | (raw[2] << 16) | (raw[3] << 24);
            } else if constexpr (U == 2) {
                reinterpret_cast<uint16_t*>(srow)[0] = (uint16_t)(raw[0] | (raw[1] << 8));
            } else {
                srow[0] = (uint8_t)raw[0];
            }
        } else {
            const int gu = group >> 4, sh = __ffs(gu) - 1;
#pragma unroll
            for (int u = 0; u < U; ++u)
                if ((u & (gu - 1)) == 0) srow[u >> sh] = (uint8_t)raw[u];
        }
    }
}

// One row with the scale format chosen at run time (uniform per call side)
template <int D, int BITS>
__device__ __forceinline__ void quant_store_row_any(float (&z)[D], int group, int sfmt, uint8_t* __restrict__ crow,
                                                    uint8_t* __restrict__ srow) {
    if (sfmt == SRFTKV_SCALE_FP32)
        quant_store_row<D, BITS, SRFTKV_SCALE_FP32>(z, group, crow, srow);
    else if (sfmt == SRFTKV_SCALE_FP16)
        quant_store_row<D, BITS, SRFTKV_SCALE_FP16>(z, group, crow, srow);
    else
        quant_store_row<D, BITS, SRFTKV_SCALE_E8M0>(z, group, crow, srow);
}

// Value of stored scale i of a row in the given format (e8m0: the byte is the
// fp32 exponent field, byte 0 reads as 0.0f)
__device__ __forceinline__ float load_scale(const uint8_t* __restrict__ srow, int i, int sfmt) {
    if (sfmt == SRFTKV_SCALE_FP32) return __ldg(reinterpret_cast<const float*>(srow) + i);
    if (sfmt == SRFTKV_SCALE_FP16) return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(srow) + i)));
    return __uint_as_float((uint32_t)__ldg(srow + i) << 23);
}

// ---------------------------------------------------------------------------
// Decode one stored row to rotated coordinates q * scale (lambda not applied).
// ---------------------------------------------------------------------------
template <int D, int BITS>
__device__ __forceinline__ void dequant_load_row(const uint8_t* __restrict__ crow, const uint8_t* __restrict__ srow,
                                                 int group, int sfmt, float (&p)[D]) {
    constexpr int WORDS = D * BITS / 32, PER = 32 / BITS, U = D / 16;
    uint32_t w[WORDS];
    if constexpr (WORDS >= 4) {
#pragma unroll
        for (int i = 0; i < WORDS / 4; ++i) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(crow) + i);
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
    } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(crow));
        w[0] = v.x;
        w[1] = v.y;
    }
    const int sh = __ffs(group >> 4) - 1;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const float sc = load_scale(srow, u >> sh, sfmt);
#pragma unroll
        for (int i = 16 * u; i < 16 * u + 16; ++i) {
            const float c = (BITS == 4) ? code_int4(w[i / PER], i % PER) : code_int8(w[i / PER], i % PER);
            p[i] = c * sc;
        }
    }
}

// fp16 pair (x_{2n}, x_{2n+1}) with the SRFT signs applied -> complex z_n
__device__ __forceinline__ void signed_pair(uint32_t w, uint32_t mask, float& re, float& im) {
    const uint32_t s = w ^ mask;
    re = __half2float(__ushort_as_half((unsigned short)(s & 0xFFFFu)));
    im = __half2float(__ushort_as_half((unsigned short)(s >> 16)));
}

// ---------------------------------------------------------------------------
// K1: fused quantize
// ---------------------------------------------------------------------------
template <int D, int BK, int BV>
__device__ __forceinline__ void quantize_tile(const CodecParams& P, const TileId& id, const uint16_t* __restrict__ buf,
                                              int lane) {
    using Gm = Geo<D>;
    constexpr int N = D / 2;
    const CodecSideK& S = P.side[id.side];
    const int t = id.t0 + lane;
    const uint16_t* row = buf + lane * Gm::ROW_H;
    float zr[N], zi[N];
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + Gm::chunk_off(c));
        signed_pair(v.x, P.sign_mask[4 * c + 0], zr[4 * c + 0], zi[4 * c + 0]);
        signed_pair(v.y, P.sign_mask[4 * c + 1], zr[4 * c + 1], zi[4 * c + 1]);
        signed_pair(v.z, P.sign_mask[4 * c + 2], zr[4 * c + 2], zi[4 * c + 2]);
        signed_pair(v.w, P.sign_mask[4 * c + 3], zr[4 * c + 3], zi[4 * c + 3]);
    }
    float z[D];
    if (S.transform == SRFTKV_TRANSFORM_SRHT) {  // d^-1/2 H (signed x): no packing, the output is real
        wht_pairs<N>(zr, zi);
#pragma unroll
        for (int n = 0; n < N; ++n) {
            z[2 * n] = zr[n] * SplitConst<D>::inv_sqrt_d;
            z[2 * n + 1] = zi[n] * SplitConst<D>::inv_sqrt_d;
        }
    } else {
        fft<N, false>(zr, zi);
        split_forward<D>(zr, zi, z);
    }
    if (t >= P.n_tokens) return;
    if (S.lambda != nullptr) {
        const float4* lr =
            reinterpret_cast<const float4*>(S.lambda + (long long)id.o * S.lambda_outer_stride + (long long)id.h * D);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) {
            const float4 l = __ldg(lr + c);
            z[4 * c] *= l.x;
            z[4 * c + 1] *= l.y;
            z[4 * c + 2] *= l.z;
            z[4 * c + 3] *= l.w;
        }
    }
    const long long vrow = packed_row(P, id, t);
    // with equal widths on both sides only one epilogue is compiled
    if (BK == BV || id.side == 0)
        quant_store_row_any<D, BK>(z, P.group, S.sfmt, S.codes + vrow * (D * BK / 8),
                               S.scales + vrow * (D / P.group) * S.sbytes);
    else
        quant_store_row_any<D, BV>(z, P.group, S.sfmt, S.codes + vrow * (D * BV / 8),
                               S.scales + vrow * (D / P.group) * S.sbytes);
}

template <int D, int BK, int BV>
__global__ void __launch_bounds__(128, Geo<D>::MIN_BLOCKS)
    srft_quantize_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                         const __grid_constant__ CodecParams P) {
    using Gm = Geo<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint8_t* bufs = smem + 128 + warp * 2 * Gm::BUF_BYTES;
    const uint32_t bar0 = ptx::smem_u32(&bars[2 * warp]), bar1 = ptx::smem_u32(&bars[2 * warp + 1]);
    if (lane == 0) {
        ptx::mbar_init(bar0, 1);
        ptx::mbar_init(bar1, 1);
        ptx::fence_barrier_init();
    }
    __syncwarp();
    const int stride = gridDim.x * Gm::WARPS;
    int tile = blockIdx.x * Gm::WARPS + warp;
    auto issue = [&](int t, int b) {
        const TileId id = decode_tile<32>(P, t);
        const CUtensorMap* tm = id.side ? &tm1 : &tm0;
        const uint32_t bar = b ? bar1 : bar0;
        const uint32_t dst = ptx::smem_u32(bufs + b * Gm::BUF_BYTES);
        ptx::mbar_arrive_expect_tx(bar, Gm::BUF_BYTES);
        ptx::tma_load_4d(dst, tm, bar, 0, id.h, id.t0, id.o);
    };
    if (lane == 0 && tile < P.total_tiles) issue(tile, 0);
    for (int it = 0; tile < P.total_tiles; ++it, tile += stride) {
        const int b = it & 1;
        const bool has_next = tile + stride < P.total_tiles;
        if (lane == 0 && has_next) issue(tile + stride, b ^ 1);
        const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(b ? bar1 : bar0, (it >> 1) & 1, P.poll_limit));
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
        quantize_tile<D, BK, BV>(P, decode_tile<32>(P, tile), reinterpret_cast<const uint16_t*>(bufs + b * Gm::BUF_BYTES), lane);
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// K2: fused dequantize
// ---------------------------------------------------------------------------
template <int D, int BK, int BV>
__global__ void __launch_bounds__(128, Geo<D>::MIN_BLOCKS)
    srft_dequantize_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                           const __grid_constant__ CodecParams P) {
    using Gm = Geo<D>;
    constexpr int N = D / 2;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* bufs = smem + 128 + warp * 2 * Gm::BUF_BYTES;
    const int stride = gridDim.x * Gm::WARPS;
    int it = 0;
    for (int tile = blockIdx.x * Gm::WARPS + warp; tile < P.total_tiles; tile += stride, ++it) {
        const TileId id = decode_tile<32>(P, tile);
        const CodecSideK& S = P.side[id.side];
        const int t = id.t0 + lane;
        const bool valid = t < P.n_tokens;
        float p[D];
        if (valid) {
            const long long vrow = packed_row(P, id, t);
            const uint8_t* srow = S.scales + vrow * (D / P.group) * S.sbytes;
            if (BK == BV || id.side == 0)
                dequant_load_row<D, BK>(S.codes + vrow * (D * BK / 8), srow, P.group, S.sfmt, p);
            else
                dequant_load_row<D, BV>(S.codes + vrow * (D * BV / 8), srow, P.group, S.sfmt, p);
            if (S.lambda != nullptr) {
                const float4* lr = reinterpret_cast<const float4*>(S.lambda + (long long)id.o * S.lambda_outer_stride +
                                                                   (long long)id.h * D);
#pragma unroll
                for (int c = 0; c < D / 4; ++c) {
                    const float4 l = __ldg(lr + c);
                    p[4 * c] *= __frcp_rn(l.x);
                    p[4 * c + 1] *= __frcp_rn(l.y);
                    p[4 * c + 2] *= __frcp_rn(l.z);
                    p[4 * c + 3] *= __frcp_rn(l.w);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < D; ++i) p[i] = 0.f;
        }
        float zr[N], zi[N];
        if (S.transform == SRFTKV_TRANSFORM_SRHT) {  // H p / sqrt(d), signs applied on output
#pragma unroll
            for (int n = 0; n < N; ++n) {
                zr[n] = p[2 * n] * SplitConst<D>::inv_sqrt_d;
                zi[n] = p[2 * n + 1] * SplitConst<D>::inv_sqrt_d;
            }
            wht_pairs<N>(zr, zi);
        } else {
            split_inverse<D>(p, zr, zi);
            fft<N, true>(zr, zi);
        }
        const int b = it & 1;
        uint16_t* buf = reinterpret_cast<uint16_t*>(bufs + b * Gm::BUF_BYTES);
        // the store issued from this buffer two tiles ago must have read it
        if (lane == 0) ptx::bulk_wait_read<1>();
        __syncwarp();
        uint16_t* row = buf + lane * Gm::ROW_H;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = 4 * c + e;
                __half2 h = __floats2half2_rn(zr[n], zi[n]);
                w[e] = *reinterpret_cast<uint32_t*>(&h) ^ P.sign_mask[n];
            }
            *reinterpret_cast<uint4*>(row + Gm::chunk_off(c)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const CUtensorMap* tm = id.side ? &tm1 : &tm0;
            ptx::tma_store_4d(tm, ptx::smem_u32(buf), 0, id.h, id.t0, id.o);
            ptx::bulk_commit();
        }
    }
    if (lane == 0) ptx::bulk_wait<0>();
}

// Tiles of `rows` tokens: counts per head, side and call, and their divisors.
static inline void set_tile_grid(const CodecCall& c, CodecParams& P, int rows) {
    P.tiles_per_head = (c.n_tokens + rows - 1) / rows;
    P.tiles_per_side = c.n_outer * c.H * P.tiles_per_head;
    P.total_tiles = c.n_sides * P.tiles_per_side;
    P.div_side = make_fastdiv(P.tiles_per_side > 0 ? (uint32_t)P.tiles_per_side : 1u);
    P.div_head = make_fastdiv(P.tiles_per_head > 0 ? (uint32_t)P.tiles_per_head : 1u);
    P.div_H = make_fastdiv((uint32_t)c.H);
}

static inline void fill_params(const CodecCall& c, CodecParams& P) {
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        P.side[s].x = d.x;
        P.side[s].codes = d.codes;
        P.side[s].scales = static_cast<uint8_t*>(d.scales);
        P.side[s].sfmt = d.scale_format;
        P.side[s].sbytes = scale_bytes(d.scale_format);
        P.side[s].lambda = d.lambda;
        P.side[s].lambda_outer_stride = d.lambda_outer_stride;
        P.side[s].bits = d.bits;
        P.side[s].transform = d.transform;
    }
    P.n_outer = c.n_outer;
    P.H = c.H;
    P.t_cap = c.t_cap;
    P.t_offset = c.t_offset;
    P.group = c.group;
    P.n_tokens = c.n_tokens;
    P.lg_group = 0;
    while ((1 << P.lg_group) < c.group) ++P.lg_group;
    set_tile_grid(c, P, 32);
    P.poll_limit = codec_poll_limit();
    for (int i = 0; i < 128; ++i) P.sign_mask[i] = 0;
    sign_masks(c.d, c.seed, P.sign_mask);
}

template <int D, int BK, int BV>
static int launch_codec(const CodecCall& c, bool quantize) {
    using Gm = Geo<D>;
    CodecParams P;
    fill_params(c, P);
    if (P.total_tiles == 0) return 0;
    CUtensorMap tm[2];
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        if (!encode_x_map(&tm[s], d.x, D, c.H, c.n_tokens, c.n_outer, Gm::ROWS, false)) return SRFTKV_ERR_CUDA;
    }
    P.fault = codec_fault_word();
    if (!P.fault) return SRFTKV_ERR_CUDA;
    auto kern = quantize ? srft_quantize_kernel<D, BK, BV> : srft_dequantize_kernel<D, BK, BV>;
    static bool attr_done[2] = {false, false};
    if (!attr_done[quantize]) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
        attr_done[quantize] = true;
    }
    const int warps_needed = P.total_tiles;
    int blocks = (warps_needed + Gm::WARPS - 1) / Gm::WARPS;
    const int cap = device_sm_count() * Gm::MIN_BLOCKS;
    if (blocks > cap) blocks = cap;
    kern<<<blocks, Gm::WARPS * 32, Gm::SMEM, c.stream>>>(tm[0], tm[1], P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("codec kernel launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return 0;
}

// All K/V width combinations of one head dimension (explicitly instantiated
// per dimension in codec_d*.cu).
template <int D>
int launch_codec_d(const CodecCall& c, bool quantize) {
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    if (bk == 4 && bv == 4) return launch_codec<D, 4, 4>(c, quantize);
    if (bk == 8 && bv == 8) return launch_codec<D, 8, 8>(c, quantize);
    if (bk == 8 && bv == 4) return launch_codec<D, 8, 4>(c, quantize);
    return launch_codec<D, 4, 8>(c, quantize);
}

}  // namespace srftkv
