// codec_small.cu -- SRFT / SRHT quantize of d = 128 head vectors with one
// warp per vector, for small calls: appending one token to every head of a
// cache is a few hundred vectors, too few to fill the GPU with one thread per
// vector, so the latency of a vector's dependent chain is what counts.
//
// Method: "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
// Apple Silicon", Methodology 1 (SRFT(x) = pack(F diag(s) x)) and 2 (sign
// multiply, radix-2 FFT, real split and packing, lambda, group absmax,
// rounding, nibble packing), the same arithmetic as the other quantize
// kernels spread over the 32 lanes of a warp:
//   lane l holds x_{4l..4l+3}, i.e. the complex points z_{2l}, z_{2l+1} of
//   z_n = u_{2n} + i u_{2n+1} (u = s x);
//   a 64-point decimation-in-frequency FFT: stages of half-size 32..2 pair
//   lane l with lane l ^ h/2 (shuffles), the last stage pairs the lane's two
//   points; the result sits in bit-reversed order;
//   two gathers put Z_{2l}, Z_{2l+1} and Z_{64-2l}, Z_{63-2l} on lane l,
//   whose split gives y_{2l}, y_{2l+1}, i.e. p_{4l..4l+3};
//   the group absmax of 16 (32) coordinates is a reduction over 4 (8) lanes.
// The SRHT variant is the in-place Walsh-Hadamard butterfly on the same
// layout (two in-lane stages, five across lanes).  Scales and codes are
// computed by group_scale and the same magic-number rounding as the other
// kernels, so every path stores the same bytes for the same z.
#include <type_traits>

#include "codec_impl.cuh"

namespace srftkv {

namespace {
constexpr int WQ_D = 128;
constexpr int WQ_WARPS = 4;  // vectors per block

// e^{-2 pi i m / 256}; per-lane indices, so from the L1-served copy of the table
__device__ __forceinline__ float2 twid(int m) { return make_float2(tw_re_lane(m), tw_im_lane(m)); }

__device__ __forceinline__ float shfl_x(float v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
__device__ __forceinline__ float shfl_i(float v, int src) { return __shfl_sync(0xffffffffu, v, src); }
}  // namespace

// P's tile fields count rows here: total_tiles = all rows of the call, tiles_per_side = rows per side.
template <int BK, int BV, int SF>
__global__ void __launch_bounds__(WQ_WARPS * 32, 1)
    srft_quantize_warp_kernel(const __grid_constant__ CodecParams P, const __half* __restrict__ x0,
                              const __half* __restrict__ x1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long r = (long long)blockIdx.x * WQ_WARPS + warp;
    if (r >= P.total_tiles) return;  // warp-uniform
    const int side = (int)(r / P.tiles_per_side);
    const long long rs = r - (long long)side * P.tiles_per_side;
    const long long per_o = (long long)P.n_tokens * P.H;
    const int o = (int)(rs / per_o);
    const int rem = (int)(rs - (long long)o * per_o), t = rem / P.H, h = rem - t * P.H;
    const CodecSideK& S = P.side[side];
    const __half* x = (side ? x1 : x0) + (((long long)o * P.n_tokens + t) * P.H + h) * WQ_D;

    // x_{4l..4l+3} with the signs of s (fp16 sign-bit flips), as fp32; lambda_{4l..4l+3} loaded alongside
    uint2 w = __ldg(reinterpret_cast<const uint2*>(x) + lane);
    float4 lam4 = make_float4(1.f, 1.f, 1.f, 1.f);
    if (S.lambda != nullptr)
        lam4 = __ldg(reinterpret_cast<const float4*>(S.lambda + (long long)o * S.lambda_outer_stride +
                                                     (long long)h * WQ_D) + lane);
    w.x ^= P.sign_mask[2 * lane];
    w.y ^= P.sign_mask[2 * lane + 1];
    const float2 u01 = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
    const float2 u23 = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
    constexpr float f = 0.08838834764831845f;  // 1/sqrt(128)
    float z[4];
    if (S.transform == SRFTKV_TRANSFORM_SRHT) {
        // H u with H_ij = (-1)^popcount(i & j): element 4l + q, bits 0-1 in the lane, bits 2-6 across lanes
        float a0 = u01.x + u01.y, a1 = u01.x - u01.y, a2 = u23.x + u23.y, a3 = u23.x - u23.y;
        float v0 = a0 + a2, v1 = a1 + a3, v2 = a0 - a2, v3 = a1 - a3;
#pragma unroll
        for (int hs = 1; hs <= 16; hs <<= 1) {
            const float q0 = shfl_x(v0, hs), q1 = shfl_x(v1, hs), q2 = shfl_x(v2, hs), q3 = shfl_x(v3, hs);
            const bool up = (lane & hs) == 0;  // the element with the bit clear gets the sum
            v0 = up ? v0 + q0 : q0 - v0;
            v1 = up ? v1 + q1 : q1 - v1;
            v2 = up ? v2 + q2 : q2 - v2;
            v3 = up ? v3 + q3 : q3 - v3;
        }
        z[0] = v0 * f;
        z[1] = v1 * f;
        z[2] = v2 * f;
        z[3] = v3 * f;
    } else {
        // z_{2l} = (ar, ai), z_{2l+1} = (br, bi); DIF stages of half-size h = 32 .. 2 across lanes
        float ar = u01.x, ai = u01.y, br = u23.x, bi = u23.y;
#pragma unroll
        for (int hs = 16; hs >= 1; hs >>= 1) {
            const int hh = 2 * hs;  // half-size of the butterfly block
            const float par = shfl_x(ar, hs), pai = shfl_x(ai, hs), pbr = shfl_x(br, hs), pbi = shfl_x(bi, hs);
            const bool up = (lane & hs) == 0;
            // lower element e = 2l + jj of a block: (partner - own) * W_{2h}^{e mod h}, W_{2h}^j = tw[128 j / h]
            const float2 w0 = twid((((2 * lane) & (hh - 1)) * (128 / hh)) & 255);
            const float2 w1 = twid((((2 * lane + 1) & (hh - 1)) * (128 / hh)) & 255);
            const float dr0 = par - ar, di0 = pai - ai, dr1 = pbr - br, di1 = pbi - bi;
            const float lr0 = dr0 * w0.x - di0 * w0.y, li0 = dr0 * w0.y + di0 * w0.x;
            const float lr1 = dr1 * w1.x - di1 * w1.y, li1 = dr1 * w1.y + di1 * w1.x;
            ar = up ? ar + par : lr0;
            ai = up ? ai + pai : li0;
            br = up ? br + pbr : lr1;
            bi = up ? bi + pbi : li1;
        }
        {  // half-size 1: the lane's own pair
            const float tr = ar, ti = ai;
            ar = tr + br;
            ai = ti + bi;
            br = tr - br;
            bi = ti - bi;
        }
        // lane l now holds Z at elements 2l, 2l+1 in bit-reversed order; gather Z_{2l} (element
        // rv = bitrev6(2l) < 32: lane rv/2, point rv%2) and Z_{2l+1} (element rv + 32: lane rv/2 + 16)
        const int rv = (int)(__brev((unsigned)(2 * lane)) >> 26), src = rv >> 1;
        const bool odd = rv & 1;
        float s0 = shfl_i(ar, src), s1 = shfl_i(ai, src), s2 = shfl_i(br, src), s3 = shfl_i(bi, src);
        const float zkr0 = odd ? s2 : s0, zki0 = odd ? s3 : s1;
        s0 = shfl_i(ar, src + 16);
        s1 = shfl_i(ai, src + 16);
        s2 = shfl_i(br, src + 16);
        s3 = shfl_i(bi, src + 16);
        const float zkr1 = odd ? s2 : s0, zki1 = odd ? s3 : s1;
        // Z_{64-2l} (Z_0 for l = 0) and Z_{63-2l}, from the lanes holding them now
        const float znr0 = shfl_i(zkr0, (32 - lane) & 31), zni0 = shfl_i(zki0, (32 - lane) & 31);
        const float znr1 = shfl_i(zkr1, 31 - lane), zni1 = shfl_i(zki1, 31 - lane);
        // split: E = (Z_k + conj Z_{N-k}) / 2, O = (Z_k - conj Z_{N-k}) / 2i, U_k = E + W_d^k O, y_k = U_k / sqrt(d)
        auto split = [&](int k, float zr, float zi, float nr, float ni, float& ur, float& ui, float& er, float& orr) {
            er = 0.5f * (zr + nr);
            const float ei = 0.5f * (zi - ni);
            orr = 0.5f * (zi + ni);
            const float oi = -0.5f * (zr - nr);
            const float2 wk = twid(2 * k);  // e^{-2 pi i k / 128}
            ur = er + (wk.x * orr - wk.y * oi);
            ui = ei + (wk.x * oi + wk.y * orr);
        };
        float u0r, u0i, e0, o0, u1r, u1i, e1, o1;
        split(2 * lane, zkr0, zki0, znr0, zni0, u0r, u0i, e0, o0);
        split(2 * lane + 1, zkr1, zki1, znr1, zni1, u1r, u1i, e1, o1);
        constexpr float c2 = 0.125f;  // sqrt(2/128)
        if (lane == 0) {  // p_0 = y_0 and p_1 = y_{d/2}, both real
            z[0] = f * u0r;
            z[1] = f * (e0 - o0);
        } else {
            z[0] = c2 * u0r;
            z[1] = c2 * u0i;
        }
        z[2] = c2 * u1r;
        z[3] = c2 * u1i;
    }
    z[0] *= lam4.x;  // all ones without lambda
    z[1] *= lam4.y;
    z[2] *= lam4.z;
    z[3] *= lam4.w;

    // group absmax over the group's lanes (4 for groups of 16, 8 for 32), then scale, rounding, packing
    float a = fmaxf(fmaxf(fabsf(z[0]), fabsf(z[1])), fmaxf(fabsf(z[2]), fabsf(z[3])));
    const int gl = P.group / 4;  // lanes per group
    for (int m = 1; m < gl; m <<= 1) a = fmaxf(a, shfl_x(a, m));
    const bool k_bits = BK == BV || side == 0;
    const int bits = k_bits ? BK : BV;
    const long long vrow = ((long long)o * P.H + h) * P.t_cap + P.t_offset + t;
    uint8_t* crow = S.codes + vrow * (WQ_D * bits / 8);
    uint8_t* srow = S.scales + vrow * (WQ_D / P.group) * S.sbytes;
    float sc, inv;
    uint32_t raw;
    auto finish = [&](auto bits_c) {
        constexpr int B = decltype(bits_c)::value;
        constexpr float MAG = kMagic + ((B == 4) ? 8.f : 128.f);
        group_scale<B, SF>(a, sc, raw, inv);
        float zm[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) zm[i] = fmaf_(z[i], inv, MAG);
        if constexpr (SF == SRFTKV_SCALE_FP16) {
            constexpr float Q = (B == 4) ? 7.f : 127.f;
            if (a > 65504.f * Q) {  // a saturated scale can push |z/scale| past Q
#pragma unroll
                for (int i = 0; i < 4; ++i) zm[i] = fminf(fmaxf(zm[i], MAG - Q), MAG + Q);
            }
        }
        if constexpr (B == 4) {  // offset-binary nibbles (q + 8), even coordinate low, flipped to two's complement
            const uint32_t q01 = f2u(zm[0]) + (f2u(zm[1]) << 4), q23 = f2u(zm[2]) + (f2u(zm[3]) << 4);
            const uint32_t word = ((q01 + (q23 << 8)) & 0xFFFFu) ^ 0x8888u;
            reinterpret_cast<uint16_t*>(crow)[lane] = (uint16_t)word;
        } else {
            reinterpret_cast<uint32_t*>(crow)[lane] = pack4_int8(zm);
        }
    };
    if (k_bits)
        finish(std::integral_constant<int, BK>{});
    else
        finish(std::integral_constant<int, BV>{});
    if ((lane & (gl - 1)) == 0) {  // the group's first lane stores its scale
        const int j = lane / gl;
        if constexpr (SF == SRFTKV_SCALE_FP32) reinterpret_cast<float*>(srow)[j] = sc;
        else if constexpr (SF == SRFTKV_SCALE_FP16) reinterpret_cast<uint16_t*>(srow)[j] = (uint16_t)raw;
        else srow[j] = (uint8_t)raw;
    }
}

template <int BK, int BV, int SF>
static int launch_warp(const CodecCall& c) {
    CodecParams P;
    fill_params(c, P);
    P.tiles_per_side = c.n_outer * c.n_tokens * c.H;  // rows, see the kernel
    P.total_tiles = c.n_sides * P.tiles_per_side;
    if (P.total_tiles == 0) return 0;
    const __half* x0 = static_cast<const __half*>(c.side[0].x);
    const __half* x1 = static_cast<const __half*>(c.side[c.n_sides > 1 ? 1 : 0].x);
    const int blocks = (P.total_tiles + WQ_WARPS - 1) / WQ_WARPS;
    srft_quantize_warp_kernel<BK, BV, SF><<<blocks, WQ_WARPS * 32, 0, c.stream>>>(P, x0, x1);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("warp quantize launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return 0;
}

template <int SF>
static int launch_warp_bits(const CodecCall& c, int bk, int bv) {
    if (bk == 4 && bv == 4) return launch_warp<4, 4, SF>(c);
    if (bk == 8 && bv == 8) return launch_warp<8, 8, SF>(c);
    if (bk == 8 && bv == 4) return launch_warp<8, 4, SF>(c);
    return launch_warp<4, 8, SF>(c);
}

int codec_quantize_warp(const CodecCall& c) {
    if (c.d != WQ_D || c.group > 32) return 1;  // a group spans at most 8 lanes
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    const int sf = c.side[0].scale_format;  // both sides share it (mixed calls are split on the host)
    if (sf == SRFTKV_SCALE_FP16) return launch_warp_bits<SRFTKV_SCALE_FP16>(c, bk, bv);
    if (sf == SRFTKV_SCALE_E8M0) return launch_warp_bits<SRFTKV_SCALE_E8M0>(c, bk, bv);
    return launch_warp_bits<SRFTKV_SCALE_FP32>(c, bk, bv);
}

}  // namespace srftkv
