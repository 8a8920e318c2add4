// codec_tc.cu -- SRFT quantize and dequantize with the transform done as a
// dense contraction on the 5th-generation tensor cores (head dimension 128).
//
// Method: "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
// Apple Silicon", Methodology 1 (SRFT(x) = pack(F diag(s) x) is a fixed real
// d x d orthogonal map R_s) and Methodology 4 (the pages' CPU path batches
// the DFT as dense matmuls; this is the GPU counterpart).  Methodology 2-3
// (lambda, group absmax, rounding, packing) run unchanged in the epilogue.
//
// For a tile of 128 head vectors X (fp16, exact), P = X . R_s^T is one
// M=128, N=128, K=128 contraction.  R_s is split into two fp16 matrices
// R_hi + R_lo (about 21 significant bits together) and both are applied, so
// each tile is 16 tcgen05.mma (K=16 each) accumulating in fp32 in tensor
// memory.  Warp roles, one persistent CTA per SM:
//   warp 0     TMA producer: x tiles (two 128-byte-swizzled k-blocks) into a
//              3-stage ring;
//   warp 1     allocates tensor memory and issues the MMAs (one thread) into
//              two accumulator buffers;
//   warps 2-9  epilogue: each reads 32 rows x 64 columns of an accumulator
//              (warp w may only touch tensor-memory lanes 32(w%4)..+31),
//              applies lambda, quantises its four 16-coordinate groups and
//              stores codes and scales straight from registers.
// R_hi / R_lo are built once per CTA in shared memory from the twiddle table
// (entries of R are closed forms of cos and sin of 2 pi jk/d).
#include "codec_impl.cuh"
#include "tcgen05.cuh"

namespace srftkv {

namespace {
constexpr int TD = 128;                       // head dimension
constexpr int TM = 128;                       // rows per tile
constexpr int TSTAGES = 3;
constexpr int T_KB_BYTES = TM * 64 * 2;       // one 128-byte-wide k-block of a tile: 16 KB
constexpr int T_A_BYTES = 2 * T_KB_BYTES;     // a full 128 x 128 fp16 tile
constexpr int T_B_BYTES = TD * TD * 2;        // R_hi or R_lo
constexpr int T_OFF_BLO = T_B_BYTES;
constexpr int T_OFF_A = 2 * T_B_BYTES;
constexpr int T_OFF_BAR = T_OFF_A + TSTAGES * T_A_BYTES;
constexpr int T_SMEM = T_OFF_BAR + 128 + 1024;  // + barriers + alignment slack
constexpr int T_WARPS = 10;
constexpr uint32_t T_IDESC = tc::idesc_f16_f32(TM, TD);
constexpr uint32_t T_TMEM_COLS = 256;         // two 128-column fp32 accumulators
}  // namespace

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ TileId decode_tile128(const CodecParams& P, int t) { return decode_tile<TM>(P, t); }

// Byte offset of element (row n, column k) of a 128 x 128 fp16 operand stored
// K-major in two 128-byte-swizzled k-blocks (the layout TMA's 128-byte swizzle
// produces and the MMA descriptors below describe).
__device__ __forceinline__ uint32_t sw128_offset(int n, int k) {
    return (uint32_t)((k >> 6) * T_KB_BYTES + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + ((k & 7) << 1));
}

template <int BK, int BV>
__global__ void __launch_bounds__(T_WARPS * 32, 1)
    srft_quantize_tc_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                            const __grid_constant__ CodecParams P) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, and still a __shared__ pointer so accesses compile to shared-memory instructions
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T_OFF_BAR);
    // barrier indices: full[0..2], empty[3..5], acc_full[6..7], acc_empty[8..9]; tensor-memory slot after them
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[10]);

    // ---- R_s = R diag(s), split into fp16 hi + lo, in the MMA operand layout ----
    {
        constexpr float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)
        constexpr float c2 = 0.125f;                        // sqrt(2/128)
        for (int idx = threadIdx.x; idx < TD * TD; idx += blockDim.x) {
            const int n = idx >> 7, k = idx & 127;
            float v;
            if (n == 0) {
                v = inv_sqrt_d;
            } else if (n == 1) {
                v = (k & 1) ? -inv_sqrt_d : inv_sqrt_d;
            } else {
                const int m = (((n >> 1) * k) & (TD - 1)) * (256 / TD);  // angle 2 pi (jk mod d)/d on the 256-point table
                v = (n & 1) ? c2 * tw_im(m) : c2 * tw_re(m);             // tw_im holds -sin
            }
            const uint32_t sbit = (k & 1) ? 0x80000000u : 0x8000u;
            if (P.sign_mask[k >> 1] & sbit) v = -v;
            const __half hi = __float2half_rn(v);
            const __half lo = __float2half_rn(v - __half2float(hi));
            const uint32_t off = sw128_offset(n, k);
            *reinterpret_cast<__half*>(smem + off) = hi;
            *reinterpret_cast<__half*>(smem + T_OFF_BLO + off) = lo;
        }
        ptx::fence_proxy_async_smem();  // generic writes -> tensor-core (async proxy) reads
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < TSTAGES; ++s) {
            ptx::mbar_init(bar(s), 1);
            ptx::mbar_init(bar(3 + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(bar(6 + a), 1);
            ptx::mbar_init(bar(8 + a), 8);
        }
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(ptx::smem_u32(tmem_slot), T_TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int stride = gridDim.x;
    bool failed = false;

    if (warp == 0) {
        if (lane == 0) {
            for (int t = blockIdx.x, i = 0; t < P.total_tiles; t += stride, ++i) {
                const int s = i % TSTAGES, use = i / TSTAGES;
                if (use > 0 && !ptx::mbar_wait_bounded(bar(3 + s), (use - 1) & 1)) {
                    failed = true;
                    break;
                }
                const TileId id = decode_tile128(P, t);
                const CUtensorMap* tm = id.side ? &tm1 : &tm0;
                const uint32_t dst = sbase + T_OFF_A + s * T_A_BYTES;
                ptx::mbar_arrive_expect_tx(bar(s), T_A_BYTES);
                ptx::tma_load_4d(dst, tm, bar(s), 0, id.h, id.t0, id.o);
                ptx::tma_load_4d(dst + T_KB_BYTES, tm, bar(s), 64, id.h, id.t0, id.o);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int t = blockIdx.x, i = 0; t < P.total_tiles; t += stride, ++i) {
                const int s = i % TSTAGES, a = i & 1;
                if (!ptx::mbar_wait_bounded(bar(s), (i / TSTAGES) & 1) ||
                    (i >= 2 && !ptx::mbar_wait_bounded(bar(8 + a), ((i >> 1) - 1) & 1))) {
                    failed = true;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem + a * TD;
                const uint32_t a_base = sbase + T_OFF_A + s * T_A_BYTES;
#pragma unroll
                for (int ks = 0; ks < TD / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * T_KB_BYTES + (ks & 3) * 32;
                    const uint64_t ad = tc::sw128_desc(a_base + koff);
                    tc::mma_f16(d_tmem, ad, tc::sw128_desc(sbase + koff), T_IDESC, ks > 0);
                    tc::mma_f16(d_tmem, ad, tc::sw128_desc(sbase + T_OFF_BLO + koff), T_IDESC, 1);
                }
                tc::commit(bar(3 + s));  // the x stage can be refilled once these MMAs are done
                tc::commit(bar(6 + a));  // accumulator a is ready for the epilogue
            }
        }
    } else {
        const int quarter = warp & 3, half = (warp - 2) >> 2;
        for (int t = blockIdx.x, i = 0; t < P.total_tiles; t += stride, ++i) {
            const int a = i & 1;
            const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar(6 + a), (i >> 1) & 1));
            if (!ok) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
            uint32_t r0[32], r1[32];
            const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16) + a * TD + half * 64;
            tc::ld_32x32b_x32(taddr, r0);
            tc::ld_32x32b_x32(taddr + 32, r1);
            tc::wait_ld(r0);
            tc::wait_ld(r1);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(8 + a));  // accumulator a may be overwritten

            const TileId id = decode_tile128(P, t);
            const CodecSideK& S = P.side[id.side];
            const int t_tok = id.t0 + 32 * quarter + lane;
            if (t_tok >= P.n_tokens) continue;
            float z[64];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                z[j] = __uint_as_float(r0[j]);
                z[32 + j] = __uint_as_float(r1[j]);
            }
            if (S.lambda != nullptr) {
                const float4* lr = reinterpret_cast<const float4*>(
                    S.lambda + (long long)id.o * S.lambda_outer_stride + (long long)id.h * TD + half * 64);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float4 l = __ldg(lr + c);
                    z[4 * c] *= l.x;
                    z[4 * c + 1] *= l.y;
                    z[4 * c + 2] *= l.z;
                    z[4 * c + 3] *= l.w;
                }
            }
            const long long vrow = packed_row(P, id, t_tok);
            const int ng = TD / P.group;
            if (BK == BV || id.side == 0)
                quant_store_row<64, BK>(z, P.group, S.codes + vrow * (TD * BK / 8) + half * (64 * BK / 8),
                                        S.scales + vrow * ng + half * (ng / 2));
            else
                quant_store_row<64, BV>(z, P.group, S.codes + vrow * (TD * BV / 8) + half * (64 * BV / 8),
                                        S.scales + vrow * ng + half * (ng / 2));
        }
    }
    if (failed) atomicOr(P.fault, 1u);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, T_TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Dequantize: X_hat = P_hat . (R_s)^T, P_hat = codes * scale / lambda
// ---------------------------------------------------------------------------
// Warp roles (one persistent CTA per SM, 10 warps):
//   warp 0     allocates tensor memory and issues the MMAs (one thread);
//   warp 1     TMA producer: the tile's code rows and scale rows, each padded
//              by 16 bytes in shared memory (conflict-free row reads), into a
//              ring of input stages;
//   warps 2-5  converters: thread = row of the tile; decode codes * scale,
//              divide by lambda, write P_hat as fp16 into a 128-byte-swizzled
//              A stage;
//   warps 6-9  epilogue: tensor memory -> fp16 -> swizzled staging -> TMA store
//              (warp w reads tensor-memory lanes 32(w%4)..+31).
// B = diag(s) R (signs folded in), split hi + lo, so X_hat = s (R^T P_hat).
// P_hat is rounded once to fp16 before the contraction; the result is rounded
// to fp16 again on output.
namespace {
constexpr int DQ_WARPS = 10;
constexpr int DQ_SP = 12;                               // padded scale row (floats), groups of 16 or 32
constexpr int DQ_OFF_A = 2 * T_B_BYTES;                 // two A stages of 32 KB
constexpr int DQ_OFF_O = DQ_OFF_A + 2 * T_A_BYTES;      // one output staging buffer of 32 KB
constexpr int DQ_OFF_IN = DQ_OFF_O + T_A_BYTES;         // input stages
template <int BK, int BV>
struct DqCfg {
    static constexpr int RBMAX = TD * (BK > BV ? BK : BV) / 8;
    static constexpr int CODE_RP = RBMAX + 16;                      // padded code row
    static constexpr int OFF_SC = TM * CODE_RP;
    static constexpr int STAGE = (OFF_SC + TM * DQ_SP * 4 + 1023) / 1024 * 1024;
    static constexpr int STAGES = (BK == 4 && BV == 4) ? 3 : 2;
    static constexpr int OFF_BAR = DQ_OFF_IN + STAGES * STAGE;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
};
}  // namespace

template <int D, int BITS>
__device__ __forceinline__ void dequant_row_smem(const uint8_t* __restrict__ crow, const float* __restrict__ srow,
                                                 int group, float (&p)[D]) {
    constexpr int WORDS = D * BITS / 32, PER = 32 / BITS, U = D / 16;
    uint32_t w[WORDS];
#pragma unroll
    for (int i = 0; i < WORDS / 4; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(crow)[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    float sc[U];
    if (group == 16) {  // one scale per 16-coordinate unit: vector loads of the (padded) scale row
#pragma unroll
        for (int i = 0; i < U / 4; ++i) {
            const float4 v = reinterpret_cast<const float4*>(srow)[i];
            sc[4 * i] = v.x;
            sc[4 * i + 1] = v.y;
            sc[4 * i + 2] = v.z;
            sc[4 * i + 3] = v.w;
        }
    } else {
        const int sh = __ffs(group >> 4) - 1;
#pragma unroll
        for (int u = 0; u < U; ++u) sc[u] = srow[u >> sh];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int i = 16 * u; i < 16 * u + 16; ++i) {
            const float c = (BITS == 4) ? code_int4(w[i / PER], i % PER) : code_int8(w[i / PER], i % PER);
            p[i] = c * sc[u];
        }
    }
}

struct DqMaps {
    CUtensorMap out[2], codes[2], scales[2];
};

template <int BK, int BV>
__global__ void __launch_bounds__(DQ_WARPS * 32, 1)
    srft_dequantize_tc_kernel(const __grid_constant__ DqMaps M, const __grid_constant__ CodecParams P) {
    using C = DqCfg<BK, BV>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, and still a __shared__ pointer so accesses compile to shared-memory instructions
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    // a_full[0,1], a_empty[2,3], acc_full[4,5], acc_empty[6,7], in_full[8..10], in_empty[11..13]; tmem slot at 14
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[14]);

    {  // B[k][n] = s_k R[n][k], hi and lo
        constexpr float inv_sqrt_d = 0.08838834764831845f;
        constexpr float c2 = 0.125f;
        for (int idx = threadIdx.x; idx < TD * TD; idx += blockDim.x) {
            const int k = idx >> 7, n = idx & 127;  // B row k (output coordinate), column n (packed coordinate)
            float v;
            if (n == 0) {
                v = inv_sqrt_d;
            } else if (n == 1) {
                v = (k & 1) ? -inv_sqrt_d : inv_sqrt_d;
            } else {
                const int m = (((n >> 1) * k) & (TD - 1)) * (256 / TD);
                v = (n & 1) ? c2 * tw_im(m) : c2 * tw_re(m);
            }
            if (P.sign_mask[k >> 1] & ((k & 1) ? 0x80000000u : 0x8000u)) v = -v;
            const __half hi = __float2half_rn(v);
            const __half lo = __float2half_rn(v - __half2float(hi));
            const uint32_t off = sw128_offset(k, n);
            *reinterpret_cast<__half*>(smem + off) = hi;
            *reinterpret_cast<__half*>(smem + T_OFF_BLO + off) = lo;
        }
        ptx::fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(bar(0 + a), 4);
            ptx::mbar_init(bar(2 + a), 1);
            ptx::mbar_init(bar(4 + a), 1);
            ptx::mbar_init(bar(6 + a), 4);
        }
        for (int st = 0; st < C::STAGES; ++st) {
            ptx::mbar_init(bar(8 + st), 1);
            ptx::mbar_init(bar(11 + st), 4);
        }
        ptx::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(ptx::smem_u32(tmem_slot), T_TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int stride = gridDim.x;
    bool failed = false;

    if (warp == 0) {
        if (lane == 0) {
            for (int t = blockIdx.x, i = 0; t < P.total_tiles; t += stride, ++i) {
                const int s = i & 1;
                if (!ptx::mbar_wait_bounded(bar(0 + s), (i >> 1) & 1) ||
                    (i >= 2 && !ptx::mbar_wait_bounded(bar(6 + s), ((i >> 1) - 1) & 1))) {
                    failed = true;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem + s * TD;
                const uint32_t a_base = sbase + DQ_OFF_A + s * T_A_BYTES;
#pragma unroll
                for (int ks = 0; ks < TD / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * T_KB_BYTES + (ks & 3) * 32;
                    const uint64_t ad = tc::sw128_desc(a_base + koff);
                    tc::mma_f16(d_tmem, ad, tc::sw128_desc(sbase + koff), T_IDESC, ks > 0);
                    tc::mma_f16(d_tmem, ad, tc::sw128_desc(sbase + T_OFF_BLO + koff), T_IDESC, 1);
                }
                tc::commit(bar(2 + s));  // A stage s may be rewritten
                tc::commit(bar(4 + s));  // accumulator s is ready
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int t = blockIdx.x, i = 0; t < P.total_tiles; t += stride, ++i) {
                const int st = i % C::STAGES, use = i / C::STAGES;
                if (use > 0 && !ptx::mbar_wait_bounded(bar(11 + st), (use - 1) & 1)) {
                    failed = true;
                    break;
                }
                const TileId id = decode_tile128(P, t);
                const int bits = (BK == BV || id.side == 0) ? BK : BV;
                const uint32_t dst = sbase + DQ_OFF_IN + st * C::STAGE;
                const int row = P.t_offset + id.t0;   // packed planes: [outer*H][t_cap] rows
                const int oh = id.o * P.H + id.h;
                ptx::mbar_arrive_expect_tx(bar(8 + st), TM * (TD * bits / 8 + 16) + TM * (TD / P.group + 4) * 4);
                ptx::tma_load_3d(dst, &M.codes[id.side], bar(8 + st), 0, row, oh);
                ptx::tma_load_3d(dst + C::OFF_SC, &M.scales[id.side], bar(8 + st), 0, row, oh);
            }
        }
    } else if (warp <= 5) {
        const int m = threadIdx.x - 64;  // row of the tile, 0..127
        for (int t = blockIdx.x, i = 0; t < P.total_tiles; t += stride, ++i) {
            const int s = i & 1, st = i % C::STAGES;
            const TileId id = decode_tile128(P, t);
            const CodecSideK& S = P.side[id.side];
            const int t_tok = id.t0 + m;
            const bool ok_in = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar(8 + st), (i / C::STAGES) & 1));
            if (!ok_in) {
                failed = true;
                break;
            }
            const uint8_t* in = smem + DQ_OFF_IN + st * C::STAGE;
            const float* srow = reinterpret_cast<const float*>(in + C::OFF_SC) + m * (TD / P.group + 4);
            float p[TD];
            if (BK == BV || id.side == 0)
                dequant_row_smem<TD, BK>(in + m * (TD * BK / 8 + 16), srow, P.group, p);
            else
                dequant_row_smem<TD, BV>(in + m * (TD * BV / 8 + 16), srow, P.group, p);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(11 + st));  // input stage consumed
            if (t_tok < P.n_tokens && S.lambda != nullptr) {
                const float4* lr = reinterpret_cast<const float4*>(S.lambda + (long long)id.o * S.lambda_outer_stride +
                                                                   (long long)id.h * TD);
#pragma unroll
                for (int c = 0; c < TD / 4; ++c) {
                    const float4 l = __ldg(lr + c);
                    p[4 * c] = __fdividef(p[4 * c], l.x);
                    p[4 * c + 1] = __fdividef(p[4 * c + 1], l.y);
                    p[4 * c + 2] = __fdividef(p[4 * c + 2], l.z);
                    p[4 * c + 3] = __fdividef(p[4 * c + 3], l.w);
                }
            }
            const bool ok = __all_sync(0xffffffffu, i < 2 || ptx::mbar_wait_bounded(bar(2 + s), ((i >> 1) - 1) & 1));
            if (!ok) {
                failed = true;
                break;
            }
            uint8_t* A = smem + DQ_OFF_A + s * T_A_BYTES;
#pragma unroll
            for (int ch = 0; ch < TD / 8; ++ch) {  // 16-byte chunk ch holds columns 8ch..8ch+7
                uint4 v;
                v.x = pack_half2(p[8 * ch + 0], p[8 * ch + 1]);
                v.y = pack_half2(p[8 * ch + 2], p[8 * ch + 3]);
                v.z = pack_half2(p[8 * ch + 4], p[8 * ch + 5]);
                v.w = pack_half2(p[8 * ch + 6], p[8 * ch + 7]);
                *reinterpret_cast<uint4*>(A + sw128_offset(m, 8 * ch)) = v;
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(0 + s));
        }
    } else {
        const int quarter = warp & 3;   // tensor-memory lanes 32*quarter..+31 = tile rows
        const int m = 32 * quarter + lane;
        const bool leader = (warp == 6 && lane == 0);
        for (int t = blockIdx.x, i = 0; t < P.total_tiles; t += stride, ++i) {
            const int s = i & 1;
            const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar(4 + s), (i >> 1) & 1));
            if (!ok) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
            uint32_t v[4][32];
            const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16) + s * TD;
#pragma unroll
            for (int j = 0; j < 4; ++j) tc::ld_32x32b_x32(taddr + 32 * j, v[j]);
#pragma unroll
            for (int j = 0; j < 4; ++j) tc::wait_ld(v[j]);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(6 + s));
            // the staging buffer: the TMA store of the previous tile must have read it
            if (leader) ptx::bulk_wait_read<0>();
            ptx::named_bar_sync(1, 128);
            uint8_t* O = smem + DQ_OFF_O;
#pragma unroll
            for (int ch = 0; ch < TD / 8; ++ch) {
                const int j = ch >> 2, c0 = (ch & 3) * 8;
                uint4 w;
                w.x = pack_half2(__uint_as_float(v[j][c0 + 0]), __uint_as_float(v[j][c0 + 1]));
                w.y = pack_half2(__uint_as_float(v[j][c0 + 2]), __uint_as_float(v[j][c0 + 3]));
                w.z = pack_half2(__uint_as_float(v[j][c0 + 4]), __uint_as_float(v[j][c0 + 5]));
                w.w = pack_half2(__uint_as_float(v[j][c0 + 6]), __uint_as_float(v[j][c0 + 7]));
                *reinterpret_cast<uint4*>(O + sw128_offset(m, 8 * ch)) = w;
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar_sync(1, 128);
            if (leader) {
                const TileId id = decode_tile128(P, t);
                const uint32_t src = sbase + DQ_OFF_O;
                ptx::tma_store_4d(&M.out[id.side], src, 0, id.h, id.t0, id.o);
                ptx::tma_store_4d(&M.out[id.side], src + T_KB_BYTES, 64, id.h, id.t0, id.o);
                ptx::bulk_commit();
            }
        }
        if (leader) ptx::bulk_wait<0>();
    }
    if (failed) atomicOr(P.fault, 1u);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, T_TMEM_COLS);
}

template <int BK, int BV>
static int launch_dq_tc(const CodecCall& c) {
    using C = DqCfg<BK, BV>;
    CodecParams P;
    fill_params(c, P);
    P.tiles_per_head = (c.n_tokens + TM - 1) / TM;
    P.tiles_per_side = c.n_outer * c.H * P.tiles_per_head;
    P.total_tiles = c.n_sides * P.tiles_per_side;
    P.fault = codec_fault_word();
    if (!P.fault) return SRFTKV_ERR_CUDA;
    DqMaps M;
    const unsigned long long tcap = (unsigned long long)c.t_cap, nrow = (unsigned long long)c.n_outer * c.H;
    const int ng = TD / c.group;
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        const int rb = TD * d.bits / 8;
        // packed planes [n_outer*H][t_cap][row], row padded by 16 bytes in shared memory
        const unsigned long long cdims[3] = {(unsigned long long)rb / 4, tcap, nrow};
        const unsigned long long cstr[2] = {(unsigned long long)rb, tcap * rb};
        const unsigned cbox[3] = {(unsigned)(rb / 4 + 4), (unsigned)TM, 1u};
        const unsigned long long sdims[3] = {(unsigned long long)ng, tcap, nrow};
        const unsigned long long sstr[2] = {ng * 4ull, tcap * ng * 4ull};
        const unsigned sbox[3] = {(unsigned)(ng + 4), (unsigned)TM, 1u};
        if (!encode_x_map(&M.out[s], d.x, TD, c.H, c.n_tokens, c.n_outer, TM, true) ||
            !encode_tiled(&M.codes[s], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, d.codes, cdims, cstr, cbox,
                          "tensor-core dequantize codes") ||
            !encode_tiled(&M.scales[s], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, d.scales, sdims, sstr, sbox,
                          "tensor-core dequantize scales"))
            return SRFTKV_ERR_CUDA;
    }
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(srft_dequantize_tc_kernel<BK, BV>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        attr = true;
    }
    int blocks = device_sm_count();
    if (blocks > P.total_tiles) blocks = P.total_tiles;
    srft_dequantize_tc_kernel<BK, BV><<<blocks, DQ_WARPS * 32, C::SMEM, c.stream>>>(M, P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tensor-core dequantize launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return SRFTKV_OK;
}

template <int BK, int BV>
static int launch_tc(const CodecCall& c) {
    CodecParams P;
    fill_params(c, P);
    P.tiles_per_head = (c.n_tokens + TM - 1) / TM;
    P.tiles_per_side = c.n_outer * c.H * P.tiles_per_head;
    P.total_tiles = c.n_sides * P.tiles_per_side;
    P.fault = codec_fault_word();
    if (!P.fault) return SRFTKV_ERR_CUDA;
    CUtensorMap tm[2];
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        if (!encode_x_map(&tm[s], d.x, TD, c.H, c.n_tokens, c.n_outer, TM, true)) return SRFTKV_ERR_CUDA;
    }
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(srft_quantize_tc_kernel<BK, BV>, cudaFuncAttributeMaxDynamicSharedMemorySize, T_SMEM);
        attr = true;
    }
    int blocks = device_sm_count();
    if (blocks > P.total_tiles) blocks = P.total_tiles;
    srft_quantize_tc_kernel<BK, BV><<<blocks, T_WARPS * 32, T_SMEM, c.stream>>>(tm[0], tm[1], P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tensor-core quantize launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return SRFTKV_OK;
}

int codec_quantize_tc(const CodecCall& c) {
    if (c.d != TD || c.group > 64) return 1;
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    if (bk == 4 && bv == 4) return launch_tc<4, 4>(c);
    if (bk == 8 && bv == 8) return launch_tc<8, 8>(c);
    if (bk == 8 && bv == 4) return launch_tc<8, 4>(c);
    return launch_tc<4, 8>(c);
}

int codec_dequantize_tc(const CodecCall& c) {
    if (c.d != TD || c.group > 32) return 1;  // scale rows must be at least 16 bytes for the TMA copy
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    if (bk == 4 && bv == 4) return launch_dq_tc<4, 4>(c);
    if (bk == 8 && bv == 8) return launch_dq_tc<8, 8>(c);
    if (bk == 8 && bv == 4) return launch_dq_tc<8, 4>(c);
    return launch_dq_tc<4, 8>(c);
}

}  // namespace srftkv
