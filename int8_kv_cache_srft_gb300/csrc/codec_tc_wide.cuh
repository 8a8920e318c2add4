// codec_tc_wide.cuh -- SRFT quantize with the transform as a dense contraction
// on the 5th-generation tensor cores for the wide head dimensions d = 192 and
// d = 256 (instantiated in codec_tc_wide192.cu and codec_tc_wide256.cu).
//
// Method: "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
// Apple Silicon", Methodology 1 (SRFT(x) = pack(F diag(s) x) is a fixed real
// d x d orthogonal map R_s), Methodology 4 (the pages' CPU path batches the
// DFT as dense matmuls; this is the GPU counterpart) and Methodology 2-3
// (lambda, group absmax, rounding, packing) in the epilogue.
//
// As at d = 128, a tile is 128 head vectors X (fp16, exact) and the product
// P = X . R_s^T takes R_s as R_hi + R_lo in fp16 (the rounding decisions need
// more than fp16's 11 bits).  R_s is scaled by 2^8 before the split so that
// R_lo stays a normal fp16 (entries near sqrt(2/d) leave residuals below
// fp16's smallest normal, where they would lose bits): about 23 bits
// together; the 2^-8 goes into the group scales.  At d = 256 (K = 256, the
// most accumulation steps) the hi and lo products also go to two fp32
// accumulators, added once in the epilogue.  What changes with d is the
// shared memory: R_hi + R_lo is 2 d^2 bytes (144 KB at d = 192, 256 KB at
// d = 256).  So
//   - the x tile streams through a ring of k-blocks (64 columns x 128 rows,
//     16 KB, the 128-byte swizzle unit) instead of whole tiles, which leaves
//     room for five stages next to R at d = 192;
//   - at d = 256 the output coordinates are split between the two CTAs of a
//     pair (NSPLIT = 2): each holds the 128 rows of R_s for its half (128 KB),
//     reads every x tile of the pair's schedule (the second read of a tile is
//     served from L2, the two CTAs run the same schedule side by side) and
//     writes the codes and scales of its half of each row; groups of at most
//     32 never straddle the halves.
// Warp roles, one persistent CTA per SM (18 warps):
//   warp 0     TMA producer of the x k-blocks;
//   warp 1     owns tensor memory and issues the MMAs (one thread): per tile
//              and k-block four K = 16 steps, hi and lo, N = d / NSPLIT;
//   warps 2-17 epilogue: units of 32 rows x 32 columns of an accumulator
//              (a warp may only touch tensor-memory lanes 32(w%4)..+31),
//              lambda, group absmax, rounding, packing, stores from registers.
#pragma once

#include "codec_impl.cuh"
#include "tcgen05.cuh"

namespace srftkv {

namespace wide {

constexpr int M = 128;                 // rows per tile
constexpr int KB_BYTES = M * 64 * 2;   // one x k-block: 128 rows x 64 fp16 columns, 128-byte swizzled
constexpr int EPI = 16;                // epilogue warps
constexpr int WARPS = 2 + EPI;
constexpr int SMEM_CAP = 232448;       // 227 KB a CTA
constexpr int RLOG2 = 8;               // R_s is held times 2^RLOG2

template <int DV, int NSPLIT>
struct Cfg {
    static constexpr int N = DV / NSPLIT;       // output coordinates of this CTA
    static constexpr int KB = DV / 64;          // k-blocks a tile
    static constexpr int B_KB = N * 128;        // one k-block of R_s: N rows of 128 bytes
    static constexpr int B_BYTES = KB * B_KB;   // R_hi (or R_lo)
    static constexpr int OFF_BLO = B_BYTES;
    static constexpr int OFF_X = 2 * B_BYTES;
    static constexpr int STAGES = (SMEM_CAP - 1024 - 256 - OFF_X) / KB_BYTES;
    static constexpr int OFF_BAR = OFF_X + STAGES * KB_BYTES;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
    static constexpr bool SPLIT_ACC = NSPLIT == 2;   // hi and lo products in two accumulators (d = 256)
    static constexpr int ACC_COLS = SPLIT_ACC ? 2 * N : N;
    static constexpr int NACC = ACC_COLS > 128 ? 2 : 4;  // tiles in flight in the 512 tensor-memory columns
    static constexpr int ACC_STRIDE = 512 / NACC;
    static_assert(ACC_COLS <= ACC_STRIDE, "tensor memory");
    static constexpr int NQ = N / 32;                   // 32-column quarters of an accumulator
    static constexpr int U = 4 * NQ;                    // epilogue units a tile
    static constexpr int UPW = NACC * U / EPI;          // units a warp takes per round of the accumulators
    static_assert(STAGES >= 3, "x stages");
    static_assert(SMEM <= SMEM_CAP, "shared memory");
    static_assert(NACC * U % EPI == 0, "units per round");
    static_assert((2 * STAGES + 2 * NACC) * 8 + 4 <= 256, "barrier area");
};

// Byte offset of element (row n, column k) of an N-row operand stored K-major
// as k-blocks of 64 columns in the 128-byte swizzle layout (the MMA
// descriptors' layout).
template <int N>
__device__ __forceinline__ uint32_t kb_offset(int n, int k) {
    return (uint32_t)((k >> 6) * (N * 128) + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + ((k & 7) << 1));
}

}  // namespace wide

// SF: the scale format of both sides (mixed calls are split on the host)
template <int BK, int BV, int SF, int DV, int NSPLIT>
__global__ void __launch_bounds__(wide::WARPS * 32, 1)
    srft_quantize_tc_wide_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                                 const __grid_constant__ CodecParams P) {
    using C = wide::Cfg<DV, NSPLIT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = (int)blockIdx.x % NSPLIT, pair = (int)blockIdx.x / NSPLIT, npairs = (int)gridDim.x / NSPLIT;
    const int n0 = half * C::N;  // this CTA's first output coordinate
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    constexpr int X_FULL = 0, X_EMPTY = C::STAGES, ACC_FULL = 2 * C::STAGES, ACC_EMPTY = 2 * C::STAGES + C::NACC;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[2 * C::STAGES + 2 * C::NACC]);

    // ---- R_s rows n0 .. n0+N-1 (R diag(s)), split into fp16 hi + lo, in the MMA operand layout ----
    {
        // cos / sin (2 pi m / d) for m < d, in double, in the x stages (not yet in use)
        float* cs = reinterpret_cast<float*>(smem + C::OFF_X);
        float* sn = cs + DV;
        for (int m = threadIdx.x; m < DV; m += blockDim.x) {
            double sv, cv;
            sincospi(2.0 * m / DV, &sv, &cv);
            cs[m] = (float)cv;
            sn[m] = (float)sv;
        }
        __syncthreads();
        const bool srht = P.side[0].transform == SRFTKV_TRANSFORM_SRHT;
        // entries times 2^RLOG2 (exact), so that the fp16 residual R_lo stays normal
        const float isd = (float)((1 << wide::RLOG2) / sqrt((double)DV)), r2 = (float)((1 << wide::RLOG2) * sqrt(2.0 / DV));
        for (int idx = threadIdx.x; idx < C::N * DV; idx += blockDim.x) {
            const int nl = idx / DV, k = idx - nl * DV, n = n0 + nl;
            float v;
            if (srht) v = (__popc(n & k) & 1) ? -isd : isd;  // Hadamard entry / sqrt(d) (d a power of two)
            else if (n == 0) v = isd;
            else if (n == 1) v = (k & 1) ? -isd : isd;
            else {
                const int m = ((n >> 1) * k) % DV;
                v = (n & 1) ? -r2 * sn[m] : r2 * cs[m];
            }
            if (P.sign_mask[k >> 1] & ((k & 1) ? 0x80000000u : 0x8000u)) v = -v;
            const __half hi = __float2half_rn(v);
            const __half lo = __float2half_rn(v - __half2float(hi));
            const uint32_t off = wide::kb_offset<C::N>(nl, k);
            *reinterpret_cast<__half*>(smem + off) = hi;
            *reinterpret_cast<__half*>(smem + C::OFF_BLO + off) = lo;
        }
        ptx::fence_proxy_async_smem();  // generic writes -> tensor-core and TMA (async proxy) accesses
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(bar(X_FULL + s), 1);
            ptx::mbar_init(bar(X_EMPTY + s), 1);
        }
        for (int a = 0; a < C::NACC; ++a) {
            ptx::mbar_init(bar(ACC_FULL + a), 1);
            ptx::mbar_init(bar(ACC_EMPTY + a), C::U);  // one arrival per (lane quarter, column quarter)
        }
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool failed = false;

    if (warp == 0) {
        if (lane == 0) {
            int kbi = 0;  // k-blocks issued so far: stage kbi % STAGES, use kbi / STAGES
            for (int t = pair; t < P.total_tiles && !failed; t += npairs) {
                const TileId id = decode_tile<wide::M>(P, t);
                const CUtensorMap* tm = id.side ? &tm1 : &tm0;
#pragma unroll 1
                for (int kb = 0; kb < C::KB; ++kb, ++kbi) {
                    const int s = kbi % C::STAGES, use = kbi / C::STAGES;
                    if (use > 0 && !ptx::mbar_wait_bounded(bar(X_EMPTY + s), (use - 1) & 1)) {
                        failed = true;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(bar(X_FULL + s), wide::KB_BYTES);
                    ptx::tma_load_4d(sbase + C::OFF_X + s * wide::KB_BYTES, tm, bar(X_FULL + s), 64 * kb, id.h, id.t0,
                                     id.o);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t IDESC = tc::idesc_f16_f32(wide::M, C::N);
            int kbi = 0;
            for (int t = pair, i = 0; t < P.total_tiles && !failed; t += npairs, ++i) {
                const int a = i % C::NACC;
                if (i >= C::NACC && !ptx::mbar_wait_bounded(bar(ACC_EMPTY + a), (i / C::NACC - 1) & 1)) {
                    failed = true;
                    break;
                }
                const uint32_t d_tmem = tmem + a * C::ACC_STRIDE;
#pragma unroll 1
                for (int kb = 0; kb < C::KB; ++kb, ++kbi) {
                    const int s = kbi % C::STAGES;
                    if (!ptx::mbar_wait_bounded(bar(X_FULL + s), (kbi / C::STAGES) & 1)) {
                        failed = true;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t x_base = sbase + C::OFF_X + s * wide::KB_BYTES;
                    const uint32_t b_base = sbase + kb * C::B_KB;
                    const uint32_t d_lo = C::SPLIT_ACC ? d_tmem + C::N : d_tmem;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ad = tc::sw128_desc(x_base + 32 * ks);
                        tc::mma_f16(d_tmem, ad, tc::sw128_desc(b_base + 32 * ks), IDESC, (kb | ks) != 0);
                        tc::mma_f16(d_lo, ad, tc::sw128_desc(b_base + C::OFF_BLO + 32 * ks), IDESC,
                                    C::SPLIT_ACC ? (kb | ks) != 0 : 1);
                    }
                    tc::commit(bar(X_EMPTY + s));  // the k-block stage can be refilled once these MMAs are done
                }
                if (failed) break;
                tc::commit(bar(ACC_FULL + a));  // accumulator a is ready for the epilogue
            }
        }
    } else {
        // Units: (lane quarter, 32-column quarter) of a tile; U a tile, NACC
        // tiles a round of the accumulators.  Warp x = ((w-2) & ~3) | (w % 4)
        // takes units x, x + 16, x + 32, ... of the round (all in its lane
        // quarter, since 16 is a multiple of 4), so every warp does UPW units.
        const int quarter = warp & 3;
        const int x = ((warp - 2) & ~3) | quarter;
        for (int r = 0; !failed; ++r) {
            if (pair + C::NACC * r * npairs >= P.total_tiles) break;
#pragma unroll 1
            for (int uj = 0; uj < C::UPW; ++uj) {
                const int u = x + wide::EPI * uj, tr = u / C::U, cq = (u % C::U) >> 2;
                const int t = pair + (C::NACC * r + tr) * npairs;
                if (t >= P.total_tiles) break;  // later units belong to later tiles
                const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar(ACC_FULL + tr), r & 1));
                if (!ok) {
                    failed = true;
                    break;
                }
                tc::fence_after_sync();
                uint32_t r0[32], r1[32];
                const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16) + tr * C::ACC_STRIDE + cq * 32;
                tc::ld_32x32b_x32(taddr, r0);
                if constexpr (C::SPLIT_ACC) tc::ld_32x32b_x32(taddr + C::N, r1);
                tc::wait_ld(r0);
                if constexpr (C::SPLIT_ACC) tc::wait_ld(r1);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(ACC_EMPTY + tr));  // this unit of accumulator tr is read

                const TileId id = decode_tile<wide::M>(P, t);
                const CodecSideK& S = P.side[id.side];
                const int t_tok = id.t0 + 32 * quarter + lane;
                if (t_tok >= P.n_tokens) continue;
                const int c0 = n0 + 32 * cq;  // first output coordinate of the unit
                float z[32];  // coordinates times 2^RLOG2
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    z[j] = C::SPLIT_ACC ? __uint_as_float(r0[j]) + __uint_as_float(r1[j]) : __uint_as_float(r0[j]);
                if (S.lambda != nullptr) {
                    const float4* lr = reinterpret_cast<const float4*>(
                        S.lambda + (long long)id.o * S.lambda_outer_stride + (long long)id.h * DV + c0);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 l = __ldg(lr + c);
                        z[4 * c] *= l.x;
                        z[4 * c + 1] *= l.y;
                        z[4 * c + 2] *= l.z;
                        z[4 * c + 3] *= l.w;
                    }
                }
                const long long vrow = packed_row(P, id, t_tok);
                const int ng = DV / P.group;
                uint8_t* srow = S.scales + (vrow * ng + c0 / P.group) * S.sbytes;
                if (BK == BV || id.side == 0)
                    quant_store_row<32, BK, SF, wide::RLOG2>(z, P.group, S.codes + vrow * (DV * BK / 8) + c0 * BK / 8,
                                                             srow);
                else
                    quant_store_row<32, BV, SF, wide::RLOG2>(z, P.group, S.codes + vrow * (DV * BV / 8) + c0 * BV / 8,
                                                             srow);
            }
        }
    }
    if (failed) atomicOr(P.fault, 1u);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

template <int BK, int BV, int SF, int DV, int NSPLIT>
static int launch_tc_wide(const CodecCall& c) {
    using C = wide::Cfg<DV, NSPLIT>;
    CodecParams P;
    fill_params(c, P);
    P.tiles_per_head = (c.n_tokens + wide::M - 1) / wide::M;
    P.tiles_per_side = c.n_outer * c.H * P.tiles_per_head;
    P.total_tiles = c.n_sides * P.tiles_per_side;
    P.fault = codec_fault_word();
    if (!P.fault) return SRFTKV_ERR_CUDA;
    CUtensorMap tm[2];
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        if (!encode_x_map(&tm[s], d.x, DV, c.H, c.n_tokens, c.n_outer, wide::M, true)) return SRFTKV_ERR_CUDA;
    }
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(srft_quantize_tc_wide_kernel<BK, BV, SF, DV, NSPLIT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        attr = true;
    }
    // persistent: one CTA an SM, in groups of NSPLIT that run the same tile schedule
    int groups = device_sm_count() / NSPLIT;
    if (groups > P.total_tiles) groups = P.total_tiles;
    if (groups < 1) groups = 1;
    srft_quantize_tc_wide_kernel<BK, BV, SF, DV, NSPLIT><<<groups * NSPLIT, wide::WARPS * 32, C::SMEM, c.stream>>>(
        tm[0], tm[1], P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tensor-core quantize launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return SRFTKV_OK;
}

// Every (K, V) width pair and scale format of one wide head dimension.
template <int DV, int NSPLIT>
int codec_quantize_tc_wide_d(const CodecCall& c) {
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    const int sf = c.side[0].scale_format;  // both sides share it (mixed calls are split on the host)
    auto go = [&](auto sfc) {
        constexpr int SF = decltype(sfc)::value;
        if (bk == 4 && bv == 4) return launch_tc_wide<4, 4, SF, DV, NSPLIT>(c);
        if (bk == 8 && bv == 8) return launch_tc_wide<8, 8, SF, DV, NSPLIT>(c);
        if (bk == 8 && bv == 4) return launch_tc_wide<8, 4, SF, DV, NSPLIT>(c);
        return launch_tc_wide<4, 8, SF, DV, NSPLIT>(c);
    };
    if (sf == SRFTKV_SCALE_FP16) return go(std::integral_constant<int, SRFTKV_SCALE_FP16>{});
    if (sf == SRFTKV_SCALE_E8M0) return go(std::integral_constant<int, SRFTKV_SCALE_E8M0>{});
    return go(std::integral_constant<int, SRFTKV_SCALE_FP32>{});
}

}  // namespace srftkv
