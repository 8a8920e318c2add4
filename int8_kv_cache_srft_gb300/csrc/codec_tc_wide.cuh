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
#include "codec_tc_common.cuh"
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
        uint32_t* smask = reinterpret_cast<uint32_t*>(sn + DV);
        for (int m = threadIdx.x; m < DV; m += blockDim.x) {
            double sv, cv;
            sincospi(2.0 * m / DV, &sv, &cv);
            cs[m] = (float)cv;
            sn[m] = (float)sv;
        }
        stage_sign_mask(smask, P.sign_mask, DV / 2);
        __syncthreads();
        const bool srht = P.side[0].transform == SRFTKV_TRANSFORM_SRHT;
        // entries times 2^RLOG2 (exact), so that the fp16 residual R_lo stays normal
        const float isd = (float)((1 << wide::RLOG2) / sqrt((double)DV)), r2 = (float)((1 << wide::RLOG2) * sqrt(2.0 / DV));
        auto entry = [&](int n, int k) -> float {
            float v;
            if (srht) v = (__popc(n & k) & 1) ? -isd : isd;  // Hadamard entry / sqrt(d) (d a power of two)
            else if (n == 0) v = isd;
            else if (n == 1) v = (k & 1) ? -isd : isd;
            else {
                const int m = ((n >> 1) * k) % DV;
                v = (n & 1) ? -r2 * sn[m] : r2 * cs[m];
            }
            return sign_flip(smask, k) ? -v : v;
        };
        // one 16-byte chunk (8 consecutive k of row n) of R_hi and of R_lo a step
        for (int c = threadIdx.x; c < C::N * DV / 8; c += blockDim.x) {
            const int nl = c / (DV / 8), k0 = (c - nl * (DV / 8)) * 8, n = n0 + nl;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) split_pair_h2(entry(n, k0 + 2 * j), entry(n, k0 + 2 * j + 1), hi[j], lo[j]);
            const uint32_t off = wide::kb_offset<C::N>(nl, k0);
            *reinterpret_cast<uint4*>(smem + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(smem + C::OFF_BLO + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
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
                const int ng = DV >> P.lg_group;
                uint8_t* srow = S.scales + (vrow * ng + (c0 >> P.lg_group)) * S.sbytes;
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
    set_tile_grid(c, P, wide::M);
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

// ---------------------------------------------------------------------------
// Dequantize at d = 192 and 256: X_hat = s (R^T P_hat), P_hat = codes * scale
// ---------------------------------------------------------------------------
// The d = 128 design (codec_tc.cu) widened:
//   warp 0      owns tensor memory and issues the MMAs (one thread): per tile
//               two contractions of N = d/2 output coordinates each, into two
//               accumulators, so the epilogue drains one half while the
//               other is computed;
//   warp 1      TMA producer: each tile's code rows and scale rows into a ring
//               of input stages.  A code row is copied as segments of 128, 64
//               or 32 bytes (96 = 64 + 32, 192 = 128 + 64, 256 = 128 + 128),
//               each with the TMA swizzle equal to its width, which keeps the
//               row-per-thread reads free of bank conflicts;
//   warps 2-9   converters: thread = half a row; codes * scale as exact fp16
//               pairs (the K order of dq_kperm), written into tensor memory
//               as the MMA's A operand, in pieces of 8 or 4 code words;
//   warps 10-17 epilogue: tensor memory -> fp16 -> global, each thread
//               storing its row's half (d bytes) straight from registers (no
//               staging buffer: the shared memory goes to R_s, 72 or 128 KB).
// B = diag(s) R in fp16 (P_hat and the output are fp16).  A side with lambda
// takes the register path (there is no room for the fp32 copy of R_s that
// the d = 128 kernel rebuilds B from).
namespace wide {
constexpr int DQ_CONV = 8, DQ_EPI = 8, DQ_WARPS = 2 + DQ_CONV + DQ_EPI;
// tensor memory: a ring of three accumulator slots of 128 columns (one output half of a tile each, so
// the epilogue has a tile and a half of slack) and one A buffer at column 384; the converters convert
// the next tile into registers before they wait for the A buffer, so one suffices
constexpr int DQ_NA = 1, DQ_SLOTS = 3;
constexpr uint32_t DQ_A_COL = 384, DQ_A_STRIDE = 128;

// Segments of a code row of rb bytes: powers of two of at most 128 bytes, largest first.
__host__ __device__ constexpr int seg_width(int rb, int s) {
    return rb == 96 ? (s == 0 ? 64 : 32) : rb == 128 ? 128 : rb == 192 ? (s == 0 ? 128 : 64) : 128;
}
__host__ __device__ constexpr int seg_count(int rb) { return rb == 128 ? 1 : 2; }
__host__ __device__ constexpr int seg_off(int rb, int s) { return s == 0 ? 0 : seg_width(rb, 0); }

template <int DV, int BK, int BV>
struct DqCfg {
    static constexpr int RBMAX = DV * (BK > BV ? BK : BV) / 8;   // code bytes a row
    static constexpr int OFF_SC = M * RBMAX;                       // 1024-aligned
    static constexpr int STAGE = (OFF_SC + M * (DV / 4) + 1023) / 1024 * 1024;  // scale rows of at most d/4 bytes
    static constexpr int B_BYTES = DV * DV * 2;                    // R_s in fp16, k-blocks of DV rows
    static constexpr int OFF_IN = B_BYTES;
    static constexpr int STAGES = (SMEM_CAP - 1024 - 256 - OFF_IN) / STAGE > 4 ? 4 : (SMEM_CAP - 1024 - 256 - OFF_IN) / STAGE;
    static constexpr int OFF_BAR = OFF_IN + STAGES * STAGE;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
    static_assert(STAGES >= 2, "input stages");
    static_assert(SMEM <= SMEM_CAP, "shared memory");
};

// Byte offset, in an input stage, of 16-byte chunk c of code row m (rows of rb bytes in swizzled segments)
__device__ __forceinline__ uint32_t code_chunk(int rb, int m, int c) {
    const int p = 16 * c;
    const int s = p >= seg_width(rb, 0) ? 1 : 0;
    const int w = seg_width(rb, s), cc = (p - seg_off(rb, s)) >> 4;
    return (uint32_t)(M * seg_off(rb, s) + m * w + (swz16(w, m, cc) << 4));
}

// Scale of 16-coordinate unit u of tile row m: fp32 planes of d = 256 as swizzled rows (64 bytes for
// group 16, 32 for group 32), every other plane as its contiguous bytes (rows of ng * sb bytes)
template <int DV>
__device__ __forceinline__ float unit_scale(const uint8_t* __restrict__ in, int m, int u, int group, int sfmt) {
    const int lg = __ffs(group) - 1;  // group: a power of two
    const int gi = (16 * u) >> lg, ng = DV >> lg;
    if (sfmt == SRFTKV_SCALE_FP32) {
        if constexpr (DV == 256) {
            const int srb = 4 * ng, b = 4 * gi;
            return *reinterpret_cast<const float*>(in + m * srb + (swz16(srb, m, b >> 4) << 4) + (b & 15));
        } else {
            return *reinterpret_cast<const float*>(in + (m * ng + gi) * 4);
        }
    }
    if (sfmt == SRFTKV_SCALE_FP16)
        return __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(in + (m * ng + gi) * 2)));
    return __uint_as_float((uint32_t)in[m * ng + gi] << 23);  // e8m0: the byte is the fp32 exponent field
}

// Scales of the NU 16-coordinate units u0 .. u0+NU-1 of tile row m (u0 even), with vector loads where the
// row layout allows: fp32 rows of d = 256 are swizzled 16-byte chunks, fp32 rows of d = 192 contiguous and
// 8-byte aligned at even groups; fp16 / e8m0 rows contiguous
template <int DV, int NU>
__device__ __forceinline__ void unit_scales(const uint8_t* __restrict__ in, int m, int u0, int group, int sfmt,
                                            float (&sc)[NU]) {
    const int ng = DV >> (__ffs(group) - 1);  // group: a power of two
    if (sfmt == SRFTKV_SCALE_FP32 && group == 16) {
        if constexpr (DV == 256) {  // 64-byte rows, 64-byte swizzle; u0 a multiple of 4
            const int srb = 64;
#pragma unroll
            for (int q = 0; q < NU / 4; ++q) {
                const float4 v = *reinterpret_cast<const float4*>(in + m * srb + (swz16(srb, m, u0 / 4 + q) << 4));
                sc[4 * q] = v.x, sc[4 * q + 1] = v.y, sc[4 * q + 2] = v.z, sc[4 * q + 3] = v.w;
            }
            if constexpr (NU % 4 == 0) return;
        } else {  // 48-byte rows; unit = group, 8-byte aligned pairs
#pragma unroll
            for (int q = 0; q < NU / 2; ++q) {
                const float2 v = *reinterpret_cast<const float2*>(in + (m * ng + u0 + 2 * q) * 4);
                sc[2 * q] = v.x, sc[2 * q + 1] = v.y;
            }
            return;
        }
    }
#pragma unroll
    for (int u = 0; u < NU; ++u) sc[u] = unit_scale<DV>(in, m, u0 + u, group, sfmt);
}

// fp16 pairs of NW consecutive 8-coordinate code words starting at word w0 of tile row m: codes * scale
// with the scale split into fp16 hi + lo (one main rounding), in the K order of dq_kperm
template <int DV, int BITS, int NW>
__device__ __forceinline__ void word_pairs(const uint8_t* __restrict__ in, int off_sc, int m, int w0, int group,
                                           int sfmt, uint32_t (&hp)[4 * NW]) {
    constexpr int RB = DV * BITS / 8;
    constexpr int NCH = NW * BITS / 16;  // 16-byte chunks of the NW words (8 coordinates = BITS bytes)
    uint32_t w[4 * NCH];
    const int c0 = w0 * BITS / 16;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const uint4 v = *reinterpret_cast<const uint4*>(in + code_chunk(RB, m, c0 + k));
        w[4 * k] = v.x;
        w[4 * k + 1] = v.y;
        w[4 * k + 2] = v.z;
        w[4 * k + 3] = v.w;
    }
    float scu[NW / 2];
    unit_scales<DV, NW / 2>(in + off_sc, m, w0 / 2, group, sfmt, scu);
#pragma unroll
    for (int u = 0; u < NW / 2; ++u) {  // unit u: words 2u, 2u+1 (16 coordinates)
        const float sc = scu[u];
        const __half h = __float2half_rn(sc);
        const uint32_t sh = half2_bcast(h), sl = half2_bcast(__float2half_rn(sc - __half2float(h)));
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int k = 2 * u + e;
            uint32_t c[4];
            if constexpr (BITS == 4) {
                const uint32_t x = w[k], xs = x >> 8;
                c[0] = codes_lo4(x);
                c[1] = codes_hi4(x);
                c[2] = codes_lo4(xs);
                c[3] = codes_hi4(xs);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)  // bytes j of the two words: coordinates 8k + j and 8k + j + 4
                    c[j] = codes_b8(__byte_perm(w[2 * k], w[2 * k + 1], j | (j << 4) | ((4 + j) << 8) | ((4 + j) << 12)));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) hp[4 * k + j] = h2fma(c[j], sh, h2mul(c[j], sl));
        }
    }
}
}  // namespace wide

struct WideDqMaps {
    CUtensorMap codes[2][2];  // [side][segment]
    CUtensorMap scales[2];
};

template <int BK, int BV, int DV>
__global__ void __launch_bounds__(wide::DQ_WARPS * 32, 1)
    srft_dequantize_tc_wide_kernel(const __grid_constant__ WideDqMaps Mp, const __grid_constant__ CodecParams P) {
    using C = wide::DqCfg<DV, BK, BV>;
    constexpr int M = wide::M, NH = DV / 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    constexpr int IN_FULL = 0, IN_EMPTY = C::STAGES, A_FULL = 2 * C::STAGES, A_EMPTY = A_FULL + wide::DQ_NA,
                  ACC_FULL = A_EMPTY + wide::DQ_NA, ACC_EMPTY = ACC_FULL + wide::DQ_SLOTS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[ACC_EMPTY + wide::DQ_SLOTS]);

    {  // B[k][q] = s_k R[n][k] with n = dq_kperm(q), fp16, in the MMA operand layout (k-blocks of DV rows)
        float* cs = reinterpret_cast<float*>(smem + C::OFF_IN);  // cos / sin (2 pi m/d) in the (unused) input stages
        float* sn = cs + DV;
        uint32_t* smask = reinterpret_cast<uint32_t*>(sn + DV);
        for (int m = threadIdx.x; m < DV; m += blockDim.x) {
            double sv, cv;
            sincospi(2.0 * m / DV, &sv, &cv);
            cs[m] = (float)cv;
            sn[m] = (float)sv;
        }
        stage_sign_mask(smask, P.sign_mask, DV / 2);
        __syncthreads();
        const bool srht = P.side[0].transform == SRFTKV_TRANSFORM_SRHT;
        const float isd = (float)(1.0 / sqrt((double)DV)), r2 = (float)sqrt(2.0 / DV);
        // one 16-byte chunk a step: B row k (output coordinate), K positions q0 .. q0+7 holding packed
        // coordinates dq_kperm(q)
        for (int c = threadIdx.x; c < DV * DV / 8; c += blockDim.x) {
            const int k = c / (DV / 8), q0 = (c - k * (DV / 8)) * 8;
            const bool flip = sign_flip(smask, k);
            uint32_t h[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int n = dq_kperm(q0 + 2 * j + e);
                    float v;
                    if (srht) v = (__popc(n & k) & 1) ? -isd : isd;
                    else if (n == 0) v = isd;
                    else if (n == 1) v = (k & 1) ? -isd : isd;
                    else {
                        const int mm = ((n >> 1) * k) % DV;
                        v = (n & 1) ? -r2 * sn[mm] : r2 * cs[mm];
                    }
                    v2[e] = flip ? -v : v;
                }
                h[j] = pack_half2(v2[0], v2[1]);
            }
            *reinterpret_cast<uint4*>(smem + wide::kb_offset<DV>(k, q0)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
        ptx::fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            ptx::mbar_init(bar(IN_FULL + st), 1);
            ptx::mbar_init(bar(IN_EMPTY + st), wide::DQ_CONV);
        }
        for (int b = 0; b < wide::DQ_NA; ++b) {
            ptx::mbar_init(bar(A_FULL + b), wide::DQ_CONV);
            ptx::mbar_init(bar(A_EMPTY + b), 1);
        }
        for (int h = 0; h < wide::DQ_SLOTS; ++h) {
            ptx::mbar_init(bar(ACC_FULL + h), 1);
            ptx::mbar_init(bar(ACC_EMPTY + h), wide::DQ_EPI / 2);  // the four epilogue warps of one output half
        }
        ptx::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int count = (P.total_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    bool failed = false;

    if (warp == 0) {
        if (lane == 0) {
            constexpr uint32_t IDESC = tc::idesc_f16_f32(M, NH);
            for (int i = 0; i < count && !failed; ++i) {
                const int b = i % wide::DQ_NA;
                if (!ptx::mbar_wait_bounded(bar(A_FULL + b), (i / wide::DQ_NA) & 1)) {
                    failed = true;
                    break;
                }
                const uint32_t a_tmem = tmem + wide::DQ_A_COL + b * wide::DQ_A_STRIDE;
#pragma unroll 1
                for (int hf = 0; hf < 2; ++hf) {
                    const int j = 2 * i + hf, sl = j % wide::DQ_SLOTS;  // half j of the call -> slot j % 3
                    if (j >= wide::DQ_SLOTS &&
                        !ptx::mbar_wait_bounded(bar(ACC_EMPTY + sl), (j / wide::DQ_SLOTS - 1) & 1)) {
                        failed = true;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t d_tmem = tmem + sl * 128;
#pragma unroll
                    for (int ks = 0; ks < DV / 16; ++ks) {
                        const uint32_t boff = (ks >> 2) * (DV * 128) + hf * NH * 128 + (ks & 3) * 32;
                        tc::mma_f16_ta(d_tmem, a_tmem + 8 * ks, tc::sw128_desc(sbase + boff), IDESC, ks > 0);
                    }
                    tc::commit(bar(ACC_FULL + sl));  // output half hf of this tile is ready
                }
                if (failed) break;
                tc::commit(bar(A_EMPTY + b));  // A buffer b may be rewritten once these MMAs are done
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int i = 0; i < count; ++i) {
                const int t = blockIdx.x + i * gridDim.x;
                const int st = i % C::STAGES, use = i / C::STAGES;
                if (use > 0 && !ptx::mbar_wait_bounded(bar(IN_EMPTY + st), (use - 1) & 1)) {
                    failed = true;
                    break;
                }
                const TileId id = decode_tile<M>(P, t);
                const int bits = (BK == BV || id.side == 0) ? BK : BV, rb = DV * bits / 8;
                const uint32_t dst = sbase + C::OFF_IN + st * C::STAGE;
                const int row = P.t_offset + id.t0;  // packed planes: [outer*H][t_cap] rows
                const int oh = id.o * P.H + id.h;
                const int sb = P.side[id.side].sbytes, ng = DV >> P.lg_group;
                // fp32 scale rows of d = 256 through the tensor map (swizzled rows); every other plane as the
                // tile's contiguous bytes by a plain bulk copy that stops at the end of this (outer, head)
                const bool flat = !(sb == 4 && DV == 256);
                const uint32_t sc_bytes = flat ? (uint32_t)(min(M, P.t_cap - row) * ng * sb) : (uint32_t)(M * ng * sb);
                ptx::mbar_arrive_expect_tx(bar(IN_FULL + st), M * rb + sc_bytes);
                for (int sg = 0; sg < wide::seg_count(rb); ++sg)
                    ptx::tma_load_3d(dst + M * wide::seg_off(rb, sg), &Mp.codes[id.side][sg], bar(IN_FULL + st),
                                     wide::seg_off(rb, sg), row, oh);
                if (flat)
                    ptx::bulk_load(dst + C::OFF_SC, P.side[id.side].scales + ((long long)oh * P.t_cap + row) * ng * sb,
                                   sc_bytes, bar(IN_FULL + st));
                else
                    ptx::tma_load_3d(dst + C::OFF_SC, &Mp.scales[id.side], bar(IN_FULL + st), 0, row, oh);
            }
        }
    } else if (warp < 2 + wide::DQ_CONV) {
        // converter warp w: tile rows = tensor-memory lanes 32(w%4)..+31, row half (w-2)/4
        const int quarter = warp & 3, m = 32 * quarter + lane, hf = (warp - 2) >> 2;
        const uint32_t lanes = tmem + ((uint32_t)(32 * quarter) << 16);
        for (int i = 0; i < count; ++i) {
            const int t = blockIdx.x + i * gridDim.x;
            const int b = i % wide::DQ_NA, st = i % C::STAGES;
            const TileId id = decode_tile<M>(P, t);
            const CodecSideK& S = P.side[id.side];
            if (!__all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar(IN_FULL + st), (i / C::STAGES) & 1))) {
                failed = true;
                break;
            }
            const uint8_t* in = smem + C::OFF_IN + st * C::STAGE;
            const bool side_k = BK == BV || id.side == 0;
            // half hf = code words hf*DV/16 .. +DV/16-1 = A columns hf*DV/4 .. +DV/4-1 (column c holds word c/4),
            // converted into registers first, then written in pieces of 8 words (32 columns) and, at d = 192,
            // one of 4 words (16 columns), each at a column offset that is a multiple of its width
            constexpr int NWA = DV == 256 ? 8 : 8, NWB = DV == 256 ? 8 : 4;
            const int wa = DV == 256 ? 16 * hf : (hf == 0 ? 0 : 16), wb = DV == 256 ? 16 * hf + 8 : (hf == 0 ? 8 : 12);
            uint32_t ha[4 * NWA], hb[4 * NWB];
            if (side_k) {
                wide::word_pairs<DV, BK, NWA>(in, C::OFF_SC, m, wa, P.group, S.sfmt, ha);
                wide::word_pairs<DV, BK, NWB>(in, C::OFF_SC, m, wb, P.group, S.sfmt, hb);
            } else {
                wide::word_pairs<DV, BV, NWA>(in, C::OFF_SC, m, wa, P.group, S.sfmt, ha);
                wide::word_pairs<DV, BV, NWB>(in, C::OFF_SC, m, wb, P.group, S.sfmt, hb);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(IN_EMPTY + st));  // input stage consumed
            if (!__all_sync(0xffffffffu,
                            i < wide::DQ_NA || ptx::mbar_wait_bounded(bar(A_EMPTY + b), (i / wide::DQ_NA - 1) & 1))) {
                failed = true;
                break;
            }
            tc::fence_after_sync();  // the MMAs that read A buffer b are complete
            const uint32_t acol = lanes + wide::DQ_A_COL + b * wide::DQ_A_STRIDE;
            tc::st_32x32b_x32(acol + 4 * wa, ha);
            if constexpr (NWB == 8) tc::st_32x32b_x32(acol + 4 * wb, hb);
            else tc::st_32x32b_x16(acol + 4 * wb, hb);
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(A_FULL + b));
        }
    } else {
        // epilogue warp w: tensor-memory lanes 32(w%4)..+31 = tile rows, output half (w-10)/4
        const int quarter = warp & 3, hf = (warp - 2 - wide::DQ_CONV) >> 2;
        for (int i = 0; i < count; ++i) {
            const int t = blockIdx.x + i * gridDim.x;
            const int j = 2 * i + hf, sl = j % wide::DQ_SLOTS;
            const uint32_t lanes = tmem + ((uint32_t)(32 * quarter) << 16) + sl * 128;
            if (!__all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar(ACC_FULL + sl), (j / wide::DQ_SLOTS) & 1))) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
            const TileId id = decode_tile<M>(P, t);
            const int t_tok = id.t0 + 32 * quarter + lane;
            const bool live = t_tok < P.n_tokens;
            uint4* dst = reinterpret_cast<uint4*>(
                reinterpret_cast<__half*>(P.side[id.side].x) +
                ((((long long)id.o * P.n_tokens + t_tok) * P.H + id.h) * DV + hf * NH));
            // the row's segment starts on 32 bytes when x does (rows of 2d bytes, halves of d bytes)
            const bool v8 = (reinterpret_cast<uintptr_t>(P.side[id.side].x) & 31u) == 0u;
            auto store32 = [&](int j, const uint32_t (&v)[32]) {  // fp32 columns 32j .. +31 -> fp16 -> global
                if (!live) return;
                uint32_t h[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) h[q] = pack_half2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
                if (v8) {
                    ptx::st_global_v8(dst + 4 * j, h[0], h[1], h[2], h[3], h[4], h[5], h[6], h[7]);
                    ptx::st_global_v8(dst + 4 * j + 2, h[8], h[9], h[10], h[11], h[12], h[13], h[14], h[15]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) dst[4 * j + q] = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                }
            };
            // two 32-column loads in flight at a time; the accumulator half is released right after the last one
            uint32_t va[32], vb[32];
            tc::ld_32x32b_x32(lanes, va);
            tc::ld_32x32b_x32(lanes + 32, vb);
            tc::wait_ld(va);
            tc::wait_ld(vb);
            if constexpr (NH == 96) {
                store32(0, va);
                tc::ld_32x32b_x32(lanes + 64, va);
                tc::wait_ld(va);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(ACC_EMPTY + sl));  // the slot may be overwritten
                store32(1, vb);
                store32(2, va);
            } else {
                store32(0, va);
                store32(1, vb);
                tc::ld_32x32b_x32(lanes + 64, va);
                tc::ld_32x32b_x32(lanes + 96, vb);
                tc::wait_ld(va);
                tc::wait_ld(vb);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(ACC_EMPTY + sl));
                store32(2, va);
                store32(3, vb);
            }
        }
    }
    if (failed) atomicOr(P.fault, 1u);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

template <int BK, int BV, int DV>
static int launch_dq_tc_wide(const CodecCall& c) {
    using C = wide::DqCfg<DV, BK, BV>;
    CodecParams P;
    fill_params(c, P);
    set_tile_grid(c, P, wide::M);
    P.fault = codec_fault_word();
    if (!P.fault) return SRFTKV_ERR_CUDA;
    WideDqMaps Mp;
    const unsigned long long tcap = (unsigned long long)c.t_cap, nrow = (unsigned long long)c.n_outer * c.H;
    const int ng = DV / c.group;
    auto swz = [](int bytes) {
        return bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
               : bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
               : bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                             : CU_TENSOR_MAP_SWIZZLE_NONE;
    };
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        const int rb = DV * d.bits / 8;
        // code plane [n_outer*H][t_cap][rb] as segments of the row, each with its own swizzle
        for (int sg = 0; sg < 2; ++sg) {
            const int g = sg < wide::seg_count(rb) ? sg : 0;
            const unsigned long long cdims[3] = {(unsigned long long)rb, tcap, nrow};
            const unsigned long long cstr[2] = {(unsigned long long)rb, tcap * rb};
            const unsigned cbox[3] = {(unsigned)wide::seg_width(rb, g), (unsigned)wide::M, 1u};
            if (!encode_tiled_swz(&Mp.codes[s][sg], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, d.codes, cdims, cstr, cbox,
                                  swz(wide::seg_width(rb, g)), "wide tensor-core dequantize codes"))
                return SRFTKV_ERR_CUDA;
        }
        if (d.scale_format != SRFTKV_SCALE_FP32 || DV != 256) {
            Mp.scales[s] = Mp.codes[s][0];  // read by plain bulk copies (no tensor map)
        } else {
            const unsigned long long sdims[3] = {(unsigned long long)ng, tcap, nrow};
            const unsigned long long sstr[2] = {ng * 4ull, tcap * ng * 4ull};
            const unsigned sbox[3] = {(unsigned)ng, (unsigned)wide::M, 1u};
            if (!encode_tiled_swz(&Mp.scales[s], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, d.scales, sdims, sstr, sbox,
                                  swz(4 * ng), "wide tensor-core dequantize scales"))
                return SRFTKV_ERR_CUDA;
        }
    }
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(srft_dequantize_tc_wide_kernel<BK, BV, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
        attr = true;
    }
    int blocks = device_sm_count();
    if (blocks > P.total_tiles) blocks = P.total_tiles;
    srft_dequantize_tc_wide_kernel<BK, BV, DV><<<blocks, wide::DQ_WARPS * 32, C::SMEM, c.stream>>>(Mp, P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("wide tensor-core dequantize launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return SRFTKV_OK;
}

// The wide tensor-core dequantize for one head dimension: 1 when the call does not fit it (a side with
// lambda, groups above 32, or scale rows that are not whole 16-byte rows of the plane).
template <int DV>
int codec_dequantize_tc_wide_d(const CodecCall& c) {
    if (c.group > 32) return 1;
    for (int s = 0; s < c.n_sides; ++s) {
        if (c.side[s].lambda) return 1;
        const long long rb = (long long)(DV / c.group) * scale_bytes(c.side[s].scale_format);
        if ((c.side[s].scale_format != SRFTKV_SCALE_FP32 || DV != 256) &&
            (((long long)c.t_cap * rb) % 16 || ((long long)c.t_offset * rb) % 16))
            return 1;
    }
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    if (bk == 4 && bv == 4) return launch_dq_tc_wide<4, 4, DV>(c);
    if (bk == 8 && bv == 8) return launch_dq_tc_wide<8, 8, DV>(c);
    if (bk == 8 && bv == 4) return launch_dq_tc_wide<8, 4, DV>(c);
    return launch_dq_tc_wide<4, 8, DV>(c);
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
