// codec_tc.cu -- SRFT quantize and dequantize with the transform done as a
// dense contraction on the 5th-generation tensor cores (head dimension 128,
// and 96 inside the same 128-wide tiles with R zero outside its 96 x 96 block).
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
//   warps 2-17 epilogue: each reads 32 rows x 32 columns of an accumulator
//              (warp w may only touch tensor-memory lanes 32(w%4)..+31),
//              applies lambda, quantises its two 16-coordinate groups and
//              stores codes and scales straight from registers.  The
//              quantisation is a chain of dependent steps per row (absmax,
//              reciprocal, rounding, packing); sixteen warps with short rows
//              keep enough of them in flight to match the load rate.
// R_hi / R_lo are built once per CTA in shared memory from the twiddle table
// (entries of R are closed forms of cos and sin of 2 pi jk/d).
#include <type_traits>

#include "codec_impl.cuh"
#include "codec_tc_common.cuh"
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
constexpr int T_SMEM = T_OFF_BAR + 256 + 1024;  // + barriers + alignment slack
constexpr int T_EPI = 16;                     // epilogue warps of the quantize kernel
constexpr int T_WARPS = 2 + T_EPI;
constexpr int T_NACC = 4;                     // fp32 accumulators of 128 columns in tensor memory
constexpr uint32_t T_TMEM_COLS = 128 * T_NACC;
}  // namespace

__device__ __forceinline__ TileId decode_tile128(const CodecParams& P, int t) { return decode_tile<TM>(P, t); }

// Entry (n, k) of the forward transform R for head dimension dv <= 128 (p = R x,
// n the packed output coordinate, k the input coordinate), before the sign of
// input k; zero outside dv x dv, so a smaller head dimension runs as the
// 128-wide contraction padded with zeros.  dv = 128 takes the compile-time
// twiddle table; other (even) dv take cs[m], sn[m] = cos, sin(2 pi m / dv),
// tabulated once per CTA (in double, rounded to float) by r_tables.
__device__ float r_entry(int n, int k, int dv, bool srht, const float* __restrict__ cs, const float* __restrict__ sn) {
    if (n >= dv || k >= dv) return 0.f;
    if (dv == TD) {
        constexpr float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)
        constexpr float c2 = 0.125f;                        // sqrt(2/128)
        if (srht) return (__popc(n & k) & 1) ? -inv_sqrt_d : inv_sqrt_d;  // Hadamard entry / sqrt(d)
        if (n == 0) return inv_sqrt_d;
        if (n == 1) return (k & 1) ? -inv_sqrt_d : inv_sqrt_d;
        const int m = (((n >> 1) * k) & (TD - 1)) * (256 / TD);  // angle 2 pi (jk mod d)/d on the 256-point table
        return (n & 1) ? c2 * tw_im_lane(m) : c2 * tw_re_lane(m);   // the imaginary part holds -sin
    }
    const float isd = (float)(1.0 / sqrt((double)dv)), r2 = (float)sqrt(2.0 / dv);
    if (n == 0) return isd;
    if (n == 1) return (k & 1) ? -isd : isd;
    const int m = ((n >> 1) * k) % dv;
    return (n & 1) ? -r2 * sn[m] : r2 * cs[m];
}

// cos, sin (2 pi m / dv) for m < dv into cs, sn (shared memory not yet in use);
// the caller synchronises the block before r_entry reads them.  A table of dv
// entries instead of an angle per entry of R: 16 K double-precision sincos per
// CTA had cost about 80 us a launch (FP64 is slow on this GPU).
__device__ __forceinline__ void r_tables(int dv, float* cs, float* sn) {
    for (int m = threadIdx.x; m < dv; m += blockDim.x) {
        double sv, cv;
        sincospi(2.0 * m / dv, &sv, &cv);
        cs[m] = (float)cv;
        sn[m] = (float)sv;
    }
}

// Byte offset of element (row n, column k) of a 128 x 128 fp16 operand stored
// K-major in two 128-byte-swizzled k-blocks (the layout TMA's 128-byte swizzle
// produces and the MMA descriptors below describe).
__device__ __forceinline__ uint32_t sw128_offset(int n, int k) {
    return (uint32_t)((k >> 6) * T_KB_BYTES + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + ((k & 7) << 1));
}

// SF: the scale format of both sides (mixed calls are split on the host);
// DV: the head dimension, 128 or a smaller one padded to the 128-wide tile
template <int BK, int BV, int SF, int DV>
__global__ void __launch_bounds__(T_WARPS * 32, 1)
    srft_quantize_tc_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                            const __grid_constant__ CodecParams P) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, and still a __shared__ pointer so accesses compile to shared-memory instructions
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T_OFF_BAR);
    // barriers: x stage full / empty, accumulator full / empty; tensor-memory slot after them
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    constexpr int X_FULL = 0, X_EMPTY = TSTAGES, ACC_FULL = 2 * TSTAGES, ACC_EMPTY = 2 * TSTAGES + T_NACC;
    static_assert((2 * TSTAGES + 2 * T_NACC) * 8 + 4 <= 256, "barrier area");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[2 * TSTAGES + 2 * T_NACC]);

    // ---- R_s = R diag(s), split into fp16 hi + lo, in the MMA operand layout ----
    // (both sides of a launch share the transform; mixed calls are split on the host)
    {
        const bool srht = P.side[0].transform == SRFTKV_TRANSFORM_SRHT;
        // angle tables (d < 128) in the x stages, which no copy has reached yet
        float* cs = reinterpret_cast<float*>(smem + T_OFF_A);
        float* sn = cs + TD;
        uint32_t* smask = reinterpret_cast<uint32_t*>(sn + TD);
        stage_sign_mask(smask, P.sign_mask, TD / 2);
        if constexpr (DV != TD) r_tables(DV, cs, sn);
        __syncthreads();
        // one 16-byte chunk (8 consecutive k of row n) of R_hi and of R_lo a step
        for (int c = threadIdx.x; c < TD * TD / 8; c += blockDim.x) {
            const int n = c >> 4, k0 = (c & 15) << 3;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = k0 + 2 * j;
                float v0 = r_entry(n, k, DV, srht, cs, sn), v1 = r_entry(n, k + 1, DV, srht, cs, sn);
                if (sign_flip(smask, k)) v0 = -v0;
                if (sign_flip(smask, k + 1)) v1 = -v1;
                split_pair_h2(v0, v1, hi[j], lo[j]);
            }
            const uint32_t off = sw128_offset(n, k0);
            *reinterpret_cast<uint4*>(smem + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(smem + T_OFF_BLO + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        ptx::fence_proxy_async_smem();  // generic writes -> tensor-core (async proxy) reads
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < TSTAGES; ++s) {
            ptx::mbar_init(bar(X_FULL + s), 1);
            ptx::mbar_init(bar(X_EMPTY + s), 1);
        }
        for (int a = 0; a < T_NACC; ++a) {
            ptx::mbar_init(bar(ACC_FULL + a), 1);
            ptx::mbar_init(bar(ACC_EMPTY + a), 4 * ((DV + 31) / 32));  // one arrival per (lane quarter, column quarter)
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
                if (use > 0 && !ptx::mbar_wait_bounded(bar(X_EMPTY + s), (use - 1) & 1)) {
                    failed = true;
                    break;
                }
                const TileId id = decode_tile128(P, t);
                const CUtensorMap* tm = id.side ? &tm1 : &tm0;
                const uint32_t dst = sbase + T_OFF_A + s * T_A_BYTES;
                ptx::mbar_arrive_expect_tx(bar(X_FULL + s), T_A_BYTES);
                ptx::tma_load_4d(dst, tm, bar(X_FULL + s), 0, id.h, id.t0, id.o);
                ptx::tma_load_4d(dst + T_KB_BYTES, tm, bar(X_FULL + s), 64, id.h, id.t0, id.o);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int t = blockIdx.x, i = 0; t < P.total_tiles; t += stride, ++i) {
                const int s = i % TSTAGES, a = i % T_NACC;
                // (P.poll_limit: the default bound, or fewer polls from the test hook; if this wait gives up
                // before any MMA was issued, no MMA is ever in flight when tensor memory is freed, and the
                // producer's copies land while the other roles' waits run out)
                if (!ptx::mbar_wait_bounded(bar(X_FULL + s), (i / TSTAGES) & 1, P.poll_limit) ||
                    (i >= T_NACC && !ptx::mbar_wait_bounded(bar(ACC_EMPTY + a), (i / T_NACC - 1) & 1))) {
                    failed = true;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem + a * TD;
                const uint32_t a_base = sbase + T_OFF_A + s * T_A_BYTES;
                // d < 128: K and N stop at d (the padding columns of x and rows of R_s are zero)
                constexpr uint32_t IDESC = tc::idesc_f16_f32(TM, DV);
#pragma unroll
                for (int ks = 0; ks < DV / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * T_KB_BYTES + (ks & 3) * 32;
                    const uint64_t ad = tc::sw128_desc(a_base + koff);
                    tc::mma_f16(d_tmem, ad, tc::sw128_desc(sbase + koff), IDESC, ks > 0);
                    tc::mma_f16(d_tmem, ad, tc::sw128_desc(sbase + T_OFF_BLO + koff), IDESC, 1);
                }
                tc::commit(bar(X_EMPTY + s));  // the x stage can be refilled once these MMAs are done
                tc::commit(bar(ACC_FULL + a));  // accumulator a is ready for the epilogue
            }
        }
    } else {
        // Work units: (lane quarter, 32-column quarter) of a tile; a warp may
        // only read tensor-memory lanes 32(w%4)..+31.  unit(): wait for
        // accumulator a, read the unit's 32 x 32 block, release the
        // accumulator, then lambda, quantise and store the 32 rows.
        const int quarter = warp & 3;
        auto unit = [&](int t, int a, int cq, uint32_t parity) -> bool {
            const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar(ACC_FULL + a), parity));
            if (!ok) return false;
            tc::fence_after_sync();
            uint32_t r0[32];
            const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16) + a * TD + cq * 32;
            tc::ld_32x32b_x32(taddr, r0);
            tc::wait_ld(r0);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ACC_EMPTY + a));  // accumulator a may be overwritten

            const TileId id = decode_tile128(P, t);
            const CodecSideK& S = P.side[id.side];
            const int t_tok = id.t0 + 32 * quarter + lane;
            if (t_tok >= P.n_tokens) return true;
            const long long vrow = packed_row(P, id, t_tok);
            const int ng = DV >> P.lg_group;
            // the unit's columns 32 cq .. +W-1 (W = 32, or 16 for the last quarter at d = 80); at d = 80 the
            // code rows (40 or 80 bytes) and scale rows (5 scales) allow only narrow stores
            auto finish = [&](auto wc) {
                constexpr int W = decltype(wc)::value;
                constexpr bool NARROW = DV == 80;
                float z[W];
#pragma unroll
                for (int j = 0; j < W; ++j) z[j] = __uint_as_float(r0[j]);
                if (S.lambda != nullptr) {
                    const float4* lr = reinterpret_cast<const float4*>(
                        S.lambda + (long long)id.o * S.lambda_outer_stride + (long long)id.h * DV + cq * 32);
#pragma unroll
                    for (int c = 0; c < W / 4; ++c) {
                        const float4 l = __ldg(lr + c);
                        z[4 * c] *= l.x;
                        z[4 * c + 1] *= l.y;
                        z[4 * c + 2] *= l.z;
                        z[4 * c + 3] *= l.w;
                    }
                }
                uint8_t* srow = S.scales + (vrow * ng + ((32 * cq) >> P.lg_group)) * S.sbytes;
                if (BK == BV || id.side == 0)
                    quant_store_row<W, BK, SF, 0, NARROW>(z, P.group, S.codes + vrow * (DV * BK / 8) + cq * (32 * BK / 8),
                                                          srow);
                else
                    quant_store_row<W, BV, SF, 0, NARROW>(z, P.group, S.codes + vrow * (DV * BV / 8) + cq * (32 * BV / 8),
                                                          srow);
            };
            if constexpr (DV % 32 != 0) {
                if (cq == DV / 32) finish(std::integral_constant<int, DV % 32>{});
                else finish(std::integral_constant<int, 32>{});
            } else {
                finish(std::integral_constant<int, 32>{});
            }
            return true;
        };
        if constexpr (DV == TD) {
            // warp w: the same column quarter (w-2)/4 of every tile
            const int cq = (warp - 2) >> 2;
            for (int t = blockIdx.x, i = 0; t < P.total_tiles; t += stride, ++i)
                if (!unit(t, i % T_NACC, cq, (i / T_NACC) & 1)) {
                    failed = true;
                    break;
                }
        } else {
            // NQ = DV/32 column quarters, 4 NQ units a tile, 16 NQ for the
            // T_NACC = 4 tiles of one round of the accumulators: each of the 16
            // warps takes NQ of them, units x, x+16, x+32, ... in tile order (x
            // keeps the warp's lane quarter: unit u's is u % 4), so at d = 96
            // the 12 units of a tile spread over all 16 warps.
            static_assert(T_NACC == 4 && T_EPI == 16, "units per warp and round");
            constexpr int NQ = (DV + 31) / 32, U = 4 * NQ;  // the last quarter is 16 columns wide at d = 80
            const int x = ((warp - 2) & ~3) | quarter;
            for (int r = 0; blockIdx.x + T_NACC * r * stride < P.total_tiles && !failed; ++r)
#pragma unroll 1
                for (int uj = 0; uj < NQ; ++uj) {
                    const int u = x + 16 * uj, tr = u / U;
                    const int t = blockIdx.x + (T_NACC * r + tr) * stride;
                    if (t >= P.total_tiles) break;  // later units belong to later tiles
                    if (!unit(t, tr, (u % U) >> 2, r & 1)) {
                        failed = true;
                        break;
                    }
                }
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
// Warp roles (one persistent CTA per SM, 18 warps):
//   warp 0      allocates tensor memory and issues the MMAs (one thread);
//   warp 1      TMA producer: the tile's code rows and scale rows, copied as
//               exact rows (TMA swizzle equal to the row length keeps the
//               row-per-thread reads free of bank conflicts), into a ring of
//               input stages;
//   warps 2-9   converters: thread = half a row of the tile; decode codes *
//               scale, write P_hat as fp16 straight into
//               tensor memory (the MMA takes A from there: no shared-memory
//               round trip, which with the B reads would otherwise exceed the
//               SM's shared-memory bandwidth);
//   warps 10-17 epilogue: tensor memory -> fp16 -> swizzled staging -> TMA
//               store (warp w reads tensor-memory lanes 32(w%4)..+31, one
//               column half; at d = 96 the six-word halves of d96_word).
// Converting is a dependent chain per row; eight warps on half rows keep
// enough of them in flight to match the load rate.
// 1/lambda scales the contraction's K index (the packed coordinate), so it is
// folded into B: B[k][q] = R_s[k][q] / lambda_n(q), rebuilt (by the MMA warp,
// from an fp32 copy of R_s, once the MMAs that read B have completed)
// whenever the tile's lambda row changes.  With lambda a CTA takes a
// contiguous range of tiles, so a rebuild comes once per (side, outer, head)
// run rather than per tile, and the converters keep the code-pair path.
// B = diag(s) R (signs folded in), so X_hat = s (R^T P_hat).  P_hat is
// rounded once to fp16 before the contraction and the result is rounded to
// fp16 again on output; R_s in fp16 (11 bits) matches that precision, so
// unlike the quantize kernel (whose rounding decisions need R to about 21
// bits, hence hi + lo) one contraction per tile suffices.
namespace {
constexpr int DQ_CONV = 8, DQ_EPI = 8;                // converter and epilogue warps
constexpr int DQ_WARPS = 2 + DQ_CONV + DQ_EPI;
constexpr int DQ_OFF_O = T_B_BYTES;                     // two output staging buffers of 32 KB (after R_s)
constexpr int DQ_OFF_IN = DQ_OFF_O + 2 * T_A_BYTES;     // input stages
constexpr int DQ_NA = 3;                                // A buffers in tensor memory
constexpr uint32_t DQ_TMEM_COLS = 512;                  // accumulators 0..255, A buffers 256..447
constexpr uint32_t DQ_A_COL = 256;                      // A buffer b: 64 columns (128 fp16 per lane) at 256 + 64 b
template <int BK, int BV>
struct DqCfg {
    static constexpr int RBMAX = TD * (BK > BV ? BK : BV) / 8;     // exact code rows (64 or 128 bytes)
    static constexpr int OFF_SC = TM * RBMAX;                       // 1024-aligned
    static constexpr int STAGE = (OFF_SC + TM * 32 + 1023) / 1024 * 1024;  // scale rows of at most 32 bytes
    static constexpr int STAGES = (BK == 4 && BV == 4) ? 4 : 3;
    static constexpr int OFF_BASE = DQ_OFF_IN + STAGES * STAGE;  // R_s in fp32, [k][q] rows of 128 (64 KB)
    static constexpr int OFF_IL = OFF_BASE + TD * TD * 4;        // 1/lambda of the current run, 128 floats
    static constexpr int OFF_BAR = OFF_IL + TD * 4;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
};
}  // namespace

// The four 16-column unit scales of columns 64 hf .. +63 of tile row m, from
// the stage in shared memory: fp32 planes as exact swizzled rows (32 bytes
// for group 16, 16 for group 32), fp16 / e8m0 planes as their contiguous
// bytes (rows of 4 to 16 bytes, unswizzled).
__device__ __forceinline__ void half_row_scales(const uint8_t* __restrict__ in, int off_sc, int m, int hf, int group,
                                                int sfmt, float (&sc)[4]) {
    if (sfmt == SRFTKV_SCALE_FP32) {
        const int srb = 4 * (TD >> (__ffs(group) - 1));  // group: a power of two (a shift, not a division)
        if (group == 16) {  // groups 4hf .. 4hf+3: chunk hf of the 32-byte row
            const float4 v = *reinterpret_cast<const float4*>(in + off_sc + m * srb + (swz16(srb, m, hf) << 4));
            sc[0] = v.x;
            sc[1] = v.y;
            sc[2] = v.z;
            sc[3] = v.w;
        } else {  // group 32: groups 2hf, 2hf+1 of the 16-byte row
            const float2 v = *reinterpret_cast<const float2*>(in + off_sc + m * srb + 8 * hf);
            sc[0] = sc[1] = v.x;
            sc[2] = sc[3] = v.y;
        }
        return;
    }
    const uint8_t* row = in + off_sc + m * (TD >> (__ffs(group) - 1)) * (sfmt == SRFTKV_SCALE_FP16 ? 2 : 1);
    if (sfmt == SRFTKV_SCALE_FP16) {
        if (group == 16) {
            const uint2 h = *reinterpret_cast<const uint2*>(row + 8 * hf);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
            sc[0] = a.x;
            sc[1] = a.y;
            sc[2] = b.x;
            sc[3] = b.y;
        } else {
            const uint32_t h = *reinterpret_cast<const uint32_t*>(row + 4 * hf);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h));
            sc[0] = sc[1] = a.x;
            sc[2] = sc[3] = a.y;
        }
    } else {  // e8m0: the byte is the fp32 exponent field
        if (group == 16) {
            const uint32_t e = *reinterpret_cast<const uint32_t*>(row + 4 * hf);
            sc[0] = __uint_as_float((e & 0xFFu) << 23);
            sc[1] = __uint_as_float(((e >> 8) & 0xFFu) << 23);
            sc[2] = __uint_as_float(((e >> 16) & 0xFFu) << 23);
            sc[3] = __uint_as_float((e >> 24) << 23);
        } else {
            const uint32_t e = *reinterpret_cast<const unsigned short*>(row + 2 * hf);
            sc[0] = sc[1] = __uint_as_float((e & 0xFFu) << 23);
            sc[2] = sc[3] = __uint_as_float((e >> 8) << 23);
        }
    }
}

// The 16-byte code chunks of half hf of tile row m (swizzled rows of 128*BITS/8 bytes)
template <int BITS, int NCH>
__device__ __forceinline__ void load_half_codes(const uint8_t* __restrict__ in, int m, int hf, uint32_t (&w)[4 * NCH]) {
    constexpr int RB = TD * BITS / 8;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int c = NCH * hf + k;
        const uint4 v = *reinterpret_cast<const uint4*>(in + m * RB + (swz16(RB, m, c) << 4));
        w[4 * k] = v.x;
        w[4 * k + 1] = v.y;
        w[4 * k + 2] = v.z;
        w[4 * k + 3] = v.w;
    }
}

// P_hat for columns 64 hf .. +63 of tile row m directly as fp16 pairs in the
// K order of dq_kperm (no lambda): codes -> exact fp16 pairs -> times the
// group scale split into fp16 hi + lo, P_hat = fp16(q s_hi + fp16(q s_lo)), one
// main rounding as when the fp32 product q s is rounded to fp16.
template <int BITS>
__device__ __forceinline__ void dequant_half_pairs(const uint8_t* __restrict__ in, int m, int hf, const float (&sc)[4],
                                                   uint32_t (&hp)[32]) {
    constexpr int NCH = 64 * BITS / 128;
    uint32_t w[4 * NCH];
    load_half_codes<BITS, NCH>(in, m, hf, w);
    uint32_t sh[4], sl[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const __half h = __float2half_rn(sc[g]);
        sh[g] = half2_bcast(h);
        sl[g] = half2_bcast(__float2half_rn(sc[g] - __half2float(h)));
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // 8-element word k of the half: coordinates 64 hf + 8k .. +7, group k/2
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
        for (int j = 0; j < 4; ++j) hp[4 * k + j] = h2fma(c[j], sh[k >> 1], h2mul(c[j], sl[k >> 1]));
    }
}

// d = 96: the two halves of a row are six 8-coordinate words each, words
// 4h..4h+3 (coordinates 32h..32h+31) and 8+2h, 9+2h (coordinates 64+16h..+15)
// for half h, so both do equal work and every tensor-memory access stays
// naturally aligned: A columns 16h..+15 and 32+8h..+7 (column c holds word
// c/4), accumulator columns 32h..+31 and 64+16h..+15 (one per coordinate).
__device__ __forceinline__ int d96_word(int hf, int k) { return k < 4 ? 4 * hf + k : 8 + 2 * hf + (k - 4); }

// The code words of half hf of tile row m (48- or 96-byte unswizzled rows):
// int4 word k is w[k], int8 word k is w[2k], w[2k+1].
template <int BITS>
__device__ __forceinline__ void d96_half_words(const uint8_t* __restrict__ in, int m, int hf,
                                               uint32_t (&w)[6 * BITS / 4]) {
    const uint8_t* row = in + m * (96 * BITS / 8);
    if constexpr (BITS == 4) {
        const uint4 a = *reinterpret_cast<const uint4*>(row + 16 * hf);
        const uint2 c = *reinterpret_cast<const uint2*>(row + 32 + 8 * hf);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = c.x; w[5] = c.y;
    } else {
        const uint4 a = *reinterpret_cast<const uint4*>(row + 32 * hf);
        const uint4 b = *reinterpret_cast<const uint4*>(row + 32 * hf + 16);
        const uint4 c = *reinterpret_cast<const uint4*>(row + 64 + 16 * hf);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        w[8] = c.x; w[9] = c.y; w[10] = c.z; w[11] = c.w;
    }
}

// The scales of half hf's three 16-coordinate units 2hf, 2hf+1, 4+hf (flat rows of 96/group scales)
__device__ __forceinline__ void d96_half_scales(const uint8_t* __restrict__ in, int off_sc, int m, int hf, int group,
                                                int sfmt, float (&sc)[3]) {
    const int lg = __ffs(group) - 1;  // group: a power of two
    const int ng = 96 >> lg, sb = sfmt == SRFTKV_SCALE_FP32 ? 4 : sfmt == SRFTKV_SCALE_FP16 ? 2 : 1;
    const uint8_t* row = in + off_sc + m * ng * sb;
    const int units[3] = {2 * hf, 2 * hf + 1, 4 + hf};
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const int gi = (16 * units[u]) >> lg;
        if (sfmt == SRFTKV_SCALE_FP32) sc[u] = *reinterpret_cast<const float*>(row + 4 * gi);
        else if (sfmt == SRFTKV_SCALE_FP16) sc[u] = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(row + 2 * gi)));
        else sc[u] = __uint_as_float((uint32_t)row[gi] << 23);
    }
}

// fp16 pairs (coordinates 8w+j, 8w+j+4; j = 0..3) of half hf of a d = 96 row,
// codes * scale with the scale split into fp16 hi + lo, in the order of the A columns
template <int BITS>
__device__ __forceinline__ void d96_half_pairs(const uint8_t* __restrict__ in, int off_sc, int m, int hf, int group,
                                               int sfmt, uint32_t (&hp)[24]) {
    uint32_t w[6 * BITS / 4];
    d96_half_words<BITS>(in, m, hf, w);
    float sc[3];
    d96_half_scales(in, off_sc, m, hf, group, sfmt, sc);
    uint32_t sh[3], sl[3];
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const __half h = __float2half_rn(sc[u]);
        sh[u] = half2_bcast(h);
        sl[u] = half2_bcast(__float2half_rn(sc[u] - __half2float(h)));
    }
#pragma unroll
    for (int k = 0; k < 6; ++k) {
        const int u = k < 4 ? k >> 1 : 2;
        uint32_t c[4];
        if constexpr (BITS == 4) {
            const uint32_t x = w[k], xs = x >> 8;
            c[0] = codes_lo4(x);
            c[1] = codes_hi4(x);
            c[2] = codes_lo4(xs);
            c[3] = codes_hi4(xs);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                c[j] = codes_b8(__byte_perm(w[2 * k], w[2 * k + 1], j | (j << 4) | ((4 + j) << 8) | ((4 + j) << 12)));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) hp[4 * k + j] = h2fma(c[j], sh[u], h2mul(c[j], sl[u]));
    }
}

// d = 80: ten 8-coordinate words a row, five a half: words 4h..4h+3
// (coordinates 32h..32h+31, A columns 16h..+15) and 8+h (coordinates
// 64+8h..+7, A columns 32+4h..+3), so both halves do equal work and each
// tensor-memory store (16 + 4 columns) is aligned to its width.  Rows are
// 40 (int4) or 80 (int8) bytes, copied flat, so only 8-byte alignment holds.
template <int BITS>
__device__ __forceinline__ void d80_half_words(const uint8_t* __restrict__ in, int m, int hf,
                                               uint32_t (&w)[5 * BITS / 4]) {
    const uint8_t* row = in + m * (80 * BITS / 8);
    if constexpr (BITS == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(row + 16 * hf);
        const uint2 b = *reinterpret_cast<const uint2*>(row + 16 * hf + 8);
        w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y;
        w[4] = *reinterpret_cast<const uint32_t*>(row + 32 + 4 * hf);
    } else {
        const uint4 a = *reinterpret_cast<const uint4*>(row + 32 * hf);
        const uint4 b = *reinterpret_cast<const uint4*>(row + 32 * hf + 16);
        const uint2 c = *reinterpret_cast<const uint2*>(row + 64 + 8 * hf);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        w[8] = c.x; w[9] = c.y;
    }
}

// fp16 pairs of half hf of a d = 80 row (units 2hf, 2hf+1 and 4; groups of 16), codes * scale with the
// scale split into fp16 hi + lo, in the order of the A columns
template <int BITS>
__device__ __forceinline__ void d80_half_pairs(const uint8_t* __restrict__ in, int off_sc, int m, int hf, int sfmt,
                                               uint32_t (&hp)[20]) {
    uint32_t w[5 * BITS / 4];
    d80_half_words<BITS>(in, m, hf, w);
    const int sb = sfmt == SRFTKV_SCALE_FP32 ? 4 : sfmt == SRFTKV_SCALE_FP16 ? 2 : 1;
    const uint8_t* srow = in + off_sc + m * 5 * sb;
    const int units[3] = {2 * hf, 2 * hf + 1, 4};
    uint32_t sh[3], sl[3];
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const int gi = units[u];
        float sc;
        if (sfmt == SRFTKV_SCALE_FP32) sc = *reinterpret_cast<const float*>(srow + 4 * gi);
        else if (sfmt == SRFTKV_SCALE_FP16) sc = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(srow + 2 * gi)));
        else sc = __uint_as_float((uint32_t)srow[gi] << 23);
        const __half h = __float2half_rn(sc);
        sh[u] = half2_bcast(h);
        sl[u] = half2_bcast(__float2half_rn(sc - __half2float(h)));
    }
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int u = k < 4 ? k >> 1 : 2;
        uint32_t c[4];
        if constexpr (BITS == 4) {
            const uint32_t x = w[k], xs = x >> 8;
            c[0] = codes_lo4(x);
            c[1] = codes_hi4(x);
            c[2] = codes_lo4(xs);
            c[3] = codes_hi4(xs);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                c[j] = codes_b8(__byte_perm(w[2 * k], w[2 * k + 1], j | (j << 4) | ((4 + j) << 8) | ((4 + j) << 12)));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) hp[4 * k + j] = h2fma(c[j], sh[u], h2mul(c[j], sl[u]));
    }
}

struct DqMaps {
    CUtensorMap out[2], codes[2], scales[2];
};

template <int BK, int BV, int DV>  // DV: head dimension, 128 or a smaller one padded to the 128-wide tile
__global__ void __launch_bounds__(DQ_WARPS * 32, 1)
    srft_dequantize_tc_kernel(const __grid_constant__ DqMaps M, const __grid_constant__ CodecParams P) {
    using C = DqCfg<BK, BV>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, and still a __shared__ pointer so accesses compile to shared-memory instructions
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    // a_full[0..2], a_empty[3..5], acc_full[6,7], acc_empty[8,9], in_full[10..13], in_empty[14..17],
    // b_free at 18; tensor-memory slot at 19
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    constexpr int A_FULL = 0, A_EMPTY = 3, ACC_FULL = 6, ACC_EMPTY = 8, IN_FULL = 10, IN_EMPTY = 14, B_FREE = 18;
    static_assert(C::STAGES <= 4, "input stages");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[19]);
    float* rbase = reinterpret_cast<float*>(smem + C::OFF_BASE);
    static_assert(C::OFF_BASE % 16 == 0, "the fp32 copy of R_s is written as float4");

    {  // B[k][q] = s_k R[n][k] with n = dq_kperm(q) (zero outside d x d), in fp16; and in fp32 for the rebuilds
        const bool srht = P.side[0].transform == SRFTKV_TRANSFORM_SRHT;
        // angle tables (d < 128) in the output staging buffers, which no epilogue has reached yet
        float* cs = reinterpret_cast<float*>(smem + DQ_OFF_O);
        float* sn = cs + TD;
        uint32_t* smask = reinterpret_cast<uint32_t*>(sn + TD);
        stage_sign_mask(smask, P.sign_mask, TD / 2);
        if constexpr (DV != TD) r_tables(DV, cs, sn);
        __syncthreads();
        // one 16-byte chunk a step: B row k (output coordinate), K positions q0 .. q0+7 holding packed
        // coordinates dq_kperm(q)
        for (int c = threadIdx.x; c < TD * TD / 8; c += blockDim.x) {
            const int k = c >> 4, q0 = (c & 15) << 3;
            const bool flip = sign_flip(smask, k);
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[j] = r_entry(dq_kperm(q0 + j), k, DV, srht, cs, sn);
                if (flip) v[j] = -v[j];
            }
            float4* rb = reinterpret_cast<float4*>(rbase + k * TD + q0);
            rb[0] = make_float4(v[0], v[1], v[2], v[3]);
            rb[1] = make_float4(v[4], v[5], v[6], v[7]);
            *reinterpret_cast<uint4*>(smem + sw128_offset(k, q0)) =
                make_uint4(pack_half2(v[0], v[1]), pack_half2(v[2], v[3]), pack_half2(v[4], v[5]), pack_half2(v[6], v[7]));
        }
        ptx::fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        for (int b = 0; b < DQ_NA; ++b) {
            ptx::mbar_init(bar(A_FULL + b), DQ_CONV);
            ptx::mbar_init(bar(A_EMPTY + b), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(bar(ACC_FULL + a), 1);
            ptx::mbar_init(bar(ACC_EMPTY + a), DQ_EPI);
        }
        for (int st = 0; st < C::STAGES; ++st) {
            ptx::mbar_init(bar(IN_FULL + st), 1);
            ptx::mbar_init(bar(IN_EMPTY + st), DQ_CONV);
        }
        ptx::mbar_init(bar(B_FREE), 1);
        ptx::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(ptx::smem_u32(tmem_slot), DQ_TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // this CTA's tiles: a contiguous range when a side has lambda (runs of one lambda row), else round-robin
    const bool contig = P.side[0].lambda != nullptr || P.side[1].lambda != nullptr;
    const int per = (P.total_tiles + gridDim.x - 1) / gridDim.x;
    const int first = contig ? blockIdx.x * per : blockIdx.x, step = contig ? 1 : gridDim.x;
    const int count = contig ? max(0, min(per, P.total_tiles - first))
                             : (P.total_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    bool failed = false;

    if (warp == 0) {
        const float* cur = nullptr;  // the lambda row B is divided by (nullptr: none)
        uint32_t bfree_parity = 0;
        for (int i = 0; i < count; ++i) {
            const int t = first + i * step;
            const TileId id = decode_tile128(P, t);
            const CodecSideK& S = P.side[id.side];
            const float* key = S.lambda == nullptr
                                   ? nullptr
                                   : S.lambda + (long long)id.o * S.lambda_outer_stride + (long long)id.h * DV;
            if (key != cur) {
                // the MMAs issued so far read B: wait for them, then rebuild B = R_s / lambda from the fp32 copy
                bool ok = true;
                if (lane == 0) {
                    tc::commit(bar(B_FREE));
                    ok = ptx::mbar_wait_bounded(bar(B_FREE), bfree_parity);
                }
                bfree_parity ^= 1u;
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                    failed = true;
                    break;
                }
                tc::fence_after_sync();
                float* il = reinterpret_cast<float*>(smem + C::OFF_IL);
                for (int c = lane; c < TD; c += 32) il[c] = (key != nullptr && c < DV) ? __frcp_rn(__ldg(key + c)) : 1.f;
                __syncwarp();
                for (int j = lane; j < TD * TD / 8; j += 32) {  // row k, K positions 8c .. 8c+7
                    const int k = j >> 4, q0 = (j & 15) * 8;
                    const float4 lo = *reinterpret_cast<const float4*>(rbase + k * TD + q0);
                    const float4 hi = *reinterpret_cast<const float4*>(rbase + k * TD + q0 + 4);
                    const float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    uint32_t h[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        h[e] = pack_half2(v[2 * e] * il[dq_kperm(q0 + 2 * e)], v[2 * e + 1] * il[dq_kperm(q0 + 2 * e + 1)]);
                    *reinterpret_cast<uint4*>(smem + sw128_offset(k, q0)) = make_uint4(h[0], h[1], h[2], h[3]);
                }
                ptx::fence_proxy_async_smem();  // generic writes -> tensor-core reads
                __syncwarp();
                cur = key;
            }
            bool ok = true;
            if (lane == 0) {
                const int s = i & 1, b = i % DQ_NA;
                ok = ptx::mbar_wait_bounded(bar(A_FULL + b), (i / DQ_NA) & 1) &&
                     (i < 2 || ptx::mbar_wait_bounded(bar(ACC_EMPTY + s), ((i >> 1) - 1) & 1));
                if (ok) {
                    tc::fence_after_sync();
                    const uint32_t d_tmem = tmem + s * TD;
                    const uint32_t a_tmem = tmem + DQ_A_COL + b * 64;
                    // d < 128: K and N stop at d (accumulator columns past d are never stored)
                    constexpr uint32_t IDESC = tc::idesc_f16_f32(TM, DV);
#pragma unroll
                    for (int ks = 0; ks < DV / 16; ++ks) {
                        const uint32_t koff = (ks >> 2) * T_KB_BYTES + (ks & 3) * 32;
                        tc::mma_f16_ta(d_tmem, a_tmem + 8 * ks, tc::sw128_desc(sbase + koff), IDESC, ks > 0);
                    }
                    tc::commit(bar(A_EMPTY + b));  // A buffer b may be rewritten
                    tc::commit(bar(ACC_FULL + s));  // accumulator s is ready
                }
            }
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                failed = true;
                break;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int i = 0; i < count; ++i) {
                const int t = first + i * step;
                const int st = i % C::STAGES, use = i / C::STAGES;
                if (use > 0 && !ptx::mbar_wait_bounded(bar(IN_EMPTY + st), (use - 1) & 1)) {
                    failed = true;
                    break;
                }
                const TileId id = decode_tile128(P, t);
                const int bits = (BK == BV || id.side == 0) ? BK : BV;
                const uint32_t dst = sbase + DQ_OFF_IN + st * C::STAGE;
                const int row = P.t_offset + id.t0;   // packed planes: [outer*H][t_cap] rows
                const int oh = id.o * P.H + id.h;
                if constexpr (DV == 80) {
                    // rows of 40 / 80 code bytes and 5 scales are no TMA rows: the tile's bytes of both planes as
                    // plain bulk copies, stopping at the end of this (outer, head)
                    const CodecSideK& S = P.side[id.side];
                    const int rows = min(TM, P.t_cap - row), rb = 80 * bits / 8, srb = 5 * S.sbytes;
                    ptx::mbar_arrive_expect_tx(bar(IN_FULL + st), (uint32_t)(rows * (rb + srb)));
                    ptx::bulk_load(dst, S.codes + ((long long)oh * P.t_cap + row) * rb, (uint32_t)(rows * rb),
                                   bar(IN_FULL + st));
                    ptx::bulk_load(dst + C::OFF_SC, S.scales + ((long long)oh * P.t_cap + row) * srb,
                                   (uint32_t)(rows * srb), bar(IN_FULL + st));
                    continue;
                }
                // fp32 scales as rows of the tile; fp16 / e8m0 scales as the tile's bytes in rows of 16
                const int sb = P.side[id.side].sbytes, ng = DV >> P.lg_group, sc_bytes = TM * ng * sb;
                const bool flat = !(sb == 4 && DV == TD);  // scale rows copied as 16-byte rows of bytes
                ptx::mbar_arrive_expect_tx(bar(IN_FULL + st), TM * (DV * bits / 8) + sc_bytes);
                ptx::tma_load_3d(dst, &M.codes[id.side], bar(IN_FULL + st), 0, row, oh);
                ptx::tma_load_3d(dst + C::OFF_SC, &M.scales[id.side], bar(IN_FULL + st), 0,
                                 flat ? row * ng * sb / 16 : row, oh);
            }
        }
    } else if (warp < 2 + DQ_CONV) {
        // converter warp w: tile rows = tensor-memory lanes 32(w%4)..+31 (the
        // quarter a warp may write), column half (w-2)/4
        const int quarter = warp & 3, m = 32 * quarter + lane, hf = (warp - 2) >> 2;

        for (int i = 0; i < count; ++i) {
            const int t = first + i * step;
            const int b = i % DQ_NA, st = i % C::STAGES;
            const TileId id = decode_tile128(P, t);
            const CodecSideK& S = P.side[id.side];
            const bool ok_in = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar(IN_FULL + st), (i / C::STAGES) & 1));
            if (!ok_in) {
                failed = true;
                break;
            }
            const uint8_t* in = smem + DQ_OFF_IN + st * C::STAGE;
            uint32_t hp[32];  // fp16 pairs in the K order of dq_kperm: column 32 hf + c
            const bool side_k = BK == BV || id.side == 0;
            // lambda is folded into B: the converters take codes * scale only
            if constexpr (DV == 80) {  // d = 80: balanced halves of five words
                uint32_t (&h20)[20] = *reinterpret_cast<uint32_t(*)[20]>(hp);
                if (side_k)
                    d80_half_pairs<BK>(in, C::OFF_SC, m, hf, S.sfmt, h20);
                else
                    d80_half_pairs<BV>(in, C::OFF_SC, m, hf, S.sfmt, h20);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(IN_EMPTY + st));  // input stage consumed
                const bool ok = __all_sync(0xffffffffu,
                                           i < DQ_NA || ptx::mbar_wait_bounded(bar(A_EMPTY + b), (i / DQ_NA - 1) & 1));
                if (!ok) {
                    failed = true;
                    break;
                }
                tc::fence_after_sync();  // the MMAs that read A buffer b are complete
                const uint32_t acol = tmem + ((uint32_t)(32 * quarter) << 16) + DQ_A_COL + b * 64;
                tc::st_32x32b_x16(acol + 16 * hf, hp);
                tc::st_32x32b_x4(acol + 32 + 4 * hf, hp + 16);
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(A_FULL + b));
                continue;
            } else if constexpr (DV != TD) {  // d = 96: balanced halves of six words (d96_word)
                uint32_t (&h24)[24] = *reinterpret_cast<uint32_t(*)[24]>(hp);
                if (side_k)
                    d96_half_pairs<BK>(in, C::OFF_SC, m, hf, P.group, S.sfmt, h24);
                else
                    d96_half_pairs<BV>(in, C::OFF_SC, m, hf, P.group, S.sfmt, h24);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(IN_EMPTY + st));  // input stage consumed
                const bool ok = __all_sync(0xffffffffu,
                                           i < DQ_NA || ptx::mbar_wait_bounded(bar(A_EMPTY + b), (i / DQ_NA - 1) & 1));
                if (!ok) {
                    failed = true;
                    break;
                }
                tc::fence_after_sync();  // the MMAs that read A buffer b are complete
                const uint32_t acol = tmem + ((uint32_t)(32 * quarter) << 16) + DQ_A_COL + b * 64;
                tc::st_32x32b_x16(acol + 16 * hf, hp);
                tc::st_32x32b_x8(acol + 32 + 8 * hf, hp + 16);
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(A_FULL + b));
                continue;
            }
            float sc[4];
            half_row_scales(in, C::OFF_SC, m, hf, P.group, S.sfmt, sc);
            if (side_k)
                dequant_half_pairs<BK>(in, m, hf, sc, hp);
            else
                dequant_half_pairs<BV>(in, m, hf, sc, hp);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(IN_EMPTY + st));  // input stage consumed
            const bool ok = __all_sync(0xffffffffu,
                                       i < DQ_NA || ptx::mbar_wait_bounded(bar(A_EMPTY + b), (i / DQ_NA - 1) & 1));
            if (!ok) {
                failed = true;
                break;
            }
            tc::fence_after_sync();  // the MMAs that read A buffer b are complete
            tc::st_32x32b_x32(tmem + ((uint32_t)(32 * quarter) << 16) + DQ_A_COL + b * 64 + 32 * hf, hp);
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(A_FULL + b));
        }
    } else {
        const int quarter = warp & 3;   // tensor-memory lanes 32*quarter..+31 = tile rows
        const int m = 32 * quarter + lane, hf = (warp - 2 - DQ_CONV) >> 2;  // and column half hf
        const bool leader = (warp == 2 + DQ_CONV && lane == 0);
        for (int i = 0; i < count; ++i) {
            const int t = first + i * step;
            const int s = i & 1;
            const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar(ACC_FULL + s), (i >> 1) & 1));
            if (!ok) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
            uint32_t v[2][32];
            const uint32_t lanes = tmem + ((uint32_t)(32 * quarter) << 16) + s * TD;
            if constexpr (DV == TD) {
#pragma unroll
                for (int j = 0; j < 2; ++j) tc::ld_32x32b_x32(lanes + 64 * hf + 32 * j, v[j]);
#pragma unroll
                for (int j = 0; j < 2; ++j) tc::wait_ld(v[j]);
            } else if constexpr (DV == 80) {  // d = 80: columns 32hf..+31 and 64+8hf..+7
                uint32_t (&v8)[8] = *reinterpret_cast<uint32_t(*)[8]>(v[1]);
                tc::ld_32x32b_x32(lanes + 32 * hf, v[0]);
                tc::ld_32x32b_x8(lanes + 64 + 8 * hf, v8);
                tc::wait_ld(v[0]);
                tc::wait_ld(v8);
            } else {  // d = 96: columns 32hf..+31 and 64+16hf..+15 (d96_word)
                uint32_t (&v16)[16] = *reinterpret_cast<uint32_t(*)[16]>(v[1]);
                tc::ld_32x32b_x32(lanes + 32 * hf, v[0]);
                tc::ld_32x32b_x16(lanes + 64 + 16 * hf, v16);
                tc::wait_ld(v[0]);
                tc::wait_ld(v16);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ACC_EMPTY + s));
            // staging buffer s: the TMA store issued from it two tiles ago must have read it
            if (leader) ptx::bulk_wait_read<1>();
            ptx::named_bar_sync(1, 32 * DQ_EPI);
            uint8_t* O = smem + DQ_OFF_O + s * T_A_BYTES;
            // 8-column chunk ch (of 8 here, 6 at d = 96, 5 at d = 80) -> its output column
            constexpr int NCHK = DV == TD ? 8 : DV == 96 ? 6 : 5;
#pragma unroll
            for (int ch = 0; ch < NCHK; ++ch) {
                const int j = ch >> 2, c0 = (ch & 3) * 8;
                const int col = DV == TD ? 64 * hf + 8 * ch
                                : DV == 96 ? (ch < 4 ? 32 * hf + 8 * ch : 64 + 16 * hf + 8 * (ch - 4))
                                           : (ch < 4 ? 32 * hf + 8 * ch : 64 + 8 * hf);
                uint4 w;
                w.x = pack_half2(__uint_as_float(v[j][c0 + 0]), __uint_as_float(v[j][c0 + 1]));
                w.y = pack_half2(__uint_as_float(v[j][c0 + 2]), __uint_as_float(v[j][c0 + 3]));
                w.z = pack_half2(__uint_as_float(v[j][c0 + 4]), __uint_as_float(v[j][c0 + 5]));
                w.w = pack_half2(__uint_as_float(v[j][c0 + 6]), __uint_as_float(v[j][c0 + 7]));
                *reinterpret_cast<uint4*>(O + sw128_offset(m, col)) = w;
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar_sync(1, 32 * DQ_EPI);
            if (leader) {
                const TileId id = decode_tile128(P, t);
                const uint32_t src = sbase + DQ_OFF_O + s * T_A_BYTES;
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
    if (warp == 0) tc::tmem_dealloc(tmem, DQ_TMEM_COLS);
}

template <int BK, int BV, int DV>
static int launch_dq_tc(const CodecCall& c) {
    using C = DqCfg<BK, BV>;
    CodecParams P;
    fill_params(c, P);
    set_tile_grid(c, P, TM);
    P.fault = codec_fault_word();
    if (!P.fault) return SRFTKV_ERR_CUDA;
    DqMaps M;
    const unsigned long long tcap = (unsigned long long)c.t_cap, nrow = (unsigned long long)c.n_outer * c.H;
    const int ng = DV / c.group;
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        const int rb = DV * d.bits / 8;
        // packed planes [n_outer*H][t_cap][row], copied as exact rows with the
        // swizzle mode equal to the row length (64/128-byte code rows, 32-byte
        // group-16 scale rows; 16-byte group-32 scale rows and the 48/96-byte
        // code rows of d = 96 unswizzled)
        auto swz = [](int bytes) {
            return bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                   : bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                   : bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                 : CU_TENSOR_MAP_SWIZZLE_NONE;
        };
        const unsigned long long cdims[3] = {(unsigned long long)rb, tcap, nrow};
        const unsigned long long cstr[2] = {(unsigned long long)rb, tcap * rb};
        const unsigned cbox[3] = {(unsigned)rb, (unsigned)TM, 1u};
        const unsigned long long sdims[3] = {(unsigned long long)ng, tcap, nrow};
        const unsigned long long sstr[2] = {ng * 4ull, tcap * ng * 4ull};
        const unsigned sbox[3] = {(unsigned)ng, (unsigned)TM, 1u};
        if (!encode_x_map(&M.out[s], d.x, DV, c.H, c.n_tokens, c.n_outer, TM, true)) return SRFTKV_ERR_CUDA;
        if (DV == 80) {  // code and scale rows read by plain bulk copies
            M.codes[s] = M.scales[s] = M.out[s];
            continue;
        }
        if (!encode_tiled_swz(&M.codes[s], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, d.codes, cdims, cstr, cbox, swz(rb),
                              "tensor-core dequantize codes"))
            return SRFTKV_ERR_CUDA;
        if (d.scale_format != SRFTKV_SCALE_FP32 || DV != TD) {
            // the plane's bytes as rows of 16; one tile is 128 * ng * sb / 16 of them
            const unsigned long long sb = (unsigned long long)scale_bytes(d.scale_format);
            const unsigned long long rdims[3] = {16ull, tcap * ng * sb / 16, nrow};
            const unsigned long long rstr[2] = {16ull, tcap * ng * sb};
            const unsigned rbox[3] = {16u, (unsigned)(TM * ng * sb / 16), 1u};
            if (!encode_tiled(&M.scales[s], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, d.scales, rdims, rstr, rbox,
                              "tensor-core dequantize scales (16-byte rows)"))
                return SRFTKV_ERR_CUDA;
        } else if (!encode_tiled_swz(&M.scales[s], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, d.scales, sdims, sstr, sbox,
                                     swz(4 * ng), "tensor-core dequantize scales")) {
            return SRFTKV_ERR_CUDA;
        }
    }
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(srft_dequantize_tc_kernel<BK, BV, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        attr = true;
    }
    int blocks = device_sm_count();
    if (blocks > P.total_tiles) blocks = P.total_tiles;
    srft_dequantize_tc_kernel<BK, BV, DV><<<blocks, DQ_WARPS * 32, C::SMEM, c.stream>>>(M, P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tensor-core dequantize launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return SRFTKV_OK;
}

template <int BK, int BV, int SF, int DV>
static int launch_tc(const CodecCall& c) {
    CodecParams P;
    fill_params(c, P);
    set_tile_grid(c, P, TM);
    P.fault = codec_fault_word();
    if (!P.fault) return SRFTKV_ERR_CUDA;
    CUtensorMap tm[2];
    for (int s = 0; s < 2; ++s) {
        const CodecSideDesc& d = c.side[s < c.n_sides ? s : 0];
        if (!encode_x_map(&tm[s], d.x, c.d, c.H, c.n_tokens, c.n_outer, TM, true)) return SRFTKV_ERR_CUDA;
    }
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(srft_quantize_tc_kernel<BK, BV, SF, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             T_SMEM);
        attr = true;
    }
    int blocks = device_sm_count();
    if (blocks > P.total_tiles) blocks = P.total_tiles;
    srft_quantize_tc_kernel<BK, BV, SF, DV><<<blocks, T_WARPS * 32, T_SMEM, c.stream>>>(tm[0], tm[1], P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tensor-core quantize launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return SRFTKV_OK;
}

template <int SF, int DV>
static int launch_tc_bits(const CodecCall& c, int bk, int bv) {
    if (bk == 4 && bv == 4) return launch_tc<4, 4, SF, DV>(c);
    if (bk == 8 && bv == 8) return launch_tc<8, 8, SF, DV>(c);
    if (bk == 8 && bv == 4) return launch_tc<8, 4, SF, DV>(c);
    return launch_tc<4, 8, SF, DV>(c);
}
template <int SF>
static int launch_tc_dim(const CodecCall& c, int bk, int bv) {
    return c.d == 96 ? launch_tc_bits<SF, 96>(c, bk, bv)
           : c.d == 80 ? launch_tc_bits<SF, 80>(c, bk, bv)
                       : launch_tc_bits<SF, TD>(c, bk, bv);
}

int codec_quantize_tc(const CodecCall& c) {
    if ((c.d != TD && c.d != 96 && c.d != 80) || c.group > 32) return 1;  // a group must fit in one epilogue thread's 32 columns
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    const int sf = c.side[0].scale_format;  // both sides share it (mixed calls are split on the host)
    if (sf == SRFTKV_SCALE_FP16) return launch_tc_dim<SRFTKV_SCALE_FP16>(c, bk, bv);
    if (sf == SRFTKV_SCALE_E8M0) return launch_tc_dim<SRFTKV_SCALE_E8M0>(c, bk, bv);
    return launch_tc_dim<SRFTKV_SCALE_FP32>(c, bk, bv);
}

template <int DV>
static int launch_dq_bits(const CodecCall& c, int bk, int bv) {
    if (bk == 4 && bv == 4) return launch_dq_tc<4, 4, DV>(c);
    if (bk == 8 && bv == 8) return launch_dq_tc<8, 8, DV>(c);
    if (bk == 8 && bv == 4) return launch_dq_tc<8, 4, DV>(c);
    return launch_dq_tc<4, 8, DV>(c);
}

int dq_tc_scale_rows_ok(const CodecCall& c) {
    // fp16 / e8m0 planes (and every plane of d = 96 and 80) are copied in rows of 16
    // bytes: a token's scale bytes times t_cap and t_offset must be whole rows;
    // at d = 80 the code planes as well
    for (int s = 0; s < c.n_sides; ++s) {
        const long long cb = (long long)c.d * c.side[s].bits / 8;
        if (c.d == 80 && (((long long)c.t_cap * cb) % 16 || ((long long)c.t_offset * cb) % 16)) return 0;
        const long long rb = (long long)(c.d / c.group) * scale_bytes(c.side[s].scale_format);
        if ((c.side[s].scale_format != SRFTKV_SCALE_FP32 || c.d != TD) &&
            (((long long)c.t_cap * rb) % 16 || ((long long)c.t_offset * rb) % 16))
            return 0;
    }
    return 1;
}

int codec_dequantize_tc(const CodecCall& c) {
    if ((c.d != TD && c.d != 96 && c.d != 80) || c.group > 32) return 1;  // scale rows of at least 16 bytes (TMA)
    if (!dq_tc_scale_rows_ok(c)) return 1;
    const int bk = c.side[0].bits, bv = c.n_sides > 1 ? c.side[1].bits : bk;
    return c.d == 96 ? launch_dq_bits<96>(c, bk, bv)
           : c.d == 80 ? launch_dq_bits<80>(c, bk, bv)
                       : launch_dq_bits<TD>(c, bk, bv);
}

}  // namespace srftkv
