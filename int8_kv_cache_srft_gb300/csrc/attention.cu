// attention.cu -- decode attention that reads the packed SRFT cache directly.
//
// Method: "Gemini on-device quantization, KV cache, Apple Silicon", section
// "Flash Attention and Metal kernel fusion": tiles of tokens with an online
// softmax, so the T-long score vector never exists in memory.  "When
// Quantization Is Free ...", Methodology 1: the SRFT R is orthogonal, so
//   q . k_hat_t = (R q) . (R k_hat_t) = sum_i (R q)_i z_hat_{t,i} / lambda_i
// and sum_t p_t v_hat_t = R^T (sum_t p_t z_hat^V_t / lambda^V).  The cache is
// therefore read in its rotated, quantised form: q is rotated once, and the
// output is rotated back once per (batch, query head), never per token.
//
// Three launches per call:
//   1. prep: q_tilde = SRFT(q) / lambda_K * sm_scale * log2(e) (one block of four
//      warps per row);
//   2. split: grid (n_splits, B*Hkv*head groups), launched as the prep's
//      programmatic dependent.  Each warp streams chunks of tokens of its
//      split; a TMA copy per plane (codes and scales of K and V) lands each chunk
//      in shared memory, swizzled (or padded) so that the ldmatrix reads that
//      follow are bank-conflict free.  Codes are turned into exact fp16
//      integers in registers and contracted on the tensor cores
//      (mma.sync m16n8k16, fp32 accumulate): S = codes_K . q_tilde per 16-token
//      tile, the per-group scale applied to the fp32 partial of each group,
//      then acc += codes_V^T . (p * scale_V).  The GQA query heads of one kv
//      head share every tile.  Per-warp online softmax states are merged in
//      shared memory into one partial (m, l, acc) per (query head, split);
//   3. combine: merge the splits, divide by l and lambda_V, inverse SRFT (one
//      block per row, launched as the split kernel's programmatic dependent).
//
// The contractions are tiny (4 query heads per kv head), so the tensor cores
// are used for what they are here: a way to do the 2 x 4 multiply-adds per
// cached element in very few instructions, leaving the issue slots for the
// dequantisation bit tricks and the softmax.  The codes are exact in fp16;
// the other operand (q_tilde, or p * scale_V) is split into two fp16 halves
// hi + lo and contracted twice, which keeps the products at ~22-bit accuracy.
#include <cuda_fp16.h>

#include <atomic>
#include <cmath>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "srft_math.cuh"

namespace srftkv {

static __device__ unsigned int g_attn_fault;

// Polls of the split kernel's wait for a chunk before the warp gives up; a
// negative value selects the default (2^20 polls, about a second).  Set only
// by srftkv_set_attention_poll_limit_for_testing.
static std::atomic<int> g_poll_limit{-1};
void attention_set_poll_limit(int polls) { g_poll_limit.store(polls < 0 ? -1 : polls); }

constexpr int kAttnWarps = 4;
constexpr int kFoldChunks = 64;  // a warp folds the V code offset out of its accumulators this often (a power of two)
#ifndef SRFTKV_ATTN_STAGES
#define SRFTKV_ATTN_STAGES 2  // TMA stages per warp (chunks in flight + 1)
#endif
#ifndef SRFTKV_ATTN_CH
#define SRFTKV_ATTN_CH 0      // tokens per chunk; 0 = 32, or 16 when a 32-token stage would exceed 9 KB
#endif

struct AttnParams {
    const uint16_t* q;     // fp16 [B][Hq][D]
    float* qt;             // fp32 [B][Hq][D] prepared queries (workspace)
    float* part_ml;        // [B*Hq][n_splits][2]  (m, l) in log2 units
    float* part_acc;       // [B*Hq][n_splits][D]
    float* out;            // fp32 [B][Hq][D]
    const int* seq_lens;   // [B] or null
    const float* lam_k;
    long long lam_k_stride;
    const float* lam_v;
    long long lam_v_stride;
    const uint8_t* vscale; // V scale plane (bytes), read directly only to size the V unit (see the split kernel)
    int B, Hq, Hkv, rep, t_cap, n_splits, group, log2_group;
    int hpg, n_hg;         // query heads per head group (<= 4) and head groups per kv head
    int sp;                // scale row (floats)
    int tr_k, tr_v;        // transform of the K and V sides (SRFTKV_TRANSFORM_*)
    int sf_k, sf_v;        // scale format of the K and V sides (SRFTKV_SCALE_*)
    float qscale;          // sm_scale * log2(e)
    uint32_t poll_limit;   // polls of a warp's wait for its next chunk before it gives up
    uint32_t sign_mask[128];
};

// ---------------------------------------------------------------------------
// Small PTX helpers
// ---------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the kernel before it in the stream still runs;
// griddep_wait blocks until that kernel has completed and its memory writes are
// visible (a no-op for a kernel launched the ordinary way).  griddep_launch_dependents
// lets the next such kernel start launching once every CTA of this one has
// called it or exited.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// two matrices (the addresses of lanes 0-15)
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t (&r)[2]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// D = A . B + D, m16n8k16, fp16 inputs, fp32 accumulators
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A . B + (c0, c1, c0, c1): the accumulator starts from per-column values
__device__ __forceinline__ void mma16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1, float c0, float c1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %10, %11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}
// (a, b) ~= hi + lo with both halves fp16: the MMA then sees a and b to about
// 22 bits instead of 11 (codes are exact in fp16, so this is the only rounding
// of the contraction inputs).
// The residuals a - hi.x and b - hi.y are exact in fp32 (hi is a rounding of
// them to 11 bits); each is one mixed-precision FMA, hi.x * -1 + a, with the
// fp16 half taken straight from the packed register instead of a widening
// convert and a subtraction.
__device__ __forceinline__ void split_h2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(a, b);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    float ra, rb;
    asm("{\n\t.reg .f16 hx, hy, m1;\n\t"
        "mov.b32 {hx, hy}, %2;\n\t"
        "mov.b16 m1, 0xBC00;\n\t"
        "fma.rn.f32.f16 %0, hx, m1, %3;\n\t"
        "fma.rn.f32.f16 %1, hy, m1, %4;\n\t}"
        : "=f"(ra), "=f"(rb)
        : "r"(hi), "f"(a), "f"(b));
    const __half2 l = __floats2half2_rn(ra, rb);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}
// Packed fp32 (one instruction for two lanes of work; IEEE rounding per lane).
__device__ __forceinline__ float2 mul2(float a0, float a1, float b0, float b1) {
    return __fmul2_rn(make_float2(a0, a1), make_float2(b0, b1));
}
__device__ __forceinline__ float2 fma2(float a0, float a1, float b0, float b1, float2 c) {
    return __ffma2_rn(make_float2(a0, a1), make_float2(b0, b1), c);
}

// Codes -> fp16 pairs in one logic op.  Bits 0xF/0xF0000 (0xF0/0xF00000)
// hold two two's-complement nibbles; XOR with 8 makes them offset binary, and
// with a zero exponent field the fp16 bit pattern is the subnormal
// (q + 8) * 2^-24 (or (q + 8) * 2^-20 for the high nibbles), exactly.  Bytes
// give (q + 128) * 2^-24.  The offset is removed after the contraction from the
// column sums of the other operand (offset * sum of B), which is small enough
// next to the signal that nothing is lost to cancellation; the unit 2^-24 is
// folded into the score and output scaling.
constexpr float kSub = 16777216.f;  // 2^24
// The XOR to offset binary is taken once per loaded word (ob4 / ob8: every
// nibble or byte at once, and it commutes with the >> 8 of the second pair),
// so each extraction is a single AND: (w & m) ^ (0x8.. & m) as one logic op
// would need two immediate operands, which one LOP3 cannot take.
__device__ __forceinline__ uint32_t ob4(uint32_t w) { return w ^ 0x88888888u; }  // int4 nibbles -> offset binary
__device__ __forceinline__ uint32_t ob8(uint32_t w) { return w ^ 0x80808080u; }  // int8 bytes -> offset binary
__device__ __forceinline__ uint32_t u4_lo(uint32_t wx) { return wx & 0x000F000Fu; }  // nibbles 0, 16 of ob4(w)
__device__ __forceinline__ uint32_t u4_hi(uint32_t wx) { return wx & 0x00F000F0u; }  // nibbles 4, 20 of ob4(w)
__device__ __forceinline__ uint32_t u8_lo(uint32_t wx) { return wx & 0x00FF00FFu; }  // bytes 0, 2 of ob8(w)
__device__ __forceinline__ float h2_sum(uint32_t h) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    return f.x + f.y;
}

// Shared-memory images of the cache planes.  TMA copies whole rows (a box
// exactly as wide as the row: a wider, zero-filled box turns each chunk into
// one small request per row and cost about 9 % of the streaming rate).  Code
// rows of at most 128 bytes land swizzled (TMA's 32/64/128-byte swizzle, the
// mode equal to the row length), which keeps the ldmatrix reads free of bank
// conflicts without padding; longer rows (fp16, or int8 at d=256) keep 16
// bytes of padding per row.
//
// Rows that are not a whole number of 16-byte chunks (int4 at d = 80: 40
// bytes) can be neither a TMA row (strides are multiples of 16 bytes) nor an
// ldmatrix row (16-byte aligned addresses).  Such planes are read as rows of
// token PAIRS (80 bytes: five 16-byte segments, the middle one holding the
// even token's last 8 bytes and the odd token's first 8), and the MMAs take
// pairs as their rows (see tile_scores_pair / tile_pv_pair).
template <int D, int BITS>
struct PlaneT {
    static constexpr int RB = D * BITS / 8;                // bytes per cached row
    static constexpr bool PAIR = RB % 16 == 8;             // read as rows of token pairs
    static constexpr bool SWZ = !PAIR && BITS != 16 && RB <= 128 && (RB & (RB - 1)) == 0;  // exact rows, swizzled
    // unswizzled rows: an odd number of 16-byte chunks is already free of
    // ldmatrix bank conflicts (48-byte int4 rows at d = 96, 80-byte int8 rows and
    // int4 pairs at d = 80); others get 16 bytes of padding
    static constexpr int RP = SWZ || PAIR || (RB / 16) % 2 == 1 ? RB : RB + 16;  // shared-memory pitch per token
    static constexpr int NSEG = 2 * RB / 16;               // 16-byte segments of a pair row (PAIR only)
};

// 16-byte chunks of a group-16 fp32 scale row (d/4 bytes; 24 at d = 96 -> 2)
template <int D>
constexpr int scale_chunks() { return (D / 4 + 15) / 16; }
template <int D>
constexpr bool pow2_dim() { return (D & (D - 1)) == 0; }

// Byte offset of 16-byte chunk `ch` of row `r` in a swizzled plane of RB-byte
// rows (TMA swizzle: address bits [4, 4+b) XOR bits [7, 7+b), b = log2(RB/16)),
// for a buffer that starts on a 1024-byte boundary.
template <int RB>
__host__ __device__ constexpr int swz_chunk(int r, int ch) {
    if constexpr ((RB & (RB - 1)) != 0) return ch;  // rows that are not a power of two are never swizzled
    return ch ^ (((r * RB) >> 7) & (RB / 16 - 1));
}

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// d = 256 with 4-bit keys keeps the K-side B fragments of q (hi, lo and the
// offset terms: 80 registers a thread) in shared memory instead of registers,
// which lets the kernel run three CTAs an SM instead of two; each 32-dim chunk
// reads them back with two 16-byte loads and one 8-byte load.
template <int D, int BK>
constexpr bool q_in_smem() { return D == 256 && BK == 4; }

template <int D, int BK, int BV>
struct AttnCfg {
    static constexpr bool QK = BK != 16, QV = BV != 16;
    static constexpr int SRB = D / 4;  // largest scale row in bytes (group 16); exact rows, no padding
    static constexpr int STAGE32 = 32 * (PlaneT<D, BK>::RP + PlaneT<D, BV>::RP + (QK ? SRB : 0) + (QV ? SRB : 0));
    // d = 192 with stages of at most 13.5 KB: 32-token chunks at 2 CTAs an SM (no register spills either)
    // beat 16-token chunks at 3 (1.04 against 1.13 ms on the decode shape); d = 256 keeps 16 (1.48 against 1.79)
    static constexpr bool WIDE32 = D == 192 && STAGE32 <= 13824;
    static constexpr int CH = SRFTKV_ATTN_CH ? SRFTKV_ATTN_CH : (STAGE32 <= 9216 || WIDE32 ? 32 : 16);  // tokens per chunk
    static constexpr bool QSM = q_in_smem<D, BK>();
    static constexpr int MINB = (D >= 256 && !QSM) || WIDE32 ? 2 : (D == 96 && BK == 4 && BV == 4) ? 4 : 3;  // CTAs an SM the kernel is compiled for
    static constexpr int NS = SRFTKV_ATTN_STAGES;
    // swizzled sub-buffers (code rows of <= 128 bytes, group-16 scale rows of
    // >= 32 bytes) start on a 1024-byte boundary, the others on 128 bytes
    static constexpr int AK = PlaneT<D, BK>::SWZ ? 1024 : 128, AV = PlaneT<D, BV>::SWZ ? 1024 : 128;
    static constexpr int AS = (QK || QV) && SRB >= 32 ? 1024 : 128;
    static constexpr int A0 = AK > AV ? (AK > AS ? AK : AS) : (AV > AS ? AV : AS);  // stage alignment
    static constexpr int OFF_KC = 0;
    static constexpr int OFF_KS = align_up(OFF_KC + CH * PlaneT<D, BK>::RP, AS);
    static constexpr int OFF_VC = align_up(OFF_KS + (QK ? CH * SRB : 0), AV);
    static constexpr int OFF_VS = align_up(OFF_VC + CH * PlaneT<D, BV>::RP, AS);
    // fp16 / e8m0 scale planes land raw (at most 2 bytes a scale) and are widened into the fp32 rows above
    static constexpr int RAWB = CH * (D / 16) * 2;
    static constexpr int OFF_KR = align_up(OFF_VS + (QV ? CH * SRB : 0), 128);
    static constexpr int OFF_VR = align_up(OFF_KR + (QK ? RAWB : 0), 128);  // a TMA destination (320 bytes of K at d = 80)
    static constexpr int STAGE = align_up(OFF_VR + (QV ? RAWB : 0), A0);
    static constexpr int WARP_BYTES = NS * STAGE;
    static constexpr int MERGE_BYTES = kAttnWarps * (4 * D + 8) * 4;
    static constexpr int BODY = kAttnWarps * WARP_BYTES > MERGE_BYTES ? kAttnWarps * WARP_BYTES : MERGE_BYTES;
    // q fragments (QSM): hi and lo [D/32][32 lanes] x 16 bytes, offset terms [D/32][32] x 8 bytes
    static constexpr int OFF_QF = BODY;
    static constexpr int QF_BYTES = QSM ? (D / 32) * 32 * (16 + 16 + 8) : 0;
    static constexpr int BARS = OFF_QF + QF_BYTES;      // mbarriers after the body (and the q fragments)
    static constexpr int SMEM = 1024 + BARS + 128;      // + slack to realign the base to 1024 bytes
    static_assert(OFF_KC % 128 == 0 && OFF_KS % 128 == 0 && OFF_VC % 128 == 0 && OFF_VS % 128 == 0 &&
                      OFF_KR % 128 == 0 && OFF_VR % 128 == 0 && STAGE % 128 == 0,
                  "TMA destinations on 128-byte boundaries");
    static_assert(OFF_QF % 16 == 0 && BARS % 8 == 0, "q fragments as 16-byte loads, mbarriers on 8 bytes");
    static constexpr bool PK = PlaneT<D, BK>::PAIR, PV = PlaneT<D, BV>::PAIR;
    static_assert(!(PK || PV) || CH == 32, "a chunk of token pairs is one 16-row MMA tile");
    // K-side B-fragment registers and code-offset terms: four and two per 32-dim chunk (int4), per 16-byte
    // segment of a pair row (int4 pairs), two and one per 16 dims (int8 / fp16)
    static constexpr int QB = PK ? 4 * PlaneT<D, BK>::NSEG : D / 8;
    static constexpr int NB = PK ? 2 * PlaneT<D, BK>::NSEG : D / 16;
    // V accumulators: eight per 32-dim chunk or pair segment (half of them useful for int4), four per 16 dims
    static constexpr int ACC = PV ? 8 * PlaneT<D, BV>::NSEG : D / 4;
    static constexpr int NSV = PV ? PlaneT<D, BV>::NSEG : BV == 4 ? D / 32 : BV == 8 ? D / 16 : 1;  // column sums of the V-side B
};

// ---------------------------------------------------------------------------
// 1. q preparation
// ---------------------------------------------------------------------------
// fp16 cache (no rotation): q times the softmax scale, one thread per row.
template <int D>
__global__ void __launch_bounds__(128) attn_prep_q_raw_kernel(const __grid_constant__ AttnParams P) {
    const int row = blockIdx.x * 128 + threadIdx.x;
    if (row >= P.B * P.Hq) return;
    const uint4* xr = reinterpret_cast<const uint4*>(P.q + (long long)row * D);
    float4* yr = reinterpret_cast<float4*>(P.qt + (long long)row * D);
#pragma unroll 4
    for (int c = 0; c < D / 8; ++c) {
        const uint4 v = __ldg(xr + c);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
        const float2 bq = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
        const float2 cc = __half22float2(*reinterpret_cast<const __half2*>(&v.z));
        const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&v.w));
        yr[2 * c] = make_float4(a.x * P.qscale, a.y * P.qscale, bq.x * P.qscale, bq.y * P.qscale);
        yr[2 * c + 1] = make_float4(cc.x * P.qscale, cc.y * P.qscale, dd.x * P.qscale, dd.y * P.qscale);
    }
    griddep_launch_dependents();  // the split kernel may start launching (it waits for this grid's end)
}

// The packed unitary DFT R of length D (the SRFT's rotation, R diag(s)):
// row 0 is the DC term 1/sqrt(D), row 1 the Nyquist term (-1)^k / sqrt(D),
// rows 2f and 2f+1 (0 < f < D/2) sqrt(2/D) cos(2 pi f k / D) and
// -sqrt(2/D) sin(2 pi f k / D).  The tables hold those two scaled functions
// of m = f k mod D, in fp32 (sincospif is within one ulp).
template <int D>
__device__ __forceinline__ void dft_tables(float* tcs, float* tsn) {
    const float c = sqrtf(2.f / (float)D);
    for (int m = threadIdx.x; m < D; m += blockDim.x) {
        float sv, cv;
        sincospif((float)(2 * m) / (float)D, &sv, &cv);
        tcs[m] = c * cv;
        tsn[m] = -c * sv;
    }
}
// m + f mod D for m, f < D
template <int D>
__device__ __forceinline__ int mod_add(int m, int f) {
    if constexpr ((D & (D - 1)) == 0) return (m + f) & (D - 1);
    else {
        m += f;
        return m >= D ? m - D : m;
    }
}
__device__ __forceinline__ bool sign_neg(const uint32_t* mask, int k) {
    return (mask[k >> 1] & ((k & 1) ? 0x80000000u : 0x8000u)) != 0u;
}
// Unnormalised Walsh-Hadamard transform (Sylvester natural order) of the D
// values a warp holds, coordinate 32 j + lane in v[j]: butterflies over the
// register index for the high bits, over the lanes (shuffles) for the low five.
template <int D>
__device__ __forceinline__ void wht_warp(float (&v)[D / 32], int lane) {
#pragma unroll
    for (int h = 1; h < D / 32; h <<= 1)
#pragma unroll
        for (int j = 0; j < D / 32; ++j)
            if (!(j & h)) {
                const float x = v[j], y = v[j + h];
                v[j] = x + y;
                v[j + h] = x - y;
            }
#pragma unroll
    for (int s2 = 1; s2 < 32; s2 <<= 1)
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
            const float o = __shfl_xor_sync(0xffffffffu, v[j], s2);
            v[j] = (lane & s2) ? o - v[j] : v[j] + o;
        }
}

// q preparation: p = R diag(s) q, times the softmax scale (log2 units) and
// 1/lambda_K, into fp32 [B][Hq][D].  One block of four warps per query row.
// SRFT: warp w takes the inputs k in [wD/4, (w+1)D/4), lane the frequencies
// f = lane + 32 j (rows 2f, 2f+1), walking k with the table index f k mod D;
// the four partial rows are summed through shared memory, and the Nyquist row
// is a sum of (-1)^k x_k.  SRHT: the Walsh-Hadamard transform across one warp.
template <int D>
__global__ void __launch_bounds__(128) attn_prep_q_kernel(const __grid_constant__ AttnParams P) {
    constexpr int NF = (D / 2 + 31) / 32, KQ = D / 4;
    __shared__ float tcs[D], tsn[D], xs[D], part[4][D], nyq[4];
    const bool srht = pow2_dim<D>() && P.tr_k == SRFTKV_TRANSFORM_SRHT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (!srht) dft_tables<D>(tcs, tsn);
    const int row = blockIdx.x;
    const int b = row / P.Hq, hq = row - b * P.Hq, hkv = hq / P.rep;
    const __half* qr = reinterpret_cast<const __half*>(P.q) + (long long)row * D;
    for (int k = threadIdx.x; k < D; k += blockDim.x) {
        const float x = __half2float(qr[k]);
        xs[k] = sign_neg(P.sign_mask, k) ? -x : x;
    }
    __syncthreads();
    const float* lam = P.lam_k ? P.lam_k + (long long)b * P.lam_k_stride + (long long)hkv * D : nullptr;
    float* yr = P.qt + (long long)row * D;
    auto emit = [&](int o, float a) { yr[o] = a * (lam ? P.qscale * __frcp_rn(lam[o]) : P.qscale); };
    const float isd = rsqrtf((float)D);
    if constexpr (pow2_dim<D>()) {
        if (srht) {
            if (warp != 0) return;
            float v[D / 32];
#pragma unroll
            for (int j = 0; j < D / 32; ++j) v[j] = xs[32 * j + lane];
            wht_warp<D>(v, lane);
#pragma unroll
            for (int j = 0; j < D / 32; ++j) emit(32 * j + lane, v[j] * isd);
            griddep_launch_dependents();
            return;
        }
    }
    const int k0 = warp * KQ;
    float re[NF], im[NF];
    int m[NF], f[NF];
#pragma unroll
    for (int j = 0; j < NF; ++j) {
        re[j] = im[j] = 0.f;
        f[j] = min(lane + 32 * j, D - 1);  // lanes past D/2 compute a row nobody stores
        m[j] = (f[j] * k0) % D;
    }
    float ny = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < KQ; ++kk) {
        const float x = xs[k0 + kk];
        ny += ((k0 + kk) & 1) ? -x : x;
#pragma unroll
        for (int j = 0; j < NF; ++j) {
            re[j] = fmaf(tcs[m[j]], x, re[j]);
            im[j] = fmaf(tsn[m[j]], x, im[j]);
            m[j] = mod_add<D>(m[j], f[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < NF; ++j) {
        const int fr = lane + 32 * j;
        if (fr < D / 2) {
            part[warp][2 * fr] = re[j];
            part[warp][2 * fr + 1] = im[j];
        }
    }
    if (lane == 0) nyq[warp] = ny;
    __syncthreads();
    for (int o = threadIdx.x; o < D; o += blockDim.x) {
        float a = (part[0][o] + part[1][o]) + (part[2][o] + part[3][o]);
        if (o == 0) a *= 0.70710678118654752f;  // sqrt(2/D) sum x / sqrt(2)
        if (o == 1) a = ((nyq[0] + nyq[1]) + (nyq[2] + nyq[3])) * isd;
        emit(o, a);
    }
    // the split kernel may start launching now (it waits for this grid's end before it reads q); signalling
    // at the start placed a small split grid unevenly over the SMs the preparation still held
    griddep_launch_dependents();
}

// ---------------------------------------------------------------------------
// 2. split kernel
// ---------------------------------------------------------------------------
// K-side B fragments (q_tilde as fp16 hi + lo) for this thread.  Column n of
// every MMA is (query head n/2 of the group, half n%2): for 4-bit keys half 0
// takes the dims of the first 16-dim group of each 32-dim chunk and half 1 the
// second, so one MMA yields both groups' partials for a head in the two
// columns one thread owns; for 8-bit and fp16 keys half 1 is zero.  The
// high-nibble rows carry q / 16, matching their 16x larger code unit.
//
// nb[j] is minus the code offset times the column sum of B for the
// accumulator columns this thread holds (4-bit: chunk j/2, column 2c + j%2;
// 8-bit: chunk j, column 2c), in the 2^-24 unit of the codes.
template <int D, int BK>
__device__ __forceinline__ void build_qb(const float* __restrict__ qrow_base, int rep, int g, int c,
                                         uint32_t (&qh)[D / 8], uint32_t (&ql)[D / 8], float (&nb)[D / 16]) {
    const int h = g >> 1, sigma = g & 1;
    const bool head_ok = h < rep;
    const float* q = qrow_base + (long long)h * D;
    auto val = [&](int dim, bool ok) -> float { return (ok && head_ok) ? q[dim] : 0.f; };
    if constexpr (BK == 4) {
        // chunk m (32 dims): thread c owns dims 8c..8c+7, which lie in half c/2
        const bool ok = (c >> 1) == sigma;
        constexpr float i16 = 0.0625f;
#pragma unroll
        for (int m = 0; m < D / 32; ++m) {
            const int base = 32 * m + 8 * c;
            split_h2(val(base + 0, ok), val(base + 4, ok), qh[4 * m + 0], ql[4 * m + 0]);
            split_h2(val(base + 1, ok) * i16, val(base + 5, ok) * i16, qh[4 * m + 1], ql[4 * m + 1]);
            split_h2(val(base + 2, ok), val(base + 6, ok), qh[4 * m + 2], ql[4 * m + 2]);
            split_h2(val(base + 3, ok) * i16, val(base + 7, ok) * i16, qh[4 * m + 3], ql[4 * m + 3]);
            // offset 8 per code; the high-nibble rows count 16x (their unit is 2^-20)
            float part = h2_sum(qh[4 * m + 0]) + h2_sum(ql[4 * m + 0]) + h2_sum(qh[4 * m + 2]) + h2_sum(ql[4 * m + 2]);
            part += 16.f * (h2_sum(qh[4 * m + 1]) + h2_sum(ql[4 * m + 1]) + h2_sum(qh[4 * m + 3]) + h2_sum(ql[4 * m + 3]));
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);  // column g's total over its 16 k rows x 2 MMAs
            nb[2 * m + 0] = (-8.f / kSub) * __shfl_sync(0xffffffffu, part, 4 * (2 * c));
            nb[2 * m + 1] = (-8.f / kSub) * __shfl_sync(0xffffffffu, part, 4 * (2 * c + 1));
        }
    } else if constexpr (BK == 8) {
        const bool ok = sigma == 0;
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
            const int base = 16 * m + 4 * c;
            split_h2(val(base + 0, ok), val(base + 2, ok), qh[2 * m + 0], ql[2 * m + 0]);
            split_h2(val(base + 1, ok), val(base + 3, ok), qh[2 * m + 1], ql[2 * m + 1]);
            float part = h2_sum(qh[2 * m]) + h2_sum(ql[2 * m]) + h2_sum(qh[2 * m + 1]) + h2_sum(ql[2 * m + 1]);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            nb[m] = (-128.f / kSub) * __shfl_sync(0xffffffffu, part, 4 * (2 * c));
        }
    } else {
        const bool ok = sigma == 0;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
            split_h2(val(16 * j + 2 * c, ok), val(16 * j + 2 * c + 1, ok), qh[2 * j + 0], ql[2 * j + 0]);
            split_h2(val(16 * j + 8 + 2 * c, ok), val(16 * j + 9 + 2 * c, ok), qh[2 * j + 1], ql[2 * j + 1]);
            nb[j] = 0.f;
        }
    }
}

// K-side B fragments for int4 keys read as token pairs (d = 80).  Segment sg
// of a pair row is bytes 16 sg .. +15 of the pair; thread c's 4-byte word of
// it is pair byte 16 sg + 4c, i.e. token (16 sg + 4c) / RB's dims 2 b .. 2 b + 7
// with b = (16 sg + 4c) mod RB, laid out exactly as a 32-dim chunk of build_qb
// (bytes 0-7 of a segment feed column half 0, bytes 8-15 half 1; the
// straddling segment's halves belong to different tokens, which is why they
// must be separate columns).
template <int D>
__device__ __forceinline__ void build_qb_pair(const float* __restrict__ qrow_base, int rep, int g, int c,
                                              uint32_t (&qh)[4 * PlaneT<D, 4>::NSEG],
                                              uint32_t (&ql)[4 * PlaneT<D, 4>::NSEG],
                                              float (&nb)[2 * PlaneT<D, 4>::NSEG]) {
    constexpr int RB = PlaneT<D, 4>::RB, NSEG = PlaneT<D, 4>::NSEG;
    const int h = g >> 1, sigma = g & 1;
    const bool ok = h < rep && (c >> 1) == sigma;
    const float* q = qrow_base + (long long)h * D;
    auto val = [&](int dim) -> float { return ok ? q[dim] : 0.f; };
    constexpr float i16 = 0.0625f;
#pragma unroll
    for (int sg = 0; sg < NSEG; ++sg) {
        const int base = 2 * ((16 * sg + 4 * c) % RB);
        split_h2(val(base + 0), val(base + 4), qh[4 * sg + 0], ql[4 * sg + 0]);
        split_h2(val(base + 1) * i16, val(base + 5) * i16, qh[4 * sg + 1], ql[4 * sg + 1]);
        split_h2(val(base + 2), val(base + 6), qh[4 * sg + 2], ql[4 * sg + 2]);
        split_h2(val(base + 3) * i16, val(base + 7) * i16, qh[4 * sg + 3], ql[4 * sg + 3]);
        float part = h2_sum(qh[4 * sg + 0]) + h2_sum(ql[4 * sg + 0]) + h2_sum(qh[4 * sg + 2]) + h2_sum(ql[4 * sg + 2]);
        part += 16.f * (h2_sum(qh[4 * sg + 1]) + h2_sum(ql[4 * sg + 1]) + h2_sum(qh[4 * sg + 3]) + h2_sum(ql[4 * sg + 3]));
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        nb[2 * sg + 0] = (-8.f / kSub) * __shfl_sync(0xffffffffu, part, 4 * (2 * c));
        nb[2 * sg + 1] = (-8.f / kSub) * __shfl_sync(0xffffffffu, part, 4 * (2 * c + 1));
    }
}

// Per-lane part of the ldmatrix row addresses into a plane image.  Lane l
// supplies row rl of the 16-row sub-tile and reads dl chunks (0 or 1) past
// the even chunk index being loaded.  off = rl times the row pitch (plus the
// chunk step when unswizzled); x16 = (dl XOR the row's swizzle) * 16, which
// for an even chunk index c gives the swizzled chunk of c + dl as c ^ x16/16.
// A sub-tile starts on a multiple of 16 rows, which never changes the swizzle.
struct LaneRow {
    uint32_t off, x16;
};
template <int RB, bool SWZ, int RP>
__device__ __forceinline__ LaneRow lane_row(int rl, int dl) {
    LaneRow L;
    if constexpr (SWZ) {
        L.off = (uint32_t)(rl * RB);
        L.x16 = (uint32_t)((dl ^ swz_chunk<RB>(rl, 0)) << 4);
    } else {
        L.off = (uint32_t)(rl * RP + dl * 16);
        L.x16 = 0;
    }
    return L;
}
// codes, plain or transposed: matrices (rows 0-7 | 8-15) x (chunk seg | seg+1)
template <int RB, bool SWZ, int RP>
__device__ __forceinline__ LaneRow lane_row_codes(int lane) {
    return lane_row<RB, SWZ, RP>((lane & 7) + ((lane >> 3) & 1) * 8, lane >> 4);
}
// fp16 V (trans): matrices (rows 0-7, seg), (rows 0-7, seg+1), (rows 8-15, seg), (rows 8-15, seg+1)
template <int RB, bool SWZ, int RP>
__device__ __forceinline__ LaneRow lane_row_v16(int lane) {
    return lane_row<RB, SWZ, RP>((lane & 7) + (lane >> 4) * 8, (lane >> 3) & 1);
}
// ldmatrix address of this lane for the sub-tile at row tr, even chunk seg
template <int RB, bool SWZ, int RP>
__device__ __forceinline__ uint32_t plane_addr(uint32_t base, const LaneRow& L, int tr, int seg) {
    if constexpr (SWZ)
        return base + L.off + (uint32_t)(tr * RB) + (((uint32_t)seg << 4) ^ L.x16);
    else
        return base + L.off + (uint32_t)(tr * RP + seg * 16);
}

// Per-thread scale addressing.  Group-16 scale rows are SRB = d/4 bytes,
// swizzled like the codes (mode = row length); so[j] is the byte offset of
// logical 16-byte chunk j of this thread's first row.  Other group sizes use
// unswizzled rows of d/group floats.
template <int D, int NCH>
__device__ __forceinline__ void scale_offsets(int row, int extra, uint32_t (&so)[NCH]) {
    constexpr int SRB = D / 4;
#pragma unroll
    for (int j = 0; j < NCH; ++j) so[j] = (uint32_t)(row * SRB + (swz_chunk<SRB>(row, j) << 4) + extra);
}
__device__ __forceinline__ float lds_f32(const uint8_t* base, uint32_t off) {
    return *reinterpret_cast<const float*>(base + off);
}

__device__ __forceinline__ float ex2(float x) {  // 2^x; ex2.approx has a relative error of about 2^-22
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Scores of one 16-token sub-tile at row tr of the stage for this thread's
// head c: s[0] for token tr+g, s[1] for token tr+g+8 (for packed keys in the
// 2^-24 unit of the codes, for fp16 keys as is).
template <int D, int BK, int G>
__device__ __forceinline__ void tile_scores(uint32_t kc, const LaneRow& LK, const uint8_t* __restrict__ ksb,
                                            const uint32_t (&kso)[scale_chunks<D>()], int sp, int lg, int tr,
                                            int lane, const uint32_t (&qh)[D / 8], const uint32_t (&ql)[D / 8],
                                            const float (&nb)[D / 16], const uint4* __restrict__ qf, float (&s)[2]) {
    using PK = PlaneT<D, BK>;
    constexpr int SRB = D / 4;
    const int g = lane >> 2;
    const float* k0 = reinterpret_cast<const float*>(ksb) + (tr + g) * sp;
    const float* k1 = reinterpret_cast<const float*>(ksb) + (tr + g + 8) * sp;
    // scale of group f for token rows tr+g (r = 0) and tr+g+8 (r = 1)
    auto ksc = [&](int f, int r) -> float {
        if constexpr (G == 16) return lds_f32(ksb, kso[f >> 2] + (tr + 8 * r) * SRB + (f & 3) * 4);
        else return (r ? k1 : k0)[f];
    };
    if constexpr (BK == 4) {
        // token g and token g+8: (half 0, half 1) partials, summed at the end
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
        // 32-dim chunk mm from its two 8-row matrices (rows 0-7, rows 8-15)
        auto chunk = [&](int mm, uint32_t rg, uint32_t rg8) {
            // this chunk's q fragments: from registers, or from shared memory (q_in_smem)
            uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
            float n0, n1;
            if constexpr (q_in_smem<D, BK>()) {
                const uint4 H = qf[mm * 32 + lane], Lo = qf[(D / 32 + mm) * 32 + lane];
                const float2 N = reinterpret_cast<const float2*>(qf + 2 * (D / 32) * 32)[mm * 32 + lane];
                h0 = H.x, h1 = H.y, h2 = H.z, h3 = H.w, l0 = Lo.x, l1 = Lo.y, l2 = Lo.z, l3 = Lo.w, n0 = N.x, n1 = N.y;
            } else {
                h0 = qh[4 * mm], h1 = qh[4 * mm + 1], h2 = qh[4 * mm + 2], h3 = qh[4 * mm + 3];
                l0 = ql[4 * mm], l1 = ql[4 * mm + 1], l2 = ql[4 * mm + 2], l3 = ql[4 * mm + 3];
                n0 = nb[2 * mm], n1 = nb[2 * mm + 1];
            }
            rg = ob4(rg);
            rg8 = ob4(rg8);
            const uint32_t rs = rg >> 8, rs8 = rg8 >> 8;
            const uint32_t x0 = u4_lo(rg), x1 = u4_lo(rg8), x2 = u4_hi(rg), x3 = u4_hi(rg8);
            const uint32_t y0 = u4_lo(rs), y1 = u4_lo(rs8), y2 = u4_hi(rs), y3 = u4_hi(rs8);
            float d[4];
            mma16816_c(d, x0, x1, x2, x3, h0, h1, n0, n1);
            mma16816(d, y0, y1, y2, y3, h2, h3);
            mma16816(d, x0, x1, x2, x3, l0, l1);
            mma16816(d, y0, y1, y2, y3, l2, l3);
            // d = (token g: half 0, half 1, token g+8: half 0, half 1) for head c
            const int ga = (32 * mm) >> lg, gb = (32 * mm + 16) >> lg;
            a0 = fma2(ksc(ga, 0), ksc(gb, 0), d[0], d[1], a0);
            a1 = fma2(ksc(ga, 1), ksc(gb, 1), d[2], d[3], a1);
        };
#pragma unroll
        for (int m2 = 0; m2 < D / 64; ++m2) {
            uint32_t r[4];
            ldsm_x4(plane_addr<PK::RB, PK::SWZ, PK::RP>(kc, LK, tr, 2 * m2), r);
            chunk(2 * m2, r[0], r[1]);
            chunk(2 * m2 + 1, r[2], r[3]);
        }
        if constexpr (D % 64 != 0) {  // an odd number of 32-dim chunks (d = 96): the last one alone
            uint32_t r[2];
            ldsm_x2(plane_addr<PK::RB, PK::SWZ, PK::RP>(kc, LK, tr, D / 32 - 1), r);
            chunk(D / 32 - 1, r[0], r[1]);
        }
        s[0] = a0.x + a0.y;
        s[1] = a1.x + a1.y;
    } else if constexpr (BK == 8) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int m2 = 0; m2 < D / 32; ++m2) {
            uint32_t r[4];
            ldsm_x4(plane_addr<PK::RB, PK::SWZ, PK::RP>(kc, LK, tr, 2 * m2), r);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int mm = 2 * m2 + hh;
                const uint32_t rg = ob8(r[2 * hh]), rg8 = ob8(r[2 * hh + 1]);
                const uint32_t x0 = u8_lo(rg), x1 = u8_lo(rg8), x2 = u8_lo(rg >> 8), x3 = u8_lo(rg8 >> 8);
                float d[4];
                mma16816_c(d, x0, x1, x2, x3, qh[2 * mm], qh[2 * mm + 1], nb[mm], 0.f);
                mma16816(d, x0, x1, x2, x3, ql[2 * mm], ql[2 * mm + 1]);
                const int gi = (16 * mm) >> lg;
                a0 = fmaf(ksc(gi, 0), d[0], a0);
                a1 = fmaf(ksc(gi, 1), d[2], a1);
            }
        }
        if constexpr (D % 32 != 0) {  // an odd number of 16-dim chunks (d = 80): the last one alone
            constexpr int mm = D / 16 - 1;
            uint32_t r[2];
            ldsm_x2(plane_addr<PK::RB, PK::SWZ, PK::RP>(kc, LK, tr, mm), r);
            r[0] = ob8(r[0]);
            r[1] = ob8(r[1]);
            const uint32_t x0 = u8_lo(r[0]), x1 = u8_lo(r[1]), x2 = u8_lo(r[0] >> 8), x3 = u8_lo(r[1] >> 8);
            float d[4];
            mma16816_c(d, x0, x1, x2, x3, qh[2 * mm], qh[2 * mm + 1], nb[mm], 0.f);
            mma16816(d, x0, x1, x2, x3, ql[2 * mm], ql[2 * mm + 1]);
            const int gi = (16 * mm) >> lg;
            a0 = fmaf(ksc(gi, 0), d[0], a0);
            a1 = fmaf(ksc(gi, 1), d[2], a1);
        }
        s[0] = a0;
        s[1] = a1;
    } else {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
            uint32_t r[4];
            ldsm_x4(plane_addr<PK::RB, PK::SWZ, PK::RP>(kc, LK, tr, 2 * j), r);
            mma16816(d, r[0], r[1], r[2], r[3], qh[2 * j], qh[2 * j + 1]);
            mma16816(d, r[0], r[1], r[2], r[3], ql[2 * j], ql[2 * j + 1]);
        }
        s[0] = d[0];
        s[1] = d[2];
    }
}

// Scores of a 32-token chunk of int4 keys read as 16 token pairs (d = 80):
// one MMA tile whose rows are pairs.  Per 16-byte segment the two column
// halves of a head are (token parity, group) pieces of the pair: half h of
// segment sg is pair byte 16 sg + 8h, token parity (16 sg + 8h) / RB, group
// 2 ((16 sg + 8h) mod RB) / G.  s[a][b] is token 16a + 2g + b.
template <int D, int G>
__device__ __forceinline__ void tile_scores_pair(uint32_t kc, const LaneRow& LK, const uint8_t* __restrict__ ksb,
                                                 int sp, int lg, int lane, const uint32_t (&qh)[4 * PlaneT<D, 4>::NSEG],
                                                 const uint32_t (&ql)[4 * PlaneT<D, 4>::NSEG],
                                                 const float (&nb)[2 * PlaneT<D, 4>::NSEG], float (&s)[2][2]) {
    using PK = PlaneT<D, 4>;
    constexpr int RB = PK::RB, NSEG = PK::NSEG, PB = 2 * RB;
    const int g = lane >> 2;
    const float* ks = reinterpret_cast<const float*>(ksb);
    float a[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [pair g | g + 8][token parity]
    auto seg = [&](int sg, uint32_t rg, uint32_t rg8) {
        rg = ob4(rg);
        rg8 = ob4(rg8);
        const uint32_t rs = rg >> 8, rs8 = rg8 >> 8;
        const uint32_t x0 = u4_lo(rg), x1 = u4_lo(rg8), x2 = u4_hi(rg), x3 = u4_hi(rg8);
        const uint32_t y0 = u4_lo(rs), y1 = u4_lo(rs8), y2 = u4_hi(rs), y3 = u4_hi(rs8);
        float d[4];
        mma16816_c(d, x0, x1, x2, x3, qh[4 * sg], qh[4 * sg + 1], nb[2 * sg], nb[2 * sg + 1]);
        mma16816(d, y0, y1, y2, y3, qh[4 * sg + 2], qh[4 * sg + 3]);
        mma16816(d, x0, x1, x2, x3, ql[4 * sg], ql[4 * sg + 1]);
        mma16816(d, y0, y1, y2, y3, ql[4 * sg + 2], ql[4 * sg + 3]);
        // d = (pair g: half 0, half 1, pair g + 8: half 0, half 1) for head c
        const int b0 = 16 * sg, b1 = 16 * sg + 8;
        const int t0 = b0 / RB, t1 = b1 / RB;  // token parity of each half
        const int f0 = (2 * (b0 % RB)) >> lg, f1 = (2 * (b1 % RB)) >> lg;
        a[0][t0] = fmaf(ks[(2 * g + t0) * sp + f0], d[0], a[0][t0]);
        a[0][t1] = fmaf(ks[(2 * g + t1) * sp + f1], d[1], a[0][t1]);
        a[1][t0] = fmaf(ks[(16 + 2 * g + t0) * sp + f0], d[2], a[1][t0]);
        a[1][t1] = fmaf(ks[(16 + 2 * g + t1) * sp + f1], d[3], a[1][t1]);
    };
#pragma unroll
    for (int m2 = 0; m2 < NSEG / 2; ++m2) {
        uint32_t r[4];
        ldsm_x4(plane_addr<PB, false, PB>(kc, LK, 0, 2 * m2), r);
        seg(2 * m2, r[0], r[1]);
        seg(2 * m2 + 1, r[2], r[3]);
    }
    if constexpr (NSEG % 2 != 0) {
        uint32_t r[2];
        ldsm_x2(plane_addr<PB, false, PB>(kc, LK, 0, NSEG - 1), r);
        seg(NSEG - 1, r[0], r[1]);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        s[i][0] = a[i][0];
        s[i][1] = a[i][1];
    }
}

// acc += V^T B for one 16-token sub-tile, B[k][n] = p(token k, head n/2) *
// scale_V(token k, group of half n%2).  p00..p11 are p for tokens 2c+e+8f of
// head g/2 (zero for padded heads and for tokens past the end, whose scale
// rows were zeroed in shared memory).  Packed values enter as offset codes in
// the 2^-24 unit (2^-20 for high nibbles); sv[] gathers this thread's share of
// the column sums of B that remove the offset afterwards.
template <int D, int BV, int G>
__device__ __forceinline__ void tile_pv(uint32_t vc, const LaneRow& LV, const uint8_t* __restrict__ vsb,
                                        const uint32_t (&vso)[scale_chunks<D>()], int sp, int lg, int tr,
                                        int lane, float p00, float p10, float p01, float p11, uint32_t amask_lo,
                                        uint32_t amask_hi, bool tail, float (&acc)[D / 4],
                                        float (&sv)[AttnCfg<D, 4, BV>::NSV]) {
    using PV = PlaneT<D, BV>;
    constexpr int SRB = D / 4;
    const int g = lane >> 2, c = lane & 3;
    // scale of group f (group 16: chunk f/4 of the row, float f%4; vso already
    // holds this thread's column offset for 4-bit values) for token rows
    // tr+2c+e, e in {0, 1, 8, 9}
    auto vsc = [&](int gv, int f_in_chunk, int e) -> float {
        if constexpr (G == 16) return lds_f32(vsb, vso[gv] + (tr + e) * SRB + f_in_chunk * 4);
        else return reinterpret_cast<const float*>(vsb)[(tr + 2 * c + e) * sp + gv];
    };
    if constexpr (BV == 4) {
        const int side = g & 1;
        // 32-dim chunk cb from its two transposed 8-row matrices (token rows 0-7, 8-15)
        auto chunk = [&](int cb, uint32_t R0, uint32_t R1) {
            // group 16: group 2cb + side lies in chunk cb/2 at float 2(cb%2) + side (side folded into vso)
            const int gv = G == 16 ? cb >> 1 : (32 * cb + 16 * side) >> lg;
            const int fc = 2 * (cb & 1);
            const float2 b0 = mul2(p00, p10, vsc(gv, fc, 0), vsc(gv, fc, 1));  // tokens 2c, 2c+1
            const float2 b1 = mul2(p01, p11, vsc(gv, fc, 8), vsc(gv, fc, 9));  // tokens 2c+8, 2c+9
            const float2 bs = __fadd2_rn(b0, b1);
            sv[cb] += bs.x + bs.y;
            uint32_t bh0, bl0, bh1, bl1;
            split_h2(b0.x, b0.y, bh0, bl0);
            split_h2(b1.x, b1.y, bh1, bl1);
            R0 = ob4(R0);
            R1 = ob4(R1);
            const uint32_t S0 = R0 >> 8, S1 = R1 >> 8;
            float(&a0)[4] = *reinterpret_cast<float(*)[4]>(&acc[8 * cb]);
            float(&a1)[4] = *reinterpret_cast<float(*)[4]>(&acc[8 * cb + 4]);
            const uint32_t x0 = u4_lo(R0), x1 = u4_hi(R0), x2 = u4_lo(R1), x3 = u4_hi(R1);
            const uint32_t y0 = u4_lo(S0), y1 = u4_hi(S0), y2 = u4_lo(S1), y3 = u4_hi(S1);
            mma16816(a0, x0, x1, x2, x3, bh0, bh1);
            mma16816(a1, y0, y1, y2, y3, bh0, bh1);
            mma16816(a0, x0, x1, x2, x3, bl0, bl1);
            mma16816(a1, y0, y1, y2, y3, bl0, bl1);
        };
#pragma unroll
        for (int cb2 = 0; cb2 < D / 64; ++cb2) {
            uint32_t r[4];
            ldsm_x4_t(plane_addr<PV::RB, PV::SWZ, PV::RP>(vc, LV, tr, 2 * cb2), r);
            chunk(2 * cb2, r[0], r[1]);
            chunk(2 * cb2 + 1, r[2], r[3]);
        }
        if constexpr (D % 64 != 0) {  // d = 96: the last 32-dim chunk alone
            uint32_t r[2];
            ldsm_x2_t(plane_addr<PV::RB, PV::SWZ, PV::RP>(vc, LV, tr, D / 32 - 1), r);
            chunk(D / 32 - 1, r[0], r[1]);
        }
    } else if constexpr (BV == 8) {
        // the half-1 columns carry nothing for 8-bit values
        const float cm = (g & 1) ? 0.f : 1.f;
        p00 *= cm;
        p10 *= cm;
        p01 *= cm;
        p11 *= cm;
#pragma unroll
        for (int s2 = 0; s2 < D / 32; ++s2) {
            uint32_t r[4];
            ldsm_x4_t(plane_addr<PV::RB, PV::SWZ, PV::RP>(vc, LV, tr, 2 * s2), r);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int cb = 2 * s2 + hh;
                const int gv = G == 16 ? cb >> 2 : (16 * cb) >> lg;
                const int fc = cb & 3;
                const float b00 = p00 * vsc(gv, fc, 0), b10 = p10 * vsc(gv, fc, 1), b01 = p01 * vsc(gv, fc, 8),
                            b11 = p11 * vsc(gv, fc, 9);
                sv[cb] += (b00 + b10) + (b01 + b11);
                uint32_t bh0, bl0, bh1, bl1;
                split_h2(b00, b10, bh0, bl0);
                split_h2(b01, b11, bh1, bl1);
                const uint32_t R0 = ob8(r[2 * hh]), R1 = ob8(r[2 * hh + 1]);
                float(&a0)[4] = *reinterpret_cast<float(*)[4]>(&acc[4 * cb]);
                const uint32_t x0 = u8_lo(R0), x1 = u8_lo(R0 >> 8), x2 = u8_lo(R1), x3 = u8_lo(R1 >> 8);
                mma16816(a0, x0, x1, x2, x3, bh0, bh1);
                mma16816(a0, x0, x1, x2, x3, bl0, bl1);
            }
        }
        if constexpr (D % 32 != 0) {  // d = 80: the last 16-dim chunk alone
            constexpr int cb = D / 16 - 1;
            uint32_t r[2];
            ldsm_x2_t(plane_addr<PV::RB, PV::SWZ, PV::RP>(vc, LV, tr, cb), r);
            const int gv = G == 16 ? cb >> 2 : (16 * cb) >> lg;
            const int fc = cb & 3;
            const float b00 = p00 * vsc(gv, fc, 0), b10 = p10 * vsc(gv, fc, 1), b01 = p01 * vsc(gv, fc, 8),
                        b11 = p11 * vsc(gv, fc, 9);
            sv[cb] += (b00 + b10) + (b01 + b11);
            uint32_t bh0, bl0, bh1, bl1;
            split_h2(b00, b10, bh0, bl0);
            split_h2(b01, b11, bh1, bl1);
            float(&a0)[4] = *reinterpret_cast<float(*)[4]>(&acc[4 * cb]);
            r[0] = ob8(r[0]);
            r[1] = ob8(r[1]);
            const uint32_t x0 = u8_lo(r[0]), x1 = u8_lo(r[0] >> 8), x2 = u8_lo(r[1]), x3 = u8_lo(r[1] >> 8);
            mma16816(a0, x0, x1, x2, x3, bh0, bh1);
            mma16816(a0, x0, x1, x2, x3, bl0, bl1);
        }
    } else {
        const float cm = (g & 1) ? 0.f : 1.f;
        uint32_t bh0, bl0, bh1, bl1;
        split_h2(p00 * cm, p10 * cm, bh0, bl0);
        split_h2(p01 * cm, p11 * cm, bh1, bl1);
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
            uint32_t r[4];
            ldsm_x4_t(plane_addr<PV::RB, PV::SWZ, PV::RP>(vc, LV, tr, 2 * j), r);
            if (tail) {  // raw fp16 rows past the end may hold anything: zero them in the A operand
                r[0] &= amask_lo;
                r[1] &= amask_lo;
                r[2] &= amask_hi;
                r[3] &= amask_hi;
            }
            float(&a0)[4] = *reinterpret_cast<float(*)[4]>(&acc[4 * j]);
            mma16816(a0, r[0], r[1], r[2], r[3], bh0, bh1);
            mma16816(a0, r[0], r[1], r[2], r[3], bl0, bl1);
        }
    }
}

// acc += V^T B for a 32-token chunk of int4 values read as 16 token pairs
// (d = 80).  The MMA's K index is the pair; per 16-byte segment sg the A rows
// of column half h (thread rows g < 4: h = 0) are dims of token parity
// (16 sg + 8h) / RB, so B[pair][n] = p(2 pair + parity, head n/2) *
// scale_V(that token, its group).  q[f][e][t] is p of token 2 (2c + e + 8f) + t
// for head g/2 (pairs 2c + e + 8f are this thread's K slots).  Segment sg
// accumulates into acc[8 sg .. 8 sg + 7] (acc_coord_pair maps them back).
template <int D, int G>
__device__ __forceinline__ void tile_pv_pair(uint32_t vc, const LaneRow& LV, const uint8_t* __restrict__ vsb, int sp,
                                             int lg, int lane, const float (&q)[2][2][2],
                                             float (&acc)[8 * PlaneT<D, 4>::NSEG], float (&sv)[PlaneT<D, 4>::NSEG]) {
    using PV = PlaneT<D, 4>;
    constexpr int RB = PV::RB, NSEG = PV::NSEG, PB = 2 * RB;
    const int g = lane >> 2, c = lane & 3, side = g & 1;
    const float* vs = reinterpret_cast<const float*>(vsb);
    auto seg = [&](int sg, uint32_t R0, uint32_t R1) {
        // this thread's column half is `side`: pair byte 16 sg + 8 side
        const int pb = 16 * sg + 8 * side;
        const int t = 16 * sg + 16 <= RB ? 0 : 16 * sg >= RB ? 1 : pb / RB;  // token parity (constant but for the straddling segment)
        const int f = (2 * (pb % RB)) >> lg;
        const float q00 = t ? q[0][0][1] : q[0][0][0], q10 = t ? q[0][1][1] : q[0][1][0];
        const float q01 = t ? q[1][0][1] : q[1][0][0], q11 = t ? q[1][1][1] : q[1][1][0];
        const int r0 = 4 * c + t;  // token of pair 2c
        const float b00 = q00 * vs[r0 * sp + f], b10 = q10 * vs[(r0 + 2) * sp + f];
        const float b01 = q01 * vs[(r0 + 16) * sp + f], b11 = q11 * vs[(r0 + 18) * sp + f];
        sv[sg] += (b00 + b10) + (b01 + b11);
        uint32_t bh0, bl0, bh1, bl1;
        split_h2(b00, b10, bh0, bl0);
        split_h2(b01, b11, bh1, bl1);
        R0 = ob4(R0);
        R1 = ob4(R1);
        const uint32_t S0 = R0 >> 8, S1 = R1 >> 8;
        float(&a0)[4] = *reinterpret_cast<float(*)[4]>(&acc[8 * sg]);
        float(&a1)[4] = *reinterpret_cast<float(*)[4]>(&acc[8 * sg + 4]);
        const uint32_t x0 = u4_lo(R0), x1 = u4_hi(R0), x2 = u4_lo(R1), x3 = u4_hi(R1);
        const uint32_t y0 = u4_lo(S0), y1 = u4_hi(S0), y2 = u4_lo(S1), y3 = u4_hi(S1);
        mma16816(a0, x0, x1, x2, x3, bh0, bh1);
        mma16816(a1, y0, y1, y2, y3, bh0, bh1);
        mma16816(a0, x0, x1, x2, x3, bl0, bl1);
        mma16816(a1, y0, y1, y2, y3, bl0, bl1);
    };
#pragma unroll
    for (int m2 = 0; m2 < NSEG / 2; ++m2) {
        uint32_t r[4];
        ldsm_x4_t(plane_addr<PB, false, PB>(vc, LV, 0, 2 * m2), r);
        seg(2 * m2, r[0], r[1]);
        seg(2 * m2 + 1, r[2], r[3]);
    }
    if constexpr (NSEG % 2 != 0) {
        uint32_t r[2];
        ldsm_x2_t(plane_addr<PB, false, PB>(vc, LV, 0, NSEG - 1), r);
        seg(NSEG - 1, r[0], r[1]);
    }
}

// Widen the raw fp16 / e8m0 scales of a staged chunk (rows of ng scales of
// sb bytes, contiguous) into the fp32 rows the compute reads: group 16 into
// the swizzled rows of d/4 bytes, other groups into plain rows of ng floats.
template <int D, int G>
__device__ __forceinline__ void widen_scales(const uint8_t* __restrict__ raw, uint8_t* __restrict__ dst, int rows,
                                             int ng, int sfmt, int lane) {
    if constexpr (G == 16 && D % 64 == 0) {
        // lane r widens row r: four scales (one 16-byte fp32 chunk) at a time
        constexpr int NG = D / 16, SRB = D / 4;
        if (lane < rows) {
#pragma unroll
            for (int j = 0; j < NG / 4; ++j) {
                float4 v;
                if (sfmt == SRFTKV_SCALE_FP16) {
                    const uint2 h = *reinterpret_cast<const uint2*>(raw + lane * NG * 2 + 8 * j);
                    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
                    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
                    v = make_float4(a.x, a.y, b.x, b.y);
                } else {
                    const uint32_t e = *reinterpret_cast<const uint32_t*>(raw + lane * NG + 4 * j);
                    v = make_float4(__uint_as_float((e & 0xFFu) << 23), __uint_as_float(((e >> 8) & 0xFFu) << 23),
                                    __uint_as_float(((e >> 16) & 0xFFu) << 23), __uint_as_float((e >> 24) << 23));
                }
                *reinterpret_cast<float4*>(dst + lane * SRB + (swz_chunk<SRB>(lane, j) << 4)) = v;
            }
        }
        return;
    }
    for (int i = lane; i < rows * ng; i += 32) {
        const int r = i / ng, f = i - r * ng;
        float v;
        if (sfmt == SRFTKV_SCALE_FP16)
            v = __half2float(__ushort_as_half(reinterpret_cast<const unsigned short*>(raw)[i]));
        else
            v = __uint_as_float((uint32_t)raw[i] << 23);  // e8m0: the byte is the fp32 exponent field
        uint32_t off;
        if constexpr (G == 16)
            off = (uint32_t)(r * (D / 4) + (swz_chunk<D / 4>(r, f >> 2) << 4) + (f & 3) * 4);
        else
            off = (uint32_t)((r * ng + f) * 4);
        *reinterpret_cast<float*>(dst + off) = v;
    }
}

// One chunk of NT 16-token sub-tiles starting at token t0 of the sequence:
// scores for all NT*16 tokens, one online-softmax update, then P.V.
// G: the group size when known at compile time (16, the common case: all
// scale-row indexing becomes immediate offsets), or 0 to read it from P.
template <int D, int BK, int BV, int NT, int G>
__device__ __forceinline__ void attn_chunk(const AttnParams& P, uint8_t* __restrict__ stage, int t0, int t_end, int lane,
                                           const LaneRow& LK, const LaneRow& LV,
                                           const uint32_t (&kso)[scale_chunks<D>()],
                                           const uint32_t (&vso)[scale_chunks<D>()],
                                           const uint32_t (&qh)[AttnCfg<D, BK, BV>::QB],
                                           const uint32_t (&ql)[AttnCfg<D, BK, BV>::QB],
                                           const float (&nb)[AttnCfg<D, BK, BV>::NB],
                                           const uint4* __restrict__ qf, int nh,
                                           float (&acc)[AttnCfg<D, BK, BV>::ACC],
                                           float (&sv)[AttnCfg<D, BK, BV>::NSV], float& svt, float& m, float& l,
                                           float mu) {
    using C = AttnCfg<D, BK, BV>;
    constexpr float SU = C::QK ? kSub : 1.f;  // scores come in units of 1/SU
    const int g = lane >> 2, c = lane & 3;
    const uint32_t kc = ptx::smem_u32(stage + C::OFF_KC), vc = ptx::smem_u32(stage + C::OFF_VC);
    float* ks = reinterpret_cast<float*>(stage + C::OFF_KS);
    float* vs = reinterpret_cast<float*>(stage + C::OFF_VS);
    const int sp = G ? D / G : P.sp;  // floats per scale row
    if ((C::QK && P.sf_k != SRFTKV_SCALE_FP32) || (C::QV && P.sf_v != SRFTKV_SCALE_FP32)) {
        if (C::QK && P.sf_k != SRFTKV_SCALE_FP32)
            widen_scales<D, G>(stage + C::OFF_KR, stage + C::OFF_KS, 16 * NT, sp, P.sf_k, lane);
        if (C::QV && P.sf_v != SRFTKV_SCALE_FP32)
            widen_scales<D, G>(stage + C::OFF_VR, stage + C::OFF_VS, 16 * NT, sp, P.sf_v, lane);
        __syncwarp();
    }
    const int lg = G == 16 ? 4 : G == 32 ? 5 : G == 64 ? 6 : P.log2_group;
    const int valid = t_end - t0;  // tokens of this chunk inside the sequence (> 0)
    const bool tail = valid < 16 * NT;
    if (tail && (C::QK || C::QV)) {
        // scale rows past the end may hold anything: zero them so they contribute exact zeros
        for (int i = valid * sp + lane; i < 16 * NT * sp; i += 32) {
            if (C::QK) ks[i] = 0.f;
            if (C::QV) vs[i] = 0.f;
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
    }

    // this thread's head is c; s[st][r] holds token 16st + g + 8r (rows of tokens), or token 16st + 2g + r
    // (rows of token pairs)
    float s[NT][2];
    if constexpr (C::PK) {
        tile_scores_pair<D, G>(kc, LK, stage + C::OFF_KS, sp, lg, lane, qh, ql, nb, s);
        if (tail) {
#pragma unroll
            for (int st = 0; st < NT; ++st)
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    if (16 * st + 2 * g + r >= valid) s[st][r] = -INFINITY;
        }
    } else {
#pragma unroll
        for (int st = 0; st < NT; ++st) {
            if (16 * st < valid)
                tile_scores<D, BK, G>(kc, LK, stage + C::OFF_KS, kso, sp, lg, 16 * st, lane, qh, ql, nb, qf, s[st]);
            else s[st][0] = s[st][1] = 0.f;
            if (tail) {
                if (16 * st + g >= valid) s[st][0] = -INFINITY;
                if (16 * st + g + 8 >= valid) s[st][1] = -INFINITY;
            }
        }
    }
    // ---- online softmax (log2 domain) ----
    // The running max m only has to move when some score of the chunk exceeds
    // it; that is tested per thread and voted, and only then is the head max
    // reduced over the 8 token rows and the state rescaled.
    float mt = -INFINITY;
#pragma unroll
    for (int st = 0; st < NT; ++st) mt = fmaxf(mt, fmaxf(s[st][0], s[st][1]));
    mt *= SU;
    if (__any_sync(0xffffffffu, mt > m)) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        const float mn = fmaxf(m, mt);
        const float f = (mn == -INFINITY) ? 1.f : ex2(m - mn);  // head c's factor
        l *= f;
        svt *= f;
#pragma unroll
        for (int i = 0; i < C::ACC; ++i) acc[i] *= f;
        const float fs = __shfl_sync(0xffffffffu, f, g >> 1);  // head g/2's factor, for the column sums
#pragma unroll
        for (int i = 0; i < C::NSV; ++i) sv[i] *= fs;
        m = mn;
    }
    // p in [0, 256 * 2^-mu] (mu: the warp's V unit, 0 unless the V scales are far from 1): the +8 keeps
    // p * scale_V clear of fp16 subnormals; it cancels in acc / l
    const float bias = (m == -INFINITY) ? 0.f : m - 8.f + mu;
    const bool offer = c < nh;  // padded heads offer zero
    const int hd = g >> 1;         // head of this thread's B columns
    if constexpr (C::PV) {
        // all p of the chunk first; q[f][e][t]: token 4c + 2e + 16f + t for head hd
        float o[NT][2];
#pragma unroll
        for (int st = 0; st < NT; ++st)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float pv = ex2(fmaf(s[st][r], SU, -bias));  // 0 for masked tokens
                l += pv;
                o[st][r] = offer ? pv : 0.f;
            }
        float q[2][2][2];
#pragma unroll
        for (int f = 0; f < 2; ++f)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if constexpr (C::PK) {  // token 16f + 2(2c + e) + t sits in pair row 2c + e, register [f][t]
                        q[f][e][t] = __shfl_sync(0xffffffffu, o[f][t], 4 * (2 * c + e) + hd);
                    } else {  // token 16f + u, u = 4c + 2e + t: row u % 8, register [f][u / 8] with u / 8 = c / 2
                        const int src = 4 * ((4 * c + 2 * e + t) & 7) + hd;
                        const float lo = __shfl_sync(0xffffffffu, o[f][0], src);
                        const float hi = __shfl_sync(0xffffffffu, o[f][1], src);
                        q[f][e][t] = (c >> 1) ? hi : lo;
                    }
                }
        tile_pv_pair<D, G>(vc, LV, stage + C::OFF_VS, sp, lg, lane, q, acc, sv);
    } else {
#pragma unroll
    for (int st = 0; st < NT; ++st) {
        if (16 * st >= valid) break;
        const float p0 = ex2(fmaf(s[st][0], SU, -bias)), p1 = ex2(fmaf(s[st][1], SU, -bias));
        l += p0 + p1;
        const float o0 = offer ? p0 : 0.f, o1 = offer ? p1 : 0.f;
        float P00, P10, P01, P11;
        if constexpr (C::PK) {  // token 16st + 2c + e + 8f sits in pair row c + 4f, register [st][e]
            P00 = __shfl_sync(0xffffffffu, o0, 4 * c + hd);
            P10 = __shfl_sync(0xffffffffu, o1, 4 * c + hd);
            P01 = __shfl_sync(0xffffffffu, o0, 4 * (c + 4) + hd);
            P11 = __shfl_sync(0xffffffffu, o1, 4 * (c + 4) + hd);
        } else {
            P00 = __shfl_sync(0xffffffffu, o0, 4 * (2 * c) + hd);
            P10 = __shfl_sync(0xffffffffu, o0, 4 * (2 * c + 1) + hd);
            P01 = __shfl_sync(0xffffffffu, o1, 4 * (2 * c) + hd);
            P11 = __shfl_sync(0xffffffffu, o1, 4 * (2 * c + 1) + hd);
        }
        const int vt = valid - 16 * st;
        const bool sub_tail = vt < 16;
        const uint32_t mlo = (2 * c < vt ? 0x0000FFFFu : 0u) | (2 * c + 1 < vt ? 0xFFFF0000u : 0u);
        const uint32_t mhi = (2 * c + 8 < vt ? 0x0000FFFFu : 0u) | (2 * c + 9 < vt ? 0xFFFF0000u : 0u);
        tile_pv<D, BV, G>(vc, LV, stage + C::OFF_VS, vso, sp, lg, 16 * st, lane, P00, P10, P01, P11, mlo, mhi,
                          sub_tail, acc, sv);
    }
    }
}

// Where accumulator entry i of thread (g, c) lives: dim and head (column) and
// whether it is meaningful.
template <int D, int BV>
__device__ __forceinline__ void acc_coord(int i, int g, int c, int& dim, int& head, bool& useful) {
    const int e = i & 3;
    head = c;  // columns 2c, 2c+1 are (head c, half 0), (head c, half 1)
    if constexpr (BV == 4) {
        const int cb = i >> 3, j = (i >> 2) & 1;
        dim = 32 * cb + 4 * g + 2 * j + (e >> 1);
        useful = (e & 1) == (g >= 4 ? 1 : 0);  // rows g < 4 are dims of half 0
    } else if constexpr (BV == 8) {
        const int cb = i >> 2;
        dim = 16 * cb + 2 * g + (e >> 1);
        useful = (e & 1) == 0;
    } else {
        const int j = i >> 2;
        dim = 16 * j + g + 8 * (e >> 1);
        useful = (e & 1) == 0;
    }
}

// The same for int4 values read as token pairs: accumulator i = 8 sg + 4j + e
// of thread (g, c) is head c, column half e % 2, A row g (+ 8 for e >= 2) of
// segment sg's x (j = 0) or y (j = 1) MMA: nibble e / 2 of pair byte
// 16 sg + 2g + j, i.e. token parity par and dim 2 (byte mod RB) + e / 2.
template <int D>
__device__ __forceinline__ void acc_coord_pair(int i, int g, int c, int& dim, int& head, bool& useful, int& par) {
    constexpr int RB = PlaneT<D, 4>::RB;
    const int sg = i >> 3, j = (i >> 2) & 1, e = i & 3;
    const int pb = 16 * sg + 2 * g + j;
    head = c;
    par = pb >= RB ? 1 : 0;
    dim = 2 * (pb - par * RB) + (e >> 1);
    useful = (e & 1) == (g >= 4 ? 1 : 0);  // rows g < 4 are bytes 0-7 of the segment: column half 0
}

// Grid (n_splits, B * Hkv * n_hg): CTA (split, (b, kv head, head group)).
// A head group is up to four query heads of one kv head (the MMA columns
// carry four heads); GQA ratios above four run as several head groups, whose
// CTAs sit next to each other in the launch order so that the second one's
// reads of the same cache rows are mostly L2 hits.
// d = 256 keeps 2 CTAs per SM (its fragments need more than a third of the register file), and so does
// d = 192 with 32-token chunks (their stages fit two CTAs' shared memory); every other instance 3
template <int D, int BK, int BV, int G>
__global__ void __launch_bounds__(kAttnWarps * 32, AttnCfg<D, BK, BV>::MINB)
    q4kv_attn_split_kernel(const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_ks,
                           const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_vs,
                           const __grid_constant__ AttnParams P) {
    using C = AttnCfg<D, BK, BV>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // swizzled TMA destinations need 1024-byte alignment: realign (offsetting
    // the shared array keeps every access in the shared window)
    uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    // the warp index through a shuffle, so the compiler knows it is warp-uniform
    // (barrier and TMA operands then stay in uniform registers)
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int bhg = blockIdx.y, hg = bhg % P.n_hg, bh = bhg / P.n_hg;
    const int b = bh / P.Hkv, hkv = bh - b * P.Hkv;
    const int h0 = hg * P.hpg, nh = min(P.hpg, P.rep - h0);  // this CTA's query heads: h0 .. h0 + nh - 1
    const int split = blockIdx.x;
    const int L = P.seq_lens ? min(max(P.seq_lens[b], 0), P.t_cap) : P.t_cap;
    const int n_chunks = (L + C::CH - 1) / C::CH;
    const int cps = (n_chunks + P.n_splits - 1) / P.n_splits;
    const int c_begin = split * cps, c_end = min(c_begin + cps, n_chunks);

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BARS);  // 4 per warp
    uint8_t* wbase = smem + warp * C::WARP_BYTES;
    constexpr int NS = C::NS;
    static_assert(NS >= 2 && NS <= 4, "stages per warp");
    if (lane == 0) {
#pragma unroll
        for (int s2 = 0; s2 < NS; ++s2) ptx::mbar_init(ptx::smem_u32(&bars[4 * warp + s2]), 1);
        ptx::fence_barrier_init();
    }
    __syncwarp();
    auto barw = [&](int s2) { return ptx::smem_u32(&bars[4 * warp + s2]); };

    uint32_t qh[C::QB], ql[C::QB];
    float nb[C::NB];
    // per-lane shared-memory addressing of the plane images
    using PK = PlaneT<D, BK>;
    using PV = PlaneT<D, BV>;
    // (pair planes: rows of 2 RB bytes)
    const LaneRow LK = PK::PAIR ? lane_row_codes<2 * PK::RB, false, 2 * PK::RB>(lane)
                                : lane_row_codes<PK::RB, PK::SWZ, PK::RP>(lane);
    const LaneRow LV = PV::PAIR   ? lane_row_codes<2 * PV::RB, false, 2 * PV::RB>(lane)
                       : BV == 16 ? lane_row_v16<PV::RB, PV::SWZ, PV::RP>(lane)
                                  : lane_row_codes<PV::RB, PV::SWZ, PV::RP>(lane);
    constexpr int SCH = scale_chunks<D>();
    uint32_t kso[SCH], vso[SCH];
    scale_offsets<D, SCH>(g, 0, kso);                               // K: row g (and g + 8)
    scale_offsets<D, SCH>(2 * c, BV == 4 ? 4 * (g & 1) : 0, vso);  // V: rows 2c (+1, +8, +9), column half
    float acc[C::ACC], sv[C::NSV], svt = 0.f;
    float m = -INFINITY, l = 0.f;  // online-softmax state for head c (log2 domain)

    const int plane_row = b * P.Hkv + hkv;  // this (batch, kv head)'s rows in the head-major planes
    const uint32_t kc_bytes = C::CH * PlaneT<D, BK>::RP, vc_bytes = C::CH * PlaneT<D, BV>::RP;
    // exact rows of d/group scales: fp32 into the compute rows, fp16 / e8m0 raw into their own area
    const uint32_t ks_bytes = C::CH * P.sp * (P.sf_k == SRFTKV_SCALE_FP32 ? 4 : P.sf_k == SRFTKV_SCALE_FP16 ? 2 : 1);
    const uint32_t vs_bytes = C::CH * P.sp * (P.sf_v == SRFTKV_SCALE_FP32 ? 4 : P.sf_v == SRFTKV_SCALE_FP16 ? 2 : 1);
    const int ks_off = P.sf_k == SRFTKV_SCALE_FP32 ? C::OFF_KS : C::OFF_KR;
    const int vs_off = P.sf_v == SRFTKV_SCALE_FP32 ? C::OFF_VS : C::OFF_VR;
    // fp16 / e8m0 planes, and every plane of a d that is not a power of two (whose
    // scale rows are not a multiple of 16 bytes), are addressed as rows of 16
    // bytes: the chunk's first one; fp32 rows of a power-of-two d as rows
    const bool kflat = !pow2_dim<D>() || P.sf_k != SRFTKV_SCALE_FP32;
    const bool vflat = !pow2_dim<D>() || P.sf_v != SRFTKV_SCALE_FP32;
    const int ks_row = kflat ? (int)(ks_bytes / 16) : 1;
    const int vs_row = vflat ? (int)(vs_bytes / 16) : 1;
    const uint32_t tx = kc_bytes + vc_bytes + (C::QK ? ks_bytes : 0) + (C::QV ? vs_bytes : 0);
    auto issue = [&](int chunk, int st) {
        const uint32_t bar = barw(st);
        uint8_t* dst = wbase + st * C::STAGE;
        const int tok = chunk * C::CH;
        ptx::mbar_arrive_expect_tx(bar, tx);
        // (pair planes: rows of two tokens)
        ptx::tma_load_3d(ptx::smem_u32(dst + C::OFF_KC), &tm_kc, bar, 0, C::PK ? tok / 2 : tok, plane_row);
        if constexpr (C::QK)
            ptx::tma_load_3d(ptx::smem_u32(dst + ks_off), &tm_ks, bar, 0, kflat ? chunk * ks_row : tok, plane_row);
        ptx::tma_load_3d(ptx::smem_u32(dst + C::OFF_VC), &tm_vc, bar, 0, C::PV ? tok / 2 : tok, plane_row);
        if constexpr (C::QV)
            ptx::tma_load_3d(ptx::smem_u32(dst + vs_off), &tm_vs, bar, 0, vflat ? chunk * vs_row : tok, plane_row);
    };

    // per-warp ring of NS stages: iteration it (counted over both passes below)
    // uses stage it % NS; NS-1 chunks are in flight
    auto prologue = [&](int it0) {
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < NS - 1; ++j)
                if (c_begin + warp + j * kAttnWarps < c_end) issue(c_begin + warp + j * kAttnWarps, (it0 + j) % NS);
        }
    };
    // The cache copies do not depend on the q preparation, which may still be
    // running (the kernel is launched as its programmatic dependent): the first
    // chunks go out first, the prepared q is read after griddep_wait.
    prologue(0);
    griddep_wait();
    if constexpr (C::PK)
        build_qb_pair<D>(P.qt + ((long long)b * P.Hq + (long long)hkv * P.rep + h0) * D, nh, g, c, qh, ql, nb);
    else
        build_qb<D, BK>(P.qt + ((long long)b * P.Hq + (long long)hkv * P.rep + h0) * D, nh, g, c, qh, ql, nb);
    uint4* qf = reinterpret_cast<uint4*>(smem + C::OFF_QF);  // (read only when q_in_smem)
    if constexpr (C::QSM) {
        // every warp built the same fragments (same query heads, same lane layout): warp 0 stores them
        if (warp == 0) {
            float2* qn = reinterpret_cast<float2*>(qf + 2 * (D / 32) * 32);
#pragma unroll
            for (int mm = 0; mm < D / 32; ++mm) {
                qf[mm * 32 + lane] = make_uint4(qh[4 * mm], qh[4 * mm + 1], qh[4 * mm + 2], qh[4 * mm + 3]);
                qf[(D / 32 + mm) * 32 + lane] = make_uint4(ql[4 * mm], ql[4 * mm + 1], ql[4 * mm + 2], ql[4 * mm + 3]);
                qn[mm * 32 + lane] = make_float2(nb[2 * mm], nb[2 * mm + 1]);
            }
        }
        __syncthreads();
    }

    // V unit.  P.V takes B = p * scale_V in fp16 with p <= 256 * 2^-mu, l and acc
    // accumulating in that unit, and the (m, l) the warp exports carry m + mu.
    // The first pass takes mu = 0, right for V scales of ordinary size.  A warp
    // whose pass overflowed (a non-finite accumulator: some scale_V * p at or
    // above 65520) or whose p-weighted mean V scale is below 2^-14 in every
    // head (the low fp16 halves of B would fall into subnormals) runs its
    // chunks once more with mu = (exponent of its largest V scale) - 6, read
    // from the scale plane, so that every B is below 2^15.
    float mu = 0.f;
    bool failed = false, undrained = false;
    int it = 0;
    // ss[i] = the sum over the 16 token slots of B's column held by this thread's
    // useful accumulators (head c; for 4-bit values its column half), in chunk i
    auto column_sums = [&](float (&ss)[C::NSV]) {
#pragma unroll
        for (int i = 0; i < C::NSV; ++i) {
            float t = sv[i];
            t += __shfl_xor_sync(0xffffffffu, t, 1);
            t += __shfl_xor_sync(0xffffffffu, t, 2);  // column g's sum
            const int col = BV == 4 ? 2 * c + (g >= 4 ? 1 : 0) : 2 * c;
            ss[i] = __shfl_sync(0xffffffffu, t, 4 * col);
        }
    };
    // acc holds sums of (code + offset) * B in the code unit.  Taking the offset
    // times the column sums out every kFoldChunks chunks (and resetting them)
    // keeps acc near the size of its signal: over a long run of chunks the
    // offset part grows far larger than the signal and its fp32 accumulation in
    // the MMAs would lose the signal's low bits when it cancels at the end.
    // svt keeps the column's running total of B for the V-range test.
    auto fold_offset = [&]() {
        if constexpr (C::QV) {
            float ss[C::NSV];
            column_sums(ss);
#pragma unroll
            for (int i = 0; i < C::NSV; ++i) {
                svt += ss[i];
                sv[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < C::ACC; ++i) {
                if constexpr (BV == 4) {
                    const float iu = ((i >> 1) & 1) ? -8.f / 1048576.f : -8.f / kSub;  // high-nibble rows: 2^-20
                    acc[i] = fmaf(iu, ss[i >> 3], acc[i]);
                } else {
                    acc[i] = fmaf(-128.f / kSub, ss[i >> 2], acc[i]);
                }
            }
        }
    };
    // one pass over this warp's chunks with V unit 2^mu_p (the first pass is called with a literal 0, so its
    // loop is the plain one; the rare second pass is a separate copy)
    auto run_pass = [&](float mu_p) {
#pragma unroll
        for (int i = 0; i < C::ACC; ++i) acc[i] = 0.f;
#pragma unroll
        for (int i = 0; i < C::NSV; ++i) sv[i] = 0.f;
        svt = 0.f;
        m = -INFINITY;
        l = 0.f;
        for (int chunk = c_begin + warp; chunk < c_end; ++it, chunk += kAttnWarps) {
            const int st = it % NS;
            const int nxt = chunk + (NS - 1) * kAttnWarps;
            if (lane == 0 && nxt < c_end) issue(nxt, (it + NS - 1) % NS);
            const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(barw(st), (it / NS) & 1, P.poll_limit));
            if (!ok) {
                if (lane == 0) {
                    atomicOr(&g_attn_fault, 1u);
                    // let this warp's copies in flight land (this stage's included) before giving up; a copy
                    // that still has not landed keeps the CTA away from its shared memory below
                    bool all = true;
                    for (int j = 0; j < NS; ++j)
                        if (chunk + j * kAttnWarps < c_end)
                            all &= ptx::mbar_wait_bounded(barw((it + j) % NS), ((it + j) / NS) & 1, 1u << 16);
                    undrained = !all;
                }
                undrained = __shfl_sync(0xffffffffu, undrained, 0);
                failed = true;
                break;
            }
            attn_chunk<D, BK, BV, C::CH / 16, G>(P, wbase + st * C::STAGE, chunk * C::CH, L, lane, LK, LV, kso, vso,
                                                 qh, ql, nb, qf, nh, acc, sv, svt, m, l, mu_p);
            __syncwarp();
            if ((it & (kFoldChunks - 1)) == kFoldChunks - 1) fold_offset();
        }
    };
    run_pass(0.f);
    if (C::QV && !failed) {
        bool redo;
        {
            bool bad = !isfinite(l) || !isfinite(svt);
#pragma unroll
            for (int i = 0; i < C::ACC; ++i) bad |= !isfinite(acc[i]);
#pragma unroll
            for (int i = 0; i < C::NSV; ++i) bad |= !isfinite(sv[i]);
            redo = __any_sync(0xffffffffu, bad);
            if (!redo) {
                // p-weighted mean V scale of this thread's column (head c, its half), averaged over the
                // column's groups, against 2^-14
                float lt = l, ss[C::NSV], tot = svt;
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
                column_sums(ss);
#pragma unroll
                for (int i = 0; i < C::NSV; ++i) tot += ss[i];
                const bool counts = c < nh && lt > 0.f;
                redo = __any_sync(0xffffffffu, counts) &&
                       __all_sync(0xffffffffu, !counts || tot < (float)C::NSV * lt * 6.103515625e-05f);
            }
        }
        if (redo) {
            // the largest V scale of this warp's chunks, from the scale plane
            const int sbv = P.sf_v == SRFTKV_SCALE_FP32 ? 4 : P.sf_v == SRFTKV_SCALE_FP16 ? 2 : 1;
            const uint8_t* vsrc = P.vscale + (size_t)plane_row * P.t_cap * P.sp * sbv;
            uint32_t vmax = 0u;
            for (int ch = c_begin + warp; ch < c_end; ch += kAttnWarps) {
                const int t = ch * C::CH + lane;
                if (lane < C::CH && t < L) {
                    const uint8_t* row = vsrc + (size_t)t * P.sp * sbv;
                    for (int f = 0; f < P.sp; ++f) {
                        float v;
                        if (P.sf_v == SRFTKV_SCALE_FP32) v = __ldg(reinterpret_cast<const float*>(row) + f);
                        else if (P.sf_v == SRFTKV_SCALE_FP16) v = __half2float(__ldg(reinterpret_cast<const __half*>(row) + f));
                        else v = __uint_as_float((uint32_t)__ldg(row + f) << 23);
                        vmax = max(vmax, __float_as_uint(fabsf(v)));
                    }
                }
            }
            vmax = __reduce_max_sync(0xffffffffu, vmax);
            int un = vmax ? (int)(vmax >> 23) - 127 - 6 : 0;
            un = min(max(un, -110), 120);  // p = 2^(8 - mu) .. stays a finite fp32 number
            if (un != 0) {
                mu = (float)un;
                prologue(it);
                run_pass(mu);
            }
        }
    }
    // the combine may start launching once every CTA is this far (it waits for the grid's end); signalling
    // earlier lets its CTAs sit on the SMs through the whole run when the grid is a single wave
    griddep_launch_dependents();
    // the failure flag is per warp; every warp still joins the merge below
    if (failed) {
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int i = 0; i < C::ACC; ++i) acc[i] = 0.f;
#pragma unroll
        for (int i = 0; i < C::NSV; ++i) sv[i] = 0.f;
    }

    // ---- remove the code offset: acc holds sums of (code + offset) * B in the
    // code unit; the column sums of B (this thread's useful column) give the rest
    float ssum[C::NSV];
    column_sums(ssum);
#pragma unroll
    for (int i = 0; i < C::ACC; ++i) {
        if constexpr (BV == 4) {
            const float unit = ((i >> 1) & 1) ? 1048576.f : kSub;  // high-nibble rows: 2^-20
            acc[i] = fmaf(unit, acc[i], -8.f * ssum[i >> 3]);
        } else if constexpr (BV == 8) {
            acc[i] = fmaf(kSub, acc[i], -128.f * ssum[i >> 2]);
        }
    }

    // ---- per-warp totals of l over the 8 token rows ----
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    const long long prow0 = (long long)b * P.Hq + (long long)hkv * P.rep + h0;
    // all warps are done with their stage buffers; a copy that never landed keeps them all out of shared memory
    if (__syncthreads_or(undrained ? 1 : 0)) {
        for (int idx = threadIdx.x; idx < nh * D; idx += blockDim.x) {
            const int h = idx / D, dim = idx - h * D;
            const long long pidx = (prow0 + h) * P.n_splits + split;
            P.part_acc[pidx * D + dim] = 0.f;
            if (dim == 0) {
                P.part_ml[pidx * 2] = -INFINITY;
                P.part_ml[pidx * 2 + 1] = 0.f;
            }
        }
        return;
    }
    float* mw = reinterpret_cast<float*>(smem);                 // [warps][4][2]
    float* aw = mw + kAttnWarps * 8;                            // [warps][4][D]
    if (g == 0) {
        mw[warp * 8 + c * 2 + 0] = m == -INFINITY ? m : m + mu;  // the state is in the unit 2^-(m + mu - 8)
        mw[warp * 8 + c * 2 + 1] = l;
    }
#pragma unroll
    for (int i = 0; i < C::ACC; ++i) {
        int dim, head;
        bool useful;
        if constexpr (C::PV) {  // the even tokens' entries (one per dim and head) first, the odd ones added below
            int par;
            acc_coord_pair<D>(i, g, c, dim, head, useful, par);
            if (useful && par == 0) aw[(warp * 4 + head) * D + dim] = acc[i];
        } else {
            acc_coord<D, BV>(i, g, c, dim, head, useful);
            if (useful) aw[(warp * 4 + head) * D + dim] = acc[i];
        }
    }
    if constexpr (C::PV) {
        __syncwarp();
#pragma unroll
        for (int i = 0; i < C::ACC; ++i) {
            int dim, head, par;
            bool useful;
            acc_coord_pair<D>(i, g, c, dim, head, useful, par);
            if (useful && par == 1) aw[(warp * 4 + head) * D + dim] += acc[i];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nh * D; idx += blockDim.x) {
        const int h = idx / D, dim = idx - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, mw[w * 8 + h * 2]);
        float Lsum = 0.f, A = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) {
                const float f = ex2(mw[w * 8 + h * 2] - M);
                Lsum += f * mw[w * 8 + h * 2 + 1];
                A += f * aw[(w * 4 + h) * D + dim];
            }
        }
        const long long pidx = (prow0 + h) * P.n_splits + split;
        P.part_acc[pidx * D + dim] = A;
        if (dim == 0) {
            P.part_ml[pidx * 2] = M;
            P.part_ml[pidx * 2 + 1] = Lsum;
        }
    }
}

// ---------------------------------------------------------------------------
// 3. combine
// ---------------------------------------------------------------------------
// One block of four warps per output row (b, hq).  Merge: every warp takes
// the running max M over the splits (split s in lane s mod 32), then warp w
// accumulates splits w, w + 4, ... (dims lane + 32 j); the four partial rows
// meet in shared memory.  Inverse SRFT x = diag(s) R^T p: warp w takes the
// frequencies f = 1 + w + 4 i and lane the coordinates k = lane + 32 j,
// walking f with the table index f k mod D; the DC and Nyquist terms are added
// in the final sum.  SRHT: the Walsh-Hadamard transform across one warp.
template <int D, bool ROT>
__global__ void __launch_bounds__(128) attn_combine_kernel(const __grid_constant__ AttnParams P) {
    constexpr int PER = (D + 31) / 32;  // dims lane + 32 j (the last j partial at d = 80)
    __shared__ __align__(16) float rows[D];
    __shared__ float part[4][D], lw[4];
    __shared__ float tcs[ROT ? D : 1], tsn[ROT ? D : 1];
    const bool srht = ROT && pow2_dim<D>() && P.tr_v == SRFTKV_TRANSFORM_SRHT;
    if (ROT && !srht) dft_tables<D>(tcs, tsn);
    griddep_wait();  // launched as the split kernel's programmatic dependent: its partials first
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x;  // (b, hq)
    const int b = row / P.Hq, hq = row - b * P.Hq, hkv = hq / P.rep;
    const int ns = P.n_splits;
    const float* ml = P.part_ml + (long long)row * ns * 2;
    const float* ac = P.part_acc + (long long)row * ns * D;
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f, o[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) o[j] = 0.f;
    if (M != -INFINITY) {
#pragma unroll 4
        for (int s = warp; s < ns; s += 4) {
            const float2 e = *reinterpret_cast<const float2*>(ml + 2 * s);
            const float w = ex2(e.x - M);  // 0 for empty splits
            L = fmaf(w, e.y, L);
            const float* a = ac + (long long)s * D + lane;
#pragma unroll
            for (int j = 0; j < PER; ++j)
                if (lane + 32 * j < D) o[j] = fmaf(w, a[32 * j], o[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < PER; ++j)
        if (lane + 32 * j < D) part[warp][lane + 32 * j] = o[j];
    if (lane == 0) lw[warp] = L;
    __syncthreads();
    const float Lsum = (lw[0] + lw[1]) + (lw[2] + lw[3]);
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    float* yr = P.out + (long long)row * D;
    for (int t = threadIdx.x; t < D; t += blockDim.x) {
        float v = ((part[0][t] + part[1][t]) + (part[2][t] + part[3][t])) * inv;
        if (ROT && P.lam_v != nullptr) v *= __frcp_rn(P.lam_v[(long long)b * P.lam_v_stride + (long long)hkv * D + t]);
        if (ROT) rows[t] = v;
        else yr[t] = v;
    }
    if constexpr (ROT) {
        __syncthreads();
        const float isd = rsqrtf((float)D);
        if constexpr (pow2_dim<D>()) {
            if (srht) {  // x = diag(s) H p / sqrt(D)
                if (warp != 0) return;
                float v[D / 32];
#pragma unroll
                for (int j = 0; j < D / 32; ++j) v[j] = rows[32 * j + lane];
                wht_warp<D>(v, lane);
#pragma unroll
                for (int j = 0; j < D / 32; ++j) {
                    const int k = 32 * j + lane;
                    const float a = v[j] * isd;
                    yr[k] = sign_neg(P.sign_mask, k) ? -a : a;
                }
                return;
            }
        }
        float a[PER];
        int m[PER], st[PER];
        const int f0 = 1 + warp;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int k = min(lane + 32 * j, D - 1);  // lanes past D (d = 80) compute a coordinate nobody stores
            a[j] = 0.f;
            m[j] = (f0 * k) % D;
            st[j] = (4 * k) % D;
        }
#pragma unroll 4
        for (int f = f0; f < D / 2; f += 4) {
            const float2 pf = *reinterpret_cast<const float2*>(rows + 2 * f);
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                a[j] = fmaf(tcs[m[j]], pf.x, a[j]);
                a[j] = fmaf(tsn[m[j]], pf.y, a[j]);
                m[j] = mod_add<D>(m[j], st[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if (lane + 32 * j < D) part[warp][lane + 32 * j] = a[j];
        __syncthreads();
        for (int k = threadIdx.x; k < D; k += blockDim.x) {
            const float x = ((part[0][k] + part[1][k]) + (part[2][k] + part[3][k])) +
                            isd * (rows[0] + ((k & 1) ? -rows[1] : rows[1]));
            yr[k] = sign_neg(P.sign_mask, k) ? -x : x;
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// A plane [B*Hkv][t_cap][row] (head-major: the rows of one (batch, kv head)
// are contiguous); a box is box_rows consecutive tokens of box_inner elements
// (the whole row, or the row plus zero-filled padding for unswizzled code rows
// longer than 128 bytes).
static bool encode_plane(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int inner_elems, int elem_bytes,
                         int box_inner, long long bh, int t_cap, int box_rows, CUtensorMapSwizzle swz) {
    const unsigned long long dims[3] = {(unsigned long long)inner_elems, (unsigned long long)t_cap,
                                        (unsigned long long)bh};
    const unsigned long long strides[2] = {(unsigned long long)inner_elems * elem_bytes,
                                           (unsigned long long)inner_elems * elem_bytes * t_cap};
    const unsigned box[3] = {(unsigned)box_inner, (unsigned)box_rows, 1u};
    return encode_tiled_swz(map, dt, 3, const_cast<void*>(base), dims, strides, box, swz, "attention cache plane");
}
static CUtensorMapSwizzle swizzle_for(int row_bytes) {
    return row_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
           : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
           : row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                              : CU_TENSOR_MAP_SWIZZLE_NONE;
}
template <int D, int BITS>
static bool encode_codes(CUtensorMap* map, const void* base, long long bh, int t_cap, int rows) {
    using PT = PlaneT<D, BITS>;
    if (PT::PAIR)  // rows of two tokens (t_cap even, checked by attention_check)
        return encode_plane(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2 * PT::RB, 1, 2 * PT::RB, bh, t_cap / 2,
                            rows / 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (PT::SWZ)
        return encode_plane(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, PT::RB, 1, PT::RB, bh, t_cap, rows,
                            swizzle_for(PT::RB));
    return encode_plane(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT32, PT::RB / 4, 4, PT::RP / 4, bh, t_cap, rows,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
}

struct AttnLaunch {
    AttnParams P;
    const srftkv_side* k;
    const srftkv_side* v;
    int d;
    cudaStream_t stream;
};

// Launch as the programmatic dependent of the kernel before it in the stream:
// it may start while that one finishes and waits for it with griddep_wait
// (the split kernel after the q preparation, the combine after the split).
template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                    Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// the split kernel's dynamic shared memory limit, once per instance
template <int D, int BK, int BV, int G>
static void split_kernel_attr() {
    static bool done = false;
    if (!done) {
        cudaFuncSetAttribute(q4kv_attn_split_kernel<D, BK, BV, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AttnCfg<D, BK, BV>::SMEM);
        done = true;
    }
}

template <int D, int BK, int BV>
static int launch_split(const AttnLaunch& A) {
    using C = AttnCfg<D, BK, BV>;
    const AttnParams& P = A.P;
    const long long bh = (long long)P.B * P.Hkv;
    CUtensorMap tkc, tks, tvc, tvs;
    if (!encode_codes<D, BK>(&tkc, A.k->codes, bh, P.t_cap, C::CH)) return SRFTKV_ERR_CUDA;
    if (!encode_codes<D, BV>(&tvc, A.v->codes, bh, P.t_cap, C::CH)) return SRFTKV_ERR_CUDA;
    // scale rows: d/group floats; group-16 rows are swizzled like code rows of the same length
    const int ng = D / P.group;
    const CUtensorMapSwizzle ssw = P.group == 16 ? swizzle_for(4 * ng) : CU_TENSOR_MAP_SWIZZLE_NONE;
    tks = tkc;
    tvs = tvc;
    // fp16 / e8m0 planes: the (batch, kv head)'s scale bytes as rows of 16 bytes; a box is one chunk's bytes
    auto raw_plane = [&](CUtensorMap* map, const void* base, int sfmt) {
        const int sb = scale_bytes(sfmt);
        return encode_plane(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 16, 1, 16, bh, P.t_cap * ng * sb / 16,
                            C::CH * ng * sb / 16, CU_TENSOR_MAP_SWIZZLE_NONE);
    };
    if (C::QK) {
        const bool ok = P.sf_k == SRFTKV_SCALE_FP32 && pow2_dim<D>()
                            ? encode_plane(&tks, A.k->scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ng, 4, ng, bh, P.t_cap,
                                           C::CH, ssw)
                            : raw_plane(&tks, A.k->scales, P.sf_k);
        if (!ok) return SRFTKV_ERR_CUDA;
    }
    if (C::QV) {
        const bool ok = P.sf_v == SRFTKV_SCALE_FP32 && pow2_dim<D>()
                            ? encode_plane(&tvs, A.v->scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ng, 4, ng, bh, P.t_cap,
                                           C::CH, ssw)
                            : raw_plane(&tvs, A.v->scales, P.sf_v);
        if (!ok) return SRFTKV_ERR_CUDA;
    }
    const bool g16 = P.group == 16;  // raw fp16 sides carry group 16
    if (g16) split_kernel_attr<D, BK, BV, 16>();
    else split_kernel_attr<D, BK, BV, 0>();
    const dim3 grid(P.n_splits, P.B * P.Hkv * P.n_hg);
    const cudaError_t e = g16 ? launch_dependent(q4kv_attn_split_kernel<D, BK, BV, 16>, grid, dim3(kAttnWarps * 32),
                                                 C::SMEM, A.stream, tkc, tks, tvc, tvs, P)
                              : launch_dependent(q4kv_attn_split_kernel<D, BK, BV, 0>, grid, dim3(kAttnWarps * 32),
                                                 C::SMEM, A.stream, tkc, tks, tvc, tvs, P);
    if (e != cudaSuccess) {
        set_error("attention launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return 0;
}

template <int D>
static int launch_all(const AttnLaunch& A) {
    const AttnParams& P = A.P;
    const int bk = A.k->bits, bv = A.v->bits;
    const bool rot = bk != 16;
    const int rows = P.B * P.Hq;
    if (!rot)
        attn_prep_q_raw_kernel<D><<<(rows + 127) / 128, 128, 0, A.stream>>>(P);
    else
        attn_prep_q_kernel<D><<<rows, 128, 0, A.stream>>>(P);
    int rc;
    if (bk == 4 && bv == 4) rc = launch_split<D, 4, 4>(A);
    else if (bk == 8 && bv == 4) rc = launch_split<D, 8, 4>(A);
    else if (bk == 4 && bv == 8) rc = launch_split<D, 4, 8>(A);
    else if (bk == 8 && bv == 8) rc = launch_split<D, 8, 8>(A);
    else rc = launch_split<D, 16, 16>(A);
    if (rc) return rc;
    cudaError_t e = rot ? launch_dependent(attn_combine_kernel<D, true>, dim3(rows), dim3(128), 0, A.stream, P)
                        : launch_dependent(attn_combine_kernel<D, false>, dim3(rows), dim3(128), 0, A.stream, P);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("attention launch failed: %s", cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    return 0;
}

// head groups of at most four query heads per kv head (the MMA columns carry four heads), as even as possible
static int head_groups(int rep) { return (rep + 3) / 4; }
static int heads_per_group(int rep) { return (rep + head_groups(rep) - 1) / head_groups(rep); }

static int auto_splits(int B, int Hq, int Hkv, int t_cap) {
    const long long pairs = (long long)B * Hkv * head_groups(Hq / Hkv);
    // about five waves of CTAs at three an SM: larger splits than eight waves cost less per split (the
    // pipeline fill and the merge) and still leave the scheduler enough CTAs to even out the tail
    const long long target = 16ll * device_sm_count();
    long long s = (target + pairs - 1) / pairs;
    // but no split shorter than 1024 tokens (eight 32-token chunks a warp): below that the per-split work
    // (q fragments, pipeline fill, merge, partial) outweighs the parallelism gained.  Small batches
    // (measured at d = 128: B = 1 or 4 over 32 K tokens, B = 1 over 128 K, B = 16 over 8 K) ran 12-24 %
    // faster than with 256-token splits and within 6 % of the best split count
    const long long max_s = (t_cap + 1023) / 1024;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    return (int)s;
}

struct WsLayout {
    size_t qt, ml, acc, total;
};
static WsLayout ws_layout(int B, int Hq, int d, int n_splits) {
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    WsLayout w;
    w.qt = 0;
    w.ml = up((size_t)B * Hq * d * 4);
    w.acc = w.ml + up((size_t)B * Hq * n_splits * 2 * 4);
    w.total = w.acc + up((size_t)B * Hq * n_splits * d * 4);
    return w;
}

static int invalid_attn(const char* msg) {
    set_error("%s", msg);
    return SRFTKV_ERR_INVALID;
}

int attention_check(const void* q, const float* out, const srftkv_side* k, const srftkv_side* v, int B, int Hq,
                    int Hkv, int d, int group, int t_cap, int n_splits) {
    if (d != 64 && d != 80 && d != 96 && d != 128 && d != 192 && d != 256)
        return invalid_attn("attention: d must be 64, 80, 96, 128, 192 or 256");
    const bool pow2d = (d & (d - 1)) == 0;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || t_cap <= 0) return invalid_attn("attention: need B >= 0, Hq, Hkv, t_cap > 0");
    if (Hq % Hkv) return invalid_attn("attention: Hq must be a multiple of Hkv");
    if (!k || !v || !q || !out) return invalid_attn("attention: q, out, k and v must not be NULL");
    const bool raw = k->bits == 16 || v->bits == 16;
    if (raw && (k->bits != 16 || v->bits != 16)) return invalid_attn("attention: bits 16 must be used on both sides");
    if (!raw && ((k->bits != 4 && k->bits != 8) || (v->bits != 4 && v->bits != 8)))
        return invalid_attn("attention: bits must be 4, 8 (or 16 on both sides)");
    if (!raw) {
        // a power-of-two d copies fp32 scale rows as rows (at least 16 bytes: group <= d/4); d = 80, 96 and 192
        // copy every scale plane as 16-byte rows of bytes and take groups of 16 (d = 80) or 16 and 32
        if (group < 16 || (group & (group - 1)) || (d == 96 ? group > 32 : group > d / 4))
            return invalid_attn("attention: group must be a power of two with 16 <= group <= d/4 (16 or 32 at d = 96)");
        if (!k->scales || !v->scales) return invalid_attn("attention: scales must not be NULL");
        const srftkv_side* sv2[2] = {k, v};
        for (auto sd : sv2) {
            if (sd->transform != SRFTKV_TRANSFORM_SRFT && sd->transform != SRFTKV_TRANSFORM_SRHT)
                return invalid_attn("attention: transform must be SRFTKV_TRANSFORM_SRFT or SRFTKV_TRANSFORM_SRHT");
            if (sd->scale_format != SRFTKV_SCALE_FP32 && sd->scale_format != SRFTKV_SCALE_FP16 &&
                sd->scale_format != SRFTKV_SCALE_E8M0)
                return invalid_attn("attention: scale_format must be SRFTKV_SCALE_FP32, _FP16 or _E8M0");
            // fp16 / e8m0 scale planes are copied as 16-byte rows: one (batch, kv head)'s scales fill whole rows
            if ((sd->scale_format != SRFTKV_SCALE_FP32 || !pow2d) &&
                ((long long)t_cap * (d / group) * scale_bytes(sd->scale_format)) % 16 != 0)
                return invalid_attn("attention: t_cap * (d/group) * scale bytes must be a multiple of 16");
            if (!pow2d && sd->transform != SRFTKV_TRANSFORM_SRFT)
                return invalid_attn("attention: the Hadamard transform needs a power-of-two d");
        }
        // int4 rows of 40 bytes (d = 80) are copied as rows of token pairs
        if (d == 80 && (k->bits == 4 || v->bits == 4) && (t_cap & 1))
            return invalid_attn("attention: int4 rows at d = 80 need an even t_cap");
        if ((reinterpret_cast<uintptr_t>(k->scales) | reinterpret_cast<uintptr_t>(v->scales)) & 15)
            return invalid_attn("attention: scales must be 16-byte aligned");
        const srftkv_side* sd[2] = {k, v};
        for (auto s : sd)
            if (s->lambda && ((reinterpret_cast<uintptr_t>(s->lambda) & 15) || s->lambda_outer_stride < 0 ||
                              (s->lambda_outer_stride & 3)))
                return invalid_attn("attention: lambda must be 16-byte aligned with a non-negative stride, multiple of 4");
    }
    if (!k->codes || !v->codes) return invalid_attn("attention: codes must not be NULL");
    if ((reinterpret_cast<uintptr_t>(k->codes) | reinterpret_cast<uintptr_t>(v->codes) |
         reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15)
        return invalid_attn("attention: q, out and codes must be 16-byte aligned");
    if ((long long)B * Hkv * head_groups(Hq / Hkv) > 65535)
        return invalid_attn("attention: B * Hkv * ceil(Hq / Hkv / 4) must be at most 65535 (the grid's second dimension)");
    if ((long long)B * Hq > (1ll << 31) - 1) return invalid_attn("attention: B * Hq too large");
    if (n_splits < 0) return invalid_attn("attention: n_splits must be >= 0");
    return SRFTKV_OK;
}

int attention_auto_splits(int B, int Hq, int Hkv, int t_cap) { return auto_splits(B, Hq, Hkv, t_cap); }

int attention_entry(const void* q, float* out, const srftkv_side* k, const srftkv_side* v, int B, int Hq, int Hkv,
                    int d, int group, int t_cap, const int* seq_lens, float sm_scale, uint64_t seed, int n_splits,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    const int rc = attention_check(q, out, k, v, B, Hq, Hkv, d, group, t_cap, n_splits);
    if (rc) return rc;
    if (B == 0) return SRFTKV_OK;
    const int rc0 = current_device_ok();
    if (rc0) return rc0;
    const bool raw = k->bits == 16;
    const int ns = n_splits ? n_splits : auto_splits(B, Hq, Hkv, t_cap);
    const WsLayout wl = ws_layout(B, Hq, d, ns);
    if (!workspace || workspace_bytes < wl.total || (reinterpret_cast<uintptr_t>(workspace) & 15)) {
        set_error("attention: workspace must be 16-byte aligned and hold %zu bytes (got %zu)", wl.total, workspace_bytes);
        return SRFTKV_ERR_INVALID;
    }
    AttnLaunch A;
    std::memset(&A.P, 0, sizeof(A.P));
    AttnParams& P = A.P;
    char* ws = static_cast<char*>(workspace);
    P.q = static_cast<const uint16_t*>(q);
    P.qt = reinterpret_cast<float*>(ws + wl.qt);
    P.part_ml = reinterpret_cast<float*>(ws + wl.ml);
    P.part_acc = reinterpret_cast<float*>(ws + wl.acc);
    P.out = out;
    P.seq_lens = seq_lens;
    P.lam_k = raw ? nullptr : k->lambda;
    P.lam_k_stride = k->lambda_outer_stride;
    P.lam_v = raw ? nullptr : v->lambda;
    P.lam_v_stride = v->lambda_outer_stride;
    P.B = B;
    P.Hq = Hq;
    P.Hkv = Hkv;
    P.rep = Hq / Hkv;
    P.n_hg = head_groups(P.rep);
    P.hpg = heads_per_group(P.rep);
    P.vscale = raw ? nullptr : static_cast<const uint8_t*>(v->scales);
    P.t_cap = t_cap;
    P.n_splits = ns;
    P.group = raw ? 16 : group;
    P.log2_group = 0;
    while ((1 << P.log2_group) < P.group) ++P.log2_group;
    P.sp = raw ? 0 : d / P.group;
    P.tr_k = raw ? 0 : k->transform;
    P.tr_v = raw ? 0 : v->transform;
    P.sf_k = raw ? 0 : k->scale_format;
    P.sf_v = raw ? 0 : v->scale_format;
    const float sc = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt((float)d);
    P.qscale = sc * 1.4426950408889634f;
    const int lim = g_poll_limit.load();
    P.poll_limit = lim < 0 ? (1u << 20) : (uint32_t)lim;
    sign_masks(d, seed, P.sign_mask);
    A.k = k;
    A.v = v;
    A.d = d;
    A.stream = stream;
    switch (d) {
        case 64: return launch_all<64>(A);
        case 80: return launch_all<80>(A);
        case 96: return launch_all<96>(A);
        case 192: return launch_all<192>(A);
        case 128: return launch_all<128>(A);
        default: return launch_all<256>(A);
    }
}

size_t attention_workspace_size(int B, int Hq, int Hkv, int d, int t_cap, int n_splits) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || t_cap <= 0 || n_splits < 0 || Hq % Hkv) return 0;
    const int ns = n_splits ? n_splits : auto_splits(B, Hq, Hkv, t_cap);
    return ws_layout(B, Hq, d, ns).total;
}

unsigned int attn_take_fault() {
    unsigned int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_attn_fault, sizeof(v));
    cudaMemcpyToSymbol(g_attn_fault, &z, sizeof(z));
    return v;
}

}  // namespace srftkv
