/*
 * srftkv.h -- C ABI of libsrftkv, a GB300 (sm_103a) library for
 * rotate-then-quantize compression of the LLM KV cache and for decode
 * attention that reads the compressed cache directly.
 *
 * Method sources (page title -- section):
 *  [WQF] "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
 *        Apple Silicon" (summary of arXiv 2605.05699) -- Methodology 1
 *        (SRFT(x) = pack(F . diag(s) . x), F the unitary DFT, s a fixed
 *        random sign vector), Methodology 2 (the fused kernel: sign multiply,
 *        log2(d/2) radix-2 Stockham FFT stages, Hermitian packing, per-channel
 *        lambda, per-group absmax, signed int4/int8 rounding, nibble packing),
 *        Methodology 3 (per-channel lambda combined with groups of 16).
 *  [GEM] "Gemini on-device quantization, KV cache, Apple Silicon" -- section
 *        "Flash Attention and Metal kernel fusion" (tiled attention with an
 *        online softmax) and "INT8/INT4 quantization strategy" (the memory
 *        formula).
 *  [KVS] "Efficient LLM inference on Apple Silicon: KVSplit key techniques"
 *        -- "Key findings" (8-bit keys with 4-bit values, K8V4).
 *  [TQ]  "TurboQuant mobile KV cache compression: quantized deployment and
 *        latency optimisation on M5 Pro and iOS" -- quantization strategy
 *        section (online quantization of each newly generated token).
 *  [AQT] "No.9: how Apple fits a 3 GB model into a phone" -- section
 *        "Multi-plane tensor: data and scale factors together" (a quantized
 *        tensor is a data plane plus a scale plane).
 *
 * Readings where the pages leave a step open (the library and its test
 * oracle implement each one independently):
 *  - sign vector: s_i = -1 iff bit 63 of output i (from 0) of a splitmix64
 *    generator seeded with sign_seed is set (Steele, Lea & Flood 2014);
 *  - forward DFT uses exp(-2 pi i nk/d)/sqrt(d);
 *  - packing: p0 = y_0, p1 = y_{d/2}, p_{2k} = sqrt2 Re y_k,
 *    p_{2k+1} = sqrt2 Im y_k (k = 1..d/2-1): an orthogonal real map;
 *  - z_i = lambda_i * p_i; scale_j = max_{i in group j} |z_i| / Q with
 *    Q = 2^(bits-1)-1; q_i = rint(z_i / scale_j) in [-Q, Q]; zero group ->
 *    scale 0 and codes 0;
 *  - int4: two's-complement nibbles, even coordinate in the low nibble;
 *    int8: two's-complement bytes;
 *  - scales are fp32; softmax scale defaults to 1/sqrt(d); a query with
 *    sequence length 0 gets a zero output;
 *  - a head dimension that is not a power of two (d = 80, 96 or 192;
 *    Methodology 1 names SRFT's freedom from the power-of-two restriction
 *    of Hadamard rotations): the same F, the unitary DFT of length d, with
 *    the same packing; the library forms it as a dense d x d map (d = 80,
 *    96, and d = 192 on the tensor cores) or as a mixed-radix FFT (d = 192:
 *    96 = 2 x 3 x 16 points) instead of radix-2 stages only.
 *
 * General conventions
 *  - Every pointer argument that names tensor data is a DEVICE pointer
 *    owned by the caller; the library allocates no device memory.  State it
 *    keeps between calls: per-device capability checks, a per-host-thread
 *    copy of the last sign vector and error message, constant twiddle tables
 *    compiled into the kernels, two device fault words (one per kernel
 *    family) and the fixed-size scratch array of
 *    q4kv_decode_attention_static (all file-scope __device__ data, held by
 *    every GPU that loads the library), and the two process-wide poll
 *    limits of the test hooks at the end of this header.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued without host synchronisation; device-side
 *    faults surface on the caller's next synchronisation.
 *  - Return codes: SRFTKV_OK, or a negative SRFTKV_ERR_*; on any error no
 *    work has been enqueued and srftkv_last_error() describes it.
 *  - Inputs must be finite; NaN/Inf behaviour is unspecified.
 *  - Supported sizes: d in {16, 32, 64, 80, 96, 128, 192, 256} for the
 *    codec and srft_transform, d in {64, 80, 96, 128, 192, 256} for
 *    attention; group a power of two dividing d with 16 <= group <= d; bits
 *    in {4, 8} for packed sides.  d = 80, 96 and 192 take the SRFT only (the
 *    Hadamard matrix needs a power of two) and 16-byte aligned code and
 *    scale planes; d = 80 takes groups of 16 (the only power of two >= 16
 *    dividing 80), d = 96 groups of 16 or 32, d = 192 groups of 16, 32 or
 *    64.
 */
#ifndef SRFTKV_H
#define SRFTKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SRFTKV_OK 0
#define SRFTKV_ERR_INVALID (-1) /* bad size, pointer, alignment or bit width */
#define SRFTKV_ERR_CUDA (-2)    /* a CUDA call or launch failed */
#define SRFTKV_ERR_DEVICE (-3)  /* current device is not sm_103 */

/* The rotation applied before quantisation (per side, field `transform`). */
#define SRFTKV_TRANSFORM_SRFT 0 /* SRFT(x) = pack(F diag(s) x), F the unitary DFT ([WQF] Methodology 1) */
#define SRFTKV_TRANSFORM_SRHT 1 /* SRHT(x) = d^(-1/2) H diag(s) x, H the Sylvester Hadamard matrix in
                                   natural order (H_ij = (-1)^popcount(i & j)); the alternative the same
                                   section names, same sign vector s, no packing needed */
/* The scale plane's number format (per side, field `scale_format`); the codes are
 * rounded against the stored scale ([WQF] Key results, memory efficiency: 3.0-3.56x). */
#define SRFTKV_SCALE_FP32 0     /* fp32 A/Q, d/group per row (4 bytes each) */
#define SRFTKV_SCALE_FP16 1     /* fp16: A/Q rounded to nearest (ties even), saturating at 65504 (2 bytes) */
#define SRFTKV_SCALE_E8M0 2     /* one byte e: scale 2^(e-127) = the smallest power of two not below A/Q,
                                   e in [1, 254]; e = 0 stores an all-zero group (scale 0) */

/*
 * One side (K or V) of a packed cache, stored as two head-major planes ([AQT]):
 *   codes  : uint8 [n_outer][H][t_cap][d*bits/8]  (row start 16-byte aligned
 *            when d*bits/8 >= 16, else d*bits/8-byte aligned)
 *   scales : fp32  [n_outer][H][t_cap][d/group]   (16-byte aligned when
 *            d/group >= 4, else 4*d/group-byte aligned)
 * so the cached rows of one (outer, head) are contiguous.  n_outer is the
 * layer index for the codec calls and the batch index for attention.  A side
 * with bits == 16 (attention only) is a raw fp16 cache [B][Hkv][t_cap][d]
 * passed in `codes`, without rotation or scales.  The fp16 rows a codec call
 * reads or writes (`x`) keep the token-major layout [n_outer][n_tokens][H][d].
 */
typedef struct srftkv_side {
    void* x;                     /* quantize: fp16 input [n_outer][n_tokens][H][d] (read, 16-byte aligned);
                                    dequantize: fp16 output, same layout (written);
                                    attention: unused */
    const float* lambda;         /* per-channel lambda, element (o, h, i) at
                                    lambda[o*lambda_outer_stride + h*d + i]; must be > 0;
                                    NULL means all ones ([WQF] Methodology 3) */
    int64_t lambda_outer_stride; /* 0 broadcasts one [H][d] table over n_outer */
    int bits;                    /* 4 or 8 (16 = raw fp16 cache, attention only) */
    void* codes;                 /* code plane (see above) */
    void* scales;                /* scale plane (see above): fp32, fp16 or e8m0 bytes per scale_format */
    int transform;               /* SRFTKV_TRANSFORM_SRFT (0) or SRFTKV_TRANSFORM_SRHT (1); ignored for bits 16 */
    int scale_format;            /* SRFTKV_SCALE_FP32 (0), _FP16 (1) or _E8M0 (2): the element type of `scales` */
} srftkv_side;

/*
 * srft_kv_quantize -- encode fp16 head vectors into the packed cache
 * ([WQF] Methodology 1-3; K8V4 via bits per side [KVS]; appending one token
 * per step is n_tokens = 1 at t_offset = current length [TQ]).
 * For each side that is not NULL and every (o, t, h) with t < n_tokens:
 *   p = T(x[o][t][h]) with T the side's transform (SRFT, or SRHT);
 *   z = lambda[o][h] * p; per group j of `group`
 *   coordinates: scales[o][h][t_offset+t][j] = max|z| / Q and
 *   codes[o][h][t_offset+t] = packed rint(z / scale).
 * Both sides are encoded by one kernel launch.  Requires
 * 0 <= t_offset, t_offset + n_tokens <= t_cap, and x rows 16-byte aligned.
 * n_outer == 0 or n_tokens == 0 is a no-op that returns SRFTKV_OK.
 * d = 80 and 96 run as the 128-wide tensor-core contraction with R zero
 * outside its d x d block (any call size); d = 192 and 256 as the wide
 * tensor-core contraction for calls of 2^17 vectors and more (2^16 for
 * srft_kv_dequantize), else as the
 * register transform (two threads per vector at d = 192).
 */
int srft_kv_quantize(const srftkv_side* k, const srftkv_side* v, int n_outer, int n_tokens,
                     int H, int d, int group, int t_cap, int t_offset, uint64_t sign_seed,
                     void* stream);

/*
 * srft_kv_dequantize -- decode tokens [t_offset, t_offset+n_tokens) of the
 * packed cache back to fp16 ([WQF] Methodology 2, run backwards):
 *   x_hat = diag(s) . F^{-1} . unpack((codes * scale) / lambda)
 * (SRHT sides: x_hat = diag(s) . H . ((codes * scale) / lambda) / sqrt(d))
 * written to side->x as [n_outer][n_tokens][H][d].  Same size rules as
 * srft_kv_quantize.  The tensor-core path copies fp16 / e8m0 scale planes
 * (every scale plane at d = 80 and 96) as rows of 16 bytes, so there
 * t_cap * (d/group) * scale bytes and t_offset * (d/group) * scale bytes must
 * be multiples of 16, and at d = 80 (code rows of 40 or 80 bytes, copied
 * flat) also t_cap * d * bits / 8 and t_offset * d * bits / 8: at d = 80
 * and 96 that is required (SRFTKV_ERR_INVALID otherwise); at d = 128 a call
 * that misses it takes the FFT path.
 */
int srft_kv_dequantize(const srftkv_side* k, const srftkv_side* v, int n_outer, int n_tokens,
                       int H, int d, int group, int t_cap, int t_offset, uint64_t sign_seed,
                       void* stream);

/*
 * q4kv_decode_attention -- one decode step of attention that reads the
 * packed cache directly ([GEM] Flash Attention section: tiles of tokens with
 * an online softmax; [WQF] Methodology 1: SRFT is orthogonal, so
 * q . k_hat = SRFT(q) . (z_hat / lambda) and the cache is never rotated
 * back per token).
 *   q        : fp16 [B][Hq][d]
 *   out      : fp32 [B][Hq][d], out[b][h] = sum_t softmax_t(sm_scale * q.k_hat_t) v_hat_t
 *              over t < seq_lens[b], with query head h reading kv head
 *              h / (Hq/Hkv); k_hat, v_hat are the dequantised (unrotated) cache.
 *   k, v     : packed sides (bits 4 or 8) or both raw fp16 (bits 16);
 *              the x field is ignored.
 *   seq_lens : device int32 [B], each in [0, t_cap]; NULL means t_cap for all.
 *   sm_scale : softmax scale; <= 0 selects 1/sqrt(d).
 *   n_splits : number of context splits (split-K) per (b, kv head); 0 picks
 *              one from the device's SM count, B*Hkv and t_cap.
 *   workspace: device scratch of at least
 *              q4kv_decode_attention_workspace_size(...) bytes (16-byte aligned)
 *              for the per-split partial results; contents need not be
 *              initialised and are overwritten.
 * Requires d in {64, 80, 96, 128, 192, 256}, Hq % Hkv == 0 (any GQA ratio:
 * ratios above 4 run as head groups of at most four query heads, so
 * B * Hkv * ceil(Hq/Hkv/4) <= 65535), and
 * for packed sides a power-of-two group with 16 <= group <= d/4 (a scale
 * row of at least 16 bytes, the smallest TMA row; 16 at d = 80, 16 or 32
 * at d = 96 and 192) and 16-byte aligned scales; anything else returns
 * SRFTKV_ERR_INVALID before any launch.  fp16 / e8m0 scale planes, and
 * every scale plane at d = 80, 96 and 192 (rows that are not a power of
 * two), are copied as rows of 16 bytes and also need t_cap * (d/group) *
 * scale bytes to be a multiple of 16; int4 rows at d = 80 (40 bytes) are
 * read as rows of token pairs and need an even t_cap; d = 80, 96 and 192
 * sides use the SRFT.
 * Launches: three kernels on `stream` (q preparation, the split kernel, the
 * combine); the last two as programmatic dependents of the kernel before them
 * (they start launching while it finishes and wait for its results on the
 * device), so the call can be captured into a CUDA graph like any other
 * stream work and orders with the caller's other work as one call would.
 * Range: the kernel forms p * scale_V in fp16.  A stretch of tokens whose
 * V scales overflow that (scales of 128 and more) or sit far below it
 * (p-weighted mean scale under 2^-14) is run a second time with the values
 * rescaled by a power of two taken from its largest V scale, so any finite
 * scale works; only such caches pay for the second pass.  Key scales are
 * applied in fp32 and have no range limit.
 */
int q4kv_decode_attention(const void* q, float* out, const srftkv_side* k, const srftkv_side* v,
                          int B, int Hq, int Hkv, int d, int group, int t_cap,
                          const int* seq_lens, float sm_scale, uint64_t sign_seed, int n_splits,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * q4kv_decode_attention_static -- q4kv_decode_attention for callers that
 * cannot allocate device memory.  (The method's pages have no counterpart:
 * this is a convenience of the library.)
 *
 * Some callers cannot allocate the workspace: a runtime that has handed all
 * device memory to its own pool, a plugin behind a C ABI with no access to
 * its host framework's allocator, code that cannot afford the implicit
 * synchronisation of cudaMalloc.  This entry point takes the same arguments
 * as q4kv_decode_attention without the workspace and uses instead a
 * file-scope device array of SRFTKV_STATIC_SCRATCH_BYTES bytes that every GPU
 * loading the library holds until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *  - The arguments are checked first, exactly as q4kv_decode_attention
 *    checks them.  With n_splits == 0 the automatic split count is lowered
 *    until the workspace (q4kv_decode_attention_workspace_size) fits in
 *    SRFTKV_STATIC_SCRATCH_BYTES; sizes whose workspace exceeds it even so
 *    (or with the n_splits given) are rejected with SRFTKV_ERR_INVALID.  The
 *    automatic choice at B=16, Hq=32, d=128 on a 152-SM GB300 (19 splits)
 *    needs about 5.3 MB and is not lowered.
 *  - The first call in a CUDA context (for the runtime's primary context:
 *    the first call on a device) looks up the array's device address with
 *    that device current and caches it under the context's ID; make that
 *    first call before any stream capture.
 *  - All calls share the one array, which keeps the last call's contents;
 *    calls whose work overlaps on the GPU (e.g. on two streams) race.
 *    Nothing in it needs to start zeroed: each call writes all it reads.
 */
#define SRFTKV_STATIC_SCRATCH_BYTES (16u << 20)
int q4kv_decode_attention_static(const void* q, float* out, const srftkv_side* k, const srftkv_side* v,
                                 int B, int Hq, int Hkv, int d, int group, int t_cap,
                                 const int* seq_lens, float sm_scale, uint64_t sign_seed, int n_splits,
                                 void* stream);

/* Bytes of workspace q4kv_decode_attention needs for these sizes (n_splits 0 = the
 * automatic choice on the current device).  Returns 0 for invalid sizes. */
size_t q4kv_decode_attention_workspace_size(int B, int Hq, int Hkv, int d, int t_cap, int n_splits);

/* Bytes of one packed vector: code plane d*bits/8 and scale plane
 * (d/group) * b with b = 4, 2 or 1 for scale_format SRFTKV_SCALE_FP32, _FP16
 * or _E8M0.  Host-only; returns SRFTKV_OK or SRFTKV_ERR_INVALID (sizes the
 * codec does not take, or an unknown scale_format). */
int srft_kv_vector_bytes(int d, int bits, int group, int scale_format, size_t* code_bytes, size_t* scale_bytes);

/*
 * srft_transform -- the bare transform, for testing ([WQF] Methodology 1).
 * x : fp16 [n][d] (16-byte aligned rows); y : fp32 [n][d].
 * inverse == 0: y = SRFT(x) (packed coordinates p);
 * inverse != 0: y = SRFT^{-1}(x) = diag(s) . F^{-1} . unpack(x).
 */
int srft_transform(const void* x, float* y, int n, int d, uint64_t sign_seed, int inverse,
                   void* stream);

/*
 * srht_transform -- the Hadamard variant of srft_transform, same arguments:
 * inverse == 0: y = SRHT(x) = d^(-1/2) H diag(s) x;
 * inverse != 0: y = diag(s) H x / sqrt(d).
 */
int srht_transform(const void* x, float* y, int n, int d, uint64_t sign_seed, int inverse,
                   void* stream);

/* Message for the last non-zero return on this host thread ("" if none). */
const char* srftkv_last_error(void);

/*
 * srftkv_device_fault -- copies the library's device-side fault word for the
 * current device into *fault (0 = none) and clears it.  A kernel whose
 * bounded wait on an asynchronous copy gives up sets a bit here and returns
 * instead of waiting forever.  Synchronises the current device.
 */
int srftkv_device_fault(unsigned int* fault);

/*
 * srftkv_set_attention_poll_limit_for_testing -- TEST HOOK, not for use in
 * production.  Sets how many times (each poll may suspend for up to about
 * 1 us) a warp of the attention split kernel polls for its next chunk of the
 * cache before it gives up; a negative value restores the default (2^20
 * polls, about a second) and 0 makes every warp give up at its first chunk.
 * A warp that gives up sets bit 8 of the fault word, waits with the default
 * bound for its own copies in flight and contributes nothing, so a call on
 * which every warp gives up leaves the fault word set and writes zero
 * outputs.  Applies to every later attention call of the process (a
 * process-wide setting, both attention entry points); the codec kernels
 * keep their bound.  Always returns SRFTKV_OK.
 */
int srftkv_set_attention_poll_limit_for_testing(int polls);

/*
 * srftkv_set_codec_poll_limit_for_testing -- TEST HOOK, not for use in
 * production.  The same for the codec's quantize kernels that wait on
 * asynchronous copies of x: how many times a warp of the register-path
 * kernels (the one-thread-per-vector FFT / WHT kernel of d <= 128, the
 * two-lane kernel of d = 192 / 256) polls for its next tile, and how many
 * times the MMA-issuing thread of the tensor-core kernel of d = 80 / 96 / 128
 * polls for its next x stage, before giving up; negative restores the default (2^20
 * polls), 0 makes them give up at their first tile.  A warp that gives up
 * sets bit 0 of the fault word, waits with the default bound for its own
 * copies in flight and returns without storing; in the tensor-core kernel
 * the MMA thread then issues nothing and the epilogue warps give up after
 * their default bound (about a second), so such a call is slow.  Either way
 * the codes and scales keep their previous contents.  Process-wide; the
 * wide tensor-core kernels, the one-warp-per-vector append kernel (no
 * asynchronous copies) and the dequantize kernels keep their bounds.
 * Always returns SRFTKV_OK.
 */
int srftkv_set_codec_poll_limit_for_testing(int polls);

#ifdef __cplusplus
}
#endif

#endif /* SRFTKV_H */
