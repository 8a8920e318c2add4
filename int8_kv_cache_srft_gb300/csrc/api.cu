// api.cu -- the C ABI of libsrftkv: argument validation, the sign vector,
// TMA tensor-map encoding, device checks and error reporting.  The entry
// points are declared and documented in include/srftkv.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace srftkv {

// ---------------------------------------------------------------------------
// Errors
// ---------------------------------------------------------------------------
static thread_local char t_err[512] = "";

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
}

static int invalid(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
    return SRFTKV_ERR_INVALID;
}

// ---------------------------------------------------------------------------
// Sign vector: s_i = -1 iff bit 63 of output i of splitmix64(seed) is set.
// splitmix64 (Steele, Lea & Flood, OOPSLA 2014): the state advances by the
// golden-ratio increment and each output is the state passed through two
// xor-shift-multiply rounds and a final xor-shift.
// ---------------------------------------------------------------------------
static uint64_t splitmix64_output(uint64_t state) {
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void sign_masks(int d, uint64_t seed, uint32_t* words) {
    // the last (d, seed) of this host thread is kept: a decode loop asks for the same one every call
    thread_local int last_d = -1;
    thread_local uint64_t last_seed = 0;
    thread_local uint32_t last_words[128];
    if (d == last_d && seed == last_seed && d <= 256) {
        for (int i = 0; i < d / 2; ++i) words[i] = (words[i] & 0x7FFF7FFFu) | last_words[i];
        return;
    }
    uint64_t state = seed;
    for (int i = 0; i < d; ++i) {
        state += 0x9E3779B97F4A7C15ull;
        const bool neg = (splitmix64_output(state) >> 63) != 0;
        if (neg) words[i / 2] |= (i & 1) ? 0x80000000u : 0x00008000u;
        else words[i / 2] &= (i & 1) ? ~0x80000000u : ~0x00008000u;
    }
    if (d <= 256) {
        for (int i = 0; i < d / 2; ++i) last_words[i] = words[i] & 0x80008000u;
        last_d = d;
        last_seed = seed;
    }
}

// ---------------------------------------------------------------------------
// Device checks
// ---------------------------------------------------------------------------
struct DevInfo {
    int checked = 0;
    int ok = 0;
    int sms = 0;
};
static DevInfo g_dev[64];
static std::mutex g_dev_mu;

int current_device_ok() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        set_error("no current CUDA device");
        return SRFTKV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo& di = g_dev[dev];
    if (!di.checked) {
        cudaDeviceProp p;
        if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) {
            set_error("cudaGetDeviceProperties failed");
            return SRFTKV_ERR_CUDA;
        }
        di.ok = (p.major == 10 && p.minor == 3);
        di.sms = p.multiProcessorCount;
        di.checked = 1;
        if (!di.ok) snprintf(t_err, sizeof(t_err), "device %d is sm_%d%d, this library is built for sm_103a", dev, p.major, p.minor);
    }
    if (!di.ok) {
        set_error("current device is not sm_103 (GB300)");
        return SRFTKV_ERR_DEVICE;
    }
    return SRFTKV_OK;
}

int device_sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && g_dev[dev].checked) return g_dev[dev].sms;
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// ---------------------------------------------------------------------------
// Device addresses of the library's __device__ variables, per CUDA context
// ---------------------------------------------------------------------------
// The address of a __device__ variable belongs to the context that loaded the
// module: it differs between contexts of one device (the primary context and a
// driver-API context, or the primary context before and after a device reset).
// So lookups are cached under the current context's ID, which CUDA never
// reuses within a process.
static PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
static PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
static std::once_flag g_ctx_once;

static bool current_context_id(unsigned long long* id) {
    std::call_once(g_ctx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    if (!g_ctx_current || !g_ctx_id) return false;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

int symbol_address(SymbolCache& cache, const void* symbol, void** out, const char* what) {
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);  // false before the runtime has made a context current
    std::lock_guard<std::mutex> lk(cache.mu);
    if (have_id)
        for (int i = 0; i < SymbolCache::kSlots; ++i)
            if (cache.id[i] == id && cache.ptr[i]) {
                *out = cache.ptr[i];
                return SRFTKV_OK;
            }
    void* p = nullptr;  // the lookup allocates nothing; it makes the device's primary context current if none is
    const cudaError_t e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess || !p) {
        set_error("cudaGetSymbolAddress failed for %s: %s", what, cudaGetErrorString(e));
        return SRFTKV_ERR_CUDA;
    }
    if (have_id || current_context_id(&id)) {
        const int slot = cache.next;
        cache.next = (cache.next + 1) % SymbolCache::kSlots;
        cache.id[slot] = id;
        cache.ptr[slot] = p;
    }
    *out = p;
    return SRFTKV_OK;
}

// ---------------------------------------------------------------------------
// TMA tensor maps
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* base, const unsigned long long* dims,
                  const unsigned long long* strides_bytes, const unsigned* box, const char* what) {
    return encode_tiled_swz(map, dt, rank, base, dims, strides_bytes, box, CU_TENSOR_MAP_SWIZZLE_NONE, what);
}

bool encode_tiled_swz(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* base, const unsigned long long* dims,
                      const unsigned long long* strides_bytes, const unsigned* box, CUtensorMapSwizzle swz,
                      const char* what, CUtensorMapL2promotion promo) {
    auto enc = encoder();
    if (!enc) {
        set_error("cuTensorMapEncodeTiled is unavailable from the driver");
        return false;
    }
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    const CUresult r = enc(map, dt, rank, base, d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, promo,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (CUresult %d) for %s", (int)r, what);
        return false;
    }
    return true;
}

bool encode_x_map(CUtensorMap* map, void* base, int d, int H, int n_tokens, int n_outer, int box_rows, bool swz128) {
    // fp16 rows x[n_outer][n_tokens][H][d]; one box = box_rows tokens of one (outer, head)
    const unsigned long long e = 2;
    if (swz128) {  // 128-byte swizzled k-blocks of 64 elements (d == 128)
        const unsigned long long dims[4] = {(unsigned long long)d, (unsigned long long)H, (unsigned long long)n_tokens,
                                            (unsigned long long)n_outer};
        const unsigned long long str[3] = {d * e, (unsigned long long)H * d * e, (unsigned long long)n_tokens * H * d * e};
        const unsigned box[4] = {64u, 1u, (unsigned)box_rows, 1u};
        // rows that are not a multiple of 256 bytes (d = 80, 96, 192): an L2 promotion wider than the row's
        // alignment would fetch part of the neighbouring head's row, read much later by another tile
        const CUtensorMapL2promotion promo = (d * e) % 256 == 0   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                             : (d * e) % 128 == 0 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                                  : CU_TENSOR_MAP_L2_PROMOTION_NONE;
        return encode_tiled_swz(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B,
                                "x rows (swizzled)", promo);
    }
    if (d <= 128) {  // rows land padded by 8 elements (the zero-filled columns past d)
        const unsigned long long dims[4] = {(unsigned long long)d, (unsigned long long)H, (unsigned long long)n_tokens,
                                            (unsigned long long)n_outer};
        const unsigned long long str[3] = {d * e, (unsigned long long)H * d * e, (unsigned long long)n_tokens * H * d * e};
        const unsigned box[4] = {(unsigned)(d + 8), 1u, (unsigned)box_rows, 1u};
        return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, base, dims, str, box, "x rows");
    }
    const int half = d / 2;  // d = 256: two halves of 128 (+8 padding) each
    const unsigned long long dims[5] = {(unsigned long long)half, 2, (unsigned long long)H, (unsigned long long)n_tokens,
                                        (unsigned long long)n_outer};
    const unsigned long long str[4] = {half * e, d * e, (unsigned long long)H * d * e,
                                       (unsigned long long)n_tokens * H * d * e};
    const unsigned box[5] = {(unsigned)(half + 8), 2u, 1u, (unsigned)box_rows, 1u};
    return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, base, dims, str, box, "x rows (d=256)");
}

// ---------------------------------------------------------------------------
// Validation helpers
// ---------------------------------------------------------------------------
static bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
static size_t min_sz(size_t a, size_t b) { return a < b ? a : b; }
// head dimensions of the codec and the SRFT: the powers of two 16..256, 80, 96 and 192
// (a non-power-of-two d runs the SRFT only: d = 80 and 96 as the 128-wide tensor-core
// contraction, d = 192 as the wide tensor-core contraction or the mixed-radix register transform)
static bool codec_d(int d) {
    return d == 16 || d == 32 || d == 64 || d == 80 || d == 96 || d == 128 || d == 192 || d == 256;
}
static bool pow2_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128 || d == 256; }

static int check_codec_sizes(int n_outer, int n_tokens, int H, int d, int group, int t_cap, int t_offset) {
    if (!codec_d(d)) return invalid("d must be one of 16, 32, 64, 80, 96, 128, 192, 256 (got %d)", d);
    if (!pow2(group) || group < 16 || group > d || d % group)
        return invalid("group must be a power of two dividing d with 16 <= group <= d (got %d)", group);
    if (n_outer < 0 || n_tokens < 0 || H <= 0) return invalid("n_outer, n_tokens must be >= 0 and H > 0");
    if (t_offset < 0 || t_cap < 0 || (long long)t_offset + n_tokens > t_cap)
        return invalid("need 0 <= t_offset and t_offset + n_tokens <= t_cap (t_offset=%d n_tokens=%d t_cap=%d)", t_offset,
                       n_tokens, t_cap);
    const long long rows = (long long)n_tokens * H, crow = (long long)t_cap * H;
    if (rows > (1ll << 31) - 64 || crow > (1ll << 31) - 64 || (long long)n_outer * ((rows + 31) / 32) * 2 > (1ll << 31) - 1)
        return invalid("sizes too large for 32-bit tile indexing");
    return SRFTKV_OK;
}

static int check_side(const srftkv_side* s, const char* name, int d, int group, bool need_x) {
    if (s->bits != 4 && s->bits != 8) return invalid("%s: bits must be 4 or 8 (got %d)", name, s->bits);
    if (s->transform != SRFTKV_TRANSFORM_SRFT && s->transform != SRFTKV_TRANSFORM_SRHT)
        return invalid("%s: transform must be SRFTKV_TRANSFORM_SRFT or SRFTKV_TRANSFORM_SRHT (got %d)", name, s->transform);
    if (s->scale_format != SRFTKV_SCALE_FP32 && s->scale_format != SRFTKV_SCALE_FP16 &&
        s->scale_format != SRFTKV_SCALE_E8M0)
        return invalid("%s: scale_format %d is not supported", name, s->scale_format);
    if (s->transform == SRFTKV_TRANSFORM_SRHT && !pow2(d))
        return invalid("%s: the Hadamard transform needs a power-of-two d (got %d)", name, d);
    if (!s->codes || !s->scales) return invalid("%s: codes and scales must not be NULL", name);
    if (need_x && !s->x) return invalid("%s: x must not be NULL", name);
    // rows of a power-of-two d are powers of two: align to the row up to 16 bytes; the planes of d = 80, 96 and
    // 192 are copied by TMA or plain bulk copies
    const size_t crow = (size_t)d * s->bits / 8, srow = (size_t)(d / group) * scale_bytes(s->scale_format);
    const size_t ca = pow2(d) ? min_sz(16, crow) : 16, sa = pow2(d) ? min_sz(16, srow) : 16;
    if (!aligned(s->codes, ca)) return invalid("%s: codes must be %zu-byte aligned", name, ca);
    if (!aligned(s->scales, sa)) return invalid("%s: scales must be %zu-byte aligned", name, sa);
    if (need_x && !aligned(s->x, 16)) return invalid("%s: x must be 16-byte aligned", name);
    if (s->lambda && (!aligned(s->lambda, 16) || (s->lambda_outer_stride % 4) != 0 || s->lambda_outer_stride < 0))
        return invalid("%s: lambda must be 16-byte aligned with a non-negative outer stride that is a multiple of 4", name);
    return SRFTKV_OK;
}

static int codec_common(const srftkv_side* k, const srftkv_side* v, int n_outer, int n_tokens, int H, int d, int group,
                        int t_cap, int t_offset, uint64_t seed, void* stream, bool quantize) {
    int rc = check_codec_sizes(n_outer, n_tokens, H, d, group, t_cap, t_offset);
    if (rc) return rc;
    if (!k && !v) return invalid("at least one of k, v must be given");
    CodecCall c;
    std::memset(&c, 0, sizeof(c));
    c.n_sides = 0;
    const srftkv_side* sides[2] = {k, v};
    const char* names[2] = {"k", "v"};
    for (int i = 0; i < 2; ++i) {
        if (!sides[i]) continue;
        rc = check_side(sides[i], names[i], d, group, true);
        if (rc) return rc;
        CodecSideDesc& s = c.side[c.n_sides++];
        s.x = sides[i]->x;
        s.codes = static_cast<uint8_t*>(sides[i]->codes);
        s.scales = sides[i]->scales;
        s.scale_format = sides[i]->scale_format;
        s.lambda = sides[i]->lambda;
        s.lambda_outer_stride = sides[i]->lambda_outer_stride;
        s.bits = sides[i]->bits;
        s.transform = sides[i]->transform;
    }
    if (n_outer == 0 || n_tokens == 0) return SRFTKV_OK;
    rc = current_device_ok();
    if (rc) return rc;
    c.n_outer = n_outer;
    c.n_tokens = n_tokens;
    c.H = H;
    c.d = d;
    c.group = group;
    c.t_cap = t_cap;
    c.t_offset = t_offset;
    c.seed = seed;
    c.stream = static_cast<cudaStream_t>(stream);
    return quantize ? codec_quantize(c) : codec_dequantize(c);
}

}  // namespace srftkv

using namespace srftkv;

extern "C" {

int srft_kv_quantize(const srftkv_side* k, const srftkv_side* v, int n_outer, int n_tokens, int H, int d, int group,
                     int t_cap, int t_offset, uint64_t sign_seed, void* stream) {
    return codec_common(k, v, n_outer, n_tokens, H, d, group, t_cap, t_offset, sign_seed, stream, true);
}

int srft_kv_dequantize(const srftkv_side* k, const srftkv_side* v, int n_outer, int n_tokens, int H, int d, int group,
                       int t_cap, int t_offset, uint64_t sign_seed, void* stream) {
    return codec_common(k, v, n_outer, n_tokens, H, d, group, t_cap, t_offset, sign_seed, stream, false);
}

int srft_kv_vector_bytes(int d, int bits, int group, int scale_format, size_t* code_bytes, size_t* scale_bytes_out) {
    if (!codec_d(d)) return invalid("d must be one of 16, 32, 64, 80, 96, 128, 192, 256");
    if (bits != 4 && bits != 8) return invalid("bits must be 4 or 8");
    if (!pow2(group) || group < 16 || group > d || d % group)
        return invalid("group must be a power of two dividing d with 16 <= group <= d");
    if (scale_format != SRFTKV_SCALE_FP32 && scale_format != SRFTKV_SCALE_FP16 && scale_format != SRFTKV_SCALE_E8M0)
        return invalid("scale_format %d is not supported", scale_format);
    if (code_bytes) *code_bytes = (size_t)d * bits / 8;
    if (scale_bytes_out) *scale_bytes_out = (size_t)(d / group) * scale_bytes(scale_format);
    return SRFTKV_OK;
}

int srft_transform(const void* x, float* y, int n, int d, uint64_t sign_seed, int inverse, void* stream) {
    if (!codec_d(d)) return invalid("d must be one of 16, 32, 64, 80, 96, 128, 192, 256");
    if (n < 0) return invalid("n must be >= 0");
    if (n == 0) return SRFTKV_OK;
    if (!x || !y) return invalid("x and y must not be NULL");
    if (!aligned(x, 16) || !aligned(y, 16)) return invalid("x and y must be 16-byte aligned");
    const int rc = current_device_ok();
    if (rc) return rc;
    return transform_launch(x, y, n, d, sign_seed, inverse != 0, false, static_cast<cudaStream_t>(stream));
}

int srht_transform(const void* x, float* y, int n, int d, uint64_t sign_seed, int inverse, void* stream) {
    if (!pow2_d(d)) return invalid("d must be one of 16, 32, 64, 128, 256");
    if (n < 0) return invalid("n must be >= 0");
    if (n == 0) return SRFTKV_OK;
    if (!x || !y) return invalid("x and y must not be NULL");
    if (!aligned(x, 16) || !aligned(y, 16)) return invalid("x and y must be 16-byte aligned");
    const int rc = current_device_ok();
    if (rc) return rc;
    return transform_launch(x, y, n, d, sign_seed, inverse != 0, true, static_cast<cudaStream_t>(stream));
}

int q4kv_decode_attention(const void* q, float* out, const srftkv_side* k, const srftkv_side* v, int B, int Hq, int Hkv,
                          int d, int group, int t_cap, const int* seq_lens, float sm_scale, uint64_t sign_seed,
                          int n_splits, void* workspace, size_t workspace_bytes, void* stream) {
    return attention_entry(q, out, k, v, B, Hq, Hkv, d, group, t_cap, seq_lens, sm_scale, sign_seed, n_splits,
                           workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t q4kv_decode_attention_workspace_size(int B, int Hq, int Hkv, int d, int t_cap, int n_splits) {
    return attention_workspace_size(B, Hq, Hkv, d, t_cap, n_splits);
}

const char* srftkv_last_error(void) { return t_err; }

int srftkv_set_attention_poll_limit_for_testing(int polls) {
    attention_set_poll_limit(polls);
    return SRFTKV_OK;
}

int srftkv_device_fault(unsigned int* fault) {
    if (!fault) return invalid("fault must not be NULL");
    if (cudaDeviceSynchronize() != cudaSuccess) {
        set_error("cudaDeviceSynchronize failed");
        return SRFTKV_ERR_CUDA;
    }
    *fault = codec_take_fault() | (attn_take_fault() << 8);
    return SRFTKV_OK;
}

}  // extern "C"
