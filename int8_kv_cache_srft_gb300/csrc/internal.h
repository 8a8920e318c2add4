// internal.h -- declarations shared by the library's translation units
// (not part of the public C ABI, see include/srftkv.h for that).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "srftkv.h"

namespace srftkv {

// One side (K or V) of a codec call, after validation.
struct CodecSideDesc {
    void* x;              // fp16 rows [n_outer][n_tokens][H][d]
    uint8_t* codes;       // [n_outer][H][t_cap][d*bits/8]
    void* scales;         // [n_outer][H][t_cap][d/group], element type per scale_format
    const float* lambda;  // [*][H][d] or null
    int64_t lambda_outer_stride;
    int bits;
    int transform;        // SRFTKV_TRANSFORM_SRFT or SRFTKV_TRANSFORM_SRHT
    int scale_format;     // SRFTKV_SCALE_FP32 / _FP16 / _E8M0
};

// bytes of one stored scale
inline int scale_bytes(int scale_format) { return scale_format == SRFTKV_SCALE_FP32 ? 4 : scale_format == SRFTKV_SCALE_FP16 ? 2 : 1; }

struct CodecCall {
    CodecSideDesc side[2];
    int n_sides;
    int n_outer, n_tokens, H, d, group, t_cap, t_offset;
    uint64_t seed;
    cudaStream_t stream;
};

// Signs of the SRFT as fp16-pair XOR masks: word n has bit 15 set when
// s_{2n} = -1 and bit 31 set when s_{2n+1} = -1 (d/2 words).
void sign_masks(int d, uint64_t seed, uint32_t* words);

// Tensor map over fp16 rows x[n_outer][n_tokens][H][d] whose box is
// box_rows consecutive tokens of one (outer, head).  Plain: rows land in
// shared memory padded by 8 elements (d <= 128; d = 256 as two padded
// halves).  swz128 (d = 128): two 64-element k-blocks in the 128-byte
// swizzle layout of the tensor-core operands.  False + message on failure.
bool encode_x_map(CUtensorMap* map, void* base, int d, int H, int n_tokens, int n_outer, int box_rows, bool swz128);

int codec_quantize(const CodecCall& c);
int codec_dequantize(const CodecCall& c);
// The register-transform codec at d = 192 and 256 (two threads per vector, codec_d192.cu, codec_d256.cu).
int launch_codec_d192(const CodecCall& c, bool quantize);
int launch_codec_d256(const CodecCall& c, bool quantize);
int transform_launch(const void* x, float* y, int n, int d, uint64_t seed, bool inverse, bool srht, cudaStream_t s);
unsigned int codec_take_fault();
unsigned int* codec_fault_word();  // device address of the codec fault word (current device)
// polls of the register-path quantize kernels' wait for a tile before they give up (2^20 unless a test
// lowered it with srftkv_set_codec_poll_limit_for_testing)
uint32_t codec_poll_limit();

void set_error(const char* fmt, ...);

// Device address of a __device__ variable in the CUDA context current on this
// thread, looked up once per context (cudaGetSymbolAddress, which allocates
// nothing) and cached under the context's ID.  SRFTKV_OK or SRFTKV_ERR_CUDA.
struct SymbolCache {
    static constexpr int kSlots = 16;
    std::mutex mu;
    unsigned long long id[kSlots] = {};
    void* ptr[kSlots] = {};
    int next = 0;
};
int symbol_address(SymbolCache& cache, const void* symbol, void** out, const char* what);
int device_sm_count();
int current_device_ok();  // SRFTKV_OK, or the error code with the message set

// Generic tiled tensor map (element strides 1); false + message on failure.
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* base, const unsigned long long* dims,
                  const unsigned long long* strides_bytes, const unsigned* box, const char* what);

bool encode_tiled_swz(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* base, const unsigned long long* dims,
                      const unsigned long long* strides_bytes, const unsigned* box, CUtensorMapSwizzle swz,
                      const char* what, CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

// Tensor-core quantize path (d = 128, group <= 64); returns 1 when the call
// is not one it handles, else SRFTKV_OK or an error code.
int codec_quantize_tc(const CodecCall& c);
// Tensor-core quantize at d = 192 and d = 256 (codec_tc_wide.cuh; groups of at most 32).
int codec_quantize_tc_wide192(const CodecCall& c);
int codec_quantize_tc_wide256(const CodecCall& c);
// Tensor-core dequantize at d = 192 and 256: 1 when the call does not fit it (lambda, groups above 32, scale rows).
int codec_dequantize_tc_wide192(const CodecCall& c);
int codec_dequantize_tc_wide256(const CodecCall& c);
// One warp per vector (d = 128, groups of at most 32): returns 1 when the call does not fit it.
int codec_quantize_warp(const CodecCall& c);
int codec_dequantize_tc(const CodecCall& c);

int attention_entry(const void* q, float* out, const srftkv_side* k, const srftkv_side* v, int B, int Hq, int Hkv,
                    int d, int group, int t_cap, const int* seq_lens, float sm_scale, uint64_t seed, int n_splits,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);
size_t attention_workspace_size(int B, int Hq, int Hkv, int d, int t_cap, int n_splits);
// Argument checks of attention_entry that do not involve the workspace (SRFTKV_OK or the error, message set).
int attention_check(const void* q, const float* out, const srftkv_side* k, const srftkv_side* v, int B, int Hq,
                    int Hkv, int d, int group, int t_cap, int n_splits);
// The split count attention_entry picks for n_splits == 0 on the current device.
int attention_auto_splits(int B, int Hq, int Hkv, int t_cap);
unsigned int attn_take_fault();
// Test hook behind srftkv_set_attention_poll_limit_for_testing (negative = the default limit).
void attention_set_poll_limit(int polls);

}  // namespace srftkv
