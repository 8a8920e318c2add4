// internal.h -- declarations shared by the library's translation units
// (not part of the public C ABI, see include/srftkv.h for that).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "srftkv.h"

namespace srftkv {

// One side (K or V) of a codec call, after validation.
struct CodecSideDesc {
    void* x;              // fp16 rows [n_outer][n_tokens][H][d]
    uint8_t* codes;       // [n_outer][t_cap][H][d*bits/8]
    float* scales;        // [n_outer][t_cap][H][d/group]
    const float* lambda;  // [*][H][d] or null
    int64_t lambda_outer_stride;
    int bits;
};

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

// 3D (d <= 128) or 4D (d == 256) tensor map over fp16 rows
// [n_outer][rows_per_outer][d] whose box is `box_rows` rows of d + 8
// elements (256: two halves of 136), so that each row lands in shared memory
// padded by 16 bytes.  Returns false and sets the error message on failure.
bool encode_row_map(CUtensorMap* map, void* base, int d, long long rows_per_outer, int n_outer, int box_rows);

int codec_quantize(const CodecCall& c);
int codec_dequantize(const CodecCall& c);
int transform_launch(const void* x, float* y, int n, int d, uint64_t seed, bool inverse, cudaStream_t s);
unsigned int codec_take_fault();

void set_error(const char* fmt, ...);
int device_sm_count();

}  // namespace srftkv
