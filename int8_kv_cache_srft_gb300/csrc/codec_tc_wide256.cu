// The tensor-core quantize and dequantize at d = 256 (codec_tc_wide.cuh): CTA pairs split the output coordinates.
#include <type_traits>

#include "codec_tc_wide.cuh"

namespace srftkv {
int codec_quantize_tc_wide256(const CodecCall& c) { return codec_quantize_tc_wide_d<256, 2>(c); }
int codec_dequantize_tc_wide256(const CodecCall& c) { return codec_dequantize_tc_wide_d<256>(c); }
}  // namespace srftkv
