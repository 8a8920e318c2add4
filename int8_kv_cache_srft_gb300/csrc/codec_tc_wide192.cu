// The tensor-core quantize and dequantize at d = 192 (codec_tc_wide.cuh): one CTA holds all of R_s.
#include <type_traits>

#include "codec_tc_wide.cuh"

namespace srftkv {
int codec_quantize_tc_wide192(const CodecCall& c) { return codec_quantize_tc_wide_d<192, 1>(c); }
int codec_dequantize_tc_wide192(const CodecCall& c) { return codec_dequantize_tc_wide_d<192>(c); }
}  // namespace srftkv
