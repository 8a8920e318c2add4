// codec_d16.cu -- quantize / dequantize kernels for head dimension 16.
#include "codec_impl.cuh"

namespace srftkv {
template int launch_codec_d<16>(const CodecCall& c, bool quantize);
}  // namespace srftkv
