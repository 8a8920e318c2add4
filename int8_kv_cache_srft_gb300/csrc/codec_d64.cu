// codec_d64.cu -- quantize / dequantize kernels for head dimension 64.
#include "codec_impl.cuh"

namespace srftkv {
template int launch_codec_d<64>(const CodecCall& c, bool quantize);
}  // namespace srftkv
