// codec_d256.cu -- quantize / dequantize kernels for head dimension 256.
#include "codec_impl.cuh"

namespace srftkv {
template int launch_codec_d<256>(const CodecCall& c, bool quantize);
}  // namespace srftkv
