// codec_d32.cu -- quantize / dequantize kernels for head dimension 32.
#include "codec_impl.cuh"

namespace srftkv {
template int launch_codec_d<32>(const CodecCall& c, bool quantize);
}  // namespace srftkv
