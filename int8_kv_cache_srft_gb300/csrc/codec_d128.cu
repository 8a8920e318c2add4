// codec_d128.cu -- quantize / dequantize kernels for head dimension 128.
#include "codec_impl.cuh"

namespace srftkv {
template int launch_codec_d<128>(const CodecCall& c, bool quantize);
}  // namespace srftkv
