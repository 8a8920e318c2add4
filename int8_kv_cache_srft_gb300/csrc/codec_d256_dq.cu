// codec_d256_dq.cu -- the d = 256 dequantize kernels (codec_pair.cuh), in a
// translation unit of their own so the two directions compile in parallel.
#include "codec_pair.cuh"

namespace srftkv {

int pair_dequantize_d256(const CodecCall& c) { return launch_pair_all<256, false>(c); }

}  // namespace srftkv
