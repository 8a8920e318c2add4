// codec_d192_dq.cu -- the d = 192 dequantize kernels (codec_pair.cuh), in a
// translation unit of their own so the two directions compile in parallel.
#include "codec_pair.cuh"

namespace srftkv {

int pair_dequantize_d192(const CodecCall& c) { return launch_pair_all<192, false>(c); }

}  // namespace srftkv
