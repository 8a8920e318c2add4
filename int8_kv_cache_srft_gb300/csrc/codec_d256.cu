// codec_d256.cu -- the d = 256 codec entry (two threads per head vector, kernels
// in codec_pair.cuh): the quantize kernels, and the dispatch to the dequantize
// kernels compiled in codec_d256_dq.cu.
#include "codec_pair.cuh"

namespace srftkv {

int launch_codec_d256(const CodecCall& c, bool quantize) {
    return quantize ? launch_pair_all<256, true>(c) : pair_dequantize_d256(c);
}

}  // namespace srftkv
