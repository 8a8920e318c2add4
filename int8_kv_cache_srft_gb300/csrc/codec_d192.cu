// codec_d192.cu -- the d = 192 codec entry (two threads per head vector, a
// 3 x 16 mixed-radix transform in each; kernels in codec_pair.cuh): the
// quantize kernels, and the dispatch to the dequantize kernels compiled in
// codec_d192_dq.cu.
#include "codec_pair.cuh"

namespace srftkv {

int launch_codec_d192(const CodecCall& c, bool quantize) {
    return quantize ? launch_pair_all<192, true>(c) : pair_dequantize_d192(c);
}

}  // namespace srftkv
