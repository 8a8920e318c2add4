// attention.cu -- placeholder (decode attention is being written)
#include "internal.h"
using namespace srftkv;
extern "C" {
int q4kv_decode_attention(const void*, float*, const srftkv_side*, const srftkv_side*, int, int, int, int, int, int,
                          const int*, float, uint64_t, int, void*, size_t, void*) {
    set_error("decode attention not built yet");
    return SRFTKV_ERR_INVALID;
}
size_t q4kv_decode_attention_workspace_size(int, int, int, int, int, int) { return 0; }
}
