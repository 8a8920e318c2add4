// attention_noalloc.cu -- decode attention for callers that cannot allocate
// device memory.
//
// q4kv_decode_attention needs a scratch workspace (the prepared queries and
// the per-split partial results).  Most callers allocate it once and pass it
// in.  Some callers cannot allocate device memory at call time at all: a
// host runtime that has already handed all device memory to its own pool, a
// plugin that sits behind a C ABI with no access to its host framework's
// allocator, or latency-critical code that cannot afford the implicit device
// synchronisation of cudaMalloc.  For them this file keeps the scratch in a
// file-scope device array of fixed size, SRFTKV_STATIC_SCRATCH_BYTES, which
// every GPU that loads the library holds until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// is only a stand-in symbol), so the address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call made in a
// CUDA context (for the runtime's usual primary context: once per device) and
// cached under that context's ID; that first call should therefore come
// before any stream capture.  All calls share the one array and it keeps the
// contents of the last call: two calls whose work overlaps on the GPU (for
// example on two streams) race on it.  Nothing in it needs to start at zero:
// every call writes all the scratch it reads.
#include <cuda_runtime.h>

#include "internal.h"

namespace srftkv {

static __device__ __align__(256) unsigned char g_attention_scratch[SRFTKV_STATIC_SCRATCH_BYTES];

// Device address of the scratch array in the current context (looked up once per context).
static int scratch_for_current_context(void** out) {
    static SymbolCache cache;
    return symbol_address(cache, g_attention_scratch, out, "the static attention scratch array");
}

}  // namespace srftkv

using namespace srftkv;

extern "C" int q4kv_decode_attention_static(const void* q, float* out, const srftkv_side* k, const srftkv_side* v,
                                            int B, int Hq, int Hkv, int d, int group, int t_cap, const int* seq_lens,
                                            float sm_scale, uint64_t sign_seed, int n_splits, void* stream) {
    // the arguments first, so that a bad call reports its own error rather than the array's size
    int rc = attention_check(q, out, k, v, B, Hq, Hkv, d, group, t_cap, n_splits);
    if (rc) return rc;
    if (B == 0) return SRFTKV_OK;
    rc = current_device_ok();
    if (rc) return rc;
    const size_t cap = (size_t)SRFTKV_STATIC_SCRATCH_BYTES;
    int ns = n_splits;
    if (ns == 0) {  // the automatic count, lowered until the workspace fits the array
        ns = attention_auto_splits(B, Hq, Hkv, t_cap);
        while (ns > 1 && attention_workspace_size(B, Hq, Hkv, d, t_cap, ns) > cap) --ns;
    }
    const size_t need = attention_workspace_size(B, Hq, Hkv, d, t_cap, ns);
    if (need > cap) {
        set_error("q4kv_decode_attention_static: these sizes need %zu bytes of scratch with %d split(s) but the static "
                  "array holds %zu; pass fewer n_splits, a smaller batch, or use q4kv_decode_attention with a caller "
                  "workspace",
                  need, ns, cap);
        return SRFTKV_ERR_INVALID;
    }
    void* scratch = nullptr;
    rc = scratch_for_current_context(&scratch);
    if (rc) return rc;
    return attention_entry(q, out, k, v, B, Hq, Hkv, d, group, t_cap, seq_lens, sm_scale, sign_seed, ns, scratch, cap,
                           static_cast<cudaStream_t>(stream));
}
