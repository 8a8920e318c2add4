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
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made on that device; that first call should therefore come
// before any stream capture.  All calls share the one array and it keeps the
// contents of the last call: two calls whose work overlaps on the GPU (for
// example on two streams) race on it.  Nothing in it needs to start at zero:
// every call writes all the scratch it reads.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace srftkv {

static __device__ __align__(256) unsigned char g_attention_scratch[SRFTKV_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
}  // namespace

// Device address of the scratch array on the current device (looked up once).
static int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        set_error("q4kv_decode_attention_static: no usable current CUDA device");
        return SRFTKV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attention_scratch);
        if (e != cudaSuccess || !p) {
            set_error("q4kv_decode_attention_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            return SRFTKV_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SRFTKV_OK;
}

}  // namespace srftkv

using namespace srftkv;

extern "C" int q4kv_decode_attention_static(const void* q, float* out, const srftkv_side* k, const srftkv_side* v,
                                            int B, int Hq, int Hkv, int d, int group, int t_cap, const int* seq_lens,
                                            float sm_scale, uint64_t sign_seed, int n_splits, void* stream) {
    const size_t need = attention_workspace_size(B, Hq, Hkv, d, t_cap, n_splits);
    if (need == 0)  // invalid sizes (or nothing to do): the shared validation reports which
        return attention_entry(q, out, k, v, B, Hq, Hkv, d, group, t_cap, seq_lens, sm_scale, sign_seed, n_splits,
                               nullptr, 0, static_cast<cudaStream_t>(stream));
    if (need > (size_t)SRFTKV_STATIC_SCRATCH_BYTES) {
        set_error("q4kv_decode_attention_static: these sizes need %zu bytes of scratch but the static array holds %zu; "
                  "pass fewer n_splits or use q4kv_decode_attention with a caller workspace",
                  need, (size_t)SRFTKV_STATIC_SCRATCH_BYTES);
        return SRFTKV_ERR_INVALID;
    }
    void* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc) return rc;
    return attention_entry(q, out, k, v, B, Hq, Hkv, d, group, t_cap, seq_lens, sm_scale, sign_seed, n_splits,
                           scratch, (size_t)SRFTKV_STATIC_SCRATCH_BYTES, static_cast<cudaStream_t>(stream));
}
