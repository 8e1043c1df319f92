// attn_fwd_noalloc: the attention forward for callers that cannot allocate device memory.
//
// attn_fwd takes its scratch (the fp16 copy of V and the per-head range data) from a workspace the
// caller allocates. Some callers cannot call cudaMalloc or a caching allocator at the point where
// they run attention: code inside a host callback or a custom allocator's own hooks, a runtime
// whose memory pool is fixed at start-up and fully handed out, or plug-in hosts that forbid device
// allocation after initialisation. For them this file holds one fixed scratch array in device
// global memory and an entry point that passes that array to attn_fwd as its workspace.
//
// The array belongs to this library's device code, which CUDA loads on a device when the library
// first needs it there (with lazy module loading, the default, that is the first
// cudaGetSymbolAddress below): the first attn_fwd_noalloc call on a device therefore reserves the
// array's 64 MiB. Callers make that first call during their initialisation.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/attn.h"

namespace {

// The scratch array. Every GPU that loads the library holds it until the process exits. In host
// code its name is only a host-side stand-in, never a device address: the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;

// Device address of the array per device ordinal, and the context it was looked up in: after a
// cudaDeviceReset the device gets a new primary context, the array a new address, and the cached one
// must not be handed to a kernel.
struct Cached {
    void* ptr = nullptr;
    unsigned long long ctx_id = 0;
    bool have_id = false;
};
Cached g_cache[kMaxDevices];

// Driver calls that identify the current context (fetched through the runtime, so the library does not
// link the driver library itself). When they are unavailable the address is looked up on every call.
typedef CUresult (*PFN_ctxGetCurrent)(CUcontext*);
typedef CUresult (*PFN_ctxGetId)(CUcontext, unsigned long long*);
PFN_ctxGetCurrent g_ctx_get_current = nullptr;
PFN_ctxGetId g_ctx_get_id = nullptr;
std::once_flag g_driver_once;

void load_driver_calls() {
    std::call_once(g_driver_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PFN_ctxGetCurrent>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PFN_ctxGetId>(fn);
    });
}

// Identifier of the calling thread's current context; false when it cannot be determined.
bool current_context_id(unsigned long long* id) {
    load_driver_calls();
    if (!g_ctx_get_current || !g_ctx_get_id) return false;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array on the current device, looked up with that device current
// (once per device and context). Returns nullptr on failure.
void* scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);  // false before the runtime made a context current
    std::lock_guard<std::mutex> lock(g_mutex);
    Cached& c = g_cache[dev];
    if (c.ptr && have_id && c.have_id && c.ctx_id == id) return c.ptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    if (!have_id) have_id = current_context_id(&id);  // the lookup made the device's context current
    c.ptr = p;
    c.ctx_id = id;
    c.have_id = have_id;
    return p;
}

}  // namespace

extern "C" attn_status attn_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                                        int H_kv, int N, int d, float scale, int causal, const int32_t* kv_len,
                                        attn_dtype in_dtype, attn_dtype out_dtype, cudaStream_t stream) {
    if (in_dtype != ATTN_BF16)  // fp32 inputs need no scratch at all
        return attn_fwd(Q, K, V, O, LSE, B, H, H_kv, N, d, scale, causal, kv_len, in_dtype, out_dtype, nullptr, 0,
                        stream);
    const size_t need = attn_workspace_bytes(B, H, H_kv, N, d, in_dtype);
    if (need == 0)  // sizes attn_fwd rejects: let it return its own error code (nothing is launched)
        return attn_fwd(Q, K, V, O, LSE, B, H, H_kv, N, d, scale, causal, kv_len, in_dtype, out_dtype, nullptr, 0,
                        stream);
    if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;  // larger than the fixed scratch
    void* scratch = scratch_for_current_device();
    if (!scratch) return ATTN_ERR_CUDA;
    return attn_fwd(Q, K, V, O, LSE, B, H, H_kv, N, d, scale, causal, kv_len, in_dtype, out_dtype, scratch,
                    ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
