// attn_fwd_noalloc: the attention forward for callers that cannot allocate device memory.
//
// attn_fwd takes its scratch (the fp16 copy of V and the per-head range data) from a workspace the
// caller allocates. Some callers cannot call cudaMalloc or a caching allocator at the point where
// they run attention: code inside a host callback or a custom allocator's own hooks, a runtime
// whose memory pool is fixed at start-up and fully handed out, or plug-in hosts that forbid device
// allocation after initialisation. For them this file holds one fixed scratch array in device
// global memory, created when the library's code is loaded on a GPU, and an entry point that
// passes that array to attn_fwd as its workspace.
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
void* g_scratch_ptr[kMaxDevices] = {};  // device address of the array, per device ordinal

// Device address of the scratch array on the current device (looked up once per device, with that
// device current). Returns nullptr on failure.
void* scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
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
