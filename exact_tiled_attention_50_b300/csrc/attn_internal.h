// Internal interface between the C-ABI front end (attn_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn_impl {

// Bits recorded in the device error word by the tensor-core kernel.
enum : uint32_t {
    ERRBIT_TIMEOUT = 1u,        // some bounded wait gave up
    ERRBIT_WAIT_Q = 2u,         // which role/wait (diagnostics only)
    ERRBIT_WAIT_KV = 4u,
    ERRBIT_WAIT_S = 8u,
    ERRBIT_WAIT_P = 16u,
    ERRBIT_WAIT_O = 32u,
    ERRBIT_WAIT_EMPTY = 64u,
    ERRBIT_WAIT_DRAIN = 128u,
};

struct TcParams {
    void* O;                  // [B,H,N,d] fp32 or bf16
    float* LSE;               // [B,H,N] or nullptr
    const int32_t* kv_len;    // [B] or nullptr
    const int32_t* v_exp;     // [B*H_kv] power-of-two exponent of the fp16 copy of V
    int B, H, H_kv, N;
    int group;                // H / H_kv
    int n_pairs;              // ceil(N / 256): CTA work units per (b, h)
    int causal;
    float scale_log2;         // scale * log2(e)
    unsigned long long wait_limit_ns;
    int debug_skip_kv_load;
};

struct F32Params {
    const float* Q;
    const float* K;
    const float* V;
    void* O;                  // fp32
    float* LSE;
    const int32_t* kv_len;
    int B, H, H_kv, N, group, causal;
    float scale;
};

// V (bf16 [rows, d] per head) -> fp16 copy scaled by 2^-e per head (e chosen so |V| * 2^-e < 2^15).
struct VPrepParams {
    const void* V;            // bf16 [B*H_kv, N, d]
    void* V16;                // fp16 [B*H_kv, N, d]
    float* partial_max;       // [B*H_kv, chunks]
    int32_t* v_exp;           // [B*H_kv]
    long long elems_per_head; // N * d
    int chunks;               // per head
    int heads;                // B * H_kv
};

constexpr int VPREP_CHUNK = 16384;  // elements of V per CTA in the fp16 conversion

cudaError_t launch_vprep(const VPrepParams& p, cudaStream_t stream);
cudaError_t launch_attn_tc(int d, bool out_bf16, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV16, const TcParams& p, cudaStream_t stream);
cudaError_t launch_attn_f32(int d, const F32Params& p, cudaStream_t stream);

// Device error word of the current device: read and clear (synchronous on `stream`).
cudaError_t read_and_clear_error(uint32_t* out, cudaStream_t stream);

}  // namespace attn_impl
