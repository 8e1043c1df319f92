// Exact-fp32 attention forward on the CUDA cores (fp32 inputs).
//
// The tensor cores have no fp32 mode accurate enough for fp32 inputs (tf32 keeps 10 mantissa bits),
// so fp32 inputs take this path: fp32 FMAs and the accurate expf/logf. Same tiled method as the
// tensor-core kernel: online softmax over key tiles with running maximum m and running sum l, the
// unnormalised accumulator rescaled by exp(m_old - m_new), a single final division, and the row
// log-sum-exp (safe_softmax_block listing of "AI训练的最大障碍不是算力,而是'内存墙'", zsdodo.com;
// section 4.1.3 of "第四章 注意力机制实战案例", aiknowledge.cn).
//
// Mapping: a CTA of 128 threads owns 32 query rows of one (b, h); four consecutive lanes share a
// row, each holding the query and output columns c = part + 4 i (interleaved, so that the four
// lanes read consecutive shared-memory banks). Key/value tiles of 32 rows are staged in shared
// memory with coalesced float4 loads.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn_internal.h"

namespace attn_impl {

namespace {
constexpr int F32_ROWS = 32;
constexpr int F32_KT = 32;
constexpr int F32_THREADS = 128;
}  // namespace

template <int D>
__global__ void __launch_bounds__(F32_THREADS) attn_fwd_f32_kernel(const F32Params p) {
    constexpr int CPT = D / 4;  // columns per thread
    __shared__ __align__(16) float sK[F32_KT][D];
    __shared__ __align__(16) float sV[F32_KT][D];

    const int bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    const int kvh = h / p.group;
    const int q_start = blockIdx.x * F32_ROWS;
    const int tid = threadIdx.x;
    const int part = tid & 3;
    const int row = q_start + (tid >> 2);
    const bool row_ok = row < p.N;

    int kv_valid = p.N;
    if (p.kv_len) {
        kv_valid = p.kv_len[b];
        kv_valid = kv_valid < 0 ? 0 : (kv_valid > p.N ? p.N : kv_valid);
    }
    const int limit = p.causal ? min(kv_valid, q_start + F32_ROWS) : kv_valid;
    const int row_lim = p.causal ? min(kv_valid, row + 1) : kv_valid;

    const float* Qp = p.Q + (static_cast<size_t>(bh) * p.N + (row_ok ? row : 0)) * D;
    const float* Kp = p.K + (static_cast<size_t>(b) * p.H_kv + kvh) * static_cast<size_t>(p.N) * D;
    const float* Vp = p.V + (static_cast<size_t>(b) * p.H_kv + kvh) * static_cast<size_t>(p.N) * D;

    float q[CPT], o[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        q[i] = row_ok ? Qp[part + 4 * i] : 0.f;
        o[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;

    for (int k0 = 0; k0 < limit; k0 += F32_KT) {
        __syncthreads();
        // stage K and V rows [k0, k0 + 32) (zero past N)
        for (int idx = tid; idx < F32_KT * D / 4; idx += F32_THREADS) {
            const int kr = idx / (D / 4), c4 = idx % (D / 4);
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (k0 + kr < p.N) {
                kv = reinterpret_cast<const float4*>(Kp + static_cast<size_t>(k0 + kr) * D)[c4];
                vv = reinterpret_cast<const float4*>(Vp + static_cast<size_t>(k0 + kr) * D)[c4];
            }
            reinterpret_cast<float4*>(&sK[kr][0])[c4] = kv;
            reinterpret_cast<float4*>(&sV[kr][0])[c4] = vv;
        }
        __syncthreads();
        float s[F32_KT];
#pragma unroll
        for (int j = 0; j < F32_KT; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < CPT; ++i) acc = fmaf(q[i], sK[j][part + 4 * i], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            s[j] = (k0 + j < row_lim) ? acc * p.scale : -INFINITY;
        }
        float mt = s[0];
#pragma unroll
        for (int j = 1; j < F32_KT; ++j) mt = fmaxf(mt, s[j]);
        const float m_new = fmaxf(m, mt);
        if (m_new == -INFINITY) continue;  // nothing valid for this row yet
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) o[i] *= alpha;
#pragma unroll
        for (int j = 0; j < F32_KT; ++j) {
            const float pj = (s[j] == -INFINITY) ? 0.f : expf(s[j] - m_new);
            psum += pj;
#pragma unroll
            for (int i = 0; i < CPT; ++i) o[i] = fmaf(pj, sV[j][part + 4 * i], o[i]);
        }
        l = fmaf(alpha, l, psum);
        m = m_new;
    }

    if (!row_ok) return;
    float* Op = static_cast<float*>(p.O) + (static_cast<size_t>(bh) * p.N + row) * D;
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int i = 0; i < CPT; ++i) Op[part + 4 * i] = o[i] * inv;
    if (p.LSE && part == 0) p.LSE[static_cast<size_t>(bh) * p.N + row] = (l > 0.f) ? m + logf(l) : -INFINITY;
}

cudaError_t launch_attn_f32(int d, const F32Params& p, cudaStream_t stream) {
    dim3 grid((p.N + F32_ROWS - 1) / F32_ROWS, p.B * p.H);
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    if (d == 64)
        attn_fwd_f32_kernel<64><<<grid, F32_THREADS, 0, stream>>>(p);
    else if (d == 128)
        attn_fwd_f32_kernel<128><<<grid, F32_THREADS, 0, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace attn_impl
