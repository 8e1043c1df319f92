// Exact-fp32 attention forward on the CUDA cores (fp32 inputs).
//
// The tensor cores have no fp32 mode accurate enough for fp32 inputs (tf32 keeps 10 mantissa bits),
// so fp32 inputs take this path: fp32 FMAs and the accurate expf/logf. Same tiled method as the
// tensor-core kernel: online softmax over key tiles with running maximum m and running sum l, the
// unnormalised accumulator rescaled by exp(m_old - m_new), a single final division, and the row
// log-sum-exp (safe_softmax_block listing of "AI训练的最大障碍不是算力,而是'内存墙'", zsdodo.com;
// section 4.1.3 of "第四章 注意力机制实战案例", aiknowledge.cn).
//
// Mapping: a CTA of 16 warps (d = 64) or 8 (d = 128) owns 8 query rows of one (b, h) and splits the
// key range into one slice per warp, so that short sequences still spread over many warps: in a warp, four
// consecutive lanes share a row and each holds a quarter of its query and output columns. Every warp
// runs the online softmax over its slice (key rows read straight from L2, 4 at a time); the partial
// results of a row are then combined in shared memory with the softmax merge rule (formula 2 of
// "闪电注意力的数学原理" on the unite.ai page: m = max m_w, l = sum l_w e^(m_w - m), O = sum O_w
// e^(m_w - m) / l).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn_internal.h"

namespace attn_impl {

namespace {
constexpr int F32_ROWS = 8;      // query rows per CTA
// key slices (warps) per CTA: 16 at d = 64, 8 at d = 128 (the merge buffer, 16 or 8 x 8 rows x d fp32,
// stays at 32 KB)
template <int D>
struct F32Cfg {
    static constexpr int WARPS = D == 64 ? 16 : 8;
    static constexpr int THREADS = 32 * WARPS;
};
}  // namespace

template <int D>
__global__ void __launch_bounds__(F32Cfg<D>::THREADS, 1) attn_fwd_f32_kernel(const F32Params p) {
    constexpr int F32_WARPS = F32Cfg<D>::WARPS;
    constexpr int F32_THREADS = F32Cfg<D>::THREADS;
    constexpr int CPL = D / 4;            // columns per lane
    constexpr int CH = 4;                 // keys per online-softmax update (their rows held in registers)
    __shared__ __align__(16) float sm_o[F32_WARPS][F32_ROWS][D];
    __shared__ float sm_m[F32_WARPS][F32_ROWS], sm_l[F32_WARPS][F32_ROWS];
    __shared__ float sm_w[F32_WARPS][F32_ROWS], sm_inv[F32_ROWS], sm_lse[F32_ROWS];

    const int bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    const int kvh = h / p.group;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, part = lane & 3;
    const int q_start = blockIdx.x * F32_ROWS;
    const int row = q_start + r;
    const bool row_ok = row < p.N;

    int kv_valid = p.N;
    if (p.kv_len) {
        kv_valid = p.kv_len[b];
        kv_valid = kv_valid < 0 ? 0 : (kv_valid > p.N ? p.N : kv_valid);
    }
    // keys any row of the CTA may attend to, split into one slice per warp
    const int limit = p.causal ? min(kv_valid, q_start + F32_ROWS) : kv_valid;
    const int per_warp = (limit + F32_WARPS - 1) / F32_WARPS;
    const int k_begin = warp * per_warp;
    const int k_end = min(limit, k_begin + per_warp);
    const int row_lim = p.causal ? min(kv_valid, row + 1) : kv_valid;  // keys < row_lim are valid

    const float* Kp = p.K + (static_cast<size_t>(b) * p.H_kv + kvh) * static_cast<size_t>(p.N) * D + part * CPL;
    const float* Vp = p.V + (static_cast<size_t>(b) * p.H_kv + kvh) * static_cast<size_t>(p.N) * D + part * CPL;

    float q[CPL], o[CPL];
    {
        const float4* q4 = reinterpret_cast<const float4*>(
            p.Q + (static_cast<size_t>(bh) * p.N + (row_ok ? row : 0)) * D + part * CPL);
#pragma unroll
        for (int i = 0; i < CPL / 4; ++i) {
            const float4 v = row_ok ? __ldg(q4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            q[4 * i] = v.x; q[4 * i + 1] = v.y; q[4 * i + 2] = v.z; q[4 * i + 3] = v.w;
        }
    }
#pragma unroll
    for (int i = 0; i < CPL; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int k0 = k_begin; k0 < k_end; k0 += CH) {  // warp-uniform loop
        // every key row of the chunk is requested before any is used, so that the chunk costs one
        // memory latency for K and one for V (issued while the exponentials run)
        float4 kv[CH][CPL / 4];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const float4* k4 = reinterpret_cast<const float4*>(Kp + static_cast<size_t>(k0 + j) * D);
#pragma unroll
            for (int i = 0; i < CPL / 4; ++i)
                kv[j][i] = (k0 + j < k_end) ? __ldg(k4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float s[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < CPL / 4; ++i) {
                acc = fmaf(q[4 * i], kv[j][i].x, acc);
                acc = fmaf(q[4 * i + 1], kv[j][i].y, acc);
                acc = fmaf(q[4 * i + 2], kv[j][i].z, acc);
                acc = fmaf(q[4 * i + 3], kv[j][i].w, acc);
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            s[j] = (k0 + j < k_end && k0 + j < row_lim) ? acc * p.scale : -INFINITY;
        }
#pragma unroll
        for (int j = 0; j < CH; ++j) {  // V rows of the chunk into the registers K used
            const float4* v4 = reinterpret_cast<const float4*>(Vp + static_cast<size_t>(k0 + j) * D);
#pragma unroll
            for (int i = 0; i < CPL / 4; ++i)
                kv[j][i] = (k0 + j < k_end) ? __ldg(v4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mt = s[0];
#pragma unroll
        for (int j = 1; j < CH; ++j) mt = fmaxf(mt, s[j]);
        const float m_new = fmaxf(m, mt);
        // no valid key yet: m_new = -inf, every probability is 0 and o, l stay 0
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
        l *= alpha;
#pragma unroll
        for (int i = 0; i < CPL; ++i) o[i] *= alpha;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const float pj = (s[j] == -INFINITY) ? 0.f : expf(s[j] - m_new);
            l += pj;
#pragma unroll
            for (int i = 0; i < CPL / 4; ++i) {
                o[4 * i] = fmaf(pj, kv[j][i].x, o[4 * i]);
                o[4 * i + 1] = fmaf(pj, kv[j][i].y, o[4 * i + 1]);
                o[4 * i + 2] = fmaf(pj, kv[j][i].z, o[4 * i + 2]);
                o[4 * i + 3] = fmaf(pj, kv[j][i].w, o[4 * i + 3]);
            }
        }
        m = m_new;
    }

    // this warp's partial result of its slice: unnormalised O, m, l per row
#pragma unroll
    for (int i = 0; i < CPL / 4; ++i)
        reinterpret_cast<float4*>(&sm_o[warp][r][part * CPL])[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    if (part == 0) {
        sm_m[warp][r] = l > 0.f ? m : -INFINITY;
        sm_l[warp][r] = l;
    }
    __syncthreads();
    // merge weights per (slice, row): e^(m_w - M) for slices with weight, 1 / L and the LSE per row
    if (threadIdx.x < F32_ROWS) {
        const int rr = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < F32_WARPS; ++w) M = fmaxf(M, sm_m[w][rr]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < F32_WARPS; ++w) {
            const float wt = sm_l[w][rr] > 0.f ? expf(sm_m[w][rr] - M) : 0.f;
            sm_w[w][rr] = wt;
            L = fmaf(wt, sm_l[w][rr], L);
        }
        sm_inv[rr] = L > 0.f ? 1.f / L : 0.f;
        sm_lse[rr] = L > 0.f ? M + logf(L) : -INFINITY;
    }
    __syncthreads();
    float* Op = static_cast<float*>(p.O) + static_cast<size_t>(bh) * p.N * D;
    for (int idx = threadIdx.x; idx < F32_ROWS * D; idx += F32_THREADS) {
        const int rr = idx / D, c = idx % D;
        if (q_start + rr >= p.N) continue;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < F32_WARPS; ++w) acc = fmaf(sm_w[w][rr], sm_o[w][rr][c], acc);
        Op[static_cast<size_t>(q_start + rr) * D + c] = acc * sm_inv[rr];
    }
    if (p.LSE && threadIdx.x < F32_ROWS && q_start + threadIdx.x < p.N)
        p.LSE[static_cast<size_t>(bh) * p.N + q_start + threadIdx.x] = sm_lse[threadIdx.x];
}

cudaError_t launch_attn_f32(int d, const F32Params& p, cudaStream_t stream) {
    dim3 grid((p.N + F32_ROWS - 1) / F32_ROWS, p.B * p.H);
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    if (d == 64)
        attn_fwd_f32_kernel<64><<<grid, F32Cfg<64>::THREADS, 0, stream>>>(p);
    else if (d == 128)
        attn_fwd_f32_kernel<128><<<grid, F32Cfg<128>::THREADS, 0, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace attn_impl
