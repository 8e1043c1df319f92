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
// runs the online softmax over its slice (key rows 4 at a time); the partial
// results of a row are then combined in shared memory with the softmax merge rule (formula 2 of
// "闪电注意力的数学原理" on the unite.ai page: m = max m_w, l = sum l_w e^(m_w - m), O = sum O_w
// e^(m_w - m) / l).
//
// Short sequences (the head's K and V together within 128 KB: N <= 256 at d = 64, N <= 128 at
// d = 128) first copy the keys the CTA needs into shared memory with two bulk copies, so that the
// key loop reads no global memory: one round trip to L2 or HBM instead of two per 4-key chunk.
// Longer sequences read the key rows from L2, every row of a chunk requested before any is used.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn_impl {

using namespace attn_sm103;

__device__ unsigned int g_attn_f32_error = 0;  // bounded waits of the staged kernel that gave up

namespace {
constexpr int F32_ROWS = 8;      // query rows per CTA
// key slices (warps) per CTA: 16 at d = 64, 8 at d = 128 (the merge buffer, 16 or 8 x 8 rows x d fp32,
// stays at 32 KB)
template <int D>
struct F32Cfg {
    static constexpr int WARPS = D == 64 ? 16 : 8;
    static constexpr int THREADS = 32 * WARPS;
};
constexpr int F32_STAGE_BYTES = 128 * 1024;  // shared memory for K and V of a short head
}  // namespace

// A key row's four floats: shared memory (staged) or the read-only global path.
template <bool STAGED>
__device__ __forceinline__ float4 ld_row4(const float4* a) {
    if constexpr (STAGED) return *a;
    else return __ldg(a);
}

// STAGED: K and V rows [0, limit) of the head are copied into shared memory first (dynamic, 2 N d
// fp32); otherwise they are read from global memory.
template <int D, bool STAGED>
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

    const size_t kv_head = (static_cast<size_t>(b) * p.H_kv + kvh) * static_cast<size_t>(p.N) * D;
    const float* Kp = p.K + kv_head + part * CPL;
    const float* Vp = p.V + kv_head + part * CPL;
    if constexpr (STAGED) {
        extern __shared__ __align__(128) float f32_kv[];  // K rows [0, N), then V rows [0, N)
        __shared__ __align__(8) uint64_t kv_bar;
        if (threadIdx.x == 0) {
            mbar_init(&kv_bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (threadIdx.x == 0 && limit > 0) {
            const uint32_t bytes = static_cast<uint32_t>(limit) * D * 4;  // whole rows: a multiple of 16
            mbar_arrive_expect_tx(&kv_bar, 2 * bytes);
            bulk_load(f32_kv, p.K + kv_head, bytes, &kv_bar);
            bulk_load(f32_kv + static_cast<size_t>(p.N) * D, p.V + kv_head, bytes, &kv_bar);
        }
        volatile int never = 0;
        const bool got = limit > 0 ? mbar_wait(&kv_bar, 0, p.wait_limit_ns, &never) : true;
        if (!__syncthreads_and(got)) {
            // the copies did not land in time: record it, wait (bounded) for them once more so that
            // none writes shared memory after the CTA has exited, and write nothing
            if (threadIdx.x == 0) {
                atomicOr(&g_attn_f32_error, 1u);
                (void)mbar_wait(&kv_bar, 0, p.wait_limit_ns, &never);
            }
            return;
        }
        Kp = f32_kv + part * CPL;
        Vp = f32_kv + static_cast<size_t>(p.N) * D + part * CPL;
    }

    // A lane's CPL columns are CPL / 4 float4 chunks; its i-th access takes chunk (i + rot) mod
    // (CPL / 4), rotated by its quarter, so that the four quarters of a row (whose chunks would share
    // bank groups: 64 or 128 bytes apart) read different bank groups in every quarter-warp phase. q and
    // o are kept in that rotated order; the dot product is a sum, so the order does not matter.
    constexpr int NCH = CPL / 4;
    const int rot = part * (NCH / 4);
    float q[CPL], o[CPL];
    {
        const float4* q4 = reinterpret_cast<const float4*>(
            p.Q + (static_cast<size_t>(bh) * p.N + (row_ok ? row : 0)) * D + part * CPL);
#pragma unroll
        for (int i = 0; i < CPL / 4; ++i) {
            const float4 v = row_ok ? __ldg(q4 + ((i + rot) % NCH)) : make_float4(0.f, 0.f, 0.f, 0.f);
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
                kv[j][i] = (k0 + j < k_end) ? ld_row4<STAGED>(k4 + (i + rot) % NCH) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float s[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            // four independent partial sums (x, y, z, w lanes of the float4s), added at the end
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int i = 0; i < CPL / 4; ++i) {
                a0 = fmaf(q[4 * i], kv[j][i].x, a0);
                a1 = fmaf(q[4 * i + 1], kv[j][i].y, a1);
                a2 = fmaf(q[4 * i + 2], kv[j][i].z, a2);
                a3 = fmaf(q[4 * i + 3], kv[j][i].w, a3);
            }
            float acc = (a0 + a1) + (a2 + a3);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            s[j] = (k0 + j < k_end && k0 + j < row_lim) ? acc * p.scale : -INFINITY;
        }
#pragma unroll
        for (int j = 0; j < CH; ++j) {  // V rows of the chunk into the registers K used
            const float4* v4 = reinterpret_cast<const float4*>(Vp + static_cast<size_t>(k0 + j) * D);
#pragma unroll
            for (int i = 0; i < CPL / 4; ++i)
                kv[j][i] = (k0 + j < k_end) ? ld_row4<STAGED>(v4 + (i + rot) % NCH) : make_float4(0.f, 0.f, 0.f, 0.f);
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
    for (int i = 0; i < CPL / 4; ++i)  // back to column order
        reinterpret_cast<float4*>(&sm_o[warp][r][part * CPL])[(i + rot) % NCH] =
            make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    if (part == 0) {
        sm_m[warp][r] = l > 0.f ? m : -INFINITY;
        sm_l[warp][r] = l;
    }
    __syncthreads();
    // merge weights per (slice, row): e^(m_w - M) for slices with weight, 1 / L and the LSE per row;
    // thread w + F32_WARPS * rr takes slice w of row rr, the maximum and the sum over a row's slices
    // are reduced across the lanes that hold them (F32_WARPS consecutive lanes)
    if (threadIdx.x < F32_WARPS * F32_ROWS) {
        const int w = threadIdx.x % F32_WARPS, rr = threadIdx.x / F32_WARPS;
        const float mw = sm_m[w][rr], lw = sm_l[w][rr];
        float M = mw;
#pragma unroll
        for (int o = F32_WARPS / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float wt = lw > 0.f ? expf(mw - M) : 0.f;
        sm_w[w][rr] = wt;
        float L = wt * lw;
        // the sum over slices in the fixed order of a butterfly (every lane of the row gets the same L)
#pragma unroll
        for (int o = F32_WARPS / 2; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (w == 0) {
            sm_inv[rr] = L > 0.f ? 1.f / L : 0.f;
            sm_lse[rr] = L > 0.f ? M + logf(L) : -INFINITY;
        }
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

template <int D>
static cudaError_t launch_f32_t(const F32Params& p, dim3 grid, cudaStream_t stream) {
    const size_t staged_bytes = 2 * static_cast<size_t>(p.N) * D * sizeof(float);
    if (staged_bytes <= F32_STAGE_BYTES) {
        static std::atomic<int> ready[64];  // once per device: the shared-memory opt-in
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || ready[dev].load(std::memory_order_acquire) == 0) {
            e = cudaFuncSetAttribute(attn_fwd_f32_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     F32_STAGE_BYTES);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) ready[dev].store(1, std::memory_order_release);
        }
        attn_fwd_f32_kernel<D, true><<<grid, F32Cfg<D>::THREADS, staged_bytes, stream>>>(p);
    } else {
        attn_fwd_f32_kernel<D, false><<<grid, F32Cfg<D>::THREADS, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_attn_f32(int d, const F32Params& p, cudaStream_t stream) {
    dim3 grid((p.N + F32_ROWS - 1) / F32_ROWS, p.B * p.H);
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    if (d == 64) return launch_f32_t<64>(p, grid, stream);
    if (d == 128) return launch_f32_t<128>(p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_f32_error(uint32_t* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_f32_error, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_attn_f32_error, &zero, sizeof(zero));
    *out = v ? (ERRBIT_TIMEOUT | ERRBIT_WAIT_KV) : 0u;
    return e;
}

}  // namespace attn_impl
