// Tensor-core attention backward for bf16 inputs on sm_103a (B300): dQ, dK, dV.
//
// The pages state the forward pass; its gradient is the chain rule through the same exact attention,
// in the recompute form of "闪电注意力：革命性地提高Transformer效率" (unite.ai, the key ideas: do not
// store the attention matrix, recompute its parts in the backward pass) with the row log-sum-exp of
// the forward: P = exp(scale Q K^T - LSE) (masked), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
// dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q.
//
// Blackwell mapping: one CTA per (key tile of 128 keys, batch, kv head); it keeps K_j and V_j in
// shared memory and accumulates dK_j and dV_j in tensor memory over every query head of its group and
// every query tile (causal: the tiles at or after the key tile). Two kernels share this mapping:
// attn_bwd_tc_kernel (d = 64, query tiles of 128 rows, described here) and attn_bwd_q64_kernel
// (d = 128, query tiles of 64 rows through a three-stage ring; described above it). Per query tile:
//   MMA warp      S^T = K_j Q_i^T, dP^T = V_j dO_i^T         (TMEM cols 0-127, 128-255)
//   warps 0-7     one key row each (warps 0-3 queries 0-63, warps 4-7 queries 64-127): P^T, dS^T ->
//                 bf16 in shared memory (128-byte swizzled)
//   MMA warp      dV += P^T dO_i, dK += dS^T Q_i (then Q_i, dO_i are released to the next loads),
//                 dQ_i = dS K_j   (dQ in cols 0-127)
//   warps 4-7     then one query row each: dQ_i scaled, staged in shared memory and added into the
//                 fp32 dQ in device memory by bulk tensor reductions (several key tiles add into the
//                 same rows); warps 0-3 write dK_j, dV_j at the end
//   warp 9        TMA loads (K_j, V_j once; Q_i, dO_i and the row statistics per tile)
// All waits are bounded as in the forward kernel; a wait that runs out records an error bit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn_impl {

using namespace attn_sm103;

__device__ unsigned int g_attn_bwd_error = 0;

namespace {

constexpr int BW_THREADS = 384;
constexpr int BW_MMA_WARP = 8;
constexpr int BW_TMA_WARP = 9;

// P^T and dS^T of one key row over 32 queries whose every pair is valid, as bf16 pairs: P = 2^(s sl -
// lse2), dS = P (dP - D), with the row statistics read as float4 and the arithmetic two-wide (the same
// single-rounded fma and product per pair as the masked form).
__device__ __forceinline__ void bwd_pds_valid32(const uint32_t (&sv)[32], const uint32_t (&dpv)[32], const float* lse2,
                                                const float* dvec, float sl, uint32_t (&pp)[16], uint32_t (&dd)[16]) {
    const float4* l4 = reinterpret_cast<const float4*>(lse2);
    const float4* d4 = reinterpret_cast<const float4*>(dvec);
    const f32x2 sl2 = make_f32x2(sl, sl);
#pragma unroll
    for (int i4 = 0; i4 < 8; ++i4) {
        const float4 lv = l4[i4], dq = d4[i4];
        const int i = 4 * i4;
        float x0, x1, x2, x3;
        split_f32x2(fma_f32x2(make_f32x2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), sl2,
                              make_f32x2(-lv.x, -lv.y)), x0, x1);
        split_f32x2(fma_f32x2(make_f32x2(__uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3])), sl2,
                              make_f32x2(-lv.z, -lv.w)), x2, x3);
        const f32x2 e01 = make_f32x2(ex2_approx(x0), ex2_approx(x1));
        const f32x2 e23 = make_f32x2(ex2_approx(x2), ex2_approx(x3));
        const f32x2 g01 = mul_f32x2(e01, add_f32x2(make_f32x2(__uint_as_float(dpv[i]), __uint_as_float(dpv[i + 1])),
                                                   make_f32x2(-dq.x, -dq.y)));
        const f32x2 g23 = mul_f32x2(e23, add_f32x2(make_f32x2(__uint_as_float(dpv[i + 2]), __uint_as_float(dpv[i + 3])),
                                                   make_f32x2(-dq.z, -dq.w)));
        float a0, a1, a2, a3, c0, c1, c2, c3;
        split_f32x2(e01, a0, a1);
        split_f32x2(e23, a2, a3);
        split_f32x2(g01, c0, c1);
        split_f32x2(g23, c2, c3);
        __nv_bfloat162 ph0 = __floats2bfloat162_rn(a0, a1), ph1 = __floats2bfloat162_rn(a2, a3);
        __nv_bfloat162 dh0 = __floats2bfloat162_rn(c0, c1), dh1 = __floats2bfloat162_rn(c2, c3);
        pp[2 * i4] = *reinterpret_cast<uint32_t*>(&ph0);
        pp[2 * i4 + 1] = *reinterpret_cast<uint32_t*>(&ph1);
        dd[2 * i4] = *reinterpret_cast<uint32_t*>(&dh0);
        dd[2 * i4 + 1] = *reinterpret_cast<uint32_t*>(&dh1);
    }
}

template <int D>
struct BwCfg {
    static constexpr int NB = D / 64;
    static constexpr int TILE = NB * 16384;   // 128 rows x D 16-bit values
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = TILE;
    static constexpr int OFF_Q = 2 * TILE;
    static constexpr int OFF_DO = 3 * TILE;
    static constexpr int OFF_PT = 4 * TILE;   // P^T  [128 keys][128 queries] bf16
    static constexpr int OFF_DST = OFF_PT + 32768;  // dS^T [128 keys][128 queries] bf16
    static constexpr int OFF_STAT = OFF_DST + 32768;  // lse2[128], dvec[128]
    static constexpr int OFF_DQS = OFF_STAT + 1024;   // dQ staging: 4 warps x (32 rows x 32 fp32), swizzled
    static constexpr int SMEM = 1024 + OFF_DQS + 4 * 4096;
    static constexpr uint32_t IDESC_SD = idesc_f16(128, 128, 1, 1, 0, 0);  // S^T, dP^T: K-major A and B
    static constexpr uint32_t IDESC_KV = idesc_f16(128, D, 1, 1, 0, 1);    // dV, dK: A K-major, B MN-major
    static constexpr uint32_t IDESC_Q = idesc_f16(128, D, 1, 1, 1, 1);     // dQ: A (dS) and B (K) MN-major
    static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 384, T_DQ = 0;
};

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void bw_fail(volatile int* abort_flag, uint32_t bits) {
    *abort_flag = 1;
    atomicOr(&g_attn_bwd_error, ERRBIT_TIMEOUT | bits);
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(BW_THREADS, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ BwdParams p) {
    using C = BwCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar_kv, bar_qdo_full, bar_qdo_empty, bar_s_full, bar_ps_full, bar_ps_empty,
        bar_dq_full, bar_dq_free, bar_done;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // causal: key tile jt has the query tiles from jt on, so the grid runs the key tiles in the slow
    // dimension and the costliest (first) key tiles of every head start first
    const int jt = p.causal ? blockIdx.y : blockIdx.x;   // key tile
    const int zkv = p.causal ? blockIdx.x : blockIdx.y;  // b * H_kv + kv head
    const int b = zkv / p.H_kv, hk = zkv - b * p.H_kv;
    const int N = p.N;
    int kv_valid = N;
    if (p.kv_len) {
        kv_valid = __ldg(p.kv_len + b);
        kv_valid = kv_valid < 0 ? 0 : (kv_valid > N ? N : kv_valid);
    }
    const int k0 = jt * 128;
    const bool any_keys = k0 < kv_valid;
    const int i_first = p.causal ? jt : 0;     // query tiles with at least one valid pair
    const int n_i = any_keys ? p.n_qt - i_first : 0;
    const int n_steps = n_i * p.group;         // (query head of the group, query tile) pairs
    const uint64_t limit_ns = p.wait_limit_ns;

    if (warp == BW_MMA_WARP) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(&bar_kv, 1);
        mbar_init(&bar_qdo_full, 1);
        mbar_init(&bar_qdo_empty, 1);
        mbar_init(&bar_s_full, 1);
        mbar_init(&bar_ps_full, 256);
        mbar_init(&bar_ps_empty, 1);
        mbar_init(&bar_dq_full, 1);
        mbar_init(&bar_dq_free, 128);
        mbar_init(&bar_done, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    // step s -> (query head, query tile)
    auto step_head = [&](int s) { return hk * p.group + s / n_i; };
    auto step_tile = [&](int s) { return i_first + s % n_i; };

    if (warp == BW_TMA_WARP) {
        // ====================================== TMA producer ======================================
        if (elect_one() && n_steps > 0) {
            mbar_arrive_expect_tx(&bar_kv, 2 * C::TILE);
            for (int bx = 0; bx < C::NB; ++bx) {
                tma_load_3d(smem + C::OFF_K + bx * 16384, &tmK, &bar_kv, bx * 64, k0, zkv);
                tma_load_3d(smem + C::OFF_V + bx * 16384, &tmV, &bar_kv, bx * 64, k0, zkv);
            }
            int issued = 0;
            for (int s = 0; s < n_steps; ++s) {
                if (s > 0 && !mbar_wait(&bar_qdo_empty, (s - 1) & 1, limit_ns, &abort_flag)) {
                    bw_fail(&abort_flag, ERRBIT_WAIT_EMPTY);
                    break;
                }
                const int bh = b * p.H + step_head(s), it = step_tile(s);
                mbar_arrive_expect_tx(&bar_qdo_full, 2 * C::TILE + 1024);
                for (int bx = 0; bx < C::NB; ++bx) {
                    tma_load_3d(smem + C::OFF_Q + bx * 16384, &tmQ, &bar_qdo_full, bx * 64, it * 128, bh);
                    tma_load_3d(smem + C::OFF_DO + bx * 16384, &tmDO, &bar_qdo_full, bx * 64, it * 128, bh);
                }
                const size_t srow = static_cast<size_t>(bh) * p.n_qt * 128 + static_cast<size_t>(it) * 128;
                bulk_load(smem + C::OFF_STAT, p.lse2 + srow, 512, &bar_qdo_full);
                bulk_load(smem + C::OFF_STAT + 512, p.dvec + srow, 512, &bar_qdo_full);
                issued = s + 1;
            }
            if (abort_flag) {  // wait (bounded) for the copies in flight before the CTA may exit
                volatile int never = 0;
                (void)mbar_wait(&bar_kv, 0, limit_ns, &never);
                if (issued > 0) (void)mbar_wait(&bar_qdo_full, (issued - 1) & 1, limit_ns, &never);
            }
        }
        __syncwarp();
    } else if (warp == BW_MMA_WARP) {
        // ======================================= MMA issuer =======================================
        auto wait_all = [&](uint64_t* bar, uint32_t parity, uint32_t bit) {
            const bool got = mbar_wait(bar, parity, limit_ns, &abort_flag);
            if (__all_sync(0xffffffffu, got)) return true;
            if (!got) bw_fail(&abort_flag, bit);
            return false;
        };
        const uint64_t dK_k = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);      // K as K-major A
        const uint64_t dV_k = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);      // V as K-major A
        const uint64_t dQ_k = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);      // Q as K-major B
        const uint64_t dDO_k = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);    // dO as K-major B
        const uint64_t dQ_mn = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16384, 1024);  // Q as MN-major B
        const uint64_t dDO_mn = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16384, 1024);
        const uint64_t dK_mn = sdesc_sw128(smem_u32(smem + C::OFF_K), 16384, 1024);  // K as MN-major B
        const uint64_t dPT_k = sdesc_sw128(smem_u32(smem + C::OFF_PT), 16, 1024);    // P^T as K-major A
        const uint64_t dDST_k = sdesc_sw128(smem_u32(smem + C::OFF_DST), 16, 1024);  // dS^T as K-major A
        const uint64_t dDS_mn = sdesc_sw128(smem_u32(smem + C::OFF_DST), 16384, 1024);  // dS as MN-major A
        // K-major operand over a 128 (or D) deep contraction: k-step kk of 16 elements
        auto kmaj = [](int kk) { return static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); };
        auto mnmaj = [](int kk) { return static_cast<uint64_t>((kk * 2048) >> 4); };
        bool ok = n_steps > 0 ? wait_all(&bar_kv, 0, ERRBIT_WAIT_KV) : true;
        for (int s = 0; s < n_steps && ok; ++s) {
            if (!wait_all(&bar_qdo_full, s & 1, ERRBIT_WAIT_Q)) { ok = false; break; }
            if (s > 0 && !wait_all(&bar_dq_free, (s - 1) & 1, ERRBIT_WAIT_O)) { ok = false; break; }
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_ss(tmem + C::T_S, dK_k + kmaj(kk), dQ_k + kmaj(kk), C::IDESC_SD, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_ss(tmem + C::T_DP, dV_k + kmaj(kk), dDO_k + kmaj(kk), C::IDESC_SD, kk > 0);
                umma_commit(&bar_s_full);
            }
            __syncwarp();
            if (!wait_all(&bar_ps_full, s & 1, ERRBIT_WAIT_P)) { ok = false; break; }
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // contraction over the 128 queries
                    umma_ss(tmem + C::T_DV, dPT_k + kmaj(kk), dDO_mn + mnmaj(kk), C::IDESC_KV, (s > 0 || kk > 0));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ss(tmem + C::T_DK, dDST_k + kmaj(kk), dQ_mn + mnmaj(kk), C::IDESC_KV, (s > 0 || kk > 0));
                umma_commit(&bar_qdo_empty);  // Q_i, dO_i read: the next tile's loads overlap the dQ product
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // contraction over the 128 keys
                    umma_ss(tmem + C::T_DQ, dDS_mn + mnmaj(kk), dK_mn + mnmaj(kk), C::IDESC_Q, kk > 0);
                umma_commit(&bar_dq_full);
                umma_commit(&bar_ps_empty);
            }
            __syncwarp();
        }
        if (elect_one()) umma_commit(&bar_done);  // every MMA issued above has completed
        __syncwarp();
        volatile int never = 0;
        const bool drained = mbar_wait(&bar_done, 0, limit_ns, &never);
        if (!__all_sync(0xffffffffu, drained) && lane == 0) bw_fail(&abort_flag, ERRBIT_WAIT_DRAIN);
    } else if (warp < 8) {
        // ==== warps 0-7: one key row each, warps 0-3 for queries 0-63 and warps 4-7 for queries 64-127;
        // P^T and dS^T into shared memory. Warps 4-7 then read dQ_i out of tensor memory as well. ====
        const int half = warp >> 2;
        const int r = (warp & 3) * 32 + lane;    // key row in the tile
        const int key = k0 + r;
        const uint32_t lane_off = tmem_lane_base(warp);
        const float sl = p.scale_log2;
        const float* lse2 = reinterpret_cast<const float*>(smem + C::OFF_STAT);
        const float* dvec = lse2 + 128;
        const uint32_t pt_row = smem_u32(smem + C::OFF_PT) + r * 128;
        const uint32_t dst_row = smem_u32(smem + C::OFF_DST) + r * 128;
        bool ok = true;
        for (int s = 0; s < n_steps && ok; ++s) {
            const int it = step_tile(s);
            const int q0 = it * 128;
            bool got = mbar_wait(&bar_s_full, s & 1, limit_ns, &abort_flag);
            got = got && mbar_wait(&bar_qdo_full, s & 1, limit_ns, &abort_flag);
            if (s > 0) got = got && mbar_wait(&bar_ps_empty, (s - 1) & 1, limit_ns, &abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (!got) bw_fail(&abort_flag, ERRBIT_WAIT_S);
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 2 * half; c < 2 * half + 2; ++c) {  // 32 queries at a time
                uint32_t sv[32], dpv[32];
                tmem_ld32(tmem + lane_off + C::T_S + c * 32, sv);
                tmem_ld32(tmem + lane_off + C::T_DP + c * 32, dpv);
                tmem_wait_ld(sv);
                tmem_wait_ld(dpv);
                uint32_t pp[16], dd[16];
                // every pair of the 32 valid: the fast path of the d = 128 kernel (no per-pair mask,
                // float4 row statistics, two-wide arithmetic)
                if (key < kv_valid && q0 + c * 32 + 31 < N && (!p.causal || key <= q0 + c * 32))
                    bwd_pds_valid32(sv, dpv, lse2 + c * 32, dvec + c * 32, sl, pp, dd);
                else
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float pv[2], dv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int qi = c * 32 + i + u;
                        const int q = q0 + qi;
                        const bool valid = key < kv_valid && q < N && (!p.causal || key <= q);
                        const float e = valid ? ex2_approx(__uint_as_float(sv[i + u]) * sl - lse2[qi]) : 0.f;
                        pv[u] = e;
                        dv[u] = e * (__uint_as_float(dpv[i + u]) - dvec[qi]);
                    }
                    __nv_bfloat162 ph = __floats2bfloat162_rn(pv[0], pv[1]);
                    __nv_bfloat162 dh = __floats2bfloat162_rn(dv[0], dv[1]);
                    pp[i / 2] = *reinterpret_cast<uint32_t*>(&ph);
                    dd[i / 2] = *reinterpret_cast<uint32_t*>(&dh);
                }
                // 32 queries = four 16-byte chunks of this row; box c / 2, chunk (c % 2) * 4 + k
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int ch = (c & 1) * 4 + k;
                    const uint32_t off = (c >> 1) * 16384 + ((ch ^ (r & 7)) << 4);
                    st_shared_v4(pt_row + off, pp[4 * k], pp[4 * k + 1], pp[4 * k + 2], pp[4 * k + 3]);
                    st_shared_v4(dst_row + off, dd[4 * k], dd[4 * k + 1], dd[4 * k + 2], dd[4 * k + 3]);
                }
            }
            fence_proxy_async_smem();  // the MMAs read P^T and dS^T through the async proxy
            tc_fence_before();
            mbar_arrive(&bar_ps_full);
            if (half == 1) {
                // dQ_i (query rows 32 (warp - 4) ..): scaled, staged in shared memory and added into device
                // memory by bulk tensor reductions (several key tiles add into the same dQ rows)
                const bool gq = mbar_wait(&bar_dq_full, s & 1, limit_ns, &abort_flag);
                if (!__all_sync(0xffffffffu, gq)) {
                    if (!gq) bw_fail(&abort_flag, ERRBIT_WAIT_O);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int bh = b * p.H + step_head(s);
                const int wq = warp & 3;
                const uint32_t stage = smem_u32(smem + C::OFF_DQS + wq * 4096);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + C::T_DQ + c * 32, v);
                    tmem_wait_ld(v);
                    if (c == D / 32 - 1) {  // tensor memory read out: the next S^T may overwrite it
                        tc_fence_before();
                        mbar_arrive(&bar_dq_free);
                    }
                    if (lane == 0) bulk_wait_group_read<0>();  // the staging buffer's previous box was read
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        st_shared_v4(stage + lane * 128 + ((k ^ (lane & 7)) << 4),
                                     __float_as_uint(__uint_as_float(v[4 * k]) * p.scale),
                                     __float_as_uint(__uint_as_float(v[4 * k + 1]) * p.scale),
                                     __float_as_uint(__uint_as_float(v[4 * k + 2]) * p.scale),
                                     __float_as_uint(__uint_as_float(v[4 * k + 3]) * p.scale));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {  // rows past N are not written by the reduction
                        tma_reduce_add_3d(&tmDQ, smem + C::OFF_DQS + wq * 4096, c * 32, it * 128 + wq * 32, bh);
                        bulk_commit_group();
                    }
                    __syncwarp();
                }
            }
        }
        if (half == 1) {
            if (lane == 0) bulk_wait_group_all();  // every reduction of this warp performed
            __syncwarp();
        }
        // ---- dK, dV of this key tile (warps 0-3): fp32 rows straight to device memory ----
        if (half == 0 && ok && n_steps > 0) {
            const bool got = mbar_wait(&bar_done, 0, limit_ns, &abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (!got) bw_fail(&abort_flag, ERRBIT_WAIT_DRAIN);
                ok = false;
            }
            tc_fence_after();
        }
        // ok and n_steps are warp-uniform; key < N is not (the last key tile of a ragged N), so every
        // lane takes part in the warp-collective tensor-memory loads and only the stores are guarded.
        if (half == 0 && ok) {
            const bool row_ok = key < N;
            const size_t orow = (static_cast<size_t>(zkv) * N + (row_ok ? key : 0)) * D;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                float* dst = (which ? p.dK : p.dV) + orow;
                const float mul = which ? p.scale : 1.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    if (n_steps > 0) {
                        tmem_ld32(tmem + lane_off + (which ? C::T_DK : C::T_DV) + c * 32, v);
                        tmem_wait_ld(v);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;
                    }
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(dst + c * 32 + i) =
                                make_float4(__uint_as_float(v[i]) * mul, __uint_as_float(v[i + 1]) * mul,
                                            __uint_as_float(v[i + 2]) * mul, __uint_as_float(v[i + 3]) * mul);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == BW_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------------------------
// d = 128: query tiles of 64 rows through a three-stage Q/dO ring, so that the next tiles' loads and
// its S^T, dP^T products overlap the current tile's P/dS work and dV, dK, dQ products. Per step s
// (query tile i of one head of the group) the MMA warp issues S^T(s), dP^T(s) (M = 128 keys, N = 64
// queries), then the second-phase products of step s - 1: dV += P^T dO, dK += dS^T Q (which release
// the ring stage), dQ^T = K^T dS^T (M = d, N = 64 queries) into one of two TMEM buffers. 512 threads:
// warps 0-7 compute P^T, dS^T (one key row per thread, 32 queries each); warps 8-11 (a warpgroup of
// their own, one TMEM lane quarter = 32 dimensions each) read dQ^T of each step, stage it as four
// [16 queries][32 dims] boxes through two buffers and reduce them into dQ, while warps 0-7 already
// work on the next step; warp 12 issues the MMAs, warp 13 loads.
// ---------------------------------------------------------------------------------------------
struct Bw2Cfg {
    static constexpr int D = 128;
    static constexpr int QT = 64;                        // query rows per step
    static constexpr int OFF_K = 0, OFF_V = 32768;       // 128 keys x 128 dims bf16, two 64-column boxes
    static constexpr int OFF_RING = 65536;
    static constexpr int QD = 16384;                     // 64 rows x 128 dims bf16: two boxes of 8 KB
    static constexpr int STAGES = 3;
    static constexpr int STAGE = 2 * QD + 1024;          // Q, dO, then lse2[64], dvec[64]
    static constexpr int OFF_PT = OFF_RING + STAGES * STAGE;  // P^T [128 keys][64 queries] bf16 (128 B rows)
    static constexpr int OFF_DST = OFF_PT + 16384;       // dS^T, same layout
    static constexpr int OFF_DQS = OFF_DST + 16384;      // 4 warps x 2 buffers x [16 queries][32 dims] fp32, swizzled
    static constexpr int SMEM = 1024 + OFF_DQS + 8 * 2048;
    static constexpr uint32_t T_S = 0, T_DP = 64, T_DQ = 128, T_DV = 256, T_DK = 384;  // dQ^T: 2 x 64 columns
    static constexpr uint32_t IDESC_SD = idesc_f16(128, 64, 1, 1, 0, 0);   // S^T, dP^T: K-major A and B
    static constexpr uint32_t IDESC_KV = idesc_f16(128, 128, 1, 1, 0, 1);  // dV, dK: A K-major, B MN-major
    static constexpr uint32_t IDESC_Q = idesc_f16(128, 64, 1, 1, 1, 1);    // dQ^T: A (K^T), B (dS^T) MN-major
};
static_assert(Bw2Cfg::SMEM <= 232448, "shared memory");
constexpr int Q64_THREADS = 512;
constexpr int Q64_DQ_WARP0 = 8;   // warps 8-11: dQ read-out
constexpr int Q64_MMA_WARP = 12;
constexpr int Q64_TMA_WARP = 13;
static_assert(Bw2Cfg::OFF_PT % 1024 == 0 && Bw2Cfg::OFF_DQS % 1024 == 0 && Bw2Cfg::STAGE % 1024 == 0, "align");

__global__ void __launch_bounds__(Q64_THREADS, 1)
    attn_bwd_q64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                        const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ BwdParams p) {
    using C = Bw2Cfg;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar_kv, bar_qdo_full[Bw2Cfg::STAGES], bar_qdo_empty[Bw2Cfg::STAGES],
        bar_s_full, bar_sdp_free, bar_ps_full, bar_ps_empty, bar_dq_full[2], bar_dq_free[2], bar_done;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int jt = p.causal ? blockIdx.y : blockIdx.x;   // key tile (128 keys); causal: costliest first
    const int zkv = p.causal ? blockIdx.x : blockIdx.y;  // b * H_kv + kv head
    const int b = zkv / p.H_kv, hk = zkv - b * p.H_kv;
    const int N = p.N;
    int kv_valid = N;
    if (p.kv_len) {
        kv_valid = __ldg(p.kv_len + b);
        kv_valid = kv_valid < 0 ? 0 : (kv_valid > N ? N : kv_valid);
    }
    const int k0 = jt * 128;
    const bool any_keys = k0 < kv_valid;
    const int n_q64 = (N + C::QT - 1) / C::QT;
    const int i_first = p.causal ? 2 * jt : 0;  // 64-row query tiles with at least one valid pair
    const int n_i = any_keys ? n_q64 - i_first : 0;
    const int n_steps = n_i * p.group;
    const uint64_t limit_ns = p.wait_limit_ns;

    if (warp == Q64_MMA_WARP) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(&bar_kv, 1);
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&bar_qdo_full[i], 1);
            mbar_init(&bar_qdo_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_dq_full[i], 1);
            mbar_init(&bar_dq_free[i], 128);
        }
        mbar_init(&bar_s_full, 1);
        mbar_init(&bar_sdp_free, 256);
        mbar_init(&bar_ps_full, 256);
        mbar_init(&bar_ps_empty, 1);
        mbar_init(&bar_done, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    auto step_head = [&](int s) { return hk * p.group + s / n_i; };
    auto step_tile = [&](int s) { return i_first + s % n_i; };
    // step s uses ring stage s % 3 for the (s / 3)-th time: that use's barrier phase parity is (s / 3) & 1
    auto stage_ptr = [&](int s) { return smem + C::OFF_RING + (s % C::STAGES) * C::STAGE; };

    if (warp == Q64_TMA_WARP) {
        // ================================ TMA producer (one lane) ================================
        if (elect_one() && n_steps > 0) {
            mbar_arrive_expect_tx(&bar_kv, 2 * 32768);
            for (int bx = 0; bx < 2; ++bx) {
                tma_load_3d(smem + C::OFF_K + bx * 16384, &tmK, &bar_kv, bx * 64, k0, zkv);
                tma_load_3d(smem + C::OFF_V + bx * 16384, &tmV, &bar_kv, bx * 64, k0, zkv);
            }
            int issued = 0;
            for (int s = 0; s < n_steps; ++s) {
                const int st = s % C::STAGES;
                if (s >= C::STAGES && !mbar_wait(&bar_qdo_empty[st], ((s / C::STAGES) - 1) & 1, limit_ns, &abort_flag)) {
                    bw_fail(&abort_flag, ERRBIT_WAIT_EMPTY);
                    break;
                }
                const int bh = b * p.H + step_head(s), it = step_tile(s);
                uint8_t* sp = stage_ptr(s);
                mbar_arrive_expect_tx(&bar_qdo_full[st], 2 * C::QD + 512);
                for (int bx = 0; bx < 2; ++bx) {
                    tma_load_3d(sp + bx * 8192, &tmQ, &bar_qdo_full[st], bx * 64, it * C::QT, bh);
                    tma_load_3d(sp + C::QD + bx * 8192, &tmDO, &bar_qdo_full[st], bx * 64, it * C::QT, bh);
                }
                const size_t srow = static_cast<size_t>(bh) * p.n_qt * 128 + static_cast<size_t>(it) * C::QT;
                bulk_load(sp + 2 * C::QD, p.lse2 + srow, 256, &bar_qdo_full[st]);
                bulk_load(sp + 2 * C::QD + 256, p.dvec + srow, 256, &bar_qdo_full[st]);
                issued = s + 1;
            }
            if (abort_flag) {  // wait (bounded) for the copies in flight before the CTA may exit
                volatile int never = 0;
                (void)mbar_wait(&bar_kv, 0, limit_ns, &never);
                for (int s = issued > C::STAGES ? issued - C::STAGES : 0; s < issued; ++s)
                    (void)mbar_wait(&bar_qdo_full[s % C::STAGES], (s / C::STAGES) & 1, limit_ns, &never);
            }
        }
        __syncwarp();
    } else if (warp == Q64_MMA_WARP) {
        // ======================================= MMA issuer =======================================
        auto wait_all = [&](uint64_t* bar, uint32_t parity, uint32_t bit) {
            const bool got = mbar_wait(bar, parity, limit_ns, &abort_flag);
            if (__all_sync(0xffffffffu, got)) return true;
            if (!got) bw_fail(&abort_flag, bit);
            return false;
        };
        const uint64_t dK_k = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);      // K as K-major A
        const uint64_t dV_k = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);      // V as K-major A
        const uint64_t dK_mn = sdesc_sw128(smem_u32(smem + C::OFF_K), 16384, 1024);  // K^T as M-major A
        const uint64_t dPT_k = sdesc_sw128(smem_u32(smem + C::OFF_PT), 16, 1024);    // P^T as K-major A
        const uint64_t dDST_k = sdesc_sw128(smem_u32(smem + C::OFF_DST), 16, 1024);  // dS^T as K-major A
        const uint64_t dDST_n = sdesc_sw128(smem_u32(smem + C::OFF_DST), 16384, 1024);  // dS^T as N-major B
        // K and V tiles: k-step kk of 16 dims (two 16 KB boxes of 64 dims); Q, dO tiles: 8 KB boxes
        auto kmaj_kv = [](int kk) { return static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); };
        auto kmaj_q = [](int kk) { return static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4); };
        auto rows16 = [](int kk) { return static_cast<uint64_t>((kk * 2048) >> 4); };  // 16 rows of 128 B
        auto col16 = [](int kk) { return static_cast<uint64_t>((kk * 32) >> 4); };      // 16 elements of a row
        bool ok = n_steps > 0 ? wait_all(&bar_kv, 0, ERRBIT_WAIT_KV) : true;
        for (int s = 0; s <= n_steps && ok; ++s) {
            if (s < n_steps) {
                // ---- S^T(s) = K Q^T, dP^T(s) = V dO^T ----
                if (!wait_all(&bar_qdo_full[s % C::STAGES], (s / C::STAGES) & 1, ERRBIT_WAIT_Q)) { ok = false; break; }
                if (s > 0 && !wait_all(&bar_sdp_free, (s - 1) & 1, ERRBIT_WAIT_P)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t sp = smem_u32(stage_ptr(s));
                    const uint64_t dQ_k = sdesc_sw128(sp, 16, 1024);
                    const uint64_t dDO_k = sdesc_sw128(sp + C::QD, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_ss(tmem + C::T_S, dK_k + kmaj_kv(kk), dQ_k + kmaj_q(kk), C::IDESC_SD, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_ss(tmem + C::T_DP, dV_k + kmaj_kv(kk), dDO_k + kmaj_q(kk), C::IDESC_SD, kk > 0);
                    umma_commit(&bar_s_full);
                }
                __syncwarp();
            }
            if (s >= 1) {
                // ---- second phase of step t = s - 1 ----
                const int t = s - 1;
                if (!wait_all(&bar_ps_full, t & 1, ERRBIT_WAIT_P)) { ok = false; break; }
                if (t >= 2 && !wait_all(&bar_dq_free[t & 1], ((t >> 1) - 1) & 1, ERRBIT_WAIT_O)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t sp = smem_u32(stage_ptr(t));
                    const uint64_t dQ_mn = sdesc_sw128(sp, 8192, 1024);            // Q as MN-major B (N = dims)
                    const uint64_t dDO_mn = sdesc_sw128(sp + C::QD, 8192, 1024);
#pragma unroll
                    for (int kk = 0; kk < C::QT / 16; ++kk)  // contraction over the 64 queries
                        umma_ss(tmem + C::T_DV, dPT_k + col16(kk), dDO_mn + rows16(kk), C::IDESC_KV, (t > 0 || kk > 0));
#pragma unroll
                    for (int kk = 0; kk < C::QT / 16; ++kk)
                        umma_ss(tmem + C::T_DK, dDST_k + col16(kk), dQ_mn + rows16(kk), C::IDESC_KV, (t > 0 || kk > 0));
                    umma_commit(&bar_qdo_empty[t % C::STAGES]);  // Q, dO of step t read: the stage may be refilled
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // dQ^T = K^T dS^T: contraction over the 128 keys
                        umma_ss(tmem + C::T_DQ + 64 * (t & 1), dK_mn + rows16(kk), dDST_n + rows16(kk), C::IDESC_Q, kk > 0);
                    umma_commit(&bar_dq_full[t & 1]);
                    umma_commit(&bar_ps_empty);
                }
                __syncwarp();
            }
        }
        if (elect_one()) umma_commit(&bar_done);  // every MMA issued above has completed
        __syncwarp();
        volatile int never = 0;
        const bool drained = mbar_wait(&bar_done, 0, limit_ns, &never);
        if (!__all_sync(0xffffffffu, drained) && lane == 0) bw_fail(&abort_flag, ERRBIT_WAIT_DRAIN);
    } else if (warp >= Q64_DQ_WARP0 && warp < Q64_DQ_WARP0 + 4) {
        // ===== warps 8-11: dQ of every step. This warp's TMEM lanes are dimensions 32 wq .. 32 wq + 31
        // (one per thread) of dQ^T; its 64 query columns leave as four [16 queries][32 dims] boxes,
        // staged 128-byte swizzled through two 2 KB buffers and added into the fp32 dQ by bulk tensor
        // reductions (rows past N are not written) =====
        const int wq = warp & 3;
        const uint32_t lane_off = tmem_lane_base(warp);
        const uint32_t stage = smem_u32(smem + C::OFF_DQS + (warp - Q64_DQ_WARP0) * 4096);
        const uint32_t colb = (lane & 3) * 4;
        for (int t = 0; t < n_steps; ++t) {
            const bool got = mbar_wait(&bar_dq_full[t & 1], (t >> 1) & 1, limit_ns, &abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (!got) bw_fail(&abort_flag, ERRBIT_WAIT_O);
                break;
            }
            tc_fence_after();
            uint32_t v0[32], v1[32];
            tmem_ld32(tmem + lane_off + C::T_DQ + 64 * (t & 1), v0);
            tmem_ld32(tmem + lane_off + C::T_DQ + 64 * (t & 1) + 32, v1);
            tmem_wait_ld(v0);
            tmem_wait_ld(v1);
            tc_fence_before();
            mbar_arrive(&bar_dq_free[t & 1]);  // the MMA warp may write this buffer's next dQ^T
            const int bh = b * p.H + step_head(t), it = step_tile(t);
#pragma unroll
            for (int hq = 0; hq < 4; ++hq) {  // queries 16 hq .. 16 hq + 15
                const uint32_t buf = stage + (hq & 1) * 2048;
                if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous box was read
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    st_shared_f32(buf + q * 128 + ((((lane >> 2) ^ (q & 7))) << 4) + colb,
                                  __uint_as_float(hq < 2 ? v0[16 * hq + q] : v1[16 * (hq - 2) + q]) * p.scale);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_reduce_add_3d(&tmDQ, smem + (buf - smem_u32(smem)), wq * 32, it * C::QT + 16 * hq, bh);
                    bulk_commit_group();
                }
                __syncwarp();
            }
        }
        if (lane == 0) bulk_wait_group_all();  // every reduction of this warp performed
        __syncwarp();
    } else if (warp < 8) {
        // ===== warps 0-7: one key row each, 32 queries (warps 0-3: queries 0-31, warps 4-7: 32-63) =====
        const int qh = warp >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;            // key row in the tile
        const int key = k0 + r;
        const uint32_t lane_off = tmem_lane_base(warp);
        const float sl = p.scale_log2;
        const uint32_t pt_row = smem_u32(smem + C::OFF_PT) + r * 128;
        const uint32_t dst_row = smem_u32(smem + C::OFF_DST) + r * 128;
        bool ok = true;
        for (int s = 0; s < n_steps && ok; ++s) {
            const int it = step_tile(s);
            const int q0 = it * C::QT + 32 * qh;
            const float* lse2 = reinterpret_cast<const float*>(stage_ptr(s) + 2 * C::QD) + 32 * qh;
            const float* dvec = lse2 + 64;
            bool got = mbar_wait(&bar_s_full, s & 1, limit_ns, &abort_flag);
            got = got && mbar_wait(&bar_qdo_full[s % C::STAGES], (s / C::STAGES) & 1, limit_ns, &abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (!got) bw_fail(&abort_flag, ERRBIT_WAIT_S);
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[32], dpv[32];
            tmem_ld32(tmem + lane_off + C::T_S + 32 * qh, sv);
            tmem_ld32(tmem + lane_off + C::T_DP + 32 * qh, dpv);
            tmem_wait_ld(sv);
            tmem_wait_ld(dpv);
            tc_fence_before();
            mbar_arrive(&bar_sdp_free);  // S^T, dP^T of this step are in registers: the next may land
            uint32_t pp[16], dd[16];
            // Every one of this thread's 32 (key, query) pairs valid (the key inside kv_len, the queries
            // below N and, causal, at or after the key): no per-pair mask, the row statistics read as
            // float4 and the arithmetic two-wide (the same single-rounded fma and product per pair).
            const bool all_valid = key < kv_valid && q0 + 31 < N && (!p.causal || key <= q0);
            if (all_valid) {
                bwd_pds_valid32(sv, dpv, lse2, dvec, sl, pp, dd);
            } else {
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float pv[2], dv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int q = q0 + i + u;
                        const bool valid = key < kv_valid && q < N && (!p.causal || key <= q);
                        const float e = valid ? ex2_approx(__uint_as_float(sv[i + u]) * sl - lse2[i + u]) : 0.f;
                        pv[u] = e;
                        dv[u] = e * (__uint_as_float(dpv[i + u]) - dvec[i + u]);
                    }
                    __nv_bfloat162 ph = __floats2bfloat162_rn(pv[0], pv[1]);
                    __nv_bfloat162 dh = __floats2bfloat162_rn(dv[0], dv[1]);
                    pp[i / 2] = *reinterpret_cast<uint32_t*>(&ph);
                    dd[i / 2] = *reinterpret_cast<uint32_t*>(&dh);
                }
            }
            // P^T, dS^T of the previous step must have been consumed by its products
            if (s > 0) {
                const bool e = mbar_wait(&bar_ps_empty, (s - 1) & 1, limit_ns, &abort_flag);
                if (!__all_sync(0xffffffffu, e)) {
                    if (!e) bw_fail(&abort_flag, ERRBIT_WAIT_EMPTY);
                    ok = false;
                    break;
                }
            }
            // 32 queries = four 16-byte chunks (4 qh .. 4 qh + 3) of this key's 128-byte row
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t off = ((4 * qh + k) ^ (r & 7)) << 4;
                st_shared_v4(pt_row + off, pp[4 * k], pp[4 * k + 1], pp[4 * k + 2], pp[4 * k + 3]);
                st_shared_v4(dst_row + off, dd[4 * k], dd[4 * k + 1], dd[4 * k + 2], dd[4 * k + 3]);
            }
            fence_proxy_async_smem();  // the MMAs read P^T and dS^T through the async proxy
            tc_fence_before();
            mbar_arrive(&bar_ps_full);
        }
        // ---- dK, dV of this key tile (warps 0-3): fp32 rows straight to device memory ----
        if (qh == 0 && ok && n_steps > 0) {
            const bool got = mbar_wait(&bar_done, 0, limit_ns, &abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (!got) bw_fail(&abort_flag, ERRBIT_WAIT_DRAIN);
                ok = false;
            }
            tc_fence_after();
        }
        // ok and n_steps are warp-uniform; key < N is not, so every lane takes part in the
        // warp-collective tensor-memory loads and only the stores are guarded.
        if (qh == 0 && ok) {
            const bool row_ok = key < N;
            const size_t orow = (static_cast<size_t>(zkv) * N + (row_ok ? key : 0)) * D;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                float* dst = (which ? p.dK : p.dV) + orow;
                const float mul = which ? p.scale : 1.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    if (n_steps > 0) {
                        tmem_ld32(tmem + lane_off + (which ? C::T_DK : C::T_DV) + c * 32, v);
                        tmem_wait_ld(v);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;
                    }
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(dst + c * 32 + i) =
                                make_float4(__uint_as_float(v[i]) * mul, __uint_as_float(v[i + 1]) * mul,
                                            __uint_as_float(v[i + 2]) * mul, __uint_as_float(v[i + 3]) * mul);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == Q64_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// D = rowsum(dO * O) and LSE in log2 units for every (padded) query row; dQ rows cleared.
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdPrepParams p) {
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);  // over bh * NQP
    const int lane = threadIdx.x & 31;
    if (row >= static_cast<long long>(p.rows) * p.NQP) return;
    const int bh = static_cast<int>(row / p.NQP), i = static_cast<int>(row % p.NQP);
    float dsum = 0.f;
    float l2 = INFINITY;  // padding rows: P = exp2(x - inf) = 0
    if (i < p.N) {
        const size_t base = (static_cast<size_t>(bh) * p.N + i) * p.d;
        const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(p.dO) + base;
        for (int c = lane; c < p.d; c += 32) {
            dsum = fmaf(__bfloat162float(dO[c]), p.O[base + c], dsum);
            p.dQ[base + c] = 0.f;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
        const float lse = p.LSE[static_cast<size_t>(bh) * p.N + i];
        l2 = lse * 1.4426950408889634f;
    }
    if (lane == 0) {
        p.lse2[row] = l2;
        p.dvec[row] = dsum;
    }
}

template <int D>
static cudaError_t launch_bwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const CUtensorMap& tmDO, const CUtensorMap& tmDQ, const BwdParams& p,
                                cudaStream_t stream) {
    auto kern = attn_bwd_tc_kernel<D>;
    static std::atomic<int> ready[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || ready[dev].load(std::memory_order_acquire) == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwCfg<D>::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) ready[dev].store(1, std::memory_order_release);
    }
    const dim3 grid = p.causal ? dim3(static_cast<unsigned>(p.B * p.H_kv), static_cast<unsigned>(p.n_qt))
                               : dim3(static_cast<unsigned>(p.n_qt), static_cast<unsigned>(p.B * p.H_kv));
    attn_bwd_tc_kernel<D><<<grid, BW_THREADS, BwCfg<D>::SMEM, stream>>>(tmQ, tmK, tmV, tmDO, tmDQ, p);
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd(int d, const BwdPrepParams& prep, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmDO, const CUtensorMap& tmDQ,
                            const BwdParams& p, cudaStream_t stream) {
    const long long rows = static_cast<long long>(prep.rows) * prep.NQP;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL || p.B * p.H_kv > 65535 || p.n_qt > 65535) return cudaErrorInvalidConfiguration;
    attn_bwd_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(prep);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (d == 128) {  // 64-row query tiles through a two-stage ring
        static std::atomic<int> ready[64];
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || ready[dev].load(std::memory_order_acquire) == 0) {
            e = cudaFuncSetAttribute(attn_bwd_q64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Bw2Cfg::SMEM);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) ready[dev].store(1, std::memory_order_release);
        }
        const dim3 grid = p.causal ? dim3(static_cast<unsigned>(p.B * p.H_kv), static_cast<unsigned>(p.n_qt))
                                   : dim3(static_cast<unsigned>(p.n_qt), static_cast<unsigned>(p.B * p.H_kv));
        attn_bwd_q64_kernel<<<grid, Q64_THREADS, Bw2Cfg::SMEM, stream>>>(tmQ, tmK, tmV, tmDO, tmDQ, p);
        return cudaGetLastError();
    }
    if (d == 64) return launch_bwd_t<64>(tmQ, tmK, tmV, tmDO, tmDQ, p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_bwd_error(uint32_t* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_bwd_error, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_attn_bwd_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace attn_impl
