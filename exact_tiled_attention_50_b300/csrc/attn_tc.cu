// Tensor-core attention forward for bf16 inputs on sm_103a (B300).
//
// Method: exact attention O = softmax(scale Q K^T) V, evaluated tile by tile with the online
// softmax: running row maximum m, running sum l, rescaling of the unnormalised accumulator by
// exp(m_old - m_new), one final division O / l, and the row log-sum-exp. Sources: the
// safe_softmax_block and flash_attention_blockwise listings of "AI训练的最大障碍不是算力,而是'内存墙'"
// (zsdodo.com); section 4.1.3 "算法流程详解" of "第四章 注意力机制实战案例" (aiknowledge.cn), whose
// accumulator form (rescale, add P V, divide once at the end) is used, with the maximum taken per row
// over the key axis; formulas 1-2 of "闪电注意力的数学原理" on "闪电注意力：革命性地提高Transformer效率"
// (unite.ai). Q-tile-outer / key-tile-inner order as in those listings, so that one CTA owns a row's
// state for its whole lifetime.
//
// Blackwell mapping (one CTA per SM, 320 threads):
//   warps 0-3  softmax warpgroup for query tile 0 (rows 0-127 of the CTA's 256 rows)
//   warps 4-7  softmax warpgroup for query tile 1 (rows 128-255)
//   warp  8    tensor-memory owner and MMA issuer (one thread issues every tcgen05.mma)
//   warp  9    TMA producer (Q tiles once, then a ring of K / V tiles)
// Tensor memory (512 columns x 128 lanes x 32 bit): S_0 [0,128), S_1 [128,256), O_0 and O_1 after
// that (d columns each). P_t (fp16, two per column) overwrites the first 64 columns of S_t after the
// softmax has read S_t into registers; the P V MMA reads P straight from tensor memory.
// The MMA thread issues, per key tile j:  PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so that while one
// warpgroup computes exponentials the tensor core works on the other tile (ping-pong).
// The lazy rescale keeps a row's reference maximum until the tile maximum exceeds it by more than
// 2^8 (log2 domain); exponentials are then at most 256 and the final O / l is unchanged, since O and
// l use the same reference. V enters the P V product as fp16 (a per-head power-of-two scale keeps
// it in range); Q K^T is bf16 x bf16 with fp32 accumulation.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn_impl {

using namespace attn_sm103;

__device__ unsigned int g_attn_error = 0;

namespace {

constexpr int BLOCK_M = 128;              // query rows per tile (tcgen05 M)
constexpr int BLOCK_N = 128;              // keys per tile
constexpr int NUM_THREADS = 320;
constexpr int MMA_WARP = 8;
constexpr int TMA_WARP = 9;
constexpr float RESCALE_THRESHOLD = 8.0f; // log2 units
constexpr uint32_t TMEM_COLS = 512;

template <int D>
struct Cfg {
    static constexpr int NB = D / 64;                 // 64-element (128-byte) boxes per row
    static constexpr int TILE_BYTES = NB * 16384;     // one 128 x D tile of 16-bit values
    static constexpr int NS = (D == 128) ? 4 : 8;     // K/V ring stages
    static constexpr int SMEM_BYTES = 1024 + 2 * TILE_BYTES + NS * TILE_BYTES;
    static constexpr uint32_t IDESC_S = idesc_f16(BLOCK_M, BLOCK_N, 1, 1, 0, 0);  // bf16, K-major both
    static constexpr uint32_t IDESC_O = idesc_f16(BLOCK_M, D, 0, 0, 0, 1);        // f16, B (V) MN-major
    static constexpr uint32_t TMEM_O = 256;
};

__device__ __forceinline__ void record_failure(volatile int* abort_flag, uint32_t bits) {
    *abort_flag = 1;
    atomicOr(&g_attn_error, ERRBIT_TIMEOUT | bits);
}

__device__ __forceinline__ int clamp_len(const int32_t* kv_len, int b, int N) {
    if (!kv_len) return N;
    int L = __ldg(kv_len + b);
    return L < 0 ? 0 : (L > N ? N : L);
}

}  // namespace

template <int D, bool OUT_BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const TcParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ0 = smem;
    uint8_t* sKV = smem + 2 * C::TILE_BYTES;

    __shared__ __align__(8) uint64_t bar_q;
    __shared__ __align__(8) uint64_t bar_kv_full[C::NS];
    __shared__ __align__(8) uint64_t bar_kv_empty[C::NS];
    __shared__ __align__(8) uint64_t bar_s_full[2];
    __shared__ __align__(8) uint64_t bar_p_full[2];
    __shared__ __align__(8) uint64_t bar_o_full[2];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work unit: (b, h, pair of 128-row query tiles); causal: heaviest pairs launch first ----
    const int BH = p.B * p.H;
    const int bh = blockIdx.x % BH;
    const int pair = p.n_pairs - 1 - static_cast<int>(blockIdx.x / BH);
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int zkv = b * p.H_kv + h / p.group;
    const int kv_valid = clamp_len(p.kv_len, b, p.N);
    int q0[2], nkv[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        q0[t] = (2 * pair + t) * BLOCK_M;
        const bool exists = q0[t] < p.N;
        const int limit = p.causal ? min(kv_valid, q0[t] + BLOCK_M) : kv_valid;
        nkv[t] = exists ? (limit + BLOCK_N - 1) / BLOCK_N : 0;
    }
    const int nmax = max(nkv[0], nkv[1]);

    // ---- setup ----
    if (warp == MMA_WARP) {
        tmem_alloc(&tmem_base_sh, TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == TMA_WARP * 32) {
        mbar_init(&bar_q, 1);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(&bar_kv_full[s], 1);
            mbar_init(&bar_kv_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar_s_full[t], 1);
            mbar_init(&bar_p_full[t], 128);
            mbar_init(&bar_o_full[t], 1);
        }
        mbar_init(&bar_drain, 1);
        abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const uint64_t limit_ns = p.wait_limit_ns;

    if (warp == TMA_WARP) {
        // ================================ TMA producer ================================
        if (lane == 0 && nmax > 0) {
            const uint64_t pol_kv = l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_first();
            uint32_t qbytes = 0;
            for (int t = 0; t < 2; ++t) qbytes += nkv[t] > 0 ? C::TILE_BYTES : 0;
            mbar_arrive_expect_tx(&bar_q, qbytes);
            for (int t = 0; t < 2; ++t)
                if (nkv[t] > 0)
                    for (int bx = 0; bx < C::NB; ++bx)
                        tma_load_3d_hint(sQ0 + t * C::TILE_BYTES + bx * 16384, &tmQ, &bar_q, bx * 64, q0[t], bh,
                                         pol_q);
            int it_done = 0;
            bool ok = true;
            for (int it = 0; it < 2 * nmax; ++it) {
                const int stage = it % C::NS;
                if (it >= C::NS) {
                    if (!mbar_wait(&bar_kv_empty[stage], ((it / C::NS) - 1) & 1, limit_ns, &abort_flag)) {
                        record_failure(&abort_flag, ERRBIT_WAIT_EMPTY);
                        ok = false;
                        break;
                    }
                }
                const int j = it >> 1;
                const bool is_v = it & 1;
                if (!is_v && j == 0 && p.debug_skip_kv_load) {
                    it_done = it + 1;
                    continue;  // failure-path test: this tile is never loaded
                }
                mbar_arrive_expect_tx(&bar_kv_full[stage], C::TILE_BYTES);
                uint8_t* dst = sKV + stage * C::TILE_BYTES;
                for (int bx = 0; bx < C::NB; ++bx)
                    tma_load_3d_hint(dst + bx * 16384, is_v ? &tmV : &tmK, &bar_kv_full[stage], bx * 64,
                                     j * BLOCK_N, zkv, pol_kv);
                it_done = it + 1;
            }
            // On failure, wait (bounded) for the copies this thread issued and nobody consumed, so
            // that no TMA write lands in shared memory after the CTA has exited.
            if (!ok || abort_flag) {
                volatile int never = 0;  // these waits must not be cut short by the abort flag
                (void)mbar_wait(&bar_q, 0, limit_ns, &never);
                const int first = it_done > C::NS ? it_done - C::NS : 0;
                for (int it = first; it < it_done; ++it) {
                    if (it == 0 && p.debug_skip_kv_load) continue;
                    (void)mbar_wait(&bar_kv_full[it % C::NS], (it / C::NS) & 1, limit_ns, &never);
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ================================ MMA issuer ================================
        if (lane == 0 && nmax > 0) {
            bool ok = mbar_wait(&bar_q, 0, limit_ns, &abort_flag);
            if (!ok) record_failure(&abort_flag, ERRBIT_WAIT_Q);
            const uint32_t sQa = smem_u32(sQ0);
            const uint32_t sKVa = smem_u32(sKV);
            auto issue_S = [&](int t, int stage) {
                const uint32_t qa = sQa + t * C::TILE_BYTES;
                const uint32_t ka = sKVa + stage * C::TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    umma_ss(tmem + t * BLOCK_N, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                            C::IDESC_S, kk > 0);
                }
            };
            auto issue_PV = [&](int t, int stage, bool accumulate) {
                const uint32_t va = sKVa + stage * C::TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < BLOCK_N / 16; ++kk)
                    umma_ts(tmem + C::TMEM_O + t * D, tmem + t * BLOCK_N + kk * 8,
                            sdesc_sw128(va + kk * 2048, 16384, 1024), C::IDESC_O, (accumulate || kk > 0));
            };
            if (ok) {
                tc_fence_after();
                // prologue: S_t(0) for both tiles from K_0 (ring position 0)
                ok = mbar_wait(&bar_kv_full[0], 0, limit_ns, &abort_flag);
                if (!ok) record_failure(&abort_flag, ERRBIT_WAIT_KV);
            }
            if (ok) {
                tc_fence_after();
                for (int t = 0; t < 2; ++t)
                    if (nkv[t] > 0) {
                        issue_S(t, 0);
                        umma_commit(&bar_s_full[t]);
                    }
                umma_commit(&bar_kv_empty[0]);
                for (int j = 0; j < nmax && ok; ++j) {
                    const int itV = 2 * j + 1, itK = 2 * j + 2;
                    const int sV = itV % C::NS, sK = itK % C::NS;
                    const bool has_next = j + 1 < nmax;
                    if (!mbar_wait(&bar_kv_full[sV], (itV / C::NS) & 1, limit_ns, &abort_flag)) {
                        record_failure(&abort_flag, ERRBIT_WAIT_KV);
                        ok = false;
                        break;
                    }
                    if (has_next && !mbar_wait(&bar_kv_full[sK], (itK / C::NS) & 1, limit_ns, &abort_flag)) {
                        record_failure(&abort_flag, ERRBIT_WAIT_KV);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int t = 0; t < 2; ++t) {
                        if (j >= nkv[t]) continue;
                        if (!mbar_wait(&bar_p_full[t], j & 1, limit_ns, &abort_flag)) {
                            record_failure(&abort_flag, ERRBIT_WAIT_P);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_PV(t, sV, j > 0);
                        if (j + 1 < nkv[t]) {
                            issue_S(t, sK);
                            umma_commit(&bar_s_full[t]);
                        } else {
                            umma_commit(&bar_o_full[t]);
                        }
                    }
                    if (!ok) break;
                    umma_commit(&bar_kv_empty[sV]);
                    if (has_next) umma_commit(&bar_kv_empty[sK]);
                }
            }
            // Drain: every MMA this thread issued has completed before tensor memory is freed.
            umma_commit(&bar_drain);
            volatile int never = 0;  // not cut short by the abort flag: the drain must finish
            if (!mbar_wait(&bar_drain, 0, limit_ns, &never)) record_failure(&abort_flag, ERRBIT_WAIT_DRAIN);
        }
        __syncwarp();
    } else {
        // ============================ softmax warpgroups ============================
        const int t = warp >> 2;            // query tile of this warpgroup
        const int wq = warp & 3;            // TMEM lane quarter
        const int r = wq * 32 + lane;       // row within the tile
        const int row = q0[t] + r;          // query index
        const uint32_t lane_off = tmem_lane_base(wq);
        const uint32_t tS = tmem + lane_off + t * BLOCK_N;
        const uint32_t tO = tmem + lane_off + C::TMEM_O + t * D;
        const float sl = p.scale_log2;
        float m_run = -INFINITY;            // reference maximum (log2 domain, already scaled)
        float l_run = 0.f;                  // running sum of exp2(s*sl - m_run)
        bool ok = true;
        const int row_lim = p.causal ? min(kv_valid, row + 1) : kv_valid;  // keys < row_lim are valid

        for (int j = 0; j < nkv[t]; ++j) {
            // tcgen05.ld/st below are warp-collective: the warp proceeds only if every lane's wait
            // succeeded
            const bool got = mbar_wait(&bar_s_full[t], j & 1, limit_ns, &abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (!got) record_failure(&abort_flag, ERRBIT_WAIT_S);
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t ra[32], rb[32], rc[32], rd[32];
            tmem_ld32(tS + 0, ra);
            tmem_ld32(tS + 32, rb);
            tmem_ld32(tS + 64, rc);
            tmem_ld32(tS + 96, rd);
            tmem_wait_ld(ra);
            tmem_wait_ld(rb);
            tmem_wait_ld(rc);
            tmem_wait_ld(rd);
            float x[128];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                x[i] = __uint_as_float(ra[i]);
                x[32 + i] = __uint_as_float(rb[i]);
                x[64 + i] = __uint_as_float(rc[i]);
                x[96 + i] = __uint_as_float(rd[i]);
            }
            const int k0 = j * BLOCK_N;
            if (k0 + BLOCK_N > kv_valid || (p.causal && k0 + BLOCK_N - 1 > q0[t])) {
                const int lim = row_lim - k0;
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i >= lim) x[i] = -INFINITY;
            }
            float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
            for (int i = 4; i < 128; i += 4) {
                mx0 = fmaxf(mx0, x[i]);
                mx1 = fmaxf(mx1, x[i + 1]);
                mx2 = fmaxf(mx2, x[i + 2]);
                mx3 = fmaxf(mx3, x[i + 3]);
            }
            const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl;
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_run = m_tile;
            } else if (m_tile > m_run + RESCALE_THRESHOLD) {
                alpha = ex2_approx(m_run - m_tile);
                l_run *= alpha;
                m_run = m_tile;
                rescale = true;
            }
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tO + c * 32, o);
                }
            }
            const float m_sub = (m_run == -INFINITY) ? 0.f : m_run;
            uint32_t pk0[32], pk1[32];
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float a0 = ex2_approx(fmaf(x[2 * i], sl, -m_sub));
                const float a1 = ex2_approx(fmaf(x[2 * i + 1], sl, -m_sub));
                const float b0 = ex2_approx(fmaf(x[64 + 2 * i], sl, -m_sub));
                const float b1 = ex2_approx(fmaf(x[64 + 2 * i + 1], sl, -m_sub));
                ls0 += a0 + a1;
                ls1 += b0 + b1;
                pk0[i] = pack_f16x2(a0, a1);
                pk1[i] = pack_f16x2(b0, b1);
            }
            l_run += ls0 + ls1;
            tmem_st32(tS + 0, pk0);
            tmem_st32(tS + 32, pk1);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar_p_full[t]);
        }

        // ---- epilogue: O / l (times the fp16 scale of V), LSE ----
        if (ok && nkv[t] > 0) {
            const bool got = mbar_wait(&bar_o_full[t], 0, limit_ns, &abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (!got) record_failure(&abort_flag, ERRBIT_WAIT_O);
                ok = false;
            }
            tc_fence_after();
        }
        if (q0[t] < p.N) {
            const bool have = ok && nkv[t] > 0;
            const float vscale = have ? ldexpf(1.0f, __ldg(p.v_exp + zkv)) : 0.f;
            const float inv = (have && l_run > 0.f) ? vscale / l_run : 0.f;
            const bool store = row < p.N;
            const size_t obase = (static_cast<size_t>(bh) * p.N + (store ? row : 0)) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (have) {
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld(o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if (store) {
                    if constexpr (OUT_BF16) {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.O) + obase + c * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                __nv_bfloat162 hv = __floats2bfloat162_rn(__uint_as_float(o[v4 * 8 + 2 * e]) * inv,
                                                                          __uint_as_float(o[v4 * 8 + 2 * e + 1]) * inv);
                                w[e] = *reinterpret_cast<uint32_t*>(&hv);
                            }
                            dst[v4] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.O) + obase + c * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4)
                            dst[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                                                  __uint_as_float(o[4 * v4 + 2]) * inv,
                                                  __uint_as_float(o[4 * v4 + 3]) * inv);
                    }
                }
            }
            if (store && p.LSE) {
                const float lse = (have && l_run > 0.f) ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
                p.LSE[static_cast<size_t>(bh) * p.N + row] = lse;
            }
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------------
// V -> fp16 with a per-head power-of-two scale: pass 1 takes |V| maxima per chunk, pass 2 picks
// the head's exponent e (so that |V| * 2^-e < 2^15) and writes V * 2^-e rounded to fp16.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) vprep_absmax_kernel(const VPrepParams p) {
    const int chunk = blockIdx.x, head = blockIdx.y;
    const long long base = static_cast<long long>(head) * p.elems_per_head + static_cast<long long>(chunk) * VPREP_CHUNK;
    const long long end = min(base + VPREP_CHUNK, static_cast<long long>(head + 1) * p.elems_per_head);
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.V) + base);
    const int nvec = static_cast<int>((end - base) / 8);  // N*d is a multiple of 64
    float m = 0.f;
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
        uint4 u = __ldg(src + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // bf16 -> fp32 is a 16-bit shift; |x| clears the sign bit
            m = fmaxf(m, __uint_as_float((w[e] << 16) & 0x7fffffffu));
            m = fmaxf(m, __uint_as_float(w[e] & 0x7fff0000u));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float r = red[0];
        for (int i = 1; i < 8; ++i) r = fmaxf(r, red[i]);
        p.partial_max[head * p.chunks + chunk] = r;
    }
}

__global__ void __launch_bounds__(256) vprep_convert_kernel(const VPrepParams p) {
    const int chunk = blockIdx.x, head = blockIdx.y;
    __shared__ int e_sh;
    if (threadIdx.x < 32) {
        float m = 0.f;
        for (int i = threadIdx.x; i < p.chunks; i += 32) m = fmaxf(m, p.partial_max[head * p.chunks + i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) {
            int E = 0;
            // |V| < 2^E; NaN/Inf inputs keep e = 0 and propagate through the result
            if (isfinite(m) && m > 0.f) (void)frexpf(m, &E);
            const int e = E > 15 ? E - 15 : 0;
            e_sh = e;
            if (chunk == 0) p.v_exp[head] = e;
        }
    }
    __syncthreads();
    const float s = ldexpf(1.0f, -e_sh);
    const long long base = static_cast<long long>(head) * p.elems_per_head + static_cast<long long>(chunk) * VPREP_CHUNK;
    const long long end = min(base + VPREP_CHUNK, static_cast<long long>(head + 1) * p.elems_per_head);
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.V) + base);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(p.V16) + base);
    const int nvec = static_cast<int>((end - base) / 8);
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
        uint4 u = __ldg(src + i);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(w[e] << 16) * s;
            const float hi = __uint_as_float(w[e] & 0xffff0000u) * s;
            w[e] = pack_f16x2(lo, hi);
        }
        dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_vprep(const VPrepParams& p, cudaStream_t stream) {
    dim3 grid(p.chunks, p.heads);
    vprep_absmax_kernel<<<grid, 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    vprep_convert_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D, bool OUT_BF16>
static cudaError_t launch_tc_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const TcParams& p, cudaStream_t stream) {
    auto kern = attn_fwd_tc_kernel<D, OUT_BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long grid = static_cast<long long>(p.n_pairs) * p.B * p.H;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(grid), NUM_THREADS, Cfg<D>::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

cudaError_t launch_attn_tc(int d, bool out_bf16, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV16, const TcParams& p, cudaStream_t stream) {
    if (d == 128) return out_bf16 ? launch_tc_t<128, true>(tmQ, tmK, tmV16, p, stream)
                                  : launch_tc_t<128, false>(tmQ, tmK, tmV16, p, stream);
    if (d == 64) return out_bf16 ? launch_tc_t<64, true>(tmQ, tmK, tmV16, p, stream)
                                 : launch_tc_t<64, false>(tmQ, tmK, tmV16, p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_error(uint32_t* out, cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int v = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&v, g_attn_error, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_attn_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace attn_impl
