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
// Blackwell mapping (one CTA per SM, 384 threads = 3 warpgroups):
//   warps 0-3  softmax warpgroup for query tile 0 (rows 0-127 of the CTA's 256 rows)
//   warps 4-7  softmax warpgroup for query tile 1 (rows 128-255)
//   warp  8    tensor-memory owner and MMA issuer (converged warp; one elected lane issues)
//   warp  9    TMA producer of the key/value tiles (K_k0 per segment, then a ring of (V_j, K_j+1))
//   warp 10    TMA producer of the query tiles Q_0, Q_1 (once per segment)
//   warp 11    idle (it completes the third warpgroup for the register split)
// Tensor memory (512 columns x 128 lanes x 32 bit): S_0 [0,128), S_1 [128,256), O_0 and O_1 after
// that (d columns each). P_t (fp16, two per column) overwrites the first 64 columns of S_t after the
// softmax has read S_t into registers; the P V MMA reads P straight from tensor memory.
// The MMA warp issues, per key tile j:  PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so that while one
// warpgroup computes exponentials the tensor core works on the other tile (ping-pong). S_t(j+1)
// overwrites the columns PV_t(j) reads P from; it is issued after PV_t(j) by the same thread and
// relies on the tensor pipe executing MMAs in issue order.
// The lazy rescale keeps a row's reference maximum until the tile maximum exceeds it by more than
// 2^15 (log2 domain); exponentials are then at most 2^15 (fp16 holds them) and the final O / l is
// unchanged, since O and l use the same reference. P is handed to the MMA warp in two halves (keys
// 0-63, 64-127) so that the first four P V k-steps overlap the second half's exponentials.
// V enters the P V product as fp16 (a per-head power-of-two scale keeps it in range); Q K^T is
// bf16 x bf16 with fp32 accumulation.
//
// fp8 variant (FP8 = true, d = 128; section "闪电注意力-3" of the unite.ai page: FP8 computation with
// a processing step that lowers the quantisation error): a pre-pass rotates Q and K by the same
// random-sign Hadamard matrix (Q K^T unchanged) and rounds Q, K and V to E4M3 with one power-of-two
// scale per 128-row tile; V is stored transposed (keys innermost) so that both products read K-major
// operands. Both products run as kind::f8f6f4 (E4M3 x E4M3, fp32 accumulation); the softmax folds
// the tiles' scales into its per-tile multiplier and writes P as E4M3 (four per TMEM column). The
// lazy-rescale threshold drops to 2^8 so that P stays below the E4M3 maximum 448.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn_impl {

using namespace attn_sm103;

__device__ unsigned int g_attn_error = 0;

namespace {

constexpr int BLOCK_M = 128;              // query rows per tile (tcgen05 M)
constexpr int BLOCK_N = 128;              // keys per tile
constexpr int NUM_THREADS = 384;          // 3 warpgroups
constexpr int MMA_WARP = 8;
constexpr int TMA_WARP = 9;                // key/value ring producer
constexpr int QLOAD_WARP = 10;             // query tile producer
constexpr uint32_t TMEM_COLS = 512;
// Register split: the block launches with 384 x 168 = 64512 registers; the two softmax
// warpgroups raise theirs to 200 and the MMA/TMA warpgroup lowers its to 104:
// 2*128*200 + 128*104 = 64512 (every sub-partition holds two softmax warps and one other warp:
// 2*200 + 104 = 504 <= 512 registers per lane).
constexpr int LAUNCH_REGS = 168;
constexpr uint32_t SOFTMAX_REGS = 200;
constexpr uint32_t CONTROL_REGS = 104;
static_assert(2 * 128 * SOFTMAX_REGS + 128 * CONTROL_REGS <= NUM_THREADS * LAUNCH_REGS, "register split");

template <int D, bool FP8>
struct Cfg {
    static_assert(!FP8 || D == 128, "the fp8 path has d = 128 (one 128-byte row per tile row)");
    static constexpr int BOX_ELEMS = FP8 ? 128 : 64;  // elements per 128-byte box row
    static constexpr int NB = D / BOX_ELEMS;          // boxes per tile row
    static constexpr int TILE_BYTES = NB * 16384;     // one 128 x D tile (fp8: also the 128 x 128 V^T tile)
    // Shared memory: Q_0, Q_1, then NP ring stages of (V_j, K_j+1), consumed together (one wait and one
    // release per key step; a segment's first stage holds only its first key tile K_k0), then the
    // epilogue's staging boxes (EPI_BUFS of 4 KB per softmax warp). With staging of its own the
    // epilogue leaves Q free, so the next segment's Q loads as soon as this segment's MMAs are done.
    static constexpr int NP = (D == 128 && !FP8) ? 2 : 4;
    // S = Q K^T k-steps: 16 bf16 or 32 E4M3 elements, 32 bytes of each row either way
    static constexpr int KSTEPS = FP8 ? D / 32 : D / 16;
    // Lazy rescale: a row keeps its reference maximum until a tile's maximum exceeds it by more than
    // this (log2 units); exponentials then stay <= 2^15, inside the fp16 range of P (65504), or
    // <= 2^8, inside the E4M3 range (448).
    static constexpr float RESCALE_THRESHOLD = FP8 ? 8.0f : 15.0f;
    static constexpr int OFF_RING = 2 * TILE_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // V slot then K slot
    static constexpr int OFF_EPI = OFF_RING + NP * STAGE_BYTES;
    // two staging boxes per warp where they fit in the 227 KB a CTA may use, else one
    static constexpr int EPI_BUFS = 1024 + OFF_EPI + 8 * 2 * 4096 <= 232448 ? 2 : 1;
    static constexpr int SMEM_BYTES = 1024 + OFF_EPI + 8 * EPI_BUFS * 4096;
    // bf16 S: K-major both; f16 P V: B (V) MN-major. fp8: E4M3 everywhere, every operand K-major
    // (V^T tile: d rows of 128 keys).
    static constexpr uint32_t IDESC_S = FP8 ? idesc_f8f6f4(BLOCK_M, BLOCK_N, 0, 0, 0, 0)
                                            : idesc_f16(BLOCK_M, BLOCK_N, 1, 1, 0, 0);
    static constexpr uint32_t IDESC_O = FP8 ? idesc_f8f6f4(BLOCK_M, D, 0, 0, 0, 0) : idesc_f16(BLOCK_M, D, 0, 0, 0, 1);
    static constexpr uint32_t TMEM_O = 256;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ void record_failure(volatile int* abort_flag, uint32_t bits) {
    *abort_flag = 1;
    atomicOr(&g_attn_error, ERRBIT_TIMEOUT | bits);
}

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2,
// 3", SC 2011): per round the 64-bit products M0 * x0 and M1 * x2 are split into halves and
// x <- (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0), the key of round r being (k0 + r W0, k1 + r W1).
// The round keys are the same for every draw of a launch and come precomputed (rk[0][r], rk[1][r]).
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, const uint32_t (&rk)[2][10]) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * x.x;
        const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * x.z;
        x = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ x.y ^ rk[0][r], static_cast<uint32_t>(p1),
                       static_cast<uint32_t>(p0 >> 32) ^ x.w ^ rk[1][r], static_cast<uint32_t>(p0));
    }
    return x;
}

// 2^k as fp32 for the exponents the merge and epilogue use (k <= 127; 0 below 2^-126, where the
// weighted contribution is negligible)
__device__ __forceinline__ float pow2i(int k) { return k < -126 ? 0.f : __int_as_float((k + 127) << 23); }

__device__ __forceinline__ int clamp_len(const int32_t* kv_len, int b, int N) {
    if (!kv_len) return N;
    int L = __ldg(kv_len + b);
    return L < 0 ? 0 : (L > N ? N : L);
}

}  // namespace

// Schedule table on the device: kv_len from the caller, batch offsets from the plan pass; reads the
// kernel's grid-constant parameter in place. Without kv_len every batch costs the same, and the
// offsets are computed here instead of read (no dependent global loads before the first tile).
struct DevSchedTab {
    const TcParams& p;
    __device__ int nb(int b) const { return key_tiles(clamp_len(p.kv_len, b, p.plan.N)); }
    __device__ long long boff(int b) const {
        if (p.kv_len == nullptr)
            return static_cast<long long>(b) * p.plan.H *
                   line_prefix(p.plan.n_pairs, key_tiles(p.plan.N), p.plan.N, p.plan.causal);
        return p.boff[b];
    }
};

// Per-segment quantities every role derives the same way.
struct SegInfo {
    int bh, zkv;
    int q0[2];       // first query row of each tile
    int n[2];        // key steps of each tile inside this piece
    int nmax;
    int kv_valid;
};

__device__ __forceinline__ SegInfo seg_info(const TcParams& p, const Segment& s) {
    SegInfo si;
    const int N = p.plan.N;
    si.kv_valid = clamp_len(p.kv_len, s.b, N);
    si.bh = s.b * p.plan.H + s.h;
    si.zkv = s.b * p.H_kv + s.h / p.group;
    si.nmax = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int q0 = s.pair * 2 * BLOCK_M + t * BLOCK_M;
        si.q0[t] = q0;
        const int lim = p.plan.causal ? min(si.kv_valid, q0 + BLOCK_M) : si.kv_valid;
        const int nkv = q0 < N ? key_tiles(lim) : 0;
        const int hi = min(s.k1, nkv);
        si.n[t] = hi > s.k0 ? hi - s.k0 : 0;
        si.nmax = max(si.nmax, si.n[t]);
    }
    return si;
}

// VAR: 0 = bf16 inputs, 1 = fp8 (E4M3) path, 2 = bf16 inputs with additive bias and dropout
template <int D, bool OUT_BF16, int VAR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                       const __grid_constant__ TcParams p) {
    constexpr bool FP8 = VAR == 1;
    constexpr bool EXTRA = VAR == 2;
    using C = Cfg<D, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    __shared__ __align__(8) uint64_t bar_q;                 // the segment's Q_0, Q_1 landed
    __shared__ __align__(8) uint64_t bar_q_empty;           // every MMA of the segment completed
    __shared__ __align__(8) uint64_t bar_full[C::NP];       // ring stage (V_j, K_j+1) landed
    __shared__ __align__(8) uint64_t bar_empty[C::NP];      // ring stage free again
    __shared__ __align__(8) uint64_t bar_s_full[2];         // S_t in TMEM
    __shared__ __align__(8) uint64_t bar_p_full[2][2];      // half h of P_t in TMEM (O_t rescaled)
    __shared__ __align__(8) uint64_t bar_o_full[2];         // last P V of the segment into O_t done
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;
    // Work-schedule walkers, one per working warp (warps 0-10), advanced by one lane; the current
    // segment is read from shared memory so that the walker state stays out of registers.
    __shared__ WalkState walk_sh[11];
    __shared__ Segment seg_sh[11];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const DevSchedTab tab{p};
    // The kernel may start while the pre-pass that precedes it on the stream still runs (programmatic
    // dependent launch). What the pre-pass writes: the fp16 V copy and its tile exponents, the batch
    // offsets and cleared flags of the schedule, and (fp8) every operand. With kv_len or fp8 the whole
    // CTA waits for it here; otherwise only the roles that read its output wait (the K/V producer
    // before its first V tile, the softmax warpgroups before their first tile exponent), so that the
    // set-up, the schedule walk and the Q and first K loads overlap the pre-pass.
    const bool dep_early = FP8 || p.kv_len != nullptr;
    if (dep_early) grid_dep_wait();
    if (warp < 11 && lane == 0) walk_init(walk_sh[warp], tab, p.plan);
    // warp-collective: the next segment of this warp's walker into seg_sh[warp]
    auto next_seg = [&]() -> bool {
        int more = 0;
        if (lane == 0) more = walk_next(walk_sh[warp], tab, p.plan, static_cast<int>(blockIdx.x), seg_sh[warp]);
        more = __shfl_sync(0xffffffffu, more, 0);
        __syncwarp();
        return more != 0;
    };

    // ---- setup ----
    if (warp == MMA_WARP) {
        tmem_alloc(&tmem_base_sh, TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == TMA_WARP * 32) {
        mbar_init(&bar_q, 1);
        mbar_init(&bar_q_empty, 1);
        for (int s = 0; s < C::NP; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar_s_full[t], 1);
            mbar_init(&bar_p_full[t][0], 128);
            mbar_init(&bar_p_full[t][1], 128);
            mbar_init(&bar_o_full[t], 1);
        }
        mbar_init(&bar_drain, 1);
        abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if (!OUT_BF16) tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const uint64_t limit_ns = p.wait_limit_ns;

    // Each role's code sits inside the branch that set its register budget, so that the register
    // allocator sees the larger budget only where it holds.
    if (warp >= 8) {
        regs_decrease<CONTROL_REGS>();
        if (warp == TMA_WARP) {
            // ============ key/value producer (one lane): K_k0 per segment, then the stage ring ============
            if (elect_one()) {
                const uint64_t pol_kv = l2_policy_evict_last();
                WalkState& walk = walk_sh[TMA_WARP];
                const Segment& s = seg_sh[TMA_WARP];
                uint32_t g = 0;        // ring stages issued
                bool ok = true;
                bool skip_k = p.debug_skip_kv_load != 0;  // failure-path test: the first K is never loaded
                bool dep_done = dep_early;                  // the pre-pass's output may be read
                while (ok && walk_next(walk, tab, p.plan, static_cast<int>(blockIdx.x), seg_sh[TMA_WARP])) {
                    const SegInfo si = seg_info(p, s);
                    if (si.nmax == 0) continue;
                    // stage 0 of the segment: K_k0 alone; stage i >= 1: V_k0+i-1 and, but for the last,
                    // K_k0+i
                    const int jend = s.k0 + si.nmax;
                    for (int j = s.k0 - 1; j < jend; ++j) {
                        const uint32_t st = g % C::NP;
                        if (g >= C::NP &&
                            !mbar_wait(&bar_empty[st], ((g / C::NP) - 1) & 1, limit_ns, &abort_flag)) {
                            record_failure(&abort_flag, ERRBIT_WAIT_EMPTY);
                            ok = false;
                            break;
                        }
                        const bool has_v = j >= s.k0, has_k = j + 1 < jend;
                        if (has_v && !dep_done) {  // the first V tile comes from the pre-pass
                            grid_dep_wait();
                            dep_done = true;
                        }
                        mbar_arrive_expect_tx(&bar_full[st], (has_v ? C::TILE_BYTES : 0) + (has_k ? C::TILE_BYTES : 0));
                        uint8_t* dst = smem + C::OFF_RING + st * C::STAGE_BYTES;
                        if (has_v) {
                            if constexpr (FP8) {  // V^T tile: keys j*128.. (innermost), all d rows
                                tma_load_3d_hint(dst, &tmV, &bar_full[st], j * BLOCK_N, 0, si.zkv, pol_kv);
                            } else {
                                for (int bx = 0; bx < C::NB; ++bx)
                                    tma_load_3d_hint(dst + bx * 16384, &tmV, &bar_full[st], bx * 64, j * BLOCK_N,
                                                     si.zkv, pol_kv);
                            }
                        }
                        if (has_k && !skip_k)
                            for (int bx = 0; bx < C::NB; ++bx)
                                tma_load_3d_hint(dst + C::TILE_BYTES + bx * 16384, &tmK, &bar_full[st],
                                                 bx * C::BOX_ELEMS, (j + 1) * BLOCK_N, si.zkv, pol_kv);
                        skip_k = false;
                        ++g;
                    }
                }
                // On failure, wait (bounded) for the copies this thread issued, so that no TMA write
                // lands in shared memory after the CTA has exited.
                if (!ok || abort_flag) {
                    volatile int never = 0;  // these waits must not be cut short by the abort flag
                    for (uint32_t gg = g > C::NP ? g - C::NP : 0; gg < g; ++gg)
                        (void)mbar_wait(&bar_full[gg % C::NP], (gg / C::NP) & 1, limit_ns, &never);
                }
            }
            __syncwarp();
        } else if (warp == QLOAD_WARP) {
            // ====================== query producer (one lane): Q_0, Q_1 per segment ======================
            if (elect_one()) {
                const uint64_t pol_q = l2_policy_evict_first();
                WalkState& walk = walk_sh[QLOAD_WARP];
                const Segment& s = seg_sh[QLOAD_WARP];
                uint32_t segq = 0;     // segments whose Q was issued
                bool ok = true;
                while (ok && walk_next(walk, tab, p.plan, static_cast<int>(blockIdx.x), seg_sh[QLOAD_WARP])) {
                    const SegInfo si = seg_info(p, s);
                    if (si.nmax == 0) continue;
                    // Q_t is reused once the previous segment's MMAs completed (the epilogue stages its
                    // output elsewhere, so this load overlaps it)
                    if (segq > 0 && !mbar_wait(&bar_q_empty, (segq - 1) & 1, limit_ns, &abort_flag)) {
                        record_failure(&abort_flag, ERRBIT_WAIT_EMPTY);
                        ok = false;
                        break;
                    }
                    uint32_t qbytes = 0;
                    qbytes += si.n[0] > 0 ? C::TILE_BYTES : 0;
                    qbytes += si.n[1] > 0 ? C::TILE_BYTES : 0;
                    mbar_arrive_expect_tx(&bar_q, qbytes);
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (si.n[t] > 0)
                            for (int bx = 0; bx < C::NB; ++bx)
                                tma_load_3d_hint(smem + t * C::TILE_BYTES + bx * 16384, &tmQ, &bar_q,
                                                 bx * C::BOX_ELEMS, si.q0[t], si.bh, pol_q);
                    ++segq;
                }
                if (!ok || abort_flag) {
                    volatile int never = 0;
                    if (segq > 0) (void)mbar_wait(&bar_q, (segq - 1) & 1, limit_ns, &never);
                }
            }
            __syncwarp();
        } else if (warp == MMA_WARP) {
            // ======================= MMA issuer (converged warp, one lane issues) =======================
            auto wait_all = [&](uint64_t* bar, uint32_t parity, uint32_t bit) {
                const bool got = mbar_wait(bar, parity, limit_ns, &abort_flag);
                if (__all_sync(0xffffffffu, got)) return true;
                if (!got) record_failure(&abort_flag, bit);
                return false;
            };
            // Descriptors are built once; a k-step or stage moves the start address, which is the
            // low field (address >> 4) of the descriptor, so offsets are added to it directly.
            const uint64_t dQ = sdesc_sw128(smem_u32(smem), 16, 1024);
            const uint64_t dRingK = sdesc_sw128(smem_u32(smem + C::OFF_RING + C::TILE_BYTES), 16, 1024);
            // V: MN-major fp16 tile (keys x d), or, fp8, the K-major V^T tile (d rows x 128 keys)
            const uint64_t dRingV = sdesc_sw128(smem_u32(smem + C::OFF_RING), FP8 ? 16 : 16384, 1024);
            auto issue_S = [&](int t, uint64_t dk) {
                const uint64_t a = dQ + static_cast<uint64_t>((t * C::TILE_BYTES) >> 4);
                const uint32_t d = tmem + t * BLOCK_N;
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    if constexpr (FP8) umma_ss_f8(d, a + off, dk + off, C::IDESC_S, kk > 0);
                    else umma_ss(d, a + off, dk + off, C::IDESC_S, kk > 0);
                }
            };
            // P V over keys [64*half, 64*half + 64): four k-steps of 16 keys (fp16 P, 2 per TMEM
            // column), or two of 32 keys (E4M3 P, 4 per column); 8 columns per k-step either way
            auto issue_PV_half = [&](int t, uint64_t dv, int half, bool accumulate) {
                const uint32_t d = tmem + C::TMEM_O + t * D;
                const uint32_t a = tmem + t * BLOCK_N;
                if constexpr (FP8) {
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        const int kk = half * 2 + k2;
                        umma_ts_f8(d, a + kk * 8, dv + static_cast<uint64_t>((kk * 32) >> 4), C::IDESC_O,
                                   (accumulate || kk > 0));
                    }
                } else {
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const int kk = half * 4 + k4;
                        umma_ts(d, a + kk * 8, dv + static_cast<uint64_t>((kk * 2048) >> 4), C::IDESC_O,
                                (accumulate || kk > 0));
                    }
                }
            };
            const Segment& s = seg_sh[MMA_WARP];
            uint32_t g = 0, segq = 0;    // ring steps consumed, segments with a Q load
            uint32_t cnt_p[2] = {0u, 0u};
            bool ok = true;
            while (ok && next_seg()) {
                const SegInfo si = seg_info(p, s);
                if (si.nmax == 0) continue;
                // the segment's first ring stage holds K_k0 alone
                const uint32_t st0 = g % C::NP;
                if (!wait_all(&bar_full[st0], (g / C::NP) & 1, ERRBIT_WAIT_KV) ||
                    !wait_all(&bar_q, segq & 1, ERRBIT_WAIT_Q)) {
                    ok = false;
                    break;
                }
                ++segq;
                tc_fence_after();
                if (elect_one()) {
                    const uint64_t dk0 = dRingK + static_cast<uint64_t>((st0 * C::STAGE_BYTES) >> 4);
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (si.n[t] > 0) {
                            issue_S(t, dk0);
                            umma_commit(&bar_s_full[t]);
                        }
                    umma_commit(&bar_empty[st0]);
                }
                __syncwarp();
                ++g;
                bool stage_ready = false;  // this step's ring stage was seen complete during the last step
                for (int jj = 0; jj < si.nmax; ++jj) {
                    const uint32_t st = g % C::NP;
                    if (!stage_ready && !wait_all(&bar_full[st], (g / C::NP) & 1, ERRBIT_WAIT_KV)) {
                        ok = false;
                        break;
                    }
                    stage_ready = false;
                    tc_fence_after();
                    const uint64_t dv = dRingV + static_cast<uint64_t>((st * C::STAGE_BYTES) >> 4);
                    const uint64_t dk = dRingK + static_cast<uint64_t>((st * C::STAGE_BYTES) >> 4);
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (!ok || jj >= si.n[t]) continue;
                        if (!wait_all(&bar_p_full[t][0], cnt_p[t] & 1, ERRBIT_WAIT_P)) {
                            ok = false;
                            continue;
                        }
                        tc_fence_after();
                        if (elect_one()) issue_PV_half(t, dv, 0, jj > 0);
                        __syncwarp();
                        if (!wait_all(&bar_p_full[t][1], cnt_p[t] & 1, ERRBIT_WAIT_P)) {
                            ok = false;
                            continue;
                        }
                        ++cnt_p[t];
                        tc_fence_after();
                        if (elect_one()) {
                            issue_PV_half(t, dv, 1, true);
                            if (jj + 1 < si.n[t]) {
                                issue_S(t, dk);
                                umma_commit(&bar_s_full[t]);
                            } else {
                                umma_commit(&bar_o_full[t]);
                            }
                        }
                        __syncwarp();
                        // Deep rings (fp8, d = 64): between the two tiles' turns, a look (without
                        // waiting) at the next step's stage; when it has landed, the next step starts on
                        // tile 0's P at once (fp8 at B1 H16 N8192: 374.8 vs 383.0 us). With the two
                        // stages of d = 128 it has rarely landed by then, and the look alone cost 1.5%.
                        if constexpr (C::NP > 2) {
                            if (t == 0 && jj + 1 < si.nmax)
                                stage_ready = __all_sync(0xffffffffu,
                                                         mbar_test_wait(smem_u32(&bar_full[(g + 1) % C::NP]),
                                                                        ((g + 1) / C::NP) & 1));
                        }
                    }
                    if (!ok) break;
                    if (elect_one()) umma_commit(&bar_empty[st]);
                    __syncwarp();
                    ++g;
                }
                if (!ok) break;
                // Q of this segment may be overwritten once these MMAs completed
                if (elect_one()) umma_commit(&bar_q_empty);
                __syncwarp();
            }
            // Drain: every MMA this warp issued has completed before tensor memory is freed.
            if (elect_one()) umma_commit(&bar_drain);
            __syncwarp();
            volatile int never = 0;  // not cut short by the abort flag: the drain must finish
            const bool drained = mbar_wait(&bar_drain, 0, limit_ns, &never);
            if (!__all_sync(0xffffffffu, drained) && lane == 0) record_failure(&abort_flag, ERRBIT_WAIT_DRAIN);
        }
    } else {
        regs_increase<SOFTMAX_REGS>();
        // ============================ softmax warpgroups ============================
        if (!dep_early) grid_dep_wait();  // tile exponents of V, flags of the schedule
        const int t = warp >> 2;            // query tile of this warpgroup
        const int wq = warp & 3;            // TMEM lane quarter
        const int r = wq * 32 + lane;       // row within the tile
        const uint32_t lane_off = tmem_lane_base(wq);
        const uint32_t tS = tmem + lane_off + t * BLOCK_N;
        const uint32_t tO = tmem + lane_off + C::TMEM_O + t * D;
        const float sl = p.scale_log2;
        const int G = p.plan.G;
        const Segment& s = seg_sh[warp];
        uint32_t cnt_s = 0, cnt_o = 0;  // S_t and O_t phases waited for
        bool ok = true;
        bool staged = false;  // this warp's staging box may still be read by the store engine

        while (ok && next_seg()) {
            // only what the key loop needs stays in registers; the rest is re-read from shared memory
            const int k0 = s.k0;
            const int q0t = s.pair * 2 * BLOCK_M + t * BLOCK_M;
            const int kv_valid = clamp_len(p.kv_len, s.b, p.plan.N);
            int nkvt = 0;
            if (q0t < p.plan.N) {
                const int hi = min(s.k1, key_tiles(p.plan.causal ? min(kv_valid, q0t + BLOCK_M) : kv_valid));
                nkvt = hi > k0 ? hi - k0 : 0;
            }

            const int row = q0t + r;                   // query index
            const int row_lim = p.plan.causal ? min(kv_valid, row + 1) : kv_valid;  // keys < row_lim are valid
            // per-tile exponents of the fp16 V copy; this piece's O holds sum P V * 2^-E with E the
            // largest exponent of the tiles seen so far (the same for every row of the tile)
            const int32_t* vexp_row = p.v_exp + static_cast<size_t>(s.b * p.H_kv + s.h / p.group) * p.n_ktiles;
            // fp8: the stored Q and K tiles stand for their values times 2^eq and 2^ek, so a score is
            // the tensor-core sum times 2^(eq + ek); both go into the multiplier of this tile
            float sl_t = sl;
            const int32_t* kexp_row = nullptr;
            if constexpr (FP8) {
                kexp_row = p.k_exp + static_cast<size_t>(s.b * p.H_kv + s.h / p.group) * p.n_ktiles;
                if (q0t < p.plan.N)
                    sl_t = ldexpf(sl, __ldg(p.q_exp + static_cast<size_t>(s.b * p.plan.H + s.h) * p.n_ktiles +
                                            q0t / BLOCK_M));
            }
            // bias + dropout: this row's bias (nullptr: none, or a row past N) and its Philox counter words
            const uint16_t* brow = nullptr;
            if constexpr (EXTRA) {
                if (p.bias && row < p.plan.N)
                    brow = p.bias + s.b * p.bias_sb + s.h * p.bias_sh + static_cast<long long>(row) * p.bias_sr;
            }
            int E = 0;
            float m_run = -INFINITY;                   // reference maximum (log2 domain, already scaled)
            float l_run = 0.f;                         // running sum of exp2(s*sl - m_run), as P V uses them

            for (int jj = 0; jj < nkvt; ++jj) {
                const int j = k0 + jj;
                const int e_j = __ldg(vexp_row + j);
                float slj = sl;
                if constexpr (FP8) slj = ldexpf(sl_t, __ldg(kexp_row + j));
                // bias + dropout: this tile's 128 bias values of the row, loaded before the wait for S
                // so that their latency overlaps it (keys past N read as 0; they are masked anyway)
                uint4 bv[EXTRA ? 16 : 1];
                if constexpr (EXTRA) {
                    const int kb = j * BLOCK_N;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int kc = kb + 8 * c;
                        if (brow == nullptr) {
                            bv[c] = make_uint4(0u, 0u, 0u, 0u);
                        } else if (kc + 8 <= p.plan.N) {
                            bv[c] = __ldg(reinterpret_cast<const uint4*>(brow + kc));
                        } else {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const uint32_t lo = kc + 2 * e < p.plan.N ? __ldg(brow + kc + 2 * e) : 0u;
                                const uint32_t hi = kc + 2 * e + 1 < p.plan.N ? __ldg(brow + kc + 2 * e + 1) : 0u;
                                w[e] = lo | (hi << 16);
                            }
                            bv[c] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                    // the row's bias two tiles ahead (one tile ahead as well at the first step) into L2,
                    // so that the loads above find it there; only 128-byte lines inside the row's N keys
                    if (brow != nullptr) {
#pragma unroll
                        for (int a = (jj == 0 ? 1 : 2); a <= 2; ++a) {
                            const int kp = kb + a * BLOCK_N;
                            if (jj + a < nkvt) {
                                if (kp + 64 <= p.plan.N) prefetch_l2(brow + kp);
                                if (kp + 128 <= p.plan.N) prefetch_l2(brow + kp + 64);
                            }
                        }
                    }
                }
                // tcgen05.ld/st below are warp-collective: the warp proceeds only if every lane's wait
                // succeeded
                const bool got = mbar_wait(&bar_s_full[t], cnt_s & 1, limit_ns, &abort_flag);
                ++cnt_s;
                if (!__all_sync(0xffffffffu, got)) {
                    if (!got) record_failure(&abort_flag, ERRBIT_WAIT_S);
                    ok = false;
                    break;
                }
                tc_fence_after();
                float x[128];
                if constexpr (EXTRA) {
                    // scores to the log2 domain with the bias added: x = S * scale*log2e + bias * log2e,
                    // in two halves so that the bias registers of a half die before the next half lands
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t ra[32], rb[32];
                        tmem_ld32(tS + 64 * hh, ra);
                        tmem_ld32(tS + 64 * hh + 32, rb);
                        tmem_wait_ld(ra);
                        tmem_wait_ld(rb);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint4 b4 = bv[8 * hh + c];
                            const uint32_t w[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = 8 * c + 2 * e;  // key within the half
                                const uint32_t s0 = i < 32 ? ra[i] : rb[i - 32];
                                const uint32_t s1 = i + 1 < 32 ? ra[i + 1] : rb[i + 1 - 32];
                                x[64 * hh + i] = fmaf(__uint_as_float(w[e] << 16), 1.4426950408889634f,
                                                      __uint_as_float(s0) * slj);
                                x[64 * hh + i + 1] = fmaf(__uint_as_float(w[e] & 0xffff0000u), 1.4426950408889634f,
                                                          __uint_as_float(s1) * slj);
                            }
                        }
                    }
                    slj = 1.0f;  // x is already in log2 units
                } else {
                    uint32_t ra[32], rb[32], rc[32], rd[32];
                    tmem_ld32(tS + 0, ra);
                    tmem_ld32(tS + 32, rb);
                    tmem_ld32(tS + 64, rc);
                    tmem_ld32(tS + 96, rd);
                    tmem_wait_ld(ra);
                    tmem_wait_ld(rb);
                    tmem_wait_ld(rc);
                    tmem_wait_ld(rd);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        x[i] = __uint_as_float(ra[i]);
                        x[32 + i] = __uint_as_float(rb[i]);
                        x[64 + i] = __uint_as_float(rc[i]);
                        x[96 + i] = __uint_as_float(rd[i]);
                    }
                }
                const int key0 = j * BLOCK_N;
                if (key0 + BLOCK_N > kv_valid || (p.plan.causal && key0 + BLOCK_N - 1 > q0t)) {
                    const int lim = row_lim - key0;
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i >= lim) x[i] = -INFINITY;
                }
                // row maximum: four independent chains of three-input maxima over x[4..123], then
                // the last four values
                float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
                for (int i = 4; i < 124; i += 8) {
                    mx0 = max3f(mx0, x[i], x[i + 1]);
                    mx1 = max3f(mx1, x[i + 2], x[i + 3]);
                    mx2 = max3f(mx2, x[i + 4], x[i + 5]);
                    mx3 = max3f(mx3, x[i + 6], x[i + 7]);
                }
                mx0 = max3f(mx0, x[124], x[125]);
                mx1 = max3f(mx1, x[126], x[127]);
                const float m_tile = max3f(mx0, mx1, fmaxf(mx2, mx3)) * slj;
                float alpha = 1.f;
                bool rescale = false;
                if (jj == 0) {
                    m_run = m_tile;
                    E = e_j;
                } else {
                    if (m_tile > m_run + C::RESCALE_THRESHOLD) {
                        alpha = ex2_approx(m_run - m_tile);
                        l_run *= alpha;
                        m_run = m_tile;
                        rescale = true;
                    }
                    if (e_j > E) {  // a tile of larger |V|: the accumulator moves to its exponent (exact)
                        alpha = ldexpf(alpha, E - e_j);
                        E = e_j;
                        rescale = true;
                    }
                }
                // Lazy rescale of O_t before any of this tile's P V lands in it (the previous P V into
                // O_t has completed: its completion preceded the S_t commit this warpgroup waited on).
                if (__any_sync(0xffffffffu, rescale)) {
                    const f32x2 al2 = make_f32x2(alpha, alpha);
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_wait_ld(o);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float a0, a1;
                            split_f32x2(
                                mul_f32x2(make_f32x2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), al2),
                                a0, a1);
                            o[2 * i] = __float_as_uint(a0);
                            o[2 * i + 1] = __float_as_uint(a1);
                        }
                        tmem_st32(tO + c * 32, o);
                    }
                }
                const float m_sub = (m_run == -INFINITY) ? 0.f : m_run;
                // P = exp2(s * scale*log2e - m), written to TMEM as fp16 pairs (E4M3 quadruples) over the
                // first 64 (32) columns of S_t, one half (64 keys) at a time; each half is announced as
                // soon as it is stored. The scale-and-subtract (and fp8's row sum) use two-wide fp32
                // instructions. A tile whose V exponent is below E enters as P * 2^(e_j - E) (folded into
                // the exponent); the row sums take P itself.
                // The row sum (O's divisor and the LSE's sum) takes P as the P V product uses it: rounded
                // to fp16 and before dropout. A row dominated by one key then divides that key's rounding
                // out of O instead of keeping it (up to 2^-12 |V| otherwise), and O, LSE stay consistent
                // for a merge of partial results. It is taken from the packed pairs after both halves are
                // handed over, while the warpgroup waits for its next S (with dropout, in the loop,
                // before the draws zero some of P). fp8 sums its fp32 exponentials in the loop (its
                // E4M3 rounding, 2^-4, would move the LSE too far).
                {
                    const int shift = e_j - E;  // <= 0, almost always 0
                    const f32x2 sl2 = make_f32x2(slj, slj);
                    const f32x2 nm2 = make_f32x2(static_cast<float>(shift) - m_sub, static_cast<float>(shift) - m_sub);
                    f32x2 acc0 = make_f32x2(0.f, 0.f), acc1 = acc0;
                    float q0 = 0.f, q1 = 0.f, q2 = 0.f, q3 = 0.f;  // the fp16 row sum of this tile, four chains
                    uint32_t pk[2][FP8 ? 16 : 32];  // both halves' P, kept for the deferred row sum
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        if constexpr (FP8) {
                            // E4M3, four keys per TMEM column: 16 columns per half
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                float e0, e1, e2, e3;
                                const int c0 = 64 * half + 4 * i;
                                split_f32x2(fma_f32x2(make_f32x2(x[c0], x[c0 + 1]), sl2, nm2), e0, e1);
                                split_f32x2(fma_f32x2(make_f32x2(x[c0 + 2], x[c0 + 3]), sl2, nm2), e2, e3);
                                e0 = ex2_approx(e0);
                                e1 = ex2_approx(e1);
                                e2 = ex2_approx(e2);
                                e3 = ex2_approx(e3);
                                acc0 = add_f32x2(acc0, make_f32x2(e0, e1));
                                acc1 = add_f32x2(acc1, make_f32x2(e2, e3));
                                pk[half][i] = pack_e4m3x4(e0, e1, e2, e3);
                            }
                            tmem_st16(tS + 16 * half, pk[half]);
                        } else {
                            uint4 rnd = make_uint4(0u, 0u, 0u, 0u);  // dropout draws of 8 keys
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                float e0, e1;
                                split_f32x2(
                                    fma_f32x2(make_f32x2(x[64 * half + 2 * i], x[64 * half + 2 * i + 1]), sl2, nm2),
                                    e0, e1);
                                pk[half][i] = pack_f16x2(ex2_approx(e0), ex2_approx(e1));
                                if constexpr (EXTRA) {
                                    if (i & 1) {
                                        q2 = add_f16lo(q2, pk[half][i]);
                                        q3 = add_f16hi(q3, pk[half][i]);
                                    } else {
                                        q0 = add_f16lo(q0, pk[half][i]);
                                        q1 = add_f16hi(q1, pk[half][i]);
                                    }
                                    if (p.drop_t != 0u) {
                                        // keys 2i, 2i+1 of this half: word (i mod 4) of the draws of their
                                        // group of 8, low half for the even key, high half for the odd one
                                        if ((i & 3) == 0)
                                            rnd = philox4x32_10(
                                                make_uint4(static_cast<uint32_t>((key0 + 64 * half + 2 * i) >> 3),
                                                           static_cast<uint32_t>(row),
                                                           static_cast<uint32_t>(s.b * p.plan.H + s.h), p.rng_offset),
                                                p.round_key);
                                        const uint32_t w = (i & 3) == 0 ? rnd.x : (i & 3) == 1 ? rnd.y
                                                         : (i & 3) == 2 ? rnd.z : rnd.w;
                                        if ((w & 0xffffu) < p.drop_t) pk[half][i] &= 0xffff0000u;  // +0, low half
                                        if ((w >> 16) < p.drop_t) pk[half][i] &= 0x0000ffffu;
                                    }
                                }
                            }
                            tmem_st32(tS + 32 * half, pk[half]);
                        }
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(&bar_p_full[t][half]);
                    }
                    if constexpr (!FP8 && !EXTRA) {
#pragma unroll
                        for (int half = 0; half < 2; ++half)
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                q0 = add_f16lo(q0, pk[half][i]);
                                q1 = add_f16hi(q1, pk[half][i]);
                                q2 = add_f16lo(q2, pk[half][i + 1]);
                                q3 = add_f16hi(q3, pk[half][i + 1]);
                            }
                    }
                    float psum;
                    if constexpr (FP8) {
                        float s0, s1, s2, s3;
                        split_f32x2(acc0, s0, s1);
                        split_f32x2(acc1, s2, s3);
                        psum = (s0 + s1) + (s2 + s3);
                    } else {
                        psum = (q0 + q1) + (q2 + q3);
                    }
                    l_run += shift == 0 ? psum : ldexpf(psum, -shift);
                }
            }
            if (!ok) break;

            // ---- end of the piece: O_t of this piece is complete once the last P V finished ----
            const bool have = nkvt > 0;
            if (have) {
                const bool got = mbar_wait(&bar_o_full[t], cnt_o & 1, limit_ns, &abort_flag);
                ++cnt_o;
                if (!__all_sync(0xffffffffu, got)) {
                    if (!got) record_failure(&abort_flag, ERRBIT_WAIT_O);
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            const bool live = have && l_run > 0.f;     // this row got weight from this piece

            if (s.kind == SEG_WRITER) {
                // partial result for the owner of the unit: unnormalised O (row fastest), m, l
                float* base = p.part + (static_cast<size_t>(blockIdx.x) * 2 + t) * (D + 3) * BLOCK_M;
                if (have) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_wait_ld(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) base[(c * 32 + i) * BLOCK_M + r] = __uint_as_float(o[i]);
                    }
                }
                base[D * BLOCK_M + r] = live ? m_run : -INFINITY;
                base[(D + 1) * BLOCK_M + r] = live ? l_run : 0.f;
                base[(D + 2) * BLOCK_M + r] = static_cast<float>(E);
                __threadfence();
                __syncwarp();
                if (lane == 0) flag_release(p.flags + (blockIdx.x * 2 + t) * 4 + wq, 1u);
                continue;
            }
            if (q0t >= p.plan.N) continue;  // a tile past the last row: nothing to write

            // COMPLETE or OWNER: gather the partial results of the unit's other pieces (owner only)
            const int W = walk_sh[warp].W;
            int c_end = blockIdx.x + 1;
            float M = live ? m_run : -INFINITY;
            int Emax = live ? E : -1000000;
            // The first two other pieces (the usual case) keep their m, l, E in registers so that each
            // output chunk needs one round trip to L2; further pieces are re-read (rare).
            int np = 0;
            const float* pb0 = nullptr;
            const float* pb1 = nullptr;
            float pm0 = -INFINITY, pl0 = 0.f, pm1 = -INFINITY, pl1 = 0.f;
            int pe0 = 0, pe1 = 0;
            if (s.kind == SEG_OWNER) {
                while (c_end < G && sched_chunk_start(p.plan, W, c_end) < s.unit_end) ++c_end;
                for (int c2 = blockIdx.x + 1; c2 < c_end && ok; ++c2) {
                    if (sched_chunk_start(p.plan, W, c2 + 1) <= sched_chunk_start(p.plan, W, c2)) continue;
                    if (!flag_wait(p.flags + (c2 * 2 + t) * 4 + wq, 1u, limit_ns, &abort_flag)) {
                        record_failure(&abort_flag, ERRBIT_WAIT_PART);
                        ok = false;
                        break;
                    }
                    const float* b2 = p.part + (static_cast<size_t>(c2) * 2 + t) * (D + 3) * BLOCK_M;
                    const float m2 = __ldcg(b2 + D * BLOCK_M + r);
                    const float l2 = __ldcg(b2 + (D + 1) * BLOCK_M + r);
                    const int e2 = static_cast<int>(__ldcg(b2 + (D + 2) * BLOCK_M + r));
                    if (np == 0) {
                        pb0 = b2; pm0 = m2; pl0 = l2; pe0 = e2;
                    } else if (np == 1) {
                        pb1 = b2; pm1 = m2; pl1 = l2; pe1 = e2;
                    }
                    ++np;
                    if (l2 > 0.f) {
                        M = fmaxf(M, m2);
                        Emax = max(Emax, e2);
                    }
                }
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
            }
            // softmax merge of the pieces: weights 2^(m_i - M) on l, 2^(m_i - M + E_i - Emax) on O
            const float w_own_l = live ? ex2_approx(m_run - M) : 0.f;
            const float w_own = live ? w_own_l * pow2i(E - Emax) : 0.f;
            const float w0l = pl0 > 0.f ? ex2_approx(pm0 - M) : 0.f;
            const float w1l = pl1 > 0.f ? ex2_approx(pm1 - M) : 0.f;
            const float w0 = pl0 > 0.f ? w0l * pow2i(pe0 - Emax) : 0.f;
            const float w1 = pl1 > 0.f ? w1l * pow2i(pe1 - Emax) : 0.f;
            float L = w_own_l * l_run + w0l * pl0 + w1l * pl1;
            int c_extra = c_end;  // first CTA whose piece is beyond the two kept in registers
            if (np > 2) {
                int k = 0;
                for (int c2 = blockIdx.x + 1; c2 < c_end; ++c2) {
                    if (sched_chunk_start(p.plan, W, c2 + 1) <= sched_chunk_start(p.plan, W, c2)) continue;
                    if (++k == 3) {
                        c_extra = c2;
                        break;
                    }
                }
                for (int c2 = c_extra; c2 < c_end; ++c2) {
                    const float* b2 = p.part + (static_cast<size_t>(c2) * 2 + t) * (D + 3) * BLOCK_M;
                    if (sched_chunk_start(p.plan, W, c2 + 1) <= sched_chunk_start(p.plan, W, c2)) continue;
                    const float l2 = __ldcg(b2 + (D + 1) * BLOCK_M + r);
                    if (l2 > 0.f) L += ex2_approx(__ldcg(b2 + D * BLOCK_M + r) - M) * l2;
                }
            }
            const int bh = s.b * p.plan.H + s.h;
            float inv = L > 0.f ? pow2i(Emax) * __frcp_rn(L) : 0.f;
            if constexpr (EXTRA) inv *= p.keep_scale;  // inverted dropout (1 without dropout)
            const bool store = row < p.plan.N;
            const size_t obase = (static_cast<size_t>(bh) * p.plan.N + (store ? row : 0)) * D;
            // this warp's staging boxes, which the store engine must have read since the warp's last
            // epilogue (long done by now: a whole segment ran in between)
            const uint32_t stage_base = smem_u32(smem + C::OFF_EPI + (t * 4 + wq) * C::EPI_BUFS * 4096);
            if (!OUT_BF16 && staged) {
                if (lane == 0) bulk_wait_group_read<0>();
                __syncwarp();
            }
            // A unit with no other pieces (the usual case) and fp32 output: two chunks per pass, both
            // read from tensor memory together and staged behind one proxy fence; the weight and the
            // normalisation fold into one factor.
            const bool fast = !OUT_BF16 && C::EPI_BUFS >= 2 && np == 0;
            if (fast) {
                const float sc = have ? w_own * inv : 0.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; c += 2) {
                    uint32_t oa[32], ob[32];
                    if (have) {
                        tmem_ld32(tO + c * 32, oa);
                        tmem_ld32(tO + (c + 1) * 32, ob);
                        tmem_wait_ld(oa);
                        tmem_wait_ld(ob);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) oa[i] = ob[i] = 0u;
                    }
                    if (c >= C::EPI_BUFS) {  // the store engine has read the buffers of the last pass
                        if (lane == 0) bulk_wait_group_read<0>();
                        __syncwarp();
                    }
                    const uint32_t bufa = stage_base + (c % C::EPI_BUFS) * 4096;
                    const uint32_t bufb = stage_base + ((c + 1) % C::EPI_BUFS) * 4096;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = lane * 128 + ((k ^ (lane & 7)) << 4);
                        st_shared_v4(bufa + off, __float_as_uint(__uint_as_float(oa[4 * k]) * sc),
                                     __float_as_uint(__uint_as_float(oa[4 * k + 1]) * sc),
                                     __float_as_uint(__uint_as_float(oa[4 * k + 2]) * sc),
                                     __float_as_uint(__uint_as_float(oa[4 * k + 3]) * sc));
                        st_shared_v4(bufb + off, __float_as_uint(__uint_as_float(ob[4 * k]) * sc),
                                     __float_as_uint(__uint_as_float(ob[4 * k + 1]) * sc),
                                     __float_as_uint(__uint_as_float(ob[4 * k + 2]) * sc),
                                     __float_as_uint(__uint_as_float(ob[4 * k + 3]) * sc));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tmO, smem + (bufa - smem_u32(smem)), c * 32, q0t + wq * 32, bh);
                        tma_store_3d(&tmO, smem + (bufb - smem_u32(smem)), (c + 1) * 32, q0t + wq * 32, bh);
                        bulk_commit_group();
                    }
                    __syncwarp();
                }
            }
#pragma unroll 1
            for (int c = 0; c < (fast ? 0 : D / 32); ++c) {
                uint32_t o[32];
                if (have) {
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld(o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                // o holds the merged, still unnormalised row values (fp32 bits)
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(have ? __uint_as_float(o[i]) * w_own : 0.f);
                if (np > 0) {  // the first two other pieces: all loads of the chunk in flight together
                    float v0[32], v1[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        v0[i] = w0 != 0.f ? __ldcg(pb0 + (c * 32 + i) * BLOCK_M + r) : 0.f;
                        v1[i] = w1 != 0.f ? __ldcg(pb1 + (c * 32 + i) * BLOCK_M + r) : 0.f;
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = __float_as_uint(fmaf(w1, v1[i], fmaf(w0, v0[i], __uint_as_float(o[i]))));
                }
                for (int c2 = c_extra; c2 < c_end; ++c2) {  // further pieces (rare)
                    if (sched_chunk_start(p.plan, W, c2 + 1) <= sched_chunk_start(p.plan, W, c2)) continue;
                    const float* b2 = p.part + (static_cast<size_t>(c2) * 2 + t) * (D + 3) * BLOCK_M;
                    if (!(__ldcg(b2 + (D + 1) * BLOCK_M + r) > 0.f)) continue;
                    const float w2 = ldexpf(ex2_approx(__ldcg(b2 + D * BLOCK_M + r) - M),
                                            static_cast<int>(__ldcg(b2 + (D + 2) * BLOCK_M + r)) - Emax);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = __float_as_uint(fmaf(w2, __ldcg(b2 + (c * 32 + i) * BLOCK_M + r), __uint_as_float(o[i])));
                }
                if constexpr (OUT_BF16) {
                    if (store) {
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
                    }
                } else {
                    // fp32 rows leave through the tensor store engine: the warp stages its 32 rows x 32
                    // columns (128-byte swizzled, 4 KB) in one of its staging boxes and one lane stores
                    // the box (rows past N are not written). Boxes are reused once the store engine has
                    // read them.
                    const uint32_t buf = stage_base + (c % C::EPI_BUFS) * 4096;
                    if (c >= C::EPI_BUFS) {
                        if (lane == 0) bulk_wait_group_read<C::EPI_BUFS - 1>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        st_shared_v4(buf + lane * 128 + ((k ^ (lane & 7)) << 4),
                                     __float_as_uint(__uint_as_float(o[4 * k]) * inv),
                                     __float_as_uint(__uint_as_float(o[4 * k + 1]) * inv),
                                     __float_as_uint(__uint_as_float(o[4 * k + 2]) * inv),
                                     __float_as_uint(__uint_as_float(o[4 * k + 3]) * inv));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tmO, smem + (buf - smem_u32(smem)), c * 32, q0t + wq * 32, bh);
                        bulk_commit_group();
                    }
                    __syncwarp();
                }
            }
            if (store && p.LSE) {
                const float lse = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
                p.LSE[static_cast<size_t>(bh) * p.plan.N + row] = lse;
            }
            if constexpr (!OUT_BF16) staged = true;
        }
    }

    // ---- teardown ----
    if (!OUT_BF16 && warp < 8 && lane == 0) bulk_wait_group_all();  // output stores performed
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------------
// V -> fp16, one 128-row key tile per CTA (a single pass: the tile stays in registers between its
// |V| maximum and the conversion). The tile's exponent e keeps |V| * 2^-e < 2^15; values too small
// for fp16 lose only absolute precision far below the result's rounding (below 2^-25 |V|max).
// ---------------------------------------------------------------------------------------------
// The schedule's batch offsets: boff[b] = sum over b' < b of H * (one head's line length in batch b'),
// computed by one block; it also clears the partial-result flags of the attention kernel.
__device__ void plan_block(const PlanParams& pl) {
    __shared__ long long part[256];
    const int tid = threadIdx.x;
    const bool act = tid < 256;  // 256 partial sums; larger blocks' other threads only clear flags
    const int per = (pl.B + 255) / 256;
    const int b0 = act ? min(pl.B, tid * per) : 0, b1 = act ? min(pl.B, b0 + per) : 0;
    long long sum = 0;
    for (int b = b0; b < b1; ++b) {
        const int nb = key_tiles(clamp_len(pl.kv_len, b, pl.N));
        sum += static_cast<long long>(pl.H) * line_prefix(pl.n_pairs, nb, pl.N, pl.causal);
    }
    if (act) part[tid] = sum;
    __syncthreads();
    if (tid == 0) {  // exclusive scan of 256 partial sums
        long long run = 0;
        for (int i = 0; i < 256; ++i) {
            const long long v = part[i];
            part[i] = run;
            run += v;
        }
        pl.boff[pl.B] = run;
    }
    __syncthreads();
    long long run = act ? part[tid] : 0;
    for (int b = b0; b < b1; ++b) {
        pl.boff[b] = run;
        const int nb = key_tiles(clamp_len(pl.kv_len, b, pl.N));
        run += static_cast<long long>(pl.H) * line_prefix(pl.n_pairs, nb, pl.N, pl.causal);
    }
    for (int i = tid; i < 8 * SCHED_MAX_CTAS; i += blockDim.x) pl.flags[i] = 0u;
}

constexpr int VPREP_THREADS = 256;
constexpr int VPREP_VECS = 128 * 128 / 8 / VPREP_THREADS;  // 16-byte vectors per thread (d = 128)

__global__ void __launch_bounds__(VPREP_THREADS) vprep_kernel(const VPrepParams p, const PlanParams pl) {
    grid_dep_launch_dependents();  // the attention kernel may start its set-up on SMs this pass leaves
    const int tile = blockIdx.x, head = blockIdx.y;
    if (head == p.heads) {  // the extra row of blocks: block 0 plans, the others have nothing to do
        if (tile == 0) plan_block(pl);
        return;
    }
    const int rows = min(128, p.N - tile * 128);
    const int nvec = rows * p.d / 8;  // d is a multiple of 64
    const size_t base = (static_cast<size_t>(head) * p.N + static_cast<size_t>(tile) * 128) * p.d;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.V) + base);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(p.V16) + base);
    uint4 u[VPREP_VECS];
    uint32_t mbits = 0;  // largest |V| as bf16 bits (the order of non-negative floats is that of their bits)
#pragma unroll
    for (int k = 0; k < VPREP_VECS; ++k) {
        const int i = threadIdx.x + k * VPREP_THREADS;
        u[k] = i < nvec ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) mbits = max(mbits, max(w[e] & 0x7fffu, (w[e] >> 16) & 0x7fffu));
    }
    mbits = __reduce_max_sync(0xffffffffu, mbits);
    __shared__ uint32_t red[VPREP_THREADS / 32];
    __shared__ int e_sh;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mbits;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t m = 0;
        for (int i = 0; i < VPREP_THREADS / 32; ++i) m = max(m, red[i]);
        const int e8 = static_cast<int>((m >> 7) & 0xffu);  // biased exponent: |V| < 2^(e8 - 126)
        const int e = (e8 == 0xff || e8 <= 141) ? 0 : e8 - 141;  // NaN/Inf propagate unscaled
        e_sh = e;
        p.v_exp[static_cast<size_t>(head) * p.n_ktiles + tile] = e;
    }
    __syncthreads();
    const int e = e_sh;
    const float sc = ldexpf(1.0f, -e);
#pragma unroll
    for (int k = 0; k < VPREP_VECS; ++k) {
        const int i = threadIdx.x + k * VPREP_THREADS;
        if (i >= nvec) continue;
        uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = __uint_as_float(w[q] << 16) * sc;
            const float hi = __uint_as_float(w[q] & 0xffff0000u) * sc;
            w[q] = pack_f16x2(lo, hi);
        }
        dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_vprep(const VPrepParams& p, const PlanParams& plan, cudaStream_t stream) {
    vprep_kernel<<<dim3(p.n_ktiles, p.heads + 1), VPREP_THREADS, 0, stream>>>(p, plan);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// fp8 pre-pass (d = 128): a persistent grid of 512-thread blocks, two per SM, each taking every G-th
// 128-row tile of the list (Q tiles, then K tiles, then V tiles), plus one block that plans the
// schedule. A tile (128 rows x 256 bytes, contiguous in BHND) reaches shared memory by one bulk copy
// into a two-stage ring: the copy of a block's next tile is in flight while it works on the current
// one, so the copy engines, not registers, hold the bytes in flight that HBM bandwidth needs.
// Q and K rows are multiplied by the signs and transformed by the unnormalised Walsh-Hadamard
// butterflies (spans 1, 2, 4, ..., 64 in that order; each output one fp32 addition or subtraction),
// then every tile is rounded to E4M3 at its own power-of-two scale. Four threads share a row (32
// elements each).
// ---------------------------------------------------------------------------------------------
constexpr int FP8P_THREADS = 512;
constexpr int FP8P_BLOCKS_PER_SM = 2;
constexpr int FP8P_STAGES = 2;
constexpr int FP8P_TILE_BYTES = 128 * 128 * 2;               // one bf16 tile, 256 bytes per row
constexpr int FP8P_SMEM = FP8P_STAGES * FP8P_TILE_BYTES;       // dynamic shared memory of the ring

// Tile exponent from the largest |x| as fp32 bits: max |x| < 2^(e8 - 126); e = max(e8 - 134, -100)
// keeps the tile's values times 2^-e below 256 = 2^8 (E4M3 holds up to 448); a zero tile gets 0.
__device__ __forceinline__ int fp8_tile_exponent(uint32_t max_abs_bits) {
    if (max_abs_bits == 0) return 0;
    const int e8 = static_cast<int>((max_abs_bits >> 23) & 0xffu);
    return max(e8 - 134, -100);
}

// Block-wide maximum of non-negative fp32 bit patterns (their order is that of the values). `bad`
// (this thread's copy wait gave up) is OR-reduced over the block by the same barrier, so that every
// thread takes the same decision.
__device__ __forceinline__ uint32_t fp8_block_max(uint32_t v, uint32_t* red, bool& bad) {
    v = __reduce_max_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    bad = __syncthreads_or(bad) != 0;
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < FP8P_THREADS / 32; ++i) m = max(m, red[i]);
    return m;
}

// 2^-e as fp32 for e in [-100, 120]
__device__ __forceinline__ float fp8_pow2_neg(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// One 128-row tile of Q or K, staged row-major in shared memory: thread t holds row t / 4, elements
// 32 (t mod 4) .. +31 as sixteen fp32 pairs. The signs are XORed into the bf16 words before they are
// widened (a sign flip is exact). Butterflies of span 1 run on single values, spans 2 .. 16 on pairs
// (two-wide fp32 adds and x - y = fma(y, -1, x), both single-rounded like the scalar forms), span 32
// pairs lanes 4r + q and 4r + (q ^ 1), span 64 lanes 4r + q and 4r + (q ^ 2), each as one fma with a
// factor of +-1; the lower element of a pair keeps x + y, the upper x - y.
template <class AfterMax>
__device__ bool fp8_prep_qk_tile(const uint8_t* stage, uint8_t* dst, int32_t* exp_out, const uint32_t* sgn,
                                 int N, int tile, uint32_t* red, bool bad, AfterMax after_max) {
    const int q4 = threadIdx.x & 3;
    const int r = threadIdx.x >> 2;
    const int row = tile * 128 + r;
    uint32_t w[16];  // bf16 pairs: element 2e in the low half of w[e], element 2e + 1 in the high half
    if (row < N) {
        // The thread's four 16-byte chunks are read in an order rotated by rot = (q4 >> 1) + 2 (r & 1):
        // rows lie 256 bytes apart, so without it the eight threads of a quarter warp (rows 2p, 2p + 1,
        // quarters 0-3) would fall on four bank groups; rotated, they cover all eight at every step.
        const int rot = ((q4 >> 1) + 2 * (r & 1)) & 3;
        const uint8_t* base = stage + r * 256 + q4 * 64;
        uint4 u0 = lds128(base + ((0 + rot) & 3) * 16);
        uint4 u1 = lds128(base + ((1 + rot) & 3) * 16);
        uint4 u2 = lds128(base + ((2 + rot) & 3) * 16);
        uint4 u3 = lds128(base + ((3 + rot) & 3) * 16);
        if (rot & 1) {  // chunk c is in u[(c - rot) & 3]: rotate back by one, then by two
            const uint4 t = u3;
            u3 = u2;
            u2 = u1;
            u1 = u0;
            u0 = t;
        }
        if (rot & 2) {
            uint4 t = u0;
            u0 = u2;
            u2 = t;
            t = u1;
            u1 = u3;
            u3 = t;
        }
        const uint4 uu[4] = {u0, u1, u2, u3};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w[4 * k] = uu[k].x;
            w[4 * k + 1] = uu[k].y;
            w[4 * k + 2] = uu[k].z;
            w[4 * k + 3] = uu[k].w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = 0u;
    }
    f32x2 b[16];
    if (sgn) {
        const uint4* s4 = reinterpret_cast<const uint4*>(sgn + q4 * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 m = s4[k];
            w[4 * k] ^= m.x;
            w[4 * k + 1] ^= m.y;
            w[4 * k + 2] ^= m.z;
            w[4 * k + 3] ^= m.w;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {  // span 1
            const float x = __uint_as_float(w[e] << 16), y = __uint_as_float(w[e] & 0xffff0000u);
            b[e] = make_f32x2(x + y, x - y);
        }
        const f32x2 neg1 = make_f32x2(-1.f, -1.f);
#pragma unroll
        for (int hp = 1; hp < 16; hp <<= 1) {  // spans 2, 4, 8, 16: pairs e and e + span/2
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                if (e & hp) continue;
                const f32x2 x = b[e], y = b[e + hp];
                b[e] = add_f32x2(x, y);
                b[e + hp] = fma_f32x2(y, neg1, x);
            }
        }
        const float s32 = (q4 & 1) ? -1.f : 1.f, s64 = (q4 & 2) ? -1.f : 1.f;
        const f32x2 m32 = make_f32x2(s32, s32), m64 = make_f32x2(s64, s64);
#pragma unroll
        for (int e = 0; e < 16; ++e) {  // span 32: mine * (+-1) + the partner's
            float x, y;
            split_f32x2(b[e], x, y);
            const f32x2 o = make_f32x2(__shfl_xor_sync(0xffffffffu, x, 1), __shfl_xor_sync(0xffffffffu, y, 1));
            b[e] = fma_f32x2(b[e], m32, o);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {  // span 64
            float x, y;
            split_f32x2(b[e], x, y);
            const f32x2 o = make_f32x2(__shfl_xor_sync(0xffffffffu, x, 2), __shfl_xor_sync(0xffffffffu, y, 2));
            b[e] = fma_f32x2(b[e], m64, o);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) b[e] = make_f32x2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
    }
    float mx = 0.f;  // largest |x| (finite inputs)
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        float x, y;
        split_f32x2(b[e], x, y);
        mx = max3f(mx, fabsf(x), fabsf(y));
    }
    const int e = fp8_tile_exponent(fp8_block_max(__float_as_uint(mx), red, bad));
    if (bad) return false;  // a copy did not land: nothing is written
    after_max();            // every thread has read the staged tile
    if (threadIdx.x == 0) *exp_out = e;
    const float sc = fp8_pow2_neg(e);
    const f32x2 sc2 = make_f32x2(sc, sc);
    if (row < N) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + static_cast<size_t>(row) * 128 + q4 * 32);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t o[4];
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
                float x0, x1, x2, x3;
                split_f32x2(mul_f32x2(b[8 * k + 2 * e4], sc2), x0, x1);
                split_f32x2(mul_f32x2(b[8 * k + 2 * e4 + 1], sc2), x2, x3);
                o[e4] = pack_e4m3x4(x0, x1, x2, x3);
            }
            d4[k] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    return true;
}

// One 128-key tile of V, staged row-major in shared memory, rounded and written transposed: dst row
// c (dimension c) holds the tile's 128 keys at columns tile*128 ..; keys past N are zero. The tile
// is copied once more, into `sm` (rows of 136 halves, 16-byte aligned) with each 8-column chunk moved
// by an XOR with the key's 16-row group (chunk ^ ((row >> 4) & 7)). Thread t then reads the pair of
// dimensions 2 (t >> 3), + 1 over keys 16 (t mod 8) .. + 15 as 32-bit words: the eight key groups of
// a warp land in eight different bank groups.
constexpr int FP8P_VT_STRIDE = 136;
template <class AfterMax>
__device__ bool fp8_prep_v_tile(const uint8_t* stage, uint8_t* dstT, int32_t* exp_out, int N, int n_cols, int tile,
                                uint32_t* red, uint16_t (*sm)[FP8P_VT_STRIDE], bool bad, AfterMax after_max) {
    uint32_t mbits = 0;  // largest |V| as bf16 bits
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int idx = threadIdx.x + k * FP8P_THREADS;  // 16-byte chunk of the tile: row idx/16
        const int row = idx >> 4, c8 = ((idx & 15) ^ ((row >> 4) & 7)) * 8;
        const uint4 u = tile * 128 + row < N ? lds128(stage + idx * 16) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(&sm[row][c8]) = u;
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) mbits = max(mbits, max(w[q] & 0x7fffu, (w[q] >> 16) & 0x7fffu));
    }
    const int e = fp8_tile_exponent(fp8_block_max(mbits << 16, red, bad));  // (its barrier synchronises sm)
    if (bad) return false;
    after_max();  // every thread has read the staged tile
    if (threadIdx.x == 0) *exp_out = e;
    const float sc = fp8_pow2_neg(e);
    const f32x2 sc2 = make_f32x2(sc, sc);
    const int cp = threadIdx.x >> 3, kg = threadIdx.x & 7, k0 = kg * 16;  // dimensions 2cp, 2cp + 1
    // the word of dimensions 2cp, 2cp + 1 in row k0 + j: chunk cp / 4 moved by kg, word cp mod 4
    const uint32_t* wrow = reinterpret_cast<const uint32_t*>(&sm[k0][(((cp >> 2) ^ kg) << 3) + 2 * (cp & 3)]);
    uint32_t lo[4], hi[4];  // E4M3 of dimension 2cp (lo) and 2cp + 1 (hi), four keys per word
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float a[4], b[4];
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            const uint32_t w0 = wrow[(4 * q + u) * (FP8P_VT_STRIDE / 2)];
            const uint32_t w1 = wrow[(4 * q + u + 1) * (FP8P_VT_STRIDE / 2)];
            split_f32x2(mul_f32x2(make_f32x2(__uint_as_float(w0 << 16), __uint_as_float(w1 << 16)), sc2), a[u],
                        a[u + 1]);
            split_f32x2(mul_f32x2(make_f32x2(__uint_as_float(w0 & 0xffff0000u), __uint_as_float(w1 & 0xffff0000u)),
                                  sc2),
                        b[u], b[u + 1]);
        }
        lo[q] = pack_e4m3x4(a[0], a[1], a[2], a[3]);
        hi[q] = pack_e4m3x4(b[0], b[1], b[2], b[3]);
    }
    uint8_t* d0 = dstT + static_cast<size_t>(2 * cp) * n_cols + tile * 128 + k0;
    *reinterpret_cast<uint4*>(d0) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(d0 + n_cols) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    return true;
}

__global__ void __launch_bounds__(FP8P_THREADS, FP8P_BLOCKS_PER_SM)
    fp8_prep_kernel(const Fp8PrepParams p, const PlanParams pl) {
    grid_dep_launch_dependents();
    extern __shared__ __align__(128) uint8_t fp8p_ring[];
    __shared__ __align__(8) uint64_t full[FP8P_STAGES];
    __shared__ uint32_t red[2][FP8P_THREADS / 32];  // block-maximum slots, alternating by tile
    __shared__ __align__(16) uint16_t vt[128][FP8P_VT_STRIDE];
    __shared__ __align__(16) uint32_t sgn[4 * 16];  // sign bits of the rotation as bf16-pair XOR masks
    const int G = static_cast<int>(gridDim.x) - 1;  // tile blocks; the last block plans the schedule
    if (static_cast<int>(blockIdx.x) == G) {
        plan_block(pl);
        return;
    }
    const int per_y = p.n_ktiles;
    const int T = per_y * (p.heads_q + 2 * p.heads_kv);  // tiles: Q heads, K heads, V heads (< 2^31)
    const size_t head_bytes = static_cast<size_t>(p.N) * 256;      // one bf16 [N, 128] slab
    if (threadIdx.x == 0) {
        for (int st = 0; st < FP8P_STAGES; ++st) mbar_init(&full[st], 1);
        fence_mbar_init();
    }
    if (p.signs && threadIdx.x < 64) {  // word e of quarter q: elements 32q + 2e (bit 15), + 1 (bit 31)
        const int el = (threadIdx.x >> 4) * 32 + 2 * (threadIdx.x & 15);
        sgn[threadIdx.x] = (__ldg(p.signs + el) < 0 ? 0x8000u : 0u) | (__ldg(p.signs + el + 1) < 0 ? 0x80000000u : 0u);
    }
    __syncthreads();
    const uint32_t* sgn_tab = p.signs ? sgn : nullptr;
    // tile i of the list into ring stage st (one thread)
    auto issue = [&](int i, int st) {
        const int y = i / per_y;
        const int tile = i - y * per_y;
        const uint8_t* src = y < p.heads_q ? static_cast<const uint8_t*>(p.Q) + static_cast<size_t>(y) * head_bytes
                           : y < p.heads_q + p.heads_kv
                               ? static_cast<const uint8_t*>(p.K) + static_cast<size_t>(y - p.heads_q) * head_bytes
                               : static_cast<const uint8_t*>(p.V) + static_cast<size_t>(y - p.heads_q - p.heads_kv) * head_bytes;
        const uint32_t bytes = static_cast<uint32_t>(min(128, p.N - tile * 128)) * 256u;
        mbar_arrive_expect_tx(&full[st], bytes);
        bulk_load(fp8p_ring + st * FP8P_TILE_BYTES, src + static_cast<size_t>(tile) * 128 * 256, bytes, &full[st]);
    };
    if (threadIdx.x == 0)
        for (int st = 0; st < FP8P_STAGES; ++st) {
            const int i = static_cast<int>(blockIdx.x) + st * G;
            if (i < T) issue(i, st);
        }
    const size_t head_elems = static_cast<size_t>(p.N) * 128;
    const int n_cols = p.n_ktiles * 128;
    volatile int never = 0;
    int k = 0;
    bool ok = true;
    bool prev_v = false;  // the block's previous tile was a V tile (its transposed reads of vt)
    for (int i = static_cast<int>(blockIdx.x); i < T; i += G, ++k) {
        const int st = k % FP8P_STAGES;
        const bool got = mbar_wait(&full[st], (k / FP8P_STAGES) & 1, p.wait_limit_ns, &never);
        const int y = i / per_y;
        const int tile = i - y * per_y;
        const bool is_v = y >= p.heads_q + p.heads_kv;
        // A V tile overwrites vt, which the previous V tile's threads may still be reading: wait for
        // them. Otherwise the block maximum's barrier orders the tiles (the reduction slots alternate).
        // Whether every copy landed is decided block-wide at that barrier.
        if (is_v && prev_v) __syncthreads();
        prev_v = is_v;
        const uint8_t* stage = fp8p_ring + st * FP8P_TILE_BYTES;
        uint32_t* rd = red[k & 1];
        // once every thread has read the staged tile, the next tile of the block may land in its stage
        auto after_max = [&]() {
            if (threadIdx.x == 0 && i + FP8P_STAGES * G < T) issue(i + FP8P_STAGES * G, st);
        };
        if (y < p.heads_q) {
            ok = fp8_prep_qk_tile(stage, p.Q8 + static_cast<size_t>(y) * head_elems,
                                  p.q_exp + static_cast<size_t>(y) * per_y + tile, sgn_tab, p.N, tile, rd, !got,
                                  after_max);
        } else if (!is_v) {
            const int h = y - p.heads_q;
            ok = fp8_prep_qk_tile(stage, p.K8 + static_cast<size_t>(h) * head_elems,
                                  p.k_exp + static_cast<size_t>(h) * per_y + tile, sgn_tab, p.N, tile, rd, !got,
                                  after_max);
        } else {
            const int h = y - p.heads_q - p.heads_kv;
            ok = fp8_prep_v_tile(stage, p.V8T + static_cast<size_t>(h) * 128 * n_cols,
                                 p.v_exp + static_cast<size_t>(h) * per_y + tile, p.N, n_cols, tile, rd, vt, !got,
                                 after_max);
        }
        if (!ok) break;  // block-uniform
    }
    if (!ok && threadIdx.x == 0) {
        // a copy that never landed: record it, then wait (bounded) for the copies still in flight so
        // that none writes shared memory after the block has exited
        atomicOr(&g_attn_error, ERRBIT_TIMEOUT | ERRBIT_WAIT_KV);
        for (int kk = k; kk < k + FP8P_STAGES; ++kk)
            if (static_cast<int>(blockIdx.x) + kk * G < T)
                (void)mbar_wait(&full[kk % FP8P_STAGES], (kk / FP8P_STAGES) & 1, p.wait_limit_ns, &never);
    }
}

cudaError_t launch_fp8_prep(const Fp8PrepParams& p, const PlanParams& plan, cudaStream_t stream) {
    if (p.d != 128 || p.sms <= 0) return cudaErrorInvalidValue;
    static std::atomic<int> ready[64];  // once per device: the shared-memory opt-in
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || ready[dev].load(std::memory_order_acquire) == 0) {
        e = cudaFuncSetAttribute(fp8_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FP8P_SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) ready[dev].store(1, std::memory_order_release);
    }
    const long long T = static_cast<long long>(p.n_ktiles) * (p.heads_q + 2LL * p.heads_kv);
    if (T >= (1LL << 30)) return cudaErrorInvalidConfiguration;  // tile indices stay in int
    const long long G = std::min<long long>(T, static_cast<long long>(FP8P_BLOCKS_PER_SM) * p.sms);
    if (G < 1) return cudaErrorInvalidValue;
    fp8_prep_kernel<<<static_cast<unsigned>(G + 1), FP8P_THREADS, FP8P_SMEM, stream>>>(p, plan);
    return cudaGetLastError();
}

template <int D, bool OUT_BF16, int VAR>
static cudaError_t launch_tc_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const CUtensorMap& tmO, const TcParams& p, cudaStream_t stream) {
    constexpr bool FP8 = VAR == 1;
    auto kern = attn_fwd_tc_kernel<D, OUT_BF16, VAR>;
    cudaError_t e = cudaSuccess;
    // once per device: shared-memory opt-in and the register check
    static std::atomic<int> ready[64];
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || ready[dev].load(std::memory_order_acquire) == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, FP8>::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        // The register split inside the kernel assumes exactly LAUNCH_REGS registers per thread at
        // launch; with fewer, the softmax warpgroups' increase could never be granted.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != LAUNCH_REGS) return cudaErrorInvalidKernelImage;
        if (dev >= 0 && dev < 64) ready[dev].store(1, std::memory_order_release);
    }
    if (p.plan.G <= 0 || p.plan.G > SCHED_MAX_CTAS) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.plan.G));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = Cfg<D, FP8>::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    // Programmatic dependent launch: the kernel may start while the pre-pass before it still runs (it
    // waits for the pre-pass's output in the roles that read it).
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    // A plan that splits units needs every CTA resident at once (an owner CTA waits, bounded, for the
    // partial results of the CTAs after it): cooperative launch. Whole-unit plans need no such guarantee.
    if (p.plan.sk) {
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, tmQ, tmK, tmV, tmO, p);
    if (e != cudaSuccess && na == 2) {
        // a driver that refuses the combination: launch cooperatively without the early start
        (void)cudaGetLastError();
        cfg.attrs = attr + 1;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, tmQ, tmK, tmV, tmO, p);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_attn_tc(int d, bool out_bf16, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV16, const CUtensorMap& tmO, const TcParams& p, cudaStream_t stream) {
    if (d == 128) return out_bf16 ? launch_tc_t<128, true, 0>(tmQ, tmK, tmV16, tmO, p, stream)
                                  : launch_tc_t<128, false, 0>(tmQ, tmK, tmV16, tmO, p, stream);
    if (d == 64) return out_bf16 ? launch_tc_t<64, true, 0>(tmQ, tmK, tmV16, tmO, p, stream)
                                 : launch_tc_t<64, false, 0>(tmQ, tmK, tmV16, tmO, p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_tc_ex(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV16,
                              const CUtensorMap& tmO, const TcParams& p, cudaStream_t stream) {
    if (d == 128) return launch_tc_t<128, false, 2>(tmQ, tmK, tmV16, tmO, p, stream);
    if (d == 64) return launch_tc_t<64, false, 2>(tmQ, tmK, tmV16, tmO, p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_tc_fp8(const CUtensorMap& tmQ8, const CUtensorMap& tmK8, const CUtensorMap& tmVT8,
                               const CUtensorMap& tmO, const TcParams& p, cudaStream_t stream) {
    return launch_tc_t<128, false, 1>(tmQ8, tmK8, tmVT8, tmO, p, stream);
}

// Line length of the worst case (every kv_len = N): the schedule needs it below 2^31.
long long plan_max_steps(int B, int H, int N, int causal) {
    const int n_pairs = (N + 2 * BLOCK_M - 1) / (2 * BLOCK_M);
    return static_cast<long long>(B) * H * line_prefix(n_pairs, key_tiles(N), N, causal);
}

SchedPlan make_plan(int B, int H, int N, int causal, bool has_kv_len, int sms, int mode) {
    SchedPlan p{};
    p.B = B;
    p.H = H;
    p.N = N;
    p.causal = causal;
    p.n_pairs = (N + 2 * BLOCK_M - 1) / (2 * BLOCK_M);
    const long long units = static_cast<long long>(B) * H * p.n_pairs;
    p.units = static_cast<int>(units);
    const int nb = key_tiles(N);
    const long long w_max = static_cast<long long>(B) * H * line_prefix(p.n_pairs, nb, N, causal);
    const long long g_cap = sms < SCHED_MAX_CTAS ? sms : SCHED_MAX_CTAS;
    // Two plans, compared by the key steps plus unit overheads of the busiest CTA (kv_len counts as N:
    // an upper bound). Stream-K: G CTAs share the line evenly, units cut by chunk boundaries pay the
    // merge penalty.
    long long g = g_cap;
    const long long g_steps = (w_max + SCHED_MIN_STEPS - 1) / SCHED_MIN_STEPS;
    if (g_steps < g) g = g_steps;
    if (g < 1) g = 1;
    const long long t_stream = (w_max + g - 1) / g + SCHED_SPLIT_PENALTY;
    // Whole units in rounds (unit r * G + c on CTA c): with equal costs every CTA runs ceil(units / G)
    // of them; with unequal costs (causal or kv_len) only one round is considered, bounded by the
    // costliest unit.
    const bool uniform = !causal && !has_kv_len;
    long long max_cost = 1;
    for (int pr = 0; pr < p.n_pairs; ++pr) {
        const long long c = pair_cost(pr, nb, N, causal);
        if (c > max_cost) max_cost = c;
    }
    const long long rounds = (units + g_cap - 1) / g_cap;
    const long long t_whole =
        uniform ? rounds * (nb + SCHED_UNIT_OVERHEAD) : (rounds == 1 ? max_cost + SCHED_UNIT_OVERHEAD : -1);
    if (mode == 1 || (mode == 0 && t_whole >= 0 && t_whole < t_stream)) {
        p.R_dp = static_cast<int>(rounds);
        p.G = static_cast<int>((units + rounds - 1) / rounds);  // the fewest CTAs for that many rounds
        p.sk = 0;
        p.S0 = static_cast<int>(w_max);  // unused: no stream-K part
        return p;
    }
    p.G = static_cast<int>(g);
    p.sk = 1;
    // data-parallel rounds only when every unit costs the same; the last one or two rounds' worth of
    // units go to the balanced stream-K part
    const long long r = uniform ? units / g - 1 : 0;
    p.R_dp = r > 0 ? static_cast<int>(r) : 0;
    p.S0 = static_cast<int>(static_cast<long long>(p.R_dp) * p.G * (nb + SCHED_UNIT_OVERHEAD));
    return p;
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
