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
    ERRBIT_WAIT_PART = 256u,    // an owner CTA waited for another CTA's partial result
};

// ---------------------------------------------------------------------------------------------
// Work schedule of the persistent tensor-core kernel (host and device code share it).
//
// A work unit is (b, h, pair): 256 query rows (two 128-row query tiles) of one head. Its cost is the
// number of 128-key steps it needs: the larger of its two tiles' key-tile counts below
// min(kv_len[b], causal limit), and at least 1 (a unit without any valid key still writes O = 0,
// LSE = -inf). Units lie on a line in (b, h, pair) order; unit u covers [off(u), off(u) + OVH +
// cost(u)): OVH = SCHED_UNIT_OVERHEAD positions stand for the fixed time of a segment (its Q load,
// first S and epilogue), then one position per key step. CTA c of G first runs R_dp data-parallel
// rounds (unit r*G + c in round r, while that unit exists), then, when the plan has a stream-K part
// (sk = 1), one contiguous chunk of the rest of the line, [S0 + (W - S0) c / G, S0 + (W - S0) (c + 1) /
// G): equal chunks of the line give every CTA the same key steps plus segment overheads, so a CTA
// with many short units gets fewer steps. A chunk boundary inside a unit's overhead belongs to the
// unit's start (the unit goes whole to the later chunk); a unit that a boundary cuts inside its key
// steps is computed in pieces over disjoint key ranges. The piece that holds the unit's first key step (the owner) is the
// last segment of its CTA; the other pieces are the first segments of the following CTAs' chunks,
// which write their partial results (unnormalised O, running max m, running sum l) to a slot of
// their own. The owner merges them with the softmax merge rule: m = max(m_a, m_b),
// O = O_a 2^(m_a - m) + O_b 2^(m_b - m), l = l_a 2^(m_a - m) + l_b 2^(m_b - m), then O / l.
// ---------------------------------------------------------------------------------------------
constexpr int SCHED_MAX_CTAS = 160;  // partial-result slots reserved in the workspace
constexpr int SCHED_MIN_STEPS = 2;   // the CTA count is capped so that chunks hold at least this many steps
// Extra time of a stream-K plan, in key steps: its CTAs run more segments (each with a Q load and an
// epilogue) and the owners of split units wait for and merge the other pieces' partial results.
// Measured on B300 against whole-unit plans (B1 H16 d128, N = 512 ... 16384, causal and not): splitting
// lost by 6-10 steps' worth on small problems and won by about 30 steps at N = 8192; the plan splits
// units only when that saves more than this.
constexpr int SCHED_SPLIT_PENALTY = 10;
// Line positions per unit before its key steps: a segment's fixed time (Q load, first S, epilogue and
// the next segment's start) measured at about two key steps' worth on B300 (B1 H16 N8192 d128).
constexpr int SCHED_UNIT_OVERHEAD = 2;

enum : int { SEG_COMPLETE = 0, SEG_OWNER = 1, SEG_WRITER = 2 };

__host__ __device__ inline int key_tiles(int kv_valid) { return (kv_valid + 127) / 128; }

// Sum of the costs of pairs [0, P) of one head in a batch with nb valid key tiles.
__host__ __device__ inline long long pair_prefix(int P, int nb, int N, int causal) {
    if (nb <= 0) return P;  // units without keys cost 1 each
    if (!causal) return static_cast<long long>(P) * nb;
    const int n_full = N > 128 ? (N - 129) / 256 + 1 : 0;  // pairs whose second tile exists
    const int Pf = P < n_full ? P : n_full;
    const int half = nb / 2;
    const long long k = Pf < half ? Pf : half;  // pairs p with 2p + 2 <= nb cost 2p + 2
    long long s = k * (k + 1) + static_cast<long long>(Pf - k) * nb;  // the rest cost nb
    if (P > n_full) s += (nb < 2 * n_full + 1 ? nb : 2 * n_full + 1);  // last pair: its first tile only
    return s;
}

__host__ __device__ inline int pair_cost(int pair, int nb, int N, int causal) {
    return static_cast<int>(pair_prefix(pair + 1, nb, N, causal) - pair_prefix(pair, nb, N, causal));
}

// Line length of pairs [0, P) of one head: their key steps and the overhead of each unit.
__host__ __device__ inline long long line_prefix(int P, int nb, int N, int causal) {
    return pair_prefix(P, nb, N, causal) + static_cast<long long>(SCHED_UNIT_OVERHEAD) * P;
}

struct SchedPlan {
    int B, H, N, n_pairs, causal;
    int units;      // B * H * n_pairs work units
    int G;          // persistent CTAs
    int R_dp;       // data-parallel rounds (the last one may be partial: units past `units` do not exist)
    int sk;         // 1: a stream-K part follows the rounds; 0: every unit is whole (no partial results)
    int S0;         // line offset where the stream-K part starts (the whole line is below 2^31)
};

struct Segment {
    int b, h, pair;
    int k0, k1;          // key steps [k0, k1) of the unit
    int cost;            // the unit's cost
    int unit_end;        // line offset just past the unit (stream-K segments; -1 in the rounds)
    int kind;            // SEG_COMPLETE, SEG_OWNER or SEG_WRITER
};

__host__ __device__ inline int sched_chunk_start(const SchedPlan& p, int W, int c) {
    return p.S0 + static_cast<int>(static_cast<long long>(W - p.S0) * c / p.G);
}

// Enumerates the segments of CTA `cta` in the order it runs them (walk_init once, then walk_next
// until it returns false). Tab provides
//   int nb(int b)              valid key tiles of batch b
//   long long boff(int b)      line offset of batch b's first unit, b = 0..B (boff(B) = W < 2^31)
// The state is a plain struct so that the kernel can keep it in shared memory, out of the registers
// of the roles that walk it.
struct WalkState {
    int W, round, sk_started, pos, chunk_end, unit_off, b, h, pair;
};

template <class Tab>
__host__ __device__ inline void walk_init(WalkState& w, const Tab& t, const SchedPlan& p) {
    w.W = static_cast<int>(t.boff(p.B));
    w.round = 0;
    w.sk_started = 0;
    w.pos = w.chunk_end = w.unit_off = 0;
    w.b = w.h = w.pair = 0;
}

template <class Tab>
__host__ __device__ inline int walk_head_cost(const Tab& t, const SchedPlan& p, int b) {
    return static_cast<int>(line_prefix(p.n_pairs, t.nb(b), p.N, p.causal));
}

// b, h, pair and unit_off of the unit that contains line position x (boff(0) <= x < W)
template <class Tab>
__host__ __device__ inline void walk_locate(WalkState& w, const Tab& t, const SchedPlan& p, int x) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {  // largest b with boff(b) <= x
        const int mid = (lo + hi + 1) / 2;
        if (t.boff(mid) <= x) lo = mid;
        else hi = mid - 1;
    }
    w.b = lo;
    const int nb = t.nb(lo);
    const int hc = walk_head_cost(t, p, lo);
    const int rem = x - static_cast<int>(t.boff(lo));
    w.h = rem / hc;
    const int r2 = rem - w.h * hc;
    int plo = 0, phi = p.n_pairs - 1;
    while (plo < phi) {  // largest pair with line_prefix(pair) <= r2
        const int mid = (plo + phi + 1) / 2;
        if (line_prefix(mid, nb, p.N, p.causal) <= r2) plo = mid;
        else phi = mid - 1;
    }
    w.pair = plo;
    w.unit_off = static_cast<int>(t.boff(lo)) + w.h * hc + static_cast<int>(line_prefix(plo, nb, p.N, p.causal));
}

template <class Tab>
__host__ __device__ inline bool walk_next(WalkState& w, const Tab& t, const SchedPlan& p, int cta, Segment& s) {
    const long long u_dp = static_cast<long long>(w.round) * p.G + cta;
    if (w.round < p.R_dp && u_dp < p.units) {
        // 32-bit arithmetic: units < 2^31 (every unit costs at least one step of a line below 2^31)
        const unsigned u = static_cast<unsigned>(u_dp);
        ++w.round;
        const unsigned np = static_cast<unsigned>(p.n_pairs);
        const unsigned bh = u / np;
        s.pair = static_cast<int>(u - bh * np);
        s.b = static_cast<int>(bh / static_cast<unsigned>(p.H));
        s.h = static_cast<int>(bh - static_cast<unsigned>(s.b) * static_cast<unsigned>(p.H));
        const int nb = t.nb(s.b);
        s.cost = pair_cost(s.pair, nb, p.N, p.causal);
        s.k0 = 0;
        s.k1 = s.cost;
        s.unit_end = -1;  // read by owners of split units only; a round's unit is whole
        s.kind = SEG_COMPLETE;
        return true;
    }
    w.round = p.R_dp;  // a partial last round ends the rounds of the CTAs past its end
    if (!p.sk) return false;
    if (!w.sk_started) {
        w.sk_started = 1;
        w.pos = sched_chunk_start(p, w.W, cta);
        w.chunk_end = sched_chunk_start(p, w.W, cta + 1);
        if (w.pos < w.chunk_end) walk_locate(w, t, p, w.pos);
    }
    if (w.pos >= w.chunk_end) return false;
    const int cost = pair_cost(w.pair, t.nb(w.b), p.N, p.causal);
    const int step0 = w.unit_off + SCHED_UNIT_OVERHEAD;  // line position of the unit's first key step
    const int end = step0 + cost;
    const int k1 = (w.chunk_end < end ? w.chunk_end : end) - step0;
    if (k1 <= 0) return false;  // the chunk ends inside this unit's overhead: the next chunk takes it
    s.b = w.b;
    s.h = w.h;
    s.pair = w.pair;
    s.cost = cost;
    s.k0 = w.pos > step0 ? w.pos - step0 : 0;
    s.k1 = k1;
    s.unit_end = end;
    s.kind = s.k0 > 0 ? SEG_WRITER : (s.k1 < cost ? SEG_OWNER : SEG_COMPLETE);
    w.pos = step0 + k1;
    w.unit_off = end;
    if (++w.pair == p.n_pairs) {
        w.pair = 0;
        if (++w.h == p.H) {
            w.h = 0;
            ++w.b;
        }
    }
    return true;
}

// Host-side table over arrays (the schedule check of the test hook).
struct HostSchedTab {
    const int* nb_;
    const long long* boff_;
    __host__ __device__ int nb(int b) const { return nb_[b]; }
    __host__ __device__ long long boff(int b) const { return boff_[b]; }
};

struct TcParams {
    void* O;                  // [B,H,N,d] fp32 or bf16
    float* LSE;               // [B,H,N] or nullptr
    const int32_t* kv_len;    // [B] or nullptr
    const int32_t* v_exp;     // [B*H_kv][n_ktiles] exponent e of each 128-key tile of the fp16 V copy
    int n_ktiles;             // ceil(N / 128)
    const long long* boff;    // [B+1] line offset of each batch's first unit (plan pass)
    float* part;              // partial results [G][2][D + 2][128] (O columns, then m, then l; row fastest)
    unsigned int* flags;      // [G][2][4] partial-result ready flags (per CTA, tile, warp), zeroed by the plan pass
    SchedPlan plan;
    int H_kv;
    int group;                // H / H_kv
    float scale_log2;         // scale * log2(e)
    unsigned long long wait_limit_ns;
    int debug_skip_kv_load;
    // fp8 path only: power-of-two exponents of the E4M3 copies of Q ([B*H][n_ktiles]) and K
    // ([B*H_kv][n_ktiles]); a tile's stored values times 2^e are the (rotated) inputs
    const int32_t* q_exp;
    const int32_t* k_exp;
    // bias + dropout variant only: additive bf16 bias (element (b, h, i, j) at
    // bias[b * bias_sb + h * bias_sh + i * bias_sr + j], strides in elements, multiples of 8) or
    // nullptr; dropout threshold t (drop iff the 16-bit draw < t; 0 = no dropout), Philox key and
    // counter word 3, and the inverse keep probability 65536 / (65536 - t)
    const uint16_t* bias;
    long long bias_sb, bias_sh, bias_sr;
    uint32_t drop_t, seed_lo, seed_hi, rng_offset;
    // the generator's ten round keys (k0 + r W0, k1 + r W1 for r = 0..9), the same for every draw of a
    // launch: computed once on the host, read by the kernel from its parameter space
    uint32_t round_key[2][10];
    float keep_scale;
};

// fp8 pre-pass: rotate Q and K (optional), round Q, K, V to E4M3 per 128-row tile, V transposed.
struct Fp8PrepParams {
    const void* Q;            // bf16 [B*H][N][d]
    const void* K;            // bf16 [B*H_kv][N][d]
    const void* V;            // bf16 [B*H_kv][N][d]
    uint8_t* Q8;              // E4M3 [B*H][N][d]
    uint8_t* K8;              // E4M3 [B*H_kv][N][d]
    uint8_t* V8T;             // E4M3 [B*H_kv][d][n_ktiles * 128] (keys past N are zero)
    int32_t* q_exp;           // [B*H][n_ktiles]
    int32_t* k_exp;           // [B*H_kv][n_ktiles]
    int32_t* v_exp;           // [B*H_kv][n_ktiles]
    const int8_t* signs;      // d values +-1 (rotation), or nullptr (no rotation)
    int N, d, n_ktiles, heads_q, heads_kv;
    int sms;                  // SMs of the device (the pre-pass runs two blocks on each)
    uint64_t wait_limit_ns;   // bound of the waits for its copies
};

struct PlanParams {
    const int32_t* kv_len;
    long long* boff;          // [B+1]
    unsigned int* flags;      // [8 * SCHED_MAX_CTAS]
    int B, H, N, n_pairs, causal;
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
    uint64_t wait_limit_ns;   // bound of the wait for the staged key rows
};

// V (bf16 [heads, N, d]) -> fp16 copy, one 128-row key tile at a time: tile j of head z is stored as
// V * 2^-e[z][j], with e the smallest non-negative exponent that keeps |V| * 2^-e below 2^15.
struct VPrepParams {
    const void* V;            // bf16 [heads, N, d]
    void* V16;                // fp16 [heads, N, d]
    int32_t* v_exp;           // [heads, n_ktiles]
    int N, d, n_ktiles, heads;
};

cudaError_t launch_vprep(const VPrepParams& p, const PlanParams& plan, cudaStream_t stream);
cudaError_t launch_fp8_prep(const Fp8PrepParams& p, const PlanParams& plan, cudaStream_t stream);
// fp8 forward (d = 128, fp32 output): maps over Q8, K8 (box 128 x 128 bytes) and V8T (keys inner)
// bias + dropout variant (bf16 inputs, fp32 output, d in {64, 128})
cudaError_t launch_attn_tc_ex(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV16,
                              const CUtensorMap& tmO, const TcParams& p, cudaStream_t stream);
cudaError_t launch_attn_tc_fp8(const CUtensorMap& tmQ8, const CUtensorMap& tmK8, const CUtensorMap& tmVT8,
                               const CUtensorMap& tmO, const TcParams& p, cudaStream_t stream);
// tmO: fp32 output map (box 32 columns x 32 rows, 128-byte swizzle); unused for bf16 output.
cudaError_t launch_attn_tc(int d, bool out_bf16, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV16, const CUtensorMap& tmO, const TcParams& p, cudaStream_t stream);

// Persistent-CTA plan for these sizes on a device with `sms` SMs (kv_len given or not).
// mode: 0 = the cheaper plan by the cost model, 1 = whole units in rounds, 2 = stream-K (test hook)
SchedPlan make_plan(int B, int H, int N, int causal, bool has_kv_len, int sms, int mode = 0);
long long plan_max_steps(int B, int H, int N, int causal);
cudaError_t launch_attn_f32(int d, const F32Params& p, cudaStream_t stream);

cudaError_t launch_attn_merge(const float* O_parts, const float* LSE_parts, int n_parts, long long rows, int d,
                              float* O, float* LSE, cudaStream_t stream);

// Backward pass (bf16 inputs): see attn_bwd.cu.
struct BwdParams {
    float* dQ;                // [B,H,N,d] fp32 (cleared by the prep kernel, reduce-added into)
    float* dK;                // [B,H_kv,N,d] fp32
    float* dV;                // [B,H_kv,N,d] fp32
    const float* lse2;        // [B*H][n_qt*128] LSE * log2(e) (+inf on padding rows)
    const float* dvec;        // [B*H][n_qt*128] rowsum(dO * O)
    const int32_t* kv_len;    // [B] or nullptr
    int B, H, H_kv, N, group, causal, n_qt;
    float scale, scale_log2;
    unsigned long long wait_limit_ns;
};

struct BwdPrepParams {
    const void* dO;           // bf16 [B,H,N,d]
    const float* O;           // fp32 [B,H,N,d]
    const float* LSE;         // fp32 [B,H,N]
    float* lse2;
    float* dvec;
    float* dQ;
    int rows, N, d, NQP;      // rows = B*H, NQP = n_qt * 128
};

cudaError_t launch_attn_bwd(int d, const BwdPrepParams& prep, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmDO, const CUtensorMap& tmDQ,
                            const BwdParams& p, cudaStream_t stream);
cudaError_t read_and_clear_bwd_error(uint32_t* out);
cudaError_t read_and_clear_f32_error(uint32_t* out);

// Device error word of the current device: read and clear (synchronous on `stream`).
cudaError_t read_and_clear_error(uint32_t* out, cudaStream_t stream);

}  // namespace attn_impl
