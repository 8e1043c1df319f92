// C ABI front end of libattn.so: argument validation, workspace layout, TMA tensor maps, dispatch.
// The operation, layouts and error conventions are documented in include/attn.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace {

constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;  // 1 s
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int> g_skip_kv_load{0};
std::atomic<int> g_plan_mode{0};
std::atomic<uint32_t> g_last_error_bits{0};
std::atomic<cudaEvent_t> g_ev_start{nullptr};
std::atomic<cudaEvent_t> g_ev_stop{nullptr};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: fp16 copy of V | per-tile V exponents | schedule batch offsets | partial-result flags |
// partial results of split work units (each piece 256-byte aligned).
struct WorkspaceLayout {
    size_t v16 = 0, vexp = 0, boff = 0, flags = 0, part = 0, total = 0;
    int n_ktiles = 0;
};

bool workspace_layout(int B, int H_kv, int N, int d, WorkspaceLayout* w) {
    const long long elems_per_head = static_cast<long long>(N) * d;
    const long long heads = static_cast<long long>(B) * H_kv;
    w->n_ktiles = (N + 127) / 128;
    w->v16 = 0;
    w->vexp = round_up(static_cast<size_t>(heads * elems_per_head) * 2, 256);
    w->boff = w->vexp + round_up(static_cast<size_t>(heads) * w->n_ktiles * sizeof(int32_t), 256);
    w->flags = w->boff + round_up(static_cast<size_t>(B + 1) * sizeof(long long), 256);
    w->part = w->flags + round_up(8 * attn_impl::SCHED_MAX_CTAS * sizeof(unsigned int), 256);
    w->total = w->part + round_up(static_cast<size_t>(attn_impl::SCHED_MAX_CTAS) * 2 * (d + 3) * 128 * sizeof(float), 256);
    return heads < 65535;  // the pre-pass grid has heads + 1 rows of blocks
}

// fp8 path: E4M3 copies of Q, K and V^T, their tile exponents, then the schedule's buffers.
struct Fp8Layout {
    size_t q8 = 0, k8 = 0, vt8 = 0, qexp = 0, kexp = 0, vexp = 0, boff = 0, flags = 0, part = 0, total = 0;
    int n_ktiles = 0;
};

bool fp8_layout(int B, int H, int H_kv, int N, int d, Fp8Layout* w) {
    const size_t hq = static_cast<size_t>(B) * H, hkv = static_cast<size_t>(B) * H_kv;
    w->n_ktiles = (N + 127) / 128;
    const size_t npad = static_cast<size_t>(w->n_ktiles) * 128;
    w->q8 = 0;
    w->k8 = round_up(hq * N * d, 256);
    w->vt8 = w->k8 + round_up(hkv * N * d, 256);
    w->qexp = w->vt8 + round_up(hkv * d * npad, 256);
    w->kexp = w->qexp + round_up(hq * w->n_ktiles * sizeof(int32_t), 256);
    w->vexp = w->kexp + round_up(hkv * w->n_ktiles * sizeof(int32_t), 256);
    w->boff = w->vexp + round_up(hkv * w->n_ktiles * sizeof(int32_t), 256);
    w->flags = w->boff + round_up(static_cast<size_t>(B + 1) * sizeof(long long), 256);
    w->part = w->flags + round_up(8 * attn_impl::SCHED_MAX_CTAS * sizeof(unsigned int), 256);
    w->total = w->part + round_up(static_cast<size_t>(attn_impl::SCHED_MAX_CTAS) * 2 * (d + 3) * 128 * sizeof(float), 256);
    return hq + 2 * hkv + 1 <= 65535;  // rows of the pre-pass grid
}

// SM count of the current device (cached per device).
int device_sms() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
    if (dev < 64) {
        const int c = cache[dev].load();
        if (c > 0) return c;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return -1;
    if (dev < 64) cache[dev].store(sms);
    return sms;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 3-D map over [slabs, rows, d] 16-bit values: box of 64 columns x 128 rows, 128-byte swizzle,
// rows past `rows` in a slab read as zero.
bool encode_rows_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int d, int rows, long long slabs,
                     unsigned box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(slabs)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows) * d * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map over the fp32 output [slabs, rows, d]: box of 32 columns x 32 rows, 128-byte swizzle
// (the layout the epilogue stages rows in); rows past `rows` are not written by stores.
bool encode_out_map(CUtensorMap* m, void* base, int d, int rows, long long slabs, unsigned box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(slabs)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(rows) * d * 4};
    cuuint32_t box[3] = {32, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map over [slabs, rows, inner] bytes (E4M3): box of 128 bytes x 128 rows, 128-byte swizzle, rows
// past `rows` read as zero.
bool encode_u8_map(CUtensorMap* m, const void* base, int inner, int rows, long long slabs) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(slabs)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows) * inner};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor maps depend only on (base address, element type, d, rows, slabs, kind), so a small cache
// keyed on those saves re-encoding them for buffers used again (the common case).
struct MapKey {
    const void* base;
    int kind, d, rows;
    long long slabs;
    bool operator==(const MapKey& o) const {
        return base == o.base && kind == o.kind && d == o.d && rows == o.rows && slabs == o.slabs;
    }
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool used;
};
constexpr int kMapCache = 32;
MapEntry g_map_cache[kMapCache];
int g_map_next = 0;
std::mutex g_map_mutex;

// MAP_Q64_BF16: bf16 rows in boxes of 64 columns x 64 rows; MAP_O16_F32: fp32 boxes of 32 columns x 16
// rows (the d = 128 backward's query tiles and dQ reductions); the others as described above.
enum { MAP_Q_BF16 = 0, MAP_K_BF16 = 1, MAP_V_F16 = 2, MAP_O_F32 = 3, MAP_U8 = 4, MAP_Q64_BF16 = 5, MAP_O16_F32 = 6 };

bool encode_rows_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int d, int rows, long long slabs,
                     unsigned box_rows);
bool encode_out_map(CUtensorMap* m, void* base, int d, int rows, long long slabs, unsigned box_rows);
bool encode_u8_map(CUtensorMap* m, const void* base, int inner, int rows, long long slabs);

bool get_map(CUtensorMap* m, int kind, const void* base, int d, int rows, long long slabs) {
    const MapKey key{base, kind, d, rows, slabs};
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        for (int i = 0; i < kMapCache; ++i)
            if (g_map_cache[i].used && g_map_cache[i].key == key) {
                *m = g_map_cache[i].map;
                return true;
            }
    }
    bool ok = false;
    if (kind == MAP_O_F32 || kind == MAP_O16_F32)
        ok = encode_out_map(m, const_cast<void*>(base), d, rows, slabs, kind == MAP_O16_F32 ? 16 : 32);
    else if (kind == MAP_U8) ok = encode_u8_map(m, base, d, rows, slabs);
    else ok = encode_rows_map(m, base, kind == MAP_V_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              d, rows, slabs, kind == MAP_Q64_BF16 ? 64 : 128);
    if (!ok) return false;
    std::lock_guard<std::mutex> lock(g_map_mutex);
    MapEntry& e = g_map_cache[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
    e.key = key;
    e.map = *m;
    e.used = true;
    return true;
}

bool sizes_ok(int B, int H, int H_kv, int N, int d) {
    if (B <= 0 || H <= 0 || H_kv <= 0 || N <= 0) return false;
    if (H % H_kv != 0) return false;
    if (d != 64 && d != 128) return false;
    if (static_cast<long long>(B) * H > 0x7fffffffLL / 2) return false;
    return true;
}

// bf16 inputs on the tensor-core path (attn_fwd and attn_fwd_ex): V -> fp16 pre-pass, then the
// persistent attention kernel; `ex` (bias + dropout) selects that variant of the kernel.
attn_status run_bf16_path(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int H_kv,
                          int N, int d, float scale, int causal, const int32_t* kv_len, attn_dtype out_dtype,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream,
                          const attn_impl::TcParams* ex) {
    WorkspaceLayout w;
    if (!workspace_layout(B, H_kv, N, d, &w)) return ATTN_ERR_UNSUPPORTED;
    if (attn_impl::plan_max_steps(B, H, N, causal) >= 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < w.total) return ATTN_ERR_INVALID_ARG;
    if (!get_encoder()) return ATTN_ERR_CUDA;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    attn_impl::VPrepParams vp{};
    vp.V = V;
    vp.V16 = ws + w.v16;
    vp.v_exp = reinterpret_cast<int32_t*>(ws + w.vexp);
    vp.N = N;
    vp.d = d;
    vp.n_ktiles = w.n_ktiles;
    vp.heads = B * H_kv;

    CUtensorMap tmQ, tmK, tmV;
    if (!get_map(&tmQ, MAP_Q_BF16, Q, d, N, static_cast<long long>(B) * H) ||
        !get_map(&tmK, MAP_K_BF16, K, d, N, static_cast<long long>(B) * H_kv) ||
        !get_map(&tmV, MAP_V_F16, vp.V16, d, N, static_cast<long long>(B) * H_kv))
        return ATTN_ERR_UNSUPPORTED;
    CUtensorMap tmO;
    memset(&tmO, 0, sizeof(tmO));
    if (out_dtype == ATTN_F32 && !get_map(&tmO, MAP_O_F32, O, d, N, static_cast<long long>(B) * H))
        return ATTN_ERR_UNSUPPORTED;

    const int sms = device_sms();
    if (sms <= 0) return ATTN_ERR_CUDA;
    attn_impl::TcParams p{};
    p.O = O;
    p.LSE = LSE;
    p.kv_len = kv_len;
    p.v_exp = vp.v_exp;
    p.n_ktiles = w.n_ktiles;
    p.boff = reinterpret_cast<const long long*>(ws + w.boff);
    p.part = reinterpret_cast<float*>(ws + w.part);
    p.flags = reinterpret_cast<unsigned int*>(ws + w.flags);
    p.plan = attn_impl::make_plan(B, H, N, causal, kv_len != nullptr, sms, g_plan_mode.load());
    p.H_kv = H_kv;
    p.group = H / H_kv;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.debug_skip_kv_load = g_skip_kv_load.load();
    if (ex) {
        p.bias = ex->bias;
        p.bias_sb = ex->bias_sb;
        p.bias_sh = ex->bias_sh;
        p.bias_sr = ex->bias_sr;
        p.drop_t = ex->drop_t;
        p.seed_lo = ex->seed_lo;
        p.seed_hi = ex->seed_hi;
        for (int r = 0; r < 10; ++r) {  // Philox4x32-10 key schedule: Weyl increments W0, W1 per round
            p.round_key[0][r] = ex->seed_lo + static_cast<uint32_t>(r) * 0x9E3779B9u;
            p.round_key[1][r] = ex->seed_hi + static_cast<uint32_t>(r) * 0xBB67AE85u;
        }
        p.rng_offset = ex->rng_offset;
        p.keep_scale = ex->keep_scale;
    }

    attn_impl::PlanParams pl{};
    pl.kv_len = kv_len;
    pl.boff = reinterpret_cast<long long*>(ws + w.boff);
    pl.flags = p.flags;
    pl.B = B; pl.H = H; pl.N = N; pl.n_pairs = p.plan.n_pairs; pl.causal = causal;

    if (attn_impl::launch_vprep(vp, pl, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    cudaEvent_t ev0 = g_ev_start.load(), ev1 = g_ev_stop.load();
    const bool timed = ev0 && ev1;
    if (timed && cudaEventRecord(ev0, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    const cudaError_t le = ex ? attn_impl::launch_attn_tc_ex(d, tmQ, tmK, tmV, tmO, p, stream)
                              : attn_impl::launch_attn_tc(d, out_dtype == ATTN_BF16, tmQ, tmK, tmV, tmO, p, stream);
    if (le != cudaSuccess) return ATTN_ERR_CUDA;
    if (timed && cudaEventRecord(ev1, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

}  // namespace

extern "C" {

size_t attn_workspace_bytes(int B, int H, int H_kv, int N, int d, attn_dtype in_dtype) {
    if (!sizes_ok(B, H, H_kv, N, d)) return 0;
    if (in_dtype != ATTN_BF16) return 0;
    WorkspaceLayout w;
    if (!workspace_layout(B, H_kv, N, d, &w)) return 0;
    return w.total;
}

attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int H_kv,
                     int N, int d, float scale, int causal, const int32_t* kv_len, attn_dtype in_dtype,
                     attn_dtype out_dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!Q || !K || !V || !O) return ATTN_ERR_INVALID_ARG;
    if (!sizes_ok(B, H, H_kv, N, d)) return ATTN_ERR_INVALID_ARG;
    if (!(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16)) return ATTN_ERR_INVALID_ARG;
    if (LSE && !aligned(LSE, 4)) return ATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return ATTN_ERR_INVALID_ARG;
    if (in_dtype != ATTN_F32 && in_dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
    if (out_dtype != ATTN_F32 && out_dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;

    if (in_dtype == ATTN_F32) {
        if (out_dtype != ATTN_F32) return ATTN_ERR_UNSUPPORTED;
        if (static_cast<long long>(B) * H > 65535) return ATTN_ERR_UNSUPPORTED;
        attn_impl::F32Params p{};
        p.Q = static_cast<const float*>(Q);
        p.K = static_cast<const float*>(K);
        p.V = static_cast<const float*>(V);
        p.O = O;
        p.LSE = LSE;
        p.kv_len = kv_len;
        p.B = B; p.H = H; p.H_kv = H_kv; p.N = N; p.group = H / H_kv; p.causal = causal;
        p.scale = scale;
        p.wait_limit_ns = g_wait_limit_ns.load();
        return attn_impl::launch_attn_f32(d, p, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }

    // bf16 inputs: tensor-core path
    return run_bf16_path(Q, K, V, O, LSE, B, H, H_kv, N, d, scale, causal, kv_len, out_dtype, workspace,
                         workspace_bytes, stream, nullptr);
}

attn_status attn_fwd_ex(const void* Q, const void* K, const void* V, float* O, float* LSE, int B, int H, int H_kv,
                        int N, int d, float scale, int causal, const int32_t* kv_len, const void* bias,
                        long long bias_stride_b, long long bias_stride_h, long long bias_stride_row, float dropout_p,
                        uint64_t seed, uint32_t offset, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!Q || !K || !V || !O) return ATTN_ERR_INVALID_ARG;
    if (!sizes_ok(B, H, H_kv, N, d)) return ATTN_ERR_INVALID_ARG;
    if (!(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16)) return ATTN_ERR_INVALID_ARG;
    if (LSE && !aligned(LSE, 4)) return ATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return ATTN_ERR_INVALID_ARG;
    if (!(dropout_p >= 0.f && dropout_p < 1.f)) return ATTN_ERR_INVALID_ARG;  // also rejects NaN
    if (bias) {
        if (!aligned(bias, 16)) return ATTN_ERR_INVALID_ARG;
        for (long long st : {bias_stride_b, bias_stride_h, bias_stride_row})
            if (st < 0 || st % 8 != 0) return ATTN_ERR_INVALID_ARG;
    }
    attn_impl::TcParams ex{};
    ex.bias = static_cast<const uint16_t*>(bias);
    ex.bias_sb = bias_stride_b;
    ex.bias_sh = bias_stride_h;
    ex.bias_sr = bias_stride_row;
    const double t = floor(static_cast<double>(dropout_p) * 65536.0);
    ex.drop_t = static_cast<uint32_t>(t);
    ex.keep_scale = static_cast<float>(65536.0 / (65536.0 - t));
    ex.seed_lo = static_cast<uint32_t>(seed & 0xffffffffull);
    ex.seed_hi = static_cast<uint32_t>(seed >> 32);
    ex.rng_offset = offset;
    return run_bf16_path(Q, K, V, O, LSE, B, H, H_kv, N, d, scale, causal, kv_len, ATTN_F32, workspace,
                         workspace_bytes, stream, &ex);
}

size_t attn_fwd_fp8_workspace_bytes(int B, int H, int H_kv, int N, int d) {
    if (!sizes_ok(B, H, H_kv, N, d) || d != 128) return 0;
    Fp8Layout w;
    if (!fp8_layout(B, H, H_kv, N, d, &w)) return 0;
    return w.total;
}

attn_status attn_fwd_fp8(const void* Q, const void* K, const void* V, float* O, float* LSE, int B, int H, int H_kv,
                         int N, int d, float scale, int causal, const int32_t* kv_len, const int8_t* signs,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!Q || !K || !V || !O) return ATTN_ERR_INVALID_ARG;
    if (!sizes_ok(B, H, H_kv, N, d)) return ATTN_ERR_INVALID_ARG;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    if (!(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16)) return ATTN_ERR_INVALID_ARG;
    if (LSE && !aligned(LSE, 4)) return ATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return ATTN_ERR_INVALID_ARG;
    Fp8Layout w;
    if (!fp8_layout(B, H, H_kv, N, d, &w)) return ATTN_ERR_UNSUPPORTED;
    if (attn_impl::plan_max_steps(B, H, N, causal) >= 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < w.total) return ATTN_ERR_INVALID_ARG;
    if (!get_encoder()) return ATTN_ERR_CUDA;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    attn_impl::Fp8PrepParams fp{};
    fp.Q = Q;
    fp.K = K;
    fp.V = V;
    fp.Q8 = ws + w.q8;
    fp.K8 = ws + w.k8;
    fp.V8T = ws + w.vt8;
    fp.q_exp = reinterpret_cast<int32_t*>(ws + w.qexp);
    fp.k_exp = reinterpret_cast<int32_t*>(ws + w.kexp);
    fp.v_exp = reinterpret_cast<int32_t*>(ws + w.vexp);
    fp.signs = signs;
    fp.N = N;
    fp.d = d;
    fp.n_ktiles = w.n_ktiles;
    fp.heads_q = B * H;
    fp.heads_kv = B * H_kv;
    fp.sms = device_sms();
    if (fp.sms <= 0) return ATTN_ERR_CUDA;
    fp.wait_limit_ns = g_wait_limit_ns.load();

    const int npad = w.n_ktiles * 128;
    CUtensorMap tmQ, tmK, tmV, tmO;
    if (!get_map(&tmQ, MAP_U8, fp.Q8, d, N, static_cast<long long>(B) * H) ||
        !get_map(&tmK, MAP_U8, fp.K8, d, N, static_cast<long long>(B) * H_kv) ||
        !get_map(&tmV, MAP_U8, fp.V8T, npad, d, static_cast<long long>(B) * H_kv) ||
        !get_map(&tmO, MAP_O_F32, O, d, N, static_cast<long long>(B) * H))
        return ATTN_ERR_UNSUPPORTED;

    const int sms = device_sms();
    if (sms <= 0) return ATTN_ERR_CUDA;
    attn_impl::TcParams p{};
    p.O = O;
    p.LSE = LSE;
    p.kv_len = kv_len;
    p.v_exp = fp.v_exp;
    p.q_exp = fp.q_exp;
    p.k_exp = fp.k_exp;
    p.n_ktiles = w.n_ktiles;
    p.boff = reinterpret_cast<const long long*>(ws + w.boff);
    p.part = reinterpret_cast<float*>(ws + w.part);
    p.flags = reinterpret_cast<unsigned int*>(ws + w.flags);
    p.plan = attn_impl::make_plan(B, H, N, causal, kv_len != nullptr, sms, g_plan_mode.load());
    p.H_kv = H_kv;
    p.group = H / H_kv;
    // the two unnormalised rotations multiply every score by d (a power of two here)
    p.scale_log2 = scale * 1.4426950408889634f / (signs ? static_cast<float>(d) : 1.0f);
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.debug_skip_kv_load = g_skip_kv_load.load();

    attn_impl::PlanParams pl{};
    pl.kv_len = kv_len;
    pl.boff = reinterpret_cast<long long*>(ws + w.boff);
    pl.flags = p.flags;
    pl.B = B; pl.H = H; pl.N = N; pl.n_pairs = p.plan.n_pairs; pl.causal = causal;

    if (attn_impl::launch_fp8_prep(fp, pl, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    cudaEvent_t ev0 = g_ev_start.load(), ev1 = g_ev_stop.load();
    const bool timed = ev0 && ev1;
    if (timed && cudaEventRecord(ev0, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (attn_impl::launch_attn_tc_fp8(tmQ, tmK, tmV, tmO, p, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (timed && cudaEventRecord(ev1, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status attn_merge(const float* O_parts, const float* LSE_parts, int n_parts, long long rows, int d, float* O,
                       float* LSE, cudaStream_t stream) {
    if (!O_parts || !LSE_parts || !O || !LSE) return ATTN_ERR_INVALID_ARG;
    if (n_parts <= 0 || rows <= 0 || (d != 64 && d != 128)) return ATTN_ERR_INVALID_ARG;
    if (!aligned(O_parts, 16) || !aligned(O, 16) || !aligned(LSE_parts, 4) || !aligned(LSE, 4)) return ATTN_ERR_INVALID_ARG;
    return attn_impl::launch_attn_merge(O_parts, LSE_parts, n_parts, rows, d, O, LSE, stream) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
    const size_t nqp = static_cast<size_t>((N + 127) / 128) * 128;
    return 2 * round_up(static_cast<size_t>(B) * H * nqp * sizeof(float), 256);
}

attn_status attn_bwd(const void* Q, const void* K, const void* V, const float* O, const void* dO, const float* LSE,
                     float* dQ, float* dK, float* dV, int B, int H, int H_kv, int N, int d, float scale, int causal,
                     const int32_t* kv_len, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return ATTN_ERR_INVALID_ARG;
    if (!sizes_ok(B, H, H_kv, N, d)) return ATTN_ERR_INVALID_ARG;
    if (!(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(dO, 16) || !aligned(O, 16) ||
        !aligned(dQ, 16) || !aligned(dK, 16) || !aligned(dV, 16) || !aligned(LSE, 4))
        return ATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return ATTN_ERR_INVALID_ARG;
    const size_t need = attn_bwd_workspace_bytes(B, H, N, d);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H_kv > 65535) return ATTN_ERR_UNSUPPORTED;
    if (!get_encoder()) return ATTN_ERR_CUDA;
    const int n_qt = (N + 127) / 128;
    const size_t half = need / 2;
    float* lse2 = static_cast<float*>(workspace);
    float* dvec = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + half);

    CUtensorMap tmQ, tmK, tmV, tmDO, tmDQ;
    // d = 128 runs the kernel with 64-row query tiles (its Q and dO maps have 64-row boxes)
    const bool q64 = d == 128;
    if (!get_map(&tmQ, q64 ? MAP_Q64_BF16 : MAP_Q_BF16, Q, d, N, static_cast<long long>(B) * H) ||
        !get_map(&tmK, MAP_K_BF16, K, d, N, static_cast<long long>(B) * H_kv) ||
        !get_map(&tmV, MAP_K_BF16, V, d, N, static_cast<long long>(B) * H_kv) ||
        !get_map(&tmDO, q64 ? MAP_Q64_BF16 : MAP_Q_BF16, dO, d, N, static_cast<long long>(B) * H) ||
        !get_map(&tmDQ, q64 ? MAP_O16_F32 : MAP_O_F32, dQ, d, N, static_cast<long long>(B) * H))
        return ATTN_ERR_UNSUPPORTED;

    attn_impl::BwdPrepParams pp{};
    pp.dO = dO; pp.O = O; pp.LSE = LSE; pp.lse2 = lse2; pp.dvec = dvec; pp.dQ = dQ;
    pp.rows = B * H; pp.N = N; pp.d = d; pp.NQP = n_qt * 128;
    attn_impl::BwdParams p{};
    p.dQ = dQ; p.dK = dK; p.dV = dV; p.lse2 = lse2; p.dvec = dvec; p.kv_len = kv_len;
    p.B = B; p.H = H; p.H_kv = H_kv; p.N = N; p.group = H / H_kv; p.causal = causal; p.n_qt = n_qt;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_limit_ns = g_wait_limit_ns.load();
    // the timing hook brackets both launches of the backward (its row-statistics pass and the kernel)
    cudaEvent_t ev0 = g_ev_start.load(), ev1 = g_ev_stop.load();
    const bool timed = ev0 && ev1;
    if (timed && cudaEventRecord(ev0, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (attn_impl::launch_attn_bwd(d, pp, tmQ, tmK, tmV, tmDO, tmDQ, p, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (timed && cudaEventRecord(ev1, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status attn_check(cudaStream_t stream) {
    uint32_t bits = 0, bwd_bits = 0, f32_bits = 0;
    if (attn_impl::read_and_clear_error(&bits, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (attn_impl::read_and_clear_bwd_error(&bwd_bits) != cudaSuccess) return ATTN_ERR_CUDA;
    if (attn_impl::read_and_clear_f32_error(&f32_bits) != cudaSuccess) return ATTN_ERR_CUDA;
    bits |= bwd_bits | f32_bits;
    g_last_error_bits.store(bits);
    return bits ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

uint32_t attn_debug_last_error_bits(void) { return g_last_error_bits.load(); }

const char* attn_status_string(attn_status s) {
    switch (s) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    }
    return "ATTN_UNKNOWN_STATUS";
}

int attn_launches_per_call(attn_dtype in_dtype) { return in_dtype == ATTN_BF16 ? 2 : 1; }

void attn_debug_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : kDefaultWaitLimitNs); }

void attn_debug_set_skip_kv_load(int on) { g_skip_kv_load.store(on ? 1 : 0); }

void attn_debug_set_plan_mode(int mode) { g_plan_mode.store(mode == 1 || mode == 2 ? mode : 0); }

int attn_debug_schedule(int B, int H, int N, int causal, const int32_t* kv_len_host, int sms, int32_t* out,
                        int max_segments) {
    if (B <= 0 || H <= 0 || N <= 0 || sms <= 0 || max_segments < 0 || (!out && max_segments > 0)) return -1;
    if (attn_impl::plan_max_steps(B, H, N, causal ? 1 : 0) >= 0x7fffffffLL) return -1;
    const attn_impl::SchedPlan plan =
        attn_impl::make_plan(B, H, N, causal ? 1 : 0, kv_len_host != nullptr, sms, g_plan_mode.load());
    std::vector<int> nb(B);
    std::vector<long long> boff(B + 1, 0);
    for (int b = 0; b < B; ++b) {
        int L = kv_len_host ? kv_len_host[b] : N;
        L = L < 0 ? 0 : (L > N ? N : L);
        nb[b] = attn_impl::key_tiles(L);
        boff[b + 1] = boff[b] + static_cast<long long>(H) * attn_impl::line_prefix(plan.n_pairs, nb[b], N, plan.causal);
    }
    const attn_impl::HostSchedTab tab{nb.data(), boff.data()};
    int n = 0;
    for (int c = 0; c < plan.G; ++c) {
        attn_impl::WalkState walk;
        attn_impl::walk_init(walk, tab, plan);
        attn_impl::Segment sg;
        while (attn_impl::walk_next(walk, tab, plan, c, sg)) {
            if (n < max_segments) {
                int32_t* o = out + 8 * static_cast<size_t>(n);
                o[0] = c; o[1] = sg.b; o[2] = sg.h; o[3] = sg.pair; o[4] = sg.k0; o[5] = sg.k1; o[6] = sg.cost;
                o[7] = sg.kind;
            }
            ++n;
        }
    }
    return n;
}

float attn_event_elapsed_ms(cudaEvent_t start, cudaEvent_t stop) {
    float ms = -1.f;
    if (!start || !stop || cudaEventElapsedTime(&ms, start, stop) != cudaSuccess) return -1.f;
    return ms;
}

void attn_set_kernel_events(cudaEvent_t start, cudaEvent_t stop) {
    g_ev_start.store(start && stop ? start : nullptr);
    g_ev_stop.store(start && stop ? stop : nullptr);
}

}  // extern "C"
