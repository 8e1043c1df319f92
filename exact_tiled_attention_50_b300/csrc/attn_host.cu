// attn_fwd_host: attention forward for inputs and outputs in host memory, with the copies to the
// device, the attention and the copies back pipelined over groups of heads.
//
// Heads are independent, so a group of key/value heads (with their query heads) can be copied in,
// computed and copied out on its own. Group k's inputs travel on one copy stream while group k - 1
// is computed on the caller's stream and group k - 2's outputs travel back on a second copy stream:
// the two PCIe directions and the kernels run at the same time instead of one after another. Every
// group's attention is an ordinary attn_fwd call on slices of the caller's device buffers, so its
// results are those of attn_fwd for those heads.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/attn.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxGroups = 64;

// Per device: the two copy streams and the events of one call's pipeline (created once, with that
// device current, and kept until the process exits).
struct Pipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t copied_in[kMaxGroups] = {}, computed[kMaxGroups] = {};
};
Pipe g_pipe[kMaxDevices];
std::mutex g_pipe_mutex;

Pipe* pipe_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    Pipe& p = g_pipe[dev];
    if (p.ready) return &p;
    const unsigned ev = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, ev) != cudaSuccess || cudaEventCreateWithFlags(&p.done, ev) != cudaSuccess)
        return nullptr;
    for (int i = 0; i < kMaxGroups; ++i)
        if (cudaEventCreateWithFlags(&p.copied_in[i], ev) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.computed[i], ev) != cudaSuccess)
            return nullptr;
    p.ready = true;
    return &p;
}

size_t elem_bytes(attn_dtype t) { return t == ATTN_F32 ? 4 : 2; }

// Groups of key/value heads per batch for these sizes: about `n_groups` in all (8 by default, at most
// 64 over every batch), never spanning two batches. With three or more per batch the first and the
// last group are half the size of the others: the first group's copy in and the last group's copy
// back are the parts of the pipeline that nothing overlaps. 0 when even one group per batch exceeds 64.
int groups_per_batch(int B, int H_kv, int n_groups) {
    long long want = n_groups > 0 ? n_groups : 8;
    if (want > kMaxGroups) want = kMaxGroups;
    long long per = (want + B - 1) / B;
    if (per >= 2) ++per;  // two half-size groups at the ends take the place of one
    if (per > H_kv) per = H_kv;
    if (per * B > kMaxGroups) per = kMaxGroups / B;
    return static_cast<int>(per);
}

// First key/value head of group i (0 <= i <= n) of a batch whose H_kv heads form n groups (n <= H_kv):
// weights 1, 2, ..., 2, 1 for n >= 3 (equal otherwise), boundaries rounded, every group kept non-empty.
int group_start(int H_kv, int n, int i) {
    if (i <= 0) return 0;
    if (i >= n) return H_kv;
    long long h;
    if (n < 3) {
        h = static_cast<long long>(H_kv) * i / n;
    } else {
        const long long W = 2LL * n - 2;
        h = (static_cast<long long>(H_kv) * (2LL * i - 1) + W / 2) / W;
    }
    if (h < i) h = i;                      // room for the i groups before
    if (h > H_kv - (n - i)) h = H_kv - (n - i);  // and for the n - i after
    return static_cast<int>(h);
}

}  // namespace

extern "C" int attn_fwd_host_groups(int B, int H_kv, int n_groups) {
    if (B <= 0 || H_kv <= 0) return -1;
    const int per = groups_per_batch(B, H_kv, n_groups);
    return per > 0 ? B * per : -1;
}

extern "C" attn_status attn_fwd_host(const void* Q_h, const void* K_h, const void* V_h, void* O_h, float* LSE_h,
                                     int B, int H, int H_kv, int N, int d, float scale, int causal,
                                     const int32_t* kv_len_h, attn_dtype in_dtype, attn_dtype out_dtype, void* Q_d,
                                     void* K_d, void* V_d, void* O_d, float* LSE_d, int32_t* kv_len_d,
                                     void* workspace, size_t workspace_bytes, int n_groups, cudaStream_t stream) {
    if (!Q_h || !K_h || !V_h || !O_h || !Q_d || !K_d || !V_d || !O_d) return ATTN_ERR_INVALID_ARG;
    if ((LSE_h == nullptr) != (LSE_d == nullptr) || (kv_len_h == nullptr) != (kv_len_d == nullptr))
        return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || H_kv <= 0 || N <= 0 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
    if ((in_dtype != ATTN_F32 && in_dtype != ATTN_BF16) || (out_dtype != ATTN_F32 && out_dtype != ATTN_BF16))
        return ATTN_ERR_INVALID_ARG;
    const int n_per = groups_per_batch(B, H_kv, n_groups);
    if (n_per <= 0) return ATTN_ERR_UNSUPPORTED;  // more than 64 groups
    const int g = H / H_kv;
    int ck = 0;  // key/value heads of the largest group
    for (int i = 0; i < n_per; ++i) {
        const int nk = group_start(H_kv, n_per, i + 1) - group_start(H_kv, n_per, i);
        if (nk > ck) ck = nk;
    }
    // the largest group's call needs the most workspace (the whole problem's is always enough)
    if (in_dtype == ATTN_BF16 && workspace_bytes < attn_workspace_bytes(1, ck * g, ck, N, d, in_dtype))
        return ATTN_ERR_INVALID_ARG;
    Pipe* pp = pipe_for_current_device();
    if (!pp) return ATTN_ERR_CUDA;

    const size_t ein = elem_bytes(in_dtype), eout = elem_bytes(out_dtype);
    const size_t head = static_cast<size_t>(N) * d;  // elements of one head's [N, d] slab
    if (cudaEventRecord(pp->start, stream) != cudaSuccess || cudaStreamWaitEvent(pp->in, pp->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(pp->out, pp->start, 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (kv_len_h &&
        cudaMemcpyAsync(kv_len_d, kv_len_h, static_cast<size_t>(B) * sizeof(int32_t), cudaMemcpyHostToDevice,
                        pp->in) != cudaSuccess)
        return ATTN_ERR_CUDA;
    int k = 0;
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < n_per; ++i, ++k) {
            const int h0 = group_start(H_kv, n_per, i);
            const int nk = group_start(H_kv, n_per, i + 1) - h0;  // key/value heads of this group
            const size_t zq = static_cast<size_t>(b) * H + static_cast<size_t>(h0) * g;  // first query head
            const size_t zk = static_cast<size_t>(b) * H_kv + h0;                          // first key/value head
            const size_t nq_el = static_cast<size_t>(nk) * g * head, nk_el = static_cast<size_t>(nk) * head;
            const uint8_t* qh = static_cast<const uint8_t*>(Q_h) + zq * head * ein;
            const uint8_t* kh = static_cast<const uint8_t*>(K_h) + zk * head * ein;
            const uint8_t* vh = static_cast<const uint8_t*>(V_h) + zk * head * ein;
            uint8_t* qd = static_cast<uint8_t*>(Q_d) + zq * head * ein;
            uint8_t* kd = static_cast<uint8_t*>(K_d) + zk * head * ein;
            uint8_t* vd = static_cast<uint8_t*>(V_d) + zk * head * ein;
            // in: this group's Q, K, V (one copy each)
            if (cudaMemcpyAsync(qd, qh, nq_el * ein, cudaMemcpyHostToDevice, pp->in) != cudaSuccess ||
                cudaMemcpyAsync(kd, kh, nk_el * ein, cudaMemcpyHostToDevice, pp->in) != cudaSuccess ||
                cudaMemcpyAsync(vd, vh, nk_el * ein, cudaMemcpyHostToDevice, pp->in) != cudaSuccess ||
                cudaEventRecord(pp->copied_in[k], pp->in) != cudaSuccess ||
                cudaStreamWaitEvent(stream, pp->copied_in[k], 0) != cudaSuccess)
                return ATTN_ERR_CUDA;
            // compute: the attention of these heads on the caller's stream
            uint8_t* od = static_cast<uint8_t*>(O_d) + zq * head * eout;
            float* ld = LSE_d ? LSE_d + zq * N : nullptr;
            const attn_status st = attn_fwd(qd, kd, vd, od, ld, 1, nk * g, nk, N, d, scale, causal,
                                            kv_len_d ? kv_len_d + b : nullptr, in_dtype, out_dtype, workspace,
                                            workspace_bytes, stream);
            if (st != ATTN_OK) return st;
            if (cudaEventRecord(pp->computed[k], stream) != cudaSuccess ||
                cudaStreamWaitEvent(pp->out, pp->computed[k], 0) != cudaSuccess)
                return ATTN_ERR_CUDA;
            // out: this group's O and LSE
            uint8_t* oh = static_cast<uint8_t*>(O_h) + zq * head * eout;
            if (cudaMemcpyAsync(oh, od, nq_el * eout, cudaMemcpyDeviceToHost, pp->out) != cudaSuccess) return ATTN_ERR_CUDA;
            if (LSE_h && cudaMemcpyAsync(LSE_h + zq * N, ld, static_cast<size_t>(nk) * g * N * sizeof(float),
                                         cudaMemcpyDeviceToHost, pp->out) != cudaSuccess)
                return ATTN_ERR_CUDA;
        }
    }
    // the call's stream reaches its end once every copy back has completed
    if (cudaEventRecord(pp->done, pp->out) != cudaSuccess || cudaStreamWaitEvent(stream, pp->done, 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}
