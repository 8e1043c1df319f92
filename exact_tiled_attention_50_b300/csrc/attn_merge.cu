// Merge of attention results computed over disjoint key sets (split-KV / sequence-parallel use).
//
// Each part i holds, for every row, the normalised output O_i over its own keys and its natural-log
// row log-sum-exp LSE_i (what attn_fwd writes). Over the union of the key sets,
//     LSE = log(sum_i exp(LSE_i)),     O = sum_i exp(LSE_i - LSE) O_i,
// which is the softmax merge rule of formula 2 in "闪电注意力的数学原理" on "闪电注意力：革命性地提高
// Transformer效率" (unite.ai), written with the per-part sums l_i = exp(LSE_i - m_i) folded into the
// log-sum-exp, and the intra/inter-block combination of "深入解析Blockwise Parallel Transformer在
// PyTorch中的实现与优化" (qqiyuan.cn). A part whose LSE is -inf (no valid key) contributes nothing.
//
// HBM-bound: one warp per row, each lane holding d/32 consecutive columns (a warp reads one whole
// row of a part: coalesced 8- or 16-byte loads), d in {64, 128}.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn_internal.h"

namespace attn_impl {

namespace {
constexpr int MERGE_THREADS = 256;

template <int CPL>  // columns per lane
__global__ void __launch_bounds__(MERGE_THREADS) attn_merge_kernel(const float* __restrict__ O_parts,
                                                                    const float* __restrict__ LSE_parts, int n_parts,
                                                                    long long rows, int d, float* __restrict__ O,
                                                                    float* __restrict__ LSE) {
    const long long row = static_cast<long long>(blockIdx.x) * (MERGE_THREADS / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float m = -INFINITY;
    for (int i = 0; i < n_parts; ++i) m = fmaxf(m, __ldg(LSE_parts + static_cast<long long>(i) * rows + row));
    float acc[CPL];
#pragma unroll
    for (int k = 0; k < CPL; ++k) acc[k] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
        for (int i = 0; i < n_parts; ++i) {
            const float li = __ldg(LSE_parts + static_cast<long long>(i) * rows + row);
            if (li == -INFINITY) continue;
            const float w = expf(li - m);
            wsum += w;
            const float* src = O_parts + (static_cast<long long>(i) * rows + row) * d + lane * CPL;
            if constexpr (CPL == 2) {
                const float2 v = __ldg(reinterpret_cast<const float2*>(src));
                acc[0] = fmaf(w, v.x, acc[0]);
                acc[1] = fmaf(w, v.y, acc[1]);
            } else {
#pragma unroll
                for (int k = 0; k < CPL; k += 4) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(src + k));
                    acc[k] = fmaf(w, v.x, acc[k]);
                    acc[k + 1] = fmaf(w, v.y, acc[k + 1]);
                    acc[k + 2] = fmaf(w, v.z, acc[k + 2]);
                    acc[k + 3] = fmaf(w, v.w, acc[k + 3]);
                }
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    float* dst = O + row * d + lane * CPL;
    if constexpr (CPL == 2) {
        *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
    } else {
#pragma unroll
        for (int k = 0; k < CPL; k += 4)
            *reinterpret_cast<float4*>(dst + k) =
                make_float4(acc[k] * inv, acc[k + 1] * inv, acc[k + 2] * inv, acc[k + 3] * inv);
    }
    if (lane == 0) LSE[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}
}  // namespace

cudaError_t launch_attn_merge(const float* O_parts, const float* LSE_parts, int n_parts, long long rows, int d,
                              float* O, float* LSE, cudaStream_t stream) {
    const long long blocks = (rows + MERGE_THREADS / 32 - 1) / (MERGE_THREADS / 32);
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (d == 128)
        attn_merge_kernel<4><<<grid, MERGE_THREADS, 0, stream>>>(O_parts, LSE_parts, n_parts, rows, d, O, LSE);
    else if (d == 64)
        attn_merge_kernel<2><<<grid, MERGE_THREADS, 0, stream>>>(O_parts, LSE_parts, n_parts, rows, d, O, LSE);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace attn_impl
