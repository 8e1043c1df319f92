/*
 * attn.h - C ABI of libattn.so: exact multi-head attention forward on NVIDIA B300 (sm_103a).
 *
 * The operation (for every batch b, query head h, query row i; kv = h / (H / H_kv)):
 *
 *     s_ij  = scale * sum_k Q[b,h,i,k] K[b,kv,j,k]
 *     valid = j < kv_len[b]  and  (causal == 0  or  j <= i)
 *     O_i   = sum_{valid j} exp(s_ij - m_i) V[b,kv,j,:] / l_i,   m_i = max_{valid j} s_ij,
 *             l_i = sum_{valid j} exp(s_ij - m_i)
 *     LSE_i = m_i + ln l_i        (natural log; a row without valid keys gets O = 0, LSE = -inf)
 *
 * This is the attention of the standard_attention listings on the pages "AI训练的最大障碍不是算力,
 * 而是'内存墙'" (zsdodo.com) and "闪电注意力：革命性地提高Transformer效率" (unite.ai), computed the
 * tiled way those pages describe: the unite.ai section "闪电注意力的数学原理" (softmax decomposition
 * and merging of per-block partial results), the running maximum / running sum recurrence of the
 * safe_softmax_block listing (zsdodo.com) and the unnormalised accumulator with one final division of
 * section 4.1.3 "算法流程详解" of "第四章 注意力机制实战案例" (aiknowledge.cn). The score matrix never
 * goes to device memory. Grouped- and multi-query heads (H_kv < H) follow the unite.ai section
 * "闪电注意力-2"; key padding (kv_len) follows the attention_mask of "动态序列处理" on
 * "基于AIFI多头注意力机制的高效序列建模实战" (qqiyuan.cn).
 *
 * Layouts (all contiguous, row-major, device memory):
 *   Q   [B, H,    N, d]     K, V [B, H_kv, N, d]     (in_dtype: bf16 or fp32, the same for all three)
 *   O   [B, H,    N, d]     (out_dtype: fp32, or bf16 for bf16 inputs)
 *   LSE [B, H,    N]        fp32, may be NULL (not written)
 *   kv_len int32 [B], may be NULL (= N for every batch); values are clamped to [0, N].
 *
 * Precision. fp32 inputs are computed in exact fp32 arithmetic (CUDA cores). bf16 inputs use the
 * tensor cores: Q K^T is exact bf16 products with fp32 accumulation; the softmax state (m, l) is
 * fp32 per row; the probabilities enter P V as fp16 and V is converted to fp16 with a power-of-two
 * scale per 128-key tile (exact for bf16 values in fp16's normal range; the accumulator follows the
 * largest tile exponent seen so far, like the running maximum), accumulating O in fp32.
 *
 * Ownership and asynchrony. The caller owns every buffer. The library never allocates device
 * memory in attn_fwd: bf16 inputs need a caller-provided workspace of attn_workspace_bytes() bytes
 * (device memory, 256-byte aligned; its contents need no initialisation and are scratch between
 * calls; two calls that overlap on the GPU must not share it). The call only enqueues work on
 * `stream` and returns; results are ready when the stream reaches that point. The library keeps
 * one device error word per device (for bounded-wait timeouts) and no other state.
 *
 * Errors. attn_fwd validates its arguments and returns without launching anything on: a NULL
 * Q/K/V/O pointer, B, H, H_kv or N <= 0, H % H_kv != 0, d not in {64, 128}, scale not finite or
 * <= 0, a Q/K/V/O/workspace pointer not 16-byte aligned (workspace: 256), too small a workspace,
 * or an unsupported dtype pair (fp32 inputs with bf16 output) -> ATTN_ERR_INVALID_ARG or
 * ATTN_ERR_UNSUPPORTED. A failed launch returns ATTN_ERR_CUDA. Every wait inside the tensor-core
 * kernel gives up after a time limit (about one second) instead of hanging the GPU; it then records
 * ATTN_ERR_TIMEOUT in the device error word, and attn_check() reports it.
 */
#ifndef EXACT_TILED_ATTENTION_B300_ATTN_H
#define EXACT_TILED_ATTENTION_B300_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,
    ATTN_ERR_UNSUPPORTED = 2,
    ATTN_ERR_CUDA = 3,
    ATTN_ERR_TIMEOUT = 4
} attn_status;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype;

/*
 * Bytes of device workspace attn_fwd needs for these sizes (0 for fp32 inputs). For bf16 inputs it
 * holds the fp16 copy of V ([B, H_kv, N, d]) with one power-of-two exponent per 128-key tile, the
 * work schedule and the partial results of work units split between CTAs. Returns 0 for invalid sizes.
 */
size_t attn_workspace_bytes(int B, int H, int H_kv, int N, int d, attn_dtype in_dtype);

/*
 * Attention forward (see the top of this file for the operation, layouts, ownership and errors).
 *   Q, K, V      device pointers, in_dtype
 *   O            device pointer, out_dtype
 *   LSE          device fp32 pointer or NULL
 *   B, H, H_kv, N, d   sizes; d in {64, 128}; H % H_kv == 0
 *   scale        score scale (typically 1/sqrt(d)); finite and > 0
 *   causal       0 or 1: mask keys j > i
 *   kv_len       device int32 [B] or NULL
 *   workspace    device pointer to attn_workspace_bytes() bytes (may be NULL when that is 0)
 *   stream       CUDA stream the work is enqueued on (0 = legacy default stream)
 */
attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int H_kv,
                     int N, int d, float scale, int causal, const int32_t* kv_len, attn_dtype in_dtype,
                     attn_dtype out_dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Attention forward with an additive bias and dropout (bf16 inputs, fp32 output): the interface of
 * the xFormers memory-efficient attention call in the EfficientAttention module of "AI训练的最大障碍
 * 不是算力,而是'内存墙'" (zsdodo.com), which passes attn_bias and a dropout probability p. Read as
 *     s_ij  = scale * q_i . k_j + bias[b,h,i,j]       (masks of attn_fwd applied on top)
 *     P_ij  = softmax_j(s_ij),   LSE_i = ln sum_j exp(s_ij)      (no dropout in either)
 *     O_i   = sum_j P_ij keep_ij / (1 - t / 65536) V_j
 * keep_ij comes from the counter-based generator Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC 2011) with key (seed mod 2^32, seed >> 32)
 * and counter (j >> 3, i, b * H + h, offset): its output words w0..w3 give eight 16-bit values
 * u_2m = w_m mod 2^16, u_2m+1 = w_m >> 16, and key j keeps its probability iff u_(j mod 8) >= t,
 * t = floor(dropout_p * 65536) (effective drop probability t / 65536). Any tiling or schedule draws
 * the same mask; a different `offset` (or seed) draws an independent one.
 *   bias       device bf16 or NULL: element (b, h, i, j) at bias[b * stride_b + h * stride_h +
 *              i * stride_row + j] (strides in elements, >= 0, multiples of 8; 16-byte aligned base;
 *              a stride of 0 broadcasts, e.g. one [N, N] bias for every batch and head). Values may
 *              be -inf (masking); the row must hold N valid entries.
 *   dropout_p  0 <= p < 1 (0: no dropout);  seed, offset: the generator's key and counter word 3
 *   workspace  attn_workspace_bytes(B, H, H_kv, N, d, ATTN_BF16) bytes, as for attn_fwd
 * Other arguments, errors and asynchrony as attn_fwd (invalid strides, alignment or p:
 * ATTN_ERR_INVALID_ARG).
 */
attn_status attn_fwd_ex(const void* Q, const void* K, const void* V, float* O, float* LSE, int B, int H, int H_kv,
                        int N, int d, float scale, int causal, const int32_t* kv_len, const void* bias,
                        long long bias_stride_b, long long bias_stride_h, long long bias_stride_row, float dropout_p,
                        uint64_t seed, uint32_t offset, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fp8 attention forward with incoherent processing (section "闪电注意力-3" of the unite.ai page names
 * FP8 computation and a processing step that lowers the quantisation error of the low-precision
 * format; this library reads the step as a random orthogonal rotation of Q and K, which leaves
 * Q K^T unchanged and spreads an outlier channel over all channels before rounding):
 *   1. if `signs` is not NULL, every row of Q and K is multiplied elementwise by signs (d values
 *      +-1, the rotation's random draw, chosen by the caller) and transformed by the Walsh-Hadamard
 *      matrix H_d (unnormalised; the factor 1/d of the two transforms moves into the score scale);
 *   2. Q, K and V are rounded to E4M3 (OCP 8-bit float: 4 exponent bits, 3 mantissa bits, max 448;
 *      round to nearest even, saturating) with one power-of-two scale per 128-row tile per head,
 *      2^e with e = max(e8 - 134, -100) for the largest |x| of the tile having fp32 exponent field e8;
 *   3. the attention of attn_fwd over the rounded values, both products on the E4M3 tensor cores
 *      with fp32 accumulation; the probabilities P enter P V as E4M3 as well.
 * Result: the attention of the rounded inputs, up to the E4M3 rounding of P (relative 2^-4 per
 * probability) and fp32 arithmetic. Not exact attention: the rounding of the inputs is part of it.
 *   Q, K, V      device bf16 pointers, [B, H, N, d] / [B, H_kv, N, d] as for attn_fwd
 *   O, LSE       device fp32 [B, H, N, d] and [B, H, N] (LSE may be NULL)
 *   d            128 only (other values: ATTN_ERR_UNSUPPORTED)
 *   scale, causal, kv_len, stream   as for attn_fwd
 *   signs        device int8 [d] with values +1 / -1, or NULL (no rotation)
 *   workspace    device, attn_fwd_fp8_workspace_bytes() bytes, 256-byte aligned: the E4M3 copies
 *                of Q, K and V (V transposed), their tile exponents, the work schedule and the
 *                partial results of split work units; scratch between calls
 * Errors as attn_fwd; timeouts of bounded waits are reported by attn_check.
 */
size_t attn_fwd_fp8_workspace_bytes(int B, int H, int H_kv, int N, int d);
attn_status attn_fwd_fp8(const void* Q, const void* K, const void* V, float* O, float* LSE, int B, int H, int H_kv,
                         int N, int d, float scale, int causal, const int32_t* kv_len, const int8_t* signs,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Backward pass of attn_fwd (bf16 inputs): the gradients of the output O with respect to Q, K and V
 * for an upstream gradient dO. The pages state the forward only; this is its chain rule in the
 * recompute form of "闪电注意力：革命性地提高Transformer效率" (unite.ai: the attention matrix is not
 * stored but rebuilt in the backward pass) from the forward's row log-sum-exp:
 *     P = exp(scale Q K^T - LSE) (masked as in attn_fwd), dV = P^T dO, dP = dO V^T,
 *     D = rowsum(dO * O), dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q;
 * grouped heads sum dK and dV over the query heads of their group.
 *   Q, dO      device bf16 [B, H, N, d];  K, V device bf16 [B, H_kv, N, d]
 *   O, LSE     device fp32 [B, H, N, d] and [B, H, N]: attn_fwd's outputs for the same inputs
 *   dQ         device fp32 [B, H, N, d]; dK, dV device fp32 [B, H_kv, N, d] (all overwritten)
 *   scale, causal, kv_len as for attn_fwd; d in {64, 128}
 *   workspace  device, attn_bwd_workspace_bytes() bytes, 256-byte aligned (row statistics)
 * Precision: P and dS enter the tensor-core products as bf16 with fp32 accumulation. Errors: as
 * attn_fwd (no launch on invalid arguments); bounded waits report ATTN_ERR_TIMEOUT via attn_check.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);
attn_status attn_bwd(const void* Q, const void* K, const void* V, const float* O, const void* dO, const float* LSE,
                     float* dQ, float* dK, float* dV, int B, int H, int H_kv, int N, int d, float scale, int causal,
                     const int32_t* kv_len, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_fwd for inputs and outputs in host memory (the operation is attn_fwd's; the overlap of
 * copies and compute is the asynchronous overlap named in section "闪电注意力-3", item 1, of
 * "闪电注意力：革命性地提高Transformer效率", unite.ai): the copies to the device, the attention and the
 * copies back are pipelined over groups of heads (heads are independent, so a group of key/value
 * heads with their query heads is copied in, computed and copied back on its own), and group k's
 * inputs cross PCIe while group k - 1 is computed and group k - 2's outputs cross back. Each group's
 * attention is an attn_fwd call on slices of the device buffers, so the results are attn_fwd's.
 *   Q_h, K_h, V_h, O_h, LSE_h, kv_len_h   host pointers, layouts and types as attn_fwd (LSE_h and
 *                kv_len_h may be NULL, then LSE_d / kv_len_d must be NULL too). Page-locked host
 *                memory lets the copies run asynchronously and overlap; pageable memory still works.
 *   Q_d, K_d, V_d, O_d, LSE_d, kv_len_d   device buffers of the same sizes, owned by the caller; they
 *                hold the inputs and outputs afterwards
 *   workspace    device, at least attn_workspace_bytes() of one group (the whole problem's size is
 *                always enough), 256-byte aligned, as for attn_fwd
 *   n_groups     head groups to aim for (0: 8); never more than 64, and a group never spans two
 *                batches; with two or more groups per batch the batch gets one more, the first and
 *                the last half the size of the others (their copies are the ones nothing overlaps):
 *                attn_fwd_host_groups() gives the number the call will use
 *   stream       the call's stream: the inputs are read after the work already on it, the kernels run
 *                on it, and it reaches the end of the call once every output is back in host memory
 *                (the copies run on two streams the library creates per device on first use and keeps)
 * Errors as attn_fwd (checked before anything is enqueued where possible); ATTN_ERR_CUDA if a copy or
 * stream operation fails. Calls on different streams (or host threads) share the copy streams, so
 * their copies queue behind each other; calls that share device buffers or a workspace must not
 * overlap.
 */
attn_status attn_fwd_host(const void* Q_h, const void* K_h, const void* V_h, void* O_h, float* LSE_h, int B, int H,
                          int H_kv, int N, int d, float scale, int causal, const int32_t* kv_len_h, attn_dtype in_dtype,
                          attn_dtype out_dtype, void* Q_d, void* K_d, void* V_d, void* O_d, float* LSE_d,
                          int32_t* kv_len_d, void* workspace, size_t workspace_bytes, int n_groups,
                          cudaStream_t stream);

/* Number of head groups attn_fwd_host uses for these sizes and n_groups (-1 on invalid sizes). */
int attn_fwd_host_groups(int B, int H_kv, int n_groups);

/*
 * Merge of attention results over disjoint key sets (split-KV or sequence-parallel attention: each
 * part attends the same queries to its own keys). For every row,
 *     LSE = log(sum_i exp(LSE_i)),   O = sum_i exp(LSE_i - LSE) O_i
 * (the softmax merge rule of formula 2, "闪电注意力的数学原理", on "闪电注意力：革命性地提高
 * Transformer效率", unite.ai; the intra/inter-block combination of "深入解析Blockwise Parallel
 * Transformer在PyTorch中的实现与优化", qqiyuan.cn). A part with LSE = -inf contributes nothing; a row
 * where every part has -inf gets O = 0, LSE = -inf.
 *   O_parts   device fp32 [n_parts, rows, d]  (each part normalised, as attn_fwd writes O)
 *   LSE_parts device fp32 [n_parts, rows]     (natural log, as attn_fwd writes LSE)
 *   O, LSE    device fp32 [rows, d] and [rows]; must not overlap the inputs
 *   d in {64, 128}; rows = B * H * N for attn_fwd outputs.
 * Errors: NULL pointers, n_parts or rows <= 0, other d, misaligned pointers (16 bytes for O buffers)
 * -> ATTN_ERR_INVALID_ARG without a launch; a failed launch -> ATTN_ERR_CUDA. Asynchronous on `stream`.
 */
attn_status attn_merge(const float* O_parts, const float* LSE_parts, int n_parts, long long rows, int d, float* O,
                       float* LSE, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the calling device's error word. Returns ATTN_OK,
 * ATTN_ERR_TIMEOUT (a bounded wait inside a kernel ran out; the results of that call are invalid)
 * or ATTN_ERR_CUDA (the stream reported an error).
 */
attn_status attn_check(cudaStream_t stream);

/*
 * Diagnostic detail of the last attn_check on this process: 0, or the device error bits it read
 * (bit 0: a bounded wait ran out; higher bits name the wait: 2 Q tile, 4 key/value stage, 8 scores,
 * 16 probabilities, 32 output, 64 free stage, 128 final drain, 256 another CTA's partial result).
 */
uint32_t attn_debug_last_error_bits(void);

/* Static, human-readable name of a status code. */
const char* attn_status_string(attn_status s);

/* Number of kernel launches attn_fwd enqueues for these arguments (1 for fp32, 2 for bf16: the V
 * conversion with the schedule plan, and the persistent attention kernel). */
int attn_launches_per_call(attn_dtype in_dtype);

/*
 * Test hooks for the failure path (not for production use).
 * attn_debug_set_wait_limit_ns: time limit of every bounded wait in the tensor-core kernel
 *   (default 1e9 ns; 0 restores the default).
 * attn_debug_set_skip_kv_load: when non-zero, the next attn_fwd calls make the TMA producer
 *   skip issuing the load of key tile 0, so the consumer's wait on it runs out and the kernel
 *   reports ATTN_ERR_TIMEOUT through attn_check(). Nothing is left in flight.
 */
void attn_debug_set_wait_limit_ns(uint64_t ns);
void attn_debug_set_skip_kv_load(int on);

/*
 * Test hook: the work plan of the following calls' persistent kernel (and of attn_debug_schedule).
 * 0 (default) = the cheaper of the two plans by the library's cost model; 1 = whole work units in
 * rounds (no unit split between CTAs); 2 = stream-K (the key range shared evenly, split units merged).
 * Results are the same under every plan; only the time differs. Other values mean 0.
 */
void attn_debug_set_plan_mode(int mode);

/*
 * Test hook (host only, no GPU needed): the work schedule the tensor-core kernel would follow for
 * these sizes on a device with `sms` SMs, with kv_len given as a HOST int32 array [B] (or NULL).
 * Writes up to max_segments records (out may be NULL when max_segments is 0) of 8 int32 (cta, b, h, pair, k0, k1, cost, kind; kind 0 = the
 * whole unit, 1 = the piece that holds the unit's first key step and merges the others, 2 = a later
 * piece that hands its partial result to that one) in the order each CTA runs them, and returns the
 * total number of segments (-1 on invalid arguments).
 */
int attn_debug_schedule(int B, int H, int N, int causal, const int32_t* kv_len_host, int sms, int32_t* out,
                        int max_segments);

/*
 * Timing hook for benchmarks: while set (both non-NULL), every attn_fwd, attn_fwd_fp8 and attn_fwd_ex
 * call records `start` on its stream immediately before the main attention kernel and `stop`
 * immediately after it (attn_bwd: around its two launches, the row-statistics pass and the kernel),
 * so that cudaEventElapsedTime gives that duration on the stream the work runs on. The events are
 * created and owned by the caller. attn_set_kernel_events(NULL, NULL) turns the hook off.
 */
void attn_set_kernel_events(cudaEvent_t start, cudaEvent_t stop);

/* Milliseconds between two recorded events (cudaEventElapsedTime); -1 on error. */
float attn_event_elapsed_ms(cudaEvent_t start, cudaEvent_t stop);

/*
 * Attention forward without any device allocation, for callers that cannot allocate device memory
 * where they run attention (inside a host callback or an allocator's own hooks, under a memory pool
 * that is fixed at start-up and fully handed out, or in plug-in hosts that forbid device allocation
 * after initialisation). The method itself has no counterpart on the pages: it is attn_fwd with its
 * scratch taken from one fixed array instead of a caller workspace.
 *
 * Arguments, layouts, results and errors are those of attn_fwd, without workspace/workspace_bytes.
 * The caller still allocates Q, K, V, O, LSE and kv_len. The scratch is a static device array of
 * ATTN_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library, which every GPU that loads the library
 * holds until the process exits. The exact size limit: a call is accepted when
 * attn_workspace_bytes(B, H, H_kv, N, d, ATTN_BF16) <= ATTN_NOALLOC_SCRATCH_BYTES (about 22.8 M
 * elements of B * H_kv * N * d at d = 128, 28 M at d = 64); larger sizes return ATTN_ERR_UNSUPPORTED
 * without launching (use attn_fwd with a workspace for those). fp32 inputs need no scratch.
 *
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current). With CUDA's lazy module loading (the default) that lookup is also what loads
 * the library's device code on the device and so reserves the 64 MiB: make the first call on each
 * device during initialisation, before memory pools are handed out and before any stream capture.
 * The address is looked up again when the device's context changes (after cudaDeviceReset). No call
 * allocates device memory (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 * Every call on a device uses the same array, and the array keeps the contents of the last call.
 * Nothing in it needs clearing: each call writes every scratch byte it reads before reading it. Two
 * calls whose work overlaps on the GPU (different streams without ordering, or different host
 * threads) race on the array and give wrong results; order them on one stream or with events.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

attn_status attn_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                             int H_kv, int N, int d, float scale, int causal, const int32_t* kv_len,
                             attn_dtype in_dtype, attn_dtype out_dtype, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_TILED_ATTENTION_B300_ATTN_H */
