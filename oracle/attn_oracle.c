/*
 * CPU oracle for exact multi-head attention forward, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call this file: it is used by tests/,
 * by __graft_entry__.smoke() (to check one small GPU result) and by bench.py's CPU-baseline and
 * reference legs. It shares no code, header or constant with the CUDA library.
 *
 * What it computes (the plain definition; the tiled method reaches the same result up to rounding):
 *   for every batch b, query head h, query row i, with kv = h / (H / H_kv):
 *     s_ij  = scale * sum_k Q[b,h,i,k] * K[b,kv,j,k]                 (fp64 products and sums)
 *     valid = (j < kv_len[b]) and (not causal or j <= i)
 *     m_i   = max_{valid j} s_ij
 *     P_ij  = exp(s_ij - m_i) / sum_{valid j} exp(s_ij - m_i)       (0 for masked j)
 *     O_i   = sum_j P_ij V[b,kv,j,:]
 *     LSE_i = m_i + ln(sum_{valid j} exp(s_ij - m_i))
 *   A row with no valid key gets O = 0 and LSE = -inf.
 *
 * Sources:
 *  - "AI训练的最大障碍不是算力,而是'内存墙'" (zsdodo.com), listing standard_attention: scores = Q K^T
 *    scaled, softmax over the key axis, weights times V; the full score matrix is stored.
 *  - "闪电注意力：革命性地提高Transformer效率" (unite.ai), section "闪电注意力的数学原理",
 *    formula 1 (softmax decomposition with the row maximum subtracted) and the standard_attention
 *    listing at the top of the page.
 *  - "基于AIFI多头注意力机制的高效序列建模实战" (qqiyuan.cn), "避坑指南": subtract the maximum before the
 *    softmax; "动态序列处理": attention_mask ignores padded positions (here: keys j >= kv_len[b]).
 *  - Grouped / multi-query heads (unite.ai page, section "闪电注意力-2", item 3): query head h reads
 *    key/value head h / (H / H_kv).
 *  - The tiled variant restates the online-softmax statistics of the safe_softmax_block listing
 *    (zsdodo.com page) with the unnormalised accumulator and single final division of the
 *    flash_attention listing in section 4.1.3 of "第四章 注意力机制实战案例" (aiknowledge.cn), the row
 *    maximum taken over the key axis.
 *
 * Inputs are fp32 arrays holding the exact input values (bf16 and fp32 values are both exactly
 * representable); every arithmetic step is fp64. Layouts are row-major: Q [B,H,N,d],
 * K and V [B,H_kv,N,d], O [B,H,N,d], LSE [B,H,N].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int check_args(int B, int H, int H_kv, int N, int d) {
    if (B <= 0 || H <= 0 || H_kv <= 0 || N <= 0 || d <= 0) return 1;
    if (H % H_kv != 0) return 1;
    return 0;
}

static int valid_key(int i, int j, int kvl, int causal) {
    if (j >= kvl) return 0;
    if (causal && j > i) return 0;
    return 1;
}

static int clamp_len(const int32_t* kv_len, int b, int N) {
    if (!kv_len) return N;
    int L = kv_len[b];
    if (L < 0) L = 0;
    if (L > N) L = N;
    return L;
}

/* Threads the following calls use (benchmark legs time the oracle on one core as well as on all). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full oracle: materialises the N x N score matrix of each (b, h) in fp64, then takes the softmax
 * of every row and multiplies by V. If P_out is not NULL it receives the probabilities
 * [B,H,N,N] (tests check their row sums).
 */
int oracle_attn_f64(const float* Q, const float* K, const float* V, double* O, double* LSE,
                    double* P_out, int B, int H, int H_kv, int N, int d, double scale, int causal,
                    const int32_t* kv_len) {
    if (check_args(B, H, H_kv, N, d)) return 1;
    const int g = H / H_kv;
    double* S = (double*)malloc(sizeof(double) * (size_t)N * (size_t)N);
    if (!S) return 2;
    for (int b = 0; b < B; ++b) {
        const int kvl = clamp_len(kv_len, b, N);
        for (int h = 0; h < H; ++h) {
            const int kvh = h / g;
            const float* q = Q + ((size_t)b * H + h) * (size_t)N * d;
            const float* k = K + ((size_t)b * H_kv + kvh) * (size_t)N * d;
            const float* v = V + ((size_t)b * H_kv + kvh) * (size_t)N * d;
            double* o = O + ((size_t)b * H + h) * (size_t)N * d;
            double* lse = LSE + ((size_t)b * H + h) * (size_t)N;

            /* S = scale * Q K^T, every entry, masked or not. */
#pragma omp parallel for schedule(static)
            for (int i = 0; i < N; ++i) {
                for (int j = 0; j < N; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += (double)q[(size_t)i * d + c] * (double)k[(size_t)j * d + c];
                    S[(size_t)i * N + j] = scale * acc;
                }
            }

            /* Row softmax (max subtracted) over the valid keys, then P V. */
#pragma omp parallel for schedule(static)
            for (int i = 0; i < N; ++i) {
                double* srow = S + (size_t)i * N;
                double m = -INFINITY;
                for (int j = 0; j < N; ++j)
                    if (valid_key(i, j, kvl, causal) && srow[j] > m) m = srow[j];
                double* orow = o + (size_t)i * d;
                for (int c = 0; c < d; ++c) orow[c] = 0.0;
                if (m == -INFINITY) {
                    lse[i] = -INFINITY;
                    if (P_out) {
                        double* prow = P_out + (((size_t)b * H + h) * (size_t)N + i) * (size_t)N;
                        for (int j = 0; j < N; ++j) prow[j] = 0.0;
                    }
                    continue;
                }
                double l = 0.0;
                for (int j = 0; j < N; ++j) {
                    double p = valid_key(i, j, kvl, causal) ? exp(srow[j] - m) : 0.0;
                    srow[j] = p;
                    l += p;
                }
                for (int j = 0; j < N; ++j) {
                    const double p = srow[j] / l;
                    srow[j] = p;
                    if (p != 0.0)
                        for (int c = 0; c < d; ++c) orow[c] += p * (double)v[(size_t)j * d + c];
                }
                lse[i] = m + log(l);
                if (P_out) {
                    double* prow = P_out + (((size_t)b * H + h) * (size_t)N + i) * (size_t)N;
                    memcpy(prow, srow, sizeof(double) * (size_t)N);
                }
            }
        }
    }
    free(S);
    return 0;
}

/*
 * Row-sampled oracle: the same definition, evaluated only for the listed query rows
 * (rows[r] = (b*H + h)*N + i). Each listed row materialises its full score row over all N keys.
 * Used where the full N x N matrices of a large workload would take too long.
 */
int oracle_attn_rows_f64(const float* Q, const float* K, const float* V, const int64_t* rows,
                         int n_rows, double* O_rows, double* LSE_rows, int B, int H, int H_kv,
                         int N, int d, double scale, int causal, const int32_t* kv_len) {
    if (check_args(B, H, H_kv, N, d)) return 1;
    const int g = H / H_kv;
    int bad = 0;
#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)N);
        if (!srow) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < n_rows; ++r) {
                const int64_t id = rows[r];
                if (id < 0 || id >= (int64_t)B * H * N) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                const int i = (int)(id % N);
                const int h = (int)((id / N) % H);
                const int b = (int)(id / ((int64_t)N * H));
                const int kvl = clamp_len(kv_len, b, N);
                const int kvh = h / g;
                const float* q = Q + (((size_t)b * H + h) * (size_t)N + i) * d;
                const float* k = K + ((size_t)b * H_kv + kvh) * (size_t)N * d;
                const float* v = V + ((size_t)b * H_kv + kvh) * (size_t)N * d;
                double* orow = O_rows + (size_t)r * d;
                for (int j = 0; j < N; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += (double)q[c] * (double)k[(size_t)j * d + c];
                    srow[j] = scale * acc;
                }
                double m = -INFINITY;
                for (int j = 0; j < N; ++j)
                    if (valid_key(i, j, kvl, causal) && srow[j] > m) m = srow[j];
                for (int c = 0; c < d; ++c) orow[c] = 0.0;
                if (m == -INFINITY) {
                    LSE_rows[r] = -INFINITY;
                    continue;
                }
                double l = 0.0;
                for (int j = 0; j < N; ++j) {
                    double p = valid_key(i, j, kvl, causal) ? exp(srow[j] - m) : 0.0;
                    srow[j] = p;
                    l += p;
                }
                for (int j = 0; j < N; ++j) {
                    const double p = srow[j] / l;
                    if (p != 0.0)
                        for (int c = 0; c < d; ++c) orow[c] += p * (double)v[(size_t)j * d + c];
                }
                LSE_rows[r] = m + log(l);
            }
            free(srow);
        }
    }
    return bad;
}

/*
 * Tiled oracle: the online-softmax recurrence over Br x Bc tiles, in fp64. Per query row it keeps
 * the running maximum m, the running sum l and an unnormalised accumulator acc; for each key tile:
 *   m_new = max(m, max_j s_ij);  p_ij = exp(s_ij - m_new);  alpha = exp(m - m_new)
 *   l = alpha * l + sum_j p_ij;  acc = alpha * acc + sum_j p_ij V_j;  m = m_new
 * and at the end O = acc / l, LSE = m + ln l. Exists only to show that the recurrence reaches the
 * full oracle's result; it is not what the GPU is compared with.
 */
int oracle_attn_tiled_f64(const float* Q, const float* K, const float* V, double* O, double* LSE,
                          int B, int H, int H_kv, int N, int d, double scale, int causal,
                          const int32_t* kv_len, int Br, int Bc) {
    if (check_args(B, H, H_kv, N, d) || Br <= 0 || Bc <= 0) return 1;
    const int g = H / H_kv;
    const int n_qblocks = (N + Br - 1) / Br;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int bh = 0; bh < B * H; ++bh) {
        for (int ib = 0; ib < n_qblocks; ++ib) {
            const int b = bh / H, h = bh % H;
            const int kvl = clamp_len(kv_len, b, N);
            const int kvh = h / g;
            const float* q = Q + (size_t)bh * N * d;
            const float* k = K + ((size_t)b * H_kv + kvh) * (size_t)N * d;
            const float* v = V + ((size_t)b * H_kv + kvh) * (size_t)N * d;
            const int i0 = ib * Br, i1 = (i0 + Br < N) ? i0 + Br : N;
            const int rows = i1 - i0;
            double* m = (double*)malloc(sizeof(double) * rows);
            double* l = (double*)malloc(sizeof(double) * rows);
            double* acc = (double*)calloc((size_t)rows * d, sizeof(double));
            double* s = (double*)malloc(sizeof(double) * Bc);
            for (int r = 0; r < rows; ++r) { m[r] = -INFINITY; l[r] = 0.0; }
            for (int j0 = 0; j0 < N; j0 += Bc) {
                const int j1 = (j0 + Bc < N) ? j0 + Bc : N;
                for (int r = 0; r < rows; ++r) {
                    const int i = i0 + r;
                    double mcur = -INFINITY;
                    for (int j = j0; j < j1; ++j) {
                        if (!valid_key(i, j, kvl, causal)) { s[j - j0] = -INFINITY; continue; }
                        double a = 0.0;
                        for (int c = 0; c < d; ++c) a += (double)q[(size_t)i * d + c] * (double)k[(size_t)j * d + c];
                        s[j - j0] = scale * a;
                        if (s[j - j0] > mcur) mcur = s[j - j0];
                    }
                    const double m_new = (mcur > m[r]) ? mcur : m[r];
                    if (m_new == -INFINITY) continue; /* nothing valid yet in this row */
                    const double alpha = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);
                    double psum = 0.0;
                    double* arow = acc + (size_t)r * d;
                    for (int c = 0; c < d; ++c) arow[c] *= alpha;
                    for (int j = j0; j < j1; ++j) {
                        const double p = (s[j - j0] == -INFINITY) ? 0.0 : exp(s[j - j0] - m_new);
                        psum += p;
                        if (p != 0.0)
                            for (int c = 0; c < d; ++c) arow[c] += p * (double)v[(size_t)j * d + c];
                    }
                    l[r] = alpha * l[r] + psum;
                    m[r] = m_new;
                }
            }
            for (int r = 0; r < rows; ++r) {
                double* orow = O + ((size_t)bh * N + i0 + r) * d;
                if (l[r] == 0.0) {
                    for (int c = 0; c < d; ++c) orow[c] = 0.0;
                    LSE[(size_t)bh * N + i0 + r] = -INFINITY;
                } else {
                    for (int c = 0; c < d; ++c) orow[c] = acc[(size_t)r * d + c] / l[r];
                    LSE[(size_t)bh * N + i0 + r] = m[r] + log(l[r]);
                }
            }
            free(m); free(l); free(acc); free(s);
        }
    }
    return 0;
}
