/*
 * FP64 CPU oracle for absorbed (latent) MLA decode over a page_size=1 FP8 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file; only the test suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or constant with the CUDA library: it decodes the
 * FP8 bytes itself, indexes the cache itself and evaluates the plain definition of
 * softmax attention in double precision, one (query row, head) at a time.
 *
 * Sources (page title and section):
 *  - "[Kimi-K3 MLA TP8] MLA performance" (ROCm/aiter issue 4541):
 *      §2 "K3 MLA geometry": one 576-wide latent entry per token (512 latent + 64 rope)
 *         shared by every query head; sm_scale = 1/sqrt(192).
 *      §3 "Entry point": nhead_kv = 1 (single latent KV head), page_size = 1.
 *      §4.1 argument table: q and kv_buffer are float8_e4m3fn, q_scale and kv_scale are
 *         float32 scalars, o is bfloat16 (tokens, heads, 512).
 *      §5.2: page_size = 1, kv_indptr deltas are token counts, kv_last_page_lens all 1,
 *         kv_indices is a per-token row list.
 *  - "Scaling Kimi K3 on AMD Instinct MI355X: Matching NVIDIA HGX B300 Throughput per
 *    GPU on AgentX", §1 "Cache" (DCP): partial answers carry normalisation information
 *    so that a softmax-weighted merge of shards is exact; §4 "MLA": heads attend
 *    independently, so padding heads does not change the real heads.
 *
 * Readings where the pages leave a step open (each is listed with its reason in the
 * design notes of the repository):
 *  - logit = sm_scale * (q_scale * q) . (kv_scale * k) over all 576 columns; V is the
 *    first 512 columns of the same row, dequantised by kv_scale.
 *  - lse is the natural log of the sum of exp(logit) over the attended positions.
 *  - For a request with T query tokens and kv_len L (the step's new entries already in
 *    the cache), query t attends positions j = 0 .. L - T + t.  For T = 1 that is all L.
 *  - An empty attended set gives o = 0 and lse = -inf, and weight 0 in a merge.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MLAO_D 576   /* latent entry width: 512 latent + 64 rope */
#define MLAO_DV 512  /* value width: the latent part of the same entry */

/*
 * float8 e4m3fn ("fn": finite, no infinities) decoded from the format definition:
 * bit 7 sign, bits 6..3 biased exponent (bias 7), bits 2..0 mantissa.  Exponent field 0
 * is subnormal (mantissa/8 * 2^-6); exponent 15 with mantissa 7 is NaN; every other
 * code is normal (1 + mantissa/8) * 2^(exponent-7).  Largest finite value is 448.
 */
double mlao_fp8_e4m3fn(unsigned code) {
    unsigned sign = (code >> 7) & 1u;
    unsigned e = (code >> 3) & 15u;
    unsigned m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return sign ? -mag : mag;
}

void mlao_fp8_table(double* out256) {
    for (unsigned c = 0; c < 256u; ++c) out256[c] = mlao_fp8_e4m3fn(c);
}

/*
 * One query row of one head against an explicit list of attended cache rows.
 *   qvec   : the 576 fp8 bytes of q[r, h, :]
 *   kv     : the cache, row-major, 576 bytes per row
 *   rows   : n_att row ids, in position order
 *   logit_scale = sm_scale * q_scale * kv_scale
 * Writes o[0..511] (fp64) and *lse.  Returns 0, or -1 if a row id is out of
 * [0, n_kv_rows), or -2 on allocation failure.
 */
int mlao_attend_one(const uint8_t* qvec, const uint8_t* kv, int64_t n_kv_rows,
                    const int32_t* rows, int64_t n_att, double logit_scale, double kv_scale,
                    double* o, double* lse) {
    double table[256];
    double qd[MLAO_D];
    double* s;
    double m, z;
    int64_t j;
    int d;

    mlao_fp8_table(table);
    for (d = 0; d < MLAO_DV; ++d) o[d] = 0.0;
    if (n_att <= 0) {
        *lse = -INFINITY;
        return 0;
    }
    for (j = 0; j < n_att; ++j)
        if (rows[j] < 0 || (int64_t)rows[j] >= n_kv_rows) return -1;
    for (d = 0; d < MLAO_D; ++d) qd[d] = table[qvec[d]];

    s = (double*)malloc(sizeof(double) * (size_t)n_att);
    if (!s) return -2;

    /* logits: s_j = logit_scale * sum_d q[d] * k_j[d] over all 576 columns */
    for (j = 0; j < n_att; ++j) {
        const uint8_t* krow = kv + (int64_t)rows[j] * MLAO_D;
        double acc = 0.0;
        for (d = 0; d < MLAO_D; ++d) acc += qd[d] * table[krow[d]];
        s[j] = logit_scale * acc;
    }
    /* softmax normaliser with the maximum taken out */
    m = s[0];
    for (j = 1; j < n_att; ++j)
        if (s[j] > m) m = s[j];
    z = 0.0;
    for (j = 0; j < n_att; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    *lse = m + log(z);
    /* weighted sum of the value part (first 512 columns), dequantised by kv_scale */
    for (j = 0; j < n_att; ++j) {
        const uint8_t* vrow = kv + (int64_t)rows[j] * MLAO_D;
        double w = s[j] / z;
        for (d = 0; d < MLAO_DV; ++d) o[d] += w * table[vrow[d]];
    }
    for (d = 0; d < MLAO_DV; ++d) o[d] *= kv_scale;
    free(s);
    return 0;
}

/*
 * Whole decode call.  q is (sum_T, H, 576) fp8 bytes, contiguous; o is (sum_T, H, 512)
 * fp64; lse is (sum_T, H) fp64.  Request b owns query tokens
 * qo_indptr[b] .. qo_indptr[b+1]-1 and cache positions kv_indptr[b] .. kv_indptr[b+1]-1,
 * whose row ids are kv_indices[kv_indptr[b] + j].
 * Returns 0; -1 on a bad row id; -2 on allocation failure; -3 on kv_len < q_len or a
 * decreasing indptr.
 */
int mlao_decode(const uint8_t* q, int H, const uint8_t* kv, int64_t n_kv_rows,
                const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                int B, double sm_scale, double q_scale, double kv_scale,
                double* o, double* lse, int n_threads) {
    const double logit_scale = sm_scale * q_scale * kv_scale;
    int64_t n_items = 0;
    int status = 0;
    int b;
    int64_t it;
    int64_t* item_row;   /* query row r (token index) of each work item */
    int* item_req;

    for (b = 0; b < B; ++b) {
        int T = qo_indptr[b + 1] - qo_indptr[b];
        int L = kv_indptr[b + 1] - kv_indptr[b];
        if (T < 0 || L < 0 || L < T) return -3;
        n_items += T;
    }
    item_row = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_items > 0 ? n_items : 1));
    item_req = (int*)malloc(sizeof(int) * (size_t)(n_items > 0 ? n_items : 1));
    if (!item_row || !item_req) {
        free(item_row);
        free(item_req);
        return -2;
    }
    it = 0;
    for (b = 0; b < B; ++b)
        for (int r = qo_indptr[b]; r < qo_indptr[b + 1]; ++r) {
            item_row[it] = r;
            item_req[it] = b;
            ++it;
        }

#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) collapse(2) reduction(min : status)
#endif
    for (it = 0; it < n_items; ++it) {
        for (int h = 0; h < H; ++h) {
            int64_t r = item_row[it];
            int bb = item_req[it];
            int T = qo_indptr[bb + 1] - qo_indptr[bb];
            int L = kv_indptr[bb + 1] - kv_indptr[bb];
            int t = (int)(r - qo_indptr[bb]);
            /* positions 0 .. L-T+t are visible to draft token t (all L when T = 1) */
            int64_t n_att = (int64_t)L - T + t + 1;
            const int32_t* rows = kv_indices + kv_indptr[bb];
            int rc = mlao_attend_one(q + (r * H + h) * MLAO_D, kv, n_kv_rows, rows, n_att,
                                     logit_scale, kv_scale, o + (r * H + h) * MLAO_DV,
                                     lse + r * H + h);
            if (rc < status) status = rc;
        }
    }
    (void)n_threads;
    free(item_row);
    free(item_req);
    return status;
}

/*
 * Softmax-weighted merge of P partial results of the same (row, head):
 *   M = max_i lse_i,  w_i = exp(lse_i - M),
 *   o = sum_i w_i o_i / sum_i w_i,  lse = M + log(sum_i w_i).
 * Partials with lse = -inf carry weight 0; if all are -inf the result is o = 0,
 * lse = -inf.  o_parts is (P, width), row-major.
 */
void mlao_merge(const double* o_parts, const double* lse_parts, int P, int64_t width,
                double* o, double* lse) {
    double M = -INFINITY, wsum = 0.0;
    int i;
    int64_t c;
    for (c = 0; c < width; ++c) o[c] = 0.0;
    for (i = 0; i < P; ++i)
        if (lse_parts[i] > M) M = lse_parts[i];
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    for (i = 0; i < P; ++i) {
        double w;
        if (lse_parts[i] == -INFINITY) continue;
        w = exp(lse_parts[i] - M);
        wsum += w;
        for (c = 0; c < width; ++c) o[c] += w * o_parts[(int64_t)i * width + c];
    }
    for (c = 0; c < width; ++c) o[c] /= wsum;
    *lse = M + log(wsum);
}

int mlao_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
