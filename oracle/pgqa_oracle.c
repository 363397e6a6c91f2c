/*
 * pgqa_oracle.c -- plain, slow, float64 CPU oracle for ragged and paged GQA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this
 * file: only the test-suite, the package smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes is the definition of softmax attention, written out row by row:
 *
 *   For request b, query head h and query row i (0 <= i < qo_len_b):
 *     g          = h / (Hq / Hk)                 (consecutive query heads share a KV head)
 *     allowed(j) = j < kv_len_b  and  (!causal or j <= i + kv_len_b - qo_len_b)
 *     s_j        = sm_scale * sum_c q[i,h,c] * k[j,g,c]              (allowed j only)
 *     m          = max_j s_j,   Z = sum_j exp(s_j - m)
 *     o[i,h,:]   = sum_j exp(s_j - m) / Z * v[j,g,:]
 *     lse[i,h]   = m + ln Z                       (natural log of sum_j exp(s_j))
 *     no allowed key:  o = 0 exactly, lse = -inf
 *
 * Sources (restated, not copied):
 *  - Atlas "Module flashinfer" API page, items ragged_prefill_bf16_hd128 / _hd256:
 *    one batched varlen launch addressed by q_indptr / kv_indptr, bf16, GQA,
 *    head_dim 128 and 256, causal selectable.
 *  - FlashInfer documentation, flashinfer_benchmark.py "Attention Flags" (--causal):
 *    bottom-right causal alignment, i.e. the last query row sees every key.
 *  - FlashInfer documentation, flashinfer.prefill / flashinfer.decode ("forward_return_lse",
 *    "single_prefill_with_kv_cache_return_lse"): the log-sum-exp output; its base is not
 *    stated there, this oracle uses the natural log over scaled scores.
 *  - vllm-rlt pull request "feat: add FlashInfer attention backend for SM120 decode",
 *    Scope / Design notes: paged decode over an NHD block table (kv_layout "NHD"),
 *    one query token per request, zero-length rows give exact zeros.
 *  - FlashInfer documentation, flashinfer.cascade, "Merge Attention States"
 *    (merge_state / merge_states): combining partial (output, lse) pairs.
 *
 * Inputs are raw bf16 bit patterns (uint16); widening bf16 to double is exact.
 * Floating point contraction is disabled at build time (-ffp-contract=off) so the x86
 * and Arm builds round identically.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper 16 bits of an IEEE-754 binary32 value. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Softmax attention of one query row over n keys (the allowed prefix 0..n-1).
 * krows[j] / vrows[j] point at the d bf16 values of key j / value j.
 * s is caller scratch of at least n doubles.
 */
static void attend_row(const uint16_t* qrow, const uint16_t* const* krows,
                       const uint16_t* const* vrows, long n, int d, double sm_scale,
                       double* s, double* o, double* lse) {
    int c;
    long j;
    if (n <= 0) {
        for (c = 0; c < d; ++c) o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (j = 0; j < n; ++j) {
        double dot = 0.0;
        for (c = 0; c < d; ++c) dot += bf16_to_double(qrow[c]) * bf16_to_double(krows[j][c]);
        s[j] = sm_scale * dot;
        if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    for (c = 0; c < d; ++c) o[c] = 0.0;
    for (j = 0; j < n; ++j) {
        double w = s[j] / z;
        for (c = 0; c < d; ++c) o[c] += w * bf16_to_double(vrows[j][c]);
    }
    *lse = m + log(z);
}

/* number of allowed keys (a prefix) for query row i of a request */
static long allowed_keys(long i, long qo_len, long kv_len, int causal) {
    if (!causal) return kv_len;
    long n = i + kv_len - qo_len + 1;
    if (n < 0) n = 0;
    if (n > kv_len) n = kv_len;
    return n;
}

/* request index b with indptr[b] <= t < indptr[b+1]; -1 when t is outside every request */
static int find_request(const int32_t* indptr, int batch, long t) {
    int lo = 0, hi = batch - 1;
    while (lo <= hi) {
        int mid = (lo + hi) / 2;
        if (t < indptr[mid]) hi = mid - 1;
        else if (t >= indptr[mid + 1]) lo = mid + 1;
        else return mid;
    }
    return -1;
}

static int pick_threads(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * Ragged (packed NHD) attention.
 *   q [total_q, Hq, d], k / v [total_kv, Hk, d]  (bf16 bits)
 *   q_indptr / kv_indptr [batch + 1]: request b owns q rows q_indptr[b]..q_indptr[b+1]-1
 *   and kv rows kv_indptr[b]..kv_indptr[b+1]-1.
 *   rows [n_rows]: which outputs to compute, each encoded t * Hq + h with t a global
 *   query row; o [n_rows, d] and lse [n_rows] receive them in that order.
 * Returns 0, or -1 on an argument error (a row outside every request, bad heads).
 */
int pgqa_oracle_ragged(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* q_indptr, const int32_t* kv_indptr, int batch,
                       int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                       double sm_scale, const int64_t* rows, long n_rows,
                       double* o, double* lse, int nthreads) {
    if (batch <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0 || head_dim <= 0)
        return -1;
    const int group = num_qo_heads / num_kv_heads;
    long max_kv = 0;
    for (int b = 0; b < batch; ++b) {
        long n = (long)kv_indptr[b + 1] - kv_indptr[b];
        if (n > max_kv) max_kv = n;
    }
    int bad = 0;
#pragma omp parallel num_threads(pick_threads(nthreads)) reduction(| : bad)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
        const uint16_t** kr = (const uint16_t**)malloc(sizeof(void*) * (size_t)(max_kv > 0 ? max_kv : 1));
        const uint16_t** vr = (const uint16_t**)malloc(sizeof(void*) * (size_t)(max_kv > 0 ? max_kv : 1));
        long r;
#pragma omp for schedule(dynamic, 4)
        for (r = 0; r < n_rows; ++r) {
            long t = (long)(rows[r] / num_qo_heads);
            int h = (int)(rows[r] % num_qo_heads);
            int b = find_request(q_indptr, batch, t);
            if (b < 0) { bad = 1; continue; }
            long i = t - q_indptr[b];
            long qo_len = (long)q_indptr[b + 1] - q_indptr[b];
            long kv_len = (long)kv_indptr[b + 1] - kv_indptr[b];
            int g = h / group;
            long n = allowed_keys(i, qo_len, kv_len, causal);
            for (long j = 0; j < n; ++j) {
                long kv_row = (long)kv_indptr[b] + j;
                kr[j] = k + ((size_t)kv_row * num_kv_heads + g) * head_dim;
                vr[j] = v + ((size_t)kv_row * num_kv_heads + g) * head_dim;
            }
            attend_row(q + ((size_t)t * num_qo_heads + h) * head_dim, kr, vr, n, head_dim,
                       sm_scale, s, o + (size_t)r * head_dim, lse + r);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return bad ? -1 : 0;
}

/*
 * Attention over a paged NHD KV cache.
 *   q [total_q, Hq, d] with q_indptr [batch + 1] (decode: q_indptr = 0,1,...,batch)
 *   k_pages / v_pages [num_pages, page_size, Hk, d]
 *   page_table [batch, page_table_stride]: key j of request b lives in page
 *   page_table[b * stride + j / page_size], slot j % page_size.  Entries past the
 *   request's last page are never read.
 *   kv_lens [batch].
 *   rows, o, lse: as for pgqa_oracle_ragged.
 * Returns 0, or -1 on an argument error (including a page id outside 0..num_pages-1).
 */
int pgqa_oracle_paged(const uint16_t* q, const int32_t* q_indptr, const uint16_t* k_pages,
                      const uint16_t* v_pages, const int32_t* page_table, int page_table_stride,
                      const int32_t* kv_lens, int page_size, long num_pages, int batch,
                      int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                      double sm_scale, const int64_t* rows, long n_rows, double* o,
                      double* lse, int nthreads) {
    if (batch <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0 || head_dim <= 0 ||
        page_size <= 0)
        return -1;
    const int group = num_qo_heads / num_kv_heads;
    long max_kv = 0;
    for (int b = 0; b < batch; ++b)
        if (kv_lens[b] > max_kv) max_kv = kv_lens[b];
    int bad = 0;
#pragma omp parallel num_threads(pick_threads(nthreads)) reduction(| : bad)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
        const uint16_t** kr = (const uint16_t**)malloc(sizeof(void*) * (size_t)(max_kv > 0 ? max_kv : 1));
        const uint16_t** vr = (const uint16_t**)malloc(sizeof(void*) * (size_t)(max_kv > 0 ? max_kv : 1));
        long r;
#pragma omp for schedule(dynamic, 4)
        for (r = 0; r < n_rows; ++r) {
            long t = (long)(rows[r] / num_qo_heads);
            int h = (int)(rows[r] % num_qo_heads);
            int b = find_request(q_indptr, batch, t);
            if (b < 0) { bad = 1; continue; }
            long i = t - q_indptr[b];
            long qo_len = (long)q_indptr[b + 1] - q_indptr[b];
            long kv_len = kv_lens[b];
            int g = h / group;
            long n = allowed_keys(i, qo_len, kv_len, causal);
            int row_bad = 0;
            for (long j = 0; j < n; ++j) {
                long page = page_table[(size_t)b * page_table_stride + j / page_size];
                if (page < 0 || page >= num_pages) { row_bad = 1; break; }
                size_t off = (((size_t)page * page_size + (size_t)(j % page_size)) * num_kv_heads + g) * head_dim;
                kr[j] = k_pages + off;
                vr[j] = v_pages + off;
            }
            if (row_bad) { bad = 1; continue; }
            attend_row(q + ((size_t)t * num_qo_heads + h) * head_dim, kr, vr, n, head_dim,
                       sm_scale, s, o + (size_t)r * head_dim, lse + r);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return bad ? -1 : 0;
}

/*
 * OCP 8-bit floating point E4M3 in its "fn" form (no infinities), decoded from the
 * format's definition: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 *   exponent 1..15: (-1)^s * 2^(e-7) * (1 + m/8)      (largest finite: 2^8 * 1.75 = 448)
 *   exponent 0:     (-1)^s * 2^(1-7) * (m/8)           (subnormals; m = 0 is a signed zero)
 *   S.1111.111:     NaN
 * The KV-cache dtype fp8_e4m3 is listed by FlashInfer documentation,
 * flashinfer_benchmark.py "Attention Flags" (--kv_dtype).
 */
static double e4m3_to_double(uint8_t bits) {
    const int sign = bits >> 7;
    const int e = (bits >> 3) & 15;
    const int m = bits & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, 1 - 7);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* decode n E4M3 bytes */
void pgqa_oracle_e4m3_decode(const uint8_t* in, long n, double* out) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_to_double(in[i]);
}

/*
 * Softmax attention of one query row over n keys stored as E4M3 bytes with one scale for
 * all keys and one for all values: key element = e4m3 * k_scale, value element =
 * e4m3 * v_scale.  krows[j] / vrows[j] point at the d bytes of key / value j.
 */
static void attend_row_e4m3(const uint16_t* qrow, const uint8_t* const* krows,
                            const uint8_t* const* vrows, long n, int d, double k_scale,
                            double v_scale, double sm_scale, double* s, double* o, double* lse) {
    int c;
    long j;
    if (n <= 0) {
        for (c = 0; c < d; ++c) o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (j = 0; j < n; ++j) {
        double dot = 0.0;
        for (c = 0; c < d; ++c)
            dot += bf16_to_double(qrow[c]) * (e4m3_to_double(krows[j][c]) * k_scale);
        s[j] = sm_scale * dot;
        if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    for (c = 0; c < d; ++c) o[c] = 0.0;
    for (j = 0; j < n; ++j) {
        double w = s[j] / z;
        for (c = 0; c < d; ++c) o[c] += w * (e4m3_to_double(vrows[j][c]) * v_scale);
    }
    *lse = m + log(z);
}

/*
 * Attention over a paged NHD KV cache held as E4M3 bytes with per-tensor scales
 * (k_scale for every key element, v_scale for every value element).  Arguments as for
 * pgqa_oracle_paged, with k_pages / v_pages holding one byte per element.
 */
int pgqa_oracle_paged_e4m3(const uint16_t* q, const int32_t* q_indptr, const uint8_t* k_pages,
                           const uint8_t* v_pages, double k_scale, double v_scale,
                           const int32_t* page_table, int page_table_stride,
                           const int32_t* kv_lens, int page_size, long num_pages, int batch,
                           int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                           double sm_scale, const int64_t* rows, long n_rows, double* o,
                           double* lse, int nthreads) {
    if (batch <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0 || head_dim <= 0 ||
        page_size <= 0)
        return -1;
    const int group = num_qo_heads / num_kv_heads;
    long max_kv = 0;
    for (int b = 0; b < batch; ++b)
        if (kv_lens[b] > max_kv) max_kv = kv_lens[b];
    int bad = 0;
#pragma omp parallel num_threads(pick_threads(nthreads)) reduction(| : bad)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
        const uint8_t** kr = (const uint8_t**)malloc(sizeof(void*) * (size_t)(max_kv > 0 ? max_kv : 1));
        const uint8_t** vr = (const uint8_t**)malloc(sizeof(void*) * (size_t)(max_kv > 0 ? max_kv : 1));
        long r;
#pragma omp for schedule(dynamic, 4)
        for (r = 0; r < n_rows; ++r) {
            long t = (long)(rows[r] / num_qo_heads);
            int h = (int)(rows[r] % num_qo_heads);
            int b = find_request(q_indptr, batch, t);
            if (b < 0) { bad = 1; continue; }
            long i = t - q_indptr[b];
            long qo_len = (long)q_indptr[b + 1] - q_indptr[b];
            long kv_len = kv_lens[b];
            int g = h / group;
            long n = allowed_keys(i, qo_len, kv_len, causal);
            int row_bad = 0;
            for (long j = 0; j < n; ++j) {
                long page = page_table[(size_t)b * page_table_stride + j / page_size];
                if (page < 0 || page >= num_pages) { row_bad = 1; break; }
                size_t off = (((size_t)page * page_size + (size_t)(j % page_size)) * num_kv_heads + g) * head_dim;
                kr[j] = k_pages + off;
                vr[j] = v_pages + off;
            }
            if (row_bad) { bad = 1; continue; }
            attend_row_e4m3(q + ((size_t)t * num_qo_heads + h) * head_dim, kr, vr, n, head_dim,
                            k_scale, v_scale, sm_scale, s, o + (size_t)r * head_dim, lse + r);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return bad ? -1 : 0;
}

/*
 * Merge of attention states (FlashInfer documentation, flashinfer.cascade,
 * "Merge Attention States"): given n_states partial results of the same rows over
 * disjoint key sets, v [n_states, n_rows, d] (each normalised over its own keys) and
 * s [n_states, n_rows] (natural-log LSE of its keys), the result over the union is
 *     S = ln sum_c exp(s_c),   V = sum_c exp(s_c - S) * v_c .
 * A state with s_c = -inf (no keys) contributes nothing; all -inf gives V = 0, S = -inf.
 */
void pgqa_oracle_merge_states(const double* v, const double* s, int n_states, long n_rows,
                              int head_dim, double* v_out, double* s_out) {
    for (long r = 0; r < n_rows; ++r) {
        double m = -INFINITY;
        for (int c = 0; c < n_states; ++c) {
            double x = s[(size_t)c * n_rows + r];
            if (x > m) m = x;
        }
        double* vo = v_out + (size_t)r * head_dim;
        for (int e = 0; e < head_dim; ++e) vo[e] = 0.0;
        if (m == -INFINITY) {
            s_out[r] = -INFINITY;
            continue;
        }
        double z = 0.0;
        for (int c = 0; c < n_states; ++c) z += exp(s[(size_t)c * n_rows + r] - m);
        for (int c = 0; c < n_states; ++c) {
            double w = exp(s[(size_t)c * n_rows + r] - m) / z;
            const double* vc = v + ((size_t)c * n_rows + r) * head_dim;
            for (int e = 0; e < head_dim; ++e) vo[e] += w * vc[e];
        }
        s_out[r] = m + log(z);
    }
}

int pgqa_oracle_threads(void) { return pick_threads(0); }
