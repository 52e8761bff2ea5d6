/*
 * rkv_oracle.c -- plain, slow CPU oracle for resident attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this file; only the
 * test suite, the smoke check and the CPU-baseline leg of the benchmark load
 * it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (all three reference pages agree on the math):
 *   output = softmax(Q . K^T * scale) . V          per query head
 *   - trueno-gpu 0.4.11, src/memory/resident/attention.rs,
 *     fn batched_multihead_attention (doc comment: "Computes: output =
 *     softmax(Q @ K^T / sqrt(d_k)) @ V", scale = 1/sqrt(head_dim)).
 *   - trustformers-core 0.2.0, src/gpu_ops/cuda/oxicuda/attention.rs,
 *     fn attention_prefill_gpu_to_gpu (causal: query i sees keys 0..=i) and
 *     fn attention_decode_gpu_to_gpu (one query, no mask).
 *   - the same page, mod gpu_tests, fn prefill_reference: naive loop,
 *     max-subtracted exponentials, normalised by the sum.
 *   - realizar 0.8.5, src/cuda/executor/cache_from_cache_from_kv_cache.rs,
 *     fn init_kv_cache_gpu / init_batched_kv_cache_gpu: GQA cache
 *     [num_kv_heads, max_len, head_dim], batched [M, num_kv_heads, max_len,
 *     head_dim].
 *   - trueno-gpu page, fn kv_cache_scatter_gpu: interleaved row -> cache[h,pos,:].
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   GQA map g(h) = h / (H/Hk) (consecutive grouping); an empty key set gives a
 *   zero row (trueno-gpu incremental_attention_gpu returns zeros for
 *   seq_len == 0); query rows at or past a sequence's valid length are zero.
 *
 * Precision: inputs are f32, every product, sum and exponential is computed
 * in double, and results are returned as double.  The softmax is the two-pass
 * max-subtracted form written out, not an online one.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* q head -> kv head, consecutive grouping (G = H / Hk query heads per kv head). */
static int kv_head_of(int h, int H, int Hk) { return h / (H / Hk); }

/*
 * One query row against a key set {0 .. n_keys-1}:
 *   s_j = (sum_d q[d] * k_j[d]) * scale
 *   p_j = exp(s_j - max s) / sum_j exp(s_j - max s)
 *   out = sum_j p_j * v_j
 * k_j = k_base + j*k_stride, v_j likewise.  n_keys == 0 -> zero row.
 * scores: caller-provided scratch of n_keys doubles.  If probs != NULL the
 * normalised probabilities are written there as well.
 */
static void attend_row(const float* q, const float* k_base, const float* v_base,
                       int64_t k_stride, int64_t v_stride, int n_keys, int D,
                       double scale, double* scores, double* out, double* probs)
{
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n_keys <= 0) return;

    /* pass 1: scores and their maximum */
    double smax = -INFINITY;
    for (int j = 0; j < n_keys; ++j) {
        const float* kj = k_base + (int64_t)j * k_stride;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += (double)q[d] * (double)kj[d];
        scores[j] = acc * scale;
        if (scores[j] > smax) smax = scores[j];
    }
    /* pass 2: exponentials and their sum */
    double sum = 0.0;
    for (int j = 0; j < n_keys; ++j) {
        scores[j] = exp(scores[j] - smax);
        sum += scores[j];
    }
    /* normalise and mix the values */
    for (int j = 0; j < n_keys; ++j) {
        double p = scores[j] / sum;
        if (probs) probs[j] = p;
        const float* vj = v_base + (int64_t)j * v_stride;
        for (int d = 0; d < D; ++d) out[d] += p * (double)vj[d];
    }
}

/* number of keys query i of a sequence of valid length len may see */
static int prefill_key_count(int i, int len, int causal)
{
    if (i >= len) return 0;          /* padded query row -> zero output */
    return causal ? i + 1 : len;     /* causal: keys 0..=i */
}

int rkv_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Prefill over interleaved activations.
 *   q, o : [B, S, H*D]      k, v : [B, S, Hk*D]     (row-major f32 / f64)
 *   seq_lens : int[B] valid lengths (<= S), or NULL for all S.
 * Returns 0, or -1 on invalid shapes.
 */
int rkv_oracle_prefill(const float* q, const float* k, const float* v, double* o,
                       int B, int S, int H, int Hk, int D, int causal,
                       const int* seq_lens, double scale)
{
    if (B < 0 || S < 0 || H <= 0 || Hk <= 0 || D <= 0 || H % Hk != 0) return -1;
    const int64_t q_row = (int64_t)H * D, kv_row = (int64_t)Hk * D;
    const int64_t n_rows = (int64_t)B * H * S;
    int rc = 0;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
        if (!scores) {
#pragma omp atomic write
            rc = -1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (!scores) continue;
            const int b = (int)(r / ((int64_t)H * S));
            const int h = (int)((r / S) % H);
            const int i = (int)(r % S);
            int len = seq_lens ? seq_lens[b] : S;
            if (len > S) len = S;
            if (len < 0) len = 0;
            const int g = kv_head_of(h, H, Hk);
            const float* qi = q + ((int64_t)b * S + i) * q_row + (int64_t)h * D;
            const float* kb = k + (int64_t)b * S * kv_row + (int64_t)g * D;
            const float* vb = v + (int64_t)b * S * kv_row + (int64_t)g * D;
            double* oi = o + ((int64_t)b * S + i) * q_row + (int64_t)h * D;
            attend_row(qi, kb, vb, kv_row, kv_row, prefill_key_count(i, len, causal), D,
                       scale, scores, oi, NULL);
        }
        free(scores);
    }
    return rc;
}

/*
 * Prefill for a sample of output rows only (for sizes too large to run whole).
 * rows[n] holds flat row ids ((b*H + h)*S + i); out is [n, D] double.
 */
int rkv_oracle_prefill_rows(const float* q, const float* k, const float* v,
                            int B, int S, int H, int Hk, int D, int causal,
                            const int* seq_lens, double scale,
                            const int64_t* rows, int64_t n, double* out)
{
    if (B < 0 || S < 0 || H <= 0 || Hk <= 0 || D <= 0 || H % Hk != 0) return -1;
    const int64_t q_row = (int64_t)H * D, kv_row = (int64_t)Hk * D;
    const int64_t total = (int64_t)B * H * S;
    int rc = 0;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n; ++t) {
            const int64_t r = rows[t];
            if (!scores || r < 0 || r >= total) {
#pragma omp atomic write
                rc = -1;
                continue;
            }
            const int b = (int)(r / ((int64_t)H * S));
            const int h = (int)((r / S) % H);
            const int i = (int)(r % S);
            int len = seq_lens ? seq_lens[b] : S;
            if (len > S) len = S;
            if (len < 0) len = 0;
            const int g = kv_head_of(h, H, Hk);
            const float* qi = q + ((int64_t)b * S + i) * q_row + (int64_t)h * D;
            const float* kb = k + (int64_t)b * S * kv_row + (int64_t)g * D;
            const float* vb = v + (int64_t)b * S * kv_row + (int64_t)g * D;
            attend_row(qi, kb, vb, kv_row, kv_row, prefill_key_count(i, len, causal), D,
                       scale, scores, out + t * D, NULL);
        }
        free(scores);
    }
    return rc;
}

/*
 * Probability row of one prefill query (b, h, i): probs[S] double, keys that
 * the query does not see are 0.  Used to check that each row sums to 1.
 */
int rkv_oracle_prefill_probs(const float* q, const float* k, const float* v,
                             int B, int S, int H, int Hk, int D, int causal,
                             const int* seq_lens, double scale,
                             int b, int h, int i, double* probs)
{
    if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= S || H % Hk != 0) return -1;
    const int64_t q_row = (int64_t)H * D, kv_row = (int64_t)Hk * D;
    int len = seq_lens ? seq_lens[b] : S;
    if (len > S) len = S;
    if (len < 0) len = 0;
    const int g = kv_head_of(h, H, Hk);
    double* scores = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double* tmp = (double*)malloc(sizeof(double) * (size_t)D);
    if (!scores || !tmp) { free(scores); free(tmp); return -1; }
    for (int j = 0; j < S; ++j) probs[j] = 0.0;
    attend_row(q + ((int64_t)b * S + i) * q_row + (int64_t)h * D,
               k + (int64_t)b * S * kv_row + (int64_t)g * D,
               v + (int64_t)b * S * kv_row + (int64_t)g * D,
               kv_row, kv_row, prefill_key_count(i, len, causal), D, scale, scores, tmp, probs);
    free(scores);
    free(tmp);
    return 0;
}

/*
 * Decode: one query token per sequence against the batched cache.
 *   q, o       : [M, H*D]
 *   k_c, v_c   : [M, Hk, Lmax, D]
 *   seq_lens   : int[M], rows 0..len-1 are attended (no mask); len <= 0 -> zeros.
 * Returns -1 if any len > Lmax (the pages reject seq_len > max_seq_len).
 */
int rkv_oracle_decode(const float* q, const float* k_c, const float* v_c, double* o,
                      int M, int H, int Hk, int D, int Lmax, const int* seq_lens,
                      double scale)
{
    if (M < 0 || H <= 0 || Hk <= 0 || D <= 0 || Lmax <= 0 || H % Hk != 0) return -1;
    for (int m = 0; m < M; ++m)
        if (seq_lens[m] > Lmax) return -1;
    const int64_t n_rows = (int64_t)M * H;
    int rc = 0;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)Lmax);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (!scores) {
#pragma omp atomic write
                rc = -1;
                continue;
            }
            const int m = (int)(r / H), h = (int)(r % H);
            const int g = kv_head_of(h, H, Hk);
            const int64_t head_base = (((int64_t)m * Hk + g) * Lmax) * D;
            attend_row(q + r * D, k_c + head_base, v_c + head_base, D, D,
                       seq_lens[m] > 0 ? seq_lens[m] : 0, D, scale, scores, o + r * D, NULL);
        }
        free(scores);
    }
    return rc;
}

/*
 * Scatter: cache[m, kh, start_pos[m] + t, :] = new[m, t, kh*D : (kh+1)*D]
 * for K and V alike.  Tokens whose target row falls outside [0, Lmax) are
 * skipped and counted once each in *overflow (if not NULL).
 */
int rkv_oracle_scatter(const float* k_new, const float* v_new, float* k_c, float* v_c,
                       int M, int T, int Hk, int D, int Lmax, const int* start_pos,
                       int* overflow)
{
    if (M < 0 || T < 0 || Hk <= 0 || D <= 0 || Lmax <= 0) return -1;
    int skipped = 0;
    for (int m = 0; m < M; ++m) {
        for (int t = 0; t < T; ++t) {
            const int64_t pos = (int64_t)start_pos[m] + t;
            if (pos < 0 || pos >= Lmax) { ++skipped; continue; }
            for (int kh = 0; kh < Hk; ++kh) {
                const int64_t src = ((int64_t)m * T + t) * Hk * D + (int64_t)kh * D;
                const int64_t dst = (((int64_t)m * Hk + kh) * Lmax + pos) * D;
                for (int d = 0; d < D; ++d) {
                    k_c[dst + d] = k_new[src + d];
                    v_c[dst + d] = v_new[src + d];
                }
            }
        }
    }
    if (overflow) *overflow += skipped;
    return 0;
}

/*
 * Prefill appended behind rows already in the batched cache (chunked prefill).
 *
 * trustformers-core attention.rs, fn attention_prefill_gpu_to_gpu states that
 * its causal mask is the from-empty-cache one and that a prefill appended to
 * an existing cache must instead run the decode path once per token
 * (fn attention_decode_gpu_to_gpu: one query against every cached row, no
 * mask).  That per-token rule is what this function computes, for a chunk of
 * T query tokens whose own K/V rows are already in the cache:
 *   query i of sequence b sits at position p0 = start_pos[b] plus i and, like
 *   a decode step of length p0 + i + 1, sees cache rows 0 .. p0+i (causal);
 *   non-causal, every valid query sees rows 0 .. p0+n-1.
 *   q, o      : [B, T, H*D]
 *   k_c, v_c  : [B, Hk, Lmax, D]
 *   start_pos : int[B], rows in the cache before the chunk
 *   q_lens    : int[B] valid query rows n of the chunk (<= T), or NULL for T;
 *               rows i >= n are zero.
 * Returns -1 on invalid shapes, a negative start or p0 + n > Lmax.
 */
int rkv_oracle_prefill_cached(const float* q, const float* k_c, const float* v_c, double* o,
                              int B, int T, int H, int Hk, int D, int Lmax, int causal,
                              const int* start_pos, const int* q_lens, double scale)
{
    if (B < 0 || T < 0 || H <= 0 || Hk <= 0 || D <= 0 || Lmax <= 0 || H % Hk != 0) return -1;
    for (int b = 0; b < B; ++b) {
        const int n = q_lens ? q_lens[b] : T;
        if (start_pos[b] < 0 || n < 0 || n > T || (int64_t)start_pos[b] + n > Lmax) return -1;
    }
    const int64_t q_row = (int64_t)H * D;
    const int64_t n_rows = (int64_t)B * H * T;
    int rc = 0;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)Lmax);
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (!scores) {
#pragma omp atomic write
                rc = -1;
                continue;
            }
            const int b = (int)(r / ((int64_t)H * T));
            const int h = (int)((r / T) % H);
            const int i = (int)(r % T);
            const int p0 = start_pos[b];
            const int n = q_lens ? q_lens[b] : T;
            int n_keys = 0;                       /* padded query row -> zero output */
            if (i < n) n_keys = causal ? p0 + i + 1 : p0 + n;
            const int g = kv_head_of(h, H, Hk);
            const int64_t head_base = (((int64_t)b * Hk + g) * Lmax) * D;
            const int64_t at = ((int64_t)b * T + i) * q_row + (int64_t)h * D;
            attend_row(q + at, k_c + head_base, v_c + head_base, D, D, n_keys, D, scale, scores,
                       o + at, NULL);
        }
        free(scores);
    }
    return rc;
}

/*
 * Rotary position embedding, GPT-NeoX half-split form, at explicit positions.
 *
 * trustformers-core attention.rs, fn rope_neox_gpu_to_gpu (partial RoPE over the
 * first rotary_ndims of each head, half-split pairs, position offset = absolute
 * position of the first row) and realizar cache_from_cache_from_kv_cache.rs,
 * fn apply_rope_to_buffer (NEOX split halves: pair (i, i + half), frequency
 * 1 / theta^(2i / dim), angle = position * frequency, x1' = x1 cos - x2 sin,
 * x2' = x1 sin + x2 cos).  With r = rotary_ndims (r = head_dim on the realizar
 * page), pair i < r/2 joins dims i and i + r/2 and turns by
 *     angle = pos * theta^(-2i / r);
 * dims r..head_dim-1 pass through unchanged.
 *   x, out    : [n_rows, n_heads * head_dim]  (out in double)
 *   positions : int[n_rows], the absolute position of each row
 * Returns -1 on invalid shapes (r odd, r > head_dim, theta <= 0).
 */
int rkv_oracle_rope(const float* x, double* out, int64_t n_rows, int n_heads, int head_dim,
                    int rotary_ndims, const int* positions, double theta)
{
    if (n_rows < 0 || n_heads <= 0 || head_dim <= 0 || rotary_ndims < 0 || rotary_ndims % 2 != 0 ||
        rotary_ndims > head_dim || !(theta > 0.0))
        return -1;
    const int half = rotary_ndims / 2;
    for (int64_t row = 0; row < n_rows; ++row) {
        const double pos = (double)positions[row];
        for (int h = 0; h < n_heads; ++h) {
            const float* xh = x + (row * n_heads + h) * (int64_t)head_dim;
            double* oh = out + (row * n_heads + h) * (int64_t)head_dim;
            for (int d = 0; d < head_dim; ++d) oh[d] = (double)xh[d];
            for (int i = 0; i < half; ++i) {
                const double angle = pos * pow(theta, -2.0 * (double)i / (double)rotary_ndims);
                const double c = cos(angle), s = sin(angle);
                const double x1 = (double)xh[i], x2 = (double)xh[i + half];
                oh[i] = x1 * c - x2 * s;
                oh[i + half] = x1 * s + x2 * c;
            }
        }
    }
    return 0;
}
