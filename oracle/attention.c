/*
 * ORACLE — test infrastructure only.  Plain, slow, fp64 CPU restatement of
 * paged decode attention.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library; the product path never does.
 * It shares no code with the CUDA path.
 *
 * What it computes, in the order the sources give it:
 *
 *  1. Append ("Incremental Serving", section "Request flow", step 2; section
 *     "Paged KV-cache layout"): the new key/value row of request b, head h is
 *     stored verbatim (storage dtype bytes) at logical position t_b - 1, i.e.
 *     physical page table_b[(t_b - 1) / P], slot (t_b - 1) % P, of the pools
 *     laid out [physical_page, head, page_offset, head_width].
 *
 *  2. Gather: key j (0 <= j < t_b) of (b, h) is
 *     K[table_b[j / P], h, j % P, :], converted exactly to fp64; same for V
 *     ("Incremental Serving", "Paged KV-cache layout": the logical page table
 *     maps logical page i to a physical page).
 *
 *  3. Scores over the prefix that includes the new key ("38 · Cached
 *     generation", section "Prepare every block, then commit every cache
 *     together", function incremental_mixture: prefix = len + 1, score =
 *     dot(q, k) * 1/sqrt(d_h)).
 *
 *  4. Stable softmax over the t_b scores (same function: softmax along the key
 *     axis; "stable softmax" in its doc comment): subtract the maximum,
 *     exponentiate, divide by the sum.
 *
 *  5. Weighted sum of the value rows, per feature (same function, the
 *     mixture loop).
 *
 * t_b counts the new token ("38 · Cached generation", section "Keep retained
 * length and final length separate": t is the number of keys read by the one
 * newest cached query).  q is fp32, widened to fp64.  Output is fp64.
 *
 * Grouped-query attention ("Rollout Serving, Caching, and Batching", KV-cache
 * memory formula: grouped-query or multi-query attention has fewer KV heads
 * than query heads): with `group` query heads per KV head, query head qh reads
 * the keys and values of KV head qh / group.  group = 1 is ordinary multi-head
 * attention.
 *
 * Sliding window (same page: a fixed window of W positions gives O(TW)
 * attention arithmetic): with window W > 0 the newest query attends to the
 * keys at positions max(0, t - W) .. t - 1 only; W = 0 means the whole prefix.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };

static double load_elem(const void* base, int64_t idx, int dtype) {
    if (dtype == ORC_F32) return (double)((const float*)base)[idx];
    uint32_t u = (uint32_t)((const uint16_t*)base)[idx] << 16;   /* bf16 is the top half of fp32 */
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Element offset of (page, head, slot, 0) in a [pages][H][P][D] pool. */
static int64_t pool_offset(int64_t page, int64_t head, int64_t slot, int H, int P, int D) {
    return ((page * H + head) * P + slot) * (int64_t)D;
}

/*
 * Step 1 for every request: write k_new / v_new rows into slot t_b - 1.
 * Returns 0, or -1 if a length or page id is out of range (nothing written
 * for that request).
 */
int orc_append(int B, int H, int D, int P, int dtype, void* k_pool, void* v_pool, int64_t n_pages,
               const void* k_new, const void* v_new, const int32_t* tables, int max_pages,
               const int32_t* seq_lens) {
    int es = dtype == ORC_F32 ? 4 : 2;
    int rc = 0;
    for (int b = 0; b < B; ++b) {
        int64_t pos = (int64_t)seq_lens[b] - 1;
        if (pos < 0 || pos / P >= max_pages) { rc = -1; continue; }
        int64_t page = tables[(int64_t)b * max_pages + pos / P];
        if (page < 0 || page >= n_pages) { rc = -1; continue; }
        for (int h = 0; h < H; ++h) {
            int64_t dst = pool_offset(page, h, pos % P, H, P, D);
            int64_t src = ((int64_t)b * H + h) * D;
            memcpy((char*)k_pool + dst * es, (const char*)k_new + src * es, (size_t)D * es);
            memcpy((char*)v_pool + dst * es, (const char*)v_new + src * es, (size_t)D * es);
        }
    }
    return rc;
}

/*
 * Steps 2-5 for one (request, head) lane whose t keys are already in the pool.
 * scores: caller scratch of t doubles.
 */
static int lane_attention(int H, int D, int P, int dtype, const void* k_pool, const void* v_pool,
                          int64_t n_pages, const float* q, const int32_t* table, int64_t t, int h,
                          int64_t window, double* scores, double* out) {
    const double scale = 1.0 / sqrt((double)D);
    const int64_t j0 = (window > 0 && t > window) ? t - window : 0;   /* first key attended */
    for (int64_t j = j0; j < t; ++j) {
        int64_t page = table[j / P];
        if (page < 0 || page >= n_pages) return -1;
        int64_t off = pool_offset(page, h, j % P, H, P, D);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)q[d] * load_elem(k_pool, off + d, dtype);
        scores[j] = dot * scale;
    }
    double m = -INFINITY;
    for (int64_t j = j0; j < t; ++j) if (scores[j] > m) m = scores[j];
    double sum = 0.0;
    for (int64_t j = j0; j < t; ++j) { scores[j] = exp(scores[j] - m); sum += scores[j]; }
    for (int64_t j = j0; j < t; ++j) scores[j] /= sum;          /* softmax weights */
    for (int d = 0; d < D; ++d) {
        double mix = 0.0;
        for (int64_t j = j0; j < t; ++j) {
            int64_t page = table[j / P];
            mix += scores[j] * load_elem(v_pool, pool_offset(page, h, j % P, H, P, D) + d, dtype);
        }
        out[d] = mix;
    }
    return 0;
}

/*
 * Batched paged decode attention, steps 1-5.
 *   H        KV heads; the query has H * group heads
 *   q        [B][H*group][D] fp32
 *   k_new    [B][H][D] storage dtype; v_new likewise
 *   tables   [B][max_pages] int32 physical page ids
 *   seq_lens [B] retained lengths t_b including the new token (>= 1)
 *   k_pool / v_pool: one layer, [n_pages][H][P][D] storage dtype (modified by step 1)
 *   out      [B][H*group][D] fp64
 *   lanes    optional list of n_lanes query lanes (b*H*group + qh) to compute;
 *            NULL = all.  Step 1 always runs for every request.
 *   threads  OpenMP threads for the lane loop (<= 0: library default)
 * Returns 0 on success, -1 on an out-of-range length or page id.
 */
int orc_paged_decode_attention_ex(int B, int H, int group, int64_t window, int D, int P,
                                  int dtype, void* k_pool, void* v_pool, int64_t n_pages,
                                  const float* q, const void* k_new, const void* v_new,
                                  const int32_t* tables, int max_pages, const int32_t* seq_lens,
                                  double* out, const int64_t* lanes, int64_t n_lanes, int threads) {
    if (group < 1 || window < 0) return -1;
    int rc = orc_append(B, H, D, P, dtype, k_pool, v_pool, n_pages, k_new, v_new, tables,
                        max_pages, seq_lens);
    if (rc != 0) return rc;
    const int HQ = H * group;
    int64_t total = lanes ? n_lanes : (int64_t)B * HQ;
    int64_t t_max = 1;
    for (int b = 0; b < B; ++b) if (seq_lens[b] > t_max) t_max = seq_lens[b];
    int bad = 0;
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    if (threads <= 0) threads = omp_get_max_threads();
#else
    threads = 1;
#endif
    #pragma omp parallel num_threads(threads) reduction(|:bad)
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)t_max);
        if (!scores) bad = 1;
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < total; ++i) {
            if (!scores) continue;
            int64_t lane = lanes ? lanes[i] : i;
            int b = (int)(lane / HQ), qh = (int)(lane % HQ);
            if (lane_attention(H, D, P, dtype, k_pool, v_pool, n_pages, q + lane * D,
                               tables + (int64_t)b * max_pages, seq_lens[b], qh / group,
                               window, scores, out + lane * D) != 0)
                bad = 1;
        }
        free(scores);
    }
    return bad ? -1 : 0;
}

/* Grouped-query attention over the whole prefix. */
int orc_paged_decode_attention_gqa(int B, int H, int group, int D, int P, int dtype, void* k_pool,
                                   void* v_pool, int64_t n_pages, const float* q,
                                   const void* k_new, const void* v_new, const int32_t* tables,
                                   int max_pages, const int32_t* seq_lens, double* out,
                                   const int64_t* lanes, int64_t n_lanes, int threads) {
    return orc_paged_decode_attention_ex(B, H, group, 0, D, P, dtype, k_pool, v_pool, n_pages, q,
                                         k_new, v_new, tables, max_pages, seq_lens, out, lanes,
                                         n_lanes, threads);
}

/* Multi-head attention: one query head per KV head. */
int orc_paged_decode_attention(int B, int H, int D, int P, int dtype, void* k_pool, void* v_pool,
                               int64_t n_pages, const float* q, const void* k_new,
                               const void* v_new, const int32_t* tables, int max_pages,
                               const int32_t* seq_lens, double* out, const int64_t* lanes,
                               int64_t n_lanes, int threads) {
    return orc_paged_decode_attention_gqa(B, H, 1, D, P, dtype, k_pool, v_pool, n_pages, q, k_new,
                                          v_new, tables, max_pages, seq_lens, out, lanes, n_lanes,
                                          threads);
}

/*
 * Batched prefill writing the paged cache ("Incremental Serving", section
 * "Paged KV-cache layout": a future batched prefill may use FlashAttention
 * while writing the same paged cache that paged decode attention reads).
 * Request b holds L0_b = seq_lens[b] - n_b cached tokens and appends
 * n_b = cu_new[b+1] - cu_new[b] new ones.  Token i of the chunk goes to
 * position L0_b + i: its key/value rows are stored there, and its output is the
 * attention of its query over positions 0 .. L0_b + i (the window's last W
 * positions if window > 0) — exactly steps 1-5 of one decode step at
 * t = L0_b + i + 1, taken for i = 0 .. n_b - 1 in order.
 *   q      [total_new][H*group][D] fp32; k_new, v_new [total_new][H][D] storage dtype
 *   out    [total_new][H*group][D] fp64
 * Returns 0, or -1 on an out-of-range length or page id.
 */
int orc_paged_prefill(int B, int H, int group, int64_t window, int D, int P, int dtype,
                      void* k_pool, void* v_pool, int64_t n_pages, const float* q,
                      const void* k_new, const void* v_new, const int32_t* cu_new,
                      const int32_t* tables, int max_pages, const int32_t* seq_lens, double* out,
                      int threads) {
    const int HQ = H * group;
    const int es = dtype == ORC_F32 ? 4 : 2;
    for (int b = 0; b < B; ++b) {
        const int n = cu_new[b + 1] - cu_new[b];
        const int64_t L0 = (int64_t)seq_lens[b] - n;
        if (n < 0 || L0 < 0) return -1;
        for (int i = 0; i < n; ++i) {
            const int64_t x = cu_new[b] + i;   /* row of this token in q / k_new / out */
            const int32_t t = (int32_t)(L0 + i + 1);
            int rc = orc_paged_decode_attention_ex(
                1, H, group, window, D, P, dtype, k_pool, v_pool, n_pages, q + x * HQ * D,
                (const char*)k_new + x * H * D * es, (const char*)v_new + x * H * D * es,
                tables + (int64_t)b * max_pages, max_pages, &t, out + x * HQ * D, NULL, 0,
                threads);
            if (rc != 0) return rc;
        }
    }
    return 0;
}

/* Threads the lane loop would use by default. */
int orc_max_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
