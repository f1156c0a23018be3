/*
 * Oracle for KV-outer block-sparse attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded CPU
 * statement of what the method computes, in double precision.  It exists so
 * that the CUDA library can be checked against something independent of it.
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load it; the library itself never does, and it shares no code,
 * header, table or constant with the library.
 *
 * Sources (the crate alice-llm 2.0.0, module sparse_attention):
 *   types.rs   - CuSeqlensQ::new / batch_of, SparseSelection layout,
 *                BlockTables layout, KvOuterIndex fields and accessors,
 *                SparseAttentionError variants.
 *   forward.rs - module doc (KV-outer forward, partial layout, log-sum-exp
 *                combine), fn kvouter_forward (argument checks, q_local_pos),
 *                fn process_work_unit (block gather, right-aligned causal
 *                mask, per-(edge, qhead lane) softmax statistics).
 *   gpu.rs     - kvouter_forward_gpu (used_kv_lens = None means the full
 *                msb * block_size range).
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes of the repository):
 *   - causal = 1 is the right-aligned rule of the code; causal = 2 the
 *     left-aligned variant (limit = the query's position in its chunk), an
 *     opt-in for the doc's reading of unknown KV lengths.
 *   - msb = floor(max_pages / pages_per_block).
 *   - The index drops an entry when its id is -1 or when the block starts at
 *     or beyond the sequence's KV length (block_id * block_size >= lk_b); a
 *     block that is only causally masked is kept.
 *   - Compact slots are listed in ascending raw-slot order; inside a slot the
 *     edges keep the (query, rank) order in which they are met; sel_slots is
 *     padded with -1 after num_sel[h].
 *   - A (query, rank) pair whose block repeats an earlier rank is its own edge.
 *   - Work splits: each non-empty slot, in CSR order, cut into consecutive
 *     pieces of at most `split_edges` edges (0 = never cut).
 *   - Combine of a row with no live partial gives out = 0 and lse = -inf.
 *   - 16-bit o partials (an opt-in the pages do not have; they keep o, m, l
 *     in f32): each o value is the nearest bfloat16 to the exact one, ties
 *     to even; m and l are kept exactly.
 *
 * Parity pins: see tests/test_oracle_pins.py (dense attention on tiny inputs,
 * permutation / padding invariance, single block, equal-key closed form,
 * brute-force index, printed fixtures).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Error kinds, in the order the pages' error enum lists them. */
enum {
    ORC_OK = 0,
    ORC_HEAD_COUNT = 1,     /* Hq must be a positive multiple of Hkv          */
    ORC_BLOCK_PAGE = 2,     /* block_size a positive multiple of page_size    */
    ORC_CU_SEQLENS = 3,     /* cu_seqlens_q empty, not from 0, or decreasing  */
    ORC_SHAPE = 4,          /* a length disagrees, or a page id >= num_pages  */
    ORC_SELECTED_RANGE = 5, /* selected id outside [-1, msb)                  */
    ORC_HEAD_DIM = 6,
    ORC_EMPTY = 7           /* Tq == 0 or Hkv == 0 or topk == 0               */
};

/* ------------------------------------------------------------------------- */
/* Types (types.rs)                                                          */
/* ------------------------------------------------------------------------- */

/* CuSeqlensQ::new: at least two entries, first 0, never decreasing. */
int orc_validate_cu_seqlens(const int64_t *prefix, int64_t len)
{
    if (len < 2 || prefix[0] != 0)
        return ORC_CU_SEQLENS;
    for (int64_t i = 1; i < len; ++i)
        if (prefix[i] < prefix[i - 1])
            return ORC_CU_SEQLENS;
    return ORC_OK;
}

/* CuSeqlensQ::batch_of: the first index whose prefix exceeds the query, minus
 * one (saturating at zero); a plain linear walk. */
int64_t orc_batch_of(const int64_t *prefix, int64_t len, int64_t query)
{
    int64_t first_greater = len;
    for (int64_t i = 0; i < len; ++i) {
        if (prefix[i] > query) {
            first_greater = i;
            break;
        }
    }
    return first_greater > 0 ? first_greater - 1 : 0;
}

/* SparseSelection::get: selected[tq_idx, hkv_idx, rank], row-major. */
int32_t orc_selection_get(const int32_t *selected, int64_t hkv, int64_t topk,
                          int64_t tq_idx, int64_t hkv_idx, int64_t rank)
{
    return selected[(tq_idx * hkv + hkv_idx) * topk + rank];
}

/* KV length of sequence b: max(used_kv_lens[b], 0), or msb * block_size when
 * no lengths are given (gpu.rs, "None" = full block coverage; forward.rs,
 * process_work_unit). */
static int64_t seq_kv_len(const int32_t *used_kv_lens, int64_t b, int64_t msb,
                          int64_t block_size)
{
    if (used_kv_lens == NULL)
        return msb * block_size;
    return used_kv_lens[b] > 0 ? (int64_t)used_kv_lens[b] : 0;
}

/* bf16 bit pattern -> float: the bf16 value is the top half of an f32. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double kv_value(const void *pages, int kv_is_bf16, int64_t offset)
{
    if (kv_is_bf16)
        return bf16_bits_to_double(((const uint16_t *)pages)[offset]);
    return (double)((const float *)pages)[offset];
}

/*
 * Nearest bfloat16 value of x, ties to even: bfloat16 keeps the sign and
 * 8-bit exponent range of binary32 with 8 significant bits, so a normal value
 * in [2^e, 2^(e+1)) lies on a grid of step 2^(e-7), and values below the
 * smallest normal 2^-126 on the subnormal grid of step 2^-133.  Results at
 * or beyond 2^128 overflow to infinity.  Used for the opt-in 16-bit o
 * partials.
 */
double orc_round_bf16(double x)
{
    if (x != x || x == 0.0 || isinf(x))
        return x;
    int k;
    frexp(x, &k);                 /* |x| = f 2^k, f in [0.5, 1): e = k - 1 */
    int step = k - 8;             /* log2 of the grid step 2^(e-7)         */
    if (step < -133)
        step = -133;
    double y = ldexp(rint(ldexp(x, -step)), step);   /* rint: ties to even */
    if (fabs(y) >= ldexp(1.0, 128))
        return x > 0 ? INFINITY : -INFINITY;
    return y;
}

void orc_round_bf16_array(const double *x, int64_t n, double *y)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = orc_round_bf16(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Step 1: the KV-outer CSR index (KvOuterIndex)                             */
/* ------------------------------------------------------------------------- */

/* Sizes the caller must allocate for orc_build_index. */
void orc_index_geometry(int64_t tq, int64_t hkv, int64_t topk, int64_t batch,
                        int64_t max_pages, int64_t block_size, int64_t page_size,
                        int64_t *msb_out, int64_t *nbs_out)
{
    int64_t ppb = (page_size > 0 && block_size % page_size == 0) ? block_size / page_size : 1;
    int64_t msb = ppb > 0 ? max_pages / ppb : 0;
    (void)tq; (void)hkv; (void)topk;
    *msb_out = msb;
    *nbs_out = batch * msb;
}

/*
 * Builds the index of KvOuterIndex (types.rs):
 *   sel_slots   [hkv, nbs]    compact slot -> raw slot b*msb + block, -1 after num_sel[h]
 *   sel_offsets [hkv, nbs+1]  head-local CSR offsets, equal to the head total after num_sel[h]
 *   num_sel     [hkv]
 *   edges       [E, 2]        (query, rank) in CSR order, heads concatenated
 *   edge_head_base [hkv+1]
 *   inv         [hkv, tq, topk]  head-local edge position, -1 if dropped
 *   splits      [S, 4]        work list (head, compact slot, abs edge start, abs edge end)
 *   totals      [3]           E, S, number of non-empty slots over all heads
 * Edge and split arrays need room for tq*hkv*topk entries.
 */
int orc_build_index(const int32_t *selected, int64_t tq, int64_t hkv, int64_t topk,
                    const int64_t *cu_seqlens_q, int64_t batch,
                    const int32_t *used_kv_lens, int64_t max_pages,
                    int64_t block_size, int64_t page_size, int64_t split_edges,
                    int32_t *sel_slots, int32_t *sel_offsets, int32_t *num_sel,
                    int32_t *edges, int64_t *edge_head_base, int32_t *inv,
                    int64_t *splits, int64_t *totals)
{
    if (block_size <= 0 || page_size <= 0 || block_size % page_size != 0)
        return ORC_BLOCK_PAGE;
    if (tq == 0 || hkv == 0 || topk == 0)
        return ORC_EMPTY;
    if (orc_validate_cu_seqlens(cu_seqlens_q, batch + 1) != ORC_OK)
        return ORC_CU_SEQLENS;
    if (cu_seqlens_q[batch] != tq)
        return ORC_SHAPE;

    int64_t msb, nbs;
    orc_index_geometry(tq, hkv, topk, batch, max_pages, block_size, page_size, &msb, &nbs);

    for (int64_t e = 0; e < tq * hkv * topk; ++e)
        if (selected[e] < -1 || selected[e] >= msb)
            return ORC_SELECTED_RANGE;

    int64_t *bucket_count = calloc((size_t)(nbs > 0 ? nbs : 1), sizeof(int64_t));
    int64_t *bucket_cursor = calloc((size_t)(nbs > 0 ? nbs : 1), sizeof(int64_t));
    int64_t head_base = 0;
    int64_t n_splits = 0;
    int64_t n_units = 0;

    for (int64_t h = 0; h < hkv; ++h) {
        edge_head_base[h] = head_base;

        /* Which (query, rank) entries survive, and which bucket each joins. */
        memset(bucket_count, 0, (size_t)(nbs > 0 ? nbs : 1) * sizeof(int64_t));
        for (int64_t i = 0; i < tq; ++i) {
            int64_t b = orc_batch_of(cu_seqlens_q, batch + 1, i);
            int64_t lk = seq_kv_len(used_kv_lens, b, msb, block_size);
            for (int64_t r = 0; r < topk; ++r) {
                int32_t blk = orc_selection_get(selected, hkv, topk, i, h, r);
                if (blk < 0 || (int64_t)blk * block_size >= lk)
                    continue;
                bucket_count[b * msb + blk] += 1;
            }
        }

        /* Compact the non-empty raw slots in ascending order. */
        int64_t j = 0;
        int64_t running = 0;
        for (int64_t slot = 0; slot < nbs; ++slot) {
            if (bucket_count[slot] == 0)
                continue;
            sel_slots[h * nbs + j] = (int32_t)slot;
            sel_offsets[h * (nbs + 1) + j] = (int32_t)running;
            bucket_cursor[slot] = running;
            running += bucket_count[slot];
            j += 1;
        }
        num_sel[h] = (int32_t)j;
        for (int64_t p = j; p <= nbs; ++p)
            sel_offsets[h * (nbs + 1) + p] = (int32_t)running;
        for (int64_t p = j; p < nbs; ++p)
            sel_slots[h * nbs + p] = -1;

        /* Append each surviving entry to its bucket in (query, rank) order. */
        for (int64_t i = 0; i < tq; ++i) {
            int64_t b = orc_batch_of(cu_seqlens_q, batch + 1, i);
            int64_t lk = seq_kv_len(used_kv_lens, b, msb, block_size);
            for (int64_t r = 0; r < topk; ++r) {
                int32_t blk = orc_selection_get(selected, hkv, topk, i, h, r);
                int64_t inv_at = (h * tq + i) * topk + r;
                if (blk < 0 || (int64_t)blk * block_size >= lk) {
                    inv[inv_at] = -1;
                    continue;
                }
                int64_t pos = bucket_cursor[b * msb + blk]++;
                edges[2 * (head_base + pos) + 0] = (int32_t)i;
                edges[2 * (head_base + pos) + 1] = (int32_t)r;
                inv[inv_at] = (int32_t)pos;
            }
        }

        /* Work list: every compact slot in order, cut into pieces. */
        for (int64_t c = 0; c < j; ++c) {
            int64_t start = head_base + sel_offsets[h * (nbs + 1) + c];
            int64_t end = head_base + sel_offsets[h * (nbs + 1) + c + 1];
            int64_t step = split_edges > 0 ? split_edges : (end - start);
            for (int64_t s = start; s < end; s += step) {
                int64_t e = s + step < end ? s + step : end;
                splits[4 * n_splits + 0] = h;
                splits[4 * n_splits + 1] = c;
                splits[4 * n_splits + 2] = s;
                splits[4 * n_splits + 3] = e;
                n_splits += 1;
            }
        }
        n_units += j;
        head_base += running;
    }
    edge_head_base[hkv] = head_base;
    totals[0] = head_base;
    totals[1] = n_splits;
    totals[2] = n_units;
    free(bucket_count);
    free(bucket_cursor);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 2: per-edge partials (forward.rs, kvouter_forward / process_work_unit) */
/* ------------------------------------------------------------------------- */

/*
 * The keys one block contributes to sequence b: positions p of block `blk`
 * with p < lk whose page (block_tables[b, p / page_size]) is not negative.
 * Writes the absolute positions and the physical page / row of each.
 * Returns the number of keys, or -1 when a page id is >= num_pages.
 */
static int64_t gather_block_keys(int64_t b, int64_t blk, int64_t lk,
                                 const int32_t *block_tables, int64_t max_pages,
                                 int64_t block_size, int64_t page_size, int64_t num_pages,
                                 int64_t *pos_out, int64_t *page_out, int64_t *row_out)
{
    int64_t ppb = block_size / page_size;
    int64_t block_start = blk * block_size;
    int64_t block_end = (blk + 1) * block_size < lk ? (blk + 1) * block_size : lk;
    int64_t n = 0;
    for (int64_t page_local = 0; page_local < ppb; ++page_local) {
        int64_t page_seq_start = block_start + page_local * page_size;
        int64_t lo = page_seq_start;
        int64_t hi = page_seq_start + page_size < block_end ? page_seq_start + page_size : block_end;
        if (hi <= lo)
            continue;
        int32_t page_id = block_tables[b * max_pages + blk * ppb + page_local];
        if (page_id < 0)
            continue;
        if ((int64_t)page_id >= num_pages)
            return -1;
        for (int64_t p = lo; p < hi; ++p) {
            pos_out[n] = p;
            page_out[n] = page_id;
            row_out[n] = p - page_seq_start;
            n += 1;
        }
    }
    return n;
}

/* Causal limit of a query: keys at absolute position <= limit stay alive.
 * Mode 1, right-aligned (forward.rs, kvouter_forward doc and
 * process_work_unit: the code's rule); mode 2, left-aligned (the doc's
 * reading for unknown KV lengths: the query's own position in its chunk,
 * an opt-in variant). */
static int64_t causal_limit(int64_t lk, int64_t qo_len, int64_t q_local, int mode)
{
    if (mode == 2)
        return q_local;
    if (lk >= qo_len)
        return lk - qo_len + q_local;
    return q_local;
}

/*
 * Partials for every edge of the index, laid out [E * qhead] rows in CSR order
 * (ForwardPartials): o = sum_p exp(s_p - m) v_p, m = max_p s_p,
 * l = sum_p exp(s_p - m), with s_p = scale * <q, k_p>; a row with no live key
 * gives (o = 0, m = -inf, l = 0).
 */
int orc_forward(const float *q, const void *k_pages, const void *v_pages, int kv_is_bf16,
                int64_t num_pages, const int32_t *sel_slots, const int32_t *sel_offsets,
                const int32_t *num_sel, const int32_t *edges, const int64_t *edge_head_base,
                int64_t nbs, int64_t msb, const int32_t *block_tables, int64_t max_pages,
                const int64_t *cu_seqlens_q, int64_t batch, const int32_t *used_kv_lens,
                int64_t hq, int64_t hkv, int64_t head_dim, int64_t block_size,
                int64_t page_size, float softmax_scale, int causal,
                double *o_partial, double *m_partial, double *l_partial)
{
    if (hkv == 0 || hq == 0 || hq % hkv != 0)
        return ORC_HEAD_COUNT;
    if (head_dim == 0 || block_size <= 0 || page_size <= 0 || block_size % page_size != 0)
        return ORC_BLOCK_PAGE;
    int64_t qhead = hq / hkv;
    int64_t page_stride = hkv * page_size * head_dim;

    int64_t *pos = malloc((size_t)block_size * sizeof(int64_t));
    int64_t *page = malloc((size_t)block_size * sizeof(int64_t));
    int64_t *row = malloc((size_t)block_size * sizeof(int64_t));
    double *score = malloc((size_t)block_size * sizeof(double));
    int status = ORC_OK;

    for (int64_t h = 0; h < hkv && status == ORC_OK; ++h) {
        for (int64_t j = 0; j < num_sel[h] && status == ORC_OK; ++j) {
            int64_t raw_slot = sel_slots[h * nbs + j];
            int64_t b = raw_slot / msb;
            int64_t blk = raw_slot % msb;
            int64_t lk = seq_kv_len(used_kv_lens, b, msb, block_size);
            int64_t qo_len = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
            int64_t n = gather_block_keys(b, blk, lk, block_tables, max_pages, block_size,
                                          page_size, num_pages, pos, page, row);
            if (n < 0) {
                status = ORC_SHAPE;
                break;
            }
            int64_t e0 = edge_head_base[h] + sel_offsets[h * (nbs + 1) + j];
            int64_t e1 = edge_head_base[h] + sel_offsets[h * (nbs + 1) + j + 1];
            for (int64_t e = e0; e < e1; ++e) {
                int64_t q_idx = edges[2 * e];
                int64_t limit = causal_limit(lk, qo_len, q_idx - cu_seqlens_q[b], causal);
                for (int64_t qh = 0; qh < qhead; ++qh) {
                    int64_t hq_abs = h * qhead + qh;
                    const float *q_row = q + (q_idx * hq + hq_abs) * head_dim;
                    int64_t out_row = e * qhead + qh;
                    double m = -INFINITY;
                    for (int64_t t = 0; t < n; ++t) {
                        if (causal && pos[t] > limit) {
                            score[t] = -INFINITY;
                            continue;
                        }
                        int64_t base = page[t] * page_stride + (h * page_size + row[t]) * head_dim;
                        double dot = 0.0;
                        for (int64_t d = 0; d < head_dim; ++d)
                            dot += (double)q_row[d] * kv_value(k_pages, kv_is_bf16, base + d);
                        score[t] = (double)softmax_scale * dot;
                        if (score[t] > m)
                            m = score[t];
                    }
                    double *o = o_partial + out_row * head_dim;
                    for (int64_t d = 0; d < head_dim; ++d)
                        o[d] = 0.0;
                    if (m == -INFINITY) {
                        m_partial[out_row] = -INFINITY;
                        l_partial[out_row] = 0.0;
                        continue;
                    }
                    double l = 0.0;
                    for (int64_t t = 0; t < n; ++t) {
                        if (score[t] == -INFINITY)
                            continue;
                        double p = exp(score[t] - m);
                        l += p;
                        int64_t base = page[t] * page_stride + (h * page_size + row[t]) * head_dim;
                        for (int64_t d = 0; d < head_dim; ++d)
                            o[d] += p * kv_value(v_pages, kv_is_bf16, base + d);
                    }
                    m_partial[out_row] = m;
                    l_partial[out_row] = l;
                }
            }
        }
    }
    free(pos);
    free(page);
    free(row);
    free(score);
    return status;
}

/* ------------------------------------------------------------------------- */
/* Step 3: log-sum-exp combine of the partials (forward.rs module doc)        */
/* ------------------------------------------------------------------------- */

/*
 * For query i and q-head hq (kv head h = hq / qhead, lane qh = hq % qhead),
 * over the ranks r whose inv[h, i, r] >= 0:
 *   M = max m_r, L = sum exp(m_r - M) l_r, out = sum exp(m_r - M) o_r / L,
 *   lse = M + log L.   No live partial: out = 0, lse = -inf.
 */
void orc_combine(const int32_t *inv, const int64_t *edge_head_base, int64_t tq,
                 int64_t hkv, int64_t topk, int64_t qhead, int64_t head_dim,
                 const double *o_partial, const double *m_partial,
                 const double *l_partial, double *out, double *lse)
{
    int64_t hq = hkv * qhead;
    for (int64_t i = 0; i < tq; ++i) {
        for (int64_t hq_abs = 0; hq_abs < hq; ++hq_abs) {
            int64_t h = hq_abs / qhead;
            int64_t qh = hq_abs % qhead;
            double *o = out + (i * hq + hq_abs) * head_dim;
            double big_m = -INFINITY;
            for (int64_t r = 0; r < topk; ++r) {
                int32_t p = inv[(h * tq + i) * topk + r];
                if (p < 0)
                    continue;
                int64_t row = (edge_head_base[h] + p) * qhead + qh;
                if (m_partial[row] > big_m)
                    big_m = m_partial[row];
            }
            for (int64_t d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            if (big_m == -INFINITY) {
                lse[i * hq + hq_abs] = -INFINITY;
                continue;
            }
            double big_l = 0.0;
            for (int64_t r = 0; r < topk; ++r) {
                int32_t p = inv[(h * tq + i) * topk + r];
                if (p < 0)
                    continue;
                int64_t row = (edge_head_base[h] + p) * qhead + qh;
                if (m_partial[row] == -INFINITY)
                    continue;
                double w = exp(m_partial[row] - big_m);
                big_l += w * l_partial[row];
                for (int64_t d = 0; d < head_dim; ++d)
                    o[d] += w * o_partial[row * head_dim + d];
            }
            for (int64_t d = 0; d < head_dim; ++d)
                o[d] /= big_l;
            lse[i * hq + hq_abs] = big_m + log(big_l);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Independent check of steps 1-3: query-outer attention over the selection  */
/* ------------------------------------------------------------------------- */

/*
 * For each requested (query i, q-head hq): the keys are the multiset union,
 * over ranks r with a kept block (same drop rule as the index), of that
 * block's keys (same page and causal rules as the forward); one softmax over
 * all of them.  `rows` lists (i, hq) pairs; NULL means every row in order.
 * Output rows follow the order of `rows`.
 */
int orc_direct(const float *q, const void *k_pages, const void *v_pages, int kv_is_bf16,
               int64_t num_pages, const int32_t *selected, int64_t tq, int64_t hkv,
               int64_t topk, const int64_t *cu_seqlens_q, int64_t batch,
               const int32_t *used_kv_lens, const int32_t *block_tables, int64_t max_pages,
               int64_t hq, int64_t head_dim, int64_t block_size, int64_t page_size,
               float softmax_scale, int causal, const int64_t *rows, int64_t n_rows,
               double *out, double *lse)
{
    if (hkv == 0 || hq == 0 || hq % hkv != 0)
        return ORC_HEAD_COUNT;
    if (head_dim == 0 || block_size <= 0 || page_size <= 0 || block_size % page_size != 0)
        return ORC_BLOCK_PAGE;
    int64_t qhead = hq / hkv;
    int64_t msb, nbs;
    orc_index_geometry(tq, hkv, topk, batch, max_pages, block_size, page_size, &msb, &nbs);
    int64_t page_stride = hkv * page_size * head_dim;
    int64_t cap = topk * block_size;
    int64_t *pos = malloc((size_t)cap * sizeof(int64_t));
    int64_t *page = malloc((size_t)cap * sizeof(int64_t));
    int64_t *row = malloc((size_t)cap * sizeof(int64_t));
    double *score = malloc((size_t)cap * sizeof(double));
    int status = ORC_OK;
    int64_t count = rows ? n_rows : tq * hq;

    for (int64_t k = 0; k < count && status == ORC_OK; ++k) {
        int64_t i = rows ? rows[2 * k] : k / hq;
        int64_t hq_abs = rows ? rows[2 * k + 1] : k % hq;
        int64_t h = hq_abs / qhead;
        int64_t b = orc_batch_of(cu_seqlens_q, batch + 1, i);
        int64_t lk = seq_kv_len(used_kv_lens, b, msb, block_size);
        int64_t qo_len = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        int64_t limit = causal_limit(lk, qo_len, i - cu_seqlens_q[b], causal);
        const float *q_row = q + (i * hq + hq_abs) * head_dim;

        int64_t n = 0;
        for (int64_t r = 0; r < topk; ++r) {
            int32_t blk = selected[(i * hkv + h) * topk + r];
            if (blk < -1 || blk >= msb) {
                status = ORC_SELECTED_RANGE;
                break;
            }
            if (blk < 0 || (int64_t)blk * block_size >= lk)
                continue;
            int64_t got = gather_block_keys(b, blk, lk, block_tables, max_pages, block_size,
                                            page_size, num_pages, pos + n, page + n, row + n);
            if (got < 0) {
                status = ORC_SHAPE;
                break;
            }
            n += got;
        }
        if (status != ORC_OK)
            break;

        double m = -INFINITY;
        for (int64_t t = 0; t < n; ++t) {
            if (causal && pos[t] > limit) {
                score[t] = -INFINITY;
                continue;
            }
            int64_t base = page[t] * page_stride + (h * page_size + row[t]) * head_dim;
            double dot = 0.0;
            for (int64_t d = 0; d < head_dim; ++d)
                dot += (double)q_row[d] * kv_value(k_pages, kv_is_bf16, base + d);
            score[t] = (double)softmax_scale * dot;
            if (score[t] > m)
                m = score[t];
        }
        double *o = out + k * head_dim;
        for (int64_t d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        if (m == -INFINITY) {
            lse[k] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            if (score[t] == -INFINITY)
                continue;
            double p = exp(score[t] - m);
            l += p;
            int64_t base = page[t] * page_stride + (h * page_size + row[t]) * head_dim;
            for (int64_t d = 0; d < head_dim; ++d)
                o[d] += p * kv_value(v_pages, kv_is_bf16, base + d);
        }
        for (int64_t d = 0; d < head_dim; ++d)
            o[d] /= l;
        lse[k] = m + log(l);
    }
    free(pos);
    free(page);
    free(row);
    free(score);
    return status;
}
