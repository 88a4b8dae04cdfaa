/*
 * oracle.c -- plain, slow CPU oracle for MiniMax-M3 lightning-indexer block
 * scoring and top-k block selection.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or constant with the CUDA library, and the CUDA library
 * never calls it.
 *
 * What it computes, and where the pages say so:
 *   - vllm.models.minimax_m3.amd.ops.index_topk, module docstring: index
 *     queries score each 128-token block of index keys, taking the max over
 *     the block, then the top-k blocks plus forced init/local blocks are
 *     selected per query token; one page is one sparse block; the index-K
 *     cache is [num_blocks, 128, head_dim] and each token has a single key
 *     that all index heads read.
 *   - same page, minimax_m3_index_score docstring: the score of a visible
 *     sparse block is the max over its index-K tokens.
 *   - same page, minimax_m3_index_decode docstring: ids are logical block ids
 *     counted from 0, unused slots -1, laid out [heads, total_q, topk].
 *   - vllm.models.minimax_m3.amd.ops.indexer_cp_exchange, module docstring:
 *     forced init/local blocks are pinned so they can never be dropped.
 *   - vllm.models.minimax_m3.amd.ops.indexer_context_parallel,
 *     indexer_context_scores: scores are scaled by sm_scale.
 *   - vllm.models.minimax_m3.amd.indexer_nvfp4, module docstring: an NVFP4
 *     key element is e4m3_rn_satfinite(e2m1 * scale).
 *   - index_topk page, minimax_m3_index_decode, the sparse-table arguments:
 *     the page table of the block-sparse attention built from one head's
 *     ids (shapes from the pages, mapping read as stated at
 *     mm3o_sparse_table).
 *
 * Readings where the pages are silent (the same list is kept with the
 * design notes): score = sm_scale * max (natural units, no log2(e)); query j
 * of a request sits at position seq_len - query_len + j and sees key tokens
 * 0..pos inclusive; tokens past pos are left out of the max; init blocks are
 * logical 0..init-1, local blocks are the `local` blocks ending at the row's
 * own block; forced blocks take top-k slots; ties go to the lower block id;
 * ids are written in ascending order followed by -1 padding.
 *
 * All arithmetic is in double.  bf16 and NVFP4 inputs are widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MM3O_D 128
#define MM3O_BLOCK 128

/* ---------------------------------------------------------------- numbers */

/* A bf16 value is the upper half of an IEEE binary32. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point (OFP8) E4M3: sign, 4 exponent bits (bias 7),
 * 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN;
 * there are no infinities, so the largest finite value is 448. */
double mm3o_e4m3_value(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* OCP MX FP4 E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit;
 * exponent 0 is subnormal (m/2).  Magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6. */
double mm3o_e2m1_value(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v;
    if (e == 0)
        v = 0.5 * m;
    else
        v = ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* Round x to E4M3, to nearest with ties to the even code, saturating finite
 * overflow to +-448 ("rn" and "satfinite").  Written as a search over the
 * 127 non-negative finite codes, which is the definition of rounding to the
 * nearest representable value. */
uint8_t mm3o_e4m3_rn_satfinite(double x)
{
    uint8_t sign = 0, best = 0;
    double a = x, bd = INFINITY;
    if (isnan(x))
        return 0x7F;
    if (signbit(x)) {
        sign = 0x80;
        a = -x;
    }
    if (a >= 448.0)
        return sign | 0x7E;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(mm3o_e4m3_value((uint8_t)c) - a);
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
            bd = d;
            best = (uint8_t)c;
        }
    }
    return sign | best;
}

/* NVFP4 key element: e4m3_rn_satfinite(e2m1 * scale), as a real value
 * (indexer_nvfp4 page, module docstring). */
double mm3o_nvfp4_value(uint8_t code, uint8_t scale)
{
    double p = mm3o_e2m1_value(code & 15) * mm3o_e4m3_value(scale);
    return mm3o_e4m3_value(mm3o_e4m3_rn_satfinite(p));
}

/* ------------------------------------------------------------- key access */

typedef struct {
    int nvfp4;
    const uint16_t *cache;   /* bf16 [pages, 128, 128] */
    const uint8_t *codes;    /* [pages, 128, 64], element 2e low nibble */
    const uint8_t *scales;   /* [pages, 128, 8], scale g covers d 16g..16g+15 */
    int64_t num_pages;
} kv_t;

/* mm3o_nvfp4_value depends only on (code, scale byte); it is evaluated once
 * per pair and remembered, so long sequences stay affordable. */
static double nvfp4_memo[256][16];
static int nvfp4_memo_ready;

static double nvfp4_element(uint8_t code, uint8_t scale)
{
    if (!nvfp4_memo_ready) {
        for (int s = 0; s < 256; ++s)
            for (int c = 0; c < 16; ++c)
                nvfp4_memo[s][c] = mm3o_nvfp4_value((uint8_t)c, (uint8_t)s);
        nvfp4_memo_ready = 1;
    }
    return nvfp4_memo[scale][code & 15];
}

static void key_vector(const kv_t *kv, int64_t page, int t, double *k)
{
    if (!kv->nvfp4) {
        const uint16_t *row = kv->cache + (page * MM3O_BLOCK + t) * MM3O_D;
        for (int d = 0; d < MM3O_D; ++d)
            k[d] = bf16_value(row[d]);
    } else {
        const uint8_t *c = kv->codes + (page * MM3O_BLOCK + t) * (MM3O_D / 2);
        const uint8_t *s = kv->scales + (page * MM3O_BLOCK + t) * (MM3O_D / 16);
        for (int d = 0; d < MM3O_D; ++d) {
            uint8_t nib = (d & 1) ? (c[d / 2] >> 4) : (c[d / 2] & 15);
            k[d] = nvfp4_element(nib, s[d / 16]);
        }
    }
}

/* ----------------------------------------------------------- block scores */

/* Scores of the causally visible blocks of one query row.
 *
 * q: the row's 128 bf16 values.  table_row: the request's block table row
 * (logical block b lives in page table_row[b]).  pos: the query position;
 * blocks 0..pos/128 are visible and token t of block b counts when
 * 128*b + t <= pos.  out[b] = sm_scale * max_t sum_d q[d] * k_t[d].
 *
 * Returns the number of visible blocks (0 when pos < 0), or -1 when the row
 * would read a table column >= table_width or a page outside [0, num_pages).
 */
static int64_t block_scores(const kv_t *kv, const uint16_t *q,
                            const int32_t *table_row, int64_t table_width,
                            int64_t pos, double sm_scale, double *out)
{
    double qd[MM3O_D], k[MM3O_D];
    int64_t nb;
    if (pos < 0)
        return 0;
    nb = pos / MM3O_BLOCK + 1;
    if (nb > table_width)
        return -1;
    for (int d = 0; d < MM3O_D; ++d)
        qd[d] = bf16_value(q[d]);
    for (int64_t b = 0; b < nb; ++b) {
        int64_t page = table_row[b];
        double best = -INFINITY;
        if (page < 0 || page >= kv->num_pages)
            return -1;
        for (int t = 0; t < MM3O_BLOCK; ++t) {
            double dot = 0.0;
            if (b * MM3O_BLOCK + t > pos)
                break;
            key_vector(kv, page, t, k);
            for (int d = 0; d < MM3O_D; ++d)
                dot += qd[d] * k[d];
            if (dot > best)
                best = dot;
        }
        out[b] = sm_scale * best;
    }
    return nb;
}

int64_t mm3o_block_scores_bf16(const uint16_t *q, const uint16_t *cache,
                               int64_t num_pages, const int32_t *table_row,
                               int64_t table_width, int64_t pos,
                               double sm_scale, double *out)
{
    kv_t kv = {0, cache, NULL, NULL, num_pages};
    return block_scores(&kv, q, table_row, table_width, pos, sm_scale, out);
}

int64_t mm3o_block_scores_nvfp4(const uint16_t *q, const uint8_t *codes,
                                const uint8_t *scales, int64_t num_pages,
                                const int32_t *table_row, int64_t table_width,
                                int64_t pos, double sm_scale, double *out)
{
    kv_t kv = {1, NULL, codes, scales, num_pages};
    return block_scores(&kv, q, table_row, table_width, pos, sm_scale, out);
}

/* -------------------------------------------------------------- selection */

typedef struct {
    double score;
    int32_t id;
} cand_t;

/* Higher score first; equal scores go to the lower block id. */
static int cand_order(const void *pa, const void *pb)
{
    const cand_t *a = (const cand_t *)pa, *b = (const cand_t *)pb;
    if (a->score > b->score)
        return -1;
    if (a->score < b->score)
        return 1;
    return (a->id > b->id) - (a->id < b->id);
}

static int int_order(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* Top-k selection for one row with nb visible blocks (0..nb-1).
 *
 * Forced blocks F: logical blocks 0..init-1 and the `local` blocks ending at
 * the row's own block c = nb-1, clipped to 0..c.  The remaining visible
 * blocks are candidates, ranked by (score desc, id asc); the first
 * topk - |F| of them join F.  out receives F and the picks in ascending id
 * order, then -1 up to topk.  Returns 0, or -1 when |F| > topk. */
int mm3o_select(const double *scores, int64_t nb, int topk, int init_blocks,
                int local_blocks, int32_t *out)
{
    int64_t c = nb - 1, ncand = 0, nf = 0;
    int32_t *ids;
    cand_t *cand;
    int64_t m, take, n = 0;
    for (int i = 0; i < topk; ++i)
        out[i] = -1;
    if (nb <= 0)
        return 0;
    cand = (cand_t *)malloc(sizeof(cand_t) * (size_t)nb);
    ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nb + topk));
    for (int64_t b = 0; b < nb; ++b) {
        int forced = (b < init_blocks) || (b > c - local_blocks);
        if (forced) {
            ids[nf++] = (int32_t)b;
        } else {
            cand[ncand].score = scores[b];
            cand[ncand].id = (int32_t)b;
            ++ncand;
        }
    }
    if (nf > topk) {
        free(cand);
        free(ids);
        return -1;
    }
    qsort(cand, (size_t)ncand, sizeof(cand_t), cand_order);
    m = topk - nf;
    take = ncand < m ? ncand : m;
    n = nf;
    for (int64_t i = 0; i < take; ++i)
        ids[n++] = cand[i].id;
    qsort(ids, (size_t)n, sizeof(int32_t), int_order);
    for (int64_t i = 0; i < n; ++i)
        out[i] = ids[i];
    free(cand);
    free(ids);
    return 0;
}

/* ------------------------------------------------------- whole problems */

/* Scores and ids for every (head, row) of a batch.
 *
 * q: bf16 [tokens, heads, 128] with the given element strides; row r of
 * request i is token i*query_len + j at position seq_lens[i]-query_len+j.
 * scores (may be NULL): double [heads, rows, out_width]; visible blocks get
 * their score, blocks past the row's own block get -inf.
 * ids (may be NULL): int32 [heads, rows, topk].
 * Returns 0, or -1 on a table/page out of range or bad selection arguments. */
static int problem(const kv_t *kv, const uint16_t *q, int64_t q_tok_stride,
                   int64_t q_head_stride, int heads, const int32_t *table,
                   int64_t table_stride, int64_t table_width,
                   const int32_t *seq_lens, int num_reqs, int query_len,
                   double sm_scale, int topk, int init_blocks,
                   int local_blocks, double *scores, int64_t out_width,
                   int32_t *ids)
{
    int64_t rows = (int64_t)num_reqs * query_len;
    double *buf = (double *)malloc(sizeof(double) * (size_t)(table_width + 1));
    int rc = 0;
    for (int i = 0; i < num_reqs && rc == 0; ++i) {
        for (int j = 0; j < query_len && rc == 0; ++j) {
            int64_t row = (int64_t)i * query_len + j;
            int64_t pos = (int64_t)seq_lens[i] - query_len + j;
            for (int h = 0; h < heads; ++h) {
                const uint16_t *qr = q + row * q_tok_stride + h * q_head_stride;
                int64_t nb = block_scores(kv, qr, table + i * table_stride,
                                          table_width, pos, sm_scale, buf);
                if (nb < 0) {
                    rc = -1;
                    break;
                }
                if (scores) {
                    double *o = scores + ((int64_t)h * rows + row) * out_width;
                    for (int64_t b = 0; b < out_width; ++b)
                        o[b] = b < nb ? buf[b] : -INFINITY;
                }
                if (ids && mm3o_select(buf, nb, topk, init_blocks, local_blocks,
                                       ids + ((int64_t)h * rows + row) * topk)) {
                    rc = -1;
                    break;
                }
            }
        }
    }
    free(buf);
    return rc;
}

int mm3o_problem_bf16(const uint16_t *q, int64_t q_tok_stride,
                      int64_t q_head_stride, int heads, const uint16_t *cache,
                      int64_t num_pages, const int32_t *table,
                      int64_t table_stride, int64_t table_width,
                      const int32_t *seq_lens, int num_reqs, int query_len,
                      double sm_scale, int topk, int init_blocks,
                      int local_blocks, double *scores, int64_t out_width,
                      int32_t *ids)
{
    kv_t kv = {0, cache, NULL, NULL, num_pages};
    return problem(&kv, q, q_tok_stride, q_head_stride, heads, table,
                   table_stride, table_width, seq_lens, num_reqs, query_len,
                   sm_scale, topk, init_blocks, local_blocks, scores,
                   out_width, ids);
}

int mm3o_problem_nvfp4(const uint16_t *q, int64_t q_tok_stride,
                       int64_t q_head_stride, int heads, const uint8_t *codes,
                       const uint8_t *scales, int64_t num_pages,
                       const int32_t *table, int64_t table_stride,
                       int64_t table_width, const int32_t *seq_lens,
                       int num_reqs, int query_len, double sm_scale, int topk,
                       int init_blocks, int local_blocks, double *scores,
                       int64_t out_width, int32_t *ids)
{
    kv_t kv = {1, NULL, codes, scales, num_pages};
    return problem(&kv, q, q_tok_stride, q_head_stride, heads, table,
                   table_stride, table_width, seq_lens, num_reqs, query_len,
                   sm_scale, topk, init_blocks, local_blocks, scores,
                   out_width, ids);
}

/* Selection from a given score tensor, as the top-k-only entry point does:
 * scores [heads, rows, >= visible] read with the given strides; visible
 * block count per row comes from seq_lens and query_len. */
int mm3o_select_problem(const double *scores, int64_t head_stride,
                        int64_t row_stride, int heads,
                        const int32_t *seq_lens, int num_reqs, int query_len,
                        int topk, int init_blocks, int local_blocks,
                        int32_t *ids)
{
    int64_t rows = (int64_t)num_reqs * query_len;
    for (int i = 0; i < num_reqs; ++i)
        for (int j = 0; j < query_len; ++j) {
            int64_t row = (int64_t)i * query_len + j;
            int64_t pos = (int64_t)seq_lens[i] - query_len + j;
            int64_t nb = pos < 0 ? 0 : pos / MM3O_BLOCK + 1;
            for (int h = 0; h < heads; ++h)
                if (mm3o_select(scores + h * head_stride + row * row_stride, nb,
                                topk, init_blocks, local_blocks,
                                ids + ((int64_t)h * rows + row) * topk))
                    return -1;
        }
    return 0;
}

/* ------------------------------------------------------ sparse page table */

/* The page table of the block-sparse attention that follows the selection,
 * for one index head (index_topk page, minimax_m3_index_decode: the
 * sparse-table arguments attention_block_table [num_reqs, >= blocks],
 * sparse_block_table_out [total_q, topk * PAGES_PER_SPARSE_BLOCK],
 * sparse_context_lens_out [total_q], block_page_stride equal to one or two
 * times PAGES_PER_SPARSE_BLOCK, one index head only).
 *
 * The pages give the shapes but not the mapping; the reading taken here:
 *   - a sparse block of 128 tokens spans P = pages_per_block attention pages
 *     of 128 / P tokens;
 *   - attention_block_table[i, b] is the physical block holding logical
 *     block b of request i, and that block's pages are
 *     attention_block_table[i, b] * block_page_stride + 0 .. P-1;
 *   - slot k of row r (the k-th id of the row, ascending) holds the P pages
 *     of that block at columns k*P .. k*P+P-1; slots whose id is -1 hold -1;
 *   - the context length of row r is the number of key tokens the row sees
 *     (0..pos) that lie in its selected blocks: the selected blocks laid end
 *     to end, the last of them cut at pos.
 * ids: [rows, topk] of one head, as the selection writes them. */
int mm3o_sparse_table(const int32_t *ids, int topk, const int32_t *seq_lens,
                      int num_reqs, int query_len, const int32_t *attn_table,
                      int64_t attn_stride, int pages_per_block,
                      int block_page_stride, int32_t *table_out,
                      int64_t table_stride, int32_t *ctx_out)
{
    for (int i = 0; i < num_reqs; ++i)
        for (int j = 0; j < query_len; ++j) {
            int64_t row = (int64_t)i * query_len + j;
            int64_t pos = (int64_t)seq_lens[i] - query_len + j;
            const int32_t *id = ids + row * topk;
            int32_t *t = table_out + row * table_stride;
            int64_t ctx = 0;
            for (int k = 0; k < topk; ++k) {
                int32_t b = id[k];
                for (int p = 0; p < pages_per_block; ++p)
                    t[(int64_t)k * pages_per_block + p] =
                        b < 0 ? -1
                              : (int32_t)((int64_t)attn_table[i * attn_stride + b] *
                                          block_page_stride + p);
                if (b < 0)
                    continue;
                if ((int64_t)b * MM3O_BLOCK > pos)
                    return -1; /* not a visible block */
                int64_t last = (int64_t)b * MM3O_BLOCK + MM3O_BLOCK - 1;
                ctx += (last < pos ? last : pos) - (int64_t)b * MM3O_BLOCK + 1;
            }
            ctx_out[row] = (int32_t)ctx;
        }
    return 0;
}
