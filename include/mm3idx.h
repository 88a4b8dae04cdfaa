/*
 * mm3idx.h -- C ABI of the GB300 (sm_103a) MiniMax-M3 lightning-indexer
 * library: causal block scoring of bf16 index queries against a paged index-K
 * cache, followed by per-(head, query token) top-k block selection with
 * forced init and local blocks.
 *
 * Sources of the operation (vLLM API pages):
 *   vllm.models.minimax_m3.amd.ops.index_topk
 *     - module docstring: index queries score each 128-token block of index
 *       keys (max over the block), then the top-k blocks plus forced init /
 *       local blocks are selected per query token; the KV page size equals the
 *       sparse block size (128), so one sparse block is one page; the index-K
 *       cache is [num_blocks, 128, head_dim] and each token has a single key
 *       that all index heads read.
 *     - minimax_m3_index_decode: fused decode scoring + top-k; ids are
 *       logical block ids counted from 0, unused slots -1, [heads, total_q, topk];
 *       caller-owned `out` for graph capture, and per-query partial top-k
 *       lists merged in a final step.
 *     - minimax_m3_index_score: score [heads, total_q, max_block], each entry
 *       the largest token score inside a 128-token block.
 *     - minimax_m3_index_topk: top-k from a precomputed score tensor.
 *   vllm.models.minimax_m3.amd.ops.indexer_context_parallel,
 *     check_context_score_inputs / indexer_context_scores: input layout rules
 *     (bf16 [tokens, heads, 128] queries with unit d stride, contiguous
 *     non-empty [pages, 128, 128] cache, int32 tables with unit inner stride),
 *     rows = requests * query_len, table at least cdiv(max_seq_len, 128)
 *     wide, max_seq_len a bound that stays fixed across graph replays, sm_scale
 *     applied to scores.
 *   vllm.models.minimax_m3.amd.ops.indexer_cp_exchange, module docstring:
 *     forced init/local blocks are pinned and never dropped; block ids must
 *     stay below 0xFFFF (local_topk_keys).
 *   vllm.models.minimax_m3.amd.indexer_nvfp4, module docstring: an NVFP4 key
 *     element is e4m3_rn_satfinite(e2m1 * scale).
 *
 * Conventions shared by every call
 *   - D = 128 and the block (page) size is 128 tokens; both are fixed.
 *   - Request i has query_len query tokens, rows i*query_len .. +query_len-1;
 *     query j sits at position pos = seq_lens[i] - query_len + j and sees key
 *     tokens 0..pos.  Its own block is c = pos / 128; blocks 0..c are visible.
 *     A prefill of one request is query_len == seq_len.
 *   - score[h, row, b] = sm_scale * max over visible tokens t of block b of
 *     sum_d q[row, h, d] * k[t, d]   (fp32; natural units).
 *   - Forced blocks of a row: 0..init_blocks-1 and c-local_blocks+1..c,
 *     clipped to 0..c.  They take top-k slots.  The other visible blocks are
 *     ranked by (score desc, id asc); the best topk - |forced| join them.
 *     Output ids are ascending, then -1 up to topk.
 *   - Every pointer is a device pointer unless its comment says otherwise.
 *     The library never allocates or frees device memory, so every address
 *     stays stable for CUDA graph capture.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous and never synchronise, except mm3idx_get_device_error.
 *   - Calls return MM3IDX_OK (0) or a negative MM3IDX_ERR_* code and launch
 *     nothing on error.  rows == 0 is a successful no-op.
 *   - Problems found only by the GPU (a page id outside [0, num_pages),
 *     seq_len > max_seq_len, seq_len < query_len, a bounded wait that ran
 *     out) set bits of a device status word instead of trapping; the affected
 *     rows are computed as if the bad page held no visible tokens, lengths
 *     are clamped to max_seq_len, and rows with pos < 0 see no blocks.
 */
#ifndef MM3IDX_H
#define MM3IDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define MM3IDX_OK                    0
#define MM3IDX_ERR_INVALID_ARGUMENT (-1)  /* null pointer or negative size     */
#define MM3IDX_ERR_Q_LAYOUT         (-2)  /* q not 16-byte aligned, strides not multiples of 8 elements */
#define MM3IDX_ERR_CACHE_LAYOUT     (-3)  /* num_pages < 1, too many pages, or misaligned cache */
#define MM3IDX_ERR_TABLE_LAYOUT     (-4)  /* table_width < cdiv(max_seq_len,128) or table_stride < table_width */
#define MM3IDX_ERR_TOO_MANY_BLOCKS  (-5)  /* cdiv(max_seq_len,128) >= 0xFFFF   */
#define MM3IDX_ERR_QUERY_LEN        (-6)  /* query_len < 1 or max_seq_len < query_len */
#define MM3IDX_ERR_TOPK             (-7)  /* topk outside 1..MM3IDX_MAX_TOPK, init/local < 0, init+local > topk */
#define MM3IDX_ERR_OUT_LAYOUT       (-8)  /* output strides overlap or width too small */
#define MM3IDX_ERR_WORKSPACE        (-9)  /* workspace too small or not 256-byte aligned */
#define MM3IDX_ERR_UNSUPPORTED      (-10) /* shape this entry point does not serve (see its comment) */
#define MM3IDX_ERR_CUDA             (-11) /* a CUDA runtime / driver call failed */

/* bits of the device status word (mm3idx_get_device_error) */
#define MM3IDX_DEV_BAD_PAGE      1  /* a block table entry outside [0, num_pages) was read */
#define MM3IDX_DEV_SEQ_TOO_LONG  2  /* seq_lens[i] > max_seq_len (clamped)  */
#define MM3IDX_DEV_SEQ_TOO_SHORT 4  /* seq_lens[i] < query_len              */
#define MM3IDX_DEV_TIMEOUT       8  /* an on-chip pipeline wait gave up; outputs of that launch are invalid */
#define MM3IDX_DEV_BAD_ROWS     16  /* ragged calls: cu_seqlens_q does not run from 0 to total_q without decreasing */

#define MM3IDX_MAX_TOPK            32  /* largest topk served                  */
#define MM3IDX_MAX_DECODE_ROWS     32  /* heads * query_len limit of the fused decode kernel */

/* workspace kinds for mm3idx_workspace_bytes */
#define MM3IDX_OP_DECODE   1
#define MM3IDX_OP_PREFILL  2
#define MM3IDX_OP_PREFILL_NVFP4 3
#define MM3IDX_OP_SCORE_NVFP4   4

/* The problem every scoring call reads.  Host struct; the pointers in it are
 * device pointers. */
typedef struct mm3idx_problem {
    const void    *idx_q;          /* bf16 [rows, heads, 128], d stride 1, 16-byte aligned */
    int64_t        q_token_stride; /* elements between consecutive rows (multiple of 8)   */
    int64_t        q_head_stride;  /* elements between consecutive heads (multiple of 8)  */
    int32_t        heads;          /* index heads, >= 1; all heads share the keys         */
    const void    *index_cache;    /* bf16 [num_pages, 128, 128] contiguous, 16-byte aligned;
                                      for the NVFP4 entry point: uint8 codes [num_pages, 128, 64],
                                      element 2e in the low nibble, 2e+1 in the high nibble */
    const void    *index_scales;   /* NVFP4 only: uint8 e4m3 [num_pages, 128, 8], scale g covers
                                      d in [16g, 16g+16); must be NULL for bf16 calls       */
    int32_t        num_pages;      /* pages in the cache, >= 1                              */
    const int32_t *block_table;    /* int32 [num_reqs, table_stride]; logical block -> page */
    int64_t        table_stride;   /* elements between table rows, >= table_width           */
    int32_t        table_width;    /* readable columns, >= cdiv(max_seq_len, 128)           */
    const int32_t *seq_lens;       /* int32 [num_reqs]                                      */
    int32_t        num_reqs;       /* requests, >= 0                                        */
    int32_t        query_len;      /* query tokens per request, >= 1                        */
    int32_t        max_seq_len;    /* bound on seq_lens fixed across graph replays (e.g. the model's max length) */
    float          sm_scale;       /* multiplies every score                                */
} mm3idx_problem_t;

/*
 * mm3idx_score -- block scores to HBM (index_topk, minimax_m3_index_score;
 * indexer_context_parallel, indexer_context_scores for the sm_scale factor).
 *
 * out: fp32, element [h, row, b] at out[h*out_head_stride + row*out_row_stride + b]
 * for b < cdiv(max_seq_len, 128).  Visible blocks get their score; blocks past
 * the row's own block get -inf.  Columns at or beyond cdiv(max_seq_len,128)
 * are not touched.  Requires out_row_stride >= cdiv(max_seq_len,128) and
 * out_head_stride >= rows * out_row_stride.  Rows with heads*query_len <= 32
 * run on the streaming decode kernel, others on the tensor-core prefill
 * kernel.  bf16 cache (NVFP4 pages: mm3idx_score_nvfp4).
 */
int mm3idx_score(const mm3idx_problem_t *p, float *out, int64_t out_head_stride,
                 int64_t out_row_stride, void *stream);

/*
 * mm3idx_score_nvfp4 -- mm3idx_score over NVFP4 index-K pages (indexer_nvfp4,
 * MiniMaxM3IndexerRocmNvfp4Impl.forward: the NVFP4 decode and prefill
 * scorers write the fp32 block scores the top-k then reads; module
 * docstring: an element is e4m3_rn_satfinite(e2m1 * scale)).  p->index_cache
 * holds the e2m1 codes and p->index_scales the e4m3 scales (layouts in
 * mm3idx_problem_t).  out as in mm3idx_score.  Rows with heads * query_len
 * <= 32 run on the streaming NVFP4 decode kernel, which dequantises each
 * page on chip (workspace may be NULL); others first dequantise every page a
 * request can see, once, into a bf16 copy in the workspace, then run on the
 * tensor-core scorer: workspace of mm3idx_workspace_bytes(
 * MM3IDX_OP_SCORE_NVFP4, ...) bytes, 256-byte aligned, no initialisation
 * needed (and num_reqs * cdiv(max_seq_len,128) <= INT_MAX / 128, else
 * MM3IDX_ERR_UNSUPPORTED).
 */
int mm3idx_score_nvfp4(const mm3idx_problem_t *p, float *out, int64_t out_head_stride,
                       int64_t out_row_stride, void *workspace, size_t workspace_bytes,
                       void *stream);

/*
 * mm3idx_topk -- top-k selection from a score tensor (index_topk,
 * minimax_m3_index_topk).  score: fp32 [heads, rows, >= visible blocks] with
 * the given strides; only each row's visible blocks 0..c are read.  out: int32,
 * element [h, row, k] at out[h*out_head_stride + row*out_row_stride + k],
 * k < topk.  seq_lens/num_reqs/query_len/max_seq_len follow the problem
 * conventions (c comes from the row's position).
 */
int mm3idx_topk(const float *score, int64_t score_head_stride,
                int64_t score_row_stride, int32_t heads,
                const int32_t *seq_lens, int32_t num_reqs, int32_t query_len,
                int32_t max_seq_len, int32_t topk, int32_t init_blocks,
                int32_t local_blocks, int32_t *out, int64_t out_head_stride,
                int64_t out_row_stride, void *stream);

/*
 * mm3idx_workspace_bytes -- device workspace the fused calls need.
 * op = MM3IDX_OP_DECODE: one ticket counter per request plus the partial
 * top-k candidate lists of requests split across CTAs (depends on the
 * current device's SM count).
 * op = MM3IDX_OP_PREFILL (selection inside the scorer): a 64-byte record
 * per tile of 128 query rows, then two candidate lists (16 keys for
 * topk <= 16, else 32; 8 bytes a key) per row of each tile a CTA touches
 * (depends on the current device's SM count); max_seq_len is not read.
 * op = MM3IDX_OP_PREFILL_NVFP4: that (rounded up to 256 bytes), then a bf16
 * copy of the keys [num_reqs * cdiv(max_seq_len,128), 128, 128] and an
 * int32 table [num_reqs, cdiv(max_seq_len,128)].
 * op = MM3IDX_OP_SCORE_NVFP4 (topk is not read): 0 when heads * query_len
 * <= 32, else the bf16 copy of the keys and its table as above.
 * Writes the size to *bytes.  Reads the current device's attributes; no
 * allocation.
 */
int mm3idx_workspace_bytes(int32_t op, int32_t heads, int32_t num_reqs,
                           int32_t query_len, int32_t max_seq_len,
                           int32_t topk, size_t *bytes);

/*
 * mm3idx_decode -- fused decode: block scores and top-k selection in one
 * persistent kernel; the fp32 score row never goes to HBM (index_topk,
 * minimax_m3_index_decode).  Requires heads * query_len <= 32.
 *
 * out: int32 [h, row, k] at out[h*out_head_stride + row*out_row_stride + k].
 * workspace: >= mm3idx_workspace_bytes(MM3IDX_OP_DECODE, ...) bytes, 256-byte
 * aligned, zero-filled before its first use.  A request longer than one
 * CTA's share of the batch leaves at most topk candidate keys per row per
 * CTA there; the last of its CTAs to finish merges them, counted by a ticket
 * per request that every completed call returns to zero, so the workspace
 * can be reused as it is.  After a call that reported MM3IDX_DEV_TIMEOUT,
 * zero it again.  Launches that share a workspace must not overlap.
 */
int mm3idx_decode(const mm3idx_problem_t *p, int32_t topk, int32_t init_blocks,
                  int32_t local_blocks, int32_t *out, int64_t out_head_stride,
                  int64_t out_row_stride, void *workspace,
                  size_t workspace_bytes, void *stream);

/*
 * mm3idx_decode_nvfp4 -- mm3idx_decode over NVFP4 index-K pages
 * (indexer_nvfp4 module docstring): p->index_cache holds the e2m1 codes and
 * p->index_scales the e4m3 scales (layouts in mm3idx_problem_t).  Each key
 * element is e4m3_rn_satfinite(e2m1 * scale), exact in bf16, scored against
 * the bf16 query like the bf16 path.  Same workspace rules as mm3idx_decode.
 */
int mm3idx_decode_nvfp4(const mm3idx_problem_t *p, int32_t topk,
                        int32_t init_blocks, int32_t local_blocks, int32_t *out,
                        int64_t out_head_stride, int64_t out_row_stride,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * The page table of the block-sparse attention that reads the selected
 * blocks (index_topk, minimax_m3_index_decode: attention_block_table,
 * sparse_block_table_out, sparse_context_lens_out, block_page_stride; the
 * pages fix their shapes, P or 2P for the stride and one index head, but not
 * the mapping, which is read as follows).  A 128-token block spans
 * P = pages_per_block attention pages of 128 / P tokens.  Logical block b of
 * request i lives in attention block attention_block_table[i, b], whose pages
 * are attention_block_table[i, b] * block_page_stride + 0 .. P-1 (stride 2P:
 * every attention block also spans P pages of something else, e.g. values).
 * Row r of the output (total_q rows) holds, at columns k*P .. k*P+P-1, the
 * pages of the row's k-th id (ids ascending, as in `out`), and -1 in the
 * slots whose id is -1.  sparse_context_lens_out[r] is the number of key
 * tokens the row sees (0..pos) that lie in its selected blocks: the selected
 * blocks laid end to end, the last one cut at pos.  Entries times
 * block_page_stride plus P must fit in int32.
 */
typedef struct mm3idx_sparse_table {
    const int32_t *attention_block_table;  /* int32 [num_reqs, attention_table_stride]     */
    int64_t        attention_table_stride; /* elements between rows, >= attention_table_width */
    int32_t        attention_table_width;  /* readable columns, >= cdiv(max_seq_len, 128)  */
    int32_t        pages_per_block;        /* P: 1..128, a divisor of 128                   */
    int32_t        block_page_stride;      /* P or 2 * P                                    */
    int32_t       *sparse_block_table_out; /* int32 [total_q, sparse_table_stride]; columns
                                              0 .. topk*P-1 written                         */
    int64_t        sparse_table_stride;    /* >= topk * P                                   */
    int32_t       *sparse_context_lens_out;/* int32 [total_q]                               */
} mm3idx_sparse_table_t;

/*
 * mm3idx_decode_sparse_table -- mm3idx_decode (bf16 cache, p->index_scales
 * NULL) or mm3idx_decode_nvfp4 (p->index_scales set) that also writes the
 * sparse page table of its ids, from a second kernel launched on `stream`
 * as a programmatic dependent of the decode (it waits for the ids on the
 * GPU, without a launch gap).  Requires p->heads == 1
 * (MM3IDX_ERR_UNSUPPORTED otherwise).  `table` is required and, unless the
 * batch is empty, so is every pointer in it (MM3IDX_ERR_INVALID_ARGUMENT,
 * as is a pages_per_block that does not divide
 * 128 or a stride other than P or 2P); attention_table_width below
 * cdiv(max_seq_len, 128) gives MM3IDX_ERR_TABLE_LAYOUT, sparse_table_stride
 * below topk * P MM3IDX_ERR_OUT_LAYOUT.  Workspace and other rules as
 * mm3idx_decode.
 */
int mm3idx_decode_sparse_table(const mm3idx_problem_t *p, int32_t topk,
                               int32_t init_blocks, int32_t local_blocks,
                               int32_t *out, int64_t out_head_stride,
                               int64_t out_row_stride,
                               const mm3idx_sparse_table_t *table,
                               void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * mm3idx_prefill -- prefill scoring on the tensor cores and top-k selection
 * (index_topk, minimax_m3_index_score then minimax_m3_index_topk).  The
 * scorer selects as it goes: each row's best candidates (a list of 16 keys
 * for topk <= 16, else 32) stay in registers and a small dependent kernel
 * merges the lists of the CTAs that shared a query tile, so no score tensor
 * is written.  Workspace:
 * mm3idx_workspace_bytes(MM3IDX_OP_PREFILL, ...) bytes, 256-byte aligned, no
 * initialisation needed.  out as in mm3idx_decode.  Any heads/query_len.
 */
int mm3idx_prefill(const mm3idx_problem_t *p, int32_t topk, int32_t init_blocks,
                   int32_t local_blocks, int32_t *out, int64_t out_head_stride,
                   int64_t out_row_stride, void *workspace,
                   size_t workspace_bytes, void *stream);

/*
 * mm3idx_prefill_nvfp4 -- mm3idx_prefill over NVFP4 index-K pages
 * (indexer_nvfp4, MiniMaxM3IndexerRocmNvfp4Impl.forward, prefill branch:
 * NVFP4 index scores followed by the top-k).  p->index_cache holds the e2m1
 * codes and p->index_scales the e4m3 scales, as for mm3idx_decode_nvfp4.
 * Every page a request can see is first dequantised, once, to bf16
 * (e4m3_rn_satfinite(e2m1 * scale), exact in bf16) into the workspace; the
 * bf16 tensor-core scorer with its selection then runs on that copy.  Workspace:
 * mm3idx_workspace_bytes(MM3IDX_OP_PREFILL_NVFP4, ...) bytes, 256-byte
 * aligned, no initialisation needed.  A block table entry outside
 * [0, num_pages) sets MM3IDX_DEV_BAD_PAGE and its block gets no visible
 * tokens, as in the bf16 calls.
 * Requires num_reqs * cdiv(max_seq_len, 128) <= INT_MAX / 128
 * (MM3IDX_ERR_UNSUPPORTED).  out as in mm3idx_prefill.
 */
int mm3idx_prefill_nvfp4(const mm3idx_problem_t *p, int32_t topk, int32_t init_blocks,
                         int32_t local_blocks, int32_t *out, int64_t out_head_stride,
                         int64_t out_row_stride, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * Ragged batches (index_topk, minimax_m3_index_score and
 * minimax_m3_index_topk: cu_seqlens_q, prefix_lens, max_query_len): request
 * i owns the query rows cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1 of a batch of
 * total_q rows; row j of it sits at position seq_lens[i] - rows_i + j (the
 * pages' prefix_lens[i] = seq_lens[i] - rows_i).  cu_seqlens_q is an int32
 * device array [num_reqs + 1], from 0 to total_q without decreasing (else
 * MM3IDX_DEV_BAD_ROWS, and rows outside their request get -1 ids).  In the
 * problem struct, query_len is the largest rows_i (max_query_len, a bound
 * that may stay fixed across graph replays); total_q must not exceed
 * num_reqs * query_len (MM3IDX_ERR_INVALID_ARGUMENT), so a workspace sized
 * with mm3idx_workspace_bytes(op, heads, num_reqs, query_len, ...) serves
 * every batch under that bound.  idx_q holds total_q rows; outputs are laid
 * out by row as in the uniform calls.
 *
 * mm3idx_score_ragged -- mm3idx_score of a ragged batch (tensor-core scorer).
 * mm3idx_topk_ragged  -- mm3idx_topk of a ragged batch's score tensor.
 * mm3idx_prefill_ragged -- mm3idx_prefill (p->index_scales NULL) or
 *   mm3idx_prefill_nvfp4 (p->index_scales set) of a ragged batch.
 */
int mm3idx_score_ragged(const mm3idx_problem_t *p, const int32_t *cu_seqlens_q,
                        int32_t total_q, float *out, int64_t out_head_stride,
                        int64_t out_row_stride, void *stream);
int mm3idx_topk_ragged(const float *score, int64_t score_head_stride,
                       int64_t score_row_stride, int32_t heads,
                       const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                       int32_t num_reqs, int32_t total_q, int32_t max_query_len,
                       int32_t max_seq_len, int32_t topk, int32_t init_blocks,
                       int32_t local_blocks, int32_t *out, int64_t out_head_stride,
                       int64_t out_row_stride, void *stream);
int mm3idx_prefill_ragged(const mm3idx_problem_t *p, const int32_t *cu_seqlens_q,
                          int32_t total_q, int32_t topk, int32_t init_blocks,
                          int32_t local_blocks, int32_t *out, int64_t out_head_stride,
                          int64_t out_row_stride, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * mm3idx_forward -- one batch of decode requests followed by prefill
 * requests, scored and selected in one call (indexer_nvfp4,
 * MiniMaxM3IndexerRocmNvfp4Impl.forward: the batch's first
 * num_decode_tokens rows go through the decode scorer and its top-k, the
 * other rows through the prefill scorer and its top-k, into one output).
 * p describes all num_reqs requests (bf16 cache, or NVFP4 pages with
 * p->index_scales set).  Requests 0 .. num_decodes-1 are decode requests of
 * p->query_len rows each (rows 0 .. num_decodes*query_len-1; requires
 * heads * query_len <= 32 when num_decodes > 0, else MM3IDX_ERR_UNSUPPORTED).
 * Requests num_decodes .. num_reqs-1 are prefill requests whose rows follow
 * those: prefill_cu_seqlens_q, an int32 device array
 * [num_reqs - num_decodes + 1], runs from 0 to prefill_total_q (offsets
 * counted from the first prefill row, as in the ragged calls), at most
 * prefill_max_query_len rows per request.  idx_q holds
 * num_decodes*query_len + prefill_total_q rows; out as in mm3idx_decode,
 * one row per query row of the whole batch.  Workspace:
 * mm3idx_forward_workspace_bytes(...) bytes, 256-byte aligned, zero-filled
 * before its first use (its decode part follows mm3idx_decode's rules).
 * The decode kernel runs first, then the prefill's kernels, in stream order.
 */
int mm3idx_forward(const mm3idx_problem_t *p, int32_t num_decodes,
                   const int32_t *prefill_cu_seqlens_q, int32_t prefill_total_q,
                   int32_t prefill_max_query_len, int32_t topk, int32_t init_blocks,
                   int32_t local_blocks, int32_t *out, int64_t out_head_stride,
                   int64_t out_row_stride, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * mm3idx_forward_workspace_bytes -- workspace of mm3idx_forward: the decode
 * workspace of num_decodes requests (MM3IDX_OP_DECODE), rounded up to 256
 * bytes, then the prefill workspace of num_prefills requests of at most
 * prefill_max_query_len rows (MM3IDX_OP_PREFILL, or MM3IDX_OP_PREFILL_NVFP4
 * when nvfp4 != 0).  Reads the current device's SM count; no allocation.
 */
int mm3idx_forward_workspace_bytes(int32_t heads, int32_t num_decodes, int32_t decode_query_len,
                                   int32_t num_prefills, int32_t prefill_max_query_len,
                                   int32_t max_seq_len, int32_t topk, int32_t nvfp4,
                                   size_t *bytes);

/*
 * mm3idx_get_device_error -- synchronises `stream`, then reads and clears the
 * device status word of the current device (MM3IDX_DEV_* bits) into *code.
 */
int mm3idx_get_device_error(void *stream, int32_t *code);

/*
 * mm3idx_decode_static -- mm3idx_decode without a caller-provided workspace.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot give the library device memory: code that has no allocator at
 * hand or is not allowed to allocate at the point of the call (for example a
 * plug-in whose host framework plans every device buffer in advance, or a C
 * caller that only holds the input and output pointers).  The scratch the
 * decode needs lives instead in one array inside this library, of
 * MM3IDX_STATIC_SCRATCH_BYTES, which every GPU that loads the library keeps
 * until the process exits.  Nothing is allocated or freed by this call.
 *
 * Arguments and results are those of mm3idx_decode (bf16 cache).  A problem
 * whose decode workspace (mm3idx_workspace_bytes with MM3IDX_OP_DECODE)
 * exceeds MM3IDX_STATIC_SCRATCH_BYTES is rejected with
 * MM3IDX_ERR_STATIC_SCRATCH.  The first call on a device looks up the
 * array's device address (once per device, with that device current); make
 * that first call before any stream capture.  All calls share the one array
 * and it keeps the previous call's contents; each call first clears the part
 * that must start at zero (the per-request tickets, with cudaMemsetAsync on
 * `stream`, which allocates nothing).  Calls whose executions overlap on the
 * GPU race on the array, so issue them in one stream or otherwise order them.
 */
#define MM3IDX_STATIC_SCRATCH_BYTES (8u << 20)  /* 8 MiB */
#define MM3IDX_ERR_STATIC_SCRATCH   (-12)       /* problem needs more scratch than the static array */
int mm3idx_decode_static(const mm3idx_problem_t *p, int32_t topk, int32_t init_blocks,
                         int32_t local_blocks, int32_t *out, int64_t out_head_stride,
                         int64_t out_row_stride, void *stream);

/*
 * mm3idx_check_wait_timeout -- exercises the failure path of the on-chip
 * pipeline waits.  The pages have no counterpart; every scoring kernel here
 * waits on shared-memory barriers through one bounded wait, and this call
 * makes that wait run out on purpose, on a barrier that nothing completes.
 *
 * Launches one CTA of `warps` warps (1..32) on `stream`.  Every warp waits on
 * the first phase of a fresh barrier; after the library's wait limit (2 s of
 * GPU wall clock) the first warp to give up raises the CTA's abort flag, the
 * others see it and stop waiting, and the kernel sets MM3IDX_DEV_TIMEOUT in
 * the device status word and returns.  No memory is read or written besides
 * the status word, and the context stays usable.  Returns
 * MM3IDX_ERR_INVALID_ARGUMENT for `warps` outside 1..32, MM3IDX_ERR_CUDA when
 * the launch fails.  Not part of any scoring call.
 */
int mm3idx_check_wait_timeout(int32_t warps, void *stream);

/* Human-readable text of a status code (static storage). */
const char *mm3idx_status_string(int status);

/* Library version, for the binding's sanity check. */
int32_t mm3idx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MM3IDX_H */
