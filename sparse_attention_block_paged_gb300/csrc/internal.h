// internal.h -- argument blocks and launcher declarations shared by the
// host-side C ABI (api.cu) and the kernel translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mm3idx {

constexpr int kD = 128;      // index head dim
constexpr int kBlock = 128;  // tokens per sparse block (= page)

// What the streaming decode kernel produces.
enum DecodeMode : int32_t { kModeScore = 0, kModeSelect = 1 };

struct DecodeArgs {
  const uint16_t* q;          // bf16 bits [rows, heads, 128]
  int64_t q_tok;              // element strides
  int64_t q_head;
  int32_t heads;
  int32_t rows_per_req;       // heads * query_len (<= 32)
  const int32_t* table;
  int64_t table_stride;
  const int32_t* seq_lens;
  int32_t num_reqs;
  int32_t query_len;
  int32_t max_seq_len;
  int32_t num_pages;
  const uint8_t* codes;       // NVFP4 only
  const uint8_t* scales;      // NVFP4 only
  float sm_scale;
  int32_t mode;
  int32_t topk, init_blocks, local_blocks;
  // score mode
  float* score;
  int64_t s_head, s_row;
  int32_t fill_width;         // cdiv(max_seq_len, 128)
  // select mode
  int32_t* ids;
  int64_t i_head, i_row;
  uint64_t* partials;         // [slots, 32 rows, tk] keys
  unsigned int* tickets;      // [num_reqs] arrivals per split request; 0 between calls
  int32_t* status;            // device status word
};

struct PrefillArgs {
  int32_t heads;
  int32_t num_reqs;
  int32_t query_len;
  int32_t max_seq_len;
  int32_t num_pages;
  const int32_t* table;
  int64_t table_stride;
  const int32_t* seq_lens;
  float sm_scale;
  float* score;
  int64_t s_head, s_row;
  const int32_t* cu;          // ragged: [num_reqs + 1] query-row offsets; nullptr: query_len each
  int32_t total_q;            // rows of the batch
  // fused selection (partials != nullptr): candidate lists instead of
  // scores, merged into ids by launch_prefill_merge
  int32_t topk, init_blocks, local_blocks;
  uint64_t* partials;         // [2 * (grid + tiles)] slots of [prefill_tk(topk) keys][128 rows]
  int32_t* tile_rec;          // [1 + tiles][kTileRecInts]: [0][0] = tile count, then one per tile
  int32_t* status;
};

// Per query tile, written by the selecting prefill kernel for the merge:
// first and last CTA holding its units, head, first row, rows, prefix,
// tile index in its request, visible blocks, units total (2 words).
constexpr int kTileRecInts = 16;

struct PrefillMergeArgs {
  const uint64_t* partials;
  const int32_t* tile_rec;
  int64_t tiles;              // a bound on the batch's tiles (the count is tile_rec[0])
  int32_t grid;               // CTAs of the prefill launch
  int32_t heads, total_q;     // bounds every record is checked against
  int32_t topk, init_blocks, local_blocks;
  int32_t* ids;
  int64_t i_head, i_row;
};

struct SelectArgs {
  const float* score;
  int64_t s_head, s_row;
  int32_t heads;
  const int32_t* seq_lens;
  int32_t num_reqs;
  int32_t query_len;          // rows per request (uniform batches)
  const int32_t* cu;          // ragged: [num_reqs + 1] query-row offsets; nullptr: uniform
  int32_t total_q;            // rows of the batch
  int32_t max_seq_len;
  int32_t topk, init_blocks, local_blocks;
  int32_t* ids;
  int64_t i_head, i_row;
  int32_t* status;
};

struct DequantArgs {
  const uint8_t* codes;       // NVFP4 [num_pages, 128, 64]
  const uint8_t* scales;      // e4m3 [num_pages, 128, 8]
  int32_t num_pages;
  const int32_t* table;
  int64_t table_stride;
  const int32_t* seq_lens;
  int32_t num_reqs;
  int32_t max_seq_len;
  int32_t width;              // cdiv(max_seq_len, 128): slots per request
  uint16_t* pages_out;        // bf16 [num_reqs * width, 128, 128]
  int32_t* table_out;         // [num_reqs, width]: slot ids (identity)
  int32_t* status;
};

// The sparse page table of one head's ids (see sparse_table.cu).
struct SparseTableArgs {
  const int32_t* ids;         // [rows, i_row] ascending ids, -1 pad
  int64_t i_row;
  int32_t topk;
  const int32_t* seq_lens;
  int32_t num_reqs;
  int32_t query_len;
  int32_t max_seq_len;
  const int32_t* attn_table;  // [num_reqs, attn_stride] logical block -> attention block
  int64_t attn_stride;
  int32_t pages_per_block;    // attention pages per 128-token block
  int32_t block_page_stride;  // pages between consecutive attention blocks
  int32_t* st_out;            // [rows, st_stride], topk * pages_per_block used
  int64_t st_stride;
  int32_t* ctx_out;           // [rows] visible tokens in the selected blocks
};

// Launchers; each returns a cudaError_t of the launch.
cudaError_t launch_decode_bf16(const CUtensorMap& kmap, const DecodeArgs& a, int grid, cudaStream_t s);
cudaError_t launch_decode_nvfp4(const DecodeArgs& a, int grid, cudaStream_t s);
cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const PrefillArgs& a,
                           int grid, cudaStream_t s);
// The merge of the selecting prefill's lists; a programmatic dependent of it.
cudaError_t launch_prefill_merge(const PrefillMergeArgs& a, cudaStream_t s);
cudaError_t launch_select(const SelectArgs& a, int num_sms, cudaStream_t s);
// -inf for the blocks past each row's own block, up to `width` (score calls).
cudaError_t launch_fill_invisible(const SelectArgs& a, int width, int num_sms, cudaStream_t s);
cudaError_t launch_dequant_pages(const DequantArgs& a, int num_sms, cudaStream_t s);
// Launched as a programmatic dependent of the kernel before it in the stream.
cudaError_t launch_sparse_table(const SparseTableArgs& a, cudaStream_t s);

// Grid sizing of the decode kernel (persistent; one CTA per SM).
int decode_ctas_per_sm();
// Keys per (slot, row) in the decode workspace for a given topk.
inline int decode_tk(int topk) { return topk <= 16 ? 16 : 32; }
// List length of the prefill scorer's fused selection.
inline int prefill_tk(int topk) { return topk <= 16 ? 16 : 32; }

}  // namespace mm3idx
