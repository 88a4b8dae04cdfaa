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
  int32_t fill_width;         // 0: leave invisible blocks untouched; else write -inf up to it
  int32_t qtiles;             // cdiv(query_len, 128)
  int64_t units_per_head;     // prefill_units_per_head(query_len, max_seq_len)
  int64_t total_units;
  int32_t status_dummy;
  int32_t* status;
};

struct SelectArgs {
  const float* score;
  int64_t s_head, s_row;
  int32_t heads;
  const int32_t* seq_lens;
  int32_t num_reqs;
  int32_t query_len;
  int32_t max_seq_len;
  int32_t topk, init_blocks, local_blocks;
  int32_t* ids;
  int64_t i_head, i_row;
  int32_t* status;
};

// Launchers; each returns a cudaError_t of the launch.
cudaError_t launch_decode_bf16(const CUtensorMap& kmap, const DecodeArgs& a, int grid, cudaStream_t s);
cudaError_t launch_decode_nvfp4(const DecodeArgs& a, int grid, cudaStream_t s);
cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const PrefillArgs& a,
                           int grid, cudaStream_t s);
cudaError_t launch_select(const SelectArgs& a, int num_sms, cudaStream_t s);
// Work units of the prefill scorer for one (request, head), counted for a
// request of max_seq_len tokens (the unit is defined in prefill.cu).
int64_t prefill_units_per_head(int32_t query_len, int32_t max_seq_len);

// Grid sizing of the decode kernel (persistent; one CTA per SM).
int decode_ctas_per_sm();
// Keys per (slot, row) in the decode workspace for a given topk.
inline int decode_tk(int topk) { return topk <= 16 ? 16 : 32; }

}  // namespace mm3idx
