// api.cu -- the extern "C" boundary declared in include/mm3idx.h: argument
// validation (the layout rules of the vLLM MiniMax-M3 pages, mapped to status
// codes instead of ValueError), TMA tensor-map encoding, grid sizing and
// kernel dispatch.  No device memory is allocated or freed here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "ptx.cuh"

using namespace mm3idx;

namespace {

constexpr int32_t kVersion = 1;
constexpr int kMaxDevices = 64;

// Device status word (MM3IDX_DEV_* bits), one per device context.
__device__ int32_t g_status_word;

struct DeviceInfo {
  int sms = 0;
  int32_t* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MM3IDX_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.sms == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return MM3IDX_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return MM3IDX_ERR_CUDA;
    d.status = static_cast<int32_t*>(p);
    d.sms = sms;
  }
  *out = &d;
  return MM3IDX_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [pages*128, 128] bf16 rows, 64-column boxes of 128 rows, 128-byte swizzle.
int make_kmap(const mm3idx_problem_t* p, CUtensorMap* m) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return MM3IDX_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD),
                              static_cast<cuuint64_t>(p->num_pages) * kBlock};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p->index_cache), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MM3IDX_OK : MM3IDX_ERR_CACHE_LAYOUT;
}

// [rows, heads, 128] bf16 queries, boxes of 64 columns x 1 head x 128 rows.
int make_qmap(const mm3idx_problem_t* p, int64_t rows, CUtensorMap* m) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return MM3IDX_ERR_CUDA;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(p->heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p->q_head_stride) * 2,
                                 static_cast<cuuint64_t>(p->q_token_stride) * 2};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->idx_q), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MM3IDX_OK : MM3IDX_ERR_Q_LAYOUT;
}

// Scratch of mm3idx_decode_static: one array per device context, kept until
// the process exits.  Host code may not use the symbol itself as a device
// address; its address is looked up once per device with that device current.
static __device__ __align__(256) uint8_t g_static_scratch[MM3IDX_STATIC_SCRATCH_BYTES];
void* g_static_scratch_ptr[kMaxDevices];
std::mutex g_static_mu;

int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MM3IDX_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return MM3IDX_ERR_CUDA;
    g_static_scratch_ptr[dev] = ptr;
  }
  *out = g_static_scratch_ptr[dev];
  return MM3IDX_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Layout rules of check_context_score_inputs / indexer_context_scores and
// minimax_m3_index_decode, as status codes.
int check_problem(const mm3idx_problem_t* p, bool nvfp4) {
  if (!p) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (p->heads < 1 || p->num_reqs < 0) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (p->query_len < 1 || p->max_seq_len < p->query_len) return MM3IDX_ERR_QUERY_LEN;
  if (static_cast<int64_t>(p->num_reqs) * p->query_len >= INT_MAX) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (!(p->sm_scale > 0.0f) || !std::isfinite(p->sm_scale)) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (cdiv(p->max_seq_len, kBlock) >= 0xFFFF) return MM3IDX_ERR_TOO_MANY_BLOCKS;
  if (p->num_reqs == 0) return MM3IDX_OK;
  if (!p->idx_q || !p->index_cache || !p->block_table || !p->seq_lens)
    return MM3IDX_ERR_INVALID_ARGUMENT;
  if (!aligned16(p->idx_q) || p->q_token_stride % 8 != 0 || p->q_head_stride % 8 != 0 ||
      p->q_token_stride <= 0 || (p->heads > 1 && p->q_head_stride <= 0))
    return MM3IDX_ERR_Q_LAYOUT;
  if (p->num_pages < 1 || p->num_pages > INT_MAX / kBlock || !aligned16(p->index_cache))
    return MM3IDX_ERR_CACHE_LAYOUT;
  if (nvfp4 != (p->index_scales != nullptr)) return MM3IDX_ERR_CACHE_LAYOUT;
  if (nvfp4 && !aligned16(p->index_scales)) return MM3IDX_ERR_CACHE_LAYOUT;
  if (p->table_width < cdiv(p->max_seq_len, kBlock) || p->table_stride < p->table_width)
    return MM3IDX_ERR_TABLE_LAYOUT;
  return MM3IDX_OK;
}

int check_topk(int32_t topk, int32_t init_blocks, int32_t local_blocks) {
  if (topk < 1 || topk > MM3IDX_MAX_TOPK || init_blocks < 0 || local_blocks < 0 ||
      static_cast<int64_t>(init_blocks) + local_blocks > topk)
    return MM3IDX_ERR_TOPK;
  return MM3IDX_OK;
}

// Row-major [heads, rows, width] with the given strides must not overlap.
bool out_ok(int64_t head_stride, int64_t row_stride, int32_t heads, int64_t rows, int64_t width) {
  if (row_stride < width) return false;
  if (heads > 1 && head_stride < rows * row_stride) return false;
  return true;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MM3IDX_OK : MM3IDX_ERR_CUDA; }

// Decode workspace: [tickets: num_reqs x 4 B, 256-aligned, zero between
// calls][partial lists: (grid + num_reqs) slots x 32 rows x tk keys].
size_t decode_ws_head(int32_t num_reqs) {
  return (static_cast<size_t>(num_reqs) * 4 + 255) / 256 * 256;
}

size_t decode_ws_bytes(int sms, int32_t heads, int32_t num_reqs, int32_t query_len, int32_t topk) {
  (void)heads;
  (void)query_len;
  const size_t slots = static_cast<size_t>(sms) * decode_ctas_per_sm() + num_reqs;
  return decode_ws_head(num_reqs) + slots * 32 * decode_tk(topk) * 8;
}

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// Prefill workspace, part A (selection fused into the scorer): tile records
// [tiles + 1][kTileRecInts] (256-aligned), then 2 * (grid + tiles) list
// slots of 128 rows x prefill_tk(topk) keys.  `rows` bounds the batch's
// query rows; tiles are bounded by heads * (cdiv(rows, 128) + num_reqs).
int64_t prefill_tiles_bound(int32_t heads, int32_t num_reqs, int64_t rows) {
  return static_cast<int64_t>(heads) * (cdiv(rows, 128) + num_reqs);
}

size_t prefill_part_a(int sms, int32_t heads, int32_t num_reqs, int32_t query_len,
                      int32_t topk) {
  const int64_t rows = static_cast<int64_t>(num_reqs) * query_len;
  const int64_t tiles = prefill_tiles_bound(heads, num_reqs, rows);
  return align256(static_cast<size_t>(tiles + 1) * kTileRecInts * 4) +
         static_cast<size_t>(2 * (sms + tiles)) * 128 * prefill_tk(topk) * 8;
}

// The bf16 copy of an NVFP4 batch's visible pages: [num_reqs *
// cdiv(max_seq_len,128), 128, 128] bf16, then its int32 table [num_reqs,
// cdiv(max_seq_len,128)].
size_t dequant_copy_bytes(int32_t num_reqs, int32_t max_seq_len) {
  const size_t slots = static_cast<size_t>(num_reqs) * cdiv(max_seq_len, kBlock);
  return slots * kBlock * kD * 2 + align256(slots * 4);
}

// Whole prefill workspace: part A, then for NVFP4 the bf16 copy of the keys.
size_t prefill_ws_bytes(int sms, int32_t heads, int32_t num_reqs, int32_t query_len,
                        int32_t max_seq_len, int32_t topk, bool nvfp4) {
  const size_t a = prefill_part_a(sms, heads, num_reqs, query_len, topk);
  if (!nvfp4) return a;
  return align256(a) + dequant_copy_bytes(num_reqs, max_seq_len);
}

// Score workspace of NVFP4 pages: none when the streaming decode kernel
// dequantises on chip (heads * query_len <= 32), else the bf16 copy.
size_t score_nvfp4_ws_bytes(int32_t heads, int32_t num_reqs, int32_t query_len,
                            int32_t max_seq_len) {
  if (static_cast<int64_t>(heads) * query_len <= MM3IDX_MAX_DECODE_ROWS) return 0;
  return dequant_copy_bytes(num_reqs, max_seq_len);
}

// Workspace of a mixed batch: the decode part (256-aligned), then the
// prefill part.
size_t forward_ws_bytes(int sms, int32_t heads, int32_t num_decodes, int32_t decode_query_len,
                        int32_t num_prefills, int32_t prefill_max_query_len, int32_t max_seq_len,
                        int32_t topk, bool nvfp4) {
  const size_t d = num_decodes > 0
      ? align256(decode_ws_bytes(sms, heads, num_decodes, decode_query_len, topk)) : 0;
  const size_t f = num_prefills > 0
      ? prefill_ws_bytes(sms, heads, num_prefills, prefill_max_query_len, max_seq_len, topk, nvfp4)
      : 0;
  return d + f;
}

DecodeArgs decode_args(const mm3idx_problem_t* p, int* status) {
  DecodeArgs a{};
  a.q = static_cast<const uint16_t*>(p->idx_q);
  a.q_tok = p->q_token_stride;
  a.q_head = p->q_head_stride;
  a.heads = p->heads;
  a.rows_per_req = p->heads * p->query_len;
  a.table = p->block_table;
  a.table_stride = p->table_stride;
  a.seq_lens = p->seq_lens;
  a.num_reqs = p->num_reqs;
  a.query_len = p->query_len;
  a.max_seq_len = p->max_seq_len;
  a.num_pages = p->num_pages;
  a.sm_scale = p->sm_scale;
  a.status = status;
  return a;
}

int decode_grid(const mm3idx_problem_t* p, int sms) {
  const int64_t bound = static_cast<int64_t>(p->num_reqs) * cdiv(p->max_seq_len, kBlock);
  int64_t g = static_cast<int64_t>(sms) * decode_ctas_per_sm();
  if (bound < g) g = bound;
  return static_cast<int>(g < 1 ? 1 : g);
}

// The sparse-table arguments (index_topk, minimax_m3_index_decode): all or
// none, one index head, stride P or 2P, table wide enough.
int check_sparse_table(const mm3idx_problem_t* p, int32_t topk, const mm3idx_sparse_table_t* t) {
  if (p->num_reqs > 0 &&
      (!t->attention_block_table || !t->sparse_block_table_out || !t->sparse_context_lens_out))
    return MM3IDX_ERR_INVALID_ARGUMENT;
  if (p->heads != 1) return MM3IDX_ERR_UNSUPPORTED;
  const int32_t P = t->pages_per_block;
  if (P < 1 || P > kBlock || kBlock % P != 0) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (t->block_page_stride != P && t->block_page_stride != 2 * P) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (t->attention_table_width < cdiv(p->max_seq_len, kBlock) ||
      t->attention_table_stride < t->attention_table_width)
    return MM3IDX_ERR_TABLE_LAYOUT;
  if (t->sparse_table_stride < static_cast<int64_t>(topk) * P) return MM3IDX_ERR_OUT_LAYOUT;
  return MM3IDX_OK;
}

// static_scratch: the workspace is the library's own array (mm3idx_decode_static):
// a problem too large for it is MM3IDX_ERR_STATIC_SCRATCH, and its tickets are
// cleared on the stream once every argument check has passed.
int run_decode(const mm3idx_problem_t* p, bool nvfp4, int32_t topk, int32_t init_blocks,
               int32_t local_blocks, int32_t* out, int64_t out_head_stride, int64_t out_row_stride,
               void* workspace, size_t workspace_bytes, void* stream,
               const mm3idx_sparse_table_t* table = nullptr, bool static_scratch = false) {
  int rc = check_problem(p, nvfp4);
  if (rc) return rc;
  if ((rc = check_topk(topk, init_blocks, local_blocks))) return rc;
  if (table && (rc = check_sparse_table(p, topk, table))) return rc;
  const int64_t rows = static_cast<int64_t>(p->num_reqs) * p->query_len;
  if (rows == 0) return MM3IDX_OK;
  if (p->heads * static_cast<int64_t>(p->query_len) > MM3IDX_MAX_DECODE_ROWS)
    return MM3IDX_ERR_UNSUPPORTED;
  if (!out || !out_ok(out_head_stride, out_row_stride, p->heads, rows, topk))
    return MM3IDX_ERR_OUT_LAYOUT;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  const size_t need = decode_ws_bytes(dev->sms, p->heads, p->num_reqs, p->query_len, topk);
  if (static_scratch && need > workspace_bytes) return MM3IDX_ERR_STATIC_SCRATCH;
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MM3IDX_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap kmap;   // bf16 pages only: the NVFP4 kernel copies whole pages untiled
  if (!nvfp4 && (rc = make_kmap(p, &kmap))) return rc;
  // The tickets must start at zero; a completed call leaves them so, but a
  // call that gave up part-way may not have.
  if (static_scratch && cudaMemsetAsync(workspace, 0, decode_ws_head(p->num_reqs), s) != cudaSuccess)
    return MM3IDX_ERR_CUDA;
  DecodeArgs a = decode_args(p, dev->status);
  a.mode = kModeSelect;
  a.topk = topk;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  a.ids = out;
  a.i_head = out_head_stride;
  a.i_row = out_row_stride;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.tickets = reinterpret_cast<unsigned int*>(ws);
  a.partials = reinterpret_cast<uint64_t*>(ws + decode_ws_head(p->num_reqs));
  const int grid = decode_grid(p, dev->sms);
  cudaError_t e;
  if (nvfp4) {
    a.codes = static_cast<const uint8_t*>(p->index_cache);
    a.scales = static_cast<const uint8_t*>(p->index_scales);
    e = launch_decode_nvfp4(a, grid, s);
  } else {
    e = launch_decode_bf16(kmap, a, grid, s);
  }
  if (e == cudaSuccess && table) {
    SparseTableArgs t{};
    t.ids = out;
    t.i_row = out_row_stride;
    t.topk = topk;
    t.seq_lens = p->seq_lens;
    t.num_reqs = p->num_reqs;
    t.query_len = p->query_len;
    t.max_seq_len = p->max_seq_len;
    t.attn_table = table->attention_block_table;
    t.attn_stride = table->attention_table_stride;
    t.pages_per_block = table->pages_per_block;
    t.block_page_stride = table->block_page_stride;
    t.st_out = table->sparse_block_table_out;
    t.st_stride = table->sparse_table_stride;
    t.ctx_out = table->sparse_context_lens_out;
    e = launch_sparse_table(t, s);
  }
  return cuda_status(e);
}

// Scores of a batch on the tensor-core scorer; cu == nullptr: query_len
// rows per request, else the ragged row offsets (total_q rows).
// Selection fused into the prefill scorer.
struct PrefillSelect {
  int32_t* ids;
  int64_t i_head, i_row;
  int32_t topk, init_blocks, local_blocks;
  uint64_t* partials;
  int32_t* tile_rec;
  int64_t tiles;              // records (a bound on the batch's tiles)
};

int prefill_scores(const mm3idx_problem_t* p, const int32_t* cu, int32_t total_q, float* out,
                   int64_t head_stride, int64_t row_stride, int sms, int32_t* status,
                   cudaStream_t s, const PrefillSelect* sel = nullptr) {
  PrefillArgs a{};
  if (sel) {
    a.topk = sel->topk;
    a.init_blocks = sel->init_blocks;
    a.local_blocks = sel->local_blocks;
    a.partials = sel->partials;
    a.tile_rec = sel->tile_rec;
  }
  a.heads = p->heads;
  a.num_reqs = p->num_reqs;
  a.query_len = p->query_len;
  a.max_seq_len = p->max_seq_len;
  a.num_pages = p->num_pages;
  a.table = p->block_table;
  a.table_stride = p->table_stride;
  a.seq_lens = p->seq_lens;
  a.sm_scale = p->sm_scale;
  a.score = out;
  a.s_head = head_stride;
  a.s_row = row_stride;
  a.cu = cu;
  a.total_q = total_q;
  a.status = status;
  // The kernel counts the units itself; a bound on them keeps tiny batches
  // from launching idle CTAs: tiles x pairs of blocks per tile.
  const int64_t tiles = cdiv(total_q, 128) + p->num_reqs;
  const int64_t bound = static_cast<int64_t>(p->heads) * tiles * ((cdiv(p->max_seq_len, kBlock) + 1) / 2);
  int64_t grid = sms;
  if (bound < grid) grid = bound;
  if (grid < 1) return MM3IDX_OK;
  CUtensorMap qmap, kmap;
  int rc;
  if ((rc = make_qmap(p, total_q, &qmap))) return rc;
  if ((rc = make_kmap(p, &kmap))) return rc;
  if ((rc = cuda_status(launch_prefill(qmap, kmap, a, static_cast<int>(grid), s)))) return rc;
  if (!sel) return MM3IDX_OK;
  PrefillMergeArgs m{};
  m.partials = sel->partials;
  m.tile_rec = sel->tile_rec;
  m.tiles = sel->tiles;
  m.grid = static_cast<int32_t>(grid);
  m.heads = p->heads;
  m.total_q = total_q;
  m.topk = sel->topk;
  m.init_blocks = sel->init_blocks;
  m.local_blocks = sel->local_blocks;
  m.ids = sel->ids;
  m.i_head = sel->i_head;
  m.i_row = sel->i_row;
  return cuda_status(launch_prefill_merge(m, s));
}

SelectArgs select_args(const float* score, int64_t sh, int64_t sr, int32_t heads,
                       const int32_t* seq_lens, int32_t num_reqs, int32_t query_len,
                       const int32_t* cu, int32_t total_q, int32_t max_seq_len, int32_t topk,
                       int32_t init_blocks, int32_t local_blocks, int32_t* out, int64_t oh,
                       int64_t orow, int32_t* status) {
  SelectArgs a{};
  a.cu = cu;
  a.total_q = total_q;
  a.score = score;
  a.s_head = sh;
  a.s_row = sr;
  a.heads = heads;
  a.seq_lens = seq_lens;
  a.num_reqs = num_reqs;
  a.query_len = query_len;
  a.max_seq_len = max_seq_len;
  a.topk = topk;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  a.ids = out;
  a.i_head = oh;
  a.i_row = orow;
  a.status = status;
  return a;
}

// The score calls on the tensor-core scorer: the scores of the visible
// blocks, then -inf past each row's block up to `width` by a row-parallel
// kernel (in the scorer's epilogue that fill fell mostly on the CTAs of the
// first, short tiles and held up their MMAs).
int score_then_fill(const mm3idx_problem_t* p, const int32_t* cu, int32_t total_q, float* out,
                    int64_t head_stride, int64_t row_stride, int32_t width, DeviceInfo* dev,
                    cudaStream_t s) {
  int rc = prefill_scores(p, cu, total_q, out, head_stride, row_stride, dev->sms, dev->status, s);
  if (rc) return rc;
  SelectArgs f = select_args(out, head_stride, row_stride, p->heads, p->seq_lens, p->num_reqs,
                             p->query_len, cu, total_q, p->max_seq_len, 1, 0, 0, nullptr, 0, 0,
                             dev->status);
  return cuda_status(launch_fill_invisible(f, width, dev->sms, s));
}

// Dequantises every page an NVFP4 batch can see, once, into a bf16 copy at
// `dst` (dequant_copy_bytes long) and points *q at it: the copy's table maps
// (request, block) to its slot, or to -1 for a block whose page id is out of
// range, so the bf16 scorer treats that block as it treats a bad page (no
// visible tokens).  Requires num_reqs * cdiv(max_seq_len,128) <= INT_MAX / 128.
int dequant_copy(const mm3idx_problem_t* p, uint8_t* dst, DeviceInfo* dev, cudaStream_t s,
                 mm3idx_problem_t* q) {
  const int64_t width = cdiv(p->max_seq_len, kBlock);
  const int64_t slots = static_cast<int64_t>(p->num_reqs) * width;
  DequantArgs d{};
  d.codes = static_cast<const uint8_t*>(p->index_cache);
  d.scales = static_cast<const uint8_t*>(p->index_scales);
  d.num_pages = p->num_pages;
  d.table = p->block_table;
  d.table_stride = p->table_stride;
  d.seq_lens = p->seq_lens;
  d.num_reqs = p->num_reqs;
  d.max_seq_len = p->max_seq_len;
  d.width = static_cast<int32_t>(width);
  d.pages_out = reinterpret_cast<uint16_t*>(dst);
  d.table_out = reinterpret_cast<int32_t*>(dst + slots * kBlock * kD * 2);
  d.status = dev->status;
  int rc = cuda_status(launch_dequant_pages(d, dev->sms, s));
  if (rc) return rc;
  *q = *p;
  q->index_cache = d.pages_out;
  q->index_scales = nullptr;
  q->num_pages = static_cast<int32_t>(slots);
  q->block_table = d.table_out;
  q->table_stride = width;
  q->table_width = static_cast<int32_t>(width);
  return MM3IDX_OK;
}

// Block scores of a uniform batch.  heads * query_len <= 32: the streaming
// decode kernel in score mode (NVFP4 pages dequantised on chip); larger row
// counts: the tensor-core scorer, on a bf16 copy of NVFP4 pages made in the
// workspace first.
int run_score(const mm3idx_problem_t* p, bool nvfp4, float* out, int64_t out_head_stride,
              int64_t out_row_stride, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_problem(p, nvfp4);
  if (rc) return rc;
  const int64_t rows = static_cast<int64_t>(p->num_reqs) * p->query_len;
  if (rows == 0) return MM3IDX_OK;
  const int32_t width = static_cast<int32_t>(cdiv(p->max_seq_len, kBlock));
  if (!out || !out_ok(out_head_stride, out_row_stride, p->heads, rows, width))
    return MM3IDX_ERR_OUT_LAYOUT;
  const bool streaming = static_cast<int64_t>(p->heads) * p->query_len <= MM3IDX_MAX_DECODE_ROWS;
  if (nvfp4 && !streaming) {
    if (static_cast<int64_t>(p->num_reqs) * width > INT_MAX / kBlock) return MM3IDX_ERR_UNSUPPORTED;
    const size_t need = score_nvfp4_ws_bytes(p->heads, p->num_reqs, p->query_len, p->max_seq_len);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return MM3IDX_ERR_WORKSPACE;
  }
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (streaming) {
    DecodeArgs a = decode_args(p, dev->status);
    a.mode = kModeScore;
    a.topk = 1;
    a.score = out;
    a.s_head = out_head_stride;
    a.s_row = out_row_stride;
    a.fill_width = width;
    if (nvfp4) {
      a.codes = static_cast<const uint8_t*>(p->index_cache);
      a.scales = static_cast<const uint8_t*>(p->index_scales);
      return cuda_status(launch_decode_nvfp4(a, decode_grid(p, dev->sms), s));
    }
    CUtensorMap kmap;
    if ((rc = make_kmap(p, &kmap))) return rc;
    return cuda_status(launch_decode_bf16(kmap, a, decode_grid(p, dev->sms), s));
  }
  mm3idx_problem_t q = *p;
  if (nvfp4 && (rc = dequant_copy(p, static_cast<uint8_t*>(workspace), dev, s, &q))) return rc;
  return score_then_fill(&q, nullptr, static_cast<int32_t>(rows), out, out_head_stride,
                         out_row_stride, width, dev, s);
}

// Ragged batches: row offsets on the device, total_q rows, at most
// max_query_len rows per request (the bound the workspace is sized with).
int check_ragged(int32_t num_reqs, int32_t max_query_len, const int32_t* cu, int32_t total_q) {
  if (total_q < 0 || max_query_len < 1) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(total_q) > static_cast<int64_t>(num_reqs) * max_query_len)
    return MM3IDX_ERR_INVALID_ARGUMENT;
  if (num_reqs > 0 && (!cu || (reinterpret_cast<uintptr_t>(cu) & 3u)))
    return MM3IDX_ERR_INVALID_ARGUMENT;
  return MM3IDX_OK;
}

int run_topk(const float* score, int64_t sh, int64_t sr, int32_t heads, const int32_t* seq_lens,
             int32_t num_reqs, int32_t query_len, const int32_t* cu, int32_t total_q,
             int32_t max_seq_len, int32_t topk, int32_t init_blocks, int32_t local_blocks,
             int32_t* out, int64_t oh, int64_t orow, void* stream) {
  if (heads < 1 || num_reqs < 0) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (query_len < 1 || max_seq_len < query_len) return MM3IDX_ERR_QUERY_LEN;
  if (cdiv(max_seq_len, kBlock) >= 0xFFFF) return MM3IDX_ERR_TOO_MANY_BLOCKS;
  int rc = check_topk(topk, init_blocks, local_blocks);
  if (rc) return rc;
  if (total_q == 0) return MM3IDX_OK;
  if (!score || !seq_lens || !out) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (!out_ok(sh, sr, heads, total_q, cdiv(max_seq_len, kBlock)) ||
      !out_ok(oh, orow, heads, total_q, topk))
    return MM3IDX_ERR_OUT_LAYOUT;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  SelectArgs a = select_args(score, sh, sr, heads, seq_lens, num_reqs, query_len, cu, total_q,
                             max_seq_len, topk, init_blocks, local_blocks, out, oh, orow,
                             dev->status);
  return cuda_status(launch_select(a, dev->sms, static_cast<cudaStream_t>(stream)));
}

// Prefill: the scorer selects as it goes (no score tensor), a dependent
// kernel merges its lists.  NVFP4 keys are first dequantised, once per
// page, into a bf16 copy in the workspace.  cu == nullptr: query_len rows
// per request; else ragged (total_q rows).
int run_prefill(const mm3idx_problem_t* p, bool nvfp4, const int32_t* cu, int32_t total_q,
                int32_t topk, int32_t init_blocks, int32_t local_blocks, int32_t* out,
                int64_t out_head_stride, int64_t out_row_stride, void* workspace,
                size_t workspace_bytes, void* stream) {
  int rc = check_problem(p, nvfp4);
  if (rc) return rc;
  if ((rc = check_topk(topk, init_blocks, local_blocks))) return rc;
  if (cu) {
    if ((rc = check_ragged(p->num_reqs, p->query_len, cu, total_q))) return rc;
  } else {
    total_q = p->num_reqs * p->query_len;   // < INT_MAX (check_problem)
  }
  const int64_t rows = total_q;
  if (rows == 0) return MM3IDX_OK;
  if (!out || !out_ok(out_head_stride, out_row_stride, p->heads, rows, topk))
    return MM3IDX_ERR_OUT_LAYOUT;
  const int64_t width = cdiv(p->max_seq_len, kBlock);
  if (nvfp4 && static_cast<int64_t>(p->num_reqs) * width > INT_MAX / kBlock)
    return MM3IDX_ERR_UNSUPPORTED;
  // The list slots depend on the grid (the SM count): a workspace short of
  // the size for a grid of none is refused before any CUDA call.
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < prefill_ws_bytes(0, p->heads, p->num_reqs, p->query_len, p->max_seq_len,
                                         topk, nvfp4))
    return MM3IDX_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  if (workspace_bytes < prefill_ws_bytes(dev->sms, p->heads, p->num_reqs, p->query_len,
                                         p->max_seq_len, topk, nvfp4))
    return MM3IDX_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t part_a = align256(prefill_part_a(dev->sms, p->heads, p->num_reqs, p->query_len, topk));
  mm3idx_problem_t q = *p;
  if (nvfp4 && (rc = dequant_copy(p, ws + part_a, dev, s, &q))) return rc;
  const int64_t tiles = prefill_tiles_bound(p->heads, p->num_reqs,
                                            static_cast<int64_t>(p->num_reqs) * p->query_len);
  PrefillSelect sel{};
  sel.ids = out;
  sel.i_head = out_head_stride;
  sel.i_row = out_row_stride;
  sel.topk = topk;
  sel.init_blocks = init_blocks;
  sel.local_blocks = local_blocks;
  sel.tile_rec = reinterpret_cast<int32_t*>(ws);
  sel.tiles = tiles;
  sel.partials = reinterpret_cast<uint64_t*>(
      ws + align256(static_cast<size_t>(tiles + 1) * kTileRecInts * 4));
  return prefill_scores(&q, cu, total_q, nullptr, 0, 0, dev->sms, dev->status, s, &sel);
}

// Every warp waits on the first phase of a barrier that nothing arrives at,
// through the bounded wait of the pipeline kernels, so the wait runs out.
__global__ void wait_timeout_check_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const bool ok = warp_wait(&bar, 0, &abort_flag);
  __syncthreads();
  if (threadIdx.x == 0 && (!ok || abort_flag)) atomicOr(status, MM3IDX_DEV_TIMEOUT);
}

}  // namespace

extern "C" {

int mm3idx_check_wait_timeout(int32_t warps, void* stream) {
  if (warps < 1 || warps > 32) return MM3IDX_ERR_INVALID_ARGUMENT;
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  wait_timeout_check_kernel<<<1, warps * 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->status);
  return cuda_status(cudaGetLastError());
}

int32_t mm3idx_version(void) { return kVersion; }

const char* mm3idx_status_string(int status) {
  switch (status) {
    case MM3IDX_OK: return "ok";
    case MM3IDX_ERR_INVALID_ARGUMENT: return "invalid argument (null pointer, negative size or non-positive sm_scale)";
    case MM3IDX_ERR_Q_LAYOUT: return "index queries must be bf16 [tokens, heads, 128], 16-byte aligned, strides multiples of 8";
    case MM3IDX_ERR_CACHE_LAYOUT: return "index cache must be contiguous, non-empty and 16-byte aligned";
    case MM3IDX_ERR_TABLE_LAYOUT: return "block table narrower than cdiv(max_seq_len, 128) or stride < width";
    case MM3IDX_ERR_TOO_MANY_BLOCKS: return "block ids must stay below 0xFFFF";
    case MM3IDX_ERR_QUERY_LEN: return "query_len must be >= 1 and <= max_seq_len";
    case MM3IDX_ERR_TOPK: return "topk must be 1..32 with 0 <= init, local and init + local <= topk";
    case MM3IDX_ERR_OUT_LAYOUT: return "output buffer too small or strides overlap";
    case MM3IDX_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case MM3IDX_ERR_UNSUPPORTED: return "shape not served by this entry point";
    case MM3IDX_ERR_CUDA: return "CUDA runtime or driver call failed";
    case MM3IDX_ERR_STATIC_SCRATCH:
      return "problem needs more decode scratch than the library's static array (MM3IDX_STATIC_SCRATCH_BYTES)";
    default: return "unknown status";
  }
}

int mm3idx_workspace_bytes(int32_t op, int32_t heads, int32_t num_reqs, int32_t query_len,
                           int32_t max_seq_len, int32_t topk, size_t* bytes) {
  if (!bytes || heads < 1 || num_reqs < 0 || query_len < 1 || max_seq_len < 1)
    return MM3IDX_ERR_INVALID_ARGUMENT;
  if (op == MM3IDX_OP_DECODE) {
    if (topk < 1 || topk > MM3IDX_MAX_TOPK) return MM3IDX_ERR_TOPK;
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    *bytes = decode_ws_bytes(dev->sms, heads, num_reqs, query_len, topk);
    return MM3IDX_OK;
  }
  if (op == MM3IDX_OP_SCORE_NVFP4) {
    *bytes = score_nvfp4_ws_bytes(heads, num_reqs, query_len, max_seq_len);
    return MM3IDX_OK;
  }
  if (op == MM3IDX_OP_PREFILL || op == MM3IDX_OP_PREFILL_NVFP4) {
    if (topk < 1 || topk > MM3IDX_MAX_TOPK) return MM3IDX_ERR_TOPK;
    DeviceInfo* dev = nullptr;   // the list slots depend on the grid
    int rc = device_info(&dev);
    if (rc) return rc;
    *bytes = prefill_ws_bytes(dev->sms, heads, num_reqs, query_len, max_seq_len, topk,
                              op == MM3IDX_OP_PREFILL_NVFP4);
    return MM3IDX_OK;
  }
  return MM3IDX_ERR_INVALID_ARGUMENT;
}

int mm3idx_score(const mm3idx_problem_t* p, float* out, int64_t out_head_stride,
                 int64_t out_row_stride, void* stream) {
  return run_score(p, false, out, out_head_stride, out_row_stride, nullptr, 0, stream);
}

int mm3idx_score_nvfp4(const mm3idx_problem_t* p, float* out, int64_t out_head_stride,
                       int64_t out_row_stride, void* workspace, size_t workspace_bytes,
                       void* stream) {
  return run_score(p, true, out, out_head_stride, out_row_stride, workspace, workspace_bytes,
                   stream);
}

int mm3idx_score_ragged(const mm3idx_problem_t* p, const int32_t* cu_seqlens_q, int32_t total_q,
                        float* out, int64_t out_head_stride, int64_t out_row_stride,
                        void* stream) {
  int rc = check_problem(p, false);
  if (rc) return rc;
  if ((rc = check_ragged(p->num_reqs, p->query_len, cu_seqlens_q, total_q))) return rc;
  if (total_q == 0) return MM3IDX_OK;
  const int32_t width = static_cast<int32_t>(cdiv(p->max_seq_len, kBlock));
  if (!out || !out_ok(out_head_stride, out_row_stride, p->heads, total_q, width))
    return MM3IDX_ERR_OUT_LAYOUT;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  return score_then_fill(p, cu_seqlens_q, total_q, out, out_head_stride, out_row_stride, width,
                         dev, static_cast<cudaStream_t>(stream));
}

int mm3idx_topk(const float* score, int64_t score_head_stride, int64_t score_row_stride,
                int32_t heads, const int32_t* seq_lens, int32_t num_reqs, int32_t query_len,
                int32_t max_seq_len, int32_t topk, int32_t init_blocks, int32_t local_blocks,
                int32_t* out, int64_t out_head_stride, int64_t out_row_stride, void* stream) {
  const int64_t rows = static_cast<int64_t>(num_reqs) * query_len;
  if (rows >= INT_MAX) return MM3IDX_ERR_INVALID_ARGUMENT;
  return run_topk(score, score_head_stride, score_row_stride, heads, seq_lens, num_reqs,
                  query_len, nullptr, static_cast<int32_t>(rows), max_seq_len, topk, init_blocks,
                  local_blocks, out, out_head_stride, out_row_stride, stream);
}

int mm3idx_topk_ragged(const float* score, int64_t score_head_stride, int64_t score_row_stride,
                       int32_t heads, const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                       int32_t num_reqs, int32_t total_q, int32_t max_query_len,
                       int32_t max_seq_len, int32_t topk, int32_t init_blocks,
                       int32_t local_blocks, int32_t* out, int64_t out_head_stride,
                       int64_t out_row_stride, void* stream) {
  int rc = check_ragged(num_reqs, max_query_len, cu_seqlens_q, total_q);
  if (rc) return rc;
  return run_topk(score, score_head_stride, score_row_stride, heads, seq_lens, num_reqs,
                  max_query_len, cu_seqlens_q, total_q, max_seq_len, topk, init_blocks,
                  local_blocks, out, out_head_stride, out_row_stride, stream);
}

int mm3idx_decode(const mm3idx_problem_t* p, int32_t topk, int32_t init_blocks,
                  int32_t local_blocks, int32_t* out, int64_t out_head_stride,
                  int64_t out_row_stride, void* workspace, size_t workspace_bytes, void* stream) {
  return run_decode(p, false, topk, init_blocks, local_blocks, out, out_head_stride,
                    out_row_stride, workspace, workspace_bytes, stream);
}

int mm3idx_decode_sparse_table(const mm3idx_problem_t* p, int32_t topk, int32_t init_blocks,
                               int32_t local_blocks, int32_t* out, int64_t out_head_stride,
                               int64_t out_row_stride, const mm3idx_sparse_table_t* table,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (!p || !table) return MM3IDX_ERR_INVALID_ARGUMENT;
  return run_decode(p, p->index_scales != nullptr, topk, init_blocks, local_blocks, out,
                    out_head_stride, out_row_stride, workspace, workspace_bytes, stream, table);
}

int mm3idx_decode_nvfp4(const mm3idx_problem_t* p, int32_t topk, int32_t init_blocks,
                        int32_t local_blocks, int32_t* out, int64_t out_head_stride,
                        int64_t out_row_stride, void* workspace, size_t workspace_bytes,
                        void* stream) {
  return run_decode(p, true, topk, init_blocks, local_blocks, out, out_head_stride,
                    out_row_stride, workspace, workspace_bytes, stream);
}

int mm3idx_prefill(const mm3idx_problem_t* p, int32_t topk, int32_t init_blocks,
                   int32_t local_blocks, int32_t* out, int64_t out_head_stride,
                   int64_t out_row_stride, void* workspace, size_t workspace_bytes, void* stream) {
  return run_prefill(p, false, nullptr, -1, topk, init_blocks, local_blocks, out,
                     out_head_stride, out_row_stride, workspace, workspace_bytes, stream);
}

int mm3idx_prefill_nvfp4(const mm3idx_problem_t* p, int32_t topk, int32_t init_blocks,
                         int32_t local_blocks, int32_t* out, int64_t out_head_stride,
                         int64_t out_row_stride, void* workspace, size_t workspace_bytes,
                         void* stream) {
  return run_prefill(p, true, nullptr, -1, topk, init_blocks, local_blocks, out,
                     out_head_stride, out_row_stride, workspace, workspace_bytes, stream);
}

int mm3idx_prefill_ragged(const mm3idx_problem_t* p, const int32_t* cu_seqlens_q,
                          int32_t total_q, int32_t topk, int32_t init_blocks,
                          int32_t local_blocks, int32_t* out, int64_t out_head_stride,
                          int64_t out_row_stride, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (!p) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (!cu_seqlens_q && p->num_reqs > 0) return MM3IDX_ERR_INVALID_ARGUMENT;
  return run_prefill(p, p->index_scales != nullptr, cu_seqlens_q, total_q, topk, init_blocks,
                     local_blocks, out, out_head_stride, out_row_stride, workspace,
                     workspace_bytes, stream);
}

int mm3idx_decode_static(const mm3idx_problem_t* p, int32_t topk, int32_t init_blocks,
                         int32_t local_blocks, int32_t* out, int64_t out_head_stride,
                         int64_t out_row_stride, void* stream) {
  int rc = check_problem(p, false);
  if (rc) return rc;
  if ((rc = check_topk(topk, init_blocks, local_blocks))) return rc;
  if (static_cast<int64_t>(p->num_reqs) * p->query_len == 0) return MM3IDX_OK;
  void* scratch = nullptr;
  if ((rc = static_scratch(&scratch))) return rc;
  // Every argument check runs before the tickets are cleared (inside
  // run_decode), so a rejected call leaves the shared array untouched.
  return run_decode(p, false, topk, init_blocks, local_blocks, out, out_head_stride,
                    out_row_stride, scratch, MM3IDX_STATIC_SCRATCH_BYTES, stream, nullptr,
                    /*static_scratch=*/true);
}

int mm3idx_forward_workspace_bytes(int32_t heads, int32_t num_decodes, int32_t decode_query_len,
                                   int32_t num_prefills, int32_t prefill_max_query_len,
                                   int32_t max_seq_len, int32_t topk, int32_t nvfp4,
                                   size_t* bytes) {
  if (!bytes || heads < 1 || num_decodes < 0 || num_prefills < 0 || decode_query_len < 1 ||
      prefill_max_query_len < 1 || max_seq_len < 1)
    return MM3IDX_ERR_INVALID_ARGUMENT;
  if (topk < 1 || topk > MM3IDX_MAX_TOPK) return MM3IDX_ERR_TOPK;
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  *bytes = forward_ws_bytes(dev->sms, heads, num_decodes, decode_query_len, num_prefills,
                            prefill_max_query_len, max_seq_len, topk, nvfp4 != 0);
  return MM3IDX_OK;
}

int mm3idx_forward(const mm3idx_problem_t* p, int32_t num_decodes,
                   const int32_t* prefill_cu_seqlens_q, int32_t prefill_total_q,
                   int32_t prefill_max_query_len, int32_t topk, int32_t init_blocks,
                   int32_t local_blocks, int32_t* out, int64_t out_head_stride,
                   int64_t out_row_stride, void* workspace, size_t workspace_bytes,
                   void* stream) {
  if (!p) return MM3IDX_ERR_INVALID_ARGUMENT;
  const bool nvfp4 = p->index_scales != nullptr;
  int rc = check_problem(p, nvfp4);
  if (rc) return rc;
  if ((rc = check_topk(topk, init_blocks, local_blocks))) return rc;
  if (num_decodes < 0 || num_decodes > p->num_reqs || prefill_max_query_len < 1)
    return MM3IDX_ERR_INVALID_ARGUMENT;
  const int32_t num_prefills = p->num_reqs - num_decodes;
  if ((rc = check_ragged(num_prefills, prefill_max_query_len, prefill_cu_seqlens_q,
                         prefill_total_q)))
    return rc;
  if (prefill_max_query_len > p->max_seq_len) return MM3IDX_ERR_QUERY_LEN;
  if (num_decodes > 0 && p->heads * static_cast<int64_t>(p->query_len) > MM3IDX_MAX_DECODE_ROWS)
    return MM3IDX_ERR_UNSUPPORTED;
  const int64_t dec_rows = static_cast<int64_t>(num_decodes) * p->query_len;
  if (dec_rows + prefill_total_q >= INT_MAX) return MM3IDX_ERR_INVALID_ARGUMENT;
  if (dec_rows + prefill_total_q == 0) return MM3IDX_OK;
  if (!out || !out_ok(out_head_stride, out_row_stride, p->heads, dec_rows + prefill_total_q, topk))
    return MM3IDX_ERR_OUT_LAYOUT;
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  const size_t dec_ws = num_decodes > 0
      ? align256(decode_ws_bytes(dev->sms, p->heads, num_decodes, p->query_len, topk)) : 0;
  const size_t need = forward_ws_bytes(dev->sms, p->heads, num_decodes, p->query_len,
                                       num_prefills, prefill_max_query_len, p->max_seq_len, topk,
                                       nvfp4);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MM3IDX_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // The decode part: requests 0 .. num_decodes-1, rows 0 .. dec_rows-1.
  if (num_decodes > 0) {
    mm3idx_problem_t d = *p;
    d.num_reqs = num_decodes;
    if ((rc = run_decode(&d, nvfp4, topk, init_blocks, local_blocks, out, out_head_stride,
                         out_row_stride, ws, dec_ws, stream)))
      return rc;
  }
  if (num_prefills == 0 || prefill_total_q == 0) return MM3IDX_OK;
  // The prefill part: the remaining requests and rows, after the decode in
  // stream order.  (Launched as a programmatic dependent of the decode, to
  // start on the SMs its CTAs free, the prefill measured 4 % slower: its CTAs'
  // equal shares started unevenly.)
  mm3idx_problem_t f = *p;
  f.num_reqs = num_prefills;
  f.query_len = prefill_max_query_len;
  f.idx_q = static_cast<const uint16_t*>(p->idx_q) + dec_rows * p->q_token_stride;
  f.block_table = p->block_table + static_cast<int64_t>(num_decodes) * p->table_stride;
  f.seq_lens = p->seq_lens + num_decodes;
  return run_prefill(&f, nvfp4, prefill_cu_seqlens_q, prefill_total_q, topk, init_blocks,
                     local_blocks, out + dec_rows * out_row_stride, out_head_stride,
                     out_row_stride, ws + dec_ws, workspace_bytes - dec_ws, stream);
}

int mm3idx_get_device_error(void* stream, int32_t* code) {
  if (!code) return MM3IDX_ERR_INVALID_ARGUMENT;
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MM3IDX_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MM3IDX_ERR_CUDA;
  const int32_t zero = 0;
  if (cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return MM3IDX_ERR_CUDA;
  *code = v;
  return MM3IDX_OK;
}

}  // extern "C"
