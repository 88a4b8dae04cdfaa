// sparse_table.cu -- the page table of the block-sparse attention that reads
// the selected blocks (vLLM MiniMax-M3 "index_topk" page,
// minimax_m3_index_decode: attention_block_table, sparse_block_table_out,
// sparse_context_lens_out, block_page_stride; one index head).
//
// One warp per query row, lane k on the row's k-th id (ids ascending, -1
// pad, as the selection writes them): the P pages of block b are
// attn_table[i, b] * block_page_stride + 0..P-1, -1 for a -1 slot; the
// row's context length is the sum over its selected blocks of their tokens
// at or before the row's position (the selected blocks end to end, the last
// one cut at pos).
//
// The kernel is launched as a programmatic dependent of the decode kernel
// that writes the ids: its CTAs may start while the decode still runs and
// wait for it with griddepcontrol.wait, so the table costs no launch gap.
// The table's work (one 4-byte load per id, P stores) is kept out of the
// decode kernel, whose end is latency-critical.
#include <cuda_runtime.h>

#include "../../include/mm3idx.h"
#include "internal.h"

namespace mm3idx {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) sparse_table_kernel(const SparseTableArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(a.num_reqs) * a.query_len;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const bool live = row < rows;
  int i = 0, pos = -1;
  if (live) {
    // Inputs the decode does not write: read them, and pull the row's
    // attention-table entries into L2, while the decode still runs.
    i = static_cast<int>(row / a.query_len);
    const int j = static_cast<int>(row - static_cast<int64_t>(i) * a.query_len);
    const int seq = min(max(__ldg(a.seq_lens + i), 0), a.max_seq_len);
    pos = seq - a.query_len + j;
    const int nb = pos >= 0 ? (pos >> 7) + 1 : 0;
    for (int k = lane * 32; k < nb; k += 32 * 32)  // one 128-byte line per lane
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a.attn_table + i * a.attn_stride + k));
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!live) return;
  const int P = a.pages_per_block;
  int32_t* st = a.st_out + row * a.st_stride;
  int ctx = 0;
  if (lane < a.topk) {
    const int b = a.ids[row * a.i_row + lane];
    // only ids the row can see (which keeps the table read in bounds even
    // when a decode that gave up left its ids unwritten)
    if (b >= 0 && pos >= 0 && b <= (pos >> 7)) {
      // unsigned: wraps like the int32 result asked for, no overflow UB
      const unsigned base = static_cast<unsigned>(__ldg(a.attn_table + i * a.attn_stride + b)) *
                            static_cast<unsigned>(a.block_page_stride);
      for (int p = 0; p < P; ++p) st[lane * P + p] = static_cast<int32_t>(base + p);
      ctx = min(kBlock, pos + 1 - b * kBlock);
    } else {
      for (int p = 0; p < P; ++p) st[lane * P + p] = -1;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ctx += __shfl_xor_sync(0xffffffffu, ctx, o);
  if (lane == 0) a.ctx_out[row] = ctx;
}

}  // namespace

cudaError_t launch_sparse_table(const SparseTableArgs& a, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.num_reqs) * a.query_len;
  if (rows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + kWarps - 1) / kWarps));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_table_kernel, a);
}

}  // namespace mm3idx
