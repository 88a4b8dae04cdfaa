// select.cu -- top-k block selection from an fp32 score tensor, one warp per
// (head, query row).
//
// Follows the vLLM MiniMax-M3 "index_topk" page, minimax_m3_index_topk
// (top-k from a precomputed score tensor, forced init/local blocks kept,
// output [heads, total_q, topk] of logical block ids counted from 0, -1 pad) and the
// "indexer_cp_exchange" page (packed 64-bit (score, id) keys, ids < 0xFFFF).
//
// Per row: forced blocks F = [0, f_lo) and [l_lo, c]; candidates are the
// visible blocks in [f_lo, l_lo).  When there are at most topk - |F| of them
// the row is simply 0..c.  Otherwise the warp streams the candidates in
// chunks of 32 * kPerLane keys, keeps a running top-m list (one key per lane,
// sorted by lane) and merges each chunk by m rounds of a warp-wide max; keys
// that cannot beat the current m-th best are dropped before the merge.
#include <cuda_runtime.h>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "ptx.cuh"
#include "warp_select.cuh"

namespace mm3idx {
namespace {

constexpr int kPerLane = 8;
constexpr int kWarpsPerBlock = 8;

__global__ void __launch_bounds__(kWarpsPerBlock * 32) select_kernel(const SelectArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(a.num_reqs) * a.query_len;
  const int64_t work = rows * a.heads;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); w < work;
       w += nwarps) {
    const int h = static_cast<int>(w / rows);
    const int64_t row = w - static_cast<int64_t>(h) * rows;
    const int i = static_cast<int>(row / a.query_len);
    const int j = static_cast<int>(row - static_cast<int64_t>(i) * a.query_len);
    const int seq = min(max(__ldg(a.seq_lens + i), 0), a.max_seq_len);
    const int pos = seq - a.query_len + j;
    const int c = pos >= 0 ? (pos >> 7) : -1;
    int32_t* out = a.ids + h * a.i_head + row * a.i_row;
    const int topk = a.topk;
    const Forced F(c, a.init_blocks, a.local_blocks);
    const int m = topk - F.nf;
    uint64_t mine = 0;  // lane r < m holds the r-th best key so far
    if (c >= 0 && F.l_lo - F.f_lo > m) {
      const float* srow = a.score + h * a.s_head + row * a.s_row;
      uint64_t thr = 0;
      for (int base = F.f_lo; base < F.l_lo; base += 32 * kPerLane) {
        uint64_t k[kPerLane];
#pragma unroll
        for (int p = 0; p < kPerLane; ++p) {
          const int idx = base + p * 32 + lane;
          k[p] = idx < F.l_lo ? make_key(__ldg(srow + idx), idx) : 0ull;
        }
        warp_topm_merge<kPerLane>(k, m, mine, thr, lane);
      }
    } else if (c >= 0) {
      // At most m candidates: take them all (any order; the writer sorts).
      const int idx = F.f_lo + lane;
      mine = (lane < m && idx < F.l_lo) ? make_key(0.f, idx) : 0ull;
    }
    warp_write_row(c, a.init_blocks, a.local_blocks, topk, mine, out, lane);
  }
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, int num_sms, cudaStream_t s) {
  const int64_t work = static_cast<int64_t>(a.num_reqs) * a.query_len * a.heads;
  int64_t blocks = (work + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  select_kernel<<<static_cast<int>(blocks), kWarpsPerBlock * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mm3idx
