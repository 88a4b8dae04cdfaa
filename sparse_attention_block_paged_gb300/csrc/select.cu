// select.cu -- top-k block selection from an fp32 score tensor, one warp per
// (head, query row).
//
// Follows the vLLM MiniMax-M3 "index_topk" page, minimax_m3_index_topk
// (top-k from a precomputed score tensor, forced init/local blocks kept,
// output [heads, total_q, topk] of 0-indexed block ids with -1 pad) and the
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

namespace mm3idx {
namespace {

constexpr int kPerLane = 8;
constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ uint64_t warp_max_key(uint64_t k) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(k >> 32));
  const uint32_t lo = __reduce_max_sync(
      0xffffffffu, static_cast<uint32_t>(k >> 32) == hi ? static_cast<uint32_t>(k) : 0u);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

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
    if (c < 0) {
      for (int k = lane; k < topk; k += 32) out[k] = -1;
      continue;
    }
    const int f_lo = min(a.init_blocks, c + 1);
    const int l_lo = max(f_lo, c - a.local_blocks + 1);
    const int nf = f_lo + (c + 1 - l_lo);
    const int m = topk - nf;
    const int ncand = l_lo - f_lo;
    if (ncand <= m) {
      for (int k = lane; k < topk; k += 32) out[k] = k <= c ? k : -1;
      continue;
    }
    const float* srow = a.score + h * a.s_head + row * a.s_row;
    uint64_t mine = 0;  // lane r < m holds the r-th best key so far
    uint64_t thr = 0;   // m-th best so far, 0 while fewer than m are known
    for (int base = f_lo; base < l_lo; base += 32 * kPerLane) {
      uint64_t k[kPerLane];
      bool any = false;
#pragma unroll
      for (int p = 0; p < kPerLane; ++p) {
        const int idx = base + p * 32 + lane;
        k[p] = 0;
        if (idx < l_lo) {
          const uint64_t key = make_key(__ldg(srow + idx), idx);
          if (key > thr) k[p] = key;
        }
        any |= k[p] != 0;
      }
      if (!__any_sync(0xffffffffu, any)) continue;
      bool list_taken = false;
      uint64_t next = 0;
      for (int r = 0; r < m; ++r) {
        uint64_t best = list_taken ? 0ull : mine;
#pragma unroll
        for (int p = 0; p < kPerLane; ++p) best = k[p] > best ? k[p] : best;
        const uint64_t win = warp_max_key(best);
        if (win == 0) break;
        if (lane == r) next = win;
        if (best == win) {
          if (!list_taken && mine == win) {
            list_taken = true;
          } else {
#pragma unroll
            for (int p = 0; p < kPerLane; ++p)
              if (k[p] == win) k[p] = 0;
          }
        }
      }
      mine = next;
      thr = __shfl_sync(0xffffffffu, mine, m - 1);
    }
    // Output: forced blocks around the picks, picks in ascending id order.
    const int bx = lane < m ? key_block(mine) : 0x7fffffff;
    int rank = 0;
    for (int q = 0; q < m; ++q) rank += __shfl_sync(0xffffffffu, bx, q) < bx;
    if (lane < m) out[f_lo + rank] = bx;
    for (int b = lane; b < f_lo; b += 32) out[b] = b;
    for (int b = l_lo + lane; b <= c; b += 32) out[f_lo + m + (b - l_lo)] = b;
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
