// warp_select.cuh -- warp-wide top-m selection over packed (score, block id)
// keys and the forced-block output rule, shared by the selector kernel and
// the decode kernel's cross-CTA merge.
//
// Selection rule (vLLM MiniMax-M3 "index_topk" page, minimax_m3_index_decode
// and minimax_m3_index_topk; "indexer_cp_exchange" module docstring): for a
// row whose own block is c, the forced blocks 0..init-1 and c-local+1..c
// (clipped to 0..c) are always kept; the best topk-|forced| of the remaining
// visible blocks, ranked by higher score then lower id, join them; the row is
// written in ascending id order and padded with -1.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace mm3idx {

// Largest key held by any lane (keys are unique, so exactly one lane owns it).
__device__ __forceinline__ uint64_t warp_max_key(uint64_t k) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(k >> 32));
  const uint32_t lo = __reduce_max_sync(
      0xffffffffu, static_cast<uint32_t>(k >> 32) == hi ? static_cast<uint32_t>(k) : 0u);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// A warp's running top-m list: lane r < m holds the r-th largest key seen so
// far in `mine` (0 = none); `thr` is the m-th largest (0 while fewer than m
// keys were seen).  Merges P more keys per lane (0 = none) into it.
template <int P>
__device__ __forceinline__ void warp_topm_merge(uint64_t (&k)[P], int m, uint64_t& mine,
                                                uint64_t& thr, int lane) {
  bool any = false;
#pragma unroll
  for (int p = 0; p < P; ++p) {
    if (k[p] <= thr) k[p] = 0;
    any |= k[p] != 0;
  }
  if (!__any_sync(0xffffffffu, any)) return;
  bool list_taken = false;
  uint64_t next = 0;
  for (int r = 0; r < m; ++r) {
    uint64_t best = list_taken ? 0ull : mine;
#pragma unroll
    for (int p = 0; p < P; ++p) best = k[p] > best ? k[p] : best;
    const uint64_t win = warp_max_key(best);
    if (win == 0) break;
    if (lane == r) next = win;
    if (best == win) {
      if (!list_taken && mine == win) {
        list_taken = true;
      } else {
#pragma unroll
        for (int p = 0; p < P; ++p)
          if (k[p] == win) k[p] = 0;
      }
    }
  }
  mine = next;
  thr = m > 0 ? __shfl_sync(0xffffffffu, mine, m - 1) : ~0ull;
}

// Forced block range of a row whose own block is c: [0, f_lo) and [l_lo, c].
struct Forced {
  int f_lo, l_lo, nf;
  __device__ __forceinline__ Forced(int c, int init_blocks, int local_blocks) {
    f_lo = min(init_blocks, c + 1);
    l_lo = max(f_lo, c - local_blocks + 1);
    nf = f_lo + (c + 1 - l_lo);
  }
};

// Writes one output row: forced blocks and the picks held in lanes 0..m-1 of
// `mine` (0 = none), in ascending id order, then -1 up to topk.
__device__ __forceinline__ void warp_write_row(int c, int init_blocks, int local_blocks, int topk,
                                               uint64_t mine, int32_t* out, int lane) {
  if (c < 0) {
    for (int k = lane; k < topk; k += 32) out[k] = -1;
    return;
  }
  const Forced F(c, init_blocks, local_blocks);
  const int m = topk - F.nf;
  const bool have = lane < m && mine != 0ull;
  const int npick = __popc(__ballot_sync(0xffffffffu, have));
  const int id = have ? key_block(mine) : 0x7fffffff;
  int rank = 0;
  for (int q = 0; q < npick; ++q) rank += __shfl_sync(0xffffffffu, id, q) < id;
  if (have) out[F.f_lo + rank] = id;
  for (int b = lane; b < F.f_lo; b += 32) out[b] = b;
  for (int b = F.l_lo + lane; b <= c; b += 32) out[F.f_lo + npick + (b - F.l_lo)] = b;
  for (int k = F.nf + npick + lane; k < topk; k += 32) out[k] = -1;
}

}  // namespace mm3idx
