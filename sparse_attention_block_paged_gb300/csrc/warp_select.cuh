// warp_select.cuh -- the forced-block rule shared by the selector kernel and
// the decode kernel's row writers.
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

// Forced block range of a row whose own block is c: [0, f_lo) and [l_lo, c].
struct Forced {
  int f_lo, l_lo, nf;
  __device__ __forceinline__ Forced(int c, int init_blocks, int local_blocks) {
    f_lo = min(init_blocks, c + 1);
    l_lo = max(f_lo, c - local_blocks + 1);
    nf = f_lo + (c + 1 - l_lo);
  }
};

}  // namespace mm3idx
