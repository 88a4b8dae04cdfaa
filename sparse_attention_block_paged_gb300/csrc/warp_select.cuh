// warp_select.cuh -- the forced-block rule, the per-thread candidate list
// and the row writer shared by the selector, decode and prefill kernels.
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

constexpr int kListLanes = 32;  // rows of a shared-memory hand-over table

// A row's best candidate keys, descending, held in registers (0 = empty).
// Insertion is a branchless compare-and-swap cascade with static indices.
template <int TK>
struct RegList {
  uint64_t v[TK];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int k = 0; k < TK; ++k) v[k] = 0ull;
  }
  // Keys at or below this cannot enter.
  __device__ __forceinline__ uint64_t floor() const { return v[TK - 1]; }
  __device__ __forceinline__ void insert(uint64_t key) {
#pragma unroll
    for (int k = 0; k < TK; ++k) {
      const uint64_t cur = v[k];
      const bool gt = key > cur;
      v[k] = gt ? key : cur;
      key = gt ? cur : key;
    }
  }
  __device__ __forceinline__ void offer(uint64_t key) {
    if (key > floor()) insert(key);
  }
  // Insertion of a key whose block comes after every block in the list (a
  // row's blocks offered in ascending order), with a short dependency chain.
  // A listed key then ranks above the new one exactly when its score is at
  // least the new one's (an equal score loses on the higher block id), so
  // the score halves alone decide: one 32-bit compare a slot instead of a
  // 64-bit one (in the prefill scorer's 16-key epilogue: causal 32K step
  // 119.5 -> 113.8 us, chunked batch 95.7 -> 91.2 us).  In a list sorted
  // descending, "v[k] ranks above key" holds exactly for k below the key's
  // place, so each new slot follows from the old slot, its predecessor and
  // the key alone (about four dependent steps instead of TK).  Only the
  // first N slots are kept (the rest stay as they are): a caller that needs
  // at most N keys spends no work on the others.
  template <int N = TK>
  __device__ __forceinline__ void offer_ascending(uint64_t key) {
    static_assert(N >= 1 && N <= TK, "slots in use");
    const uint32_t ks = static_cast<uint32_t>(key >> 32);
    if (ks <= static_cast<uint32_t>(v[N - 1] >> 32)) return;
    bool above_prev = true;  // v[k-1] ranks above key, with v[-1] above every key
    uint64_t prev = 0ull;
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const uint64_t cur = v[k];
      const bool above = static_cast<uint32_t>(cur >> 32) >= ks;
      v[k] = above ? cur : (above_prev ? key : prev);
      above_prev = above;
      prev = cur;
    }
  }
  // Replace the list by the best TK keys of itself and `b` (b sorted
  // descending): the elementwise max of the list and reversed b holds exactly
  // those keys as a bitonic sequence, which a bitonic sort orders again.
  __device__ __forceinline__ void merge_sorted(const uint64_t (&b)[TK]) {
#pragma unroll
    for (int k = 0; k < TK; ++k) v[k] = v[k] > b[TK - 1 - k] ? v[k] : b[TK - 1 - k];
    clean();
  }
  // The same for eight keys in any order (zeros for none): b is sorted first
  // (an optimal 19-comparator network for eight inputs, Knuth, The Art of
  // Computer Programming vol. 3, 5.3.4), then taken as b padded with zeros:
  // only the last eight slots meet a nonzero key.  About 107 compare-
  // exchanges for eight keys, where eight insertions move all TK slots each.
  __device__ __forceinline__ void merge8(uint64_t (&b)[8]) {
    constexpr int kNet[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6},
                                 {3, 7}, {0, 1}, {2, 3}, {4, 5}, {6, 7}, {2, 4}, {3, 5},
                                 {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
    for (int n = 0; n < 19; ++n) {
      const uint64_t x = b[kNet[n][0]], y = b[kNet[n][1]];
      b[kNet[n][0]] = x > y ? x : y;
      b[kNet[n][1]] = x > y ? y : x;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = TK - 8 + j;
      v[k] = v[k] > b[7 - j] ? v[k] : b[7 - j];
    }
    clean();
  }
  // Sort a bitonic list descending (half-cleaners, TK/2 apart down to 1).
  __device__ __forceinline__ void clean() {
#pragma unroll
    for (int half = TK / 2; half > 0; half >>= 1) {
#pragma unroll
      for (int k = 0; k < TK; ++k) {
        if ((k & half) == 0) {
          const uint64_t x = v[k], y = v[k + half];
          v[k] = x > y ? x : y;
          v[k + half] = x > y ? y : x;
        }
      }
    }
  }
  // Row-major store to a [k][kListLanes] shared-memory table at column n.
  __device__ __forceinline__ void store_cols(uint64_t* t, int n) const {
#pragma unroll
    for (int k = 0; k < TK; ++k) t[k * kListLanes + n] = v[k];
  }
};

// One thread writes one output row from its candidate list (keys sorted
// descending, 0 = none): forced blocks [0, f_lo) and [l_lo, c] around the best
// topk - |forced| picks, picks in ascending id order, then -1.  dry: the same
// work without the stores.
template <int TK>
__device__ __forceinline__ void write_row_lane(const uint64_t (&v)[TK], int c, int init_blocks,
                                               int local_blocks, int topk, int32_t* out,
                                               bool dry = false) {
  if (c < 0) {
    if (!dry)
      for (int k = 0; k < topk; ++k) out[k] = -1;
    return;
  }
  const Forced F(c, init_blocks, local_blocks);
  const int m = topk - F.nf;
  int id[TK];
  int npick = 0;
#pragma unroll
  for (int k = 0; k < TK; ++k) {
    const bool take = k < m && v[k] != 0ull;
    id[k] = take ? key_block(v[k]) : 0x7fffffff;
    npick += take;
  }
  // Bitonic sort of the ids, ascending (absent picks sort to the end).
#pragma unroll
  for (int size = 2; size <= TK; size <<= 1) {
#pragma unroll
    for (int stride = size / 2; stride > 0; stride >>= 1) {
#pragma unroll
      for (int k = 0; k < TK; ++k) {
        const int l = k ^ stride;
        if (l > k) {
          const bool up = (k & size) == 0;
          const int x = id[k], y = id[l];
          id[k] = (x < y) == up ? x : y;
          id[l] = (x < y) == up ? y : x;
        }
      }
    }
  }
  if (dry) return;
  int o = 0;
  for (int b = 0; b < F.f_lo; ++b) out[o++] = b;
#pragma unroll
  for (int k = 0; k < TK; ++k)
    if (k < npick) out[o + k] = id[k];
  o += npick;
  for (int b = F.l_lo; b <= c; ++b) out[o++] = b;
  for (; o < topk; ++o) out[o] = -1;
}

}  // namespace mm3idx
