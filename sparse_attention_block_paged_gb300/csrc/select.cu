// select.cu -- top-k block selection from an fp32 score tensor, one warp per
// (head, query row).
//
// Follows the vLLM MiniMax-M3 "index_topk" page, minimax_m3_index_topk
// (top-k from a precomputed score tensor, forced init/local blocks kept,
// output [heads, total_q, topk] of logical block ids counted from 0, -1 pad) and the
// "indexer_cp_exchange" page (ranking by score, then lower block id).
//
// Rows: query_len per request, or, for a ragged batch, the rows
// cu[i]..cu[i+1]-1 of request i (minimax_m3_index_topk: cu_seqlens_q and
// prefix_lens), row j of request i at position seq_len[i] - rows_i + j.
//
// Per row: forced blocks F = [0, f_lo) and [l_lo, c]; candidates are the
// visible blocks in [f_lo, l_lo).  When there are at most m = topk - |F| of
// them the row is simply 0..c.  Otherwise the warp takes the candidates 256
// at a time (eight per lane), as unique 64-bit keys (score bits above the
// block id, so higher score then lower id wins).  The best m so far ride
// along in lanes 0..m-1.  Per chunk:
//   1. each lane's largest score (its best four when m > 16); m rounds of a
//      warp-wide max give T, the m-th largest of these -- at least m scores
//      are >= T, so every key of the top m has a score >= T;
//   2. the keys with scores >= T (typically about m + a few) are compacted
//      into one key per lane through shared memory and sorted; lanes 0..m-1
//      keep the best;
//   3. if more than 32 scores are >= T, m rounds of a warp-wide max take the
//      best m directly instead.
// The picks' ids are then sorted across the warp and the row written.
#include <cuda_runtime.h>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "ptx.cuh"
#include "warp_select.cuh"

namespace mm3idx {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kPer = 8;  // keys per lane per chunk
constexpr unsigned kFull = 0xffffffffu;

// Bitonic sort of one key per lane; lane 0 ends with the largest.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t o = __shfl_xor_sync(kFull, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// Bitonic sort of one int per lane; lane 0 ends with the smallest.
__device__ __forceinline__ int warp_sort_asc(int v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int o = __shfl_xor_sync(kFull, v, stride);
      const bool keep_min = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_min ? min(v, o) : max(v, o);
    }
  }
  return v;
}

// Largest key held by any lane (keys are unique, so one lane holds it).
__device__ __forceinline__ uint64_t warp_max_key(uint64_t k) {
  const uint32_t hi = __reduce_max_sync(kFull, static_cast<uint32_t>(k >> 32));
  const uint32_t lo =
      __reduce_max_sync(kFull, static_cast<uint32_t>(k >> 32) == hi ? static_cast<uint32_t>(k) : 0u);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Ragged batches: the request owning `row` (the last i with cu[i] <= row)
// and the row's index j in it; false when the offsets do not place the row
// inside its request (malformed offsets).
__device__ __forceinline__ bool ragged_row(const SelectArgs& a, int64_t row, int& i, int& j,
                                           int& ql) {
  int lo = 0, hi = a.num_reqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.cu + mid) <= row) lo = mid;
    else hi = mid - 1;
  }
  i = lo;
  const int b = __ldg(a.cu + i), e = __ldg(a.cu + i + 1);
  ql = e - b;
  j = static_cast<int>(row - b);
  return b <= row && row < e;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32, 3) select_kernel(const SelectArgs a) {
  __shared__ uint64_t s_buf[kWarpsPerBlock][32];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  uint64_t* buf = s_buf[wib];
  const int64_t rows = a.total_q;
  const int64_t work = rows * a.heads;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  if (a.cu != nullptr && blockIdx.x == 0 && wib == 0) {
    // the offsets must run from 0 to total_q without decreasing
    bool bad = lane == 0 && (__ldg(a.cu) != 0 || __ldg(a.cu + a.num_reqs) != a.total_q);
    for (int i = lane; i < a.num_reqs; i += 32) bad |= __ldg(a.cu + i + 1) < __ldg(a.cu + i);
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, MM3IDX_DEV_BAD_ROWS);
  }
  // 32-bit index arithmetic when the problem allows it (64-bit divisions
  // cost more than the selection itself).
  const bool small = work < (int64_t{1} << 31);
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + wib; w < work; w += nwarps) {
    int h, i, j;
    int64_t row;
    int ql = a.query_len;
    bool row_ok = true;
    if (a.cu != nullptr) {
      h = static_cast<int>(w / rows);
      row = w - static_cast<int64_t>(h) * rows;
      row_ok = ragged_row(a, row, i, j, ql);
    } else if (small) {
      const uint32_t w32 = static_cast<uint32_t>(w), rows32 = static_cast<uint32_t>(rows);
      const uint32_t ql32 = static_cast<uint32_t>(a.query_len);
      h = static_cast<int>(w32 / rows32);
      const uint32_t r32 = w32 - static_cast<uint32_t>(h) * rows32;
      i = static_cast<int>(r32 / ql32);
      j = static_cast<int>(r32 - static_cast<uint32_t>(i) * ql32);
      row = r32;
    } else {
      h = static_cast<int>(w / rows);
      row = w - static_cast<int64_t>(h) * rows;
      i = static_cast<int>(row / a.query_len);
      j = static_cast<int>(row - static_cast<int64_t>(i) * a.query_len);
    }
    const int seq = min(max(__ldg(a.seq_lens + i), 0), a.max_seq_len);
    const int pos = seq - ql + j;
    const int c = row_ok && pos >= 0 ? (pos >> 7) : -1;
    int32_t* out = a.ids + h * a.i_head + row * a.i_row;
    const int topk = a.topk;
    if (c < 0) {
      for (int k = lane; k < topk; k += 32) out[k] = -1;
      continue;
    }
    const Forced F(c, a.init_blocks, a.local_blocks);
    const int m = topk - F.nf;
    if (F.l_lo - F.f_lo <= m) {
      // Every visible block is kept.
      for (int k = lane; k < topk; k += 32) out[k] = k <= c ? k : -1;
      continue;
    }
    const float* srow = a.score + h * a.s_head + row * a.s_row;
    uint64_t run = 0;  // lane r < m: the r-th best key so far
    for (int base = F.f_lo; m > 0 && base < F.l_lo; base += 32 * kPer) {
      float v[kPer];
#pragma unroll
      for (int p = 0; p < kPer; ++p) {
        const int idx = base + p * 32 + lane;
        v[p] = idx < F.l_lo ? __ldg(srow + idx) : -INFINITY;
      }
      const uint32_t rs = static_cast<uint32_t>(run >> 32);
      uint32_t T;
      if (m <= 16) {
        // This lane's largest score (ordered bits; 0 = none) among its
        // candidates and its best-so-far key.
        float fm = v[0];
#pragma unroll
        for (int p = 1; p < kPer; ++p) fm = fmaxf(fm, v[p]);
        const bool any = base + lane < F.l_lo;
        uint32_t lm = any ? ordered_bits(fm) : 0u;
        lm = rs > lm ? rs : lm;
        // T: the m-th largest of the 32 lane maxima (equal maxima leave
        // together, which only lowers T).  At least m lanes hold a score (the
        // best-so-far list, or, in the first chunk, more than m candidates).
        uint32_t rem = lm;
        T = lm;
        for (int r = 0; r < m; ++r) {
          const uint32_t mx = __reduce_max_sync(kFull, rem);
          if (mx == 0u) break;
          T = mx;
          if (rem == mx) rem = 0u;
        }
      } else {
        // Larger m: the m-th largest of the lanes' four best scores each
        // (a subset of the chunk's scores and the best-so-far keys, so at
        // least m scores reach it).  With the lane maxima alone, about 60 of
        // 256 N(0,1) scores reach the 29th-largest lane maximum and the
        // selection falls back to m rounds of a 64-bit warp max; the
        // 29th-largest of the lanes' best four lets about 29 through.
        uint32_t best4[4] = {0u, 0u, 0u, 0u};   // descending
        auto ins = [&](uint32_t x) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t hi = best4[k] > x ? best4[k] : x, lo = best4[k] > x ? x : best4[k];
            best4[k] = hi;
            x = lo;
          }
        };
#pragma unroll
        for (int p = 0; p < kPer; ++p)
          if (base + p * 32 + lane < F.l_lo) ins(ordered_bits(v[p]));
        ins(rs);
        T = best4[0];
        for (int r = 0; r < m; ++r) {
          const uint32_t mx = __reduce_max_sync(kFull, best4[0]);
          if (mx == 0u) break;
          T = mx;
          if (best4[0] == mx) {   // this lane's best leaves (equal ones together)
            best4[0] = best4[1];
            best4[1] = best4[2];
            best4[2] = best4[3];
            best4[3] = 0u;
          }
        }
      }
      const bool run_in = run != 0ull && rs >= T;
      uint32_t hit = 0;  // bit p: v[p] survives
#pragma unroll
      for (int p = 0; p < kPer; ++p)
        if (base + p * 32 + lane < F.l_lo && ordered_bits(v[p]) >= T) hit |= 1u << p;
      const int cnt = __popc(hit) + (run_in ? 1 : 0);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      const int total = __shfl_sync(kFull, incl, 31);
      if (total <= 32) {
        int off = incl - cnt;
        if (run_in) buf[off++] = run;
#pragma unroll
        for (int p = 0; p < kPer; ++p)
          if (hit & (1u << p)) buf[off++] = make_key(v[p], base + p * 32 + lane);
        __syncwarp();
        const uint64_t x = lane < total ? buf[lane] : 0ull;
        __syncwarp();
        const uint64_t srt = warp_sort_desc(x, lane);
        run = lane < m ? srt : 0ull;
      } else {
        // Many scores at or above T: take the best m one at a time.
        uint64_t k[kPer];
#pragma unroll
        for (int p = 0; p < kPer; ++p) {
          const int idx = base + p * 32 + lane;
          k[p] = idx < F.l_lo ? make_key(v[p], idx) : 0ull;
        }
        uint64_t next = 0;
        bool run_taken = false;
        for (int r = 0; r < m; ++r) {
          uint64_t best = run_taken ? 0ull : run;
#pragma unroll
          for (int p = 0; p < kPer; ++p) best = k[p] > best ? k[p] : best;
          const uint64_t win = warp_max_key(best);
          if (lane == r) next = win;
          if (best == win) {
            if (!run_taken && run == win) {
              run_taken = true;
            } else {
#pragma unroll
              for (int p = 0; p < kPer; ++p)
                if (k[p] == win) k[p] = 0ull;
            }
          }
        }
        run = next;
      }
    }
    // Row: forced init blocks, the m picks in ascending id order, the local
    // blocks, then -1.
    const int id = warp_sort_asc(lane < m ? key_block(run) : 0x7fffffff, lane);
    if (lane < F.f_lo) out[lane] = lane;
    if (lane < m) out[F.f_lo + lane] = id;
    for (int b = F.l_lo + lane; b <= c; b += 32) out[F.f_lo + m + (b - F.l_lo)] = b;
    for (int k = F.nf + m + lane; k < topk; k += 32) out[k] = -1;
  }
}

}  // namespace

// Blocks past each row's own block hold -inf, up to `width` (the score call's
// output contract): one warp per (head, row), lanes on consecutive blocks.
__global__ void __launch_bounds__(kWarpsPerBlock * 32) fill_invisible_kernel(const SelectArgs a,
                                                                             int width) {
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t rows = a.total_q;
  const int64_t work = rows * a.heads;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  const bool small = work < (int64_t{1} << 31);  // 32-bit index arithmetic
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + wib; w < work; w += nwarps) {
    int h, i, j, ql = a.query_len;
    int64_t row;
    bool row_ok = true;
    if (small) {
      const uint32_t w32 = static_cast<uint32_t>(w), rows32 = static_cast<uint32_t>(rows);
      h = static_cast<int>(w32 / rows32);
      row = w32 - static_cast<uint32_t>(h) * rows32;
    } else {
      h = static_cast<int>(w / rows);
      row = w - static_cast<int64_t>(h) * rows;
    }
    if (a.cu != nullptr) {
      row_ok = ragged_row(a, row, i, j, ql);
    } else if (small) {
      const uint32_t r32 = static_cast<uint32_t>(row), ql32 = static_cast<uint32_t>(a.query_len);
      i = static_cast<int>(r32 / ql32);
      j = static_cast<int>(r32 - static_cast<uint32_t>(i) * ql32);
    } else {
      i = static_cast<int>(row / a.query_len);
      j = static_cast<int>(row - static_cast<int64_t>(i) * a.query_len);
    }
    const int seq = min(max(__ldg(a.seq_lens + i), 0), a.max_seq_len);
    const int pos = seq - ql + j;
    const int c = row_ok && pos >= 0 ? (pos >> 7) : -1;
    float* srow = const_cast<float*>(a.score) + h * a.s_head + row * a.s_row;
    for (int b = c + 1 + lane; b < width; b += 32) srow[b] = -INFINITY;
  }
}

cudaError_t launch_fill_invisible(const SelectArgs& a, int width, int num_sms, cudaStream_t s) {
  // A warp per row, all rows at once (the rows are independent and short).
  const int64_t work = static_cast<int64_t>(a.total_q) * a.heads;
  int64_t blocks = (work + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int64_t cap = static_cast<int64_t>(num_sms) * 512;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) return cudaSuccess;
  fill_invisible_kernel<<<static_cast<int>(blocks), kWarpsPerBlock * 32, 0, s>>>(a, width);
  return cudaGetLastError();
}

cudaError_t launch_select(const SelectArgs& a, int num_sms, cudaStream_t s) {
  const int64_t work = static_cast<int64_t>(a.total_q) * a.heads;
  int64_t blocks = (work + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  select_kernel<<<static_cast<int>(blocks), kWarpsPerBlock * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mm3idx
