// decode_common.cuh -- the work partition, segment walker, query tile writer
// and merge warp shared by the streaming decode kernels (bf16 pages in
// decode.cu, NVFP4 pages in decode_fp4.cu).
//
// What the kernels compute follows the vLLM MiniMax-M3 "index_topk" page
// (minimax_m3_index_decode: fused decode score + top-k with a final merge of
// per-chunk partial top-k lists, ids 0-indexed with -1 pad) and
// "indexer_cp_exchange" (forced init/local blocks are pinned, packed 64-bit
// candidate keys).  The partition and merge scheme is ours:
//
//   * The work list is every (request, logical block) pair of the batch,
//     flattened request-major.  Each CTA takes one contiguous, equal share, so
//     ragged lengths cost no imbalance.  Shares are computed on the device
//     from seq_lens (no host round trip; CUDA-graph safe).
//   * A request split across CTAs leaves at most TK candidate keys per row per
//     CTA in the workspace; the last of its CTAs to take the request's ticket
//     merges all lists and writes the rows.  Split requests are streamed
//     first, so these merges overlap the rest of the stream.
#pragma once

#include <cstdint>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "ptx.cuh"
#include "warp_select.cuh"

namespace mm3idx {
namespace dec {

constexpr int kLanes = 32;  // rows per list slot

// Partition results and CTA-wide state, in shared memory.
struct Misc {
  long long lo, hi, total, p0, pl;
  int i0, il;
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ int req_len(const DecodeArgs& a, int i) {
  const int s = __ldg(a.seq_lens + i);
  return min(max(s, 0), a.max_seq_len);
}

__device__ __forceinline__ int req_blocks(const DecodeArgs& a, int i) {
  return (req_len(a, i) + kBlock - 1) / kBlock;
}

// A request with blocks occupies kSegCost + blocks positions of the list the
// CTAs share out: each request a CTA serves costs it a query tile and, when
// split, a cross-CTA merge, which the blocks alone do not count.  The extra
// positions come first and hold no work.  Measured on one GB300 over 0-20:
// 6 gave high-batch 171 -> 163 us; the spec-decode batch is within noise
// over 0-12 (57.3-58.6 us, graph replays); larger values lose again.
constexpr int kSegCost = 6;

__device__ __forceinline__ int req_slots(const DecodeArgs& a, int i) {
  const int n = req_blocks(a, i);
  return n > 0 ? n + kSegCost : 0;
}

// Walks this CTA's share [lo, hi) of the flattened (request, block) list and
// yields one segment (request, blocks [b0, b1)) at a time.  The two boundary
// segments come first -- the share's first request (whose earlier blocks
// belong to the previous CTA) and its last request (whose later blocks belong
// to the next CTA) -- so that the requests split across CTAs complete early
// and their cross-CTA merges overlap the streaming of the interior requests,
// which are whole and need no merge.
struct Walker {
  int i0, il;             // first and last request of the share
  long long p0, pl;       // their first flattened positions
  long long lo, hi;
  int stage = 0, i = 0;   // 0: first, 1: last, 2: interior requests
  long long P = 0;
  // Request r's positions start at pr; its blocks at pr + kSegCost, which
  // is what preq reports.
  __device__ bool emit(const DecodeArgs& a, int r, long long pr, int& req, int& b0, int& b1,
                       int& nb, long long& preq) const {
    const int n = req_blocks(a, r);
    const long long pb = pr + kSegCost;
    const long long s = pb > lo ? pb : lo;
    const long long e = (pb + n) < hi ? (pb + n) : hi;
    if (n == 0 || e <= s) return false;
    req = r;
    preq = pb;
    nb = n;
    b0 = static_cast<int>(s - pb);
    b1 = static_cast<int>(e - pb);
    return true;
  }
  __device__ bool next(const DecodeArgs& a, int& req, int& b0, int& b1, int& nb,
                       long long& preq) {
    if (lo >= hi) return false;
    if (stage == 0) {
      stage = 1;
      if (emit(a, i0, p0, req, b0, b1, nb, preq)) return true;
    }
    if (stage == 1) {
      stage = 2;
      i = i0 + 1;
      P = p0 + req_slots(a, i0);
      if (il != i0 && emit(a, il, pl, req, b0, b1, nb, preq)) return true;
    }
    while (i < il) {
      const int r = i;
      const long long pr = P;
      P += req_slots(a, r);
      ++i;
      if (emit(a, r, pr, req, b0, b1, nb, preq)) return true;
    }
    return false;
  }
};

__device__ __forceinline__ Walker make_walker(const Misc* m) {
  return Walker{m->i0, m->il, m->p0, m->pl, m->lo, m->hi};
}

// atomicInc's wrap-around increment with acquire-release ordering at GPU scope.
__device__ __forceinline__ unsigned int atomic_inc_acq_rel_gpu(unsigned int* p, unsigned int wrap) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(wrap) : "memory");
  return old;
}

// The CTA whose share holds flattened position x.
__device__ __forceinline__ int cta_of(long long x, long long total, int grid) {
  return static_cast<int>(((x + 1) * grid - 1) / total);
}

// One warp: total block count, this CTA's share and the first request in it.
__device__ __forceinline__ void partition(const DecodeArgs& a, Misc* m, int lane) {
  // Lengths are read kU per lane at a time so that their loads overlap.
  constexpr int kU = 8;
  long long total = 0;
  for (int b = 0; b < a.num_reqs; b += 32 * kU) {
    int raw[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = b + u * 32 + lane;
      raw[u] = i < a.num_reqs ? __ldg(a.seq_lens + i) : 0;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = b + u * 32 + lane;
      if (i >= a.num_reqs) continue;
      if (blockIdx.x == 0) {
        int bits = 0;
        if (raw[u] > a.max_seq_len) bits |= MM3IDX_DEV_SEQ_TOO_LONG;
        if (raw[u] < a.query_len) bits |= MM3IDX_DEV_SEQ_TOO_SHORT;
        if (bits) atomicOr(a.status, bits);
      }
      const int nbu = (min(max(raw[u], 0), a.max_seq_len) + kBlock - 1) / kBlock;
      total += nbu > 0 ? nbu + kSegCost : 0;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  const long long G = gridDim.x, c = blockIdx.x;
  const long long lo = total * c / G, hi = total * (c + 1) / G;
  // First request with blocks at or past lo (i0) and at or past hi - 1 (il).
  long long P = 0, p0 = total, pl = total;
  int i0 = a.num_reqs, il = a.num_reqs;
  bool need0 = true;
  for (int b = 0; b < a.num_reqs && hi > lo; b += 32) {
    const int i = b + lane;
    const long long nb = i < a.num_reqs ? req_slots(a, i) : 0;
    long long incl = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (need0) {
      const unsigned hit = __ballot_sync(0xffffffffu, i < a.num_reqs && P + incl > lo);
      if (hit) {
        const int k = __ffs(hit) - 1;
        i0 = b + k;
        p0 = P + __shfl_sync(0xffffffffu, incl - nb, k);
        need0 = false;
      }
    }
    const unsigned hitl = __ballot_sync(0xffffffffu, i < a.num_reqs && P + incl > hi - 1);
    if (hitl) {
      const int k = __ffs(hitl) - 1;
      il = b + k;
      pl = P + __shfl_sync(0xffffffffu, incl - nb, k);
      break;
    }
    P += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    m->lo = lo;
    m->hi = hi;
    m->total = total;
    m->i0 = i0;
    m->p0 = p0;
    m->il = il;
    m->pl = pl;
  }
}

// While the producer reads the lengths: pull the block table and the
// queries into L2, one 128-byte line per lane of one warp in every CTA (all
// of both for the named batches), so that the first table and query reads
// after the partition do not go to HBM.
__device__ __forceinline__ void prefetch_table_and_queries(const DecodeArgs& a, int lane) {
  const int64_t line = (static_cast<int64_t>(blockIdx.x) * 32 + lane) * 128;
  const int64_t tbytes = static_cast<int64_t>(a.num_reqs) * a.table_stride * 4;
  const int64_t qbytes = static_cast<int64_t>(a.num_reqs) * a.query_len * a.q_tok * 2;
  if (line < tbytes)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint8_t*>(a.table) + line));
  if (line < qbytes)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint8_t*>(a.q) + line));
}

// Writes request `req`'s query rows (row n = query j, head h with
// n = j*heads + h) into a K-major 128-byte-swizzled tile of MQ rows.  Rows
// past heads*query_len are left as they are: their accumulator lanes or
// columns are never read.
template <int MQ>
__device__ __forceinline__ void load_q_tile(const DecodeArgs& a, int req, uint8_t* dst, int lane) {
  const int R = a.rows_per_req;
  for (int item = lane; item < R * 16; item += 32) {
    const int n = item >> 4, ch = item & 15;
    const int j = n / a.heads, h = n - j * a.heads;
    const uint16_t* src = a.q + (static_cast<int64_t>(req) * a.query_len + j) * a.q_tok +
                          static_cast<int64_t>(h) * a.q_head + ch * 8;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
    const int sub = ch >> 3, c = ch & 7;
    uint8_t* p = dst + sub * (MQ * 128) + (n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4);
    *reinterpret_cast<uint4*>(p) = v;
  }
}

// The merge works in a spread layout: four rows per pass, row g of the pass
// on lanes 8g..8g+7, lane 8g+s holding list positions s, s+8, ... (TK/8 keys,
// descending over positions).  A bitonic step at a stride below 8 pairs a
// lane with lane ^ stride, at 8 or more two registers of one lane, so all 32
// lanes share a merge of two TK-key lists (about 6*TK/8 instructions a lane
// a step).  With one lane per row, four rows left 28 lanes idle and each
// 64-bit merge took one lane 1000-1600 cycles of dependent integer work.
template <int TK>
__device__ __forceinline__ void spread_clean_desc(uint64_t (&v)[TK / 8], int s) {
  constexpr int KL = TK / 8;
#pragma unroll
  for (int d = KL / 2; d > 0; d >>= 1) {       // strides TK/2 .. 8: registers i, i + d
#pragma unroll
    for (int i = 0; i < KL; ++i) {
      if ((i & d) == 0) {
        const uint64_t x = v[i], y = v[i + d];
        v[i] = x > y ? x : y;
        v[i + d] = x > y ? y : x;
      }
    }
  }
#pragma unroll
  for (int st = 4; st > 0; st >>= 1) {         // strides 4, 2, 1: lanes s, s ^ st
    const bool lower = (s & st) == 0;
#pragma unroll
    for (int i = 0; i < KL; ++i) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v[i], st);
      v[i] = (v[i] > o) == lower ? v[i] : o;
    }
  }
}

// a := the best TK keys of a and b (both descending), descending: the
// elementwise max of a and reversed b is a bitonic sequence holding exactly
// those keys, which a half-cleaner cascade orders.
template <int TK>
__device__ __forceinline__ void spread_merge(uint64_t (&a)[TK / 8], const uint64_t (&b)[TK / 8],
                                             int lane) {
  constexpr int KL = TK / 8;
  const int s = lane & 7;
  const int src = (lane & ~7) | (7 - s);     // holds position TK-1-p in register KL-1-i
#pragma unroll
  for (int i = 0; i < KL; ++i) {
    const uint64_t r = __shfl_sync(0xffffffffu, b[KL - 1 - i], src);
    a[i] = a[i] > r ? a[i] : r;
  }
  spread_clean_desc<TK>(a, s);
}

// Ascending bitonic sort of TK ids in the spread layout.
template <int TK>
__device__ __forceinline__ void spread_sort_asc(int (&id)[TK / 8], int s) {
  constexpr int KL = TK / 8;
#pragma unroll
  for (int size = 2; size <= TK; size <<= 1) {
#pragma unroll
    for (int st = size / 2; st > 0; st >>= 1) {
      if (st >= 8) {
        const int d = st / 8;
#pragma unroll
        for (int i = 0; i < KL; ++i) {
          if ((i & d) == 0) {
            const bool up = ((8 * i) & size) == 0;
            const int x = id[i], y = id[i + d];
            id[i] = up ? min(x, y) : max(x, y);
            id[i + d] = up ? max(x, y) : min(x, y);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < KL; ++i) {
          const int p = s + 8 * i;
          const bool up = (p & size) == 0, lower = (p & st) == 0;
          const int o = __shfl_xor_sync(0xffffffffu, id[i], st);
          id[i] = (lower == up) ? min(id[i], o) : max(id[i], o);
        }
      }
    }
  }
}

// Writes one row from its spread list (every lane of the warp takes part;
// write = false for lanes whose row does not exist): forced blocks [0, f_lo),
// the best topk - |forced| picks in ascending id order, the local blocks
// [l_lo, c], then -1.  c < 0 (no visible block): -1 throughout.
template <int TK>
__device__ __forceinline__ void spread_write_row(const uint64_t (&v)[TK / 8], int c,
                                                 int init_blocks, int local_blocks, int topk,
                                                 int32_t* out, int s, bool write) {
  constexpr int KL = TK / 8;
  const Forced F(c, init_blocks, local_blocks);
  const int m = c < 0 ? 0 : topk - F.nf;
  const int nlocal = c < 0 ? 0 : c + 1 - F.l_lo;
  const int f_lo = c < 0 ? 0 : F.f_lo;
  int id[KL];
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < KL; ++i) {
    const bool take = s + 8 * i < m && v[i] != 0ull;
    id[i] = take ? key_block(v[i]) : 0x7fffffff;
    cnt += take;
  }
  cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
  cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
  cnt += __shfl_xor_sync(0xffffffffu, cnt, 4);
  spread_sort_asc<TK>(id, s);
  if (!write) return;
#pragma unroll
  for (int i = 0; i < KL; ++i)
    if (s + 8 * i < cnt) out[f_lo + s + 8 * i] = id[i];
  for (int o = s; o < topk; o += 8) {
    if (o < f_lo) {
      out[o] = o;
    } else if (o >= f_lo + cnt) {
      const int t = o - f_lo - cnt;
      out[o] = t < nlocal ? F.l_lo + t : -1;
    }
  }
}

// Where a request's lists are: its first and last CTA (with total >= grid
// every share is non-empty, so they are first..last; with fewer blocks than
// CTAs every non-empty share is a single block, and block k sits in
// cta_of(preq + k)) and how many CTAs hold part of it.  Computed before the
// lists are handed over (64-bit divisions).
struct MergeGeom {
  int first, nseg;
  bool dense;
};

__device__ __forceinline__ MergeGeom merge_geom(int nb, long long preq, long long total) {
  MergeGeom m;
  m.dense = total >= gridDim.x;
  m.first = cta_of(preq, total, gridDim.x);
  const int last = cta_of(preq + nb - 1, total, gridDim.x);
  m.nseg = m.dense ? last - m.first + 1 : nb;
  return m;
}

// One request of the merge warp: fold the NL handed-over lists of each row
// (H: [NL][TK][32 rows]), then either write the rows (a request held by this
// CTA alone) or publish the lists ([slot][32 rows][TK]) and take the
// request's ticket, the last of its CTAs merging every CTA's lists and
// writing the rows.  Rows are taken four per pass in the spread layout.
//
// dry: the same instructions on the same path with no global access at all
// (no loads, stores or ticket; `split` picks the path).  The merge of a split
// request is often the last work of the last CTA of the batch; a dry run at
// kernel start brings this code into the instruction cache, where its first
// real run would otherwise wait on instruction fetches.
template <int TK, int NL>
__device__ __noinline__ void merge_request(const DecodeArgs& a, int req, long long preq, int seq,
                                           MergeGeom geo, long long total, const uint64_t* H,
                                           int lane, bool dry, bool split) {
  constexpr int KL = TK / 8;
  const int R = a.rows_per_req;
  const int g = lane >> 3, s = lane & 7;
  const int nseg = dry ? (split ? 2 : 1) : geo.nseg;
  const int64_t slot_stride = static_cast<int64_t>(kLanes) * TK;
  auto fold = [&](int r, uint64_t (&v)[KL]) {
#pragma unroll
    for (int i = 0; i < KL; ++i) v[i] = r < R ? H[(s + 8 * i) * kLanes + r] : 0ull;
#pragma unroll
    for (int l = 1; l < NL; ++l) {
      uint64_t o[KL];
#pragma unroll
      for (int i = 0; i < KL; ++i) o[i] = r < R ? H[(l * TK + s + 8 * i) * kLanes + r] : 0ull;
      spread_merge<TK>(v, o, lane);
    }
  };
  auto write_rows = [&](int r, const uint64_t (&v)[KL]) {
    const int rr = r < R ? r : 0;
    const int j = rr / a.heads, h = rr - j * a.heads;
    const int pr = (dry ? a.max_seq_len : seq) - a.query_len + j;
    const int cr = pr >= 0 ? (pr >> 7) : -1;
    int32_t* out = a.ids + h * a.i_head + (static_cast<int64_t>(req) * a.query_len + j) * a.i_row;
    spread_write_row<TK>(v, cr, a.init_blocks, a.local_blocks, a.topk, out, s, r < R && !dry);
  };
  if (nseg == 1) {
    for (int r0 = 0; r0 < R; r0 += 4) {
      uint64_t v[KL];
      fold(r0 + g, v);
      write_rows(r0 + g, v);
    }
    return;
  }
  // Split request: publish this CTA's lists, then take a ticket.  The
  // ticket wraps to zero on the last arrival, ready for the next call.
  for (int r0 = 0; r0 < R; r0 += 4) {
    const int r = r0 + g;
    uint64_t v[KL];
    fold(r, v);
    if (r < R && !dry) {
      uint64_t* dst = a.partials + (static_cast<int64_t>(blockIdx.x) + req) * slot_stride + r * TK;
#pragma unroll
      for (int i = 0; i < KL; ++i) dst[s + 8 * i] = v[i];
    }
  }
  // The warp barrier orders the lanes' list stores before lane 0's release;
  // lane 0's acquire, then the barrier, orders the merging lanes' reads after
  // every other CTA's release.  (Full fences around a plain atomicInc
  // measured 1-2 us slower.)
  __syncwarp();
  unsigned int ticket = nseg - 1;
  if (lane == 0 && !dry)
    ticket = atomic_inc_acq_rel_gpu(a.tickets + req, static_cast<unsigned int>(nseg - 1));
  ticket = __shfl_sync(0xffffffffu, ticket, 0);
  __syncwarp();
  if (ticket != static_cast<unsigned int>(nseg - 1)) return;
  // The last arrival: its own lists again from the hand-over, then every
  // other CTA's, eight sources' loads in flight at a time (a request of the
  // named batches spans at most eight CTAs, so one round trip).
  constexpr int kBatch = 8;
  for (int r0 = 0; r0 < R; r0 += 4) {
    const int r = r0 + g;
    uint64_t v[KL];
    fold(r, v);
    for (int base = 0; base < nseg; base += kBatch) {
      uint64_t o[kBatch][KL];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int js = base + b;
        int cj = -1;
        if (js < nseg) cj = geo.dense ? geo.first + js : cta_of(preq + js, total, gridDim.x);
        const bool load = cj >= 0 && cj != static_cast<int>(blockIdx.x) && r < R && !dry;
        const uint64_t* src = a.partials + (static_cast<int64_t>(load ? cj : 0) + req) * slot_stride +
                              r * TK;
#pragma unroll
        for (int i = 0; i < KL; ++i) o[b][i] = load ? __ldcg(src + s + 8 * i) : 0ull;
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        if (base + b < nseg) spread_merge<TK>(v, o[b], lane);
    }
    write_rows(r, v);
  }
}

// Requests with no blocks at all appear in no share: their rows are spread
// over the CTAs, one warp each (-inf scores or -1 ids).
__device__ __forceinline__ void fill_empty_requests(const DecodeArgs& a, int lane) {
  const int R = a.rows_per_req;
  for (int i = blockIdx.x; i < a.num_reqs; i += gridDim.x) {
    if (req_blocks(a, i) != 0) continue;
    if (a.mode != kModeSelect) {
      const int w = a.fill_width;
      for (int idx = lane; idx < R * w; idx += 32) {
        const int rr = idx / w, bb = idx - rr * w;
        const int j = rr / a.heads, h = rr - j * a.heads;
        a.score[h * a.s_head + (static_cast<int64_t>(i) * a.query_len + j) * a.s_row + bb] =
            -INFINITY;
      }
    } else {
      for (int idx = lane; idx < R * a.topk; idx += 32) {
        const int rr = idx / a.topk, k = idx - rr * a.topk;
        const int j = rr / a.heads, h = rr - j * a.heads;
        a.ids[h * a.i_head + (static_cast<int64_t>(i) * a.query_len + j) * a.i_row + k] = -1;
      }
    }
  }
}

// The merge warp: first the requests with no blocks; then merge_request for
// every request of this CTA's share, in the walker's order, as the scoring
// warps hand their lists over (hand-over slot seg & 1).  The walker steps to
// the next segment (and reads its length) before the wait for the current
// one's lists, so that after the share's last hand-over no global read is
// left on the way to the CTA's exit.
template <int TK, int NL>
__device__ void merge_warp(const DecodeArgs& a, Walker walker, long long total, uint64_t* sHand,
                           uint64_t* h_full, uint64_t* h_empty, volatile int* abort_flag,
                           int lane) {
  fill_empty_requests(a, lane);
  if (a.mode != kModeSelect) return;
  // Dry runs of both paths while the first lists are still being scored.
  const MergeGeom none{0, 1, true};
  merge_request<TK, NL>(a, 0, 0, 1, none, 1, sHand, lane, true, false);
  merge_request<TK, NL>(a, 0, 0, 1, none, 1, sHand, lane, true, true);
  int req, b0, b1, nb;
  long long preq;
  bool have = walker.next(a, req, b0, b1, nb, preq);
  int seq = have ? req_len(a, req) : 0;
  MergeGeom geo = have ? merge_geom(nb, preq, total) : none;
  for (int seg = 0; have; ++seg) {
    int nreq, nb0, nb1, nnb;
    long long npreq;
    const bool nhave = walker.next(a, nreq, nb0, nb1, nnb, npreq);
    const int nseq = nhave ? req_len(a, nreq) : 0;
    const MergeGeom ngeo = nhave ? merge_geom(nnb, npreq, total) : none;
    const int hs = seg & 1;
    if (!warp_wait(&h_full[hs], (seg >> 1) & 1, abort_flag)) break;
    merge_request<TK, NL>(a, req, preq, seq, geo, total, sHand + hs * NL * TK * kLanes, lane,
                          false, false);
    __syncwarp();
    if (lane == 0) mbar_arrive(&h_empty[hs]);
    req = nreq;
    preq = npreq;
    seq = nseq;
    geo = ngeo;
    have = nhave;
  }
}

// Score mode, once a request's last block has been scored: -inf for its
// blocks nb .. fill_width-1 in all its rows (one warp).
__device__ __forceinline__ void fill_past_blocks(const DecodeArgs& a, int req, int nb, int lane) {
  const int R = a.rows_per_req;
  const int w = a.fill_width - nb;
  for (int idx = lane; idx < R * w; idx += 32) {
    const int rr = idx / w, bb = nb + (idx - rr * w);
    const int j = rr / a.heads, h = rr - j * a.heads;
    a.score[h * a.s_head + (static_cast<int64_t>(req) * a.query_len + j) * a.s_row + bb] =
        -INFINITY;
  }
}

}  // namespace dec
}  // namespace mm3idx
