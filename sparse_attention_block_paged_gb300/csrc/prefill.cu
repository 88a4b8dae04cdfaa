// prefill.cu -- tensor-core causal block scorer for long query runs.
//
// Computes score[h, row, b] = sm_scale * max over the visible tokens of block
// b of q[row, h] . k[token] (vLLM MiniMax-M3 "index_topk" page,
// minimax_m3_index_score: per-token index scores for each visible sparse
// block, i.e. the largest token score inside the block, causal through the
// request's prefix).  The design is ours:
//
//   * A unit is (request, head, 128-row query tile, pair of key blocks).
//     A request's query rows are query_len per request, or for a ragged
//     batch the rows given by its row offsets (minimax_m3_index_score:
//     cu_seqlens_q).  The CTAs count the units exactly on the device (a
//     closed form per request) and each takes one contiguous, equal share,
//     so the causal triangle is spread evenly over the SMs.
//   * warp 0   : TMA producer.  The 128 x 128 bf16 query tile (two 64-column
//                boxes, 128-byte swizzle, from a 3-D map over
//                [tokens, heads, 128]) once per tile, and the two key pages of
//                each unit (from a 2-D map over [pages*128, 128]) into a
//                3-stage ring of 64 KB stages laid out as one 256-row operand.
//   * warp 1   : one thread issues tcgen05.mma, A = the query tile
//                (M = 128), B = both pages (N = 256 key tokens), K = 128, as
//                8 instructions into one of two 256-column fp32 TMEM
//                accumulators.  The tensor pipe queues only a few MMAs, so
//                the issuing thread's per-unit work (waits, commits, loop)
//                must hide behind the queued ones: N = 256 doubles the work
//                each instruction carries, and the producer hands the issuer
//                one word per stage (unit shape, new tile, end) so that the
//                issuer keeps no unit bookkeeping.
//   * warps 2-9: epilogue, two teams of four warps (one warp per TMEM lane
//                quadrant).  Team t drains block t of every unit: loads its
//                row's 128 columns with tcgen05.ld in two 64-column halves,
//                taking the causal row max of each with 3-input max, frees
//                the accumulator and stores one fp32 score per (row, block).
//                Ten warps put three on one SM sub-partition, which caps a
//                thread at 168 registers; holding all 128 columns at once
//                spilled the loop state to local memory.
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "ptx.cuh"
#include "warp_select.cuh"

namespace mm3idx {

namespace {

constexpr int kStages = 3;
constexpr int kPage = 32768;                  // 128 x 128 bf16
constexpr int kHalf = 16384;                  // 128 rows x 64 columns
constexpr int kStageBytes = 2 * kPage;        // two pages
constexpr uint32_t kTmemCols = 512;           // two 256-column accumulators
constexpr int kThreads = 320;
constexpr int oQ = 0;
constexpr int oK = oQ + kPage;
constexpr int oBar = oK + kStages * kStageBytes;
constexpr int kBars = 2 * kStages + 4 + 2 + 1;
constexpr int oInfo = oBar + kBars * 8;        // one word per stage, producer -> MMA
constexpr int oMisc = oInfo + kStages * 4;
constexpr int kSmem = oMisc + 64 + 1024;
static_assert(kSmem <= 227 * 1024, "shared memory budget");

struct Misc {
  uint32_t tmem;
  int abort;
};

// What the producer tells the MMA issuer about the unit in a stage, so that
// the issuer does no unit bookkeeping of its own.
constexpr uint32_t kInfoValid = 1u;    // 0: no more units
constexpr uint32_t kInfoTwo = 2u;      // both key blocks visible (N = 256), else N = 128
constexpr uint32_t kInfoNewTile = 4u;  // first unit of a new query tile

// Visible block count of query tile qt under a given prefix length
// (positions prefix + 128*qt .. prefix + min(128*qt + 127, query_len - 1)).
__device__ __forceinline__ int tile_blocks(int prefix, int qt, int query_len) {
  const int last = prefix + min(qt * 128 + 127, query_len - 1);
  return last < 0 ? 0 : (last >> 7) + 1;
}

// Where a request's query rows are: a uniform batch has query_len rows per
// request; a ragged one takes them from the row offsets cu (index_topk,
// minimax_m3_index_score: cu_seqlens_q).  prefix = seq_len - rows, so row j
// sits at position prefix + j.
struct ReqGeom {
  int qbeg = 0, ql = 0, prefix = 0, qtiles = 0;
};

__device__ __forceinline__ ReqGeom req_geom(const PrefillArgs& a, int i) {
  ReqGeom g;
  if (a.cu != nullptr) {
    const int b = __ldg(a.cu + i), e = __ldg(a.cu + i + 1);
    g.qbeg = min(max(b, 0), a.total_q);
    g.ql = min(max(e, g.qbeg), a.total_q) - g.qbeg;  // malformed offsets are flagged by the selector
  } else {
    g.qbeg = i * a.query_len;
    g.ql = a.query_len;
  }
  g.prefix = min(max(__ldg(a.seq_lens + i), 0), a.max_seq_len) - g.ql;
  g.qtiles = (g.ql + 127) >> 7;
  return g;
}

// Units of one query tile: its visible blocks in pairs; at least one, so
// that every tile is visited (in select mode, its record for the merge).
__device__ __forceinline__ int tile_units(const ReqGeom& g, int qt) {
  return max(1, (tile_blocks(g.prefix, qt, g.ql) + 1) >> 1);
}

// sum of ceil(k / 2) for k = 1..n
__device__ __forceinline__ int64_t half_ceil_sum(int64_t n) { return ((n + 1) >> 1) * ((n + 2) >> 1); }

// Units of one (request, head) in its tiles 0..qt-1.  A full tile t holds
// A + t + 1 visible blocks (A = (prefix + 127) / 128), so the full tiles sum
// in closed form; a request shorter than its rows (malformed) is counted
// tile by tile.
__device__ __forceinline__ int64_t units_before(const ReqGeom& g, int qt) {
  if (g.prefix < 0) {
    int64_t n = 0;
    for (int t = 0; t < qt; ++t) n += tile_units(g, t);
    return n;
  }
  const int full = g.ql >> 7;
  const int64_t A = (g.prefix + 127) >> 7;
  const int f = min(qt, full);
  int64_t n = half_ceil_sum(A + f) - half_ceil_sum(A);
  if (qt > full) n += tile_units(g, full);
  return n;
}

// In score mode a query tile occupies two positions ahead of its units in
// the list the CTAs share out: starting a tile costs a CTA a query-tile load
// that the MMAs wait for, which its unit count does not show, and the first
// CTAs' shares span dozens of small tiles (a clock64 trace of the 32K causal
// prefill: the CTA with 20 tiles waited 253 cycles a unit for query tiles,
// the median CTA 17, and ended 12 us after the median).  Score call on the
// 32K prefill: 115.4 us without the cost, 104.7 / 102.6 / 103.3 / 104.9 us
// with 1 / 2 / 3 / 4 positions.  The selecting kernel's epilogue is its
// bottleneck and hides most of the query loads: with 16-key lists a tile
// takes one position in uniform batches (32K causal prefill step 121.9 ->
// 119.7 us, NVFP4 prefill 127.5 -> 126.0 us, three runs each on one box;
// two positions measured no better) and none in ragged ones (the chunked
// batch measured 94.3 us without, 96.1 us with one).  With
// 32-key lists the end of a tile costs the epilogue the partial batch's
// merge and the 32-key list stores, about two units' work (a clock64 trace
// of the 32K prefill at topk 32: CTAs ended at a median of 110.8 us, the
// last at 132.4 us); two positions a tile: step 153.3 -> 137.9 us (1 / 2 /
// 3 / 4 positions: 139.3 / 137.9 / 138.7 / 139.7 us).
__device__ __forceinline__ int64_t pos_before(const ReqGeom& g, int qt, int cost) {
  return units_before(g, qt) + static_cast<int64_t>(cost) * qt;
}

// Iterates this CTA's share of the unit list (request, head, query tile,
// pair of key blocks).  The list holds exactly each request's units, so the
// shares are computed on the device: total() and init() are warp-collective.
// Shares are ranges of positions (units plus the tiles' costs); a share's
// units are those whose positions it holds.
// The state is kept small: the epilogue's loop also holds a 128-column
// accumulator row in registers.
struct UnitIter {
  int left = 0;  // units still to visit, this one included
  int req = 0, head = 0, qt = 0, p = 0, np = 0, nvis = 0;
  int tile = 0;     // index of the (request, head, tile) in the batch
  int64_t u = 0;    // index of the unit in the batch's list
  int64_t ulo = 0, uhi = 0;  // the share's units [ulo, uhi)
  int cost = 0;              // positions a query tile takes ahead of its units
  ReqGeom g;

  // Total positions of the batch (all lanes get it); *tiles gets its tiles.
  __device__ static int64_t total(const PrefillArgs& a, int cost, int* tiles = nullptr) {
    const int lane = threadIdx.x & 31;
    int64_t sum = 0;
    int nt = 0;
    for (int base = 0; base < a.num_reqs; base += 32) {
      const int i = base + lane;
      if (i < a.num_reqs) {
        const ReqGeom gi = req_geom(a, i);
        sum += pos_before(gi, gi.qtiles, cost);
        nt += gi.qtiles;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
      nt += __shfl_xor_sync(0xffffffffu, nt, o);
    }
    if (tiles) *tiles = nt * a.heads;
    return sum * a.heads;
  }

  __device__ __forceinline__ void load_tile() {
    nvis = tile_blocks(g.prefix, qt, g.ql);
    np = max(1, (nvis + 1) >> 1);
  }

  // The index of the first unit at position x or later (the batch's unit
  // count when there is none), with its request, head, tile and place.
  __device__ int64_t unit_at(const PrefillArgs& a, int64_t x, int& r, int& hd, int& t, int& pp,
                             int& tl) {
    const int lane = threadIdx.x & 31;
    int64_t pacc = 0, uacc = 0;  // positions and units of the requests before `base`
    int tacc = 0;                // tiles of the requests before `base`
    r = a.num_reqs;
    for (int base = 0; base < a.num_reqs; base += 32) {
      const int i = base + lane;
      int64_t pm = 0, um = 0;
      int tm = 0;
      if (i < a.num_reqs) {
        const ReqGeom gi = req_geom(a, i);
        pm = pos_before(gi, gi.qtiles, cost) * a.heads;
        um = units_before(gi, gi.qtiles) * a.heads;
        tm = gi.qtiles * a.heads;
      }
      int64_t pin = pm, uin = um;
      int tin = tm;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t py = __shfl_up_sync(0xffffffffu, pin, o);
        const int64_t uy = __shfl_up_sync(0xffffffffu, uin, o);
        const int ty = __shfl_up_sync(0xffffffffu, tin, o);
        if (lane >= o) {
          pin += py;
          uin += uy;
          tin += ty;
        }
      }
      const unsigned hit = __ballot_sync(0xffffffffu, pacc + pin > x);
      if (hit != 0u) {
        const int l = __ffs(hit) - 1;
        r = base + l;
        pacc += __shfl_sync(0xffffffffu, pin - pm, l);
        uacc += __shfl_sync(0xffffffffu, uin - um, l);
        tacc += __shfl_sync(0xffffffffu, tin - tm, l);
        break;
      }
      pacc += __shfl_sync(0xffffffffu, pin, 31);
      uacc += __shfl_sync(0xffffffffu, uin, 31);
      tacc += __shfl_sync(0xffffffffu, tin, 31);
    }
    if (r >= a.num_reqs) return uacc;
    const ReqGeom gr = req_geom(a, r);
    const int64_t pph = pos_before(gr, gr.qtiles, cost), uph = units_before(gr, gr.qtiles);
    int64_t off = x - pacc;
    hd = static_cast<int>(off / pph);
    off -= hd * pph;
    // the tile holding position `off`: the last qt with pos_before(qt) <= off
    int t_lo = 0, t_hi = gr.qtiles - 1;
    while (t_lo < t_hi) {
      const int mid = (t_lo + t_hi + 1) >> 1;
      if (pos_before(gr, mid, cost) <= off) t_lo = mid;
      else t_hi = mid - 1;
    }
    t = t_lo;
    pp = static_cast<int>(max(off - pos_before(gr, t, cost) - cost, int64_t{0}));  // past the tile's cost
    tl = tacc + hd * gr.qtiles + t;
    return uacc + hd * uph + units_before(gr, t) + pp;
  }

  // Position at the share [lo, hi) of the list (in positions, `cost` per
  // tile): its first unit, and the count of its units.
  __device__ void init(const PrefillArgs& a, int64_t lo, int64_t hi, int tile_cost) {
    cost = tile_cost;
    int r1, h1, t1, p1, tl1;
    const int64_t u_lo = unit_at(a, lo, req, head, qt, p, tile);
    const int64_t u_hi = unit_at(a, hi, r1, h1, t1, p1, tl1);
    left = static_cast<int>(u_hi - u_lo);
    u = ulo = u_lo;
    uhi = u_hi;
    if (left <= 0) return;
    g = req_geom(a, req);
    load_tile();
  }

  __device__ __forceinline__ bool valid() const { return left > 0; }
  // Next unit; true when it starts a new query tile.
  __device__ __forceinline__ bool advance(const PrefillArgs& a) {
    --left;
    ++u;
    if (++p < np) return false;
    p = 0;
    ++tile;
    if (++qt == g.qtiles) {
      qt = 0;
      if (++head == a.heads) {
        head = 0;
        // the next request with query rows (one without any has no units)
        do {
          ++req;
          if (req >= a.num_reqs) return true;  // only past the end of the list
          g = req_geom(a, req);
        } while (g.qtiles == 0);
      }
    }
    load_tile();
    return true;
  }
};

// Whether CTA c's share [total*c/G, total*(c+1)/G) of the positions is not
// empty.
__device__ __forceinline__ bool has_units(int c, int64_t total, int64_t G) {
  return total * (c + 1) / G > total * c / G;
}

// The CTA whose share [total*c/G, total*(c+1)/G) holds position x.
__device__ __forceinline__ int cta_of(int64_t x, int64_t total, int64_t G) {
  return static_cast<int>(((x + 1) * G - 1) / total);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// kSelect: instead of the scores, the top-k ids, kept in lists of TK keys
// (TK = 16 for topk <= 16, else 32), see the epilogue.
// NL: the list slots a row can need (select mode, 16-key lists): every row
// with a candidate has init + local forced blocks, so it takes
// topk - init - local picks; the slots past them never reach the output.
template <bool kSelect, int TK, int NL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + oQ;
  uint8_t* sK = sm + oK;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + oBar);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* q_full = acc_empty + 2;
  uint64_t* q_empty = q_full + 1;
  uint64_t* done_bar = q_empty + 1;
  volatile uint32_t* sInfo = reinterpret_cast<volatile uint32_t*>(sm + oInfo);
  Misc* misc = reinterpret_cast<Misc*>(sm + oMisc);
  volatile int* abort_flag = &misc->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 8);   // both epilogue teams
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(done_bar, 1);
    misc->abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
  }
  if (warp == 1) {
    tmem_alloc(&misc->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc->tmem;

  // No early launch of dependents (griddepcontrol.launch_dependents): the
  // selection's merge CTAs would sit on the SMs waiting, beside this grid,
  // which measured 20 % slower; they launch when this grid completes.

  // This CTA's equal share of the batch's positions (every warp computes it).
  const int tile_cost = kSelect ? (TK == 32 ? 2 : (a.cu == nullptr ? 1 : 0)) : 2;
  UnitIter U;
  int64_t total = 0, share_lo = 0, share_hi = 0;
  const int64_t G = gridDim.x;
  if (warp != 1) {
    int tiles = 0;
    total = UnitIter::total(a, tile_cost, &tiles);
    // the selection's merge reads the batch's tile count from the first record
    if (kSelect && blockIdx.x == 0 && warp == 0 && lane == 0) a.tile_rec[0] = tiles;
    share_lo = total * blockIdx.x / G;
    share_hi = total * (blockIdx.x + 1) / G;
    U.init(a, share_lo, share_hi, tile_cost);
  }

  if (a.cu != nullptr && blockIdx.x == 0 && warp == 0) {
    // ragged batches: the offsets must run from 0 to total_q without decreasing
    bool bad = lane == 0 && (__ldg(a.cu) != 0 || __ldg(a.cu + a.num_reqs) != a.total_q);
    for (int i = lane; i < a.num_reqs; i += 32) bad |= __ldg(a.cu + i + 1) < __ldg(a.cu + i);
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, MM3IDX_DEV_BAD_ROWS);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the units; lane 0 issues the copies.  Page ids are
    // read 32 at a time (one per lane) and broadcast with shuffles.
    const uint64_t pol_k = policy_evict_last();   // pages are re-read by later tiles
    const uint64_t pol_q = policy_evict_first();
    const int nblk = (a.max_seq_len + kBlock - 1) / kBlock;  // table entries that exist
    int pg_req = -1, pg_base = 0, pg = -1;
    uint32_t tq = 0, it = 0, st = 0, ph = 0;
    bool ok = true;
    bool new_tile = true;  // the share's first unit starts a tile for this CTA
    for (; ok && U.valid(); new_tile |= U.advance(a)) {
      const int b0 = 2 * U.p;
      if (b0 >= U.nvis) continue;  // no visible token (the tile's rows are loaded with its next unit)
      const bool two = b0 + 1 < U.nvis;
      if (U.req != pg_req || b0 < pg_base || b0 + 1 >= pg_base + 32) {
        pg_req = U.req;
        pg_base = b0;
        const int mine = pg_base + lane;
        pg = mine < nblk ? __ldg(a.table + static_cast<int64_t>(U.req) * a.table_stride + mine)
                         : -1;
      }
      const int pa = __shfl_sync(0xffffffffu, pg, b0 - pg_base);
      const int pb = __shfl_sync(0xffffffffu, pg, b0 + 1 - pg_base);
      if (it >= static_cast<uint32_t>(kStages)) ok = warp_wait(&empty[st], ph ^ 1u, abort_flag);
      if (!ok) break;
      if (lane == 0) {
        sInfo[st] = kInfoValid | (two ? kInfoTwo : 0u) | (new_tile ? kInfoNewTile : 0u);
        uint8_t* dst = sK + st * kStageBytes;
        // A page id out of range is not loaded (the epilogue gives its block
        // -inf); the other page of the pair still is.
        const bool good_a = pa >= 0 && pa < a.num_pages;
        const bool good_b = two && pb >= 0 && pb < a.num_pages;
        if (!good_a || (two && !good_b)) atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
        const uint32_t bytes = (good_a ? kPage : 0) + (good_b ? kPage : 0);
        if (bytes) {
          // Stage layout: [A cols 0-63][B cols 0-63][A cols 64-127][B cols 64-127],
          // i.e. 256 key rows per 64-column half, as the N = 256 operand.
          mbar_arrive_expect_tx(&full[st], bytes);
          if (good_a) {
            tma_load_2d(dst, &kmap, &full[st], 0, pa * 128, pol_k);
            tma_load_2d(dst + 2 * kHalf, &kmap, &full[st], 64, pa * 128, pol_k);
          }
          if (good_b) {
            tma_load_2d(dst + kHalf, &kmap, &full[st], 0, pb * 128, pol_k);
            tma_load_2d(dst + 3 * kHalf, &kmap, &full[st], 64, pb * 128, pol_k);
          }
        } else {
          mbar_arrive(&full[st]);
        }
      }
      ++it;
      if (++st == kStages) {
        st = 0;
        ph ^= 1u;
      }
      if (new_tile) {
        // The tile's query rows, once the MMAs of the previous tile are done
        // (issued after this unit's keys, which do not depend on them).
        new_tile = false;
        if (tq > 0) ok = warp_wait(q_empty, (tq - 1) & 1u, abort_flag);
        if (!ok) break;
        if (lane == 0) {
          const int tok0 = U.g.qbeg + U.qt * 128;
          mbar_arrive_expect_tx(q_full, kPage);
          tma_load_3d(sQ, &qmap, q_full, 0, U.head, tok0, pol_q);
          tma_load_3d(sQ + kHalf, &qmap, q_full, 64, U.head, tok0, pol_q);
        }
        ++tq;
      }
    }
    // Drain: let every copy started above land before the CTA may exit.
    if (lane == 0) {
      int dummy = 0;
      const uint32_t pend = it < static_cast<uint32_t>(kStages) ? it : kStages;
      for (uint32_t k = 0; k < pend; ++k) {
        const uint32_t idx = it - 1 - k;
        mbar_wait(&full[idx % kStages], (idx / kStages) & 1, &dummy);
      }
      if (tq > 0) mbar_wait(q_full, (tq - 1) & 1u, &dummy);
    }
    __syncwarp();
    // End marker for the MMA issuer, in the next stage once it is free.
    if (ok && it >= static_cast<uint32_t>(kStages)) ok = warp_wait(&empty[st], ph ^ 1u, abort_flag);
    if (ok && lane == 0) {
      sInfo[st] = 0u;
      mbar_arrive(&full[st]);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc2 = idesc_bf16_f32(128, 256);
      constexpr uint32_t idesc1 = idesc_bf16_f32(128, 128);
      const uint64_t qdesc = sdesc_kmajor_sw128(smem_u32(sQ));
      const uint64_t kdesc0 = sdesc_kmajor_sw128(smem_u32(sK));
      uint32_t tq = 0, it = 0, st = 0, ph = 0, acc = 0;
      bool ok = true;
      for (;;) {
        ok = mbar_wait(&full[st], ph, abort_flag);
        if (!ok) break;
        const uint32_t info = sInfo[st];
        if (!(info & kInfoValid)) break;
        if (info & kInfoNewTile) {
          if (tq > 0) mma_commit(q_empty);   // the previous tile's query rows
          ok = mbar_wait(q_full, tq & 1u, abort_flag);
          if (!ok) break;
          ++tq;
        }
        if (it >= 2) ok = mbar_wait(&acc_empty[acc], ((it >> 1) - 1) & 1u, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * 256;
        const uint64_t kdesc = kdesc0 + st * (kStageBytes >> 4);
        const uint32_t idesc = (info & kInfoTwo) ? idesc2 : idesc1;
        // K slice k: 32 bytes into a 128-byte row inside a 64-column half.
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16(d, qdesc + (k >> 2) * (kHalf >> 4) + (k & 3) * 2,
                   kdesc + (k >> 2) * ((2 * kHalf) >> 4) + (k & 3) * 2, idesc, k > 0 ? 1u : 0u);
        mma_commit(&empty[st]);
        mma_commit(&acc_full[acc]);
        ++it;
        acc ^= 1u;
        if (++st == kStages) {
          st = 0;
          ph ^= 1u;
        }
      }
      mma_commit(done_bar);
      int dummy = 0;
      mbar_wait(done_bar, 0, &dummy);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- epilogue
    const int team = (warp - 2) >> 2;  // which block of the pair
    const int quad = warp & 3;         // a warp may only read lanes 32*(warp%4)..+31
    const int r = quad * 32 + lane;    // query row within the tile
    uint32_t it = 0, acc = 0;
    bool ok = true;
    bool row_ok = false;
    int pos = 0;
    float* srow = nullptr;   // score mode: the row's scores
    int f_lo = 0, l_lo = 0;  // select mode: the row's forced blocks [0, f_lo), [l_lo, c]
    RegList<TK> list;  // select mode: best non-forced keys of the tile so far
    // 32-key lists take offers eight at a time (newest first, 0 = none): a
    // warp's 32 rows rarely all decline an offer, so one insertion per offer
    // moves all 32 slots nearly every unit.  The accumulator is then read 32
    // columns at a time to leave registers for the batch.
    constexpr bool kBatch = kSelect && TK == 32;
    constexpr bool kNarrow = kSelect && TK == 32;
    uint64_t batch[8];
    int nbatch = 0;  // offers in the batch (the same for the warp)
    bool new_tile = true;
    for (; ok && U.valid(); new_tile = U.advance(a)) {
      if (new_tile) {
        const int qrow = U.qt * 128 + r;  // query index inside the request
        row_ok = qrow < U.g.ql;
        pos = U.g.prefix + qrow;
        const int64_t row = U.g.qbeg + qrow;
        if constexpr (kSelect) {
          const Forced F(pos >= 0 ? pos >> 7 : -1, a.init_blocks, a.local_blocks);
          f_lo = F.f_lo;
          l_lo = F.l_lo;
          list.clear();
          if constexpr (kBatch) {
#pragma unroll
            for (int j = 0; j < 8; ++j) batch[j] = 0ull;
            nbatch = 0;
          }
        } else {
          srow = a.score + U.head * a.s_head + row * a.s_row;
        }
      }
      const int b0 = 2 * U.p;
      if (b0 < U.nvis) {
        const int b = b0 + team;
        const bool mine = b < U.nvis;
        // The block's page id, read before the wait so that its latency is
        // hidden: an id out of range means no visible tokens (-inf).
        const int page = mine ? __ldg(a.table + static_cast<int64_t>(U.req) * a.table_stride + b) : 0;
        bool got = true;
        if (lane == 0) got = mbar_wait(&acc_full[acc], (it >> 1) & 1u, abort_flag);
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // The row's 128 columns in two halves (64 registers live), then the
        // accumulator goes back.
        const int lim = row_ok ? pos - b * 128 : -1;  // columns 0..lim are visible
        float m0 = -INFINITY, m1 = -INFINITY;
        if (mine) {
          const uint32_t taddr =
              tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * 256 + team * 128;
          if constexpr (kNarrow) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              uint32_t v0[32];
              tmem_ld32(taddr + 32 * h, v0);
              tmem_ld_wait32(v0);
              if (lim >= 127) {
#pragma unroll
                for (int k = 0; k < 32; k += 4) {
                  m0 = fmax3(m0, __uint_as_float(v0[k]), __uint_as_float(v0[k + 1]));
                  m1 = fmax3(m1, __uint_as_float(v0[k + 2]), __uint_as_float(v0[k + 3]));
                }
              } else if (lim >= 0) {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                  if (32 * h + k <= lim) m0 = fmaxf(m0, __uint_as_float(v0[k]));
              }
            }
          } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t v0[32], v1[32];
            tmem_ld32(taddr + 64 * h, v0);
            tmem_ld32(taddr + 64 * h + 32, v1);
            tmem_ld_wait32x2(v0, v1);
            if (lim >= 127) {
#pragma unroll
              for (int k = 0; k < 32; k += 4) {
                m0 = fmax3(m0, __uint_as_float(v0[k]), __uint_as_float(v0[k + 1]));
                m1 = fmax3(m1, __uint_as_float(v0[k + 2]), __uint_as_float(v0[k + 3]));
                m0 = fmax3(m0, __uint_as_float(v1[k]), __uint_as_float(v1[k + 1]));
                m1 = fmax3(m1, __uint_as_float(v1[k + 2]), __uint_as_float(v1[k + 3]));
              }
            } else if (lim >= 0) {   // rows past the request's end (lim < 0) are never read
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                if (64 * h + k <= lim) m0 = fmaxf(m0, __uint_as_float(v0[k]));
                if (64 * h + 32 + k <= lim) m1 = fmaxf(m1, __uint_as_float(v1[k]));
              }
            }
          }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        if constexpr (kBatch) {
          uint64_t key = 0ull;
          if (mine && row_ok && b >= f_lo && b < l_lo) {
            const float score =
                (page >= 0 && page < a.num_pages) ? fmaxf(m0, m1) * a.sm_scale : -INFINITY;
            key = make_key(score, b);
          }
#pragma unroll
          for (int j = 7; j > 0; --j) batch[j] = batch[j - 1];
          batch[0] = key;
          if (++nbatch == 8) {
            list.merge8(batch);
#pragma unroll
            for (int j = 0; j < 8; ++j) batch[j] = 0ull;
            nbatch = 0;
          }
        } else if (mine && row_ok) {
          const float score =
              (page >= 0 && page < a.num_pages) ? fmaxf(m0, m1) * a.sm_scale : -INFINITY;
          if constexpr (kSelect) {
            if (b >= f_lo && b < l_lo) list.template offer_ascending<NL>(make_key(score, b));
          } else {
            srow[b] = score;
          }
        }
        ++it;
        acc ^= 1u;
      }
      if constexpr (kSelect) {
        // The last unit of the tile in this CTA's share: the warp's 32 lists
        // (of this team's blocks) go to the tile's slot in the workspace,
        // unless every row of the tile keeps all its blocks.  The CTA that
        // holds the tile's first unit also leaves the tile's record.  A
        // dependent kernel merges the lists after this one.
        if (U.p == U.np - 1 || U.left == 1) {
          if constexpr (kBatch) {
            if (nbatch > 0) {
              list.merge8(batch);
#pragma unroll
              for (int j = 0; j < 8; ++j) batch[j] = 0ull;
              nbatch = 0;
            }
          }
          if (U.nvis > a.topk) {
            // Key-major slot [TK][128 rows]: a warp's 32 rows store 256
            // contiguous bytes per key.
            const int64_t slot = 2 * (static_cast<int64_t>(blockIdx.x) + U.tile) + team;
            uint64_t* dst = a.partials + slot * 128 * TK + r;
#pragma unroll
            for (int k = 0; k < TK; ++k) dst[k * 128] = list.v[k];
          }
          const int64_t tfirst = U.u - U.p, tlast = tfirst + U.np - 1;
          if (warp == 2 && lane == 0 && tfirst >= U.ulo) {
            int32_t* rec = a.tile_rec + (static_cast<int64_t>(U.tile) + 1) * kTileRecInts;
            // the tile's last unit sits at position tlast + cost * (tile + 1)
            rec[1] = tlast < U.uhi ? static_cast<int>(blockIdx.x)
                                   : cta_of(tlast + static_cast<int64_t>(U.cost) * (U.tile + 1),
                                            total, G);
            rec[2] = U.head;
            rec[3] = U.g.qbeg;
            rec[4] = U.g.ql;
            rec[5] = U.g.prefix;
            rec[6] = U.qt;
            rec[7] = U.nvis;
            rec[8] = static_cast<int32_t>(total & 0xffffffff);
            rec[9] = static_cast<int32_t>(total >> 32);
            rec[0] = static_cast<int>(blockIdx.x);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && misc->abort) atomicOr(a.status, MM3IDX_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

// The fused prefill's selection, finished: warp per (query tile, lane
// quadrant).  A tile whose last row sees at most topk blocks keeps them all
// (rows 0..c); otherwise the 32 rows' lists of every CTA that held part of
// the tile (one list per team) are merged and the rows written.  Launched
// as a programmatic dependent of the prefill kernel, whose completion it
// waits for on the GPU.
constexpr int kMergeWarps = 8;

template <int TK>
__global__ void __launch_bounds__(kMergeWarps * 32, 1) prefill_merge_kernel(const PrefillMergeArgs a) {
  // Each warp builds its 32 rows in shared memory (lane = row) and writes
  // them out row by row, so the stores are contiguous.  Rows are TK + 1
  // words apart, so that the lanes' stores fall in distinct banks.
  __shared__ int32_t s_rows[kMergeWarps][32][TK + 1];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kMergeWarps + wib;
  const int64_t tile = item >> 2;
  const int q = static_cast<int>(item & 3);
  if (tile >= min(a.tiles, static_cast<int64_t>(a.tile_rec[0]))) return;  // the batch's tiles
  const int32_t* rec = a.tile_rec + (tile + 1) * kTileRecInts;
  const int c0 = rec[0], c1 = rec[1], head = rec[2], qbeg = rec[3], ql = rec[4], prefix = rec[5];
  const int qt = rec[6], nvis = rec[7];
  const int64_t total = static_cast<int64_t>(static_cast<uint32_t>(rec[8])) |
                        (static_cast<int64_t>(rec[9]) << 32);
  const int row0 = qt * 128 + q * 32;   // the warp's first row in the request
  // Every field is checked against this call's sizes: a prefill that gave up
  // (MM3IDX_DEV_TIMEOUT) may leave a record of an earlier call, which must
  // not send a read or write out of bounds.
  if (c0 < 0 || c1 < c0 || c1 >= a.grid || head < 0 || head >= a.heads || qbeg < 0 ||
      row0 >= ql || total <= 0)
    return;
  const int nrows = min(min(32, ql - row0), a.total_q - (qbeg + row0));
  if (nrows <= 0) return;
  const int r = q * 32 + lane;
  const int pos = prefix + row0 + lane;
  const int c = pos >= 0 ? pos >> 7 : -1;
  int32_t* srow = s_rows[wib][lane];
  if (nvis <= a.topk) {
    for (int t = 0; t < a.topk; ++t) srow[t] = t <= c ? t : -1;
  } else {
    RegList<TK> m;
    // With at least as many positions as CTAs every share holds some, and a
    // CTA between c0 and c1 holds units of this tile (a tile's cost
    // positions come before its first unit): no check.
    const bool dense = total >= a.grid;
    bool first = true;   // the first list is taken as it is
    for (int cj = c0; cj <= c1; ++cj) {
      if (!dense && !has_units(cj, total, a.grid)) continue;
      // The two teams' slots, key-major: the warp's 32 rows read 256
      // contiguous bytes per key.
      uint64_t l0[TK], l1[TK];
      const uint64_t* s0 = a.partials + 2 * (static_cast<int64_t>(cj) + tile) * 128 * TK + r;
      const uint64_t* s1 = s0 + 128 * TK;
#pragma unroll
      for (int k = 0; k < TK; ++k) {
        l0[k] = __ldcg(s0 + k * 128);
        l1[k] = __ldcg(s1 + k * 128);
      }
      if (first) {
#pragma unroll
        for (int k = 0; k < TK; ++k) m.v[k] = l0[k];
        first = false;
      } else {
        m.merge_sorted(l0);
      }
      m.merge_sorted(l1);
    }
    if (first) m.clear();   // no CTA held units of the tile (a malformed record)
    write_row_lane<TK>(m.v, c, a.init_blocks, a.local_blocks, a.topk, srow);
  }
  __syncwarp();
  // Row by row, lane = column (topk <= 32): contiguous stores, conflict-free
  // shared-memory reads.
  int32_t* out = a.ids + head * a.i_head + static_cast<int64_t>(qbeg + row0) * a.i_row;
  if (lane < a.topk)
    for (int rr = 0; rr < nrows; ++rr) out[rr * a.i_row + lane] = s_rows[wib][rr][lane];
}

template <bool kSelect, int TK, int NL = TK>
cudaError_t launch_prefill_t(const CUtensorMap& qmap, const CUtensorMap& kmap, const PrefillArgs& a,
                     int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<kSelect, TK, NL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, prefill_kernel<kSelect, TK, NL>, qmap, kmap, a);
}

cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const PrefillArgs& a,
                           int grid, cudaStream_t s) {
  if (a.partials == nullptr) return launch_prefill_t<false, 16>(qmap, kmap, a, grid, s);
  if (prefill_tk(a.topk) == 32) return launch_prefill_t<true, 32>(qmap, kmap, a, grid, s);
  // 16-key lists: the smallest list that holds a row's picks.  The usual
  // forced blocks (init 1-2, local 1-2) are served exactly; 3 forced blocks
  // at topk 16 (13 slots): causal 32K step 113.3 -> 106.8 us.
  const int m = a.topk - a.init_blocks - a.local_blocks;
  if (m <= 4) return launch_prefill_t<true, 16, 4>(qmap, kmap, a, grid, s);
  if (m <= 8) return launch_prefill_t<true, 16, 8>(qmap, kmap, a, grid, s);
  if (m <= 12) return launch_prefill_t<true, 16, 12>(qmap, kmap, a, grid, s);
  if (m <= 13) return launch_prefill_t<true, 16, 13>(qmap, kmap, a, grid, s);
  if (m <= 14) return launch_prefill_t<true, 16, 14>(qmap, kmap, a, grid, s);
  if (m <= 15) return launch_prefill_t<true, 16, 15>(qmap, kmap, a, grid, s);
  return launch_prefill_t<true, 16>(qmap, kmap, a, grid, s);
}

cudaError_t launch_prefill_merge(const PrefillMergeArgs& a, cudaStream_t s) {
  const int64_t warps = a.tiles * 4;
  if (warps == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((warps + kMergeWarps - 1) / kMergeWarps));
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return prefill_tk(a.topk) == 16 ? cudaLaunchKernelEx(&cfg, prefill_merge_kernel<16>, a)
                                  : cudaLaunchKernelEx(&cfg, prefill_merge_kernel<32>, a);
}

}  // namespace mm3idx
