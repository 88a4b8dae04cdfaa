// prefill.cu -- tensor-core causal block scorer for long query runs.
//
// Computes score[h, row, b] = sm_scale * max over the visible tokens of block
// b of q[row, h] . k[token] (vLLM MiniMax-M3 "index_topk" page,
// minimax_m3_index_score: per-token index scores for each visible sparse
// block, i.e. the largest token score inside the block, causal through the
// request's prefix).  The design is ours:
//
//   * A unit is (request, head, 128-row query tile, pair of key blocks).
//     Units are enumerated from host-known sizes, assuming every request is
//     max_seq_len long (a bound fixed across graph replays); units past a
//     request's real causal range do no math.  Each CTA of a persistent grid
//     takes one contiguous, equal share of the units, so the causal triangle
//     is spread evenly over the SMs.
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
//                row's 128 columns with tcgen05.ld, frees the accumulator,
//                then takes the causal row max with 3-input max and stores
//                one fp32 score per (row, block).
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "ptx.cuh"

namespace mm3idx {

// Worst-case units of one (request, head): every query tile of a request of
// max_seq_len tokens, its visible blocks taken in pairs.
int64_t prefill_units_per_head(int32_t query_len, int32_t max_seq_len) {
  const int64_t wprefix = static_cast<int64_t>(max_seq_len) - query_len;
  const int64_t qtiles = (static_cast<int64_t>(query_len) + 127) / 128;
  int64_t n = 0;
  for (int64_t qt = 0; qt < qtiles; ++qt) {
    const int64_t last = wprefix + std::min<int64_t>(qt * 128 + 127, query_len - 1);
    n += ((last >> 7) + 2) / 2;
  }
  return n;
}

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

// Iterates this CTA's share of the unit list.
struct UnitIter {
  int64_t u, hi;
  int rh, qt, p, np;  // (request*heads + head), tile, pair, scheduled pairs of the tile
  int req, head;      // rh split into its request and head
  int wprefix;        // worst-case prefix: max_seq_len - query_len
  __device__ void init(const PrefillArgs& a, int64_t lo, int64_t hi_) {
    u = lo;
    hi = hi_;
    wprefix = a.max_seq_len - a.query_len;
    if (lo >= hi_) return;
    rh = static_cast<int>(lo / a.units_per_head);
    req = rh / a.heads;
    head = rh - req * a.heads;
    int64_t off = lo - static_cast<int64_t>(rh) * a.units_per_head;
    qt = 0;
    for (;;) {
      np = (tile_blocks(wprefix, qt, a.query_len) + 1) >> 1;
      if (off < np) break;
      off -= np;
      ++qt;
    }
    p = static_cast<int>(off);
  }
  __device__ bool valid() const { return u < hi; }
  __device__ void advance(const PrefillArgs& a) {
    ++u;
    if (++p < np) return;
    p = 0;
    if (++qt == a.qtiles) {
      qt = 0;
      ++rh;
      if (++head == a.heads) {
        head = 0;
        ++req;
      }
    }
    np = (tile_blocks(wprefix, qt, a.query_len) + 1) >> 1;
  }
};

// Per-tile facts every role needs, refreshed only when the tile changes.
struct TileInfo {
  int rh = -1, qt = -1, req = -1;
  int prefix = 0, nvis = 0;  // request prefix; visible blocks of the tile
  __device__ __forceinline__ bool refresh(const PrefillArgs& a, const UnitIter& U) {
    if (U.rh == rh && U.qt == qt) return false;
    if (U.req != req) {
      req = U.req;
      prefix = min(max(__ldg(a.seq_lens + req), 0), a.max_seq_len) - a.query_len;
    }
    rh = U.rh;
    qt = U.qt;
    nvis = tile_blocks(prefix, qt, a.query_len);
    return true;
  }
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

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

  const int64_t G = gridDim.x;
  const int64_t lo = a.total_units * blockIdx.x / G;
  const int64_t hi = a.total_units * (blockIdx.x + 1) / G;
  UnitIter U;
  U.init(a, lo, hi);
  TileInfo T;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the units; lane 0 issues the copies.  Page ids are
    // read 32 at a time (one per lane) and broadcast with shuffles.
    const uint64_t pol_k = policy_evict_last();   // pages are re-read by later tiles
    const uint64_t pol_q = policy_evict_first();
    const int nblk = (a.max_seq_len + kBlock - 1) / kBlock;  // table entries that exist
    int cur_rh = -1, cur_qt = -1;
    int pg_req = -1, pg_base = 0, pg = -1;
    uint32_t tq = 0, it = 0, st = 0, ph = 0;
    bool ok = true;
    for (; ok && U.valid(); U.advance(a)) {
      T.refresh(a, U);
      const int b0 = 2 * U.p;
      if (b0 >= T.nvis) continue;  // no visible token
      const bool two = b0 + 1 < T.nvis;
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
      const bool new_tile = U.rh != cur_rh || U.qt != cur_qt;
      if (lane == 0) {
        sInfo[st] = kInfoValid | (two ? kInfoTwo : 0u) | (new_tile ? kInfoNewTile : 0u);
        uint8_t* dst = sK + st * kStageBytes;
        const bool good = pa >= 0 && pa < a.num_pages && (!two || (pb >= 0 && pb < a.num_pages));
        if (good) {
          // Stage layout: [A cols 0-63][B cols 0-63][A cols 64-127][B cols 64-127],
          // i.e. 256 key rows per 64-column half, as the N = 256 operand.
          mbar_arrive_expect_tx(&full[st], two ? 2 * kPage : kPage);
          tma_load_2d(dst, &kmap, &full[st], 0, pa * 128, pol_k);
          tma_load_2d(dst + 2 * kHalf, &kmap, &full[st], 64, pa * 128, pol_k);
          if (two) {
            tma_load_2d(dst + kHalf, &kmap, &full[st], 0, pb * 128, pol_k);
            tma_load_2d(dst + 3 * kHalf, &kmap, &full[st], 64, pb * 128, pol_k);
          }
        } else {
          atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
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
        cur_rh = U.rh;
        cur_qt = U.qt;
        if (tq > 0) ok = warp_wait(q_empty, (tq - 1) & 1u, abort_flag);
        if (!ok) break;
        if (lane == 0) {
          const int tok0 = U.req * a.query_len + U.qt * 128;
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
    float* srow = nullptr;
    for (; ok && U.valid(); U.advance(a)) {
      if (T.refresh(a, U)) {
        const int qrow = U.qt * 128 + r;  // query index inside the request
        row_ok = qrow < a.query_len;
        pos = T.prefix + qrow;
        srow = a.score + U.head * a.s_head +
               (static_cast<int64_t>(U.req) * a.query_len + qrow) * a.s_row;
      }
      const int b0 = 2 * U.p;
      if (b0 < T.nvis) {
        const int b = b0 + team;
        const bool mine = b < T.nvis;
        bool got = true;
        if (lane == 0) got = mbar_wait(&acc_full[acc], (it >> 1) & 1u, abort_flag);
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v0[32], v1[32], v2[32], v3[32];
        if (mine) {
          const uint32_t taddr =
              tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * 256 + team * 128;
          tmem_ld32(taddr, v0);
          tmem_ld32(taddr + 32, v1);
          tmem_ld32(taddr + 64, v2);
          tmem_ld32(taddr + 96, v3);
          tmem_ld_wait32x4(v0, v1, v2, v3);
        }
        // The columns are in registers: hand the accumulator back first.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        if (mine && row_ok) {
          const int lim = pos - b * 128;  // columns 0..lim are visible
          float m0 = -INFINITY, m1 = -INFINITY;
          if (lim >= 127) {
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
              m0 = fmax3(m0, __uint_as_float(v0[k]), __uint_as_float(v0[k + 1]));
              m1 = fmax3(m1, __uint_as_float(v0[k + 2]), __uint_as_float(v0[k + 3]));
              m0 = fmax3(m0, __uint_as_float(v1[k]), __uint_as_float(v1[k + 1]));
              m1 = fmax3(m1, __uint_as_float(v1[k + 2]), __uint_as_float(v1[k + 3]));
              m0 = fmax3(m0, __uint_as_float(v2[k]), __uint_as_float(v2[k + 1]));
              m1 = fmax3(m1, __uint_as_float(v2[k + 2]), __uint_as_float(v2[k + 3]));
              m0 = fmax3(m0, __uint_as_float(v3[k]), __uint_as_float(v3[k + 1]));
              m1 = fmax3(m1, __uint_as_float(v3[k + 2]), __uint_as_float(v3[k + 3]));
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              if (k <= lim) m0 = fmaxf(m0, __uint_as_float(v0[k]));
              if (32 + k <= lim) m1 = fmaxf(m1, __uint_as_float(v1[k]));
              if (64 + k <= lim) m0 = fmaxf(m0, __uint_as_float(v2[k]));
              if (96 + k <= lim) m1 = fmaxf(m1, __uint_as_float(v3[k]));
            }
          }
          srow[b] = fmaxf(m0, m1) * a.sm_scale;
        }
        ++it;
        acc ^= 1u;
      }
      // The tile's last scheduled unit: blocks past the visible ones hold
      // -inf.  Each warp of team 0 fills its 32 rows one row at a time, lanes
      // on consecutive blocks, so the stores coalesce.
      if (a.fill_width > 0 && team == 0 && U.p == U.np - 1) {
        const int row0 = U.qt * 128 + quad * 32;
        const int nrows = min(32, a.query_len - row0);
        float* base = a.score + U.head * a.s_head +
                      (static_cast<int64_t>(U.req) * a.query_len + row0) * a.s_row;
        for (int rr = 0; rr < nrows; ++rr)
          for (int b = T.nvis + lane; b < a.fill_width; b += 32) base[rr * a.s_row + b] = -INFINITY;
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

cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const PrefillArgs& a,
                           int grid, cudaStream_t s) {
  cudaError_t e =
      cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  prefill_kernel<<<grid, kThreads, kSmem, s>>>(qmap, kmap, a);
  return cudaGetLastError();
}

}  // namespace mm3idx
