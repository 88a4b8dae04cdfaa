// prefill.cu -- tensor-core causal block scorer for long query runs.
//
// Computes score[h, row, b] = sm_scale * max over the visible tokens of block
// b of q[row, h] . k[token] (vLLM MiniMax-M3 "index_topk" page,
// minimax_m3_index_score: per-token index scores for each visible sparse
// block, i.e. the largest token score inside the block, causal through the request's
// prefix).  The design is ours:
//
//   * A unit is (request, head, 128-row query tile, key block).  Units are
//     enumerated from host-known sizes, assuming every request is
//     max_seq_len long (a bound fixed across graph replays); units past a request's real
//     causal range do no math.  Each CTA of a persistent grid takes one
//     contiguous, equal share of the units, so the causal triangle is spread
//     evenly over the SMs.
//   * warp 0   : TMA producer: the 128 x 128 bf16 query tile (two 64-column
//                boxes, 128-byte swizzle, from a 3-D map over
//                [tokens, heads, 128]) once per tile, and each key page (from
//                a 2-D map over [pages*128, 128]) into a 4-stage ring.
//   * warp 1   : one thread copies each query tile into TMEM once
//                (tcgen05.cp) and issues tcgen05.mma with A (M = 128 query
//                rows) read from TMEM and B (N = 128 key tokens) from shared
//                memory, K = 128, into one of three 128-column fp32 TMEM
//                accumulators.  Reading only B from shared memory keeps the
//                operand traffic well inside shared-memory bandwidth.
//   * warps 2-9: epilogue, two teams of four warps taking alternate units:
//                tcgen05.ld of the thread's query row (128 fp32 columns),
//                causal mask only on diagonal blocks, row max with 3-input
//                max, scale, one fp32 store per (row, block).
#include <cuda_runtime.h>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "ptx.cuh"

namespace mm3idx {
namespace {

// The query tile is the MMA's A operand.  It is TMA-loaded into shared
// memory and, when kQInTmem, copied once per tile into TMEM (two 64-column
// buffers) so that every MMA reads only the key page from shared memory.
constexpr bool kQInTmem = true;
constexpr int kStages = 4;
constexpr int kAcc = kQInTmem ? 3 : 4;
constexpr uint32_t kAccCol0 = kQInTmem ? 128 : 0;  // first accumulator column
constexpr int kTile = 32768;  // 128 x 128 bf16
constexpr int kThreads = 320;
constexpr int oQ = 0;
constexpr int oK = oQ + 2 * kTile;
constexpr int oBar = oK + kStages * kTile;
constexpr int kBars = 2 * kStages + 2 * kAcc + 6 + 1;
constexpr int oMisc = oBar + kBars * 8;
constexpr int kSmem = oMisc + 64 + 1024;
constexpr uint32_t kTmemCols = 512;

struct Misc {
  uint32_t tmem;
  int abort;
};

// Visible block count of query tile qt under a given prefix length
// (positions prefix + 128*qt .. prefix + min(128*qt + 127, query_len - 1)).
__device__ __forceinline__ int tile_blocks(int prefix, int qt, int query_len) {
  const int last = prefix + min(qt * 128 + 127, query_len - 1);
  return last < 0 ? 0 : (last >> 7) + 1;
}

// Iterates this CTA's share of the unit list.
struct UnitIter {
  int64_t u, hi;
  int rh, qt, b, n;   // (request*heads + head), tile, block, scheduled blocks of the tile
  int wprefix;        // worst-case prefix: max_seq_len - query_len
  __device__ void init(const PrefillArgs& a, int64_t lo, int64_t hi_) {
    u = lo;
    hi = hi_;
    wprefix = a.max_seq_len - a.query_len;
    if (lo >= hi_) return;
    rh = static_cast<int>(lo / a.units_per_head);
    int64_t off = lo - static_cast<int64_t>(rh) * a.units_per_head;
    qt = 0;
    for (;;) {
      n = tile_blocks(wprefix, qt, a.query_len);
      if (off < n) break;
      off -= n;
      ++qt;
    }
    b = static_cast<int>(off);
  }
  __device__ bool valid() const { return u < hi; }
  __device__ void advance(const PrefillArgs& a) {
    ++u;
    if (++b < n) return;
    b = 0;
    if (++qt == a.qtiles) {
      qt = 0;
      ++rh;
    }
    n = tile_blocks(wprefix, qt, a.query_len);
  }
};

__device__ __forceinline__ int clamp_len(const PrefillArgs& a, int i) {
  return min(max(__ldg(a.seq_lens + i), 0), a.max_seq_len);
}

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
  uint64_t* acc_empty = acc_full + kAcc;
  uint64_t* q_full = acc_empty + kAcc;
  uint64_t* q_empty = q_full + 2;
  uint64_t* qtm_free = q_empty + 2;   // TMEM query buffer free again
  uint64_t* done_bar = qtm_free + 2;
  Misc* misc = reinterpret_cast<Misc*>(sm + oMisc);
  volatile int* abort_flag = &misc->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kAcc; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
      mbar_init(&qtm_free[s], 1);
    }
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_k = policy_evict_last();   // pages are re-read by later tiles
      const uint64_t pol_q = policy_evict_first();
      int cur_rh = -1, cur_qt = -1;
      uint32_t tq = 0, it = 0;
      bool ok = true;
      for (; ok && U.valid(); U.advance(a)) {
        const int req = U.rh / a.heads, head = U.rh - req * a.heads;
        const int prefix = clamp_len(a, req) - a.query_len;
        if (U.b >= tile_blocks(prefix, U.qt, a.query_len)) continue;  // no visible token
        if (U.rh != cur_rh || U.qt != cur_qt) {
          cur_rh = U.rh;
          cur_qt = U.qt;
          const int qs = tq & 1;
          if (tq >= 2) ok = mbar_wait(&q_empty[qs], ((tq >> 1) - 1) & 1, abort_flag);
          if (!ok) break;
          const int tok0 = req * a.query_len + U.qt * 128;
          mbar_arrive_expect_tx(&q_full[qs], kTile);
          tma_load_3d(sQ + qs * kTile, &qmap, &q_full[qs], 0, head, tok0, pol_q);
          tma_load_3d(sQ + qs * kTile + kTile / 2, &qmap, &q_full[qs], 64, head, tok0, pol_q);
          ++tq;
        }
        const uint32_t st = it % kStages, rnd = it / kStages;
        if (rnd > 0) ok = mbar_wait(&empty[st], (rnd - 1) & 1, abort_flag);
        if (!ok) break;
        const int page = __ldg(a.table + static_cast<int64_t>(req) * a.table_stride + U.b);
        if (page >= 0 && page < a.num_pages) {
          mbar_arrive_expect_tx(&full[st], kTile);
          tma_load_2d(sK + st * kTile, &kmap, &full[st], 0, page * 128, pol_k);
          tma_load_2d(sK + st * kTile + kTile / 2, &kmap, &full[st], 64, page * 128, pol_k);
        } else {
          atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
          mbar_arrive(&full[st]);
        }
        ++it;
      }
      // Drain: let every copy started above land before the CTA may exit.
      int dummy = 0;
      const uint32_t pend = it < static_cast<uint32_t>(kStages) ? it : kStages;
      for (uint32_t k = 0; k < pend; ++k) {
        const uint32_t idx = it - 1 - k;
        mbar_wait(&full[idx % kStages], (idx / kStages) & 1, &dummy);
      }
      if (tq > 0) mbar_wait(&q_full[(tq - 1) & 1], ((tq - 1) >> 1) & 1, &dummy);
      if (tq > 1) mbar_wait(&q_full[(tq - 2) & 1], ((tq - 2) >> 1) & 1, &dummy);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      int cur_rh = -1, cur_qt = -1;
      uint32_t tq = 0, it = 0;
      bool ok = true;
      uint32_t qaddr = 0, qtm = 0;
      for (; ok && U.valid(); U.advance(a)) {
        const int req = U.rh / a.heads;
        const int prefix = clamp_len(a, req) - a.query_len;
        if (U.b >= tile_blocks(prefix, U.qt, a.query_len)) continue;
        if (U.rh != cur_rh || U.qt != cur_qt) {
          if (tq > 0) mma_commit(kQInTmem ? &qtm_free[(tq - 1) & 1] : &q_empty[(tq - 1) & 1]);
          cur_rh = U.rh;
          cur_qt = U.qt;
          const int qs = tq & 1;
          ok = mbar_wait(&q_full[qs], (tq >> 1) & 1, abort_flag);
          if (!ok) break;
          qaddr = smem_u32(sQ + qs * kTile);
          if constexpr (kQInTmem) {
            // The MMAs of tile tq-2 read this TMEM buffer; let them finish.
            if (tq >= 2) ok = mbar_wait(&qtm_free[qs], ((tq >> 1) - 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            qtm = tmem_base + qs * 64;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tmem_cp_128x256b(qtm + k * 8,
                               sdesc_kmajor_sw128(qaddr + (k >> 2) * (kTile / 2) + (k & 3) * 32));
            mma_commit(&q_empty[qs]);   // the shared-memory tile is free once copied
          }
          ++tq;
        }
        const uint32_t st = it % kStages, rnd = it / kStages;
        ok = mbar_wait(&full[st], rnd & 1, abort_flag);
        if (!ok) break;
        const uint32_t ab = it % kAcc, ar = it / kAcc;
        if (ar > 0) ok = mbar_wait(&acc_empty[ab], (ar - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t kaddr = smem_u32(sK + st * kTile);
        const uint32_t d = tmem_base + kAccCol0 + ab * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bd = sdesc_kmajor_sw128(kaddr + (k >> 2) * (kTile / 2) + (k & 3) * 32);
          if constexpr (kQInTmem) {
            mma_bf16_ts(d, qtm + k * 8, bd, idesc, k > 0 ? 1u : 0u);
          } else {
            const uint64_t ad = sdesc_kmajor_sw128(qaddr + (k >> 2) * (kTile / 2) + (k & 3) * 32);
            mma_bf16(d, ad, bd, idesc, k > 0 ? 1u : 0u);
          }
        }
        mma_commit(&empty[st]);
        mma_commit(&acc_full[ab]);
        ++it;
      }
      if (ok && tq > 0 && !kQInTmem) mma_commit(&q_empty[(tq - 1) & 1]);
      mma_commit(done_bar);
      int dummy = 0;
      mbar_wait(done_bar, 0, &dummy);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- epilogue
    // Two teams of four warps (one warp per TMEM lane quadrant) take
    // alternate units, so two accumulators drain at once.
    const int team = (warp - 2) >> 2;
    const int quad = warp & 3;       // a warp may only read lanes 32*(warp%4)..+31
    const int r = quad * 32 + lane;  // query row within the tile
    uint32_t it = 0;
    bool ok = true;
    for (; ok && U.valid(); U.advance(a)) {
      const int req = U.rh / a.heads, head = U.rh - req * a.heads;
      const int prefix = clamp_len(a, req) - a.query_len;
      const int qrow = U.qt * 128 + r;            // query index inside the request
      const bool row_ok = qrow < a.query_len;
      const int pos = prefix + qrow;
      float* srow = a.score + head * a.s_head +
                    (static_cast<int64_t>(req) * a.query_len + qrow) * a.s_row;
      const bool active = U.b < tile_blocks(prefix, U.qt, a.query_len);
      const uint32_t mine = active ? it++ : 0u;
      if (active && (mine & 1u) == static_cast<uint32_t>(team)) {
        const uint32_t ab = mine % kAcc, ar = mine / kAcc;
        bool got = true;
        if (lane == 0) got = mbar_wait(&acc_full[ab], ar & 1, abort_flag);
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + kAccCol0 + ab * 128;
        const int lim = pos - U.b * 128;  // columns 0..lim are visible
        float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 64) {
          uint32_t v[32], w[32];
          tmem_ld32(taddr + c0, v);
          tmem_ld32(taddr + c0 + 32, w);
          tmem_ld_wait32x2(v, w);
          if (lim >= 127) {
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
              m0 = fmax3(m0, __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
              m1 = fmax3(m1, __uint_as_float(v[k + 2]), __uint_as_float(v[k + 3]));
              m0 = fmax3(m0, __uint_as_float(w[k]), __uint_as_float(w[k + 1]));
              m1 = fmax3(m1, __uint_as_float(w[k + 2]), __uint_as_float(w[k + 3]));
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              if (c0 + k <= lim) m0 = fmaxf(m0, __uint_as_float(v[k]));
              if (c0 + 32 + k <= lim) m1 = fmaxf(m1, __uint_as_float(w[k]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
        if (row_ok) srow[U.b] = fmaxf(m0, m1) * a.sm_scale;
      } else if (!active && a.fill_width > 0 && row_ok && (U.u & 1) == team) {
        srow[U.b] = -INFINITY;
      }
      // The tile's last scheduled block: blocks past the worst-case schedule.
      if (a.fill_width > 0 && row_ok && team == 0 && U.b == U.n - 1)
        for (int b = U.n; b < a.fill_width; ++b) srow[b] = -INFINITY;
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
