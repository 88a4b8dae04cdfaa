// prefill.cu -- tensor-core causal block scorer for long query runs.
//
// Computes score[h, row, b] = sm_scale * max over the visible tokens of block
// b of q[row, h] . k[token] (vLLM MiniMax-M3 "index_topk" page,
// minimax_m3_index_score: per-token index scores for each visible sparse
// block, the max over a 128-token index-K block, causal through the request's
// prefix).  The design is ours:
//
//   * A unit is (request, head, 128-row query tile, key block).  Units are
//     enumerated from host-known sizes, assuming every request is
//     max_seq_len long (a capture-stable bound); units past a request's real
//     causal range do no math.  Each CTA of a persistent grid takes one
//     contiguous, equal share of the units, so the causal triangle is spread
//     evenly over the SMs.
//   * warp 0   : TMA producer: the 128 x 128 bf16 query tile (two 64-column
//                boxes, 128-byte swizzle, from a 3-D map over
//                [tokens, heads, 128]) once per tile, and each key page (from
//                a 2-D map over [pages*128, 128]) into a 4-stage ring.
//   * warp 1   : one thread issues tcgen05.mma, M = 128 query rows,
//                N = 128 key tokens, K = 128, into one of two 128-column fp32
//                TMEM accumulators.
//   * warps 2-5: epilogue: tcgen05.ld of the thread's query row (128 fp32
//                columns), causal mask only on diagonal blocks, row max,
//                scale, one fp32 store per (row, block).
#include <cuda_runtime.h>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "ptx.cuh"

namespace mm3idx {
namespace {

constexpr int kStages = 4;
constexpr int kAcc = 2;
constexpr int kTile = 32768;  // 128 x 128 bf16
constexpr int kThreads = 192;
constexpr int oQ = 0;
constexpr int oK = oQ + 2 * kTile;
constexpr int oBar = oK + kStages * kTile;
constexpr int kBars = 2 * kStages + 2 * kAcc + 4 + 1;
constexpr int oMisc = oBar + kBars * 8;
constexpr int kSmem = oMisc + 64 + 1024;
constexpr uint32_t kTmemCols = kAcc * 128;

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

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
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
  uint64_t* done_bar = q_empty + 2;
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
      uint32_t qaddr = 0;
      for (; ok && U.valid(); U.advance(a)) {
        const int req = U.rh / a.heads;
        const int prefix = clamp_len(a, req) - a.query_len;
        if (U.b >= tile_blocks(prefix, U.qt, a.query_len)) continue;
        if (U.rh != cur_rh || U.qt != cur_qt) {
          if (tq > 0) mma_commit(&q_empty[(tq - 1) & 1]);
          cur_rh = U.rh;
          cur_qt = U.qt;
          const int qs = tq & 1;
          ok = mbar_wait(&q_full[qs], (tq >> 1) & 1, abort_flag);
          if (!ok) break;
          qaddr = smem_u32(sQ + qs * kTile);
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
        const uint32_t d = tmem_base + ab * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = sdesc_kmajor_sw128(qaddr + (k >> 2) * (kTile / 2) + (k & 3) * 32);
          const uint64_t bd = sdesc_kmajor_sw128(kaddr + (k >> 2) * (kTile / 2) + (k & 3) * 32);
          mma_bf16(d, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        mma_commit(&empty[st]);
        mma_commit(&acc_full[ab]);
        ++it;
      }
      if (ok && tq > 0) mma_commit(&q_empty[(tq - 1) & 1]);
      mma_commit(done_bar);
      int dummy = 0;
      mbar_wait(done_bar, 0, &dummy);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- epilogue
    const int quad = warp & 3;
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
      if (active) {
        const uint32_t ab = it % kAcc, ar = it / kAcc;
        bool got = true;
        if (lane == 0) got = mbar_wait(&acc_full[ab], ar & 1, abort_flag);
        got = __shfl_sync(0xffffffffu, got, 0);
        float best = -INFINITY;
        if (got) {
          tc_fence_after();
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + ab * 128;
          const int lim = pos - U.b * 128;  // columns 0..lim are visible
          float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(taddr + c0, v);
            tmem_ld_wait32(v);
            if (lim >= 127) {
#pragma unroll
              for (int k = 0; k < 32; k += 4) {
                m0 = fmaxf(m0, __uint_as_float(v[k]));
                m1 = fmaxf(m1, __uint_as_float(v[k + 1]));
                m2 = fmaxf(m2, __uint_as_float(v[k + 2]));
                m3 = fmaxf(m3, __uint_as_float(v[k + 3]));
              }
            } else {
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (c0 + k <= lim) m0 = fmaxf(m0, __uint_as_float(v[k]));
            }
          }
          best = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[ab]);
        }
        if (!bar_and(1, 128, got)) {
          ok = false;
          break;
        }
        ++it;
        if (row_ok && pos >= 0) srow[U.b] = best * a.sm_scale;
      } else if (a.fill_width > 0 && row_ok) {
        srow[U.b] = -INFINITY;
      }
      // The tile's last scheduled block: blocks past the worst-case schedule.
      if (a.fill_width > 0 && row_ok && U.b == U.n - 1)
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
