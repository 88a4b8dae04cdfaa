// decode.cu -- persistent, warp-specialised decode kernel over bf16 pages:
// causal block scoring of a few query rows per request against the paged
// index-K cache, with either the fp32 scores written out (score mode) or a
// fused top-k selector whose scores never leave the chip (select mode).
//
// What it computes follows the vLLM MiniMax-M3 "index_topk" page (module
// docstring; minimax_m3_index_decode).  The partition of the batch over the
// CTAs, the segment walker and the merge warp are in decode_common.cuh.  The
// roles of the warps:
//
//   * warp 2   : producer.  Walks the block table and TMA-loads each 32 KB page
//                (two 64-column boxes, 128-byte swizzle) into a ring of
//                pair slots: a unit of work is two consecutive blocks of one
//                request (or its last block alone), laid out as one 256-row
//                operand; writes each request's query rows into a swizzled
//                Q tile.
//   * warp 1   : one thread issues tcgen05.mma with the query rows as A
//                (M = 128, rows past heads*query_len unused) and the
//                unit's pages as B (N = 256 key tokens, or 128), K = 128;
//                fp32 accumulators in TMEM, two 256-column buffers.  Query
//                row n lands in TMEM lane n.  An MMA instruction costs about
//                the same time at N = 128 as at N = 256, so two pages per
//                instruction halve the tensor-core time per page, which
//                otherwise exceeds the time the page takes to stream from HBM.
//   * warps 0,4: epilogue, one per block of the unit.  Lane n loads its
//                row's 128 token scores with tcgen05.ld, masks only the
//                causal tail, takes the max with 3-input max, scales, and
//                either stores the score or offers the candidate key to its
//                row's sorted list, kept in registers.  At a request boundary
//                both warps hand their lists to the merge warp through shared
//                memory and go on streaming.
//   * warp 3   : merge warp (decode_common.cuh).
//
// Every wait is bounded (ptx.cuh).  A wait that gives up raises an abort flag
// shared by the CTA's roles and the MM3IDX_DEV_TIMEOUT status bit.
#include "decode_common.cuh"

namespace mm3idx {
namespace {

using namespace dec;

constexpr int kAccBufs = 2;
constexpr int kAccCols = 256;                        // a unit of two pages
constexpr uint32_t kTmemCols = kAccBufs * kAccCols;  // 512: the whole TMEM
constexpr int kPageBytes = kBlock * kD * 2;          // 32 KB bf16 page
constexpr int kHalfPage = kPageBytes / 2;            // 128 rows x 64 columns
constexpr int kSlotHalf = 2 * kHalfPage;             // one 64-column half of a pair slot
constexpr int kEpiA = 0, kMmaWarp = 1, kProdWarp = 2, kMergeWarp = 3, kEpiB = 4;
constexpr int kThreads = 160;

// Shared memory: the pair slots as two regions, one per 64-column half, so
// that the two pages of a slot are one 256-row K-major operand in each
// half ([slot][page][128 rows][128 B] per region); then the Q tiles.
// The query tile is always M = 128 rows: with two pages (N = 256) per MMA,
// the accumulator is the M = 128 layout (query row n in TMEM lane n, 256
// columns), the one the prefill scorer uses.
constexpr int MQ = 128;

template <int TK>
struct Cfg {
  static constexpr int kPairs = 2;
  static constexpr int kQBytes = MQ * kD * 2;
  static constexpr int oH0 = 0;
  static constexpr int oH1 = oH0 + kPairs * kSlotHalf;
  static constexpr int oQ = oH1 + kPairs * kSlotHalf;
  static constexpr int oHand = oQ + 2 * kQBytes;     // [2 slots][2 warps][TK][32]
  static constexpr int oBar = oHand + 2 * 2 * TK * kLanes * 8;
  static constexpr int kBars = 2 * kPairs + 2 * kAccBufs + 4 + 4 + 1;
  static constexpr int oMisc = oBar + kBars * 8;
  static constexpr int kSmem = oMisc + 64 + 1024;
  static_assert(oQ % 1024 == 0, "Q tile must be 1024-byte aligned");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}


// Row max of one block's 128 accumulator columns (this lane's TMEM lane),
// with the columns past `lim` left out when lim < 127.
__device__ __forceinline__ float acc_row_max(uint32_t taddr, int lim) {
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int c0 = 0; c0 < kBlock; c0 += 64) {
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
  return fmaxf(m0, m1);
}

// ------------------------------------------------------------------ kernel

template <int TK>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const DecodeArgs a) {
  using C = Cfg<TK>;
  constexpr int P = C::kPairs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sH0 = sm + C::oH0;
  uint8_t* sH1 = sm + C::oH1;
  uint8_t* sQ = sm + C::oQ;
  uint64_t* sHand = reinterpret_cast<uint64_t*>(sm + C::oHand);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::oBar);
  uint64_t* empty = full + P;
  uint64_t* acc_full = empty + P;
  uint64_t* acc_empty = acc_full + kAccBufs;
  uint64_t* q_full = acc_empty + kAccBufs;
  uint64_t* q_empty = q_full + 2;
  uint64_t* h_full = q_empty + 2;     // both epilogue warps handed a request's lists over
  uint64_t* h_empty = h_full + 2;     // the merge warp is done with a hand-over slot
  uint64_t* done_bar = h_empty + 2;
  Misc* misc = reinterpret_cast<Misc*>(sm + C::oMisc);
  volatile int* abort_flag = &misc->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kAccBufs; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
      mbar_init(&h_full[s], 2);
      mbar_init(&h_empty[s], 1);
    }
    mbar_init(done_bar, 1);
    misc->abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&misc->tmem, kTmemCols);
    tmem_relinquish();
  }
  // Launched as a programmatic dependent launch: everything above overlaps
  // the previous kernel on the stream, whose results (lengths, tables,
  // queries, pages) are read only after this wait.  The next kernel may be
  // scheduled as soon as this grid's CTAs make room.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kProdWarp) {
    if (lane == 0) prefetch_tensormap(&kmap);
    partition(a, misc, lane);
  } else if (warp == kMergeWarp) {
    prefetch_table_and_queries(a, lane);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc->tmem;
  const long long total = misc->total;
  Walker walker = make_walker(misc);

  int req, b0, b1, nb;
  long long preq;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    int seg = 0;
    uint32_t ut = 0;  // units issued
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      const int slot = seg & 1;
      if (seg >= 2) ok = warp_wait(&q_empty[slot], ((seg >> 1) - 1) & 1, abort_flag);
      if (!ok) break;
      // The query tile is written just before the first wait that could
      // block (slots are only freed by MMAs, which need the tile), so page
      // loads into free slots are already in flight meanwhile.
      bool q_pending = true;
      auto put_q = [&]() {
        load_q_tile<MQ>(a, req, sQ + slot * C::kQBytes, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[slot]);
        q_pending = false;
      };
      const int32_t* trow = a.table + static_cast<int64_t>(req) * a.table_stride;
      // Page ids are read 32 at a time, one per lane; units start at even
      // offsets from b0, so both pages of a unit sit in the same 32.
      for (int bc = b0; bc < b1 && ok; bc += 32) {
        const int mine = bc + lane;
        const int pg = mine < b1 ? __ldg(trow + mine) : 0;
        const int nblk = min(32, b1 - bc);
        for (int k = 0; k < nblk; k += 2) {
          const bool two = k + 1 < nblk;
          const int pa = __shfl_sync(0xffffffffu, pg, k);
          const int pb = __shfl_sync(0xffffffffu, pg, two ? k + 1 : k);
          const bool good_a = pa >= 0 && pa < a.num_pages;
          const bool good_b = two && pb >= 0 && pb < a.num_pages;
          const uint32_t st = ut % P, rnd = ut / P;
          if (rnd > 0 && q_pending) put_q();
          if (rnd > 0) ok = warp_wait(&empty[st], (rnd - 1) & 1, abort_flag);
          if (!ok) break;
          if (lane == 0) {
            // A page id out of range is not loaded (its stale bytes are
            // scored and the epilogue gives the block -inf).
            if (!good_a || (two && !good_b)) atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
            const uint32_t bytes = (good_a ? kPageBytes : 0) + (good_b ? kPageBytes : 0);
            uint8_t* h0 = sH0 + st * kSlotHalf;
            uint8_t* h1 = sH1 + st * kSlotHalf;
            if (bytes) {
              mbar_arrive_expect_tx(&full[st], bytes);
              if (good_a) {
                tma_load_2d(h0, &kmap, &full[st], 0, pa * kBlock, pol);
                tma_load_2d(h1, &kmap, &full[st], 64, pa * kBlock, pol);
              }
              if (good_b) {
                tma_load_2d(h0 + kHalfPage, &kmap, &full[st], 0, pb * kBlock, pol);
                tma_load_2d(h1 + kHalfPage, &kmap, &full[st], 64, pb * kBlock, pol);
              }
            } else {
              mbar_arrive(&full[st]);
            }
          }
          __syncwarp();
          ++ut;
        }
      }
      if (q_pending) put_q();
      ++seg;
    }
    // Let every copy this warp started land before the CTA can exit.
    if (lane == 0) {
      const uint32_t pending = ut < static_cast<uint32_t>(P) ? ut : P;
      for (uint32_t k = 0; k < pending; ++k) {
        const uint32_t idx = ut - 1 - k;
        int dummy = 0;
        mbar_wait(&full[idx % P], (idx / P) & 1, &dummy);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc2 = idesc_bf16_f32(MQ, 2 * kBlock);
      constexpr uint32_t idesc1 = idesc_bf16_f32(MQ, kBlock);
      int seg = 0;
      uint32_t ut = 0;
      bool ok = true;
      while (ok && walker.next(a, req, b0, b1, nb, preq)) {
        const int slot = seg & 1;
        ok = mbar_wait(&q_full[slot], (seg >> 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qaddr = smem_u32(sQ + slot * C::kQBytes);
        for (int b = b0; b < b1; b += 2) {
          const bool two = b + 1 < b1;
          const uint32_t st = ut % P, rnd = ut / P;
          ok = mbar_wait(&full[st], rnd & 1, abort_flag);
          if (!ok) break;
          const uint32_t ab = ut % kAccBufs, ar = ut / kAccBufs;
          if (ar > 0) ok = mbar_wait(&acc_empty[ab], (ar - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t k0 = smem_u32(sH0 + st * kSlotHalf), k1 = smem_u32(sH1 + st * kSlotHalf);
          const uint32_t d = tmem_base + ab * kAccCols;
          const uint32_t idesc = two ? idesc2 : idesc1;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ad = sdesc_kmajor_sw128(qaddr + (k >> 2) * (MQ * 128) + (k & 3) * 32);
            const uint64_t bd = sdesc_kmajor_sw128((k < 4 ? k0 : k1) + (k & 3) * 32);
            mma_bf16(d, ad, bd, idesc, k > 0 ? 1u : 0u);
          }
          mma_commit(&empty[st]);
          mma_commit(&acc_full[ab]);
          ++ut;
        }
        if (!ok) break;
        mma_commit(&q_empty[slot]);
        ++seg;
      }
      // Wait until every MMA issued above has finished before TMEM is freed.
      mma_commit(done_bar);
      int dummy = 0;
      mbar_wait(done_bar, 0, &dummy);
    }
    __syncwarp();
  } else if (warp == kEpiA || warp == kEpiB) {
    // ------------------------------------------------------------- epilogue
    const int e = warp == kEpiA ? 0 : 1;  // which block of each unit
    const int n = lane;  // query row (TMEM lane)
    const int R = a.rows_per_req;
    const int my_j = n < R ? n / a.heads : 0;
    const int my_h = n < R ? n - my_j * a.heads : 0;
    const bool select = a.mode == kModeSelect;
    RegList<TK> list;
    uint32_t ut = 0;
    int seg = 0;
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      const int seq = req_len(a, req);
      const int pos = seq - a.query_len + my_j;
      const int c = pos >= 0 ? (pos >> 7) : -1;
      const int64_t row = static_cast<int64_t>(req) * a.query_len + my_j;
      const int32_t* trow = a.table + static_cast<int64_t>(req) * a.table_stride;
      list.clear();
      int pg = 0;  // page ids 32 at a time, one per lane (units never straddle two 32s)
      for (int bu = b0; bu < b1; bu += 2, ++ut) {
        const int b = bu + e;
        const bool mine = b < b1;
        if (((bu - b0) & 31) == 0) pg = bu + lane < b1 ? __ldg(trow + bu + lane) : 0;
        const int page = __shfl_sync(0xffffffffu, pg, (b - b0) & 31);
        const uint32_t ab = ut % kAccBufs, ar = ut / kAccBufs;
        if (!warp_wait(&acc_full[ab], ar & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float m = mine ? acc_row_max(tmem_base + ab * kAccCols + e * kBlock, pos - b * kBlock)
                             : -INFINITY;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
        if (mine && n < R) {
          const float s = (page >= 0 && page < a.num_pages) ? m * a.sm_scale : -INFINITY;
          if (!select) {
            a.score[my_h * a.s_head + row * a.s_row + b] = s;
          } else if (b <= c && b >= a.init_blocks && b <= c - a.local_blocks) {
            list.offer(make_key(s, b));
          }
        }
      }
      if (!ok) break;
      if (select) {
        // Hand this request's lists to the merge warp and keep streaming.
        const int hs = seg & 1;
        if (seg >= 2 && !warp_wait(&h_empty[hs], ((seg >> 1) - 1) & 1, abort_flag)) break;
        if (n < R) list.store_cols(sHand + (hs * 2 + e) * TK * kLanes, n);
        __syncwarp();
        if (lane == 0) mbar_arrive(&h_full[hs]);
      } else if (e == 0 && b1 == nb && a.fill_width > nb) {
        fill_past_blocks(a, req, nb, lane);
      }
      ++seg;
    }
  } else if (warp == kMergeWarp) {
    // ------------------------------------------------------------ merge warp
    merge_warp<TK, 2>(a, walker, total, sHand, h_full, h_empty, abort_flag, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && misc->abort) atomicOr(a.status, MM3IDX_DEV_TIMEOUT);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int TK>
cudaError_t launch_t(const CUtensorMap& kmap, const DecodeArgs& a, int grid, cudaStream_t s) {
  using C = Cfg<TK>;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<TK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<TK>, kmap, a);
}

}  // namespace

int decode_ctas_per_sm() { return 1; }

cudaError_t launch_decode_bf16(const CUtensorMap& kmap, const DecodeArgs& a, int grid, cudaStream_t s) {
  if (decode_tk(a.topk) == 16) return launch_t<16>(kmap, a, grid, s);
  return launch_t<32>(kmap, a, grid, s);
}

}  // namespace mm3idx
