// decode_fp4.cu -- persistent, warp-specialised decode kernel over NVFP4
// index-K pages: causal block scoring of a few query rows per request, with
// the fp32 scores written out (score mode) or a fused top-k selector (select
// mode).  Each key element is e4m3_rn_satfinite(e2m1 code * e4m3 scale), one
// scale per 16 elements (vLLM MiniMax-M3 "indexer_nvfp4" page, module
// docstring); the scoring and selection rules are the bf16 kernel's
// (decode.cu), and so are the partition, walker and merge warp
// (decode_common.cuh).
//
// The dequantised page never goes through shared memory: it is written into
// tensor memory and is the MMA's A operand there (tokens on the 128 TMEM
// lanes, K = 128 elements in 64 columns of bf16 pairs), with the request's
// query rows as B (N = 16 or 32 rows, K-major in shared memory).  A page is
// then read from shared memory once, as 9 KB of codes and scales, and the
// accumulator holds one token per lane and one query row per column, so a
// block's max is a max across lanes.
//
//   * warp 4     : producer.  Per page, one TMA tiled copy of the 8 KB of
//                  codes (64-byte swizzle, so that the dequantisers' per-token
//                  loads hit distinct banks) and one bulk copy of the 1 KB of
//                  scales into a ring of raw stages; the query rows of each
//                  request into a swizzled B tile.
//   * warps 8+   : dequantisers, in groups of four (one per TMEM lane
//                  quadrant); group g takes the pages it % groups == g.  A
//                  thread owns one token: 64 code bytes, 8 scale bytes, a
//                  per-scale table lookup (eight copies of the table, so the
//                  eight lanes of a shared-memory phase read eight distinct
//                  banks) and byte permutes give its 128 bf16 values, stored
//                  with tcgen05.st into one of four TMEM A buffers.
//   * warp 5     : one thread issues tcgen05.mma, A from TMEM, B = query rows,
//                  into one of four 32-column fp32 accumulators.
//   * warps 0-3  : epilogue, one per lane quadrant.  Loads its 32 tokens x N
//                  rows with tcgen05.ld, masks the causal tail per row and
//                  reduces each row across its 32 lanes (redux max); the four
//                  quadrant maxima go to shared memory.
//   * warp 6     : selector.  Lane n = query row n: the row's block score is
//                  the max of the four quadrant maxima times sm_scale; it is
//                  stored (score mode) or offered to the row's candidate list,
//                  handed to the merge warp at the end of each request.
//   * warp 7     : merge warp (decode_common.cuh).
//
// Every wait is bounded (ptx.cuh); a wait that gives up raises the CTA's
// abort flag and MM3IDX_DEV_TIMEOUT.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "decode_common.cuh"

namespace mm3idx {
namespace {

using namespace dec;

constexpr int kCodeBytes = kBlock * kD / 2;    // 8 KB: 128 tokens x 64 B
constexpr int kScaleBytes = kBlock * kD / 16;  // 1 KB: 128 tokens x 8 B
constexpr int kRawStride = 10240;              // codes (1024-aligned), scales, pad
constexpr int kABufs = 4;                      // dequantised pages in TMEM
constexpr int kACols = 64;                     // 128 bf16 per lane
constexpr int kDBufs = 4;                      // accumulators
constexpr int kDCols = 32;
constexpr int kDCol0 = kABufs * kACols;        // accumulators after the A buffers
constexpr uint32_t kTmemCols = 512;
constexpr int kTabCopies = 8;
constexpr int kProdWarp = 4, kMmaWarp = 5, kSelWarp = 6, kMergeWarp = 7, kDeqWarp0 = 8;
static_assert(kDCol0 + kDBufs * kDCols <= static_cast<int>(kTmemCols), "TMEM budget");

// NQ: query rows in the B tile (16 or 32); DG: dequantiser groups.
template <int NQ, int TK, int DG>
struct Cfg {
  static constexpr int kWarps = kDeqWarp0 + 4 * DG;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRawStages = 12;
  static constexpr int kQBytes = NQ * kD * 2;
  static constexpr int oRaw = 0;
  static constexpr int oTab = oRaw + kRawStages * kRawStride;  // [256 scales][8 copies] x 16 B
  static constexpr int oQ = oTab + 256 * kTabCopies * 16;
  static constexpr int oPart = oQ + 2 * kQBytes;               // [kDBufs][4 quadrants][32] fp32
  static constexpr int oHand = oPart + kDBufs * 4 * 32 * 4;    // [2 slots][TK][32] keys
  static constexpr int oBar = oHand + 2 * TK * kLanes * 8;
  static constexpr int kBars = 2 * kRawStages + 2 * kABufs + 4 * kDBufs + 4 + 4 + 1;
  static constexpr int oMisc = oBar + kBars * 8;
  static constexpr int kSmem = oMisc + 64 + 1024;
  static_assert(oTab % 1024 == 0 && oQ % 1024 == 0, "swizzled tiles must be 1024-byte aligned");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// Per-scale-byte magnitude table: for scale byte s, the bf16 bits of
// e4m3_rn_satfinite(m * e4m3(s)) for the eight e2m1 magnitudes
// m = 0, .5, 1, 1.5, 2, 3, 4, 6, as low bytes (words 0-1) and high bytes
// (words 2-3) for byte-permute lookups; kTabCopies copies side by side.
__device__ void build_fp4_table(uint4* tab, int tid, int nthreads) {
  const float mags[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  for (int s = tid; s < 256; s += nthreads) {
    const __half_raw sh = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(s), __NV_E4M3);
    const float sv = __half2float(__half(sh));
    uint32_t lo[2] = {0u, 0u}, hi[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const __nv_fp8_storage_t e = __nv_cvt_float_to_fp8(mags[k] * sv, __NV_SATFINITE, __NV_E4M3);
      const __half_raw eh = __nv_cvt_fp8_to_halfraw(e, __NV_E4M3);
      const float ev = __half2float(__half(eh));
      const uint32_t bits = __float_as_uint(ev) >> 16;  // exact: <= 4 significant bits
      lo[k >> 2] |= (bits & 0xFFu) << ((k & 3) * 8);
      hi[k >> 2] |= ((bits >> 8) & 0xFFu) << ((k & 3) * 8);
    }
    const uint4 v = make_uint4(lo[0], lo[1], hi[0], hi[1]);
#pragma unroll
    for (int c = 0; c < kTabCopies; ++c) tab[s * kTabCopies + c] = v;
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// d = a ^ (b & 0x80808080): the sign bits of b into a's bytes.
__device__ __forceinline__ uint32_t xor_signs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, 0x80808080, 0x78;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Eight e2m1 codes (nibble k = element k, sign in bit 3) -> four bf16x2
// words (element 2i in the low half of word i).
__device__ __forceinline__ void dequant8(uint32_t codes, const uint4& t, uint32_t* o) {
  const uint32_t sel0 = codes & 0x7777u;
  const uint32_t sel1 = (codes >> 16) & 0x7777u;
  const uint32_t lo0 = prmt(t.x, t.y, sel0), hi0 = prmt(t.z, t.w, sel0);
  const uint32_t lo1 = prmt(t.x, t.y, sel1), hi1 = prmt(t.z, t.w, sel1);
  // Bit 7 of byte k of s0 (s1) is the sign of element k (k + 4): the sign
  // of the even element of a code byte is its bit 3, of the odd one bit 7.
  const uint32_t c4 = codes << 4;
  const uint32_t s0 = prmt(c4, codes, 0x5140u), s1 = prmt(c4, codes, 0x7362u);
  const uint32_t h0 = xor_signs(hi0, s0), h1 = xor_signs(hi1, s1);
  o[0] = prmt(lo0, h0, 0x5140u);
  o[1] = prmt(lo0, h0, 0x7362u);
  o[2] = prmt(lo1, h1, 0x5140u);
  o[3] = prmt(lo1, h1, 0x7362u);
}

template <int NQ, int TK, int DG>
__global__ void __launch_bounds__(Cfg<NQ, TK, DG>::kThreads, 1)
    decode_fp4_kernel(const __grid_constant__ CUtensorMap cmap, const DecodeArgs a) {
  using C = Cfg<NQ, TK, DG>;
  constexpr int RS = C::kRawStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sRaw = sm + C::oRaw;
  const uint4* sTab = reinterpret_cast<const uint4*>(sm + C::oTab);
  uint8_t* sQ = sm + C::oQ;
  float* sPart = reinterpret_cast<float*>(sm + C::oPart);
  uint64_t* sHand = reinterpret_cast<uint64_t*>(sm + C::oHand);
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(sm + C::oBar);
  uint64_t* raw_empty = raw_full + RS;
  uint64_t* a_full = raw_empty + RS;
  uint64_t* a_empty = a_full + kABufs;
  uint64_t* acc_full = a_empty + kABufs;
  uint64_t* acc_empty = acc_full + kDBufs;
  uint64_t* red_full = acc_empty + kDBufs;
  uint64_t* red_empty = red_full + kDBufs;
  uint64_t* q_full = red_empty + kDBufs;
  uint64_t* q_empty = q_full + 2;
  uint64_t* h_full = q_empty + 2;
  uint64_t* h_empty = h_full + 2;
  uint64_t* done_bar = h_empty + 2;
  Misc* misc = reinterpret_cast<Misc*>(sm + C::oMisc);
  volatile int* abort_flag = &misc->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 4);
    }
    for (int s = 0; s < kABufs; ++s) {
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kDBufs; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
      mbar_init(&red_full[s], 4);
      mbar_init(&red_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
      mbar_init(&h_full[s], 1);
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
  build_fp4_table(reinterpret_cast<uint4*>(sm + C::oTab), threadIdx.x, C::kThreads);
  // Programmatic dependent launch: the set-up above overlaps the previous
  // kernel on the stream; its results are read only after this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kProdWarp) {
    if (lane == 0) prefetch_tensormap(&cmap);
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
    uint32_t it = 0;
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      const int slot = seg & 1;
      if (seg >= 2) ok = warp_wait(&q_empty[slot], ((seg >> 1) - 1) & 1, abort_flag);
      if (!ok) break;
      bool q_pending = true;
      auto put_q = [&]() {
        load_q_tile<NQ>(a, req, sQ + slot * C::kQBytes, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[slot]);
        q_pending = false;
      };
      const int32_t* trow = a.table + static_cast<int64_t>(req) * a.table_stride;
      for (int bc = b0; bc < b1 && ok; bc += 32) {
        const int mine = bc + lane;
        const int pg = mine < b1 ? __ldg(trow + mine) : 0;
        const int nblk = min(32, b1 - bc);
        for (int k = 0; k < nblk; ++k) {
          const int page = __shfl_sync(0xffffffffu, pg, k);
          const bool good = page >= 0 && page < a.num_pages;
          const uint32_t st = it % RS, rnd = it / RS;
          if (rnd > 0 && q_pending) put_q();
          if (rnd > 0) ok = warp_wait(&raw_empty[st], (rnd - 1) & 1, abort_flag);
          if (!ok) break;
          if (lane == 0) {
            if (good) {
              uint8_t* dst = sRaw + st * kRawStride;
              mbar_arrive_expect_tx(&raw_full[st], kCodeBytes + kScaleBytes);
              tma_load_2d(dst, &cmap, &raw_full[st], 0, page * kBlock, pol);
              bulk_load(dst + kCodeBytes, a.scales + static_cast<int64_t>(page) * kScaleBytes,
                        kScaleBytes, &raw_full[st], pol);
            } else {
              // Not loaded: the stage's stale bytes are dequantised and
              // scored, and the selector gives the block -inf.
              atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
              mbar_arrive(&raw_full[st]);
            }
          }
          __syncwarp();
          ++it;
        }
      }
      if (q_pending) put_q();
      ++seg;
    }
    // Let every copy this warp started land before the CTA can exit.
    if (lane == 0) {
      const uint32_t pending = it < static_cast<uint32_t>(RS) ? it : RS;
      for (uint32_t k = 0; k < pending; ++k) {
        const uint32_t idx = it - 1 - k;
        int dummy = 0;
        mbar_wait(&raw_full[idx % RS], (idx / RS) & 1, &dummy);
      }
    }
    __syncwarp();
  } else if (warp >= kDeqWarp0) {
    // --------------------------------------------------------- dequantisers
    const int group = (warp - kDeqWarp0) >> 2;
    const int quad = warp & 3;           // TMEM lanes 32*quad .. +31
    const int tok = quad * 32 + lane;    // this thread's token of the page
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const int swz = (tok >> 1) & 3;      // 64-byte swizzle of the code rows
    const int copy = lane & (kTabCopies - 1);
    uint32_t it = 0;
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      for (int b = b0; b < b1; ++b, ++it) {
        if (static_cast<int>(it % DG) != group) continue;
        const uint32_t rs = it % RS, rr = it / RS;
        const uint32_t ab = it % kABufs, ar = it / kABufs;
        bool got = true;
        if (lane == 0) {
          got = mbar_wait(&raw_full[rs], rr & 1, abort_flag);
          if (got && ar > 0) got = mbar_wait(&a_empty[ab], (ar - 1) & 1, abort_flag);
        }
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        // Every lane observes the completed phase itself before reading what
        // the copies wrote (the stage cannot move on before this warp frees it).
        mbar_try_wait(&raw_full[rs], rr & 1);
        tc_fence_after();
        const uint8_t* raw = sRaw + rs * kRawStride;
        const uint8_t* crow = raw + tok * 64;
        uint4 cw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) cw[c] = *reinterpret_cast<const uint4*>(crow + ((c ^ swz) << 4));
        const uint2 scw = *reinterpret_cast<const uint2*>(raw + kCodeBytes + tok * 8);
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rs]);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // Elements 64*half .. +63: scale groups 4*half .. +3, code chunks
          // 2*half, 2*half+1 (two groups, i.e. 16 code bytes, each).
          const uint32_t sw = half ? scw.y : scw.x;
          uint4 t[4];
#pragma unroll
          for (int g = 0; g < 4; ++g) t[g] = sTab[((sw >> (8 * g)) & 0xFFu) * kTabCopies + copy];
          uint32_t o[32];
          const uint4 c0 = cw[2 * half], c1 = cw[2 * half + 1];
          dequant8(c0.x, t[0], o + 0);
          dequant8(c0.y, t[0], o + 4);
          dequant8(c0.z, t[1], o + 8);
          dequant8(c0.w, t[1], o + 12);
          dequant8(c1.x, t[2], o + 16);
          dequant8(c1.y, t[2], o + 20);
          dequant8(c1.z, t[3], o + 24);
          dequant8(c1.w, t[3], o + 28);
          tmem_st32(t_lane + ab * kACols + 32 * half, o);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[ab]);
      }
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NQ);
      int seg = 0;
      uint32_t it = 0;
      bool ok = true;
      while (ok && walker.next(a, req, b0, b1, nb, preq)) {
        const int slot = seg & 1;
        ok = mbar_wait(&q_full[slot], (seg >> 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qaddr = smem_u32(sQ + slot * C::kQBytes);
        for (int b = b0; b < b1; ++b) {
          const uint32_t aa = it % kABufs, ar = it / kABufs;
          ok = mbar_wait(&a_full[aa], ar & 1, abort_flag);
          if (!ok) break;
          const uint32_t db = it % kDBufs, dr = it / kDBufs;
          if (dr > 0) ok = mbar_wait(&acc_empty[db], (dr - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem_base + kDCol0 + db * kDCols;
          const uint32_t at = tmem_base + aa * kACols;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t bd = sdesc_kmajor_sw128(qaddr + (k >> 2) * (NQ * 128) + (k & 3) * 32);
            mma_bf16_ts(d, at + 8 * k, bd, idesc, k > 0 ? 1u : 0u);
          }
          mma_commit(&a_empty[aa]);
          mma_commit(&acc_full[db]);
          ++it;
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
  } else if (warp < 4) {
    // ------------------------------------------------------------- epilogue
    const int quad = warp;
    const int tok = quad * 32 + lane;
    const int R = a.rows_per_req;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    uint32_t it = 0;
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      // Row n (query j = n / heads) sees token t of block b iff
      // 128 b + t <= seq - query_len + j.
      const int first_pos = req_len(a, req) - a.query_len;
      for (int b = b0; b < b1; ++b, ++it) {
        const uint32_t db = it % kDBufs, dr = it / kDBufs;
        if (!warp_wait(&acc_full[db], dr & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[NQ];
        if constexpr (NQ == 16) {
          tmem_ld16(t_lane + kDCol0 + db * kDCols, v);
          tmem_ld_wait16(v);
        } else {
          tmem_ld32(t_lane + kDCol0 + db * kDCols, v);
          tmem_ld_wait32(v);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[db]);
        const int lim = first_pos - b * kBlock;  // row n sees tokens 0 .. lim + n / heads
        float mine = -INFINITY;
        if (lim >= kBlock - 1) {
#pragma unroll
          for (int n = 0; n < NQ; ++n) {
            if (n < R) {
              const float m = warp_max_f32(__uint_as_float(v[n]));
              if (lane == n) mine = m;
            }
          }
        } else {
#pragma unroll
          for (int n = 0; n < NQ; ++n) {
            if (n < R) {
              const bool vis = tok <= lim + n / a.heads;
              const float m = warp_max_f32(vis ? __uint_as_float(v[n]) : -INFINITY);
              if (lane == n) mine = m;
            }
          }
        }
        if (dr > 0 && !warp_wait(&red_empty[db], (dr - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        sPart[(db * 4 + quad) * 32 + lane] = mine;
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_full[db]);
      }
    }
  } else if (warp == kSelWarp) {
    // ------------------------------------------------------------- selector
    const int n = lane;  // query row
    const int R = a.rows_per_req;
    const int my_j = n < R ? n / a.heads : 0;
    const int my_h = n < R ? n - my_j * a.heads : 0;
    const bool select = a.mode == kModeSelect;
    RegList<TK> list;
    uint32_t it = 0;
    int seg = 0;
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      const int pos = req_len(a, req) - a.query_len + my_j;
      const int c = pos >= 0 ? (pos >> 7) : -1;
      const int64_t row = static_cast<int64_t>(req) * a.query_len + my_j;
      const int32_t* trow = a.table + static_cast<int64_t>(req) * a.table_stride;
      list.clear();
      for (int b = b0; b < b1; ++b, ++it) {
        const int page = __ldg(trow + b);
        const uint32_t db = it % kDBufs, dr = it / kDBufs;
        if (!warp_wait(&red_full[db], dr & 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_try_wait(&red_full[db], dr & 1);  // each lane's own acquire of the maxima
        const float* P = sPart + db * 4 * 32 + n;
        const float m = fmaxf(fmaxf(P[0], P[32]), fmaxf(P[64], P[96]));
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_empty[db]);
        if (n < R) {
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
        const int hs = seg & 1;
        if (seg >= 2 && !warp_wait(&h_empty[hs], ((seg >> 1) - 1) & 1, abort_flag)) break;
        if (n < R) list.store_cols(sHand + hs * TK * kLanes, n);
        __syncwarp();
        if (lane == 0) mbar_arrive(&h_full[hs]);
      } else if (b1 == nb && a.fill_width > nb) {
        fill_past_blocks(a, req, nb, lane);
      }
      ++seg;
    }
  } else if (warp == kMergeWarp) {
    // ------------------------------------------------------------ merge warp
    merge_warp<TK, 1>(a, walker, total, sHand, h_full, h_empty, abort_flag, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && misc->abort) atomicOr(a.status, MM3IDX_DEV_TIMEOUT);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int NQ, int TK, int DG>
cudaError_t launch_t(const CUtensorMap& cmap, const DecodeArgs& a, int grid, cudaStream_t s) {
  using C = Cfg<NQ, TK, DG>;
  cudaError_t e = cudaFuncSetAttribute(decode_fp4_kernel<NQ, TK, DG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_fp4_kernel<NQ, TK, DG>, cmap, a);
}

}  // namespace

// 32-key lists need more registers per thread, so they keep one group of
// dequantisers (384 threads); 16-key lists take two (512 threads).
cudaError_t launch_decode_nvfp4(const CUtensorMap& cmap, const DecodeArgs& a, int grid,
                                cudaStream_t s) {
  const bool small = a.rows_per_req <= 16, tk16 = decode_tk(a.topk) == 16;
  if (small && tk16) return launch_t<16, 16, 2>(cmap, a, grid, s);
  if (small) return launch_t<16, 32, 1>(cmap, a, grid, s);
  if (tk16) return launch_t<32, 16, 2>(cmap, a, grid, s);
  return launch_t<32, 32, 1>(cmap, a, grid, s);
}

}  // namespace mm3idx
