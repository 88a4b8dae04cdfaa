// decode_fp4.cu -- persistent, warp-specialised decode kernel over NVFP4
// index-K pages: causal block scoring of a few query rows per request, with
// the fp32 scores written out (score mode) or a fused top-k selector (select
// mode).  Each key element is e4m3_rn_satfinite(e2m1 code * e4m3 scale), one
// scale per 16 elements (vLLM MiniMax-M3 "indexer_nvfp4" page, module
// docstring); every such value is exact in bf16, so the page is dequantised
// to bf16 and scored on the tensor cores against the bf16 query rows exactly
// as the bf16 kernel (decode.cu) scores bf16 pages, with the same partition,
// walker and merge warp (decode_common.cuh).
//
// A tcgen05.mma instruction costs about the same time whatever its N, and a
// page needs eight of them (K = 128 in steps of 16), so the instruction rate
// bounds the kernel long before HBM does; each MMA therefore takes two pages
// (N = 256 key tokens) with the query rows as A (M = 128).
//
//   * warp 2   : producer.  Per page, one TMA tiled copy of the 8 KB of codes
//                (64-byte swizzle, so that the dequantisers' per-token loads
//                hit distinct banks) and one bulk copy of the 1 KB of scales
//                into a ring of raw stages, the pages further ahead pulled
//                into L2 first; the query rows of each request into the Q
//                tile.
//   * warps 3+ : dequantisers, two groups of four; group g takes page g of
//                each two-page unit.  A thread owns one token: 64 code bytes,
//                8 scale bytes, a per-scale table lookup (copies of the table
//                side by side spread the lanes' lookups over the banks) and
//                byte permutes give its 128 bf16 values, stored straight into
//                the unit's slot in the 128-byte-swizzled K-major layout of
//                the MMA's B operand (the eight lanes of a store phase hit
//                eight distinct 16-byte bank groups).
//   * warp 1   : one thread issues tcgen05.mma, A = query rows, B = the
//                unit's slot (N = 256, or 128 for a request's last odd
//                block), into one of two 256-column fp32 accumulators.
//   * warp 0   : epilogue: lane n = query row n takes its row's causal block
//                max of both blocks of each unit (decode.cu's epilogue), and
//                at the end of each request merges its candidate lists itself
//                (decode_common.cuh, merge_request): with one or two requests
//                per CTA this stalls the pipeline rarely, and the shared
//                memory of a hand-over and the registers of a merge warp go
//                to a deeper raw ring instead.
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
constexpr int kAccBufs = 2;
constexpr int kAccCols = 256;                  // a unit of two pages
constexpr uint32_t kTmemCols = kAccBufs * kAccCols;
constexpr int kHalfPage = kBlock * 64 * 2;     // 128 rows x 64 bf16 = 16 KB
constexpr int kSlotHalf = 2 * kHalfPage;       // one 64-column half of a two-page slot
constexpr int kEpiWarp = 0, kMmaWarp = 1, kProdWarp = 2, kDeqWarp0 = 3;
constexpr int kThreads = (kDeqWarp0 + 8) * 32;
constexpr int MQ = 128;                        // query tile rows (the M = 128 layout)
constexpr int kAhead = 16;                     // pages pulled into L2 ahead of the ring (< 32)

// The warp pulls one page's codes (64 lines of 128 B) and scales (8 lines)
// into L2, two or three lines per lane.
__device__ __forceinline__ void prefetch_page_l2(const DecodeArgs& a, int page, int lane) {
  const uint8_t* c = a.codes + static_cast<int64_t>(page) * kCodeBytes;
  asm volatile("prefetch.global.L2 [%0];" ::"l"(c + lane * 128));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(c + (lane + 32) * 128));
  if (lane < kScaleBytes / 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.scales + static_cast<int64_t>(page) * kScaleBytes +
                                                   lane * 128));
}

// Shared memory: the two-page slots as two regions, one per 64-column half
// ([slot][page][128 rows][128 B] each), the Q tile, the raw ring, the table,
// the epilogue's lists for its merges.  32-key lists take one raw stage less.
template <int TK>
struct Cfg {
  static constexpr int kPairs = 2;
  static constexpr int kRawStages = TK == 16 ? 5 : 4;
  static constexpr int kTabCopies = 2;
  static constexpr int kQBytes = MQ * kD * 2;
  static constexpr int oH0 = 0;
  static constexpr int oH1 = oH0 + kPairs * kSlotHalf;
  static constexpr int oQ = oH1 + kPairs * kSlotHalf;
  static constexpr int oRaw = oQ + kQBytes;
  static constexpr int oTab = oRaw + kRawStages * kRawStride;   // [256 scales][copies] x 16 B
  static constexpr int oList = oTab + 256 * kTabCopies * 16;    // [TK][32] keys
  static constexpr int oBar = oList + TK * kLanes * 8;
  static constexpr int kBars = 2 * kRawStages + 2 * kPairs + 2 * kAccBufs + 2 + 1;
  static constexpr int oMisc = oBar + kBars * 8;
  static constexpr int kSmem = oMisc + 64 + 1024;
  static_assert(oQ % 1024 == 0 && oRaw % 1024 == 0, "swizzled tiles must be 1024-byte aligned");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// Per-scale-byte magnitude table: for scale byte s, the bf16 bits of
// e4m3_rn_satfinite(m * e4m3(s)) for the eight e2m1 magnitudes
// m = 0, .5, 1, 1.5, 2, 3, 4, 6, as low bytes (words 0-1) and high bytes
// (words 2-3) for byte-permute lookups; `copies` copies side by side.
__device__ void build_fp4_table(uint4* tab, int copies, int tid, int nthreads) {
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
    for (int c = 0; c < copies; ++c) tab[s * copies + c] = v;
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
__device__ __forceinline__ uint4 dequant8(uint32_t codes, const uint4& t) {
  const uint32_t sel0 = codes & 0x7777u;
  const uint32_t sel1 = (codes >> 16) & 0x7777u;
  const uint32_t lo0 = prmt(t.x, t.y, sel0), hi0 = prmt(t.z, t.w, sel0);
  const uint32_t lo1 = prmt(t.x, t.y, sel1), hi1 = prmt(t.z, t.w, sel1);
  // Bit 7 of byte k of s0 (s1) is the sign of element k (k + 4): the sign
  // of the even element of a code byte is its bit 3, of the odd one bit 7.
  const uint32_t c4 = codes << 4;
  const uint32_t s0 = prmt(c4, codes, 0x5140u), s1 = prmt(c4, codes, 0x7362u);
  const uint32_t h0 = xor_signs(hi0, s0), h1 = xor_signs(hi1, s1);
  return make_uint4(prmt(lo0, h0, 0x5140u), prmt(lo0, h0, 0x7362u), prmt(lo1, h1, 0x5140u),
                    prmt(lo1, h1, 0x7362u));
}

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

template <int TK>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fp4_kernel(const __grid_constant__ CUtensorMap cmap, const DecodeArgs a) {
  using C = Cfg<TK>;
  constexpr int RS = C::kRawStages;
  constexpr int P = C::kPairs;
  constexpr int NC = C::kTabCopies;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sH0 = sm + C::oH0;
  uint8_t* sH1 = sm + C::oH1;
  uint8_t* sQ = sm + C::oQ;
  uint8_t* sRaw = sm + C::oRaw;
  const uint4* sTab = reinterpret_cast<const uint4*>(sm + C::oTab);
  uint64_t* sList = reinterpret_cast<uint64_t*>(sm + C::oList);
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(sm + C::oBar);
  uint64_t* raw_empty = raw_full + RS;
  uint64_t* slot_full = raw_empty + RS;    // both dequantiser groups wrote the unit
  uint64_t* slot_empty = slot_full + P;    // the unit's MMAs are done with the slot
  uint64_t* acc_full = slot_empty + P;
  uint64_t* acc_empty = acc_full + kAccBufs;
  uint64_t* q_full = acc_empty + kAccBufs;
  uint64_t* q_empty = q_full + 1;
  uint64_t* done_bar = q_empty + 1;
  Misc* misc = reinterpret_cast<Misc*>(sm + C::oMisc);
  volatile int* abort_flag = &misc->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 4);
    }
    for (int s = 0; s < P; ++s) {
      mbar_init(&slot_full[s], 8);
      mbar_init(&slot_empty[s], 1);
    }
    for (int s = 0; s < kAccBufs; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(done_bar, 1);
    misc->abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&misc->tmem, kTmemCols);
    tmem_relinquish();
  }
  build_fp4_table(reinterpret_cast<uint4*>(sm + C::oTab), NC, threadIdx.x, kThreads);
  // Programmatic dependent launch: the set-up above overlaps the previous
  // kernel on the stream; its results are read only after this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kProdWarp) {
    if (lane == 0) prefetch_tensormap(&cmap);
    partition(a, misc, lane);
  } else if (warp == kEpiWarp) {
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
    uint32_t it = 0;  // pages issued
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      // One Q tile: it is rewritten once the previous request's MMAs are
      // done, just before the first wait that could block, so that page
      // loads are already in flight meanwhile.
      bool q_pending = true;
      auto put_q = [&]() {
        if (seg > 0) ok = warp_wait(q_empty, (seg - 1) & 1, abort_flag);
        if (ok) {
          load_q_tile<MQ>(a, req, sQ, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(q_full);
        }
        q_pending = false;
      };
      const int32_t* trow = a.table + static_cast<int64_t>(req) * a.table_stride;
      // Page ids 32 at a time (one per lane), the next 32 read one chunk
      // early.  The request's first kAhead pages are pulled into L2 here,
      // and page k + kAhead when page k is issued, so that the copies into
      // the ring mostly find their pages in L2.
      int pg_next = b0 + lane < b1 ? __ldg(trow + b0 + lane) : -1;
      for (int k = 0; k < kAhead; ++k) {
        const int p = __shfl_sync(0xffffffffu, pg_next, k);
        if (p >= 0 && p < a.num_pages) prefetch_page_l2(a, p, lane);
      }
      for (int bc = b0; bc < b1 && ok; bc += 32) {
        const int pg = pg_next;
        pg_next = bc + 32 + lane < b1 ? __ldg(trow + bc + 32 + lane) : -1;
        const int nblk = min(32, b1 - bc);
        for (int k = 0; k < nblk; ++k) {
          const int page = __shfl_sync(0xffffffffu, pg, k);
          const int ka = k + kAhead;
          const int ahead = __shfl_sync(0xffffffffu, ka < 32 ? pg : pg_next, ka & 31);
          if (ahead >= 0 && ahead < a.num_pages) prefetch_page_l2(a, ahead, lane);
          const bool good = page >= 0 && page < a.num_pages;
          const uint32_t st = it % RS, rnd = it / RS;
          if (rnd > 0 && q_pending) put_q();
          if (!ok) break;
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
              // scored, and the epilogue gives the block -inf.
              atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
              mbar_arrive(&raw_full[st]);
            }
          }
          __syncwarp();
          ++it;
        }
      }
      if (ok && q_pending) put_q();
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
    const int group = (warp - kDeqWarp0) >> 2;   // which page of each unit
    const int tok = ((warp - kDeqWarp0) & 3) * 32 + lane;
    const int swz = (tok >> 1) & 3;                // 64-byte swizzle of the code rows
    const int copy = lane % NC;
    // This token's rows in the two halves of a slot (128-byte swizzle).
    const uint32_t row_off = group * kHalfPage + (tok >> 3) * 1024 + (tok & 7) * 128;
    uint32_t it = 0, ut = 0;  // pages and units so far
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      for (int bu = b0; bu < b1; bu += 2, ++ut) {
        const bool two = bu + 1 < b1;
        const bool mine = group == 0 || two;
        const uint32_t pit = it + group;           // this group's page of the unit
        it += two ? 2 : 1;
        const uint32_t st = ut % P, sr = ut / P;
        const uint32_t rs = pit % RS, rr = pit / RS;
        bool got = true;
        if (lane == 0) {
          if (mine) got = mbar_wait(&raw_full[rs], rr & 1, abort_flag);
          // The slot's previous unit must be consumed before this group
          // writes it or counts towards its next phase.
          if (got && sr > 0) got = mbar_wait(&slot_empty[st], (sr - 1) & 1, abort_flag);
        }
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        if (mine) {
          // Every lane observes the completed phase itself before reading
          // what the copies wrote.
          mbar_try_wait(&raw_full[rs], rr & 1);
          const uint8_t* raw = sRaw + rs * kRawStride;
          const uint8_t* crow = raw + tok * 64;
          uint4 cw[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) cw[c] = *reinterpret_cast<const uint4*>(crow + ((c ^ swz) << 4));
          const uint2 scw = *reinterpret_cast<const uint2*>(raw + kCodeBytes + tok * 8);
          __syncwarp();
          if (lane == 0) mbar_arrive(&raw_empty[rs]);
          uint8_t* h0 = sH0 + st * kSlotHalf + row_off;
          uint8_t* h1 = sH1 + st * kSlotHalf + row_off;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            // Scale group g: elements 16g .. 16g+15, code words 2g, 2g+1,
            // output chunks 2g, 2g+1 (8 elements each) of the 16 in the row.
            const uint32_t sb = ((g < 4 ? scw.x : scw.y) >> (8 * (g & 3))) & 0xFFu;
            const uint4 t = sTab[sb * NC + copy];
            const uint4 c = cw[g >> 1];
            const uint32_t w0 = (g & 1) ? c.z : c.x, w1 = (g & 1) ? c.w : c.y;
            uint8_t* hb = g < 4 ? h0 : h1;
            const int c0 = (2 * g) & 7, c1 = (2 * g + 1) & 7;
            *reinterpret_cast<uint4*>(hb + ((c0 ^ (tok & 7)) << 4)) = dequant8(w0, t);
            *reinterpret_cast<uint4*>(hb + ((c1 ^ (tok & 7)) << 4)) = dequant8(w1, t);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&slot_full[st]);
      }
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc2 = idesc_bf16_f32(MQ, 2 * kBlock);
      constexpr uint32_t idesc1 = idesc_bf16_f32(MQ, kBlock);
      const uint32_t qaddr = smem_u32(sQ);
      int seg = 0;
      uint32_t ut = 0;
      bool ok = true;
      while (ok && walker.next(a, req, b0, b1, nb, preq)) {
        ok = mbar_wait(q_full, seg & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        for (int b = b0; b < b1; b += 2) {
          const bool two = b + 1 < b1;
          const uint32_t st = ut % P, rnd = ut / P;
          ok = mbar_wait(&slot_full[st], rnd & 1, abort_flag);
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
          mma_commit(&slot_empty[st]);
          mma_commit(&acc_full[ab]);
          ++ut;
        }
        if (!ok) break;
        mma_commit(q_empty);
        ++seg;
      }
      // Wait until every MMA issued above has finished before TMEM is freed.
      mma_commit(done_bar);
      int dummy = 0;
      mbar_wait(done_bar, 0, &dummy);
    }
    __syncwarp();
  } else if (warp == kEpiWarp) {
    // ------------------------------------------------------------- epilogue
    const int n = lane;                   // query row (TMEM lane)
    const int R = a.rows_per_req;
    const int my_j = n < R ? n / a.heads : 0;
    const int my_h = n < R ? n - my_j * a.heads : 0;
    const bool select = a.mode == kModeSelect;
    // Requests with no blocks first, then dry runs of both merge paths
    // (decode_common.cuh), all before the first accumulator is ready.
    fill_empty_requests(a, lane);
    if (select) {
      const MergeGeom none{0, 1, true};
      merge_request<TK, 1>(a, 0, 0, 1, none, 1, sList, lane, true, false);
      merge_request<TK, 1>(a, 0, 0, 1, none, 1, sList, lane, true, true);
    }
    RegList<TK> list;
    uint32_t ut = 0;
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      const int seq = req_len(a, req);
      const int pos = seq - a.query_len + my_j;
      const MergeGeom geo = merge_geom(nb, preq, total);
      const int c = pos >= 0 ? (pos >> 7) : -1;
      const int64_t row = static_cast<int64_t>(req) * a.query_len + my_j;
      const int32_t* trow = a.table + static_cast<int64_t>(req) * a.table_stride;
      list.clear();
      int pg = 0;  // page ids 32 at a time, one per lane (units never straddle two 32s)
      for (int bu = b0; bu < b1; bu += 2, ++ut) {
        const bool two = bu + 1 < b1;
        if (((bu - b0) & 31) == 0) pg = bu + lane < b1 ? __ldg(trow + bu + lane) : 0;
        const int page0 = __shfl_sync(0xffffffffu, pg, (bu - b0) & 31);
        const int page1 = __shfl_sync(0xffffffffu, pg, (bu + 1 - b0) & 31);
        const uint32_t ab = ut % kAccBufs, ar = ut / kAccBufs;
        if (!warp_wait(&acc_full[ab], ar & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float m0 = acc_row_max(tmem_base + ab * kAccCols, pos - bu * kBlock);
        const float m1 =
            two ? acc_row_max(tmem_base + ab * kAccCols + kBlock, pos - (bu + 1) * kBlock) : -INFINITY;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
        if (n < R) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int b = bu + e;
            if (e == 1 && !two) break;
            const int page = e ? page1 : page0;
            const float s =
                (page >= 0 && page < a.num_pages) ? (e ? m1 : m0) * a.sm_scale : -INFINITY;
            if (!select) {
              a.score[my_h * a.s_head + row * a.s_row + b] = s;
            } else if (b <= c && b >= a.init_blocks && b <= c - a.local_blocks) {
              list.offer(make_key(s, b));
            }
          }
        }
      }
      if (!ok) break;
      if (select) {
        if (n < R) list.store_cols(sList, n);
        __syncwarp();
        merge_request<TK, 1>(a, req, preq, seq, geo, total, sList, lane, false, false);
        __syncwarp();
      } else if (b1 == nb && a.fill_width > nb) {
        fill_past_blocks(a, req, nb, lane);
      }
    }
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
cudaError_t launch_t(const CUtensorMap& cmap, const DecodeArgs& a, int grid, cudaStream_t s) {
  using C = Cfg<TK>;
  cudaError_t e = cudaFuncSetAttribute(decode_fp4_kernel<TK>,
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
  return cudaLaunchKernelEx(&cfg, decode_fp4_kernel<TK>, cmap, a);
}

}  // namespace

cudaError_t launch_decode_nvfp4(const CUtensorMap& cmap, const DecodeArgs& a, int grid,
                                cudaStream_t s) {
  if (decode_tk(a.topk) == 16) return launch_t<16>(cmap, a, grid, s);
  return launch_t<32>(cmap, a, grid, s);
}

}  // namespace mm3idx
