// decode.cu -- persistent, warp-specialised decode kernel: causal block
// scoring of a few query rows per request against the paged index-K cache,
// with either the fp32 scores written out (score mode) or a fused top-k
// selector whose scores never leave the chip (select mode).
//
// What it computes follows the vLLM MiniMax-M3 "index_topk" page
// (module docstring; minimax_m3_index_decode: fused decode score + adaptive
// top-k with a final merge of per-chunk partial top-k lists, ids 0-indexed
// with -1 pad) and "indexer_cp_exchange" (forced init/local blocks are
// pinned, packed 64-bit candidate keys).  The design is ours:
//
//   * The work list is every (request, logical block) pair of the batch,
//     flattened request-major.  Each CTA takes one contiguous, equal share, so
//     ragged lengths cost no imbalance.  Shares are computed on the device
//     from seq_lens (no host round trip; CUDA-graph safe).
//   * warp 2   : producer.  Walks the block table and TMA-loads each 32 KB page
//                (two 64-column boxes, 128-byte swizzle) into a ring of stages;
//                writes each request's query rows into a swizzled Q tile.
//                NVFP4: bulk-copies the 9 KB code+scale page into a raw ring.
//   * warps 5+ : (NVFP4 only) dequantise raw pages into bf16 tiles in the same
//                swizzled layout, via a per-scale-byte magnitude table.
//   * warp 1   : one thread issues tcgen05.mma with the query rows as A
//                (M = 64 or 128, rows past heads*query_len unused) and the page
//                as B (N = 128 tokens), K = 128; fp32 accumulators in TMEM,
//                four 128-column buffers.  Query row n lands in TMEM lane n.
//   * warps 0,4: epilogue, alternate blocks.  Lane n loads its row's 128
//                token scores with tcgen05.ld, masks only the causal tail,
//                takes the max with 3-input max, scales, and either stores the
//                score or offers the candidate key to its row's sorted list,
//                kept in registers.  At a request boundary both warps hand
//                their lists to the merge warp through shared memory and go
//                on streaming.
//   * warp 3   : merge warp.  Folds the two lists of each row and writes the
//                ids of requests held by one CTA (forced blocks re-pinned,
//                ascending, -1 pad).  For a request split across CTAs it
//                publishes the lists and takes a ticket; the last of the
//                request's CTAs to arrive merges all their lists and writes
//                the rows.  Split requests are streamed first, so these
//                merges overlap the rest of the stream.
//
// Every wait is bounded (ptx.cuh).  A wait that gives up raises an abort flag
// shared by the CTA's roles and the MM3IDX_DEV_TIMEOUT status bit.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "ptx.cuh"
#include "warp_select.cuh"

namespace mm3idx {
namespace {

constexpr int kAccBufs = 4;
constexpr int kAccCols = 128;                        // one page of tokens
constexpr uint32_t kTmemCols = kAccBufs * kAccCols;  // 512: the whole TMEM
constexpr int kTileBytes = kBlock * kD * 2;          // 32 KB bf16 page
constexpr int kFp4CodeBytes = kBlock * kD / 2;       // 8 KB
constexpr int kFp4ScaleBytes = kBlock * kD / 16;     // 1 KB
constexpr int kFp4RawBytes = kFp4CodeBytes + kFp4ScaleBytes;
constexpr int kLanes = 32;                           // rows per list slot
constexpr int kEpiA = 0, kMmaWarp = 1, kProdWarp = 2, kMergeWarp = 3, kEpiB = 4, kDeqWarp0 = 5;
// NVFP4: warps kDeqWarp0.. dequantise.  With 16-key lists the kernel fits
// in 128 registers per thread, so eight warps (two per SM sub-partition) can
// overlap one warp's shared-memory latencies with another's arithmetic;
// 32-key lists need more registers and keep four.

template <bool FP4, int MQ, int TK>
struct Cfg {
  // NVFP4 raw pages arrive far ahead of their use, so shared memory goes to
  // the bf16 stages between the dequantisers and the tensor core first.
  static constexpr int kStages =
      FP4 ? ((MQ == 64 && TK == 16) ? 4 : (MQ == 64 ? 3 : 2)) : (MQ == 64 ? 5 : 4);
  static constexpr int kRawStages = FP4 ? ((MQ == 64 && TK == 16) ? 4 : 6) : 0;
  static constexpr int kDeqWarps = FP4 ? (TK == 16 ? 8 : 4) : 0;
  static constexpr int kThreads = FP4 ? (kDeqWarp0 + kDeqWarps) * 32 : 160;
  static constexpr int kQBytes = MQ * kD * 2;
  static constexpr int oA = 0;
  static constexpr int oRaw = oA + kStages * kTileBytes;
  static constexpr int oQ = oRaw + kRawStages * kFp4RawBytes;
  static constexpr int oTab = oQ + 2 * kQBytes;
  static constexpr int oHand = oTab + (FP4 ? 256 * 16 : 0);  // [2 slots][2 warps][TK][32]
  static constexpr int oBar = oHand + 2 * 2 * TK * kLanes * 8;
  static constexpr int kBars = 2 * kStages + 2 * kRawStages + 2 * kAccBufs + 4 + 4 + 1;
  static constexpr int oMisc = oBar + kBars * 8;
  static constexpr int kSmem = oMisc + 64 + 1024;
  static_assert(oQ % 1024 == 0, "Q tile must be 1024-byte aligned");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

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
// 6 gave high-batch 171 -> 163 us and kept spec-decode at its faster 60.6 us;
// larger values lose again.
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
__device__ void partition(const DecodeArgs& a, Misc* m, int lane) {
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

// Writes request `req`'s query rows (row n = query j, head h with
// n = j*heads + h) into a K-major 128-byte-swizzled tile of MQ rows.  Rows
// past heads*query_len are left as they are: their accumulator lanes are
// never read.
template <int MQ>
__device__ void load_q_tile(const DecodeArgs& a, int req, uint8_t* dst, int lane) {
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

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}


// Row max of one 128-column accumulator row (this lane's TMEM lane), with the
// columns past `lim` left out when lim < 127.
__device__ __forceinline__ float acc_row_max(uint32_t taddr, int lim) {
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int c0 = 0; c0 < kAccCols; c0 += 64) {
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

// ----------------------------------------------------------- NVFP4 dequant

// Per-scale-byte magnitude table: for scale byte s, the bf16 bits of
// e4m3_rn_satfinite(m * e4m3(s)) for the eight e2m1 magnitudes
// m = 0, .5, 1, 1.5, 2, 3, 4, 6, split into low bytes (words 0-1) and high
// bytes (words 2-3) for byte-permute lookups.
__device__ void build_fp4_table(uint4* tab, int tid, int nthreads) {
  const float mags[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  for (int s = tid; s < 256; s += nthreads) {
    const __half_raw sh = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(s), __NV_E4M3);
    const float sv = __half2float(__half(sh));
    uint32_t lo[2] = {0u, 0u}, hi[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const __nv_fp8_storage_t e =
          __nv_cvt_float_to_fp8(mags[k] * sv, __NV_SATFINITE, __NV_E4M3);
      const __half_raw eh = __nv_cvt_fp8_to_halfraw(e, __NV_E4M3);
      const float ev = __half2float(__half(eh));
      const uint32_t bits = __float_as_uint(ev) >> 16;  // exact: <= 4 significant bits
      lo[k >> 2] |= (bits & 0xFFu) << ((k & 3) * 8);
      hi[k >> 2] |= ((bits >> 8) & 0xFFu) << ((k & 3) * 8);
    }
    tab[s] = make_uint4(lo[0], lo[1], hi[0], hi[1]);
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Eight e2m1 codes (nibble k = element k, sign in bit 3) -> four bf16x2 words.
__device__ __forceinline__ void dequant8(uint32_t codes, const uint4& t, uint32_t (&o)[4]) {
  const uint32_t sel0 = codes & 0x7777u;
  const uint32_t sel1 = (codes >> 16) & 0x7777u;
  const uint32_t lo0 = prmt(t.x, t.y, sel0), hi0 = prmt(t.z, t.w, sel0);
  const uint32_t lo1 = prmt(t.x, t.y, sel1), hi1 = prmt(t.z, t.w, sel1);
  const uint32_t sa = (codes << 4) & 0x80808080u;  // signs of elements 0, 2, 4, 6
  const uint32_t sb = codes & 0x80808080u;         // signs of elements 1, 3, 5, 7
  const uint32_t h0 = hi0 ^ prmt(sa, sb, 0x5140u);
  const uint32_t h1 = hi1 ^ prmt(sa, sb, 0x7362u);
  o[0] = prmt(lo0, h0, 0x5140u);
  o[1] = prmt(lo0, h0, 0x7362u);
  o[2] = prmt(lo1, h1, 0x5140u);
  o[3] = prmt(lo1, h1, 0x7362u);
}

// ------------------------------------------------------------------ kernel

template <bool FP4, int MQ, int TK>
__global__ void __launch_bounds__(Cfg<FP4, MQ, TK>::kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const DecodeArgs a) {
  using C = Cfg<FP4, MQ, TK>;
  constexpr int S = C::kStages;
  constexpr int RS = C::kRawStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sA = sm + C::oA;
  uint8_t* sRaw = sm + C::oRaw;
  uint8_t* sQ = sm + C::oQ;
  uint4* sTab = reinterpret_cast<uint4*>(sm + C::oTab);
  uint64_t* sHand = reinterpret_cast<uint64_t*>(sm + C::oHand);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::oBar);
  uint64_t* empty = full + S;
  uint64_t* raw_full = empty + S;
  uint64_t* raw_empty = raw_full + RS;
  uint64_t* acc_full = raw_empty + RS;
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
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], FP4 ? C::kDeqWarps : 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < RS; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], C::kDeqWarps);
    }
    for (int s = 0; s < kAccBufs; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 1);
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
  if constexpr (FP4) build_fp4_table(sTab, threadIdx.x, C::kThreads);
  // Launched as a programmatic dependent launch: everything above overlaps
  // the previous kernel on the stream, whose results (lengths, tables,
  // queries, pages) are read only after this wait.  The next kernel may be
  // scheduled as soon as this grid's CTAs make room.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kProdWarp) {
    if (!FP4 && lane == 0) prefetch_tensormap(&kmap);
    partition(a, misc, lane);
  } else if (warp == kMergeWarp) {
    // While the producer reads the lengths: pull the block table and the
    // queries into L2, one 128-byte line per lane of this warp in every CTA
    // (all of both for the named batches), so that the first table and
    // query reads after the partition do not go to HBM.
    const int64_t line = (static_cast<int64_t>(blockIdx.x) * 32 + lane) * 128;
    const int64_t tbytes = static_cast<int64_t>(a.num_reqs) * a.table_stride * 4;
    const int64_t qbytes = static_cast<int64_t>(a.num_reqs) * a.query_len * a.q_tok * 2;
    if (line < tbytes)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint8_t*>(a.table) + line));
    if (line < qbytes)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint8_t*>(a.q) + line));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc->tmem;
  const long long total = misc->total;
  Walker walker{misc->i0, misc->il, misc->p0, misc->pl, misc->lo, misc->hi};

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
      // The query tile is written just before the first wait that could
      // block (stages are only freed by MMAs, which need the tile), so page
      // loads into free stages are already in flight meanwhile.
      bool q_pending = true;
      auto put_q = [&]() {
        load_q_tile<MQ>(a, req, sQ + slot * C::kQBytes, lane);
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
          if constexpr (!FP4) {
            const uint32_t st = it % S, rnd = it / S;
            if (rnd > 0 && q_pending) put_q();
            if (rnd > 0) ok = warp_wait(&empty[st], (rnd - 1) & 1, abort_flag);
            if (!ok) break;
            if (lane == 0) {
              if (good) {
                mbar_arrive_expect_tx(&full[st], kTileBytes);
                tma_load_2d(sA + st * kTileBytes, &kmap, &full[st], 0, page * kBlock, pol);
                tma_load_2d(sA + st * kTileBytes + kTileBytes / 2, &kmap, &full[st], 64,
                            page * kBlock, pol);
              } else {
                atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
                mbar_arrive(&full[st]);
              }
            }
          } else {
            const uint32_t st = it % RS, rnd = it / RS;
            if (rnd > 0 && q_pending) put_q();
            if (rnd > 0) ok = warp_wait(&raw_empty[st], (rnd - 1) & 1, abort_flag);
            if (!ok) break;
            if (lane == 0) {
              if (good) {
                uint8_t* dst = sRaw + st * kFp4RawBytes;
                mbar_arrive_expect_tx(&raw_full[st], kFp4RawBytes);
                bulk_load(dst, a.codes + static_cast<int64_t>(page) * kFp4CodeBytes,
                          kFp4CodeBytes, &raw_full[st], pol);
                bulk_load(dst + kFp4CodeBytes,
                          a.scales + static_cast<int64_t>(page) * kFp4ScaleBytes,
                          kFp4ScaleBytes, &raw_full[st], pol);
              } else {
                atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
                mbar_arrive(&raw_full[st]);
              }
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
      constexpr int ring = FP4 ? RS : S;
      uint64_t* ring_full = FP4 ? raw_full : full;
      const uint32_t pending = it < static_cast<uint32_t>(ring) ? it : ring;
      for (uint32_t k = 0; k < pending; ++k) {
        const uint32_t idx = it - 1 - k;
        int dummy = 0;
        mbar_wait(&ring_full[idx % ring], (idx / ring) & 1, &dummy);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(MQ, kAccCols);
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
          const uint32_t st = it % S, rnd = it / S;
          ok = mbar_wait(&full[st], rnd & 1, abort_flag);
          if (!ok) break;
          const uint32_t ab = it % kAccBufs, ar = it / kAccBufs;
          if (ar > 0) ok = mbar_wait(&acc_empty[ab], (ar - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kaddr = smem_u32(sA + st * kTileBytes);
          const uint32_t d = tmem_base + ab * kAccCols;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ad = sdesc_kmajor_sw128(qaddr + (k >> 2) * (MQ * 128) + (k & 3) * 32);
            const uint64_t bd =
                sdesc_kmajor_sw128(kaddr + (k >> 2) * (kTileBytes / 2) + (k & 3) * 32);
            mma_bf16(d, ad, bd, idesc, k > 0 ? 1u : 0u);
          }
          mma_commit(&empty[st]);
          mma_commit(&acc_full[ab]);
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
  } else if (warp == kEpiA || warp == kEpiB) {
    // ------------------------------------------------------------- epilogue
    const int e = warp == kEpiA ? 0 : 1;
    const int n = lane;  // query row (TMEM lane)
    const int R = a.rows_per_req;
    const int my_j = n < R ? n / a.heads : 0;
    const int my_h = n < R ? n - my_j * a.heads : 0;
    const bool select = a.mode == kModeSelect;
    RegList<TK> list;
    uint32_t it = 0;
    int seg = 0;
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      const int seq = req_len(a, req);
      const int pos = seq - a.query_len + my_j;
      const int c = pos >= 0 ? (pos >> 7) : -1;
      const int64_t row = static_cast<int64_t>(req) * a.query_len + my_j;
      const int32_t* trow = a.table + static_cast<int64_t>(req) * a.table_stride;
      list.clear();
      for (int b = b0; b < b1; ++b, ++it) {
        if ((it & 1u) != static_cast<uint32_t>(e)) continue;
        const int page = __ldg(trow + b);
        const uint32_t ab = it % kAccBufs, ar = it / kAccBufs;
        if (!warp_wait(&acc_full[ab], ar & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float m = acc_row_max(tmem_base + ab * kAccCols, pos - b * kBlock);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
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
        // Hand this request's lists to the merge warp and keep streaming.
        const int hs = seg & 1;
        if (seg >= 2 && !warp_wait(&h_empty[hs], ((seg >> 1) - 1) & 1, abort_flag)) break;
        if (n < R) list.store_cols(sHand + (hs * 2 + e) * TK * kLanes, n);
        __syncwarp();
        if (lane == 0) mbar_arrive(&h_full[hs]);
      } else if (e == 0 && b1 == nb && a.fill_width > nb) {
        const int w = a.fill_width - nb;
        for (int idx = lane; idx < R * w; idx += 32) {
          const int rr = idx / w, bb = nb + (idx - rr * w);
          const int j = rr / a.heads, h = rr - j * a.heads;
          a.score[h * a.s_head + (static_cast<int64_t>(req) * a.query_len + j) * a.s_row + bb] =
              -INFINITY;
        }
      }
      ++seg;
    }
  } else if (warp == kMergeWarp) {
    // ------------------------------------------------------------ merge warp
    // Per request (in the walker's order): fold the two epilogue warps'
    // lists row by row (lane n owns row n).  A request held by one CTA is
    // written here; a split request goes through the partial slots and its
    // tickets.  With total >= grid every share is non-empty, so the
    // request's CTAs are first..last; with fewer blocks than CTAs every
    // non-empty share is a single block, so block k sits in cta_of(preq + k).
    const int n = lane;
    const int R = a.rows_per_req;
    const bool select = a.mode == kModeSelect;
    int seg = 0;
    bool ok = true;
    while (select && ok && walker.next(a, req, b0, b1, nb, preq)) {
      const int hs = seg & 1;
      if (!warp_wait(&h_full[hs], (seg >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      uint64_t* H0 = sHand + (hs * 2 + 0) * TK * kLanes;
      const uint64_t* H1 = sHand + (hs * 2 + 1) * TK * kLanes;
      RegList<TK> list;
      list.clear();
      if (n < R) {
        uint64_t other[TK];
#pragma unroll
        for (int k = 0; k < TK; ++k) {
          list.v[k] = H0[k * kLanes + n];
          other[k] = H1[k * kLanes + n];
        }
        list.merge_sorted(other);
      }
      const int first = cta_of(preq, total, gridDim.x);
      const int last = cta_of(preq + nb - 1, total, gridDim.x);
      const bool dense = total >= gridDim.x;
      const int nseg = dense ? last - first + 1 : nb;
      const int j = n < R ? n / a.heads : 0, h = n < R ? n - j * a.heads : 0;
      const int pr = req_len(a, req) - a.query_len + j;
      const int cr = pr >= 0 ? (pr >> 7) : -1;
      int32_t* out = a.ids + h * a.i_head + (static_cast<int64_t>(req) * a.query_len + j) * a.i_row;
      if (nseg == 1) {
        // Lane n writes row n: forced blocks, the best picks in ascending id
        // order (a sorting network over the TK candidate ids), then -1.
        if (n < R) write_row_lane<TK>(list.v, cr, a.init_blocks, a.local_blocks, a.topk, out);
      } else {
        // Split request: publish this CTA's lists, then take a ticket.  The
        // last of the request's CTAs to arrive folds every other CTA's lists
        // into its own and writes the rows.  Split requests are the first
        // ones each CTA streams (see Walker), so this overlaps the rest of
        // the stream.  The ticket wraps to zero on the last arrival, ready
        // for the next call.
        const int64_t slot_stride = static_cast<int64_t>(kLanes) * TK;
        if (n < R) {
          ulonglong2* dst = reinterpret_cast<ulonglong2*>(
              a.partials + (static_cast<int64_t>(blockIdx.x) + req) * slot_stride + n * TK);
#pragma unroll
          for (int k = 0; k < TK; k += 2) dst[k / 2] = make_ulonglong2(list.v[k], list.v[k + 1]);
        }
        // The warp barrier orders the lanes' list stores before lane 0's
        // release; lane 0's acquire, then the barrier, orders the merging
        // lanes' reads after every other CTA's release.  (Full fences
        // around a plain atomicInc measured 1-2 us slower.)
        __syncwarp();
        unsigned int ticket = 0;
        if (lane == 0)
          ticket = atomic_inc_acq_rel_gpu(a.tickets + req, static_cast<unsigned int>(nseg - 1));
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        __syncwarp();
        if (ticket == static_cast<unsigned int>(nseg - 1)) {
          if (n < R) {
            for (int js = 0; js < nseg; ++js) {
              const int cj = dense ? first + js : cta_of(preq + js, total, gridDim.x);
              if (cj == static_cast<int>(blockIdx.x)) continue;
              const ulonglong2* src = reinterpret_cast<const ulonglong2*>(
                  a.partials + (static_cast<int64_t>(cj) + req) * slot_stride + n * TK);
              uint64_t other[TK];
#pragma unroll
              for (int u = 0; u < TK / 2; ++u) {
                const ulonglong2 x = __ldcg(src + u);
                other[2 * u] = x.x;
                other[2 * u + 1] = x.y;
              }
              list.merge_sorted(other);
            }
            write_row_lane<TK>(list.v, cr, a.init_blocks, a.local_blocks, a.topk, out);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&h_empty[hs]);
      ++seg;
    }
    if (ok) {
      // Requests with no blocks at all appear in no share: spread them over CTAs.
      for (int i = blockIdx.x; i < a.num_reqs; i += gridDim.x) {
        if (req_blocks(a, i) != 0) continue;
        if (!select) {
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
  } else if constexpr (FP4) {
    // ---------------------------------------------------- NVFP4 dequantiser
    if (warp >= kDeqWarp0) {  // warp 3 has no role
      constexpr int kDqThreads = C::kDeqWarps * 32;
      const int dq = threadIdx.x - kDeqWarp0 * 32;  // 0..kDqThreads-1
      // A page is 1024 groups of 16 elements (128 tokens x 8).  Item
      // dq + kDqThreads*kk is token tok0 + kT*kk, scale group g.
      constexpr int kT = kDqThreads / 8, kItems = 1024 / kDqThreads;
      const int g = dq & 7, tok0 = dq >> 3, sw = tok0 & 7;
      const uint32_t row_off = (g >> 2) * (kTileBytes / 2) + (tok0 >> 3) * 1024 + sw * 128;
      // The group's two 16-byte chunks (elements 0-7 and 8-15).  Groups g and
      // g+4 of a token share their chunk positions in the two 64-column
      // halves, i.e. the same banks; groups g >= 4 store their chunks in the
      // opposite order so that each store instruction hits eight distinct
      // chunk positions per eight lanes.
      const bool swap = g >= 4;
      const uint32_t off_lo = row_off + ((((g & 3) * 2) ^ sw) << 4);
      const uint32_t off_hi = row_off + ((((g & 3) * 2 + 1) ^ sw) << 4);
      const uint32_t st_offA = swap ? off_hi : off_lo, st_offB = swap ? off_lo : off_hi;
      uint32_t it = 0;
      bool ok = true;
      while (ok && walker.next(a, req, b0, b1, nb, preq)) {
        for (int b = b0; b < b1; ++b) {
          const uint32_t rs = it % RS, rr = it / RS;
          const uint32_t st = it % S, sr = it / S;
          bool got = true;
          if (lane == 0) {
            got = mbar_wait(&raw_full[rs], rr & 1, abort_flag);
            if (got && sr > 0) got = mbar_wait(&empty[st], (sr - 1) & 1, abort_flag);
          }
          if (!__shfl_sync(0xffffffffu, got, 0)) {
            ok = false;
            break;
          }
          const uint8_t* codes = sRaw + rs * kFp4RawBytes;
          const uint8_t* scales = codes + kFp4CodeBytes;
          uint8_t* tile = sA + st * kTileBytes;
          // Thread dq covers group g of tokens tok0 + kT*kk.  All loads are
          // issued before any arithmetic so that the independent groups
          // overlap their latencies.
          uint2 cw[kItems];
          uint32_t sc[kItems];
#pragma unroll
          for (int kk = 0; kk < kItems; ++kk) {
            cw[kk] = *reinterpret_cast<const uint2*>(codes + kk * kT * 64 + dq * 8);
            sc[kk] = scales[kk * kT * 8 + dq];
          }
          uint4 t[kItems];
#pragma unroll
          for (int kk = 0; kk < kItems; ++kk) t[kk] = sTab[sc[kk]];
#pragma unroll
          for (int kk = 0; kk < kItems; ++kk) {
            uint32_t o0[4], o1[4];
            dequant8(swap ? cw[kk].y : cw[kk].x, t[kk], o0);
            dequant8(swap ? cw[kk].x : cw[kk].y, t[kk], o1);
            uint8_t* rowp = tile + kk * kT * 128;
            *reinterpret_cast<uint4*>(rowp + st_offA) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
            *reinterpret_cast<uint4*>(rowp + st_offB) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&full[st]);
            mbar_arrive(&raw_empty[rs]);
          }
          ++it;
        }
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

template <bool FP4, int MQ, int TK>
cudaError_t launch_t(const CUtensorMap& kmap, const DecodeArgs& a, int grid, cudaStream_t s) {
  using C = Cfg<FP4, MQ, TK>;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<FP4, MQ, TK>,
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
  return cudaLaunchKernelEx(&cfg, decode_kernel<FP4, MQ, TK>, kmap, a);
}

template <bool FP4>
cudaError_t dispatch(const CUtensorMap& kmap, const DecodeArgs& a, int grid, cudaStream_t s) {
  const bool small = a.rows_per_req <= 16, tk16 = decode_tk(a.topk) == 16;
  if (small && tk16) return launch_t<FP4, 64, 16>(kmap, a, grid, s);
  if (small) return launch_t<FP4, 64, 32>(kmap, a, grid, s);
  if (tk16) return launch_t<FP4, 128, 16>(kmap, a, grid, s);
  return launch_t<FP4, 128, 32>(kmap, a, grid, s);
}

}  // namespace

int decode_ctas_per_sm() { return 1; }

cudaError_t launch_decode_bf16(const CUtensorMap& kmap, const DecodeArgs& a, int grid, cudaStream_t s) {
  return dispatch<false>(kmap, a, grid, s);
}

cudaError_t launch_decode_nvfp4(const DecodeArgs& a, int grid, cudaStream_t s) {
  CUtensorMap unused{};
  return dispatch<true>(unused, a, grid, s);
}

}  // namespace mm3idx
