// decode_fp4.cu -- persistent, warp-specialised decode kernel over NVFP4
// index-K pages: causal block scoring of a few query rows per request, with
// the fp32 scores written out (score mode) or a fused top-k selector (select
// mode).  Each key element is e4m3_rn_satfinite(e2m1 code * e4m3 scale), one
// scale per 16 elements (vLLM MiniMax-M3 "indexer_nvfp4" page, module
// docstring); every such value is exact in bf16, and the products with the
// bf16 query rows are exact in the fp32 accumulators, as in the bf16 kernel
// (decode.cu).  The partition, walker and merge are decode_common.cuh's.
//
// Why not tcgen05 here: its B operand (or A) must sit in shared memory, so a
// page's 32 KB of dequantised bf16 is written to and read back from shared
// memory -- with the TMA copy and the code reads, about 100 KB of
// shared-memory traffic per 9 KB page from HBM, which bounds the kernel near
// half of the HBM rate.  With a handful of query rows the contraction itself
// is small (rows x 128 x 128 per page), so the dequantised keys instead go
// straight from registers into warp-level mma.sync (m16n8k16, bf16 in, fp32
// accumulate): keys as A (16 tokens x 16 dims), the query rows as B
// (16 dims x 8 rows, up to four row tiles), held in registers per request.
// The 128 dims of a product are taken in an order (the same for keys and
// queries) that gives each thread one 16-byte run of a token's codes and two
// of its scales.
//
//   * warp 1   : producer.  Per page, bulk copies of the 8 KB of codes and
//                the 1 KB of scales into a ring of raw stages, the pages
//                further ahead pulled into L2 first.
//   * warps 2-11: compute.  Warp w takes pages w, w+10, ... of the CTA's
//                stream: eight slabs of 16 tokens, each eight mma.sync per
//                row tile over the dequantised codes, then the causal row
//                max of the block (masked only in a request's last blocks),
//                written to the stage's score slot.
//   * warp 0   : selector.  Takes the score slots in page order, scales them
//                (a block with an out-of-range page gets -inf), offers them
//                to its rows' candidate lists (lane n = row n) or writes the
//                scores, frees the stage, and at the end of each request
//                writes or merges the rows (merge_request).
//
// Every wait is bounded (ptx.cuh); a wait that gives up raises the CTA's
// abort flag and MM3IDX_DEV_TIMEOUT.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "decode_common.cuh"
#include "nvfp4.cuh"

namespace mm3idx {
namespace {

using namespace dec;

constexpr int kCodeBytes = kBlock * kD / 2;    // 8 KB: 128 tokens x 64 B
constexpr int kScaleBytes = kBlock * kD / 16;  // 1 KB: 128 tokens x 8 B
constexpr int kStageBytes = kCodeBytes + kScaleBytes;
constexpr int kSelWarp = 0, kProdWarp = 1, kCompWarp0 = 2;
// Compute warps: ten, so that the block's twelve warps are three per SM
// sub-partition and keep the 168-register cap.  Measured on the 128-request
// NVFP4 batch: eight 0.304 ms, ten 0.290 ms, twelve (fourteen warps, a
// 128-register cap) 0.328 ms.  Pages go round-robin; dealing more of them to
// the warps on the two sub-partitions that also hold the selector and the
// producer (a quarter of the pages per sub-partition) measured 0.305 ms: the
// selector takes pages in order and waits on the warps given more.
template <int NT>
constexpr int comp_warps() { return 10; }
template <int NT>
constexpr int threads_of() { return (kCompWarp0 + comp_warps<NT>()) * 32; }
constexpr int kAhead = 16;                     // pages pulled into L2 ahead of the ring (< 32)
constexpr int kStages = 18;                    // raw ring depth (pages)
constexpr int kTabCopies = 8;                  // lane & 7 picks a copy: a quarter-warp's lookups hit distinct banks

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

// Shared memory: the raw ring (codes then scales per stage), the magnitude
// table, the score slots (32 rows per stage), the selector's lists for its
// merges, the barriers.
template <int TK>
struct Cfg {
  static constexpr int oRaw = 0;
  static constexpr int oTab = oRaw + kStages * kStageBytes;       // [256 scales][copies] x 16 B
  static constexpr int oScore = oTab + 256 * kTabCopies * 16;      // [stages][32] fp32
  static constexpr int oList = oScore + kStages * kLanes * 4;      // [TK][32] keys
  static constexpr int oBar = oList + TK * kLanes * 8;
  static constexpr int kBars = 3 * kStages;
  static constexpr int oMisc = oBar + kBars * 8;
  static constexpr int kSmem = oMisc + 64 + 128;
  static_assert(kStageBytes % 128 == 0 && oTab % 128 == 0 && oBar % 8 == 0, "alignment");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// D += A * B on the legacy warp-level tensor path: A 16x16 bf16 (row), B
// 16x8 bf16 (col), D 16x8 fp32, fragments in registers.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ------------------------------------------------------------------ kernel
//
// Fragment layout (thread t of a warp, j = t & 3, g = t >> 2): in k-step ks
// (0..7) of slab sl the thread's A registers are tokens 16*sl + g and +8,
// dims 32j + 4ks + {0,1} (a0, a1) and 32j + 4ks + {2,3} (a2, a3) -- bytes
// 16j + 2ks and 16j + 2ks + 1 of the token's codes, so its k-steps walk one
// 16-byte run, and scale groups 2j (k-steps 0-3) and 2j+1 (4-7); its B
// registers are query row 8*nt + g, the same dims.  D: rows = tokens
// 16*sl + g (c0, c1) and +8 (c2, c3), columns = query rows 8*nt + 2j, +1.
template <int TK, int NT>
__global__ void __launch_bounds__(threads_of<NT>(), 1) decode_fp4_kernel(const DecodeArgs a) {
  using C = Cfg<TK>;
  constexpr int S = kStages, NC = kTabCopies;
  constexpr int kCompWarps = comp_warps<NT>(), kThreads = threads_of<NT>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                           ~static_cast<uintptr_t>(127));
  uint8_t* sRaw = sm + C::oRaw;
  const uint4* sTab = reinterpret_cast<const uint4*>(sm + C::oTab);
  float* sScore = reinterpret_cast<float*>(sm + C::oScore);
  uint64_t* sList = reinterpret_cast<uint64_t*>(sm + C::oList);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::oBar);   // the copies landed
  uint64_t* done = full + S;                                     // the stage's scores are written
  uint64_t* empty = done + S;                                    // the selector is done with the stage
  Misc* misc = reinterpret_cast<Misc*>(sm + C::oMisc);
  volatile int* abort_flag = &misc->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&done[s], 1);
      mbar_init(&empty[s], 1);
    }
    misc->abort = 0;
    fence_barrier_init();
  }
  build_fp4_table(reinterpret_cast<uint4*>(sm + C::oTab), NC, threadIdx.x, kThreads);
  // Programmatic dependent launch: the set-up above overlaps the previous
  // kernel on the stream; its results are read only after this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kProdWarp) {
    partition(a, misc, lane);
  } else if (warp == kSelWarp) {
    prefetch_table_and_queries(a, lane);
  }
  __syncthreads();
  const long long total = misc->total;
  Walker walker = make_walker(misc);

  int req, b0, b1, nb;
  long long preq;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    uint32_t it = 0;  // pages issued
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
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
          const uint32_t st = it % S, rnd = it / S;
          if (rnd > 0) ok = warp_wait(&empty[st], (rnd - 1) & 1, abort_flag);
          if (!ok) break;
          if (lane == 0) {
            if (good) {
              uint8_t* dst = sRaw + st * kStageBytes;
              mbar_arrive_expect_tx(&full[st], kStageBytes);
              bulk_load(dst, a.codes + static_cast<int64_t>(page) * kCodeBytes, kCodeBytes,
                        &full[st], pol);
              bulk_load(dst + kCodeBytes, a.scales + static_cast<int64_t>(page) * kScaleBytes,
                        kScaleBytes, &full[st], pol);
            } else {
              // Not loaded: the stage's stale bytes are scored, and the
              // selector gives the block -inf.
              atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
              mbar_arrive(&full[st]);
            }
          }
          __syncwarp();
          ++it;
        }
      }
    }
    // Let every copy this warp started land before the CTA can exit.
    if (lane == 0) {
      const uint32_t pending = it < static_cast<uint32_t>(S) ? it : S;
      for (uint32_t k = 0; k < pending; ++k) {
        const uint32_t idx = it - 1 - k;
        int dummy = 0;
        mbar_wait(&full[idx % S], (idx / S) & 1, &dummy);
      }
    }
    __syncwarp();
  } else if (warp >= kCompWarp0) {
    // -------------------------------------------------------------- compute
    const int w = warp - kCompWarp0;
    const int j = lane & 3, g = lane >> 2;
    const int R = a.rows_per_req;
    const int copy = lane & (NC - 1);
    uint32_t pi = 0;  // pages of the stream so far
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      const uint32_t nseg = static_cast<uint32_t>(b1 - b0);
      // This warp's first page of the segment.
      const uint32_t first = (static_cast<uint32_t>(w) + kCompWarps - pi % kCompWarps) % kCompWarps;
      if (first < nseg) {
        // The request's query rows as B fragments: row 8*nt + g, dims
        // 32j .. 32j+31 (word 2ks: dims 32j+4ks, +1; word 2ks+1: +2, +3).
        uint32_t bq[NT][16];
        const int seq = req_len(a, req);
        int lim0[NT][2];  // pos - 0 for the D columns (query rows 8*nt + 2j + e) of this lane
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int n = nt * 8 + g;
          if (n < R) {
            const int jj = n / a.heads, h = n - jj * a.heads;
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + (static_cast<int64_t>(req) * a.query_len + jj) * a.q_tok +
                static_cast<int64_t>(h) * a.q_head + 32 * j);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 x = __ldg(src + v);
              bq[nt][4 * v] = x.x;
              bq[nt][4 * v + 1] = x.y;
              bq[nt][4 * v + 2] = x.z;
              bq[nt][4 * v + 3] = x.w;
            }
          } else {
#pragma unroll
            for (int v = 0; v < 16; ++v) bq[nt][v] = 0u;
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = nt * 8 + 2 * j + e;
            lim0[nt][e] = col < R ? seq - a.query_len + col / a.heads : 1 << 30;
          }
        }
        for (uint32_t k = first; k < nseg; k += kCompWarps) {
          const uint32_t p = pi + k;
          const uint32_t st = p % S, rnd = p / S;
          const int b = b0 + static_cast<int>(k);
          if (!warp_wait(&full[st], rnd & 1, abort_flag)) {
            ok = false;
            break;
          }
          // Every lane observes the completed phase itself before reading
          // what the copies wrote.
          mbar_try_wait(&full[st], rnd & 1);
          const uint8_t* raw = sRaw + st * kStageBytes;
          int lim[NT][2];
          bool masked = false;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              lim[nt][e] = lim0[nt][e] - b * kBlock;
              masked |= lim[nt][e] < kBlock - 1;
            }
          masked = __any_sync(0xffffffffu, masked);
          float m[NT][2];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) m[nt][0] = m[nt][1] = -INFINITY;
#pragma unroll 1   // unrolled by 2: 0.307 ms, fully: 0.325 ms (instruction fetch)
          for (int sl = 0; sl < 8; ++sl) {
            const int r0 = sl * 16 + g, r1 = r0 + 8;
            const uint4 ca = *reinterpret_cast<const uint4*>(raw + r0 * 64 + 16 * j);
            const uint4 cb = *reinterpret_cast<const uint4*>(raw + r1 * 64 + 16 * j);
            const uint32_t sa = *reinterpret_cast<const uint16_t*>(raw + kCodeBytes + r0 * 8 + 2 * j);
            const uint32_t sb = *reinterpret_cast<const uint16_t*>(raw + kCodeBytes + r1 * 8 + 2 * j);
            const uint4 ta0 = sTab[(sa & 0xFFu) * NC + copy], ta1 = sTab[(sa >> 8) * NC + copy];
            const uint4 tb0 = sTab[(sb & 0xFFu) * NC + copy], tb1 = sTab[(sb >> 8) * NC + copy];
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
            for (int qw = 0; qw < 4; ++qw) {
              const uint32_t wa = qw == 0 ? ca.x : qw == 1 ? ca.y : qw == 2 ? ca.z : ca.w;
              const uint32_t wb = qw == 0 ? cb.x : qw == 1 ? cb.y : qw == 2 ? cb.z : cb.w;
              const uint4 da = dequant8(wa, qw < 2 ? ta0 : ta1);
              const uint4 db = dequant8(wb, qw < 2 ? tb0 : tb1);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                mma_16816(acc[nt], da.x, db.x, da.y, db.y, bq[nt][4 * qw], bq[nt][4 * qw + 1]);
                mma_16816(acc[nt], da.z, db.z, da.w, db.w, bq[nt][4 * qw + 2], bq[nt][4 * qw + 3]);
              }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (masked) {
                // Columns (query rows) see tokens 0..lim of the block.
                acc[nt][0] = r0 <= lim[nt][0] ? acc[nt][0] : -INFINITY;
                acc[nt][1] = r0 <= lim[nt][1] ? acc[nt][1] : -INFINITY;
                acc[nt][2] = r1 <= lim[nt][0] ? acc[nt][2] : -INFINITY;
                acc[nt][3] = r1 <= lim[nt][1] ? acc[nt][3] : -INFINITY;
              }
              m[nt][0] = fmax3(m[nt][0], acc[nt][0], acc[nt][2]);
              m[nt][1] = fmax3(m[nt][1], acc[nt][1], acc[nt][3]);
            }
          }
          // Max over the block's tokens: the eight lanes of each j.
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float v = m[nt][e];
              v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
              v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
              v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
              m[nt][e] = v;
            }
          if (lane < 4) {
            float* slot = sScore + st * kLanes;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              slot[nt * 8 + 2 * lane] = m[nt][0];
              slot[nt * 8 + 2 * lane + 1] = m[nt][1];
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&done[st]);
        }
      }
      pi += nseg;
    }
  } else if (warp == kSelWarp) {
    // ------------------------------------------------------------- selector
    const int n = lane;                   // query row
    const int R = a.rows_per_req;
    const int my_j = n < R ? n / a.heads : 0;
    const int my_h = n < R ? n - my_j * a.heads : 0;
    const bool select = a.mode == kModeSelect;
    // Requests with no blocks first, then dry runs of both merge paths
    // (decode_common.cuh), all before the first scores are ready.
    fill_empty_requests(a, lane);
    if (select) {
      const MergeGeom none{0, 1, true};
      merge_request<TK, 1>(a, 0, 0, 1, none, 1, sList, lane, true, false);
      merge_request<TK, 1>(a, 0, 0, 1, none, 1, sList, lane, true, true);
    }
    RegList<TK> list;
    uint32_t pi = 0;
    bool ok = true;
    while (ok && walker.next(a, req, b0, b1, nb, preq)) {
      const int seq = req_len(a, req);
      const int pos = seq - a.query_len + my_j;
      const int c = pos >= 0 ? (pos >> 7) : -1;
      const int64_t row = static_cast<int64_t>(req) * a.query_len + my_j;
      const int32_t* trow = a.table + static_cast<int64_t>(req) * a.table_stride;
      const MergeGeom geo = merge_geom(nb, preq, total);
      list.clear();
      int pg = 0;  // page ids 32 at a time, one per lane
      for (int b = b0; b < b1; ++b, ++pi) {
        if (((b - b0) & 31) == 0) pg = b + lane < b1 ? __ldg(trow + b + lane) : 0;
        const int page = __shfl_sync(0xffffffffu, pg, (b - b0) & 31);
        const uint32_t st = pi % S, rnd = pi / S;
        if (!warp_wait(&done[st], rnd & 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_try_wait(&done[st], rnd & 1);   // each lane observes the phase before reading
        const float v = sScore[st * kLanes + n];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (n < R) {
          const float s = (page >= 0 && page < a.num_pages) ? v * a.sm_scale : -INFINITY;
          if (!select) {
            a.score[my_h * a.s_head + row * a.s_row + b] = s;
          } else if (b <= c && b >= a.init_blocks && b <= c - a.local_blocks) {
            list.offer(make_key(s, b));
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

  __syncthreads();
  if (threadIdx.x == 0 && misc->abort) atomicOr(a.status, MM3IDX_DEV_TIMEOUT);
}

template <int TK, int NT>
cudaError_t launch_t(const DecodeArgs& a, int grid, cudaStream_t s) {
  using C = Cfg<TK>;
  const int smem = C::kSmem;
  cudaError_t e = cudaFuncSetAttribute(decode_fp4_kernel<TK, NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads_of<NT>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_fp4_kernel<TK, NT>, a);
}

template <int TK>
cudaError_t launch_tk(const DecodeArgs& a, int grid, cudaStream_t s) {
  if (a.rows_per_req <= 8) return launch_t<TK, 1>(a, grid, s);
  if (a.rows_per_req <= 16) return launch_t<TK, 2>(a, grid, s);
  return launch_t<TK, 4>(a, grid, s);
}

}  // namespace

cudaError_t launch_decode_nvfp4(const DecodeArgs& a, int grid, cudaStream_t s) {
  if (decode_tk(a.topk) == 16) return launch_tk<16>(a, grid, s);
  return launch_tk<32>(a, grid, s);
}

}  // namespace mm3idx
