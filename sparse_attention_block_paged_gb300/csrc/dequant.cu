// dequant.cu -- NVFP4 index-K pages to bf16 pages, for the prefill scorer.
//
// An NVFP4 key element is e4m3_rn_satfinite(e2m1 code * e4m3 scale), one
// scale per 16 consecutive elements (vLLM MiniMax-M3 "indexer_nvfp4" page,
// module docstring); the result is exactly representable in bf16.  A prefill
// reads every key page once per 128-row query tile that sees it (up to 256
// times for a 32768-token request), so the pages are dequantised once here,
// into a bf16 copy laid out [request, logical block] in the caller's
// workspace, and the bf16 tensor-core scorer runs on that copy through an
// identity block table.  One CTA of 256 threads per page: thread t takes half
// a token row (64 elements): 32 bytes of codes and 4 scale bytes in, 128
// bytes of bf16 out, all coalesced.  The elements go through the per-scale
// byte-permute table of nvfp4.cuh (about two integer operations an element,
// where CUDA's fp8 conversions per element took about twenty).
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/mm3idx.h"
#include "internal.h"
#include "nvfp4.cuh"

namespace mm3idx {
namespace {

constexpr int kThreads = 256;
constexpr int kCopies = 4;   // table copies side by side (thread & 3 picks one)

__global__ void __launch_bounds__(kThreads) dequant_pages_kernel(const DequantArgs a) {
  __shared__ uint4 sTab[256 * kCopies];
  build_fp4_table(sTab, kCopies, threadIdx.x, kThreads);
  __syncthreads();
  const int t = threadIdx.x;
  const int copy = t & (kCopies - 1);
  const int tok = t >> 1, half = t & 1;
  const int64_t slots = static_cast<int64_t>(a.num_reqs) * a.width;
  for (int64_t slot = blockIdx.x; slot < slots; slot += gridDim.x) {
    const int req = static_cast<int>(slot / a.width);
    const int b = static_cast<int>(slot - static_cast<int64_t>(req) * a.width);
    const int seq = min(max(__ldg(a.seq_lens + req), 0), a.max_seq_len);
    const int page = b * kBlock < seq ? __ldg(a.table + req * a.table_stride + b) : 0;
    const bool bad = page < 0 || page >= a.num_pages;
    // A bad page's slot is marked -1 in the copy's table: the scorer then
    // scores that block as it scores a bad page of a bf16 cache (no visible
    // tokens) and sets the status bit.
    if (t == 0) a.table_out[slot] = bad ? -1 : static_cast<int32_t>(slot);
    if (b * kBlock >= seq) continue;  // never read by the scorer
    if (bad) {
      if (t == 0) atomicOr(a.status, MM3IDX_DEV_BAD_PAGE);
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(a.pages_out + slot * (kBlock * kD) + tok * kD + half * 64);
    const uint4* src = reinterpret_cast<const uint4*>(a.codes + static_cast<int64_t>(page) * (kBlock * kD / 2) +
                                                      tok * (kD / 2) + half * 32);
    const uint4 c0 = __ldg(src), c1 = __ldg(src + 1);
    const uint32_t sc = __ldg(reinterpret_cast<const uint32_t*>(
        a.scales + static_cast<int64_t>(page) * (kBlock * kD / 16) + tok * (kD / 16) + half * 4));
    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int g = 0; g < 4; ++g) {  // scale group: 16 elements, 8 code bytes
      const uint4 tb = sTab[((sc >> (8 * g)) & 0xffu) * kCopies + copy];
      dst[2 * g] = dequant8(cw[2 * g], tb);
      dst[2 * g + 1] = dequant8(cw[2 * g + 1], tb);
    }
  }
}

}  // namespace

cudaError_t launch_dequant_pages(const DequantArgs& a, int num_sms, cudaStream_t s) {
  const int64_t slots = static_cast<int64_t>(a.num_reqs) * a.width;
  int64_t grid = static_cast<int64_t>(num_sms) * 8;
  if (slots < grid) grid = slots;
  if (grid < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, dequant_pages_kernel, a);
}

}  // namespace mm3idx
