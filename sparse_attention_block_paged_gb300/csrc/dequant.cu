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
// bytes of bf16 out, all coalesced.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/mm3idx.h"
#include "internal.h"

namespace mm3idx {
namespace {

constexpr int kThreads = 256;

// e2m1 magnitudes of codes 0..7 (OCP MX FP4: 0, 0.5, 1, 1.5, 2, 3, 4, 6).
__device__ __forceinline__ float e2m1_magnitude(uint32_t m) {
  const float sub = (m & 1u) ? 0.5f : 0.0f;
  const uint32_t e = m >> 1;
  return e == 0 ? sub : static_cast<float>(1u << (e - 1)) * ((m & 1u) ? 1.5f : 1.0f);
}

// bf16 bits of e4m3_rn_satfinite(e2m1(code) * scale); the product is exact
// in fp32 and the e4m3 result is exact in fp16 and bf16.
__device__ __forceinline__ uint32_t nvfp4_bf16_bits(uint32_t code, float scale) {
  const float mag = e2m1_magnitude(code & 7u) * scale;
  const float v = (code & 8u) ? -mag : mag;
  const __nv_fp8_storage_t q = __nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
  const __half_raw h = __nv_cvt_fp8_to_halfraw(q, __NV_E4M3);
  return __float_as_uint(__half2float(__half(h))) >> 16;
}

__global__ void __launch_bounds__(kThreads) dequant_pages_kernel(const DequantArgs a) {
  const int t = threadIdx.x;
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
      const __half_raw sh = __nv_cvt_fp8_to_halfraw(
          static_cast<__nv_fp8_storage_t>((sc >> (8 * g)) & 0xffu), __NV_E4M3);
      const float s = __half2float(__half(sh));
      uint32_t o[8];
#pragma unroll
      for (int w = 0; w < 2; ++w) {  // 4 code bytes = 8 elements
        const uint32_t word = cw[2 * g + w];
#pragma unroll
        for (int by = 0; by < 4; ++by) {
          const uint32_t byte = (word >> (8 * by)) & 0xffu;
          o[4 * w + by] = nvfp4_bf16_bits(byte & 15u, s) | (nvfp4_bf16_bits(byte >> 4, s) << 16);
        }
      }
      dst[2 * g] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[2 * g + 1] = make_uint4(o[4], o[5], o[6], o[7]);
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
