// nvfp4.cuh -- NVFP4 index-K elements to bf16 with byte permutes: the
// per-scale magnitude table and the eight-element dequantisation shared by
// the NVFP4 decode kernel (decode_fp4.cu) and the dequant pass of the NVFP4
// prefill (dequant.cu).
//
// An element is e4m3_rn_satfinite(e2m1 code * e4m3 scale), one scale per 16
// consecutive elements (vLLM MiniMax-M3 "indexer_nvfp4" page, module
// docstring); every such value is exact in bf16.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace mm3idx {

// Per-scale-byte magnitude table: for scale byte s, the bf16 bits of
// e4m3_rn_satfinite(m * e4m3(s)) for the eight e2m1 magnitudes
// m = 0, .5, 1, 1.5, 2, 3, 4, 6, as low bytes (words 0-1) and high bytes
// (words 2-3) for byte-permute lookups; `copies` copies side by side.
__device__ inline void build_fp4_table(uint4* tab, int copies, int tid, int nthreads) {
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
  // prmt reads its selector from bits 0-15 only: one mask serves both halves.
  const uint32_t sel0 = codes & 0x77777777u;
  const uint32_t sel1 = sel0 >> 16;
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

}  // namespace mm3idx
