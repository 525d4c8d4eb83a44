// wordlane.cuh - bit helpers of the per-lane decoders: select of the r-th '1'
// of a word (two popcount halvings and a byte-select table), trailing zeros,
// and shifts with PTX semantics. The lane-per-mask-word draft GEMV (gemv.cu)
// and the block walks (blockwalk.cuh) use them.
#pragma once
#include "common.cuh"

namespace cas {

// sel8[b*8 + i] = MSB-first bit index of the (i+1)-th '1' of byte b (0 when b
// has fewer ones), built at compile time.
struct Sel8Table {
  uint8_t v[2048];
};
constexpr Sel8Table make_sel8() {
  Sel8Table t{};
  for (int b = 0; b < 256; ++b) {
    int seen = 0;
    for (int q = 7; q >= 0; --q)
      if ((b >> q) & 1) t.v[b * 8 + seen++] = (uint8_t)(7 - q);
  }
  return t;
}
__device__ const Sel8Table g_sel8 = make_sel8();

// trailing zeros (32 for 0)
__device__ __forceinline__ int tzcnt(uint32_t w) { return w ? 31 - __clz(w & (0u - w)) : 32; }

// Bit index, counted from the MSB, of the r-th '1' (1-based) of w: two
// popcount halvings, then the byte-select table.
__device__ __forceinline__ int select_msb(uint32_t w, int r) {
  const uint32_t hi = w >> 16;
  const int c1 = __popc(hi);
  const bool h = r <= c1;
  const uint32_t w16 = h ? hi : (w & 0xFFFFu);
  r = h ? r : r - c1;
  const uint32_t hb = w16 >> 8;
  const int c2 = __popc(hb);
  const bool hh = r <= c2;
  const uint32_t b = hh ? hb : (w16 & 0xFFu);
  r = hh ? r : r - c2;
  const int base = (h ? 0 : 16) + (hh ? 0 : 8);
  return base + __ldg(g_sel8.v + b * 8 + ((r - 1) & 7));
}

// Shifts with PTX semantics: shl clamps amounts of 32 or more (result 0);
// shf.l.wrap takes the amount modulo 32.
__device__ __forceinline__ uint32_t shl32(uint32_t x, uint32_t n) {
  uint32_t d;
  asm("shl.b32 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(n));
  return d;
}
__device__ __forceinline__ uint32_t shr32(uint32_t x, uint32_t n) {
  uint32_t d;
  asm("shr.b32 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(n));
  return d;
}
__device__ __forceinline__ uint32_t shfl_wrap(uint32_t lo, uint32_t hi, uint32_t n) {
  uint32_t d;
  asm("shf.l.wrap.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(lo), "r"(hi), "r"(n));
  return d;
}
__device__ __forceinline__ uint32_t mad32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

}  // namespace cas
