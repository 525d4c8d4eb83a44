// blockwalk.cuh - lane-per-block decoding of Cassandra-1 superblocks.
//
// A warp decodes 4 superblocks at once and lane L owns block L & 7 of
// superblock L >> 3: 128 positions, of which exactly k are kept. The warp
// stages the 4 superblocks' unary code streams in shared memory; each lane
// finds the code that starts its block - the code after the (k j)-th '1' of
// its stream (Cassandra blog review, section 3.2: a code is `rank` zeros then
// a one), j = L & 7 - by a warp popcount scan over the staged words and a
// shuffle search, and then walks its block with two 64-bit windows of its own:
// one over the bit-reversed mask (positions), one over the stream (codes).
// A window step shifts by one more than the count of leading zeros; a step of
// 32 or more (a gap of 32 or more positions, a code of rank 31 or more, a
// window that ran dry) is the only step with bit 5 set, so OR-ing the steps
// flags every case the windows cannot take.
#pragma once
#include "common.cuh"
#include "wordlane.cuh"

namespace cas {

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Shared-memory loads by 32-bit address, free for the compiler to schedule:
// every address they take derives from a base passed through fenced() after
// the stores it must see (and the barrier that publishes them), so no load is
// moved above those stores or reused across stagings.
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
// The same address, as a value the compiler cannot compute before this point.
__device__ __forceinline__ uint32_t fenced(uint32_t a) {
  uint32_t r;
  asm volatile("mov.u32 %0, %1;" : "=r"(r) : "r"(a) : "memory");
  return r;
}
__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }
// A read-only load whose bytes no other load reads (a warp's whole masks): not
// kept in L1, which then holds the data that is read again.
__device__ __forceinline__ uint4 ldg_once(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// Stores the low 16 bits of v (the instruction truncates the 32-bit register).
__device__ __forceinline__ void sts_u16(uint32_t a, uint32_t v) { asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "r"(v)); }

// 64-bit window (H, L) of a staged MSB-first bitstream at bit q: word rows
// `stride` bytes apart starting at address `base`, rows 0 .. maxw + 2.
__device__ __forceinline__ void bwindow(uint32_t base, uint32_t stride, int q, int maxw, uint32_t& H, uint32_t& L) {
  const int hw = min(q >> 5, maxw), sh = q & 31;
  const uint32_t a = base + stride * (uint32_t)hw;
  const uint32_t w0 = lds_u32(a), w1 = lds_u32(a + stride), w2 = lds_u32(a + 2u * stride);
  H = __funnelshift_l(w1, w0, sh);
  L = __funnelshift_l(w2, w1, sh);
}

// Index of the first '1' at or after bit b of a staged MSB-first bitstream
// (word rows `stride` bytes apart, rows 0..maxw), or -1.
__device__ __forceinline__ int bnext_one(uint32_t base, uint32_t stride, int b, int maxw) {
  int wi = b >> 5;
  if (wi > maxw) return -1;
  uint32_t h = lds_u32(base + stride * (uint32_t)wi) << (b & 31);
  int pos = b;
  while (h == 0u) {
    if (++wi > maxw) return -1;
    h = lds_u32(base + stride * (uint32_t)wi);
    pos = 32 * wi;
  }
  return pos + (int)__clz(h);
}

// Staged code streams: row u holds 2 zero words, then stream u (up to NW <=
// 32 W words, W per lane), then 4 zero words. A stream bit b sits at staged
// bit 64 + b.
template <int W, int NW = 32 * W>
struct BlockStreams {
  static constexpr int kWords = NW;
  static constexpr int kRow = 2 + NW + 4;
  uint32_t w[4][kRow];
};

// Zero words of the rows.
template <int W, int NW>
__device__ __forceinline__ void block_streams_init(BlockStreams<W, NW>& s, int lane) {
  if (lane < 4) {
    s.w[lane][0] = 0u;
    s.w[lane][1] = 0u;
#pragma unroll
    for (int i = 2 + NW; i < BlockStreams<W, NW>::kRow; ++i) s.w[lane][i] = 0u;
  }
}

// Stages stream u (nw[u] <= NW words at g[u]) into row u and returns, for
// lane = 8 t + j, the staged bit of the '1' that ends code kj - 1 of stream t
// (63, one bit before the stream, for j = 0): the lane's codes start one bit
// later. ok turns false when one of the first `present` streams holds fewer
// than 8 k codes. Ends with the staged rows visible to the whole warp.
template <int W, int k, int NW>
__device__ __forceinline__ int block_code_term(const uint32_t* const (&g)[4], const int (&nw)[4], int present,
                                               BlockStreams<W, NW>& s, int lane, bool& ok) {
  const int t = lane >> 3, j = lane & 7;
  int pc[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint32_t v[W];
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] = W * lane + i < nw[u] ? __ldg(g[u] + W * lane + i) : 0u;
    if (W == 2 && NW == 64) {
      *reinterpret_cast<uint2*>(&s.w[u][2 + 2 * lane]) = make_uint2(v[0], v[W - 1]);
    } else {
#pragma unroll
      for (int i = 0; i < W; ++i)
        if (W * lane + i < NW) s.w[u][2 + W * lane + i] = v[i];
    }
    pc[u] = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) pc[u] += __popc(v[i]);
  }
  // popcount prefixes over the lanes' words, two streams per register
  const int S01 = warp_incl_add(pc[0] | (pc[1] << 16), lane);
  const int S23 = warp_incl_add(pc[2] | (pc[3] << 16), lane);
  const int T01 = __shfl_sync(CAS_FULL, S01, 31), T23 = __shfl_sync(CAS_FULL, S23, 31);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int ones = ((u < 2 ? T01 : T23) >> (16 * (u & 1))) & 0xFFFF;
    if (u < present && ones < CAS_SB * k) ok = false;
  }
  // the lane whose words hold the (k j)-th '1' of stream t: lanes whose
  // prefix, in units of k, is below j (4 bits per stream)
  const int T = k * j;
  const int B01 = min((S01 & 0xFFFF) / k, 15) | (min((S01 >> 16) / k, 15) << 4);
  const int B23 = min((S23 & 0xFFFF) / k, 15) | (min((S23 >> 16) / k, 15) << 4);
  const int KB = B01 | (B23 << 8);
  int lo = 0;
#pragma unroll
  for (int step = 16; step >= 1; step >>= 1) {
    const int kb = __shfl_sync(CAS_FULL, KB, lo + step - 1);
    if (((kb >> (4 * t)) & 15) < j) lo += step;
  }
  const int lp = min(lo, 31);
  const int Sa = __shfl_sync(CAS_FULL, S01, lp), Sb = __shfl_sync(CAS_FULL, S23, lp);
  int before = ((t < 2 ? Sa : Sb) >> (16 * (t & 1))) & 0xFFFF;  // ones through lane lp's words
  __syncwarp();
  uint32_t v[W];
#pragma unroll
  for (int i = 0; i < W; ++i) v[i] = s.w[t][min(2 + W * lp + i, BlockStreams<W, NW>::kRow - 1)];
#pragma unroll
  for (int i = 0; i < W; ++i) before -= __popc(v[i]);
  int wsel = 0;
  uint32_t word = v[0];
#pragma unroll
  for (int i = 0; i < W - 1; ++i) {
    const int c = __popc(v[i]);
    if (T > before + c && wsel == i) {
      before += c;
      wsel = i + 1;
      word = v[i + 1];
    }
  }
  const int bit = 32 * (W * lp + wsel) + select_msb(word, max(T - before, 1));
  return j == 0 ? 63 : 64 + bit;
}

}  // namespace cas
