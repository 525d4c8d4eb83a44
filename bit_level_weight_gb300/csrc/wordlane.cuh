// wordlane.cuh - per-lane decoding of a superblock with lane = mask word.
//
// Lane L of a warp owns mask word L of a superblock of 8 blocks: block L/4,
// positions 32(L%4)..+31. Its kept values are consecutive kept ordinals and
// its pruned values consecutive pruned ordinals, so every field of them is one
// bit range of a block record and every exponent code one bit range of the
// superblock's unary stream (Cassandra blog review, section 3.2: a code is
// `rank` zeros then a one). Each lane finds where its codes start - the bit
// after the T-th '1' of the stream, T its first ordinal - and then walks its
// own cursors, with no cross-lane traffic per value:
//   position: count of leading zeros of a bit-reversed mask word, the found
//             bit cleared (32 once the word is exhausted);
//   code:     count of leading zeros of a 64-bit window of the stream
//             aligned at the lane's first code, re-aligned every 8 codes;
//   field:    a byte of a window of the lane's record fields, placed by one
//             byte permute.
// A superblock is taken only when every code is at most 31 bits (no run of
// 31 zeros), the stream fits the stage and every group of 8 codes fits its
// 64-bit window; otherwise the caller falls back to the generic decoder.
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

// A superblock's unary stream staged in shared memory: nw <= 32*W words,
// words W*l .. W*l+W-1 held by lane l, then 32 zero words.
template <int W>
struct StreamStage {
  uint32_t st[32 * W + 32];
};

template <int W>
struct StreamInfo {
  uint32_t w[W];  // this lane's words
  int S;          // ones in words 0 .. W*lane+W-1
  int ones;       // ones in the stream
  int endbit;     // stream bit after the last '1'
  bool lng;       // a run of 31 or more zeros (a code longer than 31 bits)
};

template <int W>
__device__ __forceinline__ StreamInfo<W> stage_stream(const uint32_t* __restrict__ g, int nw, StreamStage<W>& s,
                                                      int lane) {
  StreamInfo<W> in;
  int pc = 0;
#pragma unroll
  for (int i = 0; i < W; ++i) {
    const int wi = W * lane + i;
    in.w[i] = wi < nw ? __ldg(g + wi) : 0u;
    s.st[wi] = in.w[i];
    pc += __popc(in.w[i]);
  }
  s.st[32 * W + lane] = 0u;
  in.S = warp_incl_add(pc, lane);
  in.ones = __shfl_sync(CAS_FULL, in.S, 31);
  // runs of 31+ zeros across word boundaries (inside a word a run of 31 zeros
  // touches a boundary, so these pairs see every such run)
  bool run = lane == 0 && nw > 0 && __clz(in.w[0]) >= 31;
  const int lzn = __shfl_down_sync(CAS_FULL, __clz(in.w[0]), 1);
  int tzl = 32;  // trailing zeros of the word that holds the stream's last bit
#pragma unroll
  for (int i = 0; i < W; ++i) {
    const int wi = W * lane + i;
    const int tz = tzcnt(in.w[i]);
    const int lz = i + 1 < W ? __clz(in.w[i + 1 < W ? i + 1 : i]) : lzn;
    if (wi + 1 < nw && tz + lz >= 31) run = true;
    if (wi == nw - 1) tzl = tz;
  }
  in.lng = __any_sync(CAS_FULL, run);
  const int lw = nw - 1;
  tzl = __shfl_sync(CAS_FULL, tzl, (lw >= 0 ? lw / W : 0) & 31);
  in.endbit = nw > 0 ? 32 * lw + 32 - tzl : 0;
  return in;
}

// Stream bit just after the T-th '1' (0 for T = 0; T <= in.ones).
template <int W>
__device__ __forceinline__ int code_start(const StreamInfo<W>& in, int T) {
  const int l = min(warp_count_le(in.S, T - 1), 31);  // first lane whose prefix reaches T
  int before = __shfl_sync(CAS_FULL, in.S, l);
  uint32_t ws[W];
#pragma unroll
  for (int i = 0; i < W; ++i) ws[i] = __shfl_sync(CAS_FULL, in.w[i], l);
#pragma unroll
  for (int i = 0; i < W; ++i) before -= __popc(ws[i]);  // ones before lane l's words
  int wsel = 0;
  uint32_t word = ws[0];
#pragma unroll
  for (int i = 0; i < W - 1; ++i) {
    const int c = __popc(ws[i]);
    if (T > before + c && wsel == i) {
      before += c;
      wsel = i + 1;
      word = ws[i + 1];
    }
  }
  const int r = max(T - before, 1);
  return T > 0 ? 32 * (W * l + wsel) + select_msb(word, r) + 1 : 0;
}

// 64-bit window of a staged stream at bit `pos` (hi, lo).
template <int W>
__device__ __forceinline__ void window64(const StreamStage<W>& s, int pos, uint32_t& H, uint32_t& L) {
  const int hw = min(pos >> 5, 32 * W + 29), sh = pos & 31;
  H = __funnelshift_l(s.st[hw + 1], s.st[hw], sh);
  L = __funnelshift_l(s.st[hw + 2], s.st[hw + 1], sh);
}

// Group-of-8 window check: a lane with c codes that consumed u8, u16, u24
// bits by its 8th, 16th and 24th code and whose codes span `span` bits.
__device__ __forceinline__ bool windows_ok(int c, int u8, int u16, int u24, int span) {
  const int last = (c - 1) >> 3;  // -1 when the lane has no values
  const int lastu = last == 0 ? 0 : last == 1 ? u8 : last == 2 ? u16 : u24;
  return !((last > 0 && u8 > 64) || (last > 1 && u16 - u8 > 64) || (last > 2 && u24 - u16 > 64) ||
           (last >= 0 && span - lastu > 64));
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

// One walk over a lane's values: `n` values of one stream, positions from the
// bit-reversed word M, codes from the window at `start`. For value i,
// emit(i, g, e) gets g = the distance in positions from the previous value
// (the first value: its position) and the exponent e = lut[rank]; once the
// word is exhausted g is 32 (an emitted value past n must not be stored).
// Returns whether the windows held every code.
template <int W, class Emit>
__device__ __forceinline__ bool walk_lane(uint32_t M, int n, int maxn, const StreamStage<W>& s, int start, int span,
                                          const uint8_t* lut, Emit emit) {
  uint32_t H, L;
  window64(s, start, H, L);
  int used = 0, u8 = 0, u16 = 0, u24 = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if ((i & 3) == 0 && i >= maxn) break;
    if ((i & 7) == 0 && i > 0) {
      if (i == 8) u8 = used;
      if (i == 16) u16 = used;
      if (i == 24) u24 = used;
      window64(s, start + used, H, L);
    }
    const uint32_t g = __clz(M);  // positions skipped before this value
    M = shl32(M, g + 1u);
    const uint32_t r = __clz(H);  // <= 30 for every code of a checked stream
    const uint32_t e = lut[r];
    const uint32_t nb = r + 1u;
    H = shfl_wrap(L, H, nb);
    L = shl32(L, nb);
    used += (int)nb;
    emit(i, g, e);
  }
  return windows_ok(n, u8, u16, u24, span);
}

// bf16 of a field byte B placed in bytes 1 and 0 by a permute: bit 15 takes
// the byte's bit 7, bits 6..0 its bits 6..0; e << 7 fills bits 14..7.
__device__ __forceinline__ uint32_t bf16_from_byte(uint32_t src, int by, uint32_t e, uint32_t keep) {
  const uint32_t A = __byte_perm(src, 0u, 0x4400 | (by << 4) | by);
  return mad32(e, 128u, A & keep);
}

}  // namespace cas

namespace cas {

// Per-warp stage of word_tile: one code stream at a time (kept codes, then
// pruned codes) and the records that go with it.
struct WordTileStage {
  StreamStage<3> ss;      // <= 96 stream words + pad
  uint32_t rec[128 + 16];  // spec_sm + ver_lo records (64 + 64 words), or ver_pr (128 words); + pad
};

// Rebuilds one whole superblock (Cassandra-1, k = 64, m = 3, 8 blocks) as
// bf16 bit patterns: the value at position p of block i goes to
// dst[i * bstride + p]. FULL merges speculation and verification data (the
// original bits); otherwise the draft value is written and pruned positions
// are zero. mask: 32 words, sm / lo: 64 words, pr: 128 words of the
// superblock (16-byte aligned); sexp / vexp: its code streams of snw / vnw
// words; lut: exponent by rank. Returns false (warp-uniform) when the
// superblock is not taken: dst is then partly written and the caller
// rebuilds it with the generic decoder. dst + i * bstride must be 16-byte
// aligned.
template <bool FULL>
__device__ __forceinline__ bool word_tile(const uint32_t* __restrict__ mask, const uint32_t* __restrict__ sm,
                                          const uint32_t* __restrict__ lo, const uint32_t* __restrict__ pr,
                                          const uint32_t* __restrict__ sexp, int snw,
                                          const uint32_t* __restrict__ vexp, int vnw, const uint8_t* lut,
                                          WordTileStage& ts, uint16_t* dst, int bstride, int lane) {
  if (snw > 64 || (FULL && vnw > 96)) return false;
  const int blk = lane >> 2, q = lane & 3;
  uint16_t* row = dst + blk * bstride + 32 * q;
  const uint32_t mw = __ldg(mask + lane);
  const int c = __popc(mw);
  int inc = c;
  const int u1 = __shfl_up_sync(CAS_FULL, inc, 1, 4);
  if (q >= 1) inc += u1;
  const int u2 = __shfl_up_sync(CAS_FULL, inc, 2, 4);
  if (q >= 2) inc += u2;
  const int o = min(inc - c, 64);  // block-local ordinal of the lane's first kept value
  // kept values
  {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(sm) + lane);
    ts.rec[2 * lane] = a.x;
    ts.rec[2 * lane + 1] = a.y;
    if (FULL) {
      const uint2 b = __ldg(reinterpret_cast<const uint2*>(lo) + lane);
      ts.rec[64 + 2 * lane] = b.x;
      ts.rec[64 + 2 * lane + 1] = b.y;
    }
    if (lane < 16) ts.rec[128 + lane] = 0u;
    if (!FULL) {
      uint4* z = reinterpret_cast<uint4*>(row);
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      z[0] = zero;
      z[1] = zero;
      z[2] = zero;
      z[3] = zero;
    }
  }
  const StreamInfo<3> kin = stage_stream<3>(sexp, snw, ts.ss, lane);
  __syncwarp();
  const int ks = code_start(kin, 64 * blk + o);
  int kn = __shfl_down_sync(CAS_FULL, ks, 1);
  if (lane == 31) kn = kin.endbit;
  // field windows: nibble i of word i/8 is the lane's field i; the even and
  // odd fields of spec_sm (sign, 3 high mantissa bits) and ver_lo (4 low
  // mantissa bits) merged into one byte each: [s f6 f5 f4 | f3 f2 f1 f0]
  uint32_t te[4], to[4];
  {
    const uint32_t* rs = ts.rec + 8 * blk + (o >> 3);
    const int fs = 4 * (o & 7);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t f = __funnelshift_r(rs[i], rs[i + 1], fs);
      if (FULL) {
        const uint32_t g = __funnelshift_r(rs[64 + i], rs[64 + i + 1], fs);
        te[i] = ((f << 4) & 0xF0F0F0F0u) | (g & 0x0F0F0F0Fu);
        to[i] = (f & 0xF0F0F0F0u) | ((g >> 4) & 0x0F0F0F0Fu);
      } else {
        te[i] = f << 4;
        to[i] = f;
      }
    }
  }
  const int maxc = __reduce_max_sync(CAS_FULL, c);
  constexpr uint32_t keep = FULL ? 0x807Fu : 0x8070u;
  uint32_t ka = (uint32_t)__cvta_generic_to_shared(row) - 2u;  // address of the previous value
  bool ok = walk_lane<3>(__brev(mw), c, maxc, ts.ss, ks, kn - ks, lut, [&](int i, uint32_t g, uint32_t e) {
    const uint32_t v = bf16_from_byte((i & 1) ? to[i >> 3] : te[i >> 3], (i & 7) >> 1, e, keep);
    ka = mad32(g, 2u, ka + 2u);
    if (i < c) asm volatile("st.shared.u16 [%0], %1;" ::"r"(ka), "h"((uint16_t)v));
  });
  ok = ok && !kin.lng && kin.ones >= CAS_SB * 64;
  if (!FULL) return __all_sync(CAS_FULL, ok);
  // pruned values
  __syncwarp();  // every lane is done with the kept stage
  {
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(pr) + lane);
    *reinterpret_cast<uint4*>(ts.rec + 4 * lane) = b;
  }
  const StreamInfo<3> pin = stage_stream<3>(vexp, vnw, ts.ss, lane);
  __syncwarp();
  const int u0 = min(max(32 * q - o, 0), 64);  // block-local ordinal of the first pruned value
  const int ps = code_start(pin, 64 * blk + u0);
  int pn = __shfl_down_sync(CAS_FULL, ps, 1);
  if (lane == 31) pn = pin.endbit;
  uint32_t pb[8];  // byte j of the lane: (s << 7) | f of its j-th pruned value
  {
    const uint32_t* rp = ts.rec + 16 * blk + (u0 >> 2);
    const int bs = 8 * (u0 & 3);
#pragma unroll
    for (int i = 0; i < 8; ++i) pb[i] = __funnelshift_r(rp[i], rp[i + 1], bs);
  }
  const int np = 32 - c;
  const int maxp = __reduce_max_sync(CAS_FULL, np);
  uint32_t pa = (uint32_t)__cvta_generic_to_shared(row) - 2u;
  bool ok2 = walk_lane<3>(__brev(~mw), np, maxp, ts.ss, ps, pn - ps, lut, [&](int j, uint32_t g, uint32_t e) {
    const uint32_t v = bf16_from_byte(pb[j >> 2], j & 3, e, 0x807Fu);
    pa = mad32(g, 2u, pa + 2u);
    if (j < np) asm volatile("st.shared.u16 [%0], %1;" ::"r"(pa), "h"((uint16_t)v));
  });
  ok2 = ok2 && !pin.lng && pin.ones >= CAS_SB * 64;
  return __all_sync(CAS_FULL, ok && ok2);
}

}  // namespace cas
