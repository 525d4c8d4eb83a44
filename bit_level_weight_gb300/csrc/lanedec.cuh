// lanedec.cuh - per-lane cursors for superblocks with k = 64: 512 kept (and
// 512 pruned) values, 16 consecutive ordinals per lane.
//
// Lane L owns kept ordinals 16L..16L+15 of the superblock: they are the
// ordinals 16(L%4)..16(L%4)+15 of block L/4, so their sign/mantissa fields are
// one 64-bit slice of that block's record and their positions follow one
// another in that block's mask. A lane walks two cursors:
//   - a unary cursor over the superblock's exponent code stream (MSB-first,
//     staged in shared memory): each step returns the rank of the next code
//     (Cassandra blog review, section 3.2: a code is `rank` zeros and a one);
//   - a mask cursor over the block's four mask words: each step returns the
//     position of the next kept (or, on the inverted mask, pruned) value.
// Both refill from the next word with predicated moves (no divergent branch,
// no global load in the loop). A code longer than the 32 bits of one refill
// is not decoded correctly; `unary_lane_ok` detects that afterwards (the lane
// then takes the generic path).
#pragma once
#include "common.cuh"

namespace cas {

constexpr int kStageWords = 128;  // unary words staged per superblock
constexpr int kStagePad = 24;     // zero words after them (cursor read-ahead)

struct UnaryStage {
  uint32_t st[kStageWords + kStagePad];
  uint16_t pc[kStageWords];  // inclusive popcount prefix per word
};

// Stages words [0, nw) of a unary stream (nw <= kStageWords) with their
// popcount prefixes; returns the number of ones (warp-uniform).
__device__ __forceinline__ int stage_unary(const uint32_t* __restrict__ g, int nw, UnaryStage& s, int lane) {
  int before = 0;
  for (int c0 = 0; c0 < nw; c0 += 32) {
    const uint32_t wv = c0 + lane < nw ? __ldg(g + c0 + lane) : 0u;
    s.st[c0 + lane] = wv;
    const int incl = warp_incl_add(__popc(wv), lane) + before;
    s.pc[c0 + lane] = (uint16_t)incl;
    before = __shfl_sync(CAS_FULL, incl, 31);
  }
  if (lane < kStagePad) s.st[nw + lane] = 0u;
  return before;
}

// Stream bit just after the T-th '1' (T >= 1; total ones >= T), i.e. where
// code T starts; 0 for T = 0. Branch-free lower bound over the prefixes (the
// trip count depends only on nw) and a popcount select inside the word.
__device__ __forceinline__ int unary_code_start(const UnaryStage& s, int nw, int T) {
  int base = 0, n = nw;
  while (n > 1) {
    const int half = n >> 1;
    base = (int)s.pc[base + half - 1] < T ? base + half : base;
    n -= half;
  }
  const int wsel = base;  // first word whose inclusive prefix reaches T
  const int excl = wsel > 0 ? (int)s.pc[wsel - 1] : 0;
  const int r = T - excl;  // the r-th '1' of word wsel (1-based)
  const int pos = nth_set_bit(__brev(s.st[wsel]), max(r - 1, 0));
  return T > 0 ? wsel * 32 + pos + 1 : 0;
}

// Cursor over the codes of a staged stream, from bit `start`.
struct UnaryCursor {
  uint32_t h, l;        // current word (consumed bits cleared), next word
  const uint32_t* np;   // word after l
  int sr;               // start of the current code relative to h's MSB
  int hw;               // index of h's word

  __device__ __forceinline__ void init(const UnaryStage& s, int start) {
    hw = start >> 5;
    sr = start & 31;
    h = s.st[hw] & (0xFFFFFFFFu >> sr);
    l = s.st[hw + 1];
    np = s.st + hw + 2;
  }
  // Rank of the next code (garbage, but harmless, for an over-long code);
  // *z_out gets its last bit relative to word hw.
  __device__ __forceinline__ int next(int* z_out) {
    if (h == 0u) {  // the code continues in the next word
      h = l;
      l = *np++;
      sr -= 32;
      ++hw;
    }
    const int z = __clz(h);  // 32 when the code runs past this word too
    h ^= __funnelshift_rc(0x80000000u, 0u, z);
    const int rank = z - sr;
    sr = z + 1;
    *z_out = z;
    return rank;
  }
};

// True when the lane's last code (last bit hw*32 + z) is the `ones`-th '1'
// of the stream: every code of the lane was short enough for the cursor.
__device__ __forceinline__ bool unary_lane_ok(const UnaryStage& s, int nw, int hw, int z, int ones) {
  const int end = hw * 32 + z;
  const int wi = end >> 5;
  if (wi >= nw) return false;
  const uint32_t word = s.st[wi];
  const int b = end & 31;
  const uint32_t upto = word >> (31 - b);  // bits 0..b of the word, MSB-first
  const int cnt = (wi > 0 ? (int)s.pc[wi - 1] : 0) + __popc(upto);
  return (upto & 1u) && cnt == ones;
}

// Cursor over the set bits of a block's 128-bit mask (LSB-first positions),
// starting at the r-th set bit (0-based). Words are held bit-reversed so the
// next position is a clz.
struct MaskCursor {
  uint32_t cur, n1, n2, n3;
  int base;

  __device__ __forceinline__ void init(uint32_t m0, uint32_t m1, uint32_t m2, uint32_t m3, int r) {
    const int c0 = __popc(m0), c01 = c0 + __popc(m1), c012 = c01 + __popc(m2);
    const int w0 = (r >= c0) + (r >= c01) + (r >= c012);
    const int excl = w0 == 0 ? 0 : w0 == 1 ? c0 : w0 == 2 ? c01 : c012;
    const uint32_t a0 = w0 == 0 ? m0 : w0 == 1 ? m1 : w0 == 2 ? m2 : m3;
    const uint32_t a1 = w0 == 0 ? m1 : w0 == 1 ? m2 : w0 == 2 ? m3 : 0u;
    const uint32_t a2 = w0 == 0 ? m2 : w0 == 1 ? m3 : 0u;
    const uint32_t a3 = w0 == 0 ? m3 : 0u;
    const int bit = nth_set_bit(a0, min(max(r - excl, 0), 31));
    cur = __brev(a0 & (0xFFFFFFFFu << bit));
    n1 = __brev(a1);
    n2 = __brev(a2);
    n3 = __brev(a3);
    base = 32 * w0;
  }
  // Position (0..127) of the next set bit.
  __device__ __forceinline__ int next() {
    if (cur == 0u) {
      cur = n1;
      n1 = n2;
      n2 = n3;
      n3 = 0u;
      base += 32;
    }
    const int p = __clz(cur);
    cur ^= __funnelshift_rc(0x80000000u, 0u, p);
    return (base + p) & 127;
  }
};

}  // namespace cas
