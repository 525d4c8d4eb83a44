// lanedec.cuh - per-lane decoding of superblocks with k = 64: 512 kept (and
// 512 pruned) values, 16 consecutive ordinals per lane.
//
// Lane L owns kept ordinals 16L..16L+15 of the superblock: they are the
// ordinals 16(L%4)..16(L%4)+15 of block L/4, so their sign/mantissa fields are
// one 64-bit slice of that block's record. The warp first stages the
// superblock's unary exponent stream in shared memory (with popcount prefixes)
// and expands the mask into the block position of every ordinal (lane = mask
// word). Each lane then finds where its first code starts and walks a unary
// cursor (Cassandra blog review, section 3.2: a code is `rank` zeros and a
// one): each step returns the rank of the next code. The cursor refills from
// the next staged word with predicated moves; a code that spans more than one
// further word (possible only when a staged word is all zeros) takes a rare
// loop, compiled in only for such streams.
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
// popcount prefixes; returns the number of ones (warp-uniform). *long_codes
// (warp-uniform) tells whether a staged word is all zeros: only then can a
// code outlast one refill of the cursor.
__device__ __forceinline__ int stage_unary(const uint32_t* __restrict__ g, int nw, UnaryStage& s, int lane,
                                           bool* long_codes) {
  int before = 0;
  bool zero = false;
  for (int c0 = 0; c0 < nw; c0 += 32) {
    const bool in = c0 + lane < nw;
    const uint32_t wv = in ? __ldg(g + c0 + lane) : 0u;
    s.st[c0 + lane] = wv;
    zero |= in && wv == 0u;
    const int incl = warp_incl_add(__popc(wv), lane) + before;
    s.pc[c0 + lane] = (uint16_t)incl;
    before = __shfl_sync(CAS_FULL, incl, 31);
  }
  if (lane < kStagePad) s.st[nw + lane] = 0u;
  *long_codes = __any_sync(CAS_FULL, zero);
  return before;
}

// Stream bit just after the T-th '1' (T >= 1; total ones >= T), i.e. where
// code T starts; 0 for T = 0. Branch-free lower bound over the prefixes (the
// trip count depends only on nw) and a popcount select inside the word.
__device__ __forceinline__ int unary_code_start(const uint32_t* st, const uint16_t* pc, int nw, int T) {
  int base = 0, n = nw;
  while (n > 1) {
    const int half = n >> 1;
    base = (int)pc[base + half - 1] < T ? base + half : base;
    n -= half;
  }
  const int wsel = base;  // first word whose inclusive prefix reaches T
  const int excl = wsel > 0 ? (int)pc[wsel - 1] : 0;
  const int r = T - excl;  // the r-th '1' of word wsel (1-based)
  const int pos = nth_set_bit(__brev(st[wsel]), max(r - 1, 0));
  return T > 0 ? wsel * 32 + pos + 1 : 0;
}
__device__ __forceinline__ int unary_code_start(const UnaryStage& s, int nw, int T) {
  return unary_code_start(s.st, s.pc, nw, T);
}

// Cursor over the codes of a staged stream, from bit `start`.
struct UnaryCursor {
  uint32_t h, l;        // current word (consumed bits cleared), next word
  const uint32_t* np;   // word after l
  int sr;               // start of the current code relative to h's MSB
  const uint32_t* end;  // the rare loop reads no further (the 16 plain
                        // refills after it stay inside the stage pad)

  // st holds cap + kStagePad readable words (cap >= the stream's words).
  __device__ __forceinline__ void init(const uint32_t* st, int cap, int start) {
    const int hw = start >> 5;
    end = st + cap + 2;
    sr = start & 31;
    h = st[hw] & (0xFFFFFFFFu >> sr);
    l = st[hw + 1];
    np = st + hw + 2;
  }
  __device__ __forceinline__ void init(const UnaryStage& s, int start) { init(s.st, kStageWords, start); }
  // Rank of the next code. LONG: the stream has an all-zero word, so a code
  // may need more than one refill. A stream with fewer codes than asked for
  // yields garbage ranks, never a read outside the stage.
  template <bool LONG>
  __device__ __forceinline__ int next() {
    if (h == 0u) {  // the code continues in the next word
      h = l;
      l = *np++;
      sr -= 32;
    }
    if (LONG) {
      while (h == 0u && np < end) {
        h = l;
        l = *np++;
        sr -= 32;
      }
    }
    const int z = __clz(h);  // 32 only when the staged words ran out
    h ^= __funnelshift_rc(0x80000000u, 0u, z);
    const int rank = z - sr;
    sr = z + 1;
    return rank;
  }
};

// Lane L = mask word L of the superblock (block L/4, positions 32(L%4)..+31)
// writes the block position of each of its kept values at their superblock
// ordinal. Positions of a corrupt mask (a block without exactly 64 kept
// values) land at wrong ordinals but never outside the array.
// CAP: entries of pos (a power of two; 512 for k = 64, 1024 for any k).
template <int CAP = CAS_SB * 64>
__device__ __forceinline__ void expand_mask_positions(uint32_t mw, uint8_t* pos, int lane) {
  const int cnt = __popc(mw);
  int idx = warp_incl_add(cnt, lane) - cnt;
  uint32_t pv = 32u * (lane & 3);
#pragma unroll
  for (int p = 0; p < 32; ++p) {
    if ((mw >> p) & 1u) {
      pos[idx & (CAP - 1)] = (uint8_t)pv;
      ++idx;
    }
    ++pv;
  }
}

// Same for both the kept (set) and the pruned (clear) bits of the word in one
// pass: kpos gets the kept positions by kept ordinal, ppos the pruned ones by
// pruned ordinal.
__device__ __forceinline__ void expand_mask_both(uint32_t mw, uint8_t* kpos, uint8_t* ppos, int lane) {
  const int cnt = __popc(mw);
  const int kbefore = warp_incl_add(cnt, lane) - cnt;
  int ki = kbefore, pi = 32 * lane - kbefore;
  uint32_t pv = 32u * (lane & 3);
#pragma unroll
  for (int p = 0; p < 32; ++p) {
    if ((mw >> p) & 1u) {
      kpos[ki & (CAS_SB * 64 - 1)] = (uint8_t)pv;
      ++ki;
    } else {
      ppos[pi & (CAS_SB * 64 - 1)] = (uint8_t)pv;
      ++pi;
    }
    ++pv;
  }
}

}  // namespace cas

namespace cas {

// Byte i of a 16-byte group of positions.
__device__ __forceinline__ int pos_byte(uint4 pq, int i) {
  const uint32_t pw = (i >> 2) == 0 ? pq.x : (i >> 2) == 1 ? pq.y : (i >> 2) == 2 ? pq.z : pq.w;
  return (pw >> (8 * (i & 3))) & 127u;
}

// Kept values of lane L (ordinals 16L..16L+15): positions from the expanded
// mask, exponent from the unary cursor, sign and mantissa fields from the
// lane's slices of the speculation (rs) and cut-mantissa (rl) records.

template <bool FULL, bool LONG>
__device__ __forceinline__ void lane_kept_to_row(UnaryCursor& uc, uint4 pq, uint2 rs, uint2 rl,
                                                 const uint8_t* __restrict__ lut, uint16_t* row) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int pos = pos_byte(pq, i);
    const uint32_t e = lut[uc.next<LONG>() & 255];
    const int sh = 4 * (i & 7);
    const uint32_t f = (i < 8 ? rs.x : rs.y) >> sh;
    uint32_t bits = ((f & 8u) << 12) | (e << 7) | ((f & 7u) << 4);
    if (FULL) bits |= ((i < 8 ? rl.x : rl.y) >> sh) & 15u;
    row[pos] = (uint16_t)bits;
  }
}

// Pruned values of lane L (pruned ordinals 16L..16L+15) from their positions,
// the pruned exponent stream and the lane's 16 verification bytes.
template <bool LONG>
__device__ __forceinline__ void lane_pruned_to_row(UnaryCursor& uc, uint4 pq, uint4 pb,
                                                   const uint8_t* __restrict__ lut, uint16_t* row) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int pos = pos_byte(pq, i);
    const uint32_t e = lut[uc.next<LONG>() & 255];
    const uint32_t wsel = (i >> 2) == 0 ? pb.x : (i >> 2) == 1 ? pb.y : (i >> 2) == 2 ? pb.z : pb.w;
    const uint32_t byte = (wsel >> (8 * (i & 3))) & 0xFFu;
    row[pos] = (uint16_t)(((byte & 0x80u) << 8) | (e << 7) | (byte & 0x7Fu));
  }
}

// Per-warp shared scratch of the tile decoder.
struct TileStage {
  UnaryStage us;
  alignas(16) uint8_t kpos[CAS_SB * 64];  // block position of every kept ordinal
  alignas(16) uint8_t ppos[CAS_SB * 64];  // block position of every pruned ordinal
};

// Rebuilds one whole superblock (Cassandra-1, k = 64, m = 3, 8 blocks) as bf16
// bit patterns: the value at position p of block i goes to dst[i * bstride + p].
// FULL merges speculation and verification data (lossless); otherwise the
// draft value is written and pruned positions are zero. Lane L rebuilds kept
// ordinals 16L..16L+15 (and, FULL, pruned ordinals 16L..16L+15) with the
// unary cursor and the expanded mask; the unary streams are staged one after
// the other. mask: 32 words, sm / lo: 64 words, pr: 128 words of the
// superblock (16-byte aligned); sexp / vexp: its code streams. Returns false (warp-uniform) when a
// stream is longer than the stage or holds fewer than 512 codes: dst is then
// partly written and the caller rebuilds the superblock with the generic
// decoder. dst + i * bstride must be 16-byte aligned.
template <bool FULL>
__device__ __forceinline__ bool lane_sb_tile(const uint32_t* __restrict__ mask, const uint32_t* __restrict__ sm,
                                             const uint32_t* __restrict__ lo, const uint32_t* __restrict__ pr,
                                             const uint32_t* __restrict__ sexp, int snw,
                                             const uint32_t* __restrict__ vexp, int vnw,
                                             const uint8_t* __restrict__ lut, TileStage& ts, uint16_t* dst,
                                             int bstride, int lane) {
  if (snw > kStageWords || (FULL && vnw > kStageWords)) return false;
  uint16_t* row = dst + (lane >> 2) * bstride;
  const uint32_t mw = __ldg(mask + lane);
  const uint2 rs = __ldg(reinterpret_cast<const uint2*>(sm) + lane);
  uint2 rl = make_uint2(0u, 0u);
  if (FULL) rl = __ldg(reinterpret_cast<const uint2*>(lo) + lane);
  if (!FULL) {
    uint4* z = reinterpret_cast<uint4*>(row + 32 * (lane & 3));
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    z[0] = zero;
    z[1] = zero;
    z[2] = zero;
    z[3] = zero;
  }
  bool long_codes;
  const bool enough = stage_unary(sexp, snw, ts.us, lane, &long_codes) >= 16 * 32;
  if (FULL)
    expand_mask_both(mw, ts.kpos, ts.ppos, lane);
  else
    expand_mask_positions(mw, ts.kpos, lane);
  __syncwarp();
  if (!enough) return false;
  UnaryCursor uc;
  uc.init(ts.us, unary_code_start(ts.us, snw, 16 * lane));
  const uint4 kq = reinterpret_cast<const uint4*>(ts.kpos)[lane];
  if (long_codes)
    lane_kept_to_row<FULL, true>(uc, kq, rs, rl, lut, row);
  else
    lane_kept_to_row<FULL, false>(uc, kq, rs, rl, lut, row);
  if (FULL) {
    const uint4 pb = __ldg(reinterpret_cast<const uint4*>(pr) + lane);
    __syncwarp();  // every lane is done with the kept stream
    const bool enough_v = stage_unary(vexp, vnw, ts.us, lane, &long_codes) >= 16 * 32;
    __syncwarp();
    if (!enough_v) return false;
    uc.init(ts.us, unary_code_start(ts.us, vnw, 16 * lane));
    const uint4 pq = reinterpret_cast<const uint4*>(ts.ppos)[lane];
    if (long_codes)
      lane_pruned_to_row<true>(uc, pq, pb, lut, row);
    else
      lane_pruned_to_row<false>(uc, pq, pb, lut, row);
  }
  __syncwarp();
  return true;
}

// Any k and m (Cassandra-1, one whole superblock): lane L rebuilds the run of
// kept ordinals [L q, L q + q), q = ceil(8k / 32), and (FULL) the run of
// pruned ordinals [L q', L q' + q'), q' = ceil(8(128-k) / 32); runs may cross
// blocks. Positions come from the mask expanded into `pos` (1024 bytes; kept,
// then pruned), exponents from the unary cursor, record fields from global
// memory at run-time bit offsets (rec_*: words per block record). Same
// contract as lane_sb_tile; scratch: `us` and `pos` (1888 bytes).
__device__ __forceinline__ uint32_t field_g(const uint32_t* __restrict__ w, int bit, int width) {
  const int i = bit >> 5;
  return __funnelshift_r(__ldg(w + i), __ldg(w + i + 1), bit & 31) & ((1u << width) - 1u);
}

template <bool FULL, bool LONG>
__device__ __forceinline__ void runs_kept_to_tile(UnaryCursor& uc, const uint8_t* pos, const uint32_t* sm, int rec_sm,
                                                  const uint32_t* lo, int rec_lo, int k, int m, int t0, int t1,
                                                  const uint8_t* __restrict__ lut, uint16_t* dst, int bstride) {
  int b = k > 0 ? t0 / k : 0;
  int tl = t0 - b * k;
  for (int t = t0; t < t1; ++t) {
    if (tl == k) {
      ++b;
      tl = 0;
    }
    const uint32_t fld = field_g(sm + b * rec_sm, tl * (m + 1), m + 1);
    const uint32_t e = lut[uc.next<LONG>() & 255];
    uint32_t bits = ((fld >> m) << 15) | (e << 7) | ((fld & ((1u << m) - 1u)) << (7 - m));
    if (FULL && m < 7) bits |= field_g(lo + b * rec_lo, tl * (7 - m), 7 - m);
    ++tl;
    dst[b * bstride + pos[t]] = (uint16_t)bits;
  }
}

template <bool LONG>
__device__ __forceinline__ void runs_pruned_to_tile(UnaryCursor& uc, const uint8_t* pos, const uint32_t* pr, int rec_pr,
                                                    int kp, int u0, int u1, const uint8_t* __restrict__ lut,
                                                    uint16_t* dst, int bstride) {
  int b = kp > 0 ? u0 / kp : 0;
  int ul = u0 - b * kp;
  for (int u = u0; u < u1; ++u) {
    if (ul == kp) {
      ++b;
      ul = 0;
    }
    const uint32_t byte = (__ldg(pr + b * rec_pr + (ul >> 2)) >> (8 * (ul & 3))) & 0xFFu;
    const uint32_t e = lut[uc.next<LONG>() & 255];
    ++ul;
    dst[b * bstride + pos[u]] = (uint16_t)(((byte & 0x80u) << 8) | (e << 7) | (byte & 0x7Fu));
  }
}

template <bool FULL>
__device__ __forceinline__ bool runs_sb_tile(const uint32_t* __restrict__ mask, const uint32_t* __restrict__ sm,
                                             int rec_sm, const uint32_t* __restrict__ lo, int rec_lo,
                                             const uint32_t* __restrict__ pr, int rec_pr,
                                             const uint32_t* __restrict__ sexp, int snw,
                                             const uint32_t* __restrict__ vexp, int vnw, int k, int m,
                                             const uint8_t* __restrict__ lut, UnaryStage& us, uint8_t* pos,
                                             uint16_t* dst, int bstride, int lane) {
  if (snw > kStageWords || (FULL && vnw > kStageWords)) return false;
  const uint32_t mw = __ldg(mask + lane);
  if (!FULL) {
    uint4* z = reinterpret_cast<uint4*>(dst + (lane >> 2) * bstride + 32 * (lane & 3));
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    z[0] = zero;
    z[1] = zero;
    z[2] = zero;
    z[3] = zero;
  }
  const int kt = CAS_SB * k, q = (kt + 31) >> 5;
  const int t0 = min(lane * q, kt), t1 = min(t0 + q, kt);
  bool long_codes;
  const bool enough = stage_unary(sexp, snw, us, lane, &long_codes) >= kt;
  expand_mask_positions<CAS_SB * CAS_BLK>(mw, pos, lane);
  __syncwarp();
  if (!enough) return false;
  UnaryCursor uc;
  uc.init(us, unary_code_start(us, snw, t0));
  if (long_codes)
    runs_kept_to_tile<FULL, true>(uc, pos, sm, rec_sm, lo, rec_lo, k, m, t0, t1, lut, dst, bstride);
  else
    runs_kept_to_tile<FULL, false>(uc, pos, sm, rec_sm, lo, rec_lo, k, m, t0, t1, lut, dst, bstride);
  if (FULL) {
    const int kp = CAS_BLK - k, pt = CAS_SB * kp, q2 = (pt + 31) >> 5;
    const int u0 = min(lane * q2, pt), u1 = min(u0 + q2, pt);
    __syncwarp();  // every lane is done with the kept stream and positions
    const bool enough_v = stage_unary(vexp, vnw, us, lane, &long_codes) >= pt;
    expand_mask_positions<CAS_SB * CAS_BLK>(~mw, pos, lane);
    __syncwarp();
    if (!enough_v) return false;
    uc.init(us, unary_code_start(us, vnw, u0));
    if (long_codes)
      runs_pruned_to_tile<true>(uc, pos, pr, rec_pr, kp, u0, u1, lut, dst, bstride);
    else
      runs_pruned_to_tile<false>(uc, pos, pr, rec_pr, kp, u0, u1, lut, dst, bstride);
  }
  __syncwarp();
  return true;
}

// Cassandra-2, any k and m, one whole superblock (same contract as
// runs_sb_tile). Kept value t: sign and q from its spec_q field, E' = max(E, 1)
// of its 32-position group; the draft value is q * 2^(E'-127-m). FULL adds
// the distance d (unary code of the ver_d stream, read with the cursor) and
// the min(8, 7-m+d) residual bits: sig = (q << w) | residual, exponent E' - d
// when sig's leading bit is set (else 0). A lane's residual bits start at the
// exclusive warp sum of the widths of the runs before it, so the lane first
// decodes its d codes into `dbuf`. Pruned values as for Cassandra-1.
struct TileStage2 {
  UnaryStage us;
  alignas(16) uint8_t pos[CAS_SB * CAS_BLK];
  uint8_t dbuf[CAS_SB * CAS_BLK];  // distance d of every kept ordinal
  uint8_t mx[CAS_SB * 4];          // shared exponents of the superblock
};

template <bool LONG>
__device__ __forceinline__ int runs_read_d(UnaryCursor& uc, uint8_t* dbuf, int m, int t0, int t1) {
  int wsum = 0;
  for (int t = t0; t < t1; ++t) {
    const int dd = uc.next<LONG>() & 255;
    dbuf[t] = (uint8_t)dd;
    wsum += min(8, 7 - m + dd);
  }
  return wsum;
}

template <bool FULL>
__device__ __forceinline__ bool runs_sb_tile_c2(const uint32_t* __restrict__ mask, const uint32_t* __restrict__ sq,
                                                int rec_q, const uint8_t* __restrict__ smx,
                                                const uint32_t* __restrict__ vd, int dnw,
                                                const uint32_t* __restrict__ vres,
                                                const uint32_t* __restrict__ pr, int rec_pr,
                                                const uint32_t* __restrict__ vexp, int vnw, int k, int m,
                                                const uint8_t* __restrict__ lut, TileStage2& ts, uint16_t* dst,
                                                int bstride, int lane) {
  if (FULL && (dnw > kStageWords || vnw > kStageWords)) return false;
  const uint32_t mw = __ldg(mask + lane);
  if (!FULL) {
    uint4* z = reinterpret_cast<uint4*>(dst + (lane >> 2) * bstride + 32 * (lane & 3));
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    z[0] = zero;
    z[1] = zero;
    z[2] = zero;
    z[3] = zero;
  }
  const int kt = CAS_SB * k, q = (kt + 31) >> 5;
  const int t0 = min(lane * q, kt), t1 = min(t0 + q, kt);
  ts.mx[lane] = __ldg(smx + lane);
  bool long_codes = false, enough = true;
  if (FULL) enough = stage_unary(vd, dnw, ts.us, lane, &long_codes) >= kt;
  expand_mask_positions<CAS_SB * CAS_BLK>(mw, ts.pos, lane);
  __syncwarp();
  if (!enough) return false;
  int rbit = 0;
  if (FULL) {
    UnaryCursor uc;
    uc.init(ts.us, unary_code_start(ts.us, dnw, t0));
    const int wsum = long_codes ? runs_read_d<true>(uc, ts.dbuf, m, t0, t1) : runs_read_d<false>(uc, ts.dbuf, m, t0, t1);
    rbit = warp_incl_add(wsum, lane) - wsum;
  }
  const int width = m + 2;
  int b = k > 0 ? t0 / k : 0;
  int tl = t0 - b * k;
  for (int t = t0; t < t1; ++t) {
    if (tl == k) {
      ++b;
      tl = 0;
    }
    const int p = ts.pos[t];
    const uint32_t fld = field_g(sq + b * rec_q, tl * width, width);
    ++tl;
    const uint32_t sgn = fld >> (m + 1), qv = fld & ((1u << (m + 1)) - 1u);
    const int ep = max((int)ts.mx[b * 4 + (p >> 5)], 1);
    uint32_t bits;
    if (FULL) {
      const int dd = ts.dbuf[t];
      const int w = min(8, 7 - m + dd);
      const uint32_t res = field_g(vres, rbit, w);
      rbit += w;
      const uint32_t sig = ((qv << w) | res) & 0xFFu;
      const uint32_t e = (sig & 0x80u) ? (uint32_t)(ep - dd) : 0u;
      bits = (sgn << 15) | (e << 7) | (sig & 0x7Fu);
    } else {
      bits = (__float_as_uint((float)qv * pow2_biased(ep - m)) >> 16) | (sgn << 15);
    }
    dst[b * bstride + p] = (uint16_t)bits;
  }
  if (FULL) {
    const int kp = CAS_BLK - k, pt = CAS_SB * kp, q2 = (pt + 31) >> 5;
    const int u0 = min(lane * q2, pt), u1 = min(u0 + q2, pt);
    __syncwarp();  // every lane is done with the distance stream and positions
    const bool enough_v = stage_unary(vexp, vnw, ts.us, lane, &long_codes) >= pt;
    expand_mask_positions<CAS_SB * CAS_BLK>(~mw, ts.pos, lane);
    __syncwarp();
    if (!enough_v) return false;
    UnaryCursor uc;
    uc.init(ts.us, unary_code_start(ts.us, vnw, u0));
    if (long_codes)
      runs_pruned_to_tile<true>(uc, ts.pos, pr, rec_pr, kp, u0, u1, lut, dst, bstride);
    else
      runs_pruned_to_tile<false>(uc, ts.pos, pr, rec_pr, kp, u0, u1, lut, dst, bstride);
  }
  __syncwarp();
  return true;
}

}  // namespace cas
