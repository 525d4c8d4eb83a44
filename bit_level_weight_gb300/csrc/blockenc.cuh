// blockenc.cuh - warp-level encoder of one 128-element block.
//
// A warp holds the block 4 values per lane (lane L: positions 4L..4L+3) and
// writes its records and codes:
//   value pruning (Cassandra blog review, section 3.1): keep the k values of
//     largest magnitude, ties to the lower position;
//   mantissa truncation (section 3.1): kept values give their m high mantissa
//     bits to the speculation data, the 7-m low bits to the verification data;
//   exponent coding (section 3.2): Cassandra-1 writes unary codes of the
//     frequency rank, Cassandra-2 an MX shared exponent per 32 positions with
//     the exponent distance d as a unary code in the verification data.
// Destination words must be zero where fields are written (records are
// OR-ed in with atomics because several lanes share a word).
#pragma once
#include "common.cuh"

namespace cas {

struct BlockDst {
  uint32_t* mask;    // 4 words
  uint32_t* rec_s;   // C-1: spec_sm record; C-2: spec_q record
  uint32_t* rec_lo;  // C-1 only
  uint32_t* rec_pr;
  uint8_t* mx;       // C-2 only: 4 bytes
};

struct Stream {
  uint32_t* words;
  uint64_t cursor;  // bit position of the next code (warp-uniform)
  uint64_t limit;   // words available
};

__device__ __forceinline__ void or_field(uint32_t* base, uint64_t bit, uint32_t v, int width, uint64_t limit) {
  if (width <= 0) return;
  uint64_t i = bit >> 5;
  int sh = (int)(bit & 31);
  if (i < limit) atomicOr(base + i, v << sh);
  if (sh + width > 32 && i + 1 < limit) atomicOr(base + i + 1, v >> (32 - sh));
}
__device__ __forceinline__ void set_msb_bit(uint32_t* base, uint64_t pos, uint64_t limit) {
  uint64_t i = pos >> 5;
  if (i < limit) atomicOr(base + i, 0x80000000u >> (pos & 31));
}

// Loads 4 consecutive bf16 of a block into v[0..3] (lane L: positions 4L..).
__device__ __forceinline__ void load_block4(const uint16_t* blk, int lane, uint32_t v[4]) {
  uint2 raw = __ldg(reinterpret_cast<const uint2*>(blk) + lane);
  v[0] = raw.x & 0xFFFFu;
  v[1] = raw.x >> 16;
  v[2] = raw.y & 0xFFFFu;
  v[3] = raw.y >> 16;
}

// Shared exponent E of this lane's 32-position group (lanes 8g..8g+7):
// largest biased exponent among kept values, 0 when none is kept.
__device__ __forceinline__ int group_shared_exp(const uint32_t v[4], uint32_t kept) {
  int e = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if ((kept >> j) & 1) e = max(e, (int)((v[j] >> 7) & 0xFF));
  e = max(e, __shfl_xor_sync(CAS_FULL, e, 1));
  e = max(e, __shfl_xor_sync(CAS_FULL, e, 2));
  e = max(e, __shfl_xor_sync(CAS_FULL, e, 4));
  return e;
}

// Code-length totals of one block for each variable-length stream.
struct BlockBits {
  int sexp, vexp, vd, vres;
};

template <int VAR>
__device__ __forceinline__ BlockBits block_lane_bits(const uint32_t v[4], uint32_t kept, int E, int m,
                                                     const uint8_t* roe) {
  BlockBits b{0, 0, 0, 0};
  int Ep = max(E, 1);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int e = (v[j] >> 7) & 0xFF;
    if ((kept >> j) & 1) {
      if (VAR == 1) {
        b.sexp += roe[e] + 1;
      } else {
        int d = Ep - max(e, 1);
        b.vd += d + 1;
        b.vres += min(8, 7 - m + d);
      }
    } else {
      b.vexp += roe[e] + 1;
    }
  }
  return b;
}

// Encodes one block: writes mask, records and appends codes to the streams.
// Stream cursors advance by the block's totals (warp-uniform).
template <int VAR>
__device__ void encode_block(const uint32_t v[4], int k, int m, const uint8_t* roe, const BlockDst& dst,
                             Stream& sexp, Stream& vexp, Stream& vd, Stream& vres, int lane, uint64_t rec_limit) {
  uint32_t key[4] = {v[0] & 0x7FFFu, v[1] & 0x7FFFu, v[2] & 0x7FFFu, v[3] & 0x7FFFu};
  uint32_t kept = select_block4(key, k, lane);
  uint32_t mw = gather_mask_word(kept, lane);
  if (lane < 4) dst.mask[lane] = mw;

  int nk = __popc(kept);
  int t = warp_incl_add(nk, lane) - nk;  // kept ordinal of the lane's first kept value
  int u = 4 * lane - t;                  // pruned ordinal of the lane's first pruned value
  int E = 0;
  if (VAR == 2) {
    E = group_shared_exp(v, kept);
    if ((lane & 7) == 0) dst.mx[lane >> 3] = (uint8_t)E;
  }
  int Ep = max(E, 1);
  BlockBits lb = block_lane_bits<VAR>(v, kept, E, m, roe);
  int s_sexp = warp_incl_add(lb.sexp, lane) - lb.sexp;
  int s_vexp = warp_incl_add(lb.vexp, lane) - lb.vexp;
  int s_vd = warp_incl_add(lb.vd, lane) - lb.vd;
  int s_vres = warp_incl_add(lb.vres, lane) - lb.vres;
  uint64_t p_sexp = sexp.cursor + s_sexp, p_vexp = vexp.cursor + s_vexp;
  uint64_t p_vd = vd.cursor + s_vd, p_vres = vres.cursor + s_vres;

#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t x = v[j];
    uint32_t s = x >> 15, e = (x >> 7) & 0xFF, f = x & 0x7F;
    if ((kept >> j) & 1) {
      if (VAR == 1) {
        uint32_t fhi = f >> (7 - m), flo = f & ((1u << (7 - m)) - 1u);
        or_field(dst.rec_s, (uint64_t)t * (m + 1), (s << m) | fhi, m + 1, rec_limit);
        or_field(dst.rec_lo, (uint64_t)t * (7 - m), flo, 7 - m, rec_limit);
        int r = roe[e];
        set_msb_bit(sexp.words, p_sexp + r, sexp.limit);
        p_sexp += r + 1;
      } else {
        int d = Ep - max((int)e, 1);
        int sh = 7 - m + d;
        uint32_t sig = (e ? 0x80u : 0u) | f;
        uint32_t q = sh < 8 ? (sig >> sh) : 0u;
        int w = min(sh, 8);
        or_field(dst.rec_s, (uint64_t)t * (m + 2), (s << (m + 1)) | q, m + 2, rec_limit);
        set_msb_bit(vd.words, p_vd + d, vd.limit);
        p_vd += d + 1;
        or_field(vres.words, p_vres, sig & ((1u << w) - 1u), w, vres.limit);
        p_vres += w;
      }
      ++t;
    } else {
      or_field(dst.rec_pr, (uint64_t)u * 8, (s << 7) | f, 8, rec_limit);
      int r = roe[e];
      set_msb_bit(vexp.words, p_vexp + r, vexp.limit);
      p_vexp += r + 1;
      ++u;
    }
  }
  sexp.cursor += __shfl_sync(CAS_FULL, s_sexp + lb.sexp, 31);
  vexp.cursor += __shfl_sync(CAS_FULL, s_vexp + lb.vexp, 31);
  vd.cursor += __shfl_sync(CAS_FULL, s_vd + lb.vd, 31);
  vres.cursor += __shfl_sync(CAS_FULL, s_vres + lb.vres, 31);
}

}  // namespace cas
