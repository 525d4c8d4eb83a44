// sbdecode.cuh - warp-level decoder of one superblock of an encoded tensor.
//
// Lane L < 4*nb owns mask word L of the superblock: block L>>2, positions
// 32*(L&3)..+31 of that block (for Cassandra-2 also exactly one shared-exponent
// group). A popcount prefix over the mask words gives each lane the ordinal of
// its first kept and first pruned value; the unary exponent streams are
// decoded once per superblock into shared memory, indexed by those ordinals.
//
// Draft value (Cassandra blog review, section 3.1): pruned -> 0, kept ->
// sign, exponent and the m high mantissa bits. Full value: kept values add the
// cut mantissa bits, pruned values come from the verification record and
// their own unary exponent code. Cassandra-2 (section 3.2): the draft value is
// q * 2^(E' - 127 - m); the full value rebuilds the 8-bit significand from q,
// the unary distance d and the residual bits.
#pragma once
#include "common.cuh"

namespace cas {

constexpr int kResWords = 256 + 2;  // worst case residual words of a superblock (8 x 128 x 8 bits / 32) + pad

struct SbScratch {
  uint8_t* code;   // [1024] C-1: exponent of kept ordinal; C-2: distance d of kept ordinal
  uint8_t* vcode;  // [1024] exponent of pruned ordinal
  uint32_t* res;   // [kResWords] C-2 residual stream of the superblock
};

struct SbInfo {
  int64_t n;
  int j, nb;
  int64_t gb0;
  uint32_t mw;  // this lane's mask word (0 for idle lanes)
  int o, uo;    // superblock ordinals of this lane's first kept / pruned value
  int rbit;     // C-2: bit offset of this lane's first residual in the staged stream
};

// Decodes the streams of superblock s into scratch. FULL also decodes the
// verification streams. Ends with __syncwarp().
template <int VAR, bool FULL>
__device__ __forceinline__ SbInfo sb_prepare(const WView& w, int64_t s, const uint8_t* lut, SbScratch sc, int lane) {
  SbInfo in;
  in.n = s / w.nsr;
  in.j = (int)(s % w.nsr);
  in.nb = min(CAS_SB, w.nbr - CAS_SB * in.j);
  in.gb0 = in.n * w.nbr + CAS_SB * in.j;
  in.mw = lane < 4 * in.nb ? __ldg(w.mask + in.gb0 * 4 + lane) : 0u;
  int cnt = __popc(in.mw);
  in.o = warp_incl_add(cnt, lane) - cnt;
  int pc = lane < 4 * in.nb ? 32 - cnt : 0;
  in.uo = warp_incl_add(pc, lane) - pc;
  in.rbit = 0;
  if (VAR == 1) {
    uint32_t a, b;
    stream_range(w.sidx, s, w.lim_sexp, a, b);
    warp_decode_unary(w.sexp + a, (int)(b - a), lut, sc.code, in.nb * w.k, lane);
  } else if (FULL) {
    uint32_t a, b;
    stream_range(w.vdidx, s, w.lim_vd, a, b);
    warp_decode_unary_raw(w.vd + a, (int)(b - a), sc.code, in.nb * w.k, lane);
    uint32_t ra, rb;
    stream_range(w.vresidx, s, w.lim_vres, ra, rb);
    int nres = min((int)(rb - ra), kResWords - 2);
    for (int i = lane; i < nres; i += 32) sc.res[i] = __ldg(w.vres + ra + i);
    if (lane < 2) sc.res[nres + lane] = 0u;
  }
  if (FULL) {
    uint32_t a, b;
    stream_range(w.vidx, s, w.lim_vexp, a, b);
    warp_decode_unary(w.vexp + a, (int)(b - a), lut, sc.vcode, in.nb * (CAS_BLK - w.k), lane);
  }
  __syncwarp();
  if (VAR == 2 && FULL) {
    int sum = 0;
    for (int i = 0; i < cnt; ++i) sum += min(8, 7 - w.m + (int)sc.code[in.o + i]);
    in.rbit = warp_incl_add(sum, lane) - sum;
  }
  return in;
}

// Walks the 32 positions of this lane's mask word in order; at(p) returns
// the bf16 bit pattern of position p (draft or, FULL, exact value).
template <int VAR, bool FULL>
struct SbRebuilder {
  const uint32_t *rs, *rl, *rp;
  const uint8_t *code, *vcode;
  const uint32_t* res;
  int m, o, uo, t, u, Ep, rb;
  float scale;
  uint32_t mw;

  __device__ __forceinline__ SbRebuilder(const WView& w, const SbInfo& in, SbScratch sc, int lane) {
    const int k = w.k;
    m = w.m;
    const int blk = lane >> 2, g = lane & 3;
    const int64_t gb = in.gb0 + blk;
    o = in.o;
    uo = in.uo;
    t = o - k * blk;
    u = uo - (CAS_BLK - k) * blk;
    rs = VAR == 1 ? w.ssm + gb * w.rec_sm : w.sq + gb * w.rec_q;
    rl = w.vlo + gb * w.rec_lo;
    rp = w.vpr + gb * w.rec_pr;
    code = sc.code;
    vcode = sc.vcode;
    res = sc.res;
    Ep = VAR == 2 ? max((int)__ldg(w.smx + gb * 4 + g), 1) : 1;
    scale = VAR == 2 ? pow2_biased(Ep - m) : 0.f;
    rb = in.rbit;
    mw = in.mw;
  }

  __device__ __forceinline__ uint32_t at(int p) {
    uint32_t bits = 0;
    if ((mw >> p) & 1u) {
      if (VAR == 1) {
        uint32_t fld = get_field(rs, t * (m + 1), m + 1);
        uint32_t f = (fld & ((1u << m) - 1u)) << (7 - m);
        if (FULL && m < 7) f |= get_field(rl, t * (7 - m), 7 - m);
        bits = ((fld >> m) << 15) | ((uint32_t)code[o] << 7) | f;
      } else {
        uint32_t fld = get_field(rs, t * (m + 2), m + 2);
        uint32_t s = (fld >> (m + 1)) & 1u, q = fld & ((1u << (m + 1)) - 1u);
        if (!FULL) {
          bits = (__float_as_uint((float)q * scale) >> 16) | (s << 15);
        } else {
          int d = code[o];
          int wd = min(7 - m + d, 8);
          uint32_t r = get_field(res, rb, wd);
          rb += wd;
          uint32_t sig = ((q << wd) | r) & 0xFFu;
          uint32_t e = (sig & 0x80u) ? (uint32_t)(Ep - d) : 0u;
          bits = (s << 15) | (e << 7) | (sig & 0x7Fu);
        }
      }
      ++t;
      ++o;
    } else {
      if (FULL) {
        uint32_t byte = (__ldg(rp + (u >> 2)) >> ((u & 3) * 8)) & 0xFFu;
        bits = ((byte >> 7) << 15) | ((uint32_t)vcode[uo] << 7) | (byte & 0x7Fu);
      }
      ++u;
      ++uo;
    }
    return bits;
  }
};

// Rebuilds the 32 values of this lane's mask word as bf16 bit patterns,
// packed in pairs (out[i] = value 2i | value 2i+1 << 16).
template <int VAR, bool FULL>
__device__ __forceinline__ void sb_rebuild_word(const WView& w, const SbInfo& in, SbScratch sc, int lane,
                                                uint32_t out[16]) {
  SbRebuilder<VAR, FULL> rb(w, in, sc, lane);
#pragma unroll
  for (int p = 0; p < 32; ++p) {
    const uint32_t bits = rb.at(p);
    if (p & 1)
      out[p >> 1] |= bits << 16;
    else
      out[p >> 1] = bits;
  }
}

// Same values stored one by one to dst[0..31] (a rolled loop: little register
// pressure, for fallback paths inside register-heavy kernels).
template <int VAR, bool FULL>
__device__ __forceinline__ void sb_rebuild_store(const WView& w, const SbInfo& in, SbScratch sc, int lane,
                                                 uint16_t* dst) {
  SbRebuilder<VAR, FULL> rb(w, in, sc, lane);
#pragma unroll 1
  for (int p = 0; p < 32; ++p) dst[p] = (uint16_t)rb.at(p);
}

}  // namespace cas
