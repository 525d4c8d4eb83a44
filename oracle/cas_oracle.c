/*
 * cas_oracle.c - plain, slow CPU oracle of the Cassandra bit-level split.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header, table or constant with the CUDA library;
 * the on-disk format below is restated here from its definition.
 *
 * Sources (the method is described only in prose; no code is printed):
 *   [B3.1] Cassandra blog review, marsggbo.github.io/blog/2026/20260722-cassandra,
 *          section 3.1: unstructured value pruning keeps the most salient values,
 *          mantissa truncation cuts the low mantissa bits of the kept values, and
 *          both the pruned values and the cut bits go to the verification data;
 *          the draft loads only speculation data and zero-fills the rest; the
 *          target merges both losslessly.
 *   [B3.2] same page, section 3.2: the exponent is the bottleneck; Cassandra-1
 *          codes it with frequency-ranked unary codes ("count zeros until a
 *          one"), Cassandra-2 uses an MX-style shared exponent.
 *   [F11]  Cassandra paper (arXiv 2605.26558), Fig. 11 caption: data is managed
 *          in superblocks.
 *
 * Readings where the pages are silent (each one is listed with its reason in the
 * design notes of the repository):
 *   - saliency key = bf16 bits & 0x7FFF (monotone in |x| for finite values);
 *     k largest keys kept per 128-element block, ties to the lower position;
 *   - truncation toward zero (the cut bits are stored verbatim);
 *   - one rank table per tensor: exponents sorted by (count desc, exponent asc);
 *     rank r is coded as r zero bits then a one bit, no length cap;
 *   - Cassandra-2: 32-position groups, shared E = max biased exponent of the
 *     group's kept values, element = sign + (m+1) magnitude bits;
 *   - superblock = 8 consecutive blocks of one row; variable-length streams are
 *     word aligned per superblock and indexed by u32 word offsets;
 *   - all sections in one buffer, each on a 256-byte boundary, padding zero.
 *
 * Style: every step is written out bit by bit, with no blocking, fusion or
 * table tricks, so that it can be checked by eye against the definitions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define BLK 128           /* elements per block (value-pruning granule)        */
#define SB_BLOCKS 8       /* blocks per superblock                             */
#define GROUP 32          /* Cassandra-2 shared-exponent group                 */

/* Section indices of the encoded buffer (format definition). */
enum {
  S_MASK = 0,        /* u32[nblk][4] keep mask                                 */
  S_SPEC_SM,         /* C-1: per block ceil(k(m+1)/32) words, (s<<m)|f_hi      */
  S_SPEC_EXP,        /* C-1: unary codes of kept exponents, MSB-first          */
  S_SPEC_SBIDX,      /* C-1: u32[nsb+1] word offsets into S_SPEC_EXP           */
  S_SPEC_MX,         /* C-2: u8[nblk][4] shared exponent per group             */
  S_SPEC_Q,          /* C-2: per block ceil(k(m+2)/32) words, (s<<(m+1))|q     */
  S_VER_LO,          /* C-1: per block ceil(k(7-m)/32) words, f_lo             */
  S_VER_D,           /* C-2: unary codes of d, MSB-first                       */
  S_VER_D_SBIDX,     /* C-2: u32[nsb+1]                                        */
  S_VER_RES,         /* C-2: residual significand bits, LSB-first              */
  S_VER_RES_SBIDX,   /* C-2: u32[nsb+1]                                        */
  S_VER_PR,          /* both: per block ceil((128-k)/4) words, (s<<7)|f bytes  */
  S_VER_EXP,         /* both: unary codes of pruned exponents, MSB-first       */
  S_VER_SBIDX,       /* both: u32[nsb+1]                                       */
  NSEC
};

enum { ORC_OK = 0, ORC_INVALID = -1, ORC_SHAPE = -2, ORC_NONFINITE = -3, ORC_CORRUPT = -7 };

/* ---------------------------------------------------------------- bf16 fields */
static int bf_sign(uint16_t b) { return (b >> 15) & 1; }
static int bf_exp(uint16_t b) { return (b >> 7) & 0xFF; }
static int bf_man(uint16_t b) { return b & 0x7F; }

static double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Exact conversion of a value known to be representable in bf16.
 * Returns 0xFFFF-tagged failure through *ok when it is not. */
static uint16_t f64_to_bf16_exact(double v, int* ok) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((double)f != v || (u & 0xFFFFu) != 0) *ok = 0;
  return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- bit I/O
 * Two bit orders are used:
 *   LSB-first: bit i of the stream is bit (i & 31) of word i >> 5.
 *   MSB-first: bit i of the stream is bit 31 - (i & 31) of word i >> 5, so a
 *              count of leading zeros walks a unary code.                    */
static void put_lsb(uint32_t* w, uint64_t pos, int bit) {
  if (bit) w[pos >> 5] |= 1u << (pos & 31);
}
static int get_lsb(const uint32_t* w, uint64_t pos) { return (w[pos >> 5] >> (pos & 31)) & 1; }
static void put_msb(uint32_t* w, uint64_t pos, int bit) {
  if (bit) w[pos >> 5] |= 0x80000000u >> (pos & 31);
}
static int get_msb(const uint32_t* w, uint64_t pos) { return (w[pos >> 5] >> (31 - (pos & 31))) & 1; }

static void put_field(uint32_t* w, uint64_t off, uint32_t v, int width) {
  for (int i = 0; i < width; ++i) put_lsb(w, off + (uint64_t)i, (v >> i) & 1);
}
static uint32_t get_field(const uint32_t* w, uint64_t off, int width) {
  uint32_t v = 0;
  for (int i = 0; i < width; ++i) v |= (uint32_t)get_lsb(w, off + (uint64_t)i) << i;
  return v;
}
/* unary code of r: r zero bits then a one bit ([B3.2] "count zeros until a one") */
static uint64_t put_unary(uint32_t* w, uint64_t pos, int r) {
  for (int i = 0; i < r; ++i) put_msb(w, pos + (uint64_t)i, 0);
  put_msb(w, pos + (uint64_t)r, 1);
  return (uint64_t)r + 1;
}
/* reads one code; returns -1 when more than 255 zeros are seen or the stream
 * would be overrun (limit is the number of valid bits) */
static int get_unary(const uint32_t* w, uint64_t* pos, uint64_t limit) {
  int r = 0;
  while (1) {
    if (*pos >= limit) return -1;
    int b = get_msb(w, *pos);
    (*pos)++;
    if (b) return r;
    if (++r > 255) return -1;
  }
}

static uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
static uint64_t align256(uint64_t a) { return (a + 255) & ~(uint64_t)255; }

/* ---------------------------------------------------------------- rank table
 * [B3.2]: frequent exponents get short codes. Histogram of the biased
 * exponent over every element of the tensor.                                */
void orc_exp_hist(const uint16_t* w, int64_t n, uint64_t* counts) {
  for (int e = 0; e < 256; ++e) counts[e] = 0;
  for (int64_t i = 0; i < n; ++i) counts[bf_exp(w[i])]++;
}

/* Sort exponents by (count desc, exponent asc). Plain selection sort. Unseen
 * exponents fall to the tail in ascending order, so every finite input is
 * codable. */
void orc_rank_table(const uint64_t* counts, uint8_t* exp_of_rank, uint8_t* rank_of_exp) {
  int used[256];
  for (int e = 0; e < 256; ++e) used[e] = 0;
  for (int r = 0; r < 256; ++r) {
    int best = -1;
    for (int e = 0; e < 256; ++e) {
      if (used[e]) continue;
      if (best < 0 || counts[e] > counts[best]) best = e; /* ties keep the lower e */
    }
    used[best] = 1;
    exp_of_rank[r] = (uint8_t)best;
    rank_of_exp[best] = (uint8_t)r;
  }
}

/* ---------------------------------------------------------------- value pruning
 * [B3.1] keep the most salient values. Element i of a block is kept iff fewer
 * than k elements outrank it, where j outranks i when key_j > key_i, or when
 * key_j == key_i and j < i. key = bits & 0x7FFF. B is a parameter so tests can
 * brute-force tiny blocks; the format always uses B = 128. */
void orc_select_block(const uint16_t* blk, int B, int k, uint8_t* keep) {
  for (int i = 0; i < B; ++i) {
    int ki = blk[i] & 0x7FFF, above = 0;
    for (int j = 0; j < B; ++j) {
      int kj = blk[j] & 0x7FFF;
      if (kj > ki || (kj == ki && j < i)) above++;
    }
    keep[i] = (uint8_t)(above < k);
  }
}

/* ---------------------------------------------------------------- Cassandra-2 helpers
 * [B3.2] MX shared exponent. E = max biased exponent over the group's kept
 * values (0 when none are kept); E' = max(E,1). A kept value with biased
 * exponent e has effective exponent e' = max(e,1) and 8-bit significand
 * sig = (e != 0 ? 0x80 : 0) | f, i.e. |x| = sig * 2^(e' - 134).
 * d = E' - e' >= 0; the draft keeps q = sig >> (7 - m + d), which has m+1 bits;
 * the verification data keeps d (unary) and the w = min(8, 7-m+d) bits below. */
static int group_E(const uint16_t* blk, const uint8_t* keep, int g) {
  int E = 0;
  for (int p = g * GROUP; p < (g + 1) * GROUP; ++p)
    if (keep[p] && bf_exp(blk[p]) > E) E = bf_exp(blk[p]);
  return E;
}
static int eff_exp(int e) { return e > 0 ? e : 1; }
static int sig8(uint16_t b) { return (bf_exp(b) != 0 ? 0x80 : 0) | bf_man(b); }

/* ---------------------------------------------------------------- geometry */
typedef struct {
  int64_t N, K, nbr, nblk, nsr, nsb;
  int variant, k, m;
  uint64_t rec_sm, rec_q, rec_lo, rec_pr; /* words per block */
} geom;

static int make_geom(geom* g, int64_t N, int64_t K, int variant, int k, int m) {
  if (N < 0 || K < 0 || (variant != 1 && variant != 2) || k < 0 || k > BLK || m < 0 || m > 7)
    return ORC_INVALID;
  if (K % BLK) return ORC_SHAPE;
  g->N = N; g->K = K; g->variant = variant; g->k = k; g->m = m;
  g->nbr = K / BLK;
  g->nblk = N * g->nbr;
  g->nsr = (g->nbr + SB_BLOCKS - 1) / SB_BLOCKS;
  g->nsb = N * g->nsr;
  g->rec_sm = ceil_div((uint64_t)k * (uint64_t)(m + 1), 32);
  g->rec_q = ceil_div((uint64_t)k * (uint64_t)(m + 2), 32);
  g->rec_lo = ceil_div((uint64_t)k * (uint64_t)(7 - m), 32);
  g->rec_pr = ceil_div((uint64_t)(BLK - k) * 8, 32);
  return ORC_OK;
}
/* first and one-past-last global block id of superblock s */
static void sb_blocks(const geom* g, int64_t s, int64_t* b0, int64_t* b1) {
  int64_t n = s / g->nsr, j = s % g->nsr;
  int64_t lo = j * SB_BLOCKS, hi = lo + SB_BLOCKS;
  if (hi > g->nbr) hi = g->nbr;
  *b0 = n * g->nbr + lo;
  *b1 = n * g->nbr + hi;
}

/* ---------------------------------------------------------------- encode
 * Writes the sections of one tensor (W row-major [N][K]) with the given rank
 * table. When buf is NULL only off/len/total are computed. Returns ORC_* .  */
int orc_encode(const uint16_t* W, int64_t N, int64_t K, int variant, int k, int m,
               const uint8_t* rank_of_exp, uint8_t* buf, uint64_t* off, uint64_t* len,
               uint64_t* total) {
  geom g;
  int st = make_geom(&g, N, K, variant, k, m);
  if (st) return st;
  for (int64_t i = 0; i < N * K; ++i)
    if (bf_exp(W[i]) == 255) return ORC_NONFINITE;

  uint8_t* keep = (uint8_t*)malloc((size_t)(N * K > 0 ? N * K : 1));
  for (int64_t b = 0; b < g.nblk; ++b) orc_select_block(W + b * BLK, BLK, k, keep + b * BLK);

  /* pass 1: bit length of every variable-length stream of every superblock */
  uint64_t* bits_sexp = (uint64_t*)calloc((size_t)g.nsb + 1, 8);
  uint64_t* bits_vexp = (uint64_t*)calloc((size_t)g.nsb + 1, 8);
  uint64_t* bits_vd = (uint64_t*)calloc((size_t)g.nsb + 1, 8);
  uint64_t* bits_vres = (uint64_t*)calloc((size_t)g.nsb + 1, 8);
  for (int64_t s = 0; s < g.nsb; ++s) {
    int64_t b0, b1;
    sb_blocks(&g, s, &b0, &b1);
    for (int64_t b = b0; b < b1; ++b) {
      const uint16_t* blk = W + b * BLK;
      const uint8_t* kb = keep + b * BLK;
      for (int p = 0; p < BLK; ++p) {
        int e = bf_exp(blk[p]);
        if (!kb[p]) {
          bits_vexp[s] += (uint64_t)rank_of_exp[e] + 1;
        } else if (variant == 1) {
          bits_sexp[s] += (uint64_t)rank_of_exp[e] + 1;
        } else {
          int Ep = eff_exp(group_E(blk, kb, p / GROUP));
          int d = Ep - eff_exp(e);
          int sh = 7 - m + d;
          bits_vd[s] += (uint64_t)d + 1;
          bits_vres[s] += (uint64_t)(sh < 8 ? sh : 8);
        }
      }
    }
  }
  /* word offsets (exclusive scan of word-rounded lengths) */
  uint64_t* idx_sexp = (uint64_t*)calloc((size_t)g.nsb + 1, 8);
  uint64_t* idx_vexp = (uint64_t*)calloc((size_t)g.nsb + 1, 8);
  uint64_t* idx_vd = (uint64_t*)calloc((size_t)g.nsb + 1, 8);
  uint64_t* idx_vres = (uint64_t*)calloc((size_t)g.nsb + 1, 8);
  for (int64_t s = 0; s < g.nsb; ++s) {
    idx_sexp[s + 1] = idx_sexp[s] + ceil_div(bits_sexp[s], 32);
    idx_vexp[s + 1] = idx_vexp[s] + ceil_div(bits_vexp[s], 32);
    idx_vd[s + 1] = idx_vd[s] + ceil_div(bits_vd[s], 32);
    idx_vres[s + 1] = idx_vres[s] + ceil_div(bits_vres[s], 32);
  }
  int too_big = idx_sexp[g.nsb] > 0xFFFFFFFFull || idx_vexp[g.nsb] > 0xFFFFFFFFull ||
                idx_vd[g.nsb] > 0xFFFFFFFFull || idx_vres[g.nsb] > 0xFFFFFFFFull;

  uint64_t nb = (uint64_t)g.nblk, nsbi = (uint64_t)g.nsb + 1;
  for (int i = 0; i < NSEC; ++i) len[i] = 0;
  len[S_MASK] = nb * 16;
  len[S_VER_PR] = nb * g.rec_pr * 4;
  len[S_VER_EXP] = idx_vexp[g.nsb] * 4;
  len[S_VER_SBIDX] = nsbi * 4;
  if (variant == 1) {
    len[S_SPEC_SM] = nb * g.rec_sm * 4;
    len[S_SPEC_EXP] = idx_sexp[g.nsb] * 4;
    len[S_SPEC_SBIDX] = nsbi * 4;
    len[S_VER_LO] = nb * g.rec_lo * 4;
  } else {
    len[S_SPEC_MX] = nb * 4;
    len[S_SPEC_Q] = nb * g.rec_q * 4;
    len[S_VER_D] = idx_vd[g.nsb] * 4;
    len[S_VER_D_SBIDX] = nsbi * 4;
    len[S_VER_RES] = idx_vres[g.nsb] * 4;
    len[S_VER_RES_SBIDX] = nsbi * 4;
  }
  uint64_t run = 0;
  for (int i = 0; i < NSEC; ++i) {
    off[i] = align256(run);
    run = off[i] + len[i];
  }
  *total = align256(run);

  if (buf && !too_big) {
    memset(buf, 0, (size_t)*total);
    uint32_t* mask = (uint32_t*)(buf + off[S_MASK]);
    uint32_t* ssm = (uint32_t*)(buf + off[S_SPEC_SM]);
    uint32_t* sexp = (uint32_t*)(buf + off[S_SPEC_EXP]);
    uint32_t* sidx = (uint32_t*)(buf + off[S_SPEC_SBIDX]);
    uint8_t* smx = buf + off[S_SPEC_MX];
    uint32_t* sq = (uint32_t*)(buf + off[S_SPEC_Q]);
    uint32_t* vlo = (uint32_t*)(buf + off[S_VER_LO]);
    uint32_t* vd = (uint32_t*)(buf + off[S_VER_D]);
    uint32_t* vdidx = (uint32_t*)(buf + off[S_VER_D_SBIDX]);
    uint32_t* vres = (uint32_t*)(buf + off[S_VER_RES]);
    uint32_t* vresidx = (uint32_t*)(buf + off[S_VER_RES_SBIDX]);
    uint32_t* vpr = (uint32_t*)(buf + off[S_VER_PR]);
    uint32_t* vexp = (uint32_t*)(buf + off[S_VER_EXP]);
    uint32_t* vidx = (uint32_t*)(buf + off[S_VER_SBIDX]);

    for (int64_t s = 0; s <= g.nsb; ++s) {
      vidx[s] = (uint32_t)idx_vexp[s];
      if (variant == 1) {
        sidx[s] = (uint32_t)idx_sexp[s];
      } else {
        vdidx[s] = (uint32_t)idx_vd[s];
        vresidx[s] = (uint32_t)idx_vres[s];
      }
    }
    for (int64_t s = 0; s < g.nsb; ++s) {
      int64_t b0, b1;
      sb_blocks(&g, s, &b0, &b1);
      uint64_t p_sexp = idx_sexp[s] * 32, p_vexp = idx_vexp[s] * 32;
      uint64_t p_vd = idx_vd[s] * 32, p_vres = idx_vres[s] * 32;
      for (int64_t b = b0; b < b1; ++b) {
        const uint16_t* blk = W + b * BLK;
        const uint8_t* kb = keep + b * BLK;
        int Eg[4] = {0, 0, 0, 0};
        if (variant == 2)
          for (int gi = 0; gi < 4; ++gi) {
            Eg[gi] = group_E(blk, kb, gi);
            smx[b * 4 + gi] = (uint8_t)Eg[gi];
          }
        int t = 0, u = 0; /* ordinal among kept / pruned in this block */
        for (int p = 0; p < BLK; ++p) {
          uint16_t x = blk[p];
          int s_ = bf_sign(x), e = bf_exp(x), f = bf_man(x);
          if (kb[p]) {
            put_lsb(mask + b * 4, (uint64_t)p, 1);
            if (variant == 1) {
              int fhi = f >> (7 - m), flo = f & ((1 << (7 - m)) - 1);
              put_field(ssm + b * g.rec_sm, (uint64_t)t * (uint64_t)(m + 1),
                        (uint32_t)((s_ << m) | fhi), m + 1);
              put_field(vlo + b * g.rec_lo, (uint64_t)t * (uint64_t)(7 - m), (uint32_t)flo, 7 - m);
              p_sexp += put_unary(sexp, p_sexp, rank_of_exp[e]);
            } else {
              int Ep = eff_exp(Eg[p / GROUP]);
              int d = Ep - eff_exp(e);
              int sh = 7 - m + d;
              int sg = sig8(x);
              int q = sh < 8 ? (sg >> sh) : 0;
              int w = sh < 8 ? sh : 8;
              put_field(sq + b * g.rec_q, (uint64_t)t * (uint64_t)(m + 2),
                        (uint32_t)((s_ << (m + 1)) | q), m + 2);
              p_vd += put_unary(vd, p_vd, d);
              put_field(vres, p_vres, (uint32_t)(sg & ((1 << w) - 1)), w);
              p_vres += (uint64_t)w;
            }
            t++;
          } else {
            put_field(vpr + b * g.rec_pr, (uint64_t)u * 8, (uint32_t)((s_ << 7) | f), 8);
            p_vexp += put_unary(vexp, p_vexp, rank_of_exp[e]);
            u++;
          }
        }
      }
    }
  }
  free(keep);
  free(bits_sexp); free(bits_vexp); free(bits_vd); free(bits_vres);
  free(idx_sexp); free(idx_vexp); free(idx_vd); free(idx_vres);
  return too_big ? ORC_INVALID : ORC_OK;
}

/* ---------------------------------------------------------------- draft values by definition
 * The speculation value of every element computed straight from W, without the
 * encoded form. Cassandra-1 [B3.1]: pruned -> +0, kept -> mantissa truncated to
 * its m high bits. Cassandra-2 [B3.2]: kept -> sign * floor(|x| / u) * u with
 * u = 2^(E' - 127 - m), evaluated in double precision. */
int orc_draft_values(const uint16_t* W, int64_t N, int64_t K, int variant, int k, int m,
                     uint16_t* out) {
  geom g;
  int st = make_geom(&g, N, K, variant, k, m);
  if (st) return st;
  uint8_t keep[BLK];
  int ok = 1;
  for (int64_t b = 0; b < g.nblk; ++b) {
    const uint16_t* blk = W + b * BLK;
    uint16_t* ob = out + b * BLK;
    orc_select_block(blk, BLK, k, keep);
    for (int p = 0; p < BLK; ++p) {
      if (!keep[p]) {
        ob[p] = 0;
        continue;
      }
      if (variant == 1) {
        ob[p] = (uint16_t)(blk[p] & ~((1u << (7 - m)) - 1u));
      } else {
        int Ep = eff_exp(group_E(blk, keep, p / GROUP));
        double a = fabs(bf16_to_f64(blk[p]));
        double u = ldexp(1.0, Ep - 127 - m);
        double v = floor(a / u) * u;
        if (bf_sign(blk[p])) v = -v;
        ob[p] = f64_to_bf16_exact(v, &ok);
      }
    }
  }
  return ok ? ORC_OK : ORC_CORRUPT;
}

/* ---------------------------------------------------------------- decode
 * Parses an encoded buffer. full = 0 gives the draft (speculation data only,
 * zero-filled), full = 1 merges speculation and verification data back to the
 * original bits. Returns ORC_CORRUPT on a malformed stream. */
int orc_decode(const uint8_t* buf, const uint64_t* off, int64_t N, int64_t K, int variant, int k,
               int m, const uint8_t* exp_of_rank, int full, uint16_t* out) {
  geom g;
  int st = make_geom(&g, N, K, variant, k, m);
  if (st) return st;
  const uint32_t* mask = (const uint32_t*)(buf + off[S_MASK]);
  const uint32_t* ssm = (const uint32_t*)(buf + off[S_SPEC_SM]);
  const uint32_t* sexp = (const uint32_t*)(buf + off[S_SPEC_EXP]);
  const uint32_t* sidx = (const uint32_t*)(buf + off[S_SPEC_SBIDX]);
  const uint8_t* smx = buf + off[S_SPEC_MX];
  const uint32_t* sq = (const uint32_t*)(buf + off[S_SPEC_Q]);
  const uint32_t* vlo = (const uint32_t*)(buf + off[S_VER_LO]);
  const uint32_t* vd = (const uint32_t*)(buf + off[S_VER_D]);
  const uint32_t* vdidx = (const uint32_t*)(buf + off[S_VER_D_SBIDX]);
  const uint32_t* vres = (const uint32_t*)(buf + off[S_VER_RES]);
  const uint32_t* vresidx = (const uint32_t*)(buf + off[S_VER_RES_SBIDX]);
  const uint32_t* vpr = (const uint32_t*)(buf + off[S_VER_PR]);
  const uint32_t* vexp = (const uint32_t*)(buf + off[S_VER_EXP]);
  const uint32_t* vidx = (const uint32_t*)(buf + off[S_VER_SBIDX]);
  int ok = 1;

  for (int64_t s = 0; s < g.nsb; ++s) {
    int64_t b0, b1;
    sb_blocks(&g, s, &b0, &b1);
    uint64_t p_sexp = 0, e_sexp = 0, p_vexp = 0, e_vexp = 0;
    uint64_t p_vd = 0, e_vd = 0, p_vres = 0, e_vres = 0;
    if (variant == 1) { p_sexp = (uint64_t)sidx[s] * 32; e_sexp = (uint64_t)sidx[s + 1] * 32; }
    else {
      p_vd = (uint64_t)vdidx[s] * 32; e_vd = (uint64_t)vdidx[s + 1] * 32;
      p_vres = (uint64_t)vresidx[s] * 32; e_vres = (uint64_t)vresidx[s + 1] * 32;
    }
    p_vexp = (uint64_t)vidx[s] * 32; e_vexp = (uint64_t)vidx[s + 1] * 32;
    for (int64_t b = b0; b < b1; ++b) {
      uint16_t* ob = out + b * BLK;
      int t = 0, u = 0, nkept = 0;
      for (int p = 0; p < BLK; ++p) nkept += get_lsb(mask + b * 4, (uint64_t)p);
      if (nkept != k) return ORC_CORRUPT;
      for (int p = 0; p < BLK; ++p) {
        if (get_lsb(mask + b * 4, (uint64_t)p)) {
          if (variant == 1) {
            uint32_t fs = get_field(ssm + b * g.rec_sm, (uint64_t)t * (uint64_t)(m + 1), m + 1);
            int s_ = (fs >> m) & 1, fhi = fs & ((1u << m) - 1);
            int r = get_unary(sexp, &p_sexp, e_sexp);
            if (r < 0) return ORC_CORRUPT;
            int e = exp_of_rank[r];
            int f = fhi << (7 - m);
            if (full) f |= (int)get_field(vlo + b * g.rec_lo, (uint64_t)t * (uint64_t)(7 - m), 7 - m);
            ob[p] = (uint16_t)((s_ << 15) | (e << 7) | f);
          } else {
            int Ep = eff_exp(smx[b * 4 + p / GROUP]);
            uint32_t fs = get_field(sq + b * g.rec_q, (uint64_t)t * (uint64_t)(m + 2), m + 2);
            int s_ = (fs >> (m + 1)) & 1, q = fs & ((1u << (m + 1)) - 1);
            if (!full) {
              double v = ldexp((double)q, Ep - 127 - m);
              if (s_) v = -v;
              ob[p] = f64_to_bf16_exact(v, &ok);
            } else {
              int d = get_unary(vd, &p_vd, e_vd);
              if (d < 0 || d >= Ep) return ORC_CORRUPT;
              int sh = 7 - m + d, w = sh < 8 ? sh : 8;
              if (p_vres + (uint64_t)w > e_vres) return ORC_CORRUPT;
              int res = (int)get_field(vres, p_vres, w);
              p_vres += (uint64_t)w;
              int sg = ((q << w) | res) & 0xFF;
              int e = (sg & 0x80) ? Ep - d : 0;
              if ((sg & 0x80) == 0 && d != Ep - 1) return ORC_CORRUPT;
              ob[p] = (uint16_t)((s_ << 15) | (e << 7) | (sg & 0x7F));
            }
          }
          t++;
        } else {
          if (!full) {
            ob[p] = 0;
          } else {
            int sf = (int)get_field(vpr + b * g.rec_pr, (uint64_t)u * 8, 8);
            int r = get_unary(vexp, &p_vexp, e_vexp);
            if (r < 0) return ORC_CORRUPT;
            ob[p] = (uint16_t)(((sf >> 7) << 15) | (exp_of_rank[r] << 7) | (sf & 0x7F));
          }
          u++;
        }
      }
    }
  }
  return ok ? ORC_OK : ORC_CORRUPT;
}

/* ---------------------------------------------------------------- GEMV / GEMM
 * y[v][n] = sum_k A[n][k] * x[v][k], every product and sum in double. A and x
 * are bf16 bit patterns. Also returns the error normaliser sum_k |A x|. This is
 * the plain definition; the draft GEMV feeds it the draft values, the verify
 * GEMM the original values. */
void orc_matvec(const uint16_t* A, int64_t N, int64_t K, const uint16_t* x, int nvec, double* y,
                double* absdot) {
  for (int v = 0; v < nvec; ++v)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t kk = 0; kk < K; ++kk) {
        double p = bf16_to_f64(A[n * K + kk]) * bf16_to_f64(x[(int64_t)v * K + kk]);
        acc += p;
        aacc += fabs(p);
      }
      y[(int64_t)v * N + n] = acc;
      if (absdot) absdot[(int64_t)v * N + n] = aacc;
    }
}
