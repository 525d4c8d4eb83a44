// gemv.cu - fused draft decode + GEMV: y[v][n] = sum_k D(W)[n][k] x[v][k].
//
// Reads only the speculation sections (mask, sign/mantissa records, unary
// exponent stream and its superblock index; Cassandra-2: shared exponents and
// q records). The draft does full-size FLOPs and saves bandwidth (Cassandra
// blog review, section 3.1), so the kernel moves only the speculation bytes
// and its cost is the integer work of decoding them.
//
// Every kernel maps one warp to one superblock (row n, up to 8 blocks), stages
// x once per CTA by a TMA bulk copy, and adds its partial sums to y with one
// fp32 atomic per (superblock, vector); y is cleared first. Kernels:
//   draft_gemv_fast_kernel   Cassandra-1, k = 64, m = 3, whole superblocks:
//                            16 ordinals per lane, unary cursor over the
//                            stream staged in shared memory (lanedec.cuh);
//   draft_gemv_fast2_kernel  Cassandra-2, k = 64, m = 3, up to 2 vectors;
//   draft_gemv_runs_kernel   any k, m, both variants, whole superblocks: runs
//                            of ordinals across blocks;
//   draft_gemv_kernel        rows ending in a partial superblock: per-lane
//                            runs with cursors over '1' bits of the mask and
//                            of the stream read from global memory (below).
// draft_gemv_kernel: a lane locates the start of its run - the mask word and
// bit of its first kept position, and the bit after the t0-th '1' of the unary
// exponent stream - with warp popcount prefixes, shuffle binary searches and
// a popcount select within a word, then walks it with two cursors over '1'
// bits held in two-word windows: one over the bit-reversed mask (next kept
// position), one over the unary stream (code end; rank = distance from the
// previous end). The rank table gives exponent << 23, OR-ed with the sign and
// mantissa field into an fp32 value multiplied with x.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "lanedec.cuh"
#include "sbdecode.cuh"
#include "wordlane.cuh"
#include "blockwalk.cuh"

namespace cas {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxVec = 4;

struct GemvArgs {
  WView w;
  Lut lut;
  const uint16_t* x;
  float* y;
  int sexp_words;  // words of the unary exponent section (read bound)
  // An fp32 input transformed in the x staging (lane-per-block kernel only),
  // the bf16 result also written to xn by CTA 0. xop: 0 none (x is bf16),
  // 1 RMSNorm, x = bf16(xf / sqrt(mean(xf^2) + eps) * gamma); 2 rounding,
  // x = bf16(xf); 3 SiLU * mul, x = bf16(silu(g) * u) of xf rows [g | u] of 2K.
  int xop = 0;
  const float* xf = nullptr;
  const uint16_t* gamma = nullptr;
  uint16_t* xn = nullptr;
  float eps = 0.f;
  // How the lane-per-block kernel writes y: 0, fp32 atomics into a y the
  // caller cleared; rows of exactly 32 blocks (one chunk per row, so one warp
  // owns each row's sum) 1, a plain store, or 2, a plain add.
  int ymode = 0;
};

// Set when a bounded wait on the x staging copy gave up (read by
// cas_device_status).
__device__ int g_gemv_wait_status = 0;
// Spin limit of the first wait on the x staging copy (the wait after it keeps
// the full limit); lowered only by the failure-detection test hook.
__device__ uint32_t g_first_wait_spins = kSpinLimit;

constexpr int kRecWords = CAS_SB * 32 + 2;  // staged records of a superblock (+pad)
constexpr int kMaskWords = 40;                 // bit-reversed mask words (+zero pad)
constexpr int kWarpWords = kRecWords + kMaskWords;

// Cursor over the '1' bits of an MSB-first bitstream held as a two-word
// window (h: current word with consumed bits cleared, l: next word). `base`
// is the stream bit index of h's MSB. Used for the mask (bit-reversed, a '1'
// per kept position) and for the unary codes (a '1' ends each code).
struct OnesCursor {
  uint32_t h, l;
  int base;
  // bit index of the next '1', consuming it; `more` fetches the following
  // word (stream bit index base + 64) when the window shifts.
  template <class More>
  __device__ __forceinline__ int next(More more) {
    for (int guard = 0; h == 0 && guard < 64; ++guard) {  // window word exhausted
      h = l;
      l = more(base + 64);
      base += 32;
    }
    int z = __clz(h);
    h &= 0x7FFFFFFFu >> z;
    return base + z;
  }
};

template <int VAR, int NV>
__global__ void __launch_bounds__(kThreads) draft_gemv_kernel(GemvArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  const WView& w = a.w;
  const int K = (int)w.K;
  const int xbytes = NV * K * 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + xbytes);
  uint32_t* lut23 = reinterpret_cast<uint32_t*>(smem + xbytes + 16);  // exponent << 23 by rank
  uint32_t* wbuf = lut23 + 256 + warp * kWarpWords;
  uint32_t* s_rec = wbuf;                 // sign/mantissa records of the superblock
  uint32_t* s_mw = wbuf + kRecWords;      // bit-reversed mask words

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_tx(bar, (uint32_t)xbytes);
    bulk_g2s(xs, a.x, (uint32_t)xbytes, bar);
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) lut23[i] = (uint32_t)a.lut.v[i] << 23;
  if (lane < kMaskWords - 32) s_mw[32 + lane] = 0u;
  bool ok = mbar_wait_bounded(bar, 0, g_first_wait_spins);
  if (!__syncthreads_and(ok)) {
    if (threadIdx.x == 0) atomicExch(&g_gemv_wait_status, CAS_ERR_TIMEOUT);
    mbar_wait_bounded(bar, 0);  // let an in-flight copy land before the CTA exits
    return;
  }

  const int k = w.k, m = w.m, nsr = w.nsr, nbr = w.nbr;
  const int width = VAR == 1 ? m + 1 : m + 2;
  const uint32_t fmask = (1u << width) - 1u;
  const int rec = VAR == 1 ? w.rec_sm : w.rec_q;
  const uint32_t* recs = VAR == 1 ? w.ssm : w.sq;
  const int nsb = (int)w.nsb;
  const int stride = gridDim.x * kWarps;
  for (int s = blockIdx.x * kWarps + warp; s < nsb; s += stride) {
    const int n = s / nsr;
    const int j = s - n * nsr;
    const int nb = min(CAS_SB, nbr - CAS_SB * j);
    const int64_t gb0 = (int64_t)n * nbr + CAS_SB * j;
    const uint32_t mw = lane < 4 * nb ? __ldg(w.mask + gb0 * 4 + lane) : 0u;
    s_mw[lane] = __brev(mw);
    {
      const uint32_t* rsrc = recs + gb0 * rec;
      for (int i = lane; i < nb * rec; i += 32) s_rec[i] = __ldg(rsrc + i);
    }
    const int cnt = __popc(mw);
    const int incl = warp_incl_add(cnt, lane);
    const int kt = nb * k;
    const int q = (kt + 31) >> 5;
    const int t0 = min(lane * q, kt), t1 = min(t0 + q, kt);
    // mask word and bit of the lane's first kept position
    const int wi = min(warp_count_le(incl, t0), 31);
    const int pre = __shfl_sync(CAS_FULL, incl - cnt, wi);
    const uint32_t wsel = __shfl_sync(CAS_FULL, mw, wi);
    const int bitpos = t0 < kt ? nth_set_bit(wsel, t0 - pre) : 0;
    // unary stream: bit after the t0-th '1' (start of code t0)
    const uint32_t* stream = nullptr;
    int ebit = 0, slim = 0;  // slim: stream words readable from `stream`
    if (VAR == 1) {
      const uint32_t sb0 = __ldg(w.sidx + s), sb1 = __ldg(w.sidx + s + 1);
      stream = w.sexp + sb0;
      slim = (int)(a.sexp_words - sb0);
      const int nwords = (int)(sb1 - sb0);
      int before = 0;
      bool done = t0 == 0 || t0 >= kt;
      for (int c0 = 0; c0 < nwords; c0 += 32) {
        if (!__any_sync(CAS_FULL, !done)) break;
        uint32_t wv = c0 + lane < nwords ? __ldg(stream + c0 + lane) : 0u;
        int ones = __popc(wv);
        int oincl = warp_incl_add(ones, lane);
        int total = __shfl_sync(CAS_FULL, oincl, 31);
        int need = t0 - before;  // 1-based index of the '1' that ends code t0-1
        int wk = min(warp_count_le(oincl, need - 1), 31);
        int oexcl = __shfl_sync(CAS_FULL, oincl - ones, wk);
        uint32_t word = __shfl_sync(CAS_FULL, wv, wk);
        if (!done && need <= total) {
          ebit = (c0 + wk) * 32 + nth_set_bit(__brev(word), need - oexcl - 1) + 1;
          done = true;
        }
        before += total;
      }
    }
    __syncwarp();
    float acc[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[v] = 0.f;
    if (t0 < t1) {
      const uint16_t* xrow = xs + CAS_BLK * CAS_SB * j;
      // positions: cursor over the bit-reversed mask words from (wi, bitpos)
      OnesCursor pc;
      pc.h = s_mw[wi] & (0xFFFFFFFFu >> bitpos);
      pc.l = s_mw[wi + 1];
      pc.base = 32 * wi;
      auto more_mask = [&](int bitidx) { return s_mw[min(bitidx >> 5, kMaskWords - 1)]; };
      auto more_code = [&](int bitidx) { return (bitidx >> 5) < slim ? __ldg(stream + (bitidx >> 5)) : 0u; };
      // codes: cursor over the unary stream from the word holding ebit
      OnesCursor cc;
      int prev = ebit;  // stream bit where the current code starts
      if (VAR == 1) {
        const int e0 = ebit & ~31;
        cc.h = more_code(e0) & (0xFFFFFFFFu >> (ebit & 31));
        cc.l = more_code(e0 + 32);
        cc.base = e0;
      }
      float scale = 0.f;
      int gcur = -1;
      {
        int b = t0 / k, tl = t0 - b * k;  // block and block-local ordinal of t0
        for (int t = t0; t < t1; ++t) {
          const int pos = pc.next(more_mask);
          if (tl == k) {
            ++b;
            tl = 0;
          }
          const int bit = b * rec * 32 + tl * width;
          ++tl;
          const uint32_t fld = __funnelshift_r(s_rec[bit >> 5], s_rec[(bit >> 5) + 1], bit & 31) & fmask;
          float val;
          if (VAR == 1) {
            const int end = cc.next(more_code);
            const uint32_t e23 = lut23[(end - prev) & 255];
            prev = end + 1;
            val = __uint_as_float(((fld >> m) << 31) | e23 | ((fld & (fmask >> 1)) << (23 - m)));
          } else {
            const int g = pos >> 5;
            if (g != gcur) {
              gcur = g;
              scale = pow2_biased(max((int)__ldg(w.smx + gb0 * 4 + g), 1) - m);
            }
            val = (float)(fld & (fmask >> 1)) * scale;
            val = (fld >> (m + 1)) ? -val : val;
          }
          const uint16_t* xp = xrow + (pos & 1023);
#pragma unroll
          for (int v = 0; v < NV; ++v) acc[v] = fmaf(val, bf2f(xp[v * K]), acc[v]);
        }
      }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      float r = warp_sumf(acc[v]);
      if (lane == 0) atomicAdd(a.y + (int64_t)v * w.N + n, r);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ fast path
// Cassandra-1, k = 64, m = 3, rows made of whole superblocks (K % 1024 == 0).
// One warp per superblock, visited in row-major order; lane L owns kept
// ordinals 16L..16L+15 (block L/4). The warp stages the superblock's unary
// exponent stream in shared memory with its popcount prefixes; each lane finds
// where its first code starts (a lower bound over the prefixes and a popcount
// select) and where its first kept position is (popcounts of the block's four
// mask words), then walks 16 steps: next code -> rank -> exponent, next set
// mask bit -> position, 4-bit record field -> sign and mantissa, fp32 value
// times x (bf16 in shared memory, staged once per CTA by a TMA bulk copy).
// Superblocks whose stream exceeds the stage (or holds fewer than 512 codes)
// go through the generic superblock decoder.
struct LaneStage {
  UnaryStage us;
  alignas(16) uint8_t pos[CAS_SB * 64];  // block position of every kept ordinal
};
union LaneWarp {
  LaneStage ls;
  uint8_t code[1024];  // generic decoder scratch (exponents by kept ordinal)
};


template <int NV>
__device__ __forceinline__ void gemv_superblock_generic(const WView& w, int64_t s, const uint8_t* lut8,
                                                        uint8_t* scratch, const uint16_t* xsb, int K, int lane,
                                                        float acc[NV]) {
  SbScratch sc{scratch, nullptr, nullptr};
  const SbInfo in = sb_prepare<1, false>(w, s, lut8, sc, lane);
  uint32_t v[16];
  sb_rebuild_word<1, false>(w, in, sc, lane, v);
  const uint16_t* xp = xsb + 32 * lane;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      acc[q] = fmaf(bf2f(v[i] & 0xFFFFu), bf2f(xp[q * K + 2 * i]), acc[q]);
      acc[q] = fmaf(bf2f(v[i] >> 16), bf2f(xp[q * K + 2 * i + 1]), acc[q]);
    }
  }
  __syncwarp();
}

// The lane's 16 kept values times x: value = sign, exponent (rank table) and
// the 3 high mantissa bits of the record field; x is bf16 in shared memory.
template <int NV, bool LONG>
__device__ __forceinline__ void lane_kept_dot(UnaryCursor& uc, uint4 pq, uint2 rr, const uint8_t* lut8,
                                              const uint16_t* xl, int K, float acc[NV]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t pw = (i >> 2) == 0 ? pq.x : (i >> 2) == 1 ? pq.y : (i >> 2) == 2 ? pq.z : pq.w;
    const int pos = (pw >> (8 * (i & 3))) & 127u;
    const uint32_t e = lut8[uc.next<LONG>() & 255];
    const uint32_t f = (i < 8 ? rr.x : rr.y) >> (4 * (i & 7));
    const float val = __uint_as_float(((f & 8u) << 28) | (e << 23) | ((f & 7u) << 20));
#pragma unroll
    for (int q = 0; q < NV; ++q) acc[q] = fmaf(val, bf2f(xl[q * K + pos]), acc[q]);
  }
}

template <int NV>
__global__ void __launch_bounds__(kThreads, 4) draft_gemv_fast_kernel(GemvArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  const WView& w = a.w;
  const int K = (int)w.K;
  const int xbytes = NV * K * 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + xbytes);
  uint8_t* lut8 = smem + xbytes + 16;
  LaneWarp& lw = reinterpret_cast<LaneWarp*>(smem + xbytes + 16 + 256)[warp];

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_tx(bar, (uint32_t)xbytes);
    bulk_g2s(xs, a.x, (uint32_t)xbytes, bar);
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) lut8[i] = a.lut.v[i];
  bool ok = mbar_wait_bounded(bar, 0, g_first_wait_spins);
  if (!__syncthreads_and(ok)) {
    if (threadIdx.x == 0) atomicExch(&g_gemv_wait_status, CAS_ERR_TIMEOUT);
    mbar_wait_bounded(bar, 0);  // let an in-flight copy land before the CTA exits
    return;
  }

  const int nsr = w.nsr;
  const int nsb = (int)w.nsb;
  const int stride = gridDim.x * kWarps;
  const int dn = stride / nsr, dj = stride - dn * nsr;  // (row, column) step of the superblock loop
  const uint32_t lim = (uint32_t)a.sexp_words;
  int s = blockIdx.x * kWarps + warp;
  int n = s / nsr, j = s - n * nsr;
  for (; s < nsb; s += stride) {
    // superblock s = n * nsr + j is blocks gb0 .. gb0 + 7 (rows are whole superblocks)
    const int64_t gb0 = (int64_t)s * CAS_SB;
    const uint32_t mw = __ldg(w.mask + gb0 * 4 + lane);
    const uint2 rr = __ldg(reinterpret_cast<const uint2*>(w.ssm + gb0 * 8) + lane);
    const uint32_t sb1 = min(__ldg(w.sidx + s + 1), lim), sb0 = min(__ldg(w.sidx + s), sb1);
    const int nw = (int)(sb1 - sb0);
    const uint16_t* xsb = xs + CAS_BLK * CAS_SB * j;
    float acc[NV];
#pragma unroll
    for (int q = 0; q < NV; ++q) acc[q] = 0.f;
    bool fast = nw <= kStageWords, long_codes = false;
    if (fast) {
      fast = stage_unary(w.sexp + sb0, nw, lw.ls.us, lane, &long_codes) >= 16 * 32;
      expand_mask_positions(mw, lw.ls.pos, lane);
    }
    __syncwarp();
    if (fast) {
      UnaryCursor uc;
      uc.init(lw.ls.us, unary_code_start(lw.ls.us, nw, 16 * lane));
      const uint4 pq = reinterpret_cast<const uint4*>(lw.ls.pos)[lane];
      const uint16_t* xl = xsb + CAS_BLK * (lane >> 2);
      if (long_codes)
        lane_kept_dot<NV, true>(uc, pq, rr, lut8, xl, K, acc);
      else
        lane_kept_dot<NV, false>(uc, pq, rr, lut8, xl, K, acc);
    }
    __syncwarp();
    if (!fast) {
#pragma unroll
      for (int q = 0; q < NV; ++q) acc[q] = 0.f;
      gemv_superblock_generic<NV>(w, s, lut8, lw.code, xsb, K, lane, acc);
    }
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      const float r = warp_sumf(acc[q]);
      if (lane == 0) atomicAdd(a.y + (int64_t)q * w.N + n, r);
    }
    n += dn;
    j += dj;
    if (j >= nsr) {
      j -= nsr;
      ++n;
    }
  }
}

// ------------------------------------------------------------------ any k, m
// Rows made of whole superblocks, any k and m, both variants. Lane L takes
// the run of kept ordinals [L q, L q + q) of the superblock (q = ceil(8k/32),
// runs may cross blocks). The warp stages the superblock's records (and, for
// Cassandra-1, its unary stream; for Cassandra-2, its shared exponents) in
// shared memory and expands the mask into the block position of every kept
// ordinal; each lane then walks its run: block position, record field at a
// run-time bit offset, exponent (unary cursor, or the group's shared exponent
// for Cassandra-2), times x. Superblocks whose unary stream exceeds the stage
// take the generic decoder.
struct RunsWarp {
  UnaryStage us;                               // Cassandra-1 codes
  uint32_t rec[CAS_SB * 36 + 2];               // records of the 8 blocks (<= 36 words each) + pad
  alignas(16) uint8_t pos[CAS_SB * CAS_BLK];   // block position of every kept ordinal
  uint8_t mx[CAS_SB * 4];                      // Cassandra-2 shared exponents
};
union RunsScratch {
  RunsWarp r;
  uint8_t code[CAS_SB * CAS_BLK];  // generic decoder: exponents by kept ordinal
};

template <int VAR, int NV, bool LONG>
__device__ __forceinline__ void run_dot(const RunsWarp& rw, UnaryCursor& uc, const uint8_t* lut8, int k, int m,
                                        int rec, int t0, int t1, const uint16_t* xsb, int K, float acc[NV]) {
  const int width = VAR == 1 ? m + 1 : m + 2;
  const uint32_t fmask = (1u << width) - 1u;
  int b = k > 0 ? t0 / k : 0;
  int tl = t0 - b * k;
  for (int t = t0; t < t1; ++t) {
    if (tl == k) {
      ++b;
      tl = 0;
    }
    const int p = rw.pos[t];
    const uint32_t fld = get_field(rw.rec + b * rec, tl * width, width) & fmask;
    ++tl;
    float val;
    if (VAR == 1) {
      const uint32_t e = lut8[uc.next<LONG>() & 255];
      val = __uint_as_float(((fld >> m) << 31) | (e << 23) | ((fld & (fmask >> 1)) << (23 - m)));
    } else {
      const float scale = pow2_biased(max((int)rw.mx[b * 4 + (p >> 5)], 1) - m);
      const float qv = (float)(fld & (fmask >> 1)) * scale;
      val = (fld >> (m + 1)) ? -qv : qv;
    }
    const uint16_t* xp = xsb + CAS_BLK * b + p;
#pragma unroll
    for (int q = 0; q < NV; ++q) acc[q] = fmaf(val, bf2f(xp[q * K]), acc[q]);
  }
}

template <int VAR, int NV>
__global__ void __launch_bounds__(kThreads) draft_gemv_runs_kernel(GemvArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  const WView& w = a.w;
  const int K = (int)w.K;
  const int xbytes = NV * K * 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + xbytes);
  uint8_t* lut8 = smem + xbytes + 16;
  RunsScratch& rs = reinterpret_cast<RunsScratch*>(smem + xbytes + 16 + 256)[warp];

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_tx(bar, (uint32_t)xbytes);
    bulk_g2s(xs, a.x, (uint32_t)xbytes, bar);
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) lut8[i] = a.lut.v[i];
  bool ok = mbar_wait_bounded(bar, 0, g_first_wait_spins);
  if (!__syncthreads_and(ok)) {
    if (threadIdx.x == 0) atomicExch(&g_gemv_wait_status, CAS_ERR_TIMEOUT);
    mbar_wait_bounded(bar, 0);  // let an in-flight copy land before the CTA exits
    return;
  }

  const int k = w.k, m = w.m, nsr = w.nsr;
  const int rec = VAR == 1 ? w.rec_sm : w.rec_q;
  const uint32_t* recs = VAR == 1 ? w.ssm : w.sq;
  const int nsb = (int)w.nsb;
  const int kt = CAS_SB * k, q = (kt + 31) >> 5;
  const int t0 = min(lane * q, kt), t1 = min(t0 + q, kt);
  const int stride = gridDim.x * kWarps;
  const uint32_t lim = (uint32_t)a.sexp_words;
  for (int s = blockIdx.x * kWarps + warp; s < nsb; s += stride) {
    const int n = s / nsr;
    const int j = s - n * nsr;
    const int64_t gb0 = (int64_t)s * CAS_SB;  // rows are whole superblocks
    const uint16_t* xsb = xs + CAS_BLK * CAS_SB * j;
    float acc[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[v] = 0.f;
    int nw = 0;
    uint32_t sb0 = 0;
    if (VAR == 1) {
      const uint32_t sb1 = min(__ldg(w.sidx + s + 1), lim);
      sb0 = min(__ldg(w.sidx + s), sb1);
      nw = (int)(sb1 - sb0);
    }
    bool fast = VAR == 2 || nw <= kStageWords, long_codes = false;
    if (fast) {
      const uint32_t* rsrc = recs + gb0 * rec;
      for (int i = lane; i < CAS_SB * rec; i += 32) rs.r.rec[i] = __ldg(rsrc + i);
      if (lane < 2) rs.r.rec[CAS_SB * rec + lane] = 0u;
      if (VAR == 2) rs.r.mx[lane] = __ldg(w.smx + gb0 * 4 + lane);
      if (VAR == 1) fast = stage_unary(w.sexp + sb0, nw, rs.r.us, lane, &long_codes) >= kt;
      expand_mask_positions<CAS_SB * CAS_BLK>(__ldg(w.mask + gb0 * 4 + lane), rs.r.pos, lane);
    }
    __syncwarp();
    if (fast) {
      UnaryCursor uc;
      if (VAR == 1) uc.init(rs.r.us, unary_code_start(rs.r.us, nw, t0));
      if (long_codes)
        run_dot<VAR, NV, true>(rs.r, uc, lut8, k, m, rec, t0, t1, xsb, K, acc);
      else
        run_dot<VAR, NV, false>(rs.r, uc, lut8, k, m, rec, t0, t1, xsb, K, acc);
    }
    __syncwarp();
    if (!fast) {  // Cassandra-1 stream longer than the stage
#pragma unroll
      for (int v = 0; v < NV; ++v) acc[v] = 0.f;
      SbScratch sc{rs.code, nullptr, nullptr};
      const SbInfo in = sb_prepare<1, false>(w, s, lut8, sc, lane);
      uint32_t v[16];
      sb_rebuild_word<1, false>(w, in, sc, lane, v);
      const uint16_t* xp = xsb + 32 * lane;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
#pragma unroll
        for (int qq = 0; qq < NV; ++qq) {
          acc[qq] = fmaf(bf2f(v[i] & 0xFFFFu), bf2f(xp[qq * K + 2 * i]), acc[qq]);
          acc[qq] = fmaf(bf2f(v[i] >> 16), bf2f(xp[qq * K + 2 * i + 1]), acc[qq]);
        }
      }
      __syncwarp();
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const float r = warp_sumf(acc[v]);
      if (lane == 0) atomicAdd(a.y + (int64_t)v * w.N + n, r);
    }
  }
}

// Cassandra-2 fast path (k = 64, m = 3, whole superblocks). The speculation
// data has no unary stream: each kept value is a 5-bit field (sign, 4-bit q)
// and each 32-position mask word is exactly one shared-exponent group. Phase
// 2 stores the signed q by ordinal; phase 3 (lane = mask word = group)
// accumulates q * x and multiplies the sum once by the group's scale
// 2^(E' - 127 - m).
constexpr int kFastSkew = 512 + 16;  // values by ordinal, index t + t/32 (bank skew)
struct Fast2Warp {
  uint32_t rec[80 + 2];  // spec_q records of the 8 blocks (10 words each) + pad
  float val[kFastSkew];
};

template <int NV>
__global__ void __launch_bounds__(kThreads) draft_gemv_fast2_kernel(GemvArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  const WView& w = a.w;
  const int K = (int)w.K;
  const int xbytes = NV * K * 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + xbytes);
  Fast2Warp& fw = reinterpret_cast<Fast2Warp*>(smem + xbytes + 16)[warp];

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_tx(bar, (uint32_t)xbytes);
    bulk_g2s(xs, a.x, (uint32_t)xbytes, bar);
  }
  bool ok = mbar_wait_bounded(bar, 0, g_first_wait_spins);
  if (!__syncthreads_and(ok)) {
    if (threadIdx.x == 0) atomicExch(&g_gemv_wait_status, CAS_ERR_TIMEOUT);
    mbar_wait_bounded(bar, 0);  // let an in-flight copy land before the CTA exits
    return;
  }

  const int N = (int)w.N, nbr = w.nbr;
  const int nsb = (int)w.nsb;
  const int stride = gridDim.x * kWarps;
  int jcur = -1;
  float xr[NV][32];
  for (int sc = blockIdx.x * kWarps + warp; sc < nsb; sc += stride) {
    const int j = sc / N;
    const int n = sc - j * N;
    if (j != jcur) {
      jcur = j;
      const uint16_t* xp = xs + CAS_BLK * CAS_SB * j + 32 * lane;
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int p = 0; p < 32; ++p) xr[v][p] = bf2f(xp[v * K + p]);
    }
    const int64_t gb0 = (int64_t)n * nbr + CAS_SB * j;
    const uint32_t mw = __ldg(w.mask + gb0 * 4 + lane);
    const int cnt = __popc(mw);
    const int o = warp_incl_add(cnt, lane) - cnt;
    const float scale = pow2_biased(max((int)__ldg(w.smx + gb0 * 4 + lane), 1) - 3);
    const uint32_t* rsrc = w.sq + gb0 * 10;
    fw.rec[lane] = __ldg(rsrc + lane);
    fw.rec[32 + lane] = __ldg(rsrc + 32 + lane);
    if (lane < 16) fw.rec[64 + lane] = __ldg(rsrc + 64 + lane);
    __syncwarp();
    // phase 2: signed q by ordinal
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int t = lane + 32 * i;
      const int tl = lane + 32 * (i & 1);  // ordinal within block i/2
      const int bit = 5 * tl;
      const int wsel = 10 * (i >> 1) + (bit >> 5);
      const uint32_t fld = __funnelshift_r(fw.rec[wsel], fw.rec[wsel + 1], bit & 31) & 31u;
      const float q = (float)(fld & 15u);
      fw.val[t + (t >> 5)] = (fld >> 4) ? -q : q;
    }
    __syncwarp();
    // phase 3: positions of mask word `lane` (one shared-exponent group)
    float acc[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[v] = 0.f;
    int t = o;
#pragma unroll
    for (int p = 0; p < 32; ++p) {
      if ((mw >> p) & 1u) {
        const float val = fw.val[t + (t >> 5)];
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[v] = fmaf(val, xr[v][p], acc[v]);
        ++t;
      }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      float r = warp_sumf(acc[v] * scale);
      if (lane == 0) atomicAdd(a.y + (int64_t)v * w.N + n, r);
    }
    __syncwarp();
  }
}

template <int NV>
int launch_fast2(const GemvArgs& a, cudaStream_t st) {
  size_t smem = (size_t)NV * a.w.K * 2 + 16 + kWarps * sizeof(Fast2Warp);
  auto kern = draft_gemv_fast2_kernel<NV>;
  int per_sm = occupancy((const void*)kern, kThreads, smem);
  if (per_sm < 1) return CAS_ERR_CUDA;
  int64_t need = (a.w.nsb + kWarps - 1) / kWarps;
  int g = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sm_count() * per_sm));
  return launch_k(kern, g, kThreads, smem, st, a);
}

template <int NV>
int launch_fast(const GemvArgs& a, cudaStream_t st) {
  size_t smem = (size_t)NV * a.w.K * 2 + 16 + 256 + kWarps * sizeof(LaneWarp);
  auto kern = draft_gemv_fast_kernel<NV>;
  int per_sm = occupancy((const void*)kern, kThreads, smem);
  if (per_sm < 1) return CAS_ERR_CUDA;
  int64_t need = (a.w.nsb + kWarps - 1) / kWarps;
  int g = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sm_count() * per_sm));
  return launch_k(kern, g, kThreads, smem, st, a);
}

template <int VAR, int NV>
int launch_runs(const GemvArgs& a, cudaStream_t st) {
  size_t smem = (size_t)NV * a.w.K * 2 + 16 + 256 + kWarps * sizeof(RunsScratch);
  auto kern = draft_gemv_runs_kernel<VAR, NV>;
  int per_sm = occupancy((const void*)kern, kThreads, smem);
  if (per_sm < 1) return CAS_ERR_CUDA;
  int64_t need = (a.w.nsb + kWarps - 1) / kWarps;
  int g = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sm_count() * per_sm));
  return launch_k(kern, g, kThreads, smem, st, a);
}

template <int VAR, int NV>
int launch(const GemvArgs& a, cudaStream_t st) {
  size_t smem = (size_t)NV * a.w.K * 2 + 16 + 1024 + kWarps * kWarpWords * 4;
  auto kern = draft_gemv_kernel<VAR, NV>;
  int per_sm = occupancy((const void*)kern, kThreads, smem);
  if (per_sm < 1) return CAS_ERR_CUDA;
  int64_t need = (a.w.nsb + kWarps - 1) / kWarps;
  int g = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sm_count() * per_sm));
  return launch_k(kern, g, kThreads, smem, st, a);
}

// ------------------------------------------------------------------ word path
// Cassandra-1, k = 64, m = 3, rows made of whole superblocks, 1 or 2 vectors.
// Lane L owns mask word L of the superblock (block L/4, positions
// 32(L%4)..+31). Its kept values are consecutive ordinals, so their 4-bit
// sign/mantissa fields are one bit range of the block record and their
// exponent codes one bit range of the superblock's unary stream: each lane
// walks three cursors of its own, with no cross-lane traffic per value.
//   position: count of leading zeros of the bit-reversed mask word, the found
//             bit cleared; once the word is exhausted the count is 32, which
//             points at a zero pad float of x;
//   exponent: count of leading zeros of a 64-bit window of the code stream
//             aligned at the lane's first code (rank -> exponent by a table),
//             re-aligned after every 8 codes;
//   field:    nibble i of the lane's field window, moved into the sign and
//             mantissa bits of an fp32 by one byte permute.
// x is staged per CTA as fp32 with one zero pad float after every 32
// positions, so lane L's 32 positions start on bank L and the lanes' gathers
// of one step spread over the banks. Each warp takes a contiguous run of
// superblocks and adds its sum to y once per row. Superblocks the fast walk
// cannot take (a run of 31 or more zeros in the code stream, a lane's codes
// wider than its windows, a stream longer than 64 words) go through the
// generic superblock decoder.
constexpr int kXGroup = 33;   // staged floats per 32 positions (32 + a zero pad)
constexpr int kWordLut = 64;  // exponent by rank, ranks 0..63

struct WordStage {
  uint32_t st[64 + 32];  // stream words of the superblock, then zeros / read-ahead
  uint32_t rec[64 + 8];  // sign/mantissa records of the 8 blocks, then pad
};
union WordScratch {
  WordStage ws;
  uint8_t code[CAS_SB * CAS_BLK];  // generic decoder: exponents by kept ordinal
};

__host__ __device__ constexpr int word_x_floats(int K) { return ((K / 32) * kXGroup + 3) & ~3; }


// The generic superblock decoder for what the word walk cannot take. Kept out
// of line so that its registers do not count against the fast path.
template <int NV>
__device__ __noinline__ void word_fallback(WView w, int64_t s, const uint8_t* lut8, uint8_t* code, const float* xb,
                                           int xfl, float* part) {
  const int lane = threadIdx.x & 31;
  SbScratch ss{code, nullptr, nullptr};
  const SbInfo in = sb_prepare<1, false>(w, s, lut8, ss, lane);
  uint32_t v[16];
  sb_rebuild_word<1, false>(w, in, ss, lane, v);
#pragma unroll
  for (int q = 0; q < NV; ++q) part[q] = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      part[q] = fmaf(bf2f(v[i] & 0xFFFFu), xb[q * xfl + 2 * i], part[q]);
      part[q] = fmaf(bf2f(v[i] >> 16), xb[q * xfl + 2 * i + 1], part[q]);
    }
  }
  __syncwarp();
}

// 32 registers per thread (8 CTAs of 256 per SM); superblocks for the generic
// decoder wait in a per-warp list in shared memory until the warp's run is
// done, so nothing of that decoder is live in the hot loop.
template <int NV>
__global__ void __launch_bounds__(kThreads, 8) draft_gemv_word_kernel(GemvArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint8_t lut8[256];  // exponent by rank
  const WView& w = a.w;
  const int K = (int)w.K;
  const int xfl = word_x_floats(K);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* xs = reinterpret_cast<float*>(smem);
  WordScratch& sc = reinterpret_cast<WordScratch*>(smem + (size_t)NV * xfl * 4)[warp];

  // x -> fp32, position p of vector v at v*xfl + (p/32)*33 + p%32; pads zero
  for (int v = 0; v < NV; ++v) {
    const uint4* xv = reinterpret_cast<const uint4*>(a.x + (size_t)v * K);
    for (int i = threadIdx.x; i < K / 8; i += kThreads) {
      const uint4 pr = __ldg(xv + i);
      const int p = 8 * i;
      float* d = xs + v * xfl + (p >> 5) * kXGroup + (p & 31);
      d[0] = bf2f(pr.x & 0xFFFFu);
      d[1] = bf2f(pr.x >> 16);
      d[2] = bf2f(pr.y & 0xFFFFu);
      d[3] = bf2f(pr.y >> 16);
      d[4] = bf2f(pr.z & 0xFFFFu);
      d[5] = bf2f(pr.z >> 16);
      d[6] = bf2f(pr.w & 0xFFFFu);
      d[7] = bf2f(pr.w >> 16);
    }
    for (int g = threadIdx.x; g < K / 32; g += kThreads) xs[v * xfl + g * kXGroup + 32] = 0.f;
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) lut8[i] = a.lut.v[i];
  if (lane < 8) sc.ws.rec[64 + lane] = 0u;
  __syncthreads();

  const int nsr = w.nsr;
  const int nsb = (int)w.nsb;
  const int nwarps = gridDim.x * kWarps;
  const int gw = blockIdx.x * kWarps + warp;
  const int per = (nsb + nwarps - 1) / nwarps;
  const int s0 = min(gw * per, nsb), s1 = min(s0 + per, nsb);
  const uint32_t lim = (uint32_t)a.sexp_words;
  const int blk = lane >> 2;
  const uint32_t x_a = smem_addr(xs) + 4u * (uint32_t)(lane * kXGroup);
  int* fb = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(&sc) + sizeof(WordScratch) * (kWarps - warp)) +
            warp * per;  // this warp's list of superblocks for the generic decoder
  int nfb = 0;
  int n = s0 / nsr, j = s0 - n * nsr;
  float acc[NV];
#pragma unroll
  for (int q = 0; q < NV; ++q) acc[q] = 0.f;
  for (int s = s0; s < s1; ++s) {
    const int64_t gb0 = (int64_t)s * CAS_SB;
    const uint32_t mw = __ldg(w.mask + gb0 * 4 + lane);
    const uint2 rr = __ldg(reinterpret_cast<const uint2*>(w.ssm + gb0 * 8) + lane);
    uint32_t sb0, sb1;
    stream_range(w.sidx, s, lim, sb0, sb1);
    const int nw = (int)(sb1 - sb0);
    float part[NV];
#pragma unroll
    for (int q = 0; q < NV; ++q) part[q] = 0.f;
    bool fast = nw <= 64;
    if (fast) {
      WordStage& ws = sc.ws;
      ws.rec[2 * lane] = rr.x;
      ws.rec[2 * lane + 1] = rr.y;
      // stream words 2l, 2l+1 in lane l, with popcount prefixes
      const uint32_t* gs = w.sexp + sb0;
      const uint32_t w0 = 2 * lane < nw ? __ldg(gs + 2 * lane) : 0u;
      const uint32_t w1 = 2 * lane + 1 < nw ? __ldg(gs + 2 * lane + 1) : 0u;
      ws.st[2 * lane] = w0;
      ws.st[2 * lane + 1] = w1;
      ws.st[64 + lane] = 0u;
      const int b1 = __popc(w1);
      const int S = warp_incl_add(__popc(w0) + b1, lane);  // ones through word 2l+1
      const int ncodes = __shfl_sync(CAS_FULL, S, 31);
      // runs of 31+ zeros (a code of rank >= 31) across word boundaries
      const int tz0 = tzcnt(w0), tz1 = tzcnt(w1);
      const int lz1 = __clz(w1), lzn = __shfl_down_sync(CAS_FULL, __clz(w0), 1);
      const bool run = (2 * lane + 1 < nw && tz0 + lz1 >= 31) || (2 * lane + 2 < nw && tz1 + lzn >= 31) ||
                       (lane == 0 && nw > 0 && __clz(w0) >= 31);
      const bool lng = __any_sync(CAS_FULL, run);
      const int lw = nw - 1;  // the stream ends inside word nw-1
      const int tzl = __shfl_sync(CAS_FULL, (lw & 1) ? tz1 : tz0, (lw >> 1) & 31);
      const int endbit = nw > 0 ? 32 * lw + 32 - tzl : 0;
      // block-local ordinal of the lane's first kept value
      const int c = __popc(mw);
      int inc = c;
      const int u1 = __shfl_up_sync(CAS_FULL, inc, 1, 4);
      if ((lane & 3) >= 1) inc += u1;
      const int u2 = __shfl_up_sync(CAS_FULL, inc, 2, 4);
      if ((lane & 3) >= 2) inc += u2;
      const int o = min(inc - c, 64);
      // start of the lane's first code: just after the T-th '1'
      const int T = 64 * blk + o;
      const int l = min(warp_count_le(S, T - 1), 31);  // first lane whose prefix reaches T
      const int Sl = __shfl_sync(CAS_FULL, S, l), bl = __shfl_sync(CAS_FULL, b1, l);
      const uint32_t x0 = __shfl_sync(CAS_FULL, w0, l), x1 = __shfl_sync(CAS_FULL, w1, l);
      const int q0 = Sl - bl;  // ones through word 2l
      const bool in0 = T <= q0;
      const uint32_t wsel = in0 ? x0 : x1;
      const int rr1 = T - (in0 ? q0 - __popc(x0) : q0);
      const int start = T > 0 ? 32 * (2 * l + (in0 ? 0 : 1)) + select_msb(wsel, max(rr1, 1)) + 1 : 0;
      int nxt = __shfl_down_sync(CAS_FULL, start, 1);
      if (lane == 31) nxt = endbit;
      const int span = nxt - start;
      __syncwarp();
      // field window: fields o..o+31 of block blk's record, nibble i = field i
      const uint32_t* rp = ws.rec + 8 * blk + (o >> 3);
      const int fs = 4 * (o & 7);
      uint32_t fo[4], fe[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        fo[q] = __funnelshift_r(rp[q], rp[q + 1], fs);  // odd fields in high nibbles
        fe[q] = fo[q] << 4;                              // even fields moved up
      }
      // code window: 64 bits from `start`
      int hw = start >> 5, sh = start & 31;
      uint32_t H = __funnelshift_l(ws.st[hw + 1], ws.st[hw], sh);
      uint32_t Lw = __funnelshift_l(ws.st[hw + 2], ws.st[hw + 1], sh);
      uint32_t M = __brev(mw);
      const uint32_t xa = x_a + 4u * (uint32_t)(j * (32 * kXGroup));
      const int maxc = __reduce_max_sync(CAS_FULL, c);
      int used = 0, u8 = 0, u16 = 0, u24 = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if ((i & 3) == 0 && i >= maxc) break;
        if ((i & 7) == 0 && i > 0) {  // re-align the code window every 8 codes
          if (i == 8) u8 = used;
          if (i == 16) u16 = used;
          if (i == 24) u24 = used;
          const int pos = start + used;
          hw = min(pos >> 5, 93);
          sh = pos & 31;
          H = __funnelshift_l(ws.st[hw + 1], ws.st[hw], sh);
          Lw = __funnelshift_l(ws.st[hw + 2], ws.st[hw + 1], sh);
        }
        const uint32_t p = __clz(M);  // 32 once the word is exhausted: zero pad
        M &= ~shr32(0x80000000u, p);  // p = 32 clears nothing
        const uint32_t r = __clz(H);  // <= 30 for every code of a checked stream
        const uint32_t e = lut8[r];
        const uint32_t nb = r + 1u;
        H = shfl_wrap(Lw, H, nb);
        Lw = shl32(Lw, nb);
        used += (int)nb;
        const uint32_t src = (i & 1) ? fo[i >> 3] : fe[i >> 3];
        const int by = (i & 7) >> 1;
        const uint32_t A = __byte_perm(src, 0u, (by << 12) | (by << 8) | 0x44);
        const float val = __uint_as_float(mad32(e, 0x800000u, A & 0x80700000u));
        const uint32_t xp = mad32((uint32_t)p, 4u, xa);
#pragma unroll
        for (int q = 0; q < NV; ++q) part[q] = fmaf(val, lds_f32(xp + 4u * (uint32_t)(q * xfl)), part[q]);
      }
      // every group of 8 codes must have fit its 64-bit window: full groups by
      // the bits they consumed, the lane's last group by its true end
      const int last = (c - 1) >> 3;  // -1 when the lane has no values
      const bool bad = (last > 0 && u8 > 64) || (last > 1 && u16 - u8 > 64) || (last > 2 && u24 - u16 > 64) ||
                       (last >= 0 && span - (last == 0 ? 0 : last == 1 ? u8 : last == 2 ? u16 : u24) > 64);
      fast = !lng && ncodes >= 512 && !__any_sync(CAS_FULL, bad);
    }
    __syncwarp();
    if (!fast) {  // decoded after the run; nothing of it is added now
      if (lane == 0) fb[nfb] = s;
      ++nfb;
#pragma unroll
      for (int q = 0; q < NV; ++q) part[q] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < NV; ++q) acc[q] += part[q];
    // next superblock; the row's sum goes to y when the row ends
    if (++j == nsr || s + 1 == s1) {
#pragma unroll
      for (int q = 0; q < NV; ++q) {
        const float r = warp_sumf(acc[q]);
        if (lane == 0) atomicAdd(a.y + (int64_t)q * w.N + n, r);
        acc[q] = 0.f;
      }
      if (j == nsr) {
        j = 0;
        ++n;
      }
    }
  }
  // superblocks the word walk did not take: the generic decoder, one row
  // segment each
  __syncwarp();
  for (int i = 0; i < nfb; ++i) {
    const int sf = fb[i];
    const int nf = sf / nsr, jf = sf - nf * nsr;
    float part[NV];
    word_fallback<NV>(w, sf, lut8, sc.code, xs + jf * (32 * kXGroup) + lane * kXGroup, xfl, part);
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      const float r = warp_sumf(part[q]);
      if (lane == 0) atomicAdd(a.y + (int64_t)q * w.N + nf, r);
    }
  }
}

template <int NV>
size_t word_smem(int64_t K) {
  return (size_t)NV * word_x_floats((int)K) * 4 + kWarps * sizeof(WordScratch);
}
// superblocks per warp of a launch with g CTAs
inline int word_per(int64_t nsb, int g) { return (int)((nsb + (int64_t)g * kWarps - 1) / ((int64_t)g * kWarps)); }

// ------------------------------------------------------------------ block path
// Cassandra-1, m = 3, k = 64 or 38 (keep 50 % or 30 %), rows of whole
// superblocks with at least 32 blocks (K >= 4096), 1 or 2 vectors. A warp
// takes a chunk of 32 consecutive blocks (4 superblocks) and lane L owns block
// L of it: 128 positions with exactly k kept values, so every lane decodes the
// same number of values.
// Per chunk the warp stages the 4 superblocks' code streams and its blocks'
// bit-reversed mask words in shared memory; each lane finds where its block's
// codes start (the bit after the (k j)-th '1' of its superblock's stream, j
// the block's place in it) by a warp popcount scan and a shuffle search, and
// then walks two cursors of its own (the exponent cursor re-aligned from
// shared memory every 8 values, the position cursor every 16 for k = 64, 8
// for k = 38):
//   position: a 64-bit window of the bit-reversed mask starting just after the
//             last found position; one more than its count of leading zeros
//             is the distance n to the next kept position, and the window
//             shifts by n (a funnel shift of the two words);
//   exponent: the same over the code stream starting at the next code: the
//             count of leading zeros is the rank.
// Every shift must be below 32. A larger one - a gap of 32 or more positions,
// a code of rank 31 or more, a window that runs dry (count 32) - is the only
// case with bit 5 set, so OR-ing every shift finds all of them at once; a
// lane that met one walks its block again by scanning the staged words
// (block_walk_scan), which takes any gap and any code. Chunks whose streams
// do not fit the stage go to the generic decoder after the warp's run. x is
// staged per CTA as fp32 with 129 floats per block, so position p of block b
// sits on bank (b + p) % 32 and the 32 lanes, which advance through their
// blocks at about the same pace, spread over the banks.
constexpr int kBThreads = 512;
constexpr int kBWarps = kBThreads / 32;
constexpr int kBXRow = CAS_BLK + 1;   // staged floats per block
// bytes after x: the reads of a failed walk (up to position 127 + 16 * 33 of
// the last block) stay inside
constexpr int kBXPad = 2304;
constexpr int kBMaskRows = 8;         // zero row, 4 mask words, 3 zero rows

constexpr int kBStreamWords = BlockStreams<2>::kRow;
struct BlockStage {
  BlockStreams<2> st;             // the chunk's code streams
  uint32_t ms[kBMaskRows][32];    // row 1 + i, column l: bit-reversed mask word i of lane l's block
  uint32_t fs[8][32];             // row i, column l: word i of the sign/mantissa record of lane l's block
};
static_assert(sizeof(BlockStage) >= CAS_SB * CAS_BLK, "the generic decoder's scratch overlays the stage");
static_assert(sizeof(BlockStage) % 16 == 0, "stage alignment");

__host__ __device__ constexpr int block_x_floats(int nbr) { return (nbr * kBXRow + 3) & ~3; }

// The block walk without windows: every position and code found by a scan
// of the staged words, so gaps and codes of any length are taken. For a lane
// whose windowed walk ran dry; false when the staged data runs out (the
// encoding is inconsistent).
template <int NV>
struct ScanSum {
  float part[NV];
  bool ok;
};
template <int NV>
__device__ __noinline__ ScanSum<NV> block_walk_scan(uint32_t ms_a, uint32_t st_a, uint32_t fs_a, uint32_t lut_a,
                                                    uint32_t xbase, int xfl, int cq0, int keep) {
  ScanSum<NV> r;
  int cur = -1, qc = cq0;
#pragma unroll
  for (int q = 0; q < NV; ++q) r.part[q] = 0.f;
  r.ok = false;
  for (int i = 0; i < keep; ++i) {
    const int pb = bnext_one(ms_a, 128u, 32 + cur + 1, kBMaskRows - 1);
    const int tb = bnext_one(st_a, 4u, qc + 1, kBStreamWords - 1);
    if (pb < 0 || pb >= 32 + CAS_BLK || tb < 0) return r;
    cur = pb - 32;
    const uint32_t E = lds_u32(lut_a + 4u * (uint32_t)min(tb - qc - 1, 255));  // rank tb - qc - 1
    qc = tb;
    const uint32_t f = (lds_u32(fs_a + 128u * (uint32_t)(i >> 3)) >> (4 * (i & 7))) & 15u;
    const float val = __uint_as_float(((f & 8u) << 28) | E | ((f & 7u) << 20));
#pragma unroll
    for (int q = 0; q < NV; ++q) r.part[q] = fmaf(val, lds_f32(xbase + 4u * (uint32_t)(cur + q * xfl)), r.part[q]);
  }
  r.ok = true;
  return r;
}

template <int NV, int KEEP>
__global__ void __launch_bounds__(kBThreads, 3) draft_gemv_block_kernel(GemvArgs a) {
  pdl_wait();
  pdl_trigger();
  constexpr int kRec = (KEEP * 4 + 31) / 32;  // sign/mantissa record words per block
  constexpr int kGroups = (KEEP + 7) / 8;
  // groups of 8 values per re-alignment of the position window: 16 of 64
  // positions in 128 almost never span more than its 64 bits (a window that
  // runs dry is caught like a long gap); 16 of 38 often would
  constexpr int kPosGroups = KEEP == 64 ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t lut32[256];  // exponent << 23 by rank
  __shared__ uint8_t lut8[256];    // exponent by rank (generic decoder)
  const WView& w = a.w;
  const int K = (int)w.K;
  const int nbr = w.nbr;
  const int xfl = block_x_floats(nbr);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* xs = reinterpret_cast<float*>(smem);
  BlockStage& bs = reinterpret_cast<BlockStage*>(smem + (size_t)NV * xfl * 4 + kBXPad)[warp];

  // x -> fp32, position p of vector v at v*xfl + (p/128)*129 + p%128
  // fp32 inputs are read 4 values per load, several loads in flight per thread
  if (a.xop >= 2) {  // an fp32 input, rounded (or SiLU * mul first) to bf16 like the glue kernels
    for (int v = 0; v < NV; ++v) {
      const float4* src = reinterpret_cast<const float4*>(a.xf + (size_t)v * (a.xop == 3 ? 2 * K : K));
#pragma unroll 4
      for (int i = threadIdx.x; i < K / 4; i += kBThreads) {
        float4 f = __ldg(src + i);
        if (a.xop == 3) {
          const float4 u = __ldg(src + K / 4 + i);
          f = make_float4(silu_mul_f(f.x, u.x), silu_mul_f(f.y, u.y), silu_mul_f(f.z, u.z), silu_mul_f(f.w, u.w));
        }
        const uint32_t b0 = f2bf(f.x), b1 = f2bf(f.y), b2 = f2bf(f.z), b3 = f2bf(f.w);
        const int p = 4 * i;
        float* d = xs + v * xfl + (p >> 7) * kBXRow + (p & 127);
        d[0] = bf2f(b0);
        d[1] = bf2f(b1);
        d[2] = bf2f(b2);
        d[3] = bf2f(b3);
        if (blockIdx.x == 0) reinterpret_cast<uint2*>(a.xn + (size_t)v * K)[i] = make_uint2(b0 | (b1 << 16), b2 | (b3 << 16));
      }
    }
  } else if (a.xop == 1) {  // the input is fp32: RMSNorm first, rounded to bf16 like the unfused glue
    __shared__ float red[kBWarps];
    for (int v = 0; v < NV; ++v) {
      const float4* xr = reinterpret_cast<const float4*>(a.xf + (size_t)v * K);
      float ss = 0.f;
#pragma unroll 4
      for (int i = threadIdx.x; i < K / 4; i += kBThreads) {
        const float4 f = __ldg(xr + i);
        const int p = 4 * i;
        float* d = xs + v * xfl + (p >> 7) * kBXRow + (p & 127);
        d[0] = f.x;
        d[1] = f.y;
        d[2] = f.z;
        d[3] = f.w;
        ss = fmaf(f.x, f.x, ss);
        ss = fmaf(f.y, f.y, ss);
        ss = fmaf(f.z, f.z, ss);
        ss = fmaf(f.w, f.w, ss);
      }
      ss = warp_sumf(ss);
      if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
      __syncthreads();
      float tot = (threadIdx.x & 31) < kBWarps ? red[threadIdx.x & 31] : 0.f;
      tot = warp_sumf(tot);
      const float inv = rsqrtf(tot / (float)K + a.eps);
      const uint2* gm = reinterpret_cast<const uint2*>(a.gamma);
#pragma unroll 4
      for (int i = threadIdx.x; i < K / 4; i += kBThreads) {
        const int p = 4 * i;
        float* d = xs + v * xfl + (p >> 7) * kBXRow + (p & 127);
        const uint2 g = __ldg(gm + i);
        const uint32_t b0 = f2bf(d[0] * inv * bf2f(g.x & 0xFFFFu)), b1 = f2bf(d[1] * inv * bf2f(g.x >> 16));
        const uint32_t b2 = f2bf(d[2] * inv * bf2f(g.y & 0xFFFFu)), b3 = f2bf(d[3] * inv * bf2f(g.y >> 16));
        d[0] = bf2f(b0);
        d[1] = bf2f(b1);
        d[2] = bf2f(b2);
        d[3] = bf2f(b3);
        if (blockIdx.x == 0) reinterpret_cast<uint2*>(a.xn + (size_t)v * K)[i] = make_uint2(b0 | (b1 << 16), b2 | (b3 << 16));
      }
      __syncthreads();
    }
  }
  for (int v = 0; v < NV && a.xop == 0; ++v) {
    const uint4* xv = reinterpret_cast<const uint4*>(a.x + (size_t)v * K);
    for (int i = threadIdx.x; i < K / 8; i += kBThreads) {
      const uint4 pr = __ldg(xv + i);
      const int p = 8 * i;
      float* d = xs + v * xfl + (p >> 7) * kBXRow + (p & 127);
      d[0] = bf2f(pr.x & 0xFFFFu);
      d[1] = bf2f(pr.x >> 16);
      d[2] = bf2f(pr.y & 0xFFFFu);
      d[3] = bf2f(pr.y >> 16);
      d[4] = bf2f(pr.z & 0xFFFFu);
      d[5] = bf2f(pr.z >> 16);
      d[6] = bf2f(pr.w & 0xFFFFu);
      d[7] = bf2f(pr.w >> 16);
    }
  }
  for (int i = threadIdx.x; i < kBXPad / 4; i += kBThreads) xs[NV * xfl + i] = 0.f;
  for (int i = threadIdx.x; i < 256; i += kBThreads) {
    lut32[i] = (uint32_t)a.lut.v[i] << 23;
    lut8[i] = a.lut.v[i];
  }
  __syncthreads();

  const int64_t nsb = w.nsb;
  const int nch = (int)((nsb + 3) / 4);
  const int nwarps = gridDim.x * kBWarps;
  // chunks dealt round-robin over the CTAs (chunk c to CTA c % gridDim.x), so
  // a small matrix spreads evenly over the CTAs of the wave, and so over the SMs
  const int gw = warp * gridDim.x + blockIdx.x;
  const int per = (nch + nwarps - 1) / nwarps;
  const uint32_t lim = (uint32_t)a.sexp_words;
  const int t = lane >> 3, j = lane & 7;
  const uint32_t ms_a0 = smem_addr(&bs.ms[0][lane]);
  const uint32_t fs_a0 = smem_addr(&bs.fs[0][lane]);
  const uint32_t st_a0 = smem_addr(&bs.st.w[t][0]);
  const uint32_t lut_a = smem_addr(lut32);  // rank r at lut_a + 4r
  const uint32_t xs_a = smem_addr(xs);
  int* fb = reinterpret_cast<int*>(smem + (size_t)NV * xfl * 4 + kBXPad + kBWarps * sizeof(BlockStage)) + warp * per;
  int nfb = 0;
  // zero rows and words of the stage, written once
  block_streams_init(bs.st, lane);
  bs.ms[0][lane] = 0u;
  bs.ms[5][lane] = 0u;
  bs.ms[6][lane] = 0u;
  bs.ms[7][lane] = 0u;

  for (int c = gw; c < nch; c += nwarps) {
    // row and block in the row of the chunk's first block
    const uint32_t row0 = (uint32_t)c * 32u / (uint32_t)nbr;  // block indices fit 32 bits (launch checks)
    const uint32_t jb0 = (uint32_t)c * 32u - row0 * (uint32_t)nbr;
    // the chunk's streams; a stream longer than the stage sends the chunk to
    // the generic decoder
    uint32_t sa[4];
    int nw[4];
    bool fast = true;
    const int64_t s0 = (int64_t)c * 4;
    const uint32_t ix = lane <= 4 && s0 + lane <= nsb ? __ldg(w.sidx + s0 + lane) : 0u;  // index words s0 .. s0+4
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t i0 = __shfl_sync(CAS_FULL, ix, u), i1 = __shfl_sync(CAS_FULL, ix, u + 1);
      uint32_t a0 = 0u, b0 = 0u;
      if (s0 + u < nsb) stream_clamp(i0, i1, lim, a0, b0);
      sa[u] = a0;
      nw[u] = (int)(b0 - a0);
      fast = fast && nw[u] <= 64;
    }
    const int64_t g = (int64_t)c * 32 + lane;  // this lane's block
    const bool valid = (int64_t)c * 4 + t < nsb;
    const int64_t gl = valid ? g : (int64_t)c * 32;
    if (fast) {
      const uint4 mk = ldg_once(reinterpret_cast<const uint4*>(w.mask) + gl);
      uint32_t fw[kRec];
      if (KEEP == 64) {
        const uint4 fA = __ldg(reinterpret_cast<const uint4*>(w.ssm + gl * 8));
        const uint4 fB = __ldg(reinterpret_cast<const uint4*>(w.ssm + gl * 8) + 1);
        fw[0] = fA.x;
        fw[1] = fA.y;
        fw[2] = fA.z;
        fw[3] = fA.w;
        fw[kRec > 4 ? 4 : 0] = fB.x;
        fw[kRec > 5 ? 5 : 0] = fB.y;
        fw[kRec > 6 ? 6 : 0] = fB.z;
        fw[kRec > 7 ? 7 : 0] = fB.w;
      } else {
#pragma unroll
        for (int i = 0; i < kRec; ++i) fw[i] = __ldg(w.ssm + gl * kRec + i);
      }
      bs.ms[1][lane] = valid ? __brev(mk.x) : 0u;
      bs.ms[2][lane] = valid ? __brev(mk.y) : 0u;
      bs.ms[3][lane] = valid ? __brev(mk.z) : 0u;
      bs.ms[4][lane] = valid ? __brev(mk.w) : 0u;
#pragma unroll
      for (int i = 0; i < kRec; ++i) bs.fs[i][lane] = fw[i];
      const uint32_t* gsx[4] = {w.sexp + sa[0], w.sexp + sa[1], w.sexp + sa[2], w.sexp + sa[3]};
      const int present = nsb - (int64_t)c * 4 < 4 ? (int)(nsb - (int64_t)c * 4) : 4;
      // staged bit of the '1' before the block's first code
      const int cq0 = block_code_term<2, KEEP>(gsx, nw, present, bs.st, lane, fast);
      const uint32_t ms_a = fenced(ms_a0), fs_a = fenced(fs_a0), st_a = fenced(st_a0);
      // cursors
      // row and block in the row (nbr >= 32: the chunk wraps at most once)
      uint32_t jb = valid ? jb0 + (uint32_t)lane : jb0;
      const uint32_t nr = row0 + (jb >= (uint32_t)nbr ? 1u : 0u);
      jb = jb >= (uint32_t)nbr ? jb - (uint32_t)nbr : jb;
      const uint32_t xbase = xs_a + 4u * jb * kBXRow;
      uint32_t xa = xbase - 4u;  // x address of the last found position (-1 at first)
      uint32_t Hp, Lp, Hc, Lc;
      bwindow(ms_a, 128u, 32, kBMaskRows - 3, Hp, Lp);
      bwindow(st_a, 4u, cq0 + 1, kBStreamWords - 3, Hc, Lc);
      uint32_t used = 0u, cor = 0u;
      float part[NV];
#pragma unroll
      for (int q = 0; q < NV; ++q) part[q] = 0.f;
#pragma unroll
      for (int gi = 0; gi < kGroups; ++gi) {
        if (gi > 0) {
          if (gi % kPosGroups == 0) {
            const int cur = min((int)(xa - xbase) >> 2, CAS_BLK - 1);
            xa = xbase + 4u * (uint32_t)cur;
            bwindow(ms_a, 128u, 33 + cur, kBMaskRows - 3, Hp, Lp);  // rows <= 7 since cur <= 127
          }
          bwindow(st_a, 4u, cq0 + 1 + (int)used, kBStreamWords - 3, Hc, Lc);
        }
        const uint32_t fo = lds_u32(fs_a + 128u * gi), fe = fo << 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (8 * gi + i >= KEEP) break;
          const uint32_t np = __clz(Hp) + 1u;  // distance to the next kept position
          xa = mad32(np, 4u, xa);
          Hp = shfl_wrap(Lp, Hp, np);
          Lp = shfl_wrap(0u, Lp, np);
          const uint32_t nc = __clz(Hc) + 1u;  // rank + 1
          const uint32_t E = lds_u32(lut_a - 4u + 4u * nc);
          Hc = shfl_wrap(Lc, Hc, nc);
          Lc = shfl_wrap(0u, Lc, nc);
          used += nc;
          cor |= np | nc;
          const int by = i >> 1;
          const uint32_t A = __byte_perm((i & 1) ? fo : fe, 0u, (by << 12) | (by << 8) | 0x44);
          const float val = __uint_as_float((A & 0x80700000u) | E);
#pragma unroll
          for (int q = 0; q < NV; ++q) part[q] = fmaf(val, lds_f32(xa + 4u * (uint32_t)(q * xfl)), part[q]);
        }
      }
      // a lane whose windows ran dry scans its block again (divergent, rare)
      bool bad = false;
      if (valid && (cor & 32u)) {
        const ScanSum<NV> r = block_walk_scan<NV>(ms_a, st_a, fs_a, lut_a, xbase, xfl, cq0, KEEP);
#pragma unroll
        for (int q = 0; q < NV; ++q) part[q] = r.part[q];
        bad = !r.ok;
      }
      fast = fast && !__any_sync(CAS_FULL, bad);
      if (fast && a.ymode) {  // the chunk is row nr, all of it
#pragma unroll
        for (int q = 0; q < NV; ++q) {
          const float sA = warp_sumf(part[q]);
          if (lane == 0) {
            float* d = a.y + (int64_t)q * w.N + nr;
            *d = a.ymode == 2 ? *d + sA : sA;
          }
        }
      } else if (fast) {
        const uint32_t nA = __shfl_sync(CAS_FULL, nr, 0);
        const uint32_t nB = __reduce_max_sync(CAS_FULL, valid ? nr : nA);  // rows of a chunk: nA and maybe nA + 1
#pragma unroll
        for (int q = 0; q < NV; ++q) {
          const float v = valid ? part[q] : 0.f;
          if (nA == nB) {
            const float sA = warp_sumf(v);
            if (lane == 0) atomicAdd(a.y + (int64_t)q * w.N + nA, sA);
          } else {
            const float sA = warp_sumf(nr == nA ? v : 0.f), sB = warp_sumf(nr == nA ? 0.f : v);
            if (lane == 0) {
              atomicAdd(a.y + (int64_t)q * w.N + nA, sA);
              atomicAdd(a.y + (int64_t)q * w.N + nB, sB);
            }
          }
        }
      }
      __syncwarp();
    }
    if (!fast) {  // decoded after the run; nothing of it was added
      if (lane == 0) fb[nfb] = c;
      ++nfb;
    }
  }
  // chunks the block walk did not take: the generic decoder, one superblock
  // at a time
  __syncwarp();
  uint8_t* code = reinterpret_cast<uint8_t*>(&bs);
  for (int i = 0; i < nfb; ++i) {
    const int cf = fb[i];
    float row[NV];  // the chunk's row sum (ymode: the chunk is one whole row)
#pragma unroll
    for (int q = 0; q < NV; ++q) row[q] = 0.f;
    int64_t nf = 0;
    for (int u = 0; u < 4; ++u) {
      const int64_t sf = (int64_t)cf * 4 + u;
      if (sf >= nsb) break;
      nf = sf / w.nsr;
      const int jf = (int)(sf - nf * w.nsr);
      float part[NV];
      word_fallback<NV>(w, sf, lut8, code, xs + (jf * CAS_SB + (lane >> 2)) * kBXRow + 32 * (lane & 3), xfl, part);
#pragma unroll
      for (int q = 0; q < NV; ++q) {
        const float r = warp_sumf(part[q]);
        row[q] += r;
        if (lane == 0 && !a.ymode) atomicAdd(a.y + (int64_t)q * w.N + nf, r);
      }
    }
    if (a.ymode && lane == 0) {
#pragma unroll
      for (int q = 0; q < NV; ++q) {
        float* d = a.y + (int64_t)q * w.N + nf;
        *d = a.ymode == 2 ? *d + row[q] : row[q];
      }
    }
  }
}

template <int NV>
size_t block_smem(int64_t nbr) {
  return (size_t)NV * block_x_floats((int)nbr) * 4 + kBXPad + kBWarps * sizeof(BlockStage);
}
// chunks per warp of a launch with g CTAs
inline int block_per(int64_t nsb, int g) {
  const int64_t nch = (nsb + 3) / 4;
  return (int)((nch + (int64_t)g * kBWarps - 1) / ((int64_t)g * kBWarps));
}

template <int NV, int KEEP>
int launch_block(const GemvArgs& a, cudaStream_t st) {
  auto kern = draft_gemv_block_kernel<NV, KEEP>;
  const int max_per_sm = occupancy((const void*)kern, kBThreads, block_smem<NV>(a.w.nbr));
  if (max_per_sm < 1) return CAS_ERR_CUDA;
  // one full wave (chunks are dealt round-robin over the CTAs), at most a CTA per chunk
  const int64_t nch = (a.w.nsb + 3) / 4;
  if (nch * 32 >= (int64_t)1 << 32) return CAS_ERR_INVALID;  // 32-bit block indices
  int g = (int)std::max<int64_t>(1, std::min<int64_t>(nch, (int64_t)sm_count() * max_per_sm));
  size_t smem = block_smem<NV>(a.w.nbr) + (size_t)kBWarps * block_per(a.w.nsb, g) * sizeof(int);
  const int per_sm = occupancy((const void*)kern, kBThreads, smem);
  if (per_sm < 1) return CAS_ERR_CUDA;
  if ((int64_t)g > (int64_t)sm_count() * per_sm) {
    g = sm_count() * per_sm;
    smem = block_smem<NV>(a.w.nbr) + (size_t)kBWarps * block_per(a.w.nsb, g) * sizeof(int);
  }
  return launch_k(kern, g, kBThreads, smem, st, a);
}

template <int NV>
int launch_word(const GemvArgs& a, cudaStream_t st) {
  auto kern = draft_gemv_word_kernel<NV>;
  // the smem of the fallback lists depends on the grid, the grid on the
  // occupancy: size the lists for the largest grid that can be resident
  const int max_per_sm = occupancy((const void*)kern, kThreads, word_smem<NV>(a.w.K));
  if (max_per_sm < 1) return CAS_ERR_CUDA;
  // at least 4 superblocks per warp: each CTA stages x once
  const int64_t need = (a.w.nsb + 4 * kWarps - 1) / (4 * kWarps);
  int g = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sm_count() * max_per_sm));
  size_t smem = word_smem<NV>(a.w.K) + (size_t)kWarps * word_per(a.w.nsb, g) * sizeof(int);
  const int per_sm = occupancy((const void*)kern, kThreads, smem);
  if (per_sm < 1) return CAS_ERR_CUDA;
  if ((int64_t)g > (int64_t)sm_count() * per_sm) {  // the lists cost a resident CTA per SM
    g = sm_count() * per_sm;
    smem = word_smem<NV>(a.w.K) + (size_t)kWarps * word_per(a.w.nsb, g) * sizeof(int);
  }
  return launch_k(kern, g, kThreads, smem, st, a);
}

// Whether the lane-per-block kernel takes a call (it alone forms the bf16
// input from an fp32 one in its staging). The 3-4 vector kernel (fast) covers
// Cassandra-1 with k = 64, m = 3 on rows of whole superblocks (K % 1024 == 0):
// every lane then owns exactly 16 ordinals in one 64-bit slice of one record.
template <int VAR>
bool block_path(const GemvArgs& a, int nvec) {
  return VAR == 1 && nvec <= 2 && a.w.m == 3 && (a.w.k == 64 || a.w.k == 38) && a.w.nbr % CAS_SB == 0 &&
         a.w.nbr >= 32 && block_smem<2>(a.w.nbr) <= 200 * 1024;
}

template <int VAR>
int dispatch(const GemvArgs& a, int nvec, cudaStream_t st) {
  const bool fast = a.w.k == 64 && a.w.m == 3 && a.w.nbr % CAS_SB == 0;
  if (block_path<VAR>(a, nvec)) {
    if (a.w.k == 64) return nvec == 1 ? launch_block<1, 64>(a, st) : launch_block<2, 64>(a, st);
    return nvec == 1 ? launch_block<1, 38>(a, st) : launch_block<2, 38>(a, st);
  }
  if (fast && VAR == 1 && nvec <= 2 && word_smem<2>(a.w.K) <= 200 * 1024)
    return nvec == 1 ? launch_word<1>(a, st) : launch_word<2>(a, st);
  if (fast && VAR == 1) {
    switch (nvec) {
      case 1: return launch_fast<1>(a, st);
      case 2: return launch_fast<2>(a, st);
      case 3: return launch_fast<3>(a, st);
      default: return launch_fast<4>(a, st);
    }
  }
  if (fast && VAR == 2 && nvec <= 2) return nvec == 1 ? launch_fast2<1>(a, st) : launch_fast2<2>(a, st);
  if (a.w.nbr % CAS_SB == 0) {
    switch (nvec) {
      case 1: return launch_runs<VAR, 1>(a, st);
      case 2: return launch_runs<VAR, 2>(a, st);
      case 3: return launch_runs<VAR, 3>(a, st);
      default: return launch_runs<VAR, 4>(a, st);
    }
  }
  switch (nvec) {
    case 1: return launch<VAR, 1>(a, st);
    case 2: return launch<VAR, 2>(a, st);
    case 3: return launch<VAR, 3>(a, st);
    default: return launch<VAR, 4>(a, st);
  }
}

}  // namespace

int set_first_wait_spins(uint32_t spins) {
  return cudaMemcpyToSymbol(g_first_wait_spins, &spins, sizeof(spins)) == cudaSuccess ? CAS_OK : CAS_ERR_CUDA;
}

int corrupt_status_gemv(bool clear) {
#ifdef CAS_DEBUG
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_corrupt_status, sizeof(int)) != cudaSuccess) return CAS_ERR_CUDA;
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(g_corrupt_status, &z, sizeof(int));
  }
  return v;
#else
  (void)clear;
  return 0;
#endif
}

int gemv_wait_status(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_wait_status, sizeof(int)) != cudaSuccess) return CAS_ERR_CUDA;
  if (clear && v) {
    int z = 0;
    cudaMemcpyToSymbol(g_gemv_wait_status, &z, sizeof(int));
  }
  return v;
}

}  // namespace cas

using namespace cas;

namespace cas {
namespace {

// y (+)= D(W) x; with xf, x = bf16(rmsnorm(xf) * gamma) written to xn first.
int draft_gemv_call(const cas_weights* W, const uint16_t* x, const float* xf, int xop, const uint16_t* gamma,
                    float eps, uint16_t* xn, int nvec, float* y, bool accumulate, cudaStream_t st) {
  int s = check_weights(W);
  if (s) return s;
  if (nvec < 1 || nvec > kMaxVec) return CAS_ERR_INVALID;
  if ((int64_t)nvec * W->K * 2 > 200 * 1024) return CAS_ERR_INVALID;  // x must fit in shared memory
  if (xop < 0 || xop > 3 || (xop != 0) != (xf != nullptr)) return CAS_ERR_INVALID;
  if (xf && (!xn || !aligned16(xf) || !aligned16(xn) || W->K < 1 || W->K > 16384)) return CAS_ERR_INVALID;
  if (xop == 1 && (!gamma || !(eps >= 0.f))) return CAS_ERR_INVALID;
  if (!xf && (!x || !aligned16(x))) return CAS_ERR_INVALID;
  if (W->N == 0 && !xf) return CAS_OK;  // nothing to write (y may be an empty tensor)
  if (W->N > 0 && (!y || !aligned16(y))) return CAS_ERR_INVALID;
  // superblock indices stay 32-bit, with room for the grid stride
  if (W->K > 0 && W->N * ((W->K / CAS_BLK + CAS_SB - 1) / CAS_SB) >= (1ll << 30)) return CAS_ERR_INVALID;
  GemvArgs a;
  a.w = make_view(W);
  for (int i = 0; i < 256; ++i) a.lut.v[i] = W->exp_of_rank[i];
  a.x = x;
  a.y = y;
  a.sexp_words = (int)(W->len[CAS_SEC_SPEC_EXP] / 4);
  const bool block = W->N > 0 && W->K > 0 && (W->p.variant == 1 ? block_path<1>(a, nvec) : block_path<2>(a, nvec));
  // rows of one chunk: the kernel writes each row once, no clearing first
  if (block && a.w.nbr == 32) a.ymode = accumulate ? 2 : 1;
  // y cleared first (a zero-fill kernel) unless the kernel writes every row once
  const bool clear = !accumulate && !a.ymode && W->N > 0;
  if (W->K == 0) return clear ? zero_f32(y, (int64_t)nvec * W->N, st) : CAS_OK;
  if (xf) {
    const bool fused = block;
    if (!fused) {  // the transformed input first (the glue kernel), then the plain GEMV
      if (xop == 1)
        s = cas_add_rmsnorm(const_cast<float*>(xf), nullptr, nvec, (int)W->K, gamma, eps, xn, st);
      else if (xop == 2)
        s = cas_f32_to_bf16(xf, (int64_t)nvec * W->K, xn, st);
      else
        s = cas_silu_mul(xf, nvec, (int)W->K, xn, st);
      if (s || W->N == 0) return s;
      a.x = xn;
    } else {
      a.xop = xop;
      a.xf = xf;
      a.gamma = gamma;
      a.xn = xn;
      a.eps = eps;
    }
  }
  if (clear)
    if (const int e = zero_f32(y, (int64_t)nvec * W->N, st)) return e;
  return W->p.variant == 1 ? dispatch<1>(a, nvec, st) : dispatch<2>(a, nvec, st);
}

}  // namespace
}  // namespace cas

extern "C" int cas_draft_gemv(const cas_weights* W, const uint16_t* x, int nvec, float* y, void* stream) {
  return draft_gemv_call(W, x, nullptr, 0, nullptr, 0.f, nullptr, nvec, y, false, (cudaStream_t)stream);
}

extern "C" int cas_draft_gemv_accumulate(const cas_weights* W, const uint16_t* x, int nvec, float* y, void* stream) {
  return draft_gemv_call(W, x, nullptr, 0, nullptr, 0.f, nullptr, nvec, y, true, (cudaStream_t)stream);
}

extern "C" int cas_draft_gemv_rmsnorm(const cas_weights* W, const float* x, int nvec, const uint16_t* gamma, float eps,
                                      uint16_t* xn, float* y, void* stream) {
  if (!x) return CAS_ERR_INVALID;
  return draft_gemv_call(W, nullptr, x, 1, gamma, eps, xn, nvec, y, false, (cudaStream_t)stream);
}

extern "C" int cas_draft_gemv_f32(const cas_weights* W, const float* x, int nvec, int op, const uint16_t* gamma,
                                  float eps, uint16_t* xn, float* y, int accumulate, void* stream) {
  if (!x || op < CAS_X_ROUND || op > CAS_X_SILU_MUL) return CAS_ERR_INVALID;
  const int xop = op == CAS_X_RMSNORM ? 1 : op == CAS_X_ROUND ? 2 : 3;
  return draft_gemv_call(W, nullptr, x, xop, gamma, eps, xn, nvec, y, accumulate != 0, (cudaStream_t)stream);
}
