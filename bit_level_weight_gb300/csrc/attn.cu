// attn.cu - attention over the compressed KV cache.
//
// Draft decode (Cassandra blog review, section 3.1: the draft reads only the
// speculation data, zero-filled): softmax(q K~^T / sqrt(128)) V~ with K~, V~
// the draft values of the cache, then the exact bf16 tail tokens.
// Verify: T queries over the exact cache (both streams merged, lossless),
// causal among the last T tokens.
//
// Split over tokens (flash decoding): a CTA takes one (sequence, kv head,
// token chunk). The number of chunks is fixed at launch so that the grid is
// one wave of resident CTAs; each CTA derives its range of 32-token steps
// from the sequence length held on the device. Per 32-token step its 4 warps
// each decode one superblock (8 tokens) of K and of V. Kernels:
//   attn_draft_fused_kernel  draft, up to 4 query vectors per kv head: K
//                            scores computed in the per-lane decode, V into a
//                            bf16 tile, CUDA-core P.V (lane = 4 dimensions);
//   attn_chunk_kernel        draft with more query vectors: K and V tiles,
//                            scores with lane = token, CUDA-core P.V;
//   attn_mma_kernel          verify: K and V tiles, S = Q K^T, online softmax
//                            and P.V on tensor cores.
// GQA: the q heads h*G .. h*G+G-1 (times the T query tokens) share kv head h.
// Chunk partials (max, sum, unnormalised output) go to the workspace; a
// combine kernel merges them, adds the tail tokens and normalises.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "kvview.cuh"
#include "blockwalk.cuh"
#include "lanedec.cuh"
#include "mma.cuh"
#include "sbdecode.cuh"

namespace cas {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = 4;
constexpr int kChunk = 256;      // smallest chunk the workspace is sized for
constexpr int kStepTok = 32;     // tokens per step (4 superblocks)
constexpr int kRow = CAS_BLK + 8;  // bf16 tile row stride (272 B: conflict-free 16-byte rows)
constexpr int kPart = CAS_BLK + 2; // floats per partial: o[128], m, l
constexpr int kTileSlack = 1024;   // bytes after the verify V tile: stores of a failed walk stay inside
constexpr int kMaxBatch = 8;
constexpr int kMaxT = 16;

constexpr int kQvPerCta = 32;  // query vectors per CTA (8 per warp)
// per-warp decode scratch: the cursor decoder's staged stream, or kept codes +
// pruned codes + the Cassandra-2 residual words of one superblock
// (a multiple of 16 bytes: the tile decoder reads its position arrays as uint4)
// Cassandra-1 caches need the stage or 2 x 1024 code bytes, Cassandra-2 caches
// also the residual words of a superblock.
constexpr int kScratchC1 = (((int)sizeof(TileStage) > 2048 ? (int)sizeof(TileStage) : 2048) + 15) & ~15;
constexpr int kScratchC2 =
    (((int)sizeof(TileStage) > 2048 + 4 * kResWords ? (int)sizeof(TileStage) : 2048 + 4 * kResWords) + 15) & ~15;
static_assert(kScratchC1 % 16 == 0 && kScratchC2 % 16 == 0 && alignof(TileStage) <= 16, "per-warp scratch alignment");
static_assert(kScratchC2 >= (int)sizeof(TileStage2) && alignof(TileStage2) <= 16, "Cassandra-2 stage fits");
// The draft decodes no pruned codes: its generic decoder needs 1024 code bytes,
// so a Cassandra-1 draft takes just the cursor stage (8 resident CTAs of the
// fused kernel fit in shared memory).
constexpr int kScratchDraftC1 = (((int)sizeof(TileStage) > 1024 ? (int)sizeof(TileStage) : 1024) + 15) & ~15;
static_assert(kScratchDraftC1 <= kScratchC1 && kScratchDraftC1 % 16 == 0, "draft scratch");

struct AttnArgs {
  KvDev kv[kMaxBatch];
  const uint16_t* q;  // [B][T][Hq][128]
  float* part;        // [B][T][Hq][nchunk][kPart]
  int B, T, Hq, G, nchunk, ngroups, qv_alloc;
  int scr_warp;       // per-warp decode scratch bytes (kScratchC1 or kScratchC2)
  float scale;
};

__device__ __forceinline__ float warp_maxf(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(CAS_FULL, v, d));
  return v;
}

// Decodes superblock sb of stream st (n tokens) into tile rows [row0, row0+8)
// as bf16; rows of tokens that do not exist are zero.
template <bool FULL>
__device__ __forceinline__ void decode_sb_tile(const KvDev& d, int st, int64_t n, int64_t sb, uint16_t* tile, int row0,
                                               const uint8_t* lut, uint8_t* scratch, int lane) {
  const int64_t nsb = (n + CAS_SB - 1) / CAS_SB;
  if (sb < nsb && d.variant == 1 && d.k == 64 && d.m == 3 && CAS_SB * (sb + 1) <= n) {
    // whole superblock of 8 tokens: per-lane cursors
    const uint32_t* sidx = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, st);
    const uint32_t* vidx = (const uint32_t*)kv_sec(d, CAS_KV_VER_SBIDX, st);
    const uint32_t a0 = sidx[sb], a1 = sidx[sb + 1];
    const uint32_t v0 = FULL ? vidx[sb] : 0u, v1 = FULL ? vidx[sb + 1] : 0u;
    if (lane_sb_tile<FULL>((const uint32_t*)kv_sec(d, CAS_KV_MASK, st) + sb * 32,
                           (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, st) + sb * 64,
                           (const uint32_t*)kv_sec(d, CAS_KV_VER_LO, st) + sb * 64,
                           (const uint32_t*)kv_sec(d, CAS_KV_VER_PR, st) + sb * 128,
                           (const uint32_t*)kv_sec(d, CAS_KV_SPEC_EXP, st) + a0, (int)(a1 - a0),
                           (const uint32_t*)kv_sec(d, CAS_KV_VER_EXP, st) + v0, (int)(v1 - v0), lut,
                           *reinterpret_cast<TileStage*>(scratch), tile + row0 * kRow, kRow, lane))
      return;
  }
  if (sb < nsb && d.variant == 1 && CAS_SB * (sb + 1) <= n && !(d.k == 64 && d.m == 3)) {
    // whole superblock, other k or m: per-lane runs
    const uint32_t* sidx = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, st);
    const uint32_t* vidx = (const uint32_t*)kv_sec(d, CAS_KV_VER_SBIDX, st);
    const uint32_t a0 = sidx[sb], a1 = sidx[sb + 1];
    const uint32_t v0 = FULL ? vidx[sb] : 0u, v1 = FULL ? vidx[sb + 1] : 0u;
    TileStage& ts = *reinterpret_cast<TileStage*>(scratch);
    if (runs_sb_tile<FULL>((const uint32_t*)kv_sec(d, CAS_KV_MASK, st) + sb * 32,
                           (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, st) + sb * CAS_SB * d.rec_sm, d.rec_sm,
                           (const uint32_t*)kv_sec(d, CAS_KV_VER_LO, st) + sb * CAS_SB * d.rec_lo, d.rec_lo,
                           (const uint32_t*)kv_sec(d, CAS_KV_VER_PR, st) + sb * CAS_SB * d.rec_pr, d.rec_pr,
                           (const uint32_t*)kv_sec(d, CAS_KV_SPEC_EXP, st) + a0, (int)(a1 - a0),
                           (const uint32_t*)kv_sec(d, CAS_KV_VER_EXP, st) + v0, (int)(v1 - v0), d.k, d.m, lut,
                           ts.us, ts.kpos, tile + row0 * kRow, kRow, lane))
      return;
  }
  if (sb < nsb && d.variant == 2 && CAS_SB * (sb + 1) <= n) {
    // whole Cassandra-2 superblock: per-lane runs
    const uint32_t* didx = (const uint32_t*)kv_sec(d, CAS_KV_VER_D_SBIDX, st);
    const uint32_t* ridx = (const uint32_t*)kv_sec(d, CAS_KV_VER_RES_SBIDX, st);
    const uint32_t* vidx = (const uint32_t*)kv_sec(d, CAS_KV_VER_SBIDX, st);
    const uint32_t d0 = FULL ? didx[sb] : 0u, d1 = FULL ? didx[sb + 1] : 0u;
    const uint32_t v0 = FULL ? vidx[sb] : 0u, v1 = FULL ? vidx[sb + 1] : 0u;
    const uint32_t r0 = FULL ? ridx[sb] : 0u;
    if (runs_sb_tile_c2<FULL>((const uint32_t*)kv_sec(d, CAS_KV_MASK, st) + sb * 32,
                              (const uint32_t*)kv_sec(d, CAS_KV_SPEC_Q, st) + sb * CAS_SB * d.rec_q, d.rec_q,
                              kv_sec(d, CAS_KV_SPEC_MX, st) + sb * 32,
                              (const uint32_t*)kv_sec(d, CAS_KV_VER_D, st) + d0, (int)(d1 - d0),
                              (const uint32_t*)kv_sec(d, CAS_KV_VER_RES, st) + r0,
                              (const uint32_t*)kv_sec(d, CAS_KV_VER_PR, st) + sb * CAS_SB * d.rec_pr, d.rec_pr,
                              (const uint32_t*)kv_sec(d, CAS_KV_VER_EXP, st) + v0, (int)(v1 - v0), d.k, d.m, lut,
                              *reinterpret_cast<TileStage2*>(scratch), tile + row0 * kRow, kRow, lane))
      return;
  }
  // generic decoder (other k, m, Cassandra-2, partial superblocks, fallback):
  // lane L writes mask word L, zeros past the stream's tokens
  uint16_t* dst = tile + (row0 + (lane >> 2)) * kRow + 32 * (lane & 3);
  int nb = 0;
  if (sb < nsb && d.variant == 1) {
    SbScratch sc{scratch, scratch + 1024, nullptr};
    WView w = kv_stream_view(d, st, n);
    SbInfo in = sb_prepare<1, FULL>(w, sb, lut, sc, lane);
    nb = in.nb;
    if (lane < 4 * nb) sb_rebuild_store<1, FULL>(w, in, sc, lane, dst);
  } else if (sb < nsb) {
    SbScratch sc{scratch, scratch + 1024, reinterpret_cast<uint32_t*>(scratch + 2048)};
    WView w = kv_stream_view(d, st, n);
    SbInfo in = sb_prepare<2, FULL>(w, sb, lut, sc, lane);
    nb = in.nb;
    if (lane < 4 * nb) sb_rebuild_store<2, FULL>(w, in, sc, lane, dst);
  }
  if (lane >= 4 * nb) {
    uint4* z = reinterpret_cast<uint4*>(dst);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    z[0] = zero;
    z[1] = zero;
    z[2] = zero;
    z[3] = zero;
  }
  __syncwarp();
}

template <bool FULL, int QPW>
__global__ void __launch_bounds__(kThreads) attn_chunk_kernel(AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Kt = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Vt = Kt + kStepTok * kRow;
  float* Qs = reinterpret_cast<float*>(Vt + kStepTok * kRow);  // [nq][128], pre-scaled
  uint8_t* lutK = reinterpret_cast<uint8_t*>(Qs + a.qv_alloc * CAS_BLK);
  uint8_t* lutV = lutK + 256;
  uint8_t* scr = lutV + 256;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t* wscr = scr + warp * a.scr_warp;
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z / a.ngroups;
  const int qv0 = (blockIdx.z % a.ngroups) * kQvPerCta;
  const KvDev& d = a.kv[b];
  const int H = d.H, T = a.T, G = a.G, nq = min(T * G - qv0, kQvPerCta);
  const int64_t n = *(volatile const int64_t*)&kv_state(d)->n_tokens;
  const int64_t steps = (n + kStepTok - 1) / kStepTok;
  const int64_t t_begin = steps * chunk / a.nchunk * kStepTok;
  const int64_t t_end = min(n, steps * (chunk + 1) / a.nchunk * kStepTok);

  // query vectors qv = j * G + g (query token j, head h*G+g), scaled; this
  // CTA takes qv0 .. qv0 + nq - 1 (local index qv - qv0)
  for (int i = threadIdx.x; i < nq * CAS_BLK; i += kThreads) {
    int qv = qv0 + i / CAS_BLK, dd = i % CAS_BLK;
    int j = qv / G, g = qv % G;
    Qs[i] = bf2f(a.q[(((int64_t)b * T + j) * a.Hq + h * G + g) * CAS_BLK + dd]) * a.scale;
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) {
    lutK[i] = kv_exp_of_rank(d, h)[i];
    lutV[i] = kv_exp_of_rank(d, H + h)[i];
  }
  __syncthreads();

  float m_[QPW], l_[QPW], o_[QPW][4];
#pragma unroll
  for (int i = 0; i < QPW; ++i) {
    m_[i] = -INFINITY;
    l_[i] = 0.f;
    o_[i][0] = o_[i][1] = o_[i][2] = o_[i][3] = 0.f;
  }
  for (int64_t t0 = t_begin; t0 < t_end; t0 += kStepTok) {
    int64_t sb = t0 / CAS_SB + warp;
    decode_sb_tile<FULL>(d, h, n, sb, Kt, warp * CAS_SB, lutK, wscr, lane);
    decode_sb_tile<FULL>(d, H + h, n, sb, Vt, warp * CAS_SB, lutV, wscr, lane);
    __syncthreads();
    const int64_t tok = t0 + lane;
    // scores: lane = token
    float s[QPW];
#pragma unroll
    for (int i = 0; i < QPW; ++i) s[i] = 0.f;
    const uint4* krow = reinterpret_cast<const uint4*>(Kt + lane * kRow);
    for (int c = 0; c < CAS_BLK / 8; ++c) {
      const uint4 k8 = krow[c];
      const float k0 = __uint_as_float(k8.x << 16), k1 = __uint_as_float(k8.x & 0xFFFF0000u);
      const float k2 = __uint_as_float(k8.y << 16), k3 = __uint_as_float(k8.y & 0xFFFF0000u);
      const float k4 = __uint_as_float(k8.z << 16), k5 = __uint_as_float(k8.z & 0xFFFF0000u);
      const float k6 = __uint_as_float(k8.w << 16), k7 = __uint_as_float(k8.w & 0xFFFF0000u);
#pragma unroll
      for (int i = 0; i < QPW; ++i) {
        int qv = warp + kWarps * i;
        if (qv < nq) {
          const float4 qa = reinterpret_cast<const float4*>(Qs + qv * CAS_BLK)[2 * c];
          const float4 qb = reinterpret_cast<const float4*>(Qs + qv * CAS_BLK)[2 * c + 1];
          s[i] = fmaf(qa.x, k0, fmaf(qa.y, k1, fmaf(qa.z, k2, fmaf(qa.w, k3, s[i]))));
          s[i] = fmaf(qb.x, k4, fmaf(qb.y, k5, fmaf(qb.z, k6, fmaf(qb.w, k7, s[i]))));
        }
      }
    }
#pragma unroll
    for (int i = 0; i < QPW; ++i) {
      int qv = warp + kWarps * i;
      if (qv >= nq) continue;
      int64_t last = FULL ? n - T + (qv0 + qv) / G : n - 1;  // causal among the last T tokens (verify)
      float si = (tok < t_end && tok <= last) ? s[i] : -INFINITY;
      float mx = warp_maxf(si);
      float mnew = fmaxf(m_[i], mx);
      float p = (si == -INFINITY) ? 0.f : __expf(si - mnew);
      float corr = (m_[i] == -INFINITY) ? 0.f : __expf(m_[i] - mnew);
      if (mnew == -INFINITY) corr = 1.f;
      l_[i] = l_[i] * corr + warp_sumf(p);
      m_[i] = mnew;
      float acc0 = o_[i][0] * corr, acc1 = o_[i][1] * corr, acc2 = o_[i][2] * corr, acc3 = o_[i][3] * corr;
      for (int t = 0; t < kStepTok; ++t) {
        float pt = __shfl_sync(CAS_FULL, p, t);
        const uint2 v4 = reinterpret_cast<const uint2*>(Vt + t * kRow)[lane];
        acc0 = fmaf(pt, __uint_as_float(v4.x << 16), acc0);
        acc1 = fmaf(pt, __uint_as_float(v4.x & 0xFFFF0000u), acc1);
        acc2 = fmaf(pt, __uint_as_float(v4.y << 16), acc2);
        acc3 = fmaf(pt, __uint_as_float(v4.y & 0xFFFF0000u), acc3);
      }
      o_[i][0] = acc0; o_[i][1] = acc1; o_[i][2] = acc2; o_[i][3] = acc3;
    }
    __syncthreads();
  }
  // partials
#pragma unroll
  for (int i = 0; i < QPW; ++i) {
    int qv = warp + kWarps * i;
    if (qv >= nq) continue;
    int j = (qv0 + qv) / G, g = (qv0 + qv) % G;
    float* dst = a.part + ((((int64_t)b * T + j) * a.Hq + h * G + g) * a.nchunk + chunk) * kPart;
    reinterpret_cast<float2*>(dst)[2 * lane] = make_float2(o_[i][0], o_[i][1]);
    reinterpret_cast<float2*>(dst)[2 * lane + 1] = make_float2(o_[i][2], o_[i][3]);
    if (lane == 0) {
      dst[CAS_BLK] = m_[i];
      dst[CAS_BLK + 1] = l_[i];
    }
  }
}

// ---------------------------------------------------------------- exact tiles by block walks
// Cassandra-1 caches with k = 64, m = 3: superblock sb (8 tokens) of the K and
// V streams of head h rebuilt exactly into tile rows row0 .. row0+7 of Kt and
// Vt by one warp (blockwalk.cuh). Lane 8t + j walks token j of stream K (t <
// 2) or V (t >= 2): its 64 kept values for even t (sign and 3 high mantissa
// bits joined with the 4 cut bits), its 64 pruned values for odd t (the pruned
// byte), so the four staged code streams are K kept, K pruned, V kept, V
// pruned. A group of 8 values whose positions or codes do not all end in the
// 64-bit windows (a code longer than the window: an exponent the calibrated
// table ranks far down) is taken by scanning. Streams longer than the stage go
// to decode_sb_tile. Returns false when a walk stepped 32 or more anyway (a
// gap of 32 or more, a code of 31 to 63 bits inside a full window): its rows
// are then wrong and its stores may have run up to 782 bytes past its row.
struct KvBlockStage {
  BlockStreams<3, 80> st;  // codes: K kept, K pruned, V kept, V pruned
  uint32_t ms[7][32];      // row i, column l: bit-reversed word i of lane l's positions; rows 4-6 zero
};
static_assert(sizeof(KvBlockStage) % 16 == 0, "stage alignment");

__device__ __forceinline__ bool kv_block_tiles(const KvDev& d, int h, int64_t n, int64_t sb, uint16_t* Kt, uint16_t* Vt,
                                            int row0, const uint32_t* lut7k, const uint32_t* lut7v,
                                            const uint8_t* lutK, const uint8_t* lutV, uint8_t* scratch, int lane) {
  KvBlockStage& vs = *reinterpret_cast<KvBlockStage*>(scratch);
  const int H = d.H, t = lane >> 3, j = lane & 7;
  const bool pruned = t & 1;
  const int st = t < 2 ? h : H + h;
  const int64_t nsb = (n + CAS_SB - 1) / CAS_SB, tok = sb * CAS_SB + j;
  const bool valid = sb < nsb && tok < n;
  uint16_t* row = (t < 2 ? Kt : Vt) + (row0 + j) * kRow;
  if (!valid) {  // a token past the cache: a zero row
    uint4* z = reinterpret_cast<uint4*>(row);
    for (int i = (int)pruned; i < CAS_BLK / 8; i += 2) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (sb >= nsb) {
    __syncwarp();
    return true;
  }
  const uint32_t* gs[4];
  int nw[4];
  bool fast = true;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int su = u < 2 ? h : H + h;
    uint32_t a0, b0;
    if (u & 1)
      stream_range((const uint32_t*)kv_sec(d, CAS_KV_VER_SBIDX, su), sb, (uint32_t)d.cap_b, a0, b0);
    else
      stream_range((const uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, su), sb, (uint32_t)d.cap_a, a0, b0);
    gs[u] = (const uint32_t*)kv_sec(d, (u & 1) ? CAS_KV_VER_EXP : CAS_KV_SPEC_EXP, su) + a0;
    nw[u] = (int)(b0 - a0);
    fast = fast && nw[u] <= BlockStreams<3, 80>::kWords;
  }
  int q0 = 0;
  if (fast) {
    block_streams_init(vs.st, lane);
#pragma unroll
    for (int r = 4; r < 7; ++r) vs.ms[r][lane] = 0u;
    const uint4 mk = __ldg(reinterpret_cast<const uint4*>(kv_sec(d, CAS_KV_MASK, st)) + (valid ? tok : 0));
    const uint32_t inv = pruned ? 0xFFFFFFFFu : 0u;
    vs.ms[0][lane] = valid ? __brev(mk.x ^ inv) : 0u;
    vs.ms[1][lane] = valid ? __brev(mk.y ^ inv) : 0u;
    vs.ms[2][lane] = valid ? __brev(mk.z ^ inv) : 0u;
    vs.ms[3][lane] = valid ? __brev(mk.w ^ inv) : 0u;
    q0 = block_code_term<3, 64>(gs, nw, CAS_SB * (sb + 1) <= n ? 4 : 0, vs.st, lane, fast);
  }
  if (!fast) {  // streams longer than the stage, or too few codes: the tile decoder
    __syncwarp();
    decode_sb_tile<true>(d, h, n, sb, Kt, row0, lutK, scratch, lane);
    decode_sb_tile<true>(d, H + h, n, sb, Vt, row0, lutV, scratch, lane);
    return true;
  }
  const uint32_t ms_a = fenced(smem_addr(&vs.ms[0][lane])), st_a = fenced(smem_addr(&vs.st.w[t][0]));
  const uint32_t lut_a = smem_addr(t < 2 ? lut7k : lut7v);
  const uint32_t* ra = pruned ? (const uint32_t*)kv_sec(d, CAS_KV_VER_PR, st) + tok * 16
                              : (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, st) + tok * 8;
  const uint32_t* rb = pruned ? ra + 1 : (const uint32_t*)kv_sec(d, CAS_KV_VER_LO, st) + tok * 8;
  const int rs = pruned ? 2 : 1;
  const uint32_t tb = smem_addr(row);
  uint32_t ta = tb - 2u;
  uint32_t cor = 0u;
  if (valid) {
    uint32_t Hp, Lp, Hc, Lc;
    bwindow(ms_a, 128u, 0, 4, Hp, Lp);
    bwindow(st_a, 4u, q0 + 1, BlockStreams<3, 80>::kRow - 3, Hc, Lc);
    uint32_t used = 0u;
    uint32_t an = __ldg(ra), bn = __ldg(rb);
#pragma unroll 1
    for (int gi = 0; gi < 8; ++gi) {
      const uint32_t aw = an, bw = bn;
      if (gi < 7) {
        an = __ldg(ra + rs * (gi + 1));
        bn = __ldg(rb + rs * (gi + 1));
      }
      if (gi > 0) {
        const int cur = min((int)(ta - tb) >> 1, CAS_BLK - 1);
        ta = tb + 2u * (uint32_t)cur;
        bwindow(ms_a, 128u, cur + 1, 4, Hp, Lp);
        bwindow(st_a, 4u, q0 + 1 + (int)used, BlockStreams<3, 80>::kRow - 3, Hc, Lc);
      }
      // bytes [s f6 .. f0] of the group's values 0, 2, 4, 6 (ev) and 1, 3, 5, 7 (od)
      const uint32_t ev = pruned ? __byte_perm(aw, bw, 0x6420) : ((aw << 4) & 0xF0F0F0F0u) | (bw & 0x0F0F0F0Fu);
      const uint32_t od = pruned ? __byte_perm(aw, bw, 0x7531) : (aw & 0xF0F0F0F0u) | ((bw >> 4) & 0x0F0F0F0Fu);
      if (__popc(Hp) + __popc(Lp) < 8 || __popc(Hc) + __popc(Lc) < 8) {  // this group by scanning
        int cur = (int)(ta - tb) >> 1, qt = q0 + (int)used;
        for (int i = 0; i < 8; ++i) {
          const int pb = bnext_one(ms_a, 128u, cur + 1, 6);
          const int eb = bnext_one(st_a, 4u, qt + 1, BlockStreams<3, 80>::kRow - 1);
          if (pb < 0 || pb >= CAS_BLK || eb < 0) {
            cor |= 32u;
            break;
          }
          const uint32_t E = lds_u32(lut_a + 4u * (uint32_t)min(eb - qt - 1, 255));
          used += (uint32_t)(eb - qt);
          qt = eb;
          cur = pb;
          const uint32_t by = (((i & 1) ? od : ev) >> (8 * (i >> 1))) & 0xFFu;
          sts_u16(tb + 2u * (uint32_t)cur, ((by & 0x80u) << 8) | E | (by & 0x7Fu));
        }
        ta = tb + 2u * (uint32_t)max(cur, -1);
        continue;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t np = __clz(Hp) + 1u;
        ta = mad32(np, 2u, ta);
        Hp = shfl_wrap(Lp, Hp, np);
        Lp = shfl_wrap(0u, Lp, np);
        const uint32_t nc = __clz(Hc) + 1u;  // rank + 1
        const uint32_t E = lds_u32(lut_a - 4u + 4u * nc);
        Hc = shfl_wrap(Lc, Hc, nc);
        Lc = shfl_wrap(0u, Lc, nc);
        used += nc;
        cor |= np | nc;
        const uint32_t A = __byte_perm((i & 1) ? od : ev, 0u, (uint32_t)(i >> 1) * 0x11u | 0x4400u);
        sts_u16(ta, (A & 0x807Fu) | E);
      }
    }
  }
  return !__any_sync(CAS_FULL, valid && (cor & 32u));
}

// Tensor-core variant of the chunk kernel (up to 32 query vectors per CTA in
// MT m16 tiles): per 32-token step, after the K and V superblocks are
// decoded into the tiles, S = Q K^T (mma m16n8k16, bf16 inputs, fp32
// accumulators; Q is the unscaled bf16 query, the 1/sqrt(128) scale is applied
// to S in fp32), the online softmax runs on the S fragments (rows shared by
// the 4 lanes of a quad), and O += P V with P split into two bf16 terms
// (p = hi + lo, |p - hi - lo| <= 2^-17 p) so the product keeps fp32-like
// precision. With MT = 2, warps 2i and 2i+1 take m-tile i and split the 128
// output dimensions; with MT = 1 the 4 warps split them four ways (each
// warp recomputes the m-tile's S, which is cheap next to the decode).
template <bool FULL, int MT>
__global__ void __launch_bounds__(kThreads, MT == 2 ? 4 : 5) attn_mma_kernel(AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Kt = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Vt = Kt + kStepTok * kRow;
  uint16_t* Qt = Vt + kStepTok * kRow + kTileSlack / 2;  // [16 MT][kRow], rows >= nq zero
  uint8_t* lutK = reinterpret_cast<uint8_t*>(Qt + 16 * MT * kRow);
  uint8_t* lutV = lutK + 256;
  uint32_t* lut7K = reinterpret_cast<uint32_t*>(lutV + 256);  // exponent << 7 by rank
  uint32_t* lut7V = lut7K + 256;
  uint8_t* scr = reinterpret_cast<uint8_t*>(lut7V + 256);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t* wscr = scr + warp * a.scr_warp;
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z / a.ngroups;
  const int qv0 = (blockIdx.z % a.ngroups) * kQvPerCta;
  const KvDev& d = a.kv[b];
  const int H = d.H, T = a.T, G = a.G, nq = min(T * G - qv0, kQvPerCta);
  const int64_t n = *(volatile const int64_t*)&kv_state(d)->n_tokens;
  const int64_t steps = (n + kStepTok - 1) / kStepTok;
  const int64_t t_begin = steps * chunk / a.nchunk * kStepTok;
  const int64_t t_end = min(n, steps * (chunk + 1) / a.nchunk * kStepTok);

  for (int i = threadIdx.x; i < 16 * MT * CAS_BLK; i += kThreads) {
    const int r = i / CAS_BLK, dd = i % CAS_BLK;
    uint16_t v = 0;
    if (r < nq) {
      const int qv = qv0 + r, j = qv / G, g = qv % G;
      v = a.q[(((int64_t)b * T + j) * a.Hq + h * G + g) * CAS_BLK + dd];
    }
    Qt[r * kRow + dd] = v;
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) {
    lutK[i] = kv_exp_of_rank(d, h)[i];
    lutV[i] = kv_exp_of_rank(d, H + h)[i];
    lut7K[i] = (uint32_t)lutK[i] << 7;
    lut7V[i] = (uint32_t)lutV[i] << 7;
  }
  __syncthreads();
  const bool walk = FULL && d.variant == 1 && d.k == 64 && d.m == 3;

  constexpr int WPM = 4 / MT;       // warps per m-tile
  constexpr int NT = 16 / WPM;      // 8-dim output tiles per warp
  const int mt = MT == 1 ? 0 : warp / WPM;
  const int dbase = (warp % WPM) * NT * 8;
  const int g = lane >> 2, tq = lane & 3;
  const int r0 = mt * 16 + g, r1 = r0 + 8;  // local query rows of this lane
  // last token each row may attend to (causal among the last T tokens for verify); -1: no row
  const int64_t last0 = r0 < nq ? (FULL ? n - T + (qv0 + r0) / G : n - 1) : -1;
  const int64_t last1 = r1 < nq ? (FULL ? n - T + (qv0 + r1) / G : n - 1) : -1;
  float o[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const bool active = mt * 16 < nq;

  for (int64_t t0 = t_begin; t0 < t_end; t0 += kStepTok) {
    const int64_t sb = t0 / CAS_SB + warp;
    bool bad = false;
    if (walk) {
      bad = !kv_block_tiles(d, h, n, sb, Kt, Vt, warp * CAS_SB, lut7K, lut7V, lutK, lutV, wscr, lane);
    } else {
      decode_sb_tile<FULL>(d, h, n, sb, Kt, warp * CAS_SB, lutK, wscr, lane);
      decode_sb_tile<FULL>(d, H + h, n, sb, Vt, warp * CAS_SB, lutV, wscr, lane);
    }
    if (__syncthreads_or(bad)) {  // a failed walk may have stored into other warps' rows: rebuild all
      decode_sb_tile<FULL>(d, h, n, sb, Kt, warp * CAS_SB, lutK, wscr, lane);
      decode_sb_tile<FULL>(d, H + h, n, sb, Vt, warp * CAS_SB, lutV, wscr, lane);
      __syncthreads();
    }
    if (active) {
      // S = Q K^T: 16 rows x 32 tokens
      float s[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < CAS_BLK / 16; ++ks) {
        uint32_t af[4];
        ldmatrix_x4(af, Qt + (mt * 16 + (lane & 15)) * kRow + ks * 16 + (lane >> 4) * 8);
#pragma unroll
        for (int nt2 = 0; nt2 < 2; ++nt2) {
          uint32_t bf[4];
          const int mi = lane >> 3;
          ldmatrix_x4(bf, Kt + (nt2 * 16 + (mi >> 1) * 8 + (lane & 7)) * kRow + ks * 16 + (mi & 1) * 8);
          mma_bf16(s[2 * nt2], af, bf[0], bf[1]);
          mma_bf16(s[2 * nt2 + 1], af, bf[2], bf[3]);
        }
      }
      // online softmax on the fragments
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t tok = t0 + nt * 8 + 2 * tq + (e & 1);
          const bool ok = tok < t_end && tok <= (e < 2 ? last0 : last1);
          s[nt][e] = ok ? s[nt][e] * a.scale : -INFINITY;
        }
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(CAS_FULL, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(CAS_FULL, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(CAS_FULL, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(CAS_FULL, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float c0 = mn0 == -INFINITY ? 1.f : (m0 == -INFINITY ? 0.f : __expf(m0 - mn0));
      const float c1 = mn1 == -INFINITY ? 1.f : (m1 == -INFINITY ? 0.f : __expf(m1 - mn1));
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mref = e < 2 ? mn0 : mn1;
          const float p = s[nt][e] == -INFINITY ? 0.f : __expf(s[nt][e] - mref);
          s[nt][e] = p;
        }
        sum0 += s[nt][0] + s[nt][1];
        sum1 += s[nt][2] + s[nt][3];
      }
      sum0 += __shfl_xor_sync(CAS_FULL, sum0, 1);
      sum0 += __shfl_xor_sync(CAS_FULL, sum0, 2);
      sum1 += __shfl_xor_sync(CAS_FULL, sum1, 1);
      sum1 += __shfl_xor_sync(CAS_FULL, sum1, 2);
      l0 = l0 * c0 + sum0;
      l1 = l1 * c1 + sum1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        o[i][0] *= c0;
        o[i][1] *= c0;
        o[i][2] *= c1;
        o[i][3] *= c1;
      }
      // O += P V over two 16-token k-steps; P = hi + lo in bf16
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const float* sp = s[2 * kk + half];
          const uint32_t h01 = pack_bf16x2(sp[0], sp[1]), h23 = pack_bf16x2(sp[2], sp[3]);
          const float e0 = sp[0] - __uint_as_float(h01 << 16), e1 = sp[1] - __uint_as_float(h01 & 0xFFFF0000u);
          const float e2 = sp[2] - __uint_as_float(h23 << 16), e3 = sp[3] - __uint_as_float(h23 & 0xFFFF0000u);
          ph[2 * half] = h01;
          ph[2 * half + 1] = h23;
          pl[2 * half] = pack_bf16x2(e0, e1);
          pl[2 * half + 1] = pack_bf16x2(e2, e3);
        }
        // A fragment order: (row g, k lo), (row g+8, k lo), (row g, k hi), (row g+8, k hi)
        const uint32_t ah[4] = {ph[0], ph[1], ph[2], ph[3]};
        const uint32_t al[4] = {pl[0], pl[1], pl[2], pl[3]};
#pragma unroll
        for (int i = 0; i < NT; i += 2) {
          uint32_t bv[4];
          const int mi = lane >> 3;
          ldmatrix_x4_trans(bv, Vt + (kk * 16 + (mi & 1) * 8 + (lane & 7)) * kRow + dbase + i * 8 + (mi >> 1) * 8);
          mma_bf16(o[i], ah, bv[0], bv[1]);
          mma_bf16(o[i], al, bv[0], bv[1]);
          mma_bf16(o[i + 1], ah, bv[2], bv[3]);
          mma_bf16(o[i + 1], al, bv[2], bv[3]);
        }
      }
    }
    __syncthreads();
  }
  // partials: O (unnormalised), max and sum of every query row
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = rr ? r1 : r0;
    if (!active || r >= nq) continue;
    const int qv = qv0 + r, j = qv / G, gg = qv % G;
    float* dst = a.part + ((((int64_t)b * T + j) * a.Hq + h * G + gg) * a.nchunk + chunk) * kPart;
#pragma unroll
    for (int i = 0; i < NT; ++i)
      *reinterpret_cast<float2*>(dst + dbase + i * 8 + 2 * tq) = make_float2(o[i][2 * rr], o[i][2 * rr + 1]);
    if (warp % WPM == 0 && tq == 0) {
      dst[CAS_BLK] = rr ? m1 : m0;
      dst[CAS_BLK + 1] = rr ? l1 : l0;
    }
  }
}

// ---------------------------------------------------------------- fused draft
// Draft attention with at most 4 query vectors per kv head (T = 1, GQA up to
// 4:1). The K side needs no tile: lane L decodes its 16 kept K values of
// token L/4 (per-lane cursors, as for the tiles) and multiplies each with the
// 4 query vectors at its position (q4: dims x 4, pre-scaled, one 16-byte load
// per value); the 4 lanes of a token add their partial scores.

template <bool LONG>
__device__ __forceinline__ float4 lane_kept_qdot(UnaryCursor& uc, uint4 kq, uint2 rs, const uint8_t* __restrict__ lut,
                                                 const float4* q4) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int pos = pos_byte(kq, i);
    const uint32_t e = lut[uc.next<LONG>() & 255];
    const uint32_t f = (i < 8 ? rs.x : rs.y) >> (4 * (i & 7));
    const float val = __uint_as_float(((f & 8u) << 28) | (e << 23) | ((f & 7u) << 20));
    const float4 q = q4[pos];
    acc.x = fmaf(val, q.x, acc.x);
    acc.y = fmaf(val, q.y, acc.y);
    acc.z = fmaf(val, q.z, acc.z);
    acc.w = fmaf(val, q.w, acc.w);
  }
  return acc;
}


// Scores of the 8 tokens of superblock sb of K stream st against the 4 query
// vectors into out[8][4] (float4 per token). Only for whole Cassandra-1
// superblocks with k = 64, m = 3 and a stream that fits the stage; returns
// false otherwise (nothing written, warp-uniform).
__device__ __forceinline__ bool lane_sb_scores(const KvDev& d, int st, int64_t n, int64_t sb, const uint8_t* lut,
                                               uint8_t* scratch, const float4* q4, float4* out, int lane) {
  const int64_t nsb = (n + CAS_SB - 1) / CAS_SB;
  if (!(sb < nsb && d.variant == 1 && d.k == 64 && d.m == 3 && CAS_SB * (sb + 1) <= n)) return false;
  const uint32_t* sidx = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, st);
  const uint32_t a0 = sidx[sb], a1 = sidx[sb + 1];
  const int snw = (int)(a1 - a0);
  if (snw > kStageWords) return false;
  TileStage& ts = *reinterpret_cast<TileStage*>(scratch);
  const uint32_t mw = __ldg((const uint32_t*)kv_sec(d, CAS_KV_MASK, st) + sb * 32 + lane);
  const uint2 rs = __ldg(reinterpret_cast<const uint2*>((const uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, st) + sb * 64) + lane);
  bool long_codes;
  const bool enough =
      stage_unary((const uint32_t*)kv_sec(d, CAS_KV_SPEC_EXP, st) + a0, snw, ts.us, lane, &long_codes) >= 16 * 32;
  expand_mask_positions(mw, ts.kpos, lane);
  __syncwarp();
  if (!enough) return false;
  UnaryCursor uc;
  uc.init(ts.us, unary_code_start(ts.us, snw, 16 * lane));
  const uint4 kq = reinterpret_cast<const uint4*>(ts.kpos)[lane];
  float4 acc = long_codes ? lane_kept_qdot<true>(uc, kq, rs, lut, q4) : lane_kept_qdot<false>(uc, kq, rs, lut, q4);
#pragma unroll
  for (int x = 1; x <= 2; x <<= 1) {
    acc.x += __shfl_xor_sync(CAS_FULL, acc.x, x);
    acc.y += __shfl_xor_sync(CAS_FULL, acc.y, x);
    acc.z += __shfl_xor_sync(CAS_FULL, acc.z, x);
    acc.w += __shfl_xor_sync(CAS_FULL, acc.w, x);
  }
  if ((lane & 3) == 0) out[lane >> 2] = acc;
  __syncwarp();
  return true;
}

// Any k, m, both variants, one whole superblock: lane L takes the kept
// ordinals [ceil(k q / 4), ceil(k (q+1) / 4)) of block b = L / 4 (q = L % 4), so
// the 4 lanes of a token still add their partial scores; record fields are
// read at run-time offsets, exponents from the unary cursor (Cassandra-1) or
// the group's shared exponent (Cassandra-2). Scratch: TileStage (C-1) or
// TileStage2 (C-2); same contract as lane_sb_scores.
template <int VAR, bool LONG>
__device__ __forceinline__ float4 quarter_qdot(UnaryCursor& uc, const uint8_t* pos, const uint32_t* rec, const uint8_t* mx,
                                               int m, int b, int o0, int o1, int k, const uint8_t* __restrict__ lut,
                                               const float4* q4) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int width = VAR == 1 ? m + 1 : m + 2;
  for (int o = o0; o < o1; ++o) {
    const int p = pos[b * k + o];
    const uint32_t fld = field_g(rec, o * width, width);
    float val;
    if (VAR == 1) {
      const uint32_t e = lut[uc.next<LONG>() & 255];
      val = __uint_as_float(((fld >> m) << 31) | (e << 23) | ((fld & ((1u << m) - 1u)) << (23 - m)));
    } else {
      const float qv = (float)(fld & ((1u << (m + 1)) - 1u)) * pow2_biased(max((int)mx[b * 4 + (p >> 5)], 1) - m);
      val = (fld >> (m + 1)) ? -qv : qv;
    }
    const float4 q = q4[p];
    acc.x = fmaf(val, q.x, acc.x);
    acc.y = fmaf(val, q.y, acc.y);
    acc.z = fmaf(val, q.z, acc.z);
    acc.w = fmaf(val, q.w, acc.w);
  }
  return acc;
}

__device__ __forceinline__ bool quarter_sb_scores(const KvDev& d, int st, int64_t n, int64_t sb, const uint8_t* lut,
                                                  uint8_t* scratch, const float4* q4, float4* out, int lane) {
  const int64_t nsb = (n + CAS_SB - 1) / CAS_SB;
  if (!(sb < nsb && CAS_SB * (sb + 1) <= n)) return false;
  const int k = d.k, m = d.m, b = lane >> 2, q = lane & 3;
  const int o0 = (k * q + 3) >> 2, o1 = (k * (q + 1) + 3) >> 2;
  const uint32_t mw = __ldg((const uint32_t*)kv_sec(d, CAS_KV_MASK, st) + sb * 32 + lane);
  float4 acc;
  if (d.variant == 1) {
    const uint32_t* sidx = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, st);
    const uint32_t a0 = sidx[sb], a1 = sidx[sb + 1];
    const int snw = (int)(a1 - a0);
    if (snw > kStageWords) return false;
    TileStage& ts = *reinterpret_cast<TileStage*>(scratch);
    bool long_codes;
    const bool enough =
        stage_unary((const uint32_t*)kv_sec(d, CAS_KV_SPEC_EXP, st) + a0, snw, ts.us, lane, &long_codes) >= CAS_SB * k;
    expand_mask_positions<CAS_SB * CAS_BLK>(mw, ts.kpos, lane);
    __syncwarp();
    if (!enough) return false;
    UnaryCursor uc;
    uc.init(ts.us, unary_code_start(ts.us, snw, b * k + o0));
    const uint32_t* rec = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, st) + (sb * CAS_SB + b) * d.rec_sm;
    acc = long_codes ? quarter_qdot<1, true>(uc, ts.kpos, rec, nullptr, m, b, o0, o1, k, lut, q4)
                     : quarter_qdot<1, false>(uc, ts.kpos, rec, nullptr, m, b, o0, o1, k, lut, q4);
  } else {
    TileStage2& ts = *reinterpret_cast<TileStage2*>(scratch);
    ts.mx[lane] = __ldg(kv_sec(d, CAS_KV_SPEC_MX, st) + sb * 32 + lane);
    expand_mask_positions<CAS_SB * CAS_BLK>(mw, ts.pos, lane);
    __syncwarp();
    UnaryCursor uc;  // unused for Cassandra-2
    const uint32_t* rec = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_Q, st) + (sb * CAS_SB + b) * d.rec_q;
    acc = quarter_qdot<2, false>(uc, ts.pos, rec, ts.mx, m, b, o0, o1, k, lut, q4);
  }
#pragma unroll
  for (int x = 1; x <= 2; x <<= 1) {
    acc.x += __shfl_xor_sync(CAS_FULL, acc.x, x);
    acc.y += __shfl_xor_sync(CAS_FULL, acc.y, x);
    acc.z += __shfl_xor_sync(CAS_FULL, acc.z, x);
    acc.w += __shfl_xor_sync(CAS_FULL, acc.w, x);
  }
  if (q == 0) out[b] = acc;
  __syncwarp();
  return true;
}

// Per 32-token step warp w scores its K superblock (tokens 8w..8w+7 of the
// step) into sc, decodes its V superblock into the V tile, and after the
// barrier runs query vector w over the 32 tokens (online softmax, P.V with
// lane = 4 dims) exactly as the chunk kernel. Superblocks the cursors do not
// cover (partial, Cassandra-2, other k or m, long streams) are decoded into a
// K tile and scored from it.
__global__ void __launch_bounds__(kThreads, 8) attn_draft_fused_kernel(AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Kt = reinterpret_cast<uint16_t*>(smem);  // fallback K tile
  uint16_t* Vt = Kt + kStepTok * kRow;
  float4* q4 = reinterpret_cast<float4*>(Vt + kStepTok * kRow);  // [128] dims x 4 query vectors
  float4* sc = q4 + CAS_BLK;                                      // [32] tokens x 4 query vectors
  uint8_t* lutK = reinterpret_cast<uint8_t*>(sc + kStepTok);
  uint8_t* lutV = lutK + 256;
  uint8_t* scr = lutV + 256;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t* wscr = scr + warp * a.scr_warp;
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const KvDev& d = a.kv[b];
  const int H = d.H, G = a.G, nq = min(a.T * G, 4);
  const int64_t n = *(volatile const int64_t*)&kv_state(d)->n_tokens;
  const int64_t steps = (n + kStepTok - 1) / kStepTok;
  const int64_t t_begin = steps * chunk / a.nchunk * kStepTok;
  const int64_t t_end = min(n, steps * (chunk + 1) / a.nchunk * kStepTok);

  // q4[dd] = the 4 query vectors (q heads h*G .. h*G+3 of token 0) at dimension dd, scaled
  for (int i = threadIdx.x; i < 4 * CAS_BLK; i += kThreads) {
    const int r = i & 3, dd = i >> 2;
    float v = 0.f;
    if (r < nq) v = bf2f(a.q[((int64_t)b * a.Hq + h * G + r) * CAS_BLK + dd]) * a.scale;
    reinterpret_cast<float*>(q4)[i] = v;
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) {
    lutK[i] = kv_exp_of_rank(d, h)[i];
    lutV[i] = kv_exp_of_rank(d, H + h)[i];
  }
  __syncthreads();

  const int qv = warp;  // query vector run by this warp (if < nq)
  float m = -INFINITY, l = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
  for (int64_t t0 = t_begin; t0 < t_end; t0 += kStepTok) {
    const int64_t sb = t0 / CAS_SB + warp;
    const bool scored = (d.variant == 1 && d.k == 64 && d.m == 3)
                            ? lane_sb_scores(d, h, n, sb, lutK, wscr, q4, sc + warp * CAS_SB, lane)
                            : quarter_sb_scores(d, h, n, sb, lutK, wscr, q4, sc + warp * CAS_SB, lane);
    if (!scored) {
      decode_sb_tile<false>(d, h, n, sb, Kt, warp * CAS_SB, lutK, wscr, lane);
      // lane = (token lane / 4 of this superblock, query vector lane % 4)
      const uint32_t* kr = reinterpret_cast<const uint32_t*>(Kt + (warp * CAS_SB + (lane >> 2)) * kRow);
      const float* qf = reinterpret_cast<const float*>(q4) + (lane & 3);
      float acc = 0.f;
      for (int dd = 0; dd < CAS_BLK; dd += 2) {
        const uint32_t k2 = kr[dd >> 1];
        acc = fmaf(bf2f(k2 & 0xFFFFu), qf[4 * dd], acc);
        acc = fmaf(bf2f(k2 >> 16), qf[4 * dd + 4], acc);
      }
      reinterpret_cast<float*>(sc + warp * CAS_SB + (lane >> 2))[lane & 3] = acc;
      __syncwarp();
    }
    decode_sb_tile<false>(d, H + h, n, sb, Vt, warp * CAS_SB, lutV, wscr, lane);
    __syncthreads();
    if (qv < nq) {
      const int64_t tok = t0 + lane;
      const float si = tok < t_end ? reinterpret_cast<const float*>(sc + lane)[qv] : -INFINITY;
      const float mx = warp_maxf(si);
      const float mnew = fmaxf(m, mx);
      const float p = (si == -INFINITY) ? 0.f : __expf(si - mnew);
      float corr = (m == -INFINITY) ? 0.f : __expf(m - mnew);
      if (mnew == -INFINITY) corr = 1.f;
      l = l * corr + warp_sumf(p);
      m = mnew;
      float acc0 = o0 * corr, acc1 = o1 * corr, acc2 = o2 * corr, acc3 = o3 * corr;
      for (int t = 0; t < kStepTok; ++t) {
        const float pt = __shfl_sync(CAS_FULL, p, t);
        const uint2 v4 = reinterpret_cast<const uint2*>(Vt + t * kRow)[lane];
        acc0 = fmaf(pt, __uint_as_float(v4.x << 16), acc0);
        acc1 = fmaf(pt, __uint_as_float(v4.x & 0xFFFF0000u), acc1);
        acc2 = fmaf(pt, __uint_as_float(v4.y << 16), acc2);
        acc3 = fmaf(pt, __uint_as_float(v4.y & 0xFFFF0000u), acc3);
      }
      o0 = acc0;
      o1 = acc1;
      o2 = acc2;
      o3 = acc3;
    }
    __syncthreads();
  }
  if (qv < nq) {
    float* dst = a.part + (((int64_t)b * a.Hq + h * G + qv) * a.nchunk + chunk) * kPart;
    reinterpret_cast<float2*>(dst)[2 * lane] = make_float2(o0, o1);
    reinterpret_cast<float2*>(dst)[2 * lane + 1] = make_float2(o2, o3);
    if (lane == 0) {
      dst[CAS_BLK] = m;
      dst[CAS_BLK + 1] = l;
    }
  }
}

constexpr int kCombineWarps = 32;  // warps of a combine CTA (each merges every 32nd chunk)

struct CombineArgs {
  const float* part;
  const uint16_t* q;       // [B][T][Hq][128]
  const uint16_t* tail_k;  // [B][n_tail][Hkv][128] or null
  const uint16_t* tail_v;
  float* o;                // [B][T][Hq][128]
  const int64_t* ntok[kMaxBatch];
  int T, Hq, Hkv, G, nchunk, n_tail;
  float scale;
};

// One CTA of 32 warps per (sequence, query token, q head). Warp w merges
// chunks w, w+32, ... with lane L holding dims 4L..4L+3 (online max / sum);
// the warp results and the bf16 tail tokens are merged in shared memory.
__global__ void __launch_bounds__(kCombineWarps * 32) attn_combine_kernel(CombineArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float wm[kCombineWarps], wl[kCombineWarps];
  __shared__ float4 wo[kCombineWarps][32];
  __shared__ float ts[kMaxT];
  const int hq = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n = *(volatile const int64_t*)a.ntok[b];
  const int used = n > 0 ? a.nchunk : 0;
  const float* P = a.part + (((int64_t)b * a.T + j) * a.Hq + hq) * a.nchunk * kPart;
  const int hk = hq / a.G;
  // tail scores (exact bf16 tokens), warp 0
  if (warp == 0) {
    const uint16_t* qp = a.q + (((int64_t)b * a.T + j) * a.Hq + hq) * CAS_BLK + 4 * lane;
    for (int t = 0; t < a.n_tail; ++t) {
      const uint16_t* kp = a.tail_k + (((int64_t)b * a.n_tail + t) * a.Hkv + hk) * CAS_BLK + 4 * lane;
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) s = fmaf(bf2f(qp[i]), bf2f(kp[i]), s);
      s = warp_sumf(s) * a.scale;
      if (lane == 0) ts[t] = s;
    }
  }
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  // four chunks per warp and pass, their loads issued before any is used
  constexpr int kU = 4;
  for (int c0 = warp; c0 < used; c0 += kU * kCombineWarps) {
    float mc[kU], lc[kU];
    float4 oc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = c0 + u * kCombineWarps;
      mc[u] = -INFINITY;
      lc[u] = 0.f;
      oc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < used) {
        mc[u] = P[c * kPart + CAS_BLK];
        lc[u] = P[c * kPart + CAS_BLK + 1];
        // partials sit at a 130-float (520-byte) stride: 8-byte aligned, so two float2 loads
        const float2 oa = reinterpret_cast<const float2*>(P + c * kPart)[2 * lane];
        const float2 ob = reinterpret_cast<const float2*>(P + c * kPart)[2 * lane + 1];
        oc[u] = make_float4(oa.x, oa.y, ob.x, ob.y);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (mc[u] == -INFINITY) continue;
      const float mn = fmaxf(M, mc[u]);
      const float fa = M == -INFINITY ? 0.f : __expf(M - mn), fb = __expf(mc[u] - mn);
      L = L * fa + lc[u] * fb;
      O = make_float4(O.x * fa + oc[u].x * fb, O.y * fa + oc[u].y * fb, O.z * fa + oc[u].z * fb,
                      O.w * fa + oc[u].w * fb);
      M = mn;
    }
  }
  if (lane == 0) {
    wm[warp] = M;
    wl[warp] = L;
  }
  wo[warp][lane] = O;
  __syncthreads();
  if (warp == 0) {
    float Mt = -INFINITY;
    for (int w = 0; w < kCombineWarps; ++w) Mt = fmaxf(Mt, wm[w]);
    for (int t = 0; t < a.n_tail; ++t) Mt = fmaxf(Mt, ts[t]);
    float Lt = 0.f;
    float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < kCombineWarps; ++w) {
      if (wm[w] == -INFINITY) continue;
      const float f = __expf(wm[w] - Mt);
      Lt += wl[w] * f;
      const float4 o = wo[w][lane];
      Ot = make_float4(Ot.x + o.x * f, Ot.y + o.y * f, Ot.z + o.z * f, Ot.w + o.w * f);
    }
    for (int t = 0; t < a.n_tail; ++t) {
      const float f = __expf(ts[t] - Mt);
      Lt += f;
      const uint16_t* vp = a.tail_v + (((int64_t)b * a.n_tail + t) * a.Hkv + hk) * CAS_BLK + 4 * lane;
      Ot = make_float4(Ot.x + f * bf2f(vp[0]), Ot.y + f * bf2f(vp[1]), Ot.z + f * bf2f(vp[2]), Ot.w + f * bf2f(vp[3]));
    }
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    reinterpret_cast<float4*>(a.o + (((int64_t)b * a.T + j) * a.Hq + hq) * CAS_BLK)[lane] =
        make_float4(Ot.x * inv, Ot.y * inv, Ot.z * inv, Ot.w * inv);
  }
}

size_t chunk_smem(int qv_alloc, int scr_warp) {
  return (size_t)2 * kStepTok * kRow * 2 + (size_t)qv_alloc * CAS_BLK * 4 + 512 + (size_t)kWarps * scr_warp;
}

int nchunks(int64_t max_tokens) { return (int)((max_tokens + kChunk - 1) / kChunk); }

size_t mma_smem(int mt, int scr_warp) {
  return (size_t)2 * kStepTok * kRow * 2 + kTileSlack + (size_t)16 * mt * kRow * 2 + 512 + 2048 +
         (size_t)kWarps * scr_warp;
}

// Sets a.nchunk to one wave of resident CTAs (at most the workspace's count).
int one_wave(AttnArgs& a, int Hkv, const void* kern, size_t smem) {
  const int per_sm = occupancy(kern, kThreads, smem);
  if (per_sm < 1) return CAS_ERR_CUDA;
  const int64_t slots = (int64_t)per_sm * sm_count();
  a.nchunk = (int)std::max<int64_t>(1, std::min<int64_t>(a.nchunk, slots / ((int64_t)Hkv * a.B * a.ngroups)));
  return CAS_OK;
}

int launch_fused(AttnArgs& a, int Hkv, cudaStream_t st) {
  if (a.scr_warp == kScratchC1) a.scr_warp = kScratchDraftC1;  // every cache is Cassandra-1
  const size_t smem = (size_t)2 * kStepTok * kRow * 2 + (size_t)CAS_BLK * 16 + (size_t)kStepTok * 16 + 512 +
                      (size_t)kWarps * a.scr_warp;
  const int s = one_wave(a, Hkv, (const void*)attn_draft_fused_kernel, smem);
  if (s) return s;
  return launch_k(attn_draft_fused_kernel, dim3(a.nchunk, Hkv, a.B), kThreads, smem, st, a);
}


// ---------------------------------------------------------------- block draft
// Draft attention for Cassandra-1 caches with k = 64, m = 3 and at most 4
// query vectors per kv head (blockwalk.cuh). A warp takes 32 tokens at a time
// (4 superblocks of a stream) with lane = token: it walks the token's 64 kept
// K values and multiplies each with the 4 query vectors at its position (one
// 16-byte load of a dims x 4 query table), runs the online softmax per query
// vector over its 32 scores, walks the 64 kept V values of the same tokens
// into a zero-filled bf16 tile, and adds P V on tensor cores as O^T += V^T P^T
// (mma m16n8k16: A = the tile, transposed by ldmatrix; B = P in bf16 as hi +
// lo, |p - hi - lo| <= 2^-17 p; C = 128 dims x 8 query columns, 4 used). Each
// warp keeps its own softmax state over every 4th step of the CTA's chunk;
// the 4 warps merge at the end. A lane whose windows ran dry rescans its
// token (K) or makes the whole warp rebuild its V rows by scanning (its
// stores may have run into the next rows); superblocks whose streams do not
// fit the stage are decoded by decode_sb_tile and scored from the tile.
constexpr int kDRow = CAS_BLK + 8;     // V tile row (272 B)
constexpr int kDPRow = 40;             // P^T stage row: 32 tokens + pad (conflict-free ldmatrix)
constexpr int kDWarpPad = 512;         // bytes after a warp's V tile: stores of a failed walk stay inside
struct DraftStage {
  union {
    struct {
      BlockStreams<2> st;  // codes of the step's 4 superblocks (K, then V)
      uint32_t ms[7][32];  // row i, column l: bit-reversed mask word i of token l; rows 4-6 zero
    } w;
    uint8_t tile_scratch[kScratchDraftC1];  // decode_sb_tile's stage
  } u;
  uint16_t ph[8][kDPRow], pl[8][kDPRow];  // P^T hi / lo: query vector x token (rows 4-7 zero)
  uint16_t vt[kStepTok * kDRow + kDWarpPad / 2];  // V tile: token x dim (+ slack)
};
static_assert(sizeof(DraftStage) % 16 == 0, "draft stage alignment");

// The K walk of one token without windows (any gap, any code length): the
// scores against the 4 query vectors, or ok = false when the staged data runs
// out (the encoding is inconsistent).
__device__ __noinline__ float4 draft_k_scan(uint32_t ms_a, uint32_t st_a, int q0, uint32_t lutk_a,
                                            const uint32_t* __restrict__ rec, uint32_t q4_a, bool& ok) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int cur = -1, q = q0;
  ok = false;
  for (int i = 0; i < 64; ++i) {
    const int p = bnext_one(ms_a, 128u, cur + 1, 6);
    const int e = bnext_one(st_a, 4u, q + 1, BlockStreams<2>::kRow - 1);
    if (p < 0 || p >= CAS_BLK || e < 0) return acc;
    cur = p;
    const uint32_t E = lds_u32(lutk_a + 4u * (uint32_t)min(e - q - 1, 255));
    q = e;
    const uint32_t f = (__ldg(rec + (i >> 3)) >> (4 * (i & 7))) & 15u;
    const float v = __uint_as_float(((f & 8u) << 28) | E | ((f & 7u) << 20));
    const float4 qq = *reinterpret_cast<const float4*>(__cvta_shared_to_generic(q4_a + 16u * (uint32_t)p));
    acc.x = fmaf(v, qq.x, acc.x);
    acc.y = fmaf(v, qq.y, acc.y);
    acc.z = fmaf(v, qq.z, acc.z);
    acc.w = fmaf(v, qq.w, acc.w);
  }
  ok = true;
  return acc;
}

// The V walk of one token without windows into its tile row; false when the
// staged data runs out.
__device__ __noinline__ bool draft_v_scan(uint32_t ms_a, uint32_t st_a, int q0, uint32_t lutv_a,
                                          const uint32_t* __restrict__ rec, uint32_t row_a) {
  int cur = -1, q = q0;
  for (int i = 0; i < 64; ++i) {
    const int p = bnext_one(ms_a, 128u, cur + 1, 6);
    const int e = bnext_one(st_a, 4u, q + 1, BlockStreams<2>::kRow - 1);
    if (p < 0 || p >= CAS_BLK || e < 0) return false;
    cur = p;
    const uint32_t E = lds_u32(lutv_a + 4u * (uint32_t)min(e - q - 1, 255));
    q = e;
    const uint32_t f = (__ldg(rec + (i >> 3)) >> (4 * (i & 7))) & 15u;
    sts_u16(row_a + 2u * (uint32_t)p, ((f & 8u) << 12) | E | ((f & 7u) << 4));
  }
  return true;
}

__global__ void __launch_bounds__(kThreads, 4) attn_draft_block_kernel(AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  float4* q4 = reinterpret_cast<float4*>(smem);  // [128] dims x 4 query vectors, scaled
  uint32_t* lutk = reinterpret_cast<uint32_t*>(q4 + CAS_BLK);  // exponent << 23 by rank (K)
  uint32_t* lutv = lutk + 256;                                  // exponent << 7 by rank (V)
  uint8_t* lut8k = reinterpret_cast<uint8_t*>(lutv + 256);      // exponent by rank (generic decoder)
  uint8_t* lut8v = lut8k + 256;
  DraftStage* stages = reinterpret_cast<DraftStage*>(lut8v + 256);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  DraftStage& ds = stages[warp];
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const KvDev& d = a.kv[b];
  const int H = d.H, G = a.G, nq = min(a.T * G, 4);
  const int64_t n = *(volatile const int64_t*)&kv_state(d)->n_tokens;
  const int64_t nsb = (n + CAS_SB - 1) / CAS_SB;
  const int64_t steps = (n + kStepTok - 1) / kStepTok;
  const int64_t s_begin = steps * chunk / a.nchunk, s_end = steps * (chunk + 1) / a.nchunk;

  for (int i = threadIdx.x; i < 4 * CAS_BLK; i += kThreads) {
    const int r = i & 3, dd = i >> 2;
    float v = 0.f;
    if (r < nq) v = bf2f(a.q[((int64_t)b * a.Hq + h * G + r) * CAS_BLK + dd]) * a.scale;
    reinterpret_cast<float*>(q4)[i] = v;
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) {
    const uint8_t ek = kv_exp_of_rank(d, h)[i], ev = kv_exp_of_rank(d, H + h)[i];
    lutk[i] = (uint32_t)ek << 23;
    lutv[i] = (uint32_t)ev << 7;
    lut8k[i] = ek;
    lut8v[i] = ev;
  }
  block_streams_init(ds.u.w.st, lane);
#pragma unroll
  for (int r = 4; r < 7; ++r) ds.u.w.ms[r][lane] = 0u;
  for (int i = lane; i < 8 * kDPRow; i += 32) {
    (&ds.ph[0][0])[i] = 0;
    (&ds.pl[0][0])[i] = 0;
  }
  __syncthreads();

  const uint32_t q4_a = smem_addr(q4), lutk_a = smem_addr(lutk), lutv_a = smem_addr(lutv);
  const uint32_t ms_a0 = smem_addr(&ds.u.w.ms[0][lane]), st_a0 = smem_addr(&ds.u.w.st.w[lane >> 3][0]);
  const uint32_t vt_a = smem_addr(ds.vt), row_a = vt_a + 2u * (uint32_t)(lane * kDRow);
  const uint32_t* sidxK = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, h);
  const uint32_t* sidxV = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, H + h);
  const uint32_t lim = (uint32_t)d.cap_a;
  const int gq = lane >> 2, tq = lane & 3;
  float mst[4], lst[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    mst[q] = -INFINITY;
    lst[q] = 0.f;
  }
  float c[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) c[mt][0] = c[mt][1] = c[mt][2] = c[mt][3] = 0.f;

  for (int64_t s = s_begin + warp; s < s_end; s += kWarps) {
    const int64_t t0 = s * kStepTok, tok = t0 + lane, sb0 = t0 / CAS_SB;
    const bool valid = tok < n;
    const int64_t tk = valid ? tok : t0;
    // superblocks of the step with all 8 tokens (their streams hold 512 codes)
    int whole = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) whole += CAS_SB * (sb0 + u + 1) <= n ? 1 : 0;
    float sc[4];
    // ---- K: scores of token tok against the query vectors
    {
      const uint32_t* g4[4];
      int nw[4];
      bool fast = true;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t a0 = 0u, b0 = 0u;
        if (sb0 + u < nsb) stream_range(sidxK, sb0 + u, lim, a0, b0);
        g4[u] = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_EXP, h) + a0;
        nw[u] = (int)(b0 - a0);
        fast = fast && nw[u] <= 64;
      }
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (fast) {
        const uint4 mk = __ldg(reinterpret_cast<const uint4*>(kv_sec(d, CAS_KV_MASK, h)) + tk);
        const uint32_t* rec = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, h) + tk * 8;
        ds.u.w.ms[0][lane] = valid ? __brev(mk.x) : 0u;
        ds.u.w.ms[1][lane] = valid ? __brev(mk.y) : 0u;
        ds.u.w.ms[2][lane] = valid ? __brev(mk.z) : 0u;
        ds.u.w.ms[3][lane] = valid ? __brev(mk.w) : 0u;
        uint32_t fn = __ldg(rec);  // the next group's record word
        const int q0 = block_code_term<2, 64>(g4, nw, whole, ds.u.w.st, lane, fast);
        const uint32_t ms_a = fenced(ms_a0), st_a = fenced(st_a0);
        uint32_t xa = q4_a - 16u;  // query table address of the last found position (-1 at first)
        uint32_t Hp, Lp, Hc, Lc;
        bwindow(ms_a, 128u, 0, 4, Hp, Lp);
        bwindow(st_a, 4u, q0 + 1, BlockStreams<2>::kRow - 3, Hc, Lc);
        uint32_t used = 0u, cor = 0u;
        bool pstale = false;  // the position window lags the cursor (after a scanned group)
#pragma unroll 1
        for (int gi = 0; gi < 8; ++gi) {
          const uint32_t fo = fn, fe = fn << 4;
          if (gi < 7) fn = __ldg(rec + gi + 1);
          if (gi > 0) {
            // the position window every 16 values (a window that runs dry
            // is caught like a long gap), the code window every 8
            if ((gi & 1) == 0 || pstale) {
              const int cur = min((int)(xa - q4_a) >> 4, CAS_BLK - 1);
              xa = q4_a + 16u * (uint32_t)cur;
              bwindow(ms_a, 128u, cur + 1, 4, Hp, Lp);
            }
            bwindow(st_a, 4u, q0 + 1 + (int)used, BlockStreams<2>::kRow - 3, Hc, Lc);
          }
          pstale = false;
          // a group whose 8 codes do not all end in the window (a code longer
          // than the window: an exponent the tables rank far down) is taken by
          // scanning; the walk goes on after it
          if (__popc(Hc) + __popc(Lc) < 8) {
            int cur = (int)(xa - q4_a) >> 4, qt = q0 + (int)used;
            for (int i = 0; i < 8; ++i) {
              const int pb = bnext_one(ms_a, 128u, cur + 1, 6);
              const int eb = bnext_one(st_a, 4u, qt + 1, BlockStreams<2>::kRow - 1);
              if (pb < 0 || pb >= CAS_BLK || eb < 0) {
                cor |= 32u;
                break;
              }
              const uint32_t E = lds_u32(lutk_a + 4u * (uint32_t)min(eb - qt - 1, 255));
              used += (uint32_t)(eb - qt);
              qt = eb;
              cur = pb;
              const uint32_t f = (fo >> (4 * i)) & 15u;
              const float v = __uint_as_float(((f & 8u) << 28) | E | ((f & 7u) << 20));
              float4 qq;
              asm("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                  : "=f"(qq.x), "=f"(qq.y), "=f"(qq.z), "=f"(qq.w)
                  : "r"(q4_a + 16u * (uint32_t)cur));
              acc.x = fmaf(v, qq.x, acc.x);
              acc.y = fmaf(v, qq.y, acc.y);
              acc.z = fmaf(v, qq.z, acc.z);
              acc.w = fmaf(v, qq.w, acc.w);
            }
            xa = q4_a + 16u * (uint32_t)max(cur, -1);
            pstale = true;
            continue;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t np = __clz(Hp) + 1u;
            xa = mad32(np, 16u, xa);
            Hp = shfl_wrap(Lp, Hp, np);
            Lp = shfl_wrap(0u, Lp, np);
            const uint32_t nc = __clz(Hc) + 1u;
            const uint32_t E = lds_u32(lutk_a - 4u + 4u * nc);
            Hc = shfl_wrap(Lc, Hc, nc);
            Lc = shfl_wrap(0u, Lc, nc);
            used += nc;
            cor |= np | nc;
            const int by = i >> 1;
            const uint32_t A = __byte_perm((i & 1) ? fo : fe, 0u, (by << 12) | (by << 8) | 0x44);
            const float v = __uint_as_float((A & 0x80700000u) | E);
            float4 qq;
            asm("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(qq.x), "=f"(qq.y), "=f"(qq.z), "=f"(qq.w) : "r"(xa));
            acc.x = fmaf(v, qq.x, acc.x);
            acc.y = fmaf(v, qq.y, acc.y);
            acc.z = fmaf(v, qq.z, acc.z);
            acc.w = fmaf(v, qq.w, acc.w);
          }
        }
        if (valid && (cor & 32u)) {  // rescan this token (divergent, rare)
          bool ok;
          acc = draft_k_scan(ms_a, st_a, q0, lutk_a, rec, q4_a, ok);
          if (!ok) acc = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncwarp();
      }
      if (!fast) {  // a stream longer than the stage: K tile, then scores from it
        for (int u = 0; u < 4; ++u)
          decode_sb_tile<false>(d, h, n, sb0 + u, ds.vt, CAS_SB * u, lut8k, ds.u.tile_scratch, lane);
        const uint32_t* kr = reinterpret_cast<const uint32_t*>(ds.vt + lane * kDRow);
        for (int dd = 0; dd < CAS_BLK; dd += 2) {
          const uint32_t k2 = kr[dd >> 1];
          const float4 qa = q4[dd], qb = q4[dd + 1];
          const float k0 = bf2f(k2 & 0xFFFFu), k1 = bf2f(k2 >> 16);
          acc.x = fmaf(k0, qa.x, fmaf(k1, qb.x, acc.x));
          acc.y = fmaf(k0, qa.y, fmaf(k1, qb.y, acc.y));
          acc.z = fmaf(k0, qa.z, fmaf(k1, qb.z, acc.z));
          acc.w = fmaf(k0, qa.w, fmaf(k1, qb.w, acc.w));
        }
        block_streams_init(ds.u.w.st, lane);
#pragma unroll
        for (int r = 4; r < 7; ++r) ds.u.w.ms[r][lane] = 0u;
        __syncwarp();
      }
      sc[0] = valid ? acc.x : -INFINITY;
      sc[1] = valid ? acc.y : -INFINITY;
      sc[2] = valid ? acc.z : -INFINITY;
      sc[3] = valid ? acc.w : -INFINITY;
    }
    // ---- online softmax per query vector; P^T (hi, lo) to the stage
    float corr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float mnew = fmaxf(mst[q], warp_maxf(sc[q]));
      const float p = sc[q] == -INFINITY ? 0.f : __expf(sc[q] - mnew);
      corr[q] = mst[q] == -INFINITY ? (mnew == -INFINITY ? 1.f : 0.f) : __expf(mst[q] - mnew);
      lst[q] = lst[q] * corr[q] + warp_sumf(p);
      mst[q] = mnew;
      const uint32_t hi = pack_bf16x2(p, 0.f) & 0xFFFFu;
      const float lo = p - __uint_as_float(hi << 16);
      ds.ph[q][lane] = (uint16_t)hi;
      ds.pl[q][lane] = (uint16_t)(pack_bf16x2(lo, 0.f) & 0xFFFFu);
    }
    // ---- V: draft values of the 32 tokens into the tile
    {
      const uint32_t* g4[4];
      int nw[4];
      bool fast = true;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t a0 = 0u, b0 = 0u;
        if (sb0 + u < nsb) stream_range(sidxV, sb0 + u, lim, a0, b0);
        g4[u] = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_EXP, H + h) + a0;
        nw[u] = (int)(b0 - a0);
        fast = fast && nw[u] <= 64;
      }
      if (fast) {
        const uint4 mk = __ldg(reinterpret_cast<const uint4*>(kv_sec(d, CAS_KV_MASK, H + h)) + tk);
        const uint32_t* rec = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, H + h) + tk * 8;
        uint32_t fn = __ldg(rec);  // the next group's record word
        // zero the token's row (pruned dims, tokens past the cache)
        uint4* zr = reinterpret_cast<uint4*>(ds.vt + lane * kDRow);
#pragma unroll
        for (int i = 0; i < CAS_BLK / 8; ++i) zr[i] = make_uint4(0u, 0u, 0u, 0u);
        ds.u.w.ms[0][lane] = valid ? __brev(mk.x) : 0u;
        ds.u.w.ms[1][lane] = valid ? __brev(mk.y) : 0u;
        ds.u.w.ms[2][lane] = valid ? __brev(mk.z) : 0u;
        ds.u.w.ms[3][lane] = valid ? __brev(mk.w) : 0u;
        const int q0 = block_code_term<2, 64>(g4, nw, whole, ds.u.w.st, lane, fast);
        const uint32_t ms_a = fenced(ms_a0), st_a = fenced(st_a0);
        uint32_t ta = row_a - 2u;
        uint32_t Hp, Lp, Hc, Lc;
        bwindow(ms_a, 128u, 0, 4, Hp, Lp);
        bwindow(st_a, 4u, q0 + 1, BlockStreams<2>::kRow - 3, Hc, Lc);
        uint32_t used = 0u, cor = 0u;
        if (valid) {
#pragma unroll 1
          for (int gi = 0; gi < 8; ++gi) {
            const uint32_t fo = fn, fe = fn << 4;
            if (gi < 7) fn = __ldg(rec + gi + 1);
            if (gi > 0) {
              const int cur = min((int)(ta - row_a) >> 1, CAS_BLK - 1);
              ta = row_a + 2u * (uint32_t)cur;
              bwindow(ms_a, 128u, cur + 1, 4, Hp, Lp);
              bwindow(st_a, 4u, q0 + 1 + (int)used, BlockStreams<2>::kRow - 3, Hc, Lc);
            }
            if (__popc(Hc) + __popc(Lc) < 8) {  // as for K
              int cur = (int)(ta - row_a) >> 1, qt = q0 + (int)used;
              for (int i = 0; i < 8; ++i) {
                const int pb = bnext_one(ms_a, 128u, cur + 1, 6);
                const int eb = bnext_one(st_a, 4u, qt + 1, BlockStreams<2>::kRow - 1);
                if (pb < 0 || pb >= CAS_BLK || eb < 0) {
                  cor |= 32u;
                  break;
                }
                const uint32_t E = lds_u32(lutv_a + 4u * (uint32_t)min(eb - qt - 1, 255));
                used += (uint32_t)(eb - qt);
                qt = eb;
                cur = pb;
                const uint32_t f = (fo >> (4 * i)) & 15u;
                sts_u16(row_a + 2u * (uint32_t)cur, ((f & 8u) << 12) | E | ((f & 7u) << 4));
              }
              ta = row_a + 2u * (uint32_t)max(cur, -1);
              continue;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t np = __clz(Hp) + 1u;
              ta = mad32(np, 2u, ta);
              Hp = shfl_wrap(Lp, Hp, np);
              Lp = shfl_wrap(0u, Lp, np);
              const uint32_t nc = __clz(Hc) + 1u;
              const uint32_t E = lds_u32(lutv_a - 4u + 4u * nc);
              Hc = shfl_wrap(Lc, Hc, nc);
              Lc = shfl_wrap(0u, Lc, nc);
              used += nc;
              cor |= np | nc;
              const int by = i >> 1;
              const uint32_t A = __byte_perm((i & 1) ? fo : fe, 0u, by * 0x11 | 0x4400);
              sts_u16(ta, (A & 0x8070u) | E);
            }
          }
        }
        // a walk that ran dry may have stored into the next rows: every lane
        // rebuilds its row by scanning
        if (__any_sync(CAS_FULL, valid && (cor & 32u))) {
          __syncwarp();
#pragma unroll
          for (int i = 0; i < CAS_BLK / 8; ++i) zr[i] = make_uint4(0u, 0u, 0u, 0u);
          bool ok = !valid || draft_v_scan(ms_a, st_a, q0, lutv_a, rec, row_a);
          if (!ok)
            for (int i = 0; i < CAS_BLK / 8; ++i) zr[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }
      if (!fast) {
        for (int u = 0; u < 4; ++u)
          decode_sb_tile<false>(d, H + h, n, sb0 + u, ds.vt, CAS_SB * u, lut8v, ds.u.tile_scratch, lane);
        block_streams_init(ds.u.w.st, lane);
#pragma unroll
        for (int r = 4; r < 7; ++r) ds.u.w.ms[r][lane] = 0u;
        __syncwarp();
      }
    }
    // ---- O^T += V^T P^T: rescale, then 2 k-steps x 8 m-tiles x (hi, lo)
    const float ca = tq == 0 ? corr[0] : corr[2], cb = tq == 0 ? corr[1] : corr[3];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      c[mt][0] *= ca;
      c[mt][1] *= cb;
      c[mt][2] *= ca;
      c[mt][3] *= cb;
    }
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t bh[2], bl[2];
      {
        const int r = lane & 7, kh = (lane >> 3) & 1;
        const uint32_t ah = smem_addr(&ds.ph[r][16 * ks + 8 * kh]), al = smem_addr(&ds.pl[r][16 * ks + 8 * kh]);
        asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(bh[0]), "=r"(bh[1]) : "r"(ah));
        asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(bl[0]), "=r"(bl[1]) : "r"(al));
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t av[4];
        const int tr = 16 * ks + (lane & 7) + ((lane >> 4) & 1) * 8, dc = 16 * mt + ((lane >> 3) & 1) * 8;
        ldmatrix_x4_trans(av, ds.vt + tr * kDRow + dc);
        mma_bf16(c[mt], av, bh[0], bh[1]);
        mma_bf16(c[mt], av, bl[0], bl[1]);
      }
    }
    __syncwarp();
  }
  // merge the 4 warps' states: o[w][q][dim] over the V tiles
  __syncthreads();
  float* ow = reinterpret_cast<float*>(stages);  // [4][4][128]
  __shared__ float wm[kWarps][4], wl[kWarps][4];
  if (lane < 4) {
    wm[warp][lane] = lane == 0 ? mst[0] : lane == 1 ? mst[1] : lane == 2 ? mst[2] : mst[3];
    wl[warp][lane] = lane == 0 ? lst[0] : lane == 1 ? lst[1] : lane == 2 ? lst[2] : lst[3];
  }
  if (tq < 2) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d0 = 16 * mt + gq;
      ow[(warp * 4 + 2 * tq) * CAS_BLK + d0] = c[mt][0];
      ow[(warp * 4 + 2 * tq + 1) * CAS_BLK + d0] = c[mt][1];
      ow[(warp * 4 + 2 * tq) * CAS_BLK + d0 + 8] = c[mt][2];
      ow[(warp * 4 + 2 * tq + 1) * CAS_BLK + d0 + 8] = c[mt][3];
    }
  }
  __syncthreads();
  // warp q writes query vector q's partial
  if (warp < nq) {
    const int q = warp;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) M = fmaxf(M, wm[w2][q]);
    float L = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      if (wm[w2][q] == -INFINITY) continue;
      const float f = __expf(wm[w2][q] - M);
      L += wl[w2][q] * f;
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] += f * ow[(w2 * 4 + q) * CAS_BLK + 4 * lane + i];
    }
    float* dst = a.part + (((int64_t)b * a.Hq + h * G + q) * a.nchunk + chunk) * kPart;
    reinterpret_cast<float2*>(dst)[2 * lane] = make_float2(o[0], o[1]);
    reinterpret_cast<float2*>(dst)[2 * lane + 1] = make_float2(o[2], o[3]);
    if (lane == 0) {
      dst[CAS_BLK] = M;
      dst[CAS_BLK + 1] = L;
    }
  }
}

int launch_draft_block(AttnArgs& a, int Hkv, cudaStream_t st) {
  const size_t smem = (size_t)CAS_BLK * 16 + 2 * 256 * 4 + 2 * 256 + (size_t)kWarps * sizeof(DraftStage);
  const int s = one_wave(a, Hkv, (const void*)attn_draft_block_kernel, smem);
  if (s) return s;
  return launch_k(attn_draft_block_kernel, dim3(a.nchunk, Hkv, a.B), kThreads, smem, st, a);
}

template <bool FULL, int MT>
int launch_mma(AttnArgs& a, int Hkv, cudaStream_t st) {
  // the block walks' stage (every Cassandra-1 cache uses a C-1 scratch)
  if (a.scr_warp == kScratchC1) a.scr_warp = std::max<int>(kScratchC1, (int)sizeof(KvBlockStage));
  const size_t smem = mma_smem(MT, a.scr_warp);
  auto kern = attn_mma_kernel<FULL, MT>;
  const int s = one_wave(a, Hkv, (const void*)kern, smem);
  if (s) return s;
  return launch_k(kern, dim3(a.nchunk, Hkv, a.B * a.ngroups), kThreads, smem, st, a);
}

// a.nchunk on entry: the most chunks the workspace holds; on return: the
// chunks launched (one wave of resident CTAs, at most that many).
template <bool FULL, int QPW>
int launch_chunk(AttnArgs& a, int Hkv, cudaStream_t st) {
  size_t smem = chunk_smem(a.qv_alloc, a.scr_warp);
  auto kern = attn_chunk_kernel<FULL, QPW>;
  const int s = one_wave(a, Hkv, (const void*)kern, smem);
  if (s) return s;
  dim3 grid(a.nchunk, Hkv, a.B * a.ngroups);
  return launch_k(kern, grid, kThreads, smem, st, a);
}

int run_attn(bool full, const cas_kv* const* kv, int B, const uint16_t* q, int T, int Hq, const uint16_t* tail_k,
             const uint16_t* tail_v, int n_tail, float* o, void* ws, uint64_t ws_bytes, cudaStream_t st) {
  if (!kv || B < 1 || B > kMaxBatch || !q || !o || T < 1 || T > kMaxT || Hq < 1 || !aligned16(q) || !aligned16(o))
    return CAS_ERR_INVALID;
  if (n_tail < 0 || n_tail > kMaxT || (n_tail > 0 && (!tail_k || !tail_v))) return CAS_ERR_INVALID;
  int Hkv = 0;
  int64_t Tm = 0;
  AttnArgs a{};
  CombineArgs c{};
  for (int i = 0; i < B; ++i) {
    int s = check_kv(kv[i]);
    if (s) return s;
    if (i == 0) Hkv = kv[i]->n_kv_heads;
    if (kv[i]->n_kv_heads != Hkv || kv[i]->p.keep_per_block != kv[0]->p.keep_per_block ||
        kv[i]->p.mant_bits != kv[0]->p.mant_bits)
      return CAS_ERR_INVALID;
    Tm = std::max(Tm, kv[i]->max_tokens);
    a.kv[i] = make_kv_dev(kv[i]);
    a.scr_warp = std::max(a.scr_warp, kv[i]->p.variant == 1 ? kScratchC1 : kScratchC2);
    c.ntok[i] = (const int64_t*)((uint8_t*)kv[i]->base + kv[i]->off[CAS_KV_STATE]);
  }
  if (Hq % Hkv) return CAS_ERR_INVALID;
  int G = Hq / Hkv;
  if (T * G > kWarps * 16) return CAS_ERR_INVALID;
  uint64_t need = cas_attn_workspace_bytes(B, Hq, T, Tm);
  if (!ws || ws_bytes < need || !aligned16(ws)) return CAS_ERR_BUFFER;
  a.q = q;
  a.part = (float*)ws;
  a.B = B;
  a.T = T;
  a.Hq = Hq;
  a.G = G;
  a.nchunk = nchunks(Tm);
  a.scale = 1.0f / std::sqrt((float)CAS_BLK);
  a.ngroups = (T * G + kQvPerCta - 1) / kQvPerCta;
  a.qv_alloc = std::min(T * G, kQvPerCta);
  int qpw = (std::min(T * G, kQvPerCta) + kWarps - 1) / kWarps;
  int s;
  bool block_ok = true;  // every cache Cassandra-1 with k = 64, m = 3
  for (int i = 0; i < B; ++i)
    block_ok = block_ok && kv[i]->p.variant == 1 && kv[i]->p.keep_per_block == 64 && kv[i]->p.mant_bits == 3;
  if (!full && T == 1 && a.qv_alloc <= 4 && block_ok) {
    s = launch_draft_block(a, Hkv, st);
  } else if (!full && T == 1 && a.qv_alloc <= 4) {
    s = launch_fused(a, Hkv, st);
  } else if (!full) {
    s = qpw <= 4 ? launch_chunk<false, 4>(a, Hkv, st) : launch_chunk<false, 8>(a, Hkv, st);
  } else {
    s = a.qv_alloc > 16 ? launch_mma<true, 2>(a, Hkv, st) : launch_mma<true, 1>(a, Hkv, st);
  }
  if (s) return s;
  c.part = a.part;
  c.q = q;
  c.tail_k = tail_k;
  c.tail_v = tail_v;
  c.o = o;
  c.T = T;
  c.Hq = Hq;
  c.Hkv = Hkv;
  c.G = G;
  c.nchunk = a.nchunk;
  c.n_tail = full ? 0 : n_tail;
  c.scale = a.scale;
  return launch_k(attn_combine_kernel, dim3(Hq, T, B), kCombineWarps * 32, 0, st, c);
}

}  // namespace
}  // namespace cas

using namespace cas;

extern "C" uint64_t cas_attn_workspace_bytes(int B, int Hq, int T, int64_t max_tokens) {
  if (B < 1 || Hq < 1 || T < 1 || max_tokens < 1) return 0;
  return (uint64_t)B * T * Hq * nchunks(max_tokens) * kPart * sizeof(float);
}

extern "C" int cas_draft_attn_decode(const cas_kv* const* kv, int batch, const uint16_t* q, int n_q_heads,
                                     const uint16_t* tail_k, const uint16_t* tail_v, int n_tail, float* o,
                                     void* workspace, uint64_t workspace_bytes, void* stream) {
  return run_attn(false, kv, batch, q, 1, n_q_heads, tail_k, tail_v, n_tail, o, workspace, workspace_bytes,
                  (cudaStream_t)stream);
}

extern "C" int cas_verify_attn(const cas_kv* const* kv, int batch, const uint16_t* q, int T, int n_q_heads, float* o,
                               void* workspace, uint64_t workspace_bytes, void* stream) {
  return run_attn(true, kv, batch, q, T, n_q_heads, nullptr, nullptr, 0, o, workspace, workspace_bytes,
                  (cudaStream_t)stream);
}

// ------------------------------------------------------------------ no-allocation variant
// Some callers cannot allocate device memory at the time they decode: a host
// runtime whose memory plan is fixed at start-up and forbids later
// allocation, or an embedding application that owns every allocation and
// hands this library only its inputs and outputs. For them the draft
// attention keeps its chunk partials in this fixed array instead of a
// caller-provided workspace. It is part of the library's device image, so
// every GPU that loads the library holds it until the process exits.
namespace {

constexpr uint64_t kStaticScratchBytes = 8ull << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

// Device address of g_attn_scratch in the current context. The host symbol is
// only a stand-in, so the address is looked up on every call: a context that
// was rebuilt (cudaDeviceReset) or another context on the same device holds
// the array at another address.
int static_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return CAS_ERR_CUDA;
  *out = p;
  return CAS_OK;
}

}  // namespace

extern "C" int cas_draft_attn_decode_noalloc(const cas_kv* const* kv, int batch, const uint16_t* q, int n_q_heads,
                                             const uint16_t* tail_k, const uint16_t* tail_v, int n_tail, float* o,
                                             void* stream) {
  if (!kv || batch < 1 || batch > kMaxBatch || n_q_heads < 1) return CAS_ERR_INVALID;
  int64_t Tm = 0;
  for (int i = 0; i < batch; ++i) {
    const int s = check_kv(kv[i]);  // the same descriptor errors as the workspace version
    if (s) return s;
    Tm = std::max(Tm, kv[i]->max_tokens);
  }
  const uint64_t need = cas_attn_workspace_bytes(batch, n_q_heads, 1, Tm);
  if (need > kStaticScratchBytes) return CAS_ERR_BUFFER;
  void* ws = nullptr;
  int s = static_scratch(&ws);
  if (s) return s;
  // every partial the combine step reads is written by the chunk step of this
  // same call, so nothing in the array needs clearing between calls
  return run_attn(false, kv, batch, q, 1, n_q_heads, tail_k, tail_v, n_tail, o, ws, kStaticScratchBytes,
                  (cudaStream_t)stream);
}
