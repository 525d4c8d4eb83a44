// gemm.cu - verify: lossless reconstruct + GEMM, Y[t][n] = sum_k W[n][k] X[t][k].
//
// The target merges speculation and verification data back to the original
// bits (Cassandra blog review, section 3.1) and runs T = draft length + 1
// tokens at once, so the product is a small dense contraction. A CTA takes a
// tile of 16 rows by one superblock column (up to 1024 k): its 8 warps
// rebuild the 16 row-superblocks bit-exactly into a shared-memory tile, then
// split the k16 steps of the tile among themselves on the tensor cores
// (mma m16n8k16, bf16 inputs, fp32 accumulation; T <= 8 uses one n8 tile, T <= 16
// two). Warp partials are summed in shared memory and added to Y with fp32
// atomics; Y is cleared first. Cassandra-1 with k = 64, m = 3 on rows of whole
// superblocks rebuilds the tile by block walks (verify_gemm_block_kernel,
// blockwalk.cuh); other k, m and Cassandra-2 by the per-lane run decoders of
// lanedec.cuh; rows ending in a partial superblock by the generic warp
// decoder of sbdecode.cuh.
#include <cuda_runtime.h>

#include <algorithm>

#include "lanedec.cuh"
#include "mma.cuh"
#include "sbdecode.cuh"
#include "wordlane.cuh"
#include "blockwalk.cuh"

namespace cas {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 16;
// Tile row: the 8 blocks of a row-superblock, each followed by 8 bf16 of
// padding (blocks start in different banks, so the decoder's scattered
// stores spread), then 8 more (rows start 4 banks apart: conflict-free
// ldmatrix).
constexpr int kBlkStride = CAS_BLK + 8;
constexpr int kTileStride = kBlkStride * CAS_SB + 8;
// tile column of k-step ks (16 columns)
__device__ __forceinline__ int tile_col(int ks) { return kBlkStride * (ks >> 3) + 16 * (ks & 7); }

struct GemmArgs {
  WView w;
  Lut lut;
  const uint16_t* X;
  float* Y;
  int T;
};

// Per-warp decode scratch: the cursor decoder's stage, or the generic
// decoder's kept + pruned codes (+ Cassandra-2 residual words); a multiple of
// 16 bytes (the cursor decoder reads its position arrays as uint4). The warp
// partials of the product reuse this region after the decode.
template <int VAR>
__host__ __device__ constexpr int scratch_warp() {
  constexpr int generic = 2048 + (VAR == 2 ? kResWords * 4 : 0);
  return (((int)sizeof(TileStage) > generic ? (int)sizeof(TileStage) : generic) + 15) & ~15;
}
static_assert(scratch_warp<1>() % 16 == 0 && alignof(TileStage) <= 16, "per-warp scratch alignment");
static_assert(scratch_warp<2>() >= (int)sizeof(TileStage2) && alignof(TileStage2) <= 16, "Cassandra-2 stage fits");
static_assert(kWarps * scratch_warp<1>() >= kWarps * 256 * 4, "warp partials fit in the scratch");

// MODE 2: rows of whole superblocks, any k, m (runs_sb_tile, Cassandra-2:
// runs_sb_tile_c2); MODE 0: generic. (Cassandra-1 with k = 64, m = 3 runs
// verify_gemm_block_kernel below.)
template <int VAR, int NT, int MODE>
__global__ void __launch_bounds__(kThreads, 4) verify_gemm_kernel(GemmArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  const WView& w = a.w;
  uint16_t* tile = reinterpret_cast<uint16_t*>(smem);  // [16][kTileStride]
  uint8_t* s_lut = smem + kRows * kTileStride * 2;
  uint8_t* scratch = s_lut + 256;
  float* red = reinterpret_cast<float*>(scratch);  // [8][16][16], after the decode
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t* wscr = scratch + warp * scratch_warp<VAR>();
  SbScratch sc{wscr, wscr + 1024, reinterpret_cast<uint32_t*>(wscr + 2048)};
  TileStage& ts = *reinterpret_cast<TileStage*>(wscr);
  for (int i = threadIdx.x; i < 256; i += kThreads) s_lut[i] = a.lut.v[i];
  __syncthreads();

  const int64_t ntile = (w.N + kRows - 1) / kRows;
  const int64_t ntasks = ntile * w.nsr;
  const int K = (int)w.K, T = a.T;
  const uint32_t* X32 = reinterpret_cast<const uint32_t*>(a.X);
  for (int64_t task = blockIdx.x; task < ntasks; task += gridDim.x) {
    int64_t rt = task / w.nsr;
    int j = (int)(task % w.nsr);
    int nb = min(CAS_SB, w.nbr - CAS_SB * j);
    // 1) rebuild rows rt*16 + {warp, warp + 8}
    for (int r = warp; r < kRows; r += kWarps) {
      int64_t n = rt * kRows + r;
      uint4* dst = reinterpret_cast<uint4*>(tile + r * kTileStride + kBlkStride * (lane >> 2) + 32 * (lane & 3));
      bool done = false;
      if (n < w.N && MODE != 0) {
        const int64_t s = n * w.nsr + j;
        const int64_t gb0 = n * w.nbr + CAS_SB * j;
        uint32_t v0, v1;
        stream_range(w.vidx, s, w.lim_vexp, v0, v1);
        if (VAR == 2) {
          uint32_t d0, d1, r0, r1;
          stream_range(w.vdidx, s, w.lim_vd, d0, d1);
          stream_range(w.vresidx, s, w.lim_vres, r0, r1);
          done = runs_sb_tile_c2<true>(w.mask + gb0 * 4, w.sq + gb0 * w.rec_q, w.rec_q, w.smx + gb0 * 4,
                                       w.vd + d0, (int)(d1 - d0), w.vres + r0,
                                       w.vpr + gb0 * w.rec_pr, w.rec_pr, w.vexp + v0, (int)(v1 - v0), w.k, w.m,
                                       s_lut, *reinterpret_cast<TileStage2*>(wscr), tile + r * kTileStride,
                                       kBlkStride, lane);
        } else {
          uint32_t a0, a1;
          stream_range(w.sidx, s, w.lim_sexp, a0, a1);
          done = runs_sb_tile<true>(w.mask + gb0 * 4, w.ssm + gb0 * w.rec_sm, w.rec_sm, w.vlo + gb0 * w.rec_lo,
                                    w.rec_lo, w.vpr + gb0 * w.rec_pr, w.rec_pr, w.sexp + a0, (int)(a1 - a0),
                                    w.vexp + v0, (int)(v1 - v0), w.k, w.m, s_lut, ts.us, ts.kpos,
                                    tile + r * kTileStride, kBlkStride, lane);
        }
      }
      if (done) {
      } else if (n < w.N) {
        SbInfo in = sb_prepare<VAR, true>(w, n * w.nsr + j, s_lut, sc, lane);
        if (lane < 4 * nb) {
          uint32_t v[16];
          sb_rebuild_word<VAR, true>(w, in, sc, lane, v);
          dst[0] = make_uint4(v[0], v[1], v[2], v[3]);
          dst[1] = make_uint4(v[4], v[5], v[6], v[7]);
          dst[2] = make_uint4(v[8], v[9], v[10], v[11]);
          dst[3] = make_uint4(v[12], v[13], v[14], v[15]);
        }
        __syncwarp();
      } else if (lane < 4 * nb) {
        uint4 z = make_uint4(0, 0, 0, 0);
        dst[0] = z; dst[1] = z; dst[2] = z; dst[3] = z;
      }
    }
    // 2) tensor-core product of the tile with X[:, tile columns]. This warp's X
    // fragments (k-steps warp, warp + 8, ...) are loaded before the barrier so
    // their latency overlaps the other warps' decode.
    const int g = lane >> 2, tq = lane & 3;
    const int ksteps = nb * (CAS_BLK / 16);
    constexpr int kKsPerWarp = CAS_BLK * CAS_SB / 16 / kWarps;
    uint32_t xb[kKsPerWarp][NT][2];
#pragma unroll
    for (int i = 0; i < kKsPerWarp; ++i) {
      const int ks = warp + kWarps * i;
      const int col = CAS_BLK * CAS_SB * j + ks * 16 + 2 * tq;
#pragma unroll
      for (int q = 0; q < NT; ++q) {
        const int tok = q * 8 + g;
        xb[i][q][0] = xb[i][q][1] = 0u;
        if (ks < ksteps && tok < T) {
          xb[i][q][0] = __ldg(X32 + ((int64_t)tok * K + col) / 2);
          xb[i][q][1] = __ldg(X32 + ((int64_t)tok * K + col + 8) / 2);
        }
      }
    }
    __syncthreads();
    float c[NT][4];
#pragma unroll
    for (int q = 0; q < NT; ++q) c[q][0] = c[q][1] = c[q][2] = c[q][3] = 0.f;
#pragma unroll
    for (int i = 0; i < kKsPerWarp; ++i) {
      const int ks = warp + kWarps * i;
      if (ks < ksteps) {
        uint32_t af[4];
        ldmatrix_x4(af, tile + (lane & 15) * kTileStride + tile_col(ks) + (lane >> 4) * 8);
#pragma unroll
        for (int q = 0; q < NT; ++q) mma_bf16(c[q], af, xb[i][q][0], xb[i][q][1]);
      }
    }
    // 3) reduce warp partials: red[warp][row][token]
    float* rw = red + warp * 256;
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      rw[g * 16 + q * 8 + 2 * tq] = c[q][0];
      rw[g * 16 + q * 8 + 2 * tq + 1] = c[q][1];
      rw[(g + 8) * 16 + q * 8 + 2 * tq] = c[q][2];
      rw[(g + 8) * 16 + q * 8 + 2 * tq + 1] = c[q][3];
    }
    __syncthreads();
    {
      int r = threadIdx.x >> 4, tt = threadIdx.x & 15;
      int64_t n = rt * kRows + r;
      if (tt < T && tt < NT * 8 && n < w.N) {
        float sum = 0.f;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) sum += red[ww * 256 + r * 16 + tt];
        atomicAdd(a.Y + (int64_t)tt * w.N + n, sum);
      }
    }
    __syncthreads();
  }
}

template <int VAR, int NT, int MODE>
int launch(const GemmArgs& a, cudaStream_t st) {
  size_t smem = (size_t)kRows * kTileStride * 2 + 256 + kWarps * scratch_warp<VAR>();
  auto kern = verify_gemm_kernel<VAR, NT, MODE>;
  int per_sm = occupancy((const void*)kern, kThreads, smem);
  if (per_sm < 1) return CAS_ERR_CUDA;
  int64_t ntasks = (a.w.N + kRows - 1) / kRows * a.w.nsr;
  int g = (int)std::max<int64_t>(1, std::min<int64_t>(ntasks, (int64_t)sm_count() * per_sm));
  return launch_k(kern, g, kThreads, smem, st, a);
}


// ------------------------------------------------------------------ block path
// Cassandra-1, k = 64, m = 3, rows of whole superblocks. A CTA of 8 warps
// takes 16 rows by one superblock column; warp w rebuilds rows 2w and 2w + 1.
// Each block is walked by two lanes (blockwalk.cuh): lane 8t + j takes block j
// of row 2w + (t >> 1), its 64 kept values for even t and its 64 pruned
// values for odd t, so the warp's four staged code streams are row 0 kept, row
// 0 pruned, row 1 kept, row 1 pruned and every lane walks 64 values:
// positions from a window over the bit-reversed mask (or its complement),
// exponents from a window over its stream. A kept value joins its sign and 3
// high mantissa bits with the 4 cut bits of the verification record, a pruned
// value is its byte of the pruned record; both are laid out as even and odd
// bytes per group of 8, so the per-value code is the same for both kinds. Each
// bf16 goes to its position in the tile. When a lane meets a step of 32 or more
// (a long gap or code), the stores of its failed walk may land up to 655
// positions past its block's start (position 127 at a re-alignment, then 16
// steps of at most 33) - in the warp's own rows, the next warp's first row, or
// the slack after the tile - so that warp and the next one rebuild
// their rows by scanning the staged words instead; streams longer than the
// stage go to the generic decoder. Then the product runs as in
// verify_gemm_kernel.
constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr int kVRows = 2 * kVWarps;
// Tile layout (bf16 elements): block j of row r at vrow(r) + 132 j. In 4-byte
// banks a block is 66 words (2 banks on) and a row 528 words plus 4 after
// every odd row, so the 16 blocks a warp writes (rows 2w and 2w + 1) start on
// 16 different even banks, and rows 0..7 start on 8 different multiples of 4
// (conflict-free A-fragment loads). The scattered 16-bit stores of the walk
// then meet each other on a bank only when two lanes' positions drift apart.
constexpr int kVBlk = CAS_BLK + 4;
constexpr int kVRowLen = kVBlk * CAS_SB;
__host__ __device__ constexpr int vrow(int r) { return r * kVRowLen + 8 * (r >> 1); }
// slack after the tile (bytes): a failed walk stores up to position
// 7 * 132 + 655 of the last row
constexpr int kVPad = ((vrow(kVRows - 1) + 7 * kVBlk + 656 - vrow(kVRows)) * 2 + 127) / 128 * 128;
constexpr int kVTile = vrow(kVRows) + kVPad / 2;  // elements
static_assert(vrow(kVRows - 1) + 7 * kVBlk + 656 <= kVTile, "slack covers a failed walk of the last row");
static_assert(7 * kVBlk + 656 - kVRowLen <= kVRowLen, "a failed walk stays within the next row");
// The tile's k-step ks (16 columns) and A fragment (mma m16n8k16, row-major):
// rows g, g + 8 and columns 2 tq (+ 8) of the step, one 32-bit load each.
__device__ __forceinline__ void vtile_afrag(uint32_t a[4], uint32_t tile_a, int ks, int g, int tq) {
  const uint32_t c = 2u * (uint32_t)(kVBlk * (ks >> 3) + 16 * (ks & 7) + 2 * tq);
  const uint32_t r0 = tile_a + 2u * (uint32_t)vrow(g) + c, r1 = tile_a + 2u * (uint32_t)vrow(g + 8) + c;
  a[0] = lds_u32(r0);
  a[1] = lds_u32(r1);
  a[2] = lds_u32(r0 + 16u);
  a[3] = lds_u32(r1 + 16u);
}

using VerifyStreams = BlockStreams<3, 80>;
struct VerifyStage {
  VerifyStreams st;    // codes: row 0 kept, row 0 pruned, row 1 kept, row 1 pruned (up to 80 words each)
  uint32_t ms[7][32];  // row i, column l: bit-reversed word i of lane l's positions; rows 4-6 zero
};
static_assert(sizeof(VerifyStage) % 16 == 0, "stage alignment");
static_assert(sizeof(VerifyStage) >= 2048, "the generic decoder's codes fit in the stage");
static_assert(kVWarps * sizeof(VerifyStage) >= kVWarps * 256 * 4, "warp partials fit over the stages");

// Zero rows and words of a warp's stage.
__device__ __forceinline__ void verify_stage_init(VerifyStage& vs, int lane) {
  block_streams_init(vs.st, lane);
#pragma unroll
  for (int r = 4; r < 7; ++r) vs.ms[r][lane] = 0u;
}

// The walk of one lane's 64 values without windows: every position and code
// found by a scan of the staged words (any gap, any code length), the record
// read again through the cache. For a warp whose windowed walk stepped 32 or
// more; false when the staged data runs out (the encoding is inconsistent).
__device__ __noinline__ bool verify_lane_scan(uint32_t ms_a, uint32_t st_a, int q0, uint32_t lut_a, bool pruned,
                                              const uint32_t* __restrict__ ra, const uint32_t* __restrict__ rb,
                                              uint32_t tb) {
  int cur = -1, q = q0;
  for (int i = 0; i < 64; ++i) {
    const int p = bnext_one(ms_a, 128u, cur + 1, 6);
    const int e = bnext_one(st_a, 4u, q + 1, VerifyStreams::kRow - 1);
    if (p < 0 || p >= CAS_BLK || e < 0) return false;
    cur = p;
    const uint32_t E = lds_u32(lut_a + 4u * (uint32_t)min(e - q, 256));  // rank e - q - 1
    q = e;
    uint32_t b;
    if (pruned) {
      b = (__ldg(ra + (i >> 2)) >> (8 * (i & 3))) & 255u;
    } else {
      const int sh = 4 * (i & 7);
      b = (((__ldg(ra + (i >> 3)) >> sh) & 15u) << 4) | ((__ldg(rb + (i >> 3)) >> sh) & 15u);
    }
    sts_u16(tb + 2u * (uint32_t)cur, ((b & 0x80u) << 8) | E | (b & 0x7Fu));
  }
  return true;
}

template <int NT>
__global__ void __launch_bounds__(kVThreads, 4) verify_gemm_block_kernel(GemmArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t lut7[256];  // exponent << 7 by rank
  __shared__ uint8_t lut8[256];   // exponent by rank (generic decoder)
  __shared__ uint32_t s_bad;      // bit w: warp w's walk stepped 32 or more in this task
  const WView& w = a.w;
  uint16_t* tile = reinterpret_cast<uint16_t*>(smem);
  VerifyStage& vs = reinterpret_cast<VerifyStage*>(smem + kVTile * 2)[threadIdx.x >> 5];
  float* red = reinterpret_cast<float*>(smem + kVTile * 2);  // [warps][16][16], over the stages after the decode
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 256; i += kVThreads) {
    lut7[i] = (uint32_t)a.lut.v[i] << 7;
    lut8[i] = a.lut.v[i];
  }
  if (threadIdx.x == 0) s_bad = 0u;
  __syncthreads();

  const int64_t ntile = (w.N + kVRows - 1) / kVRows;
  const int64_t ntasks = ntile * w.nsr;
  const int K = (int)w.K, T = a.T;
  const uint32_t* X32 = reinterpret_cast<const uint32_t*>(a.X);
  const int t = lane >> 3, j = lane & 7;
  const bool pruned = t & 1;
  const uint32_t ms_a0 = smem_addr(&vs.ms[0][lane]), st_a0 = smem_addr(&vs.st.w[t][0]);
  const uint32_t lut_a = smem_addr(lut7) - 4u;  // rank c - 1 at lut_a + 4c
  const uint32_t tile_a = smem_addr(tile);
  for (int64_t task = blockIdx.x; task < ntasks; task += gridDim.x) {
    // task indices fit 32 bits (launch checks): 32-bit division
    const uint32_t nsr32 = (uint32_t)w.nsr;
    const uint32_t rt32 = (uint32_t)task / nsr32;
    const int64_t rt = rt32;
    const int col = (int)((uint32_t)task - rt32 * nsr32);
    const int64_t r0 = rt * kVRows + 2 * warp;  // the warp's first row
    const int64_t n = r0 + (t >> 1);            // this lane's row
    const bool valid = n < w.N;
    // 1) rebuild rows r0, r0 + 1 of the tile (the stage's zero words first: the
    // previous task's partials and the generic decoder write over them)
    verify_stage_init(vs, lane);
    // stream u (row r0 + u / 2, kept codes for even u, pruned for odd) is
    // located by lane u
    uint32_t ua = 0u, ub = 0u;
    if (lane < 4 && r0 + (lane >> 1) < w.N) {
      const int64_t s = (r0 + (lane >> 1)) * w.nsr + col;
      if (lane & 1)
        stream_range(w.vidx, s, w.lim_vexp, ua, ub);
      else
        stream_range(w.sidx, s, w.lim_sexp, ua, ub);
    }
    const int present = r0 + 1 < w.N ? 4 : (r0 < w.N ? 2 : 0);
    const uint32_t* gs[4];
    int nw[4];
    bool fast = true;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t a0 = __shfl_sync(CAS_FULL, ua, u);
      nw[u] = (int)__shfl_sync(CAS_FULL, ub - ua, u);
      gs[u] = ((u & 1) ? w.vexp : w.sexp) + a0;
      fast = fast && nw[u] <= VerifyStreams::kWords;
    }
    const int64_t gb = (valid ? n : r0) * w.nbr + CAS_SB * col + j;  // this lane's block
    const uint32_t tb = tile_a + 2u * (uint32_t)(vrow(2 * warp + (t >> 1)) + kVBlk * j);
    int q0s = 0;
    if (fast) {
      const uint4 mk = ldg_once(reinterpret_cast<const uint4*>(w.mask) + gb);
      // the lane's records: kept, spec_sm and ver_lo words (one each per group
      // of 8); pruned, ver_pr words (two per group)
      const uint32_t* ra = pruned ? w.vpr + gb * 16 : w.ssm + gb * 8;
      const uint32_t* rb = pruned ? w.vpr + gb * 16 + 1 : w.vlo + gb * 8;
      const int rs = pruned ? 2 : 1;
      const uint32_t inv = pruned ? 0xFFFFFFFFu : 0u;
      vs.ms[0][lane] = valid ? __brev(mk.x ^ inv) : 0u;
      vs.ms[1][lane] = valid ? __brev(mk.y ^ inv) : 0u;
      vs.ms[2][lane] = valid ? __brev(mk.z ^ inv) : 0u;
      vs.ms[3][lane] = valid ? __brev(mk.w ^ inv) : 0u;
      const int q0 = block_code_term<3, 64>(gs, nw, present, vs.st, lane, fast);
      const uint32_t ms_a = fenced(ms_a0), st_a = fenced(st_a0);
      uint32_t ta = tb - 2u;  // tile address of the last found position (-1 at first)
      uint32_t Hp, Lp, Hc, Lc;
      bwindow(ms_a, 128u, 0, 4, Hp, Lp);
      bwindow(st_a, 4u, q0 + 1, VerifyStreams::kRow - 3, Hc, Lc);
      uint32_t used = 0u, cor = 0u;
      uint32_t an = __ldg(ra), bn = __ldg(rb);  // the next group's record words
#pragma unroll 1
      for (int gi = 0; gi < 8; ++gi) {
        const uint32_t aw = an, bw = bn;
        if (gi < 7) {
          ra += rs;
          rb += rs;
          an = __ldg(ra);
          bn = __ldg(rb);
        }
        if (gi > 0) {
          // the position window is re-aligned every 16 values (16 of the
          // block's 64 positions almost never span more than its 64 bits, and
          // a window that runs dry is caught like a long gap), the code window
          // every 8
          if ((gi & 1) == 0) {
            const int cur = min((int)(ta - tb) >> 1, CAS_BLK - 1);
            ta = tb + 2u * (uint32_t)cur;
            bwindow(ms_a, 128u, cur + 1, 4, Hp, Lp);  // rows <= 6 since cur <= 127
          }
          bwindow(st_a, 4u, q0 + 1 + (int)used, VerifyStreams::kRow - 3, Hc, Lc);
        }
        // bytes [s f6 .. f0] of the group's values 0, 2, 4, 6 (ev) and 1, 3, 5, 7 (od)
        const uint32_t ev = pruned ? __byte_perm(aw, bw, 0x6420)
                                   : ((aw << 4) & 0xF0F0F0F0u) | (bw & 0x0F0F0F0Fu);
        const uint32_t od = pruned ? __byte_perm(aw, bw, 0x7531)
                                   : (aw & 0xF0F0F0F0u) | ((bw >> 4) & 0x0F0F0F0Fu);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t np = __clz(Hp) + 1u;  // distance to the next position
          ta = mad32(np, 2u, ta);
          Hp = shfl_wrap(Lp, Hp, np);
          Lp = shfl_wrap(0u, Lp, np);
          const uint32_t nc = __clz(Hc) + 1u;  // rank + 1
          const uint32_t E = lds_u32(lut_a + 4u * nc);
          Hc = shfl_wrap(Lc, Hc, nc);
          Lc = shfl_wrap(0u, Lc, nc);
          used += nc;
          cor |= np | nc;
          const uint32_t A = __byte_perm((i & 1) ? od : ev, 0u, (uint32_t)(i >> 1) * 0x11u | 0x4400u);
          sts_u16(ta, (A & 0x807Fu) | E);
        }
      }
      if (__any_sync(CAS_FULL, valid && (cor & 32u)) && lane == 0) atomicOr(&s_bad, 1u << warp);
      q0s = q0;
    }
    // a step of 32 or more in this warp or the one before: rebuild by the scan
    // walk (a failed walk may have stored into the blocks after it)
    __syncthreads();
    const uint32_t bad = s_bad;
    if (((bad >> warp) & 1u || (warp > 0 && ((bad >> (warp - 1)) & 1u))) && fast) {
      const uint32_t* ra = pruned ? w.vpr + gb * 16 : w.ssm + gb * 8;
      const uint32_t* rb = pruned ? w.vpr + gb * 16 + 1 : w.vlo + gb * 8;
      const bool ok = !valid || verify_lane_scan(fenced(ms_a0), fenced(st_a0), q0s, lut_a, pruned, ra, rb, tb);
      fast = __all_sync(CAS_FULL, ok);
    }
    __syncwarp();
    if (!fast) {  // the generic decoder, one row-superblock at a time
      SbScratch sc{reinterpret_cast<uint8_t*>(&vs), reinterpret_cast<uint8_t*>(&vs) + 1024, nullptr};
      for (int u = 0; u < 2; ++u) {
        if (r0 + u >= w.N) break;
        const SbInfo in = sb_prepare<1, true>(w, (r0 + u) * w.nsr + col, lut8, sc, lane);
        uint32_t v[16];
        sb_rebuild_word<1, true>(w, in, sc, lane, v);
        uint2* dst = reinterpret_cast<uint2*>(tile + vrow(2 * warp + u) + kVBlk * (lane >> 2) + 32 * (lane & 3));
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_uint2(v[2 * i], v[2 * i + 1]);
        __syncwarp();
      }
    }
    // 2) tensor-core product of the tile with X[:, tile columns]. The lane's
    // B fragment words of k-step warp + 8 i: token gq (+ 8), columns
    // 1024 col + 16 (warp + 8 i) + 2 tq (+ 8), as words of bf16 pairs (K is
    // a multiple of 1024 here).
    const int gq = lane >> 2, tq = lane & 3;
    constexpr int kKs = CAS_BLK * CAS_SB / 16 / kVWarps;
    uint32_t xb[kKs][NT][2];
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      const int tok = q * 8 + gq;
      const uint32_t* xq = X32 + (size_t)min(tok, T - 1) * (size_t)(K / 2) + 512 * col + 8 * warp + tq;
#pragma unroll
      for (int i = 0; i < kKs; ++i) {
        xb[i][q][0] = tok < T ? __ldg(xq + 64 * i) : 0u;
        xb[i][q][1] = tok < T ? __ldg(xq + 64 * i + 4) : 0u;
      }
    }
    __syncthreads();
    float acc[NT][4];
#pragma unroll
    for (int q = 0; q < NT; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
#pragma unroll
    for (int i = 0; i < kKs; ++i) {
      const int ks = warp + kVWarps * i;
      uint32_t af[4];
      vtile_afrag(af, fenced(tile_a), ks, gq, tq);
#pragma unroll
      for (int q = 0; q < NT; ++q) mma_bf16(acc[q], af, xb[i][q][0], xb[i][q][1]);
    }
    // 3) reduce warp partials: red[warp][row][token]
    float* rw = red + warp * 256;
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      rw[gq * 16 + q * 8 + 2 * tq] = acc[q][0];
      rw[gq * 16 + q * 8 + 2 * tq + 1] = acc[q][1];
      rw[(gq + 8) * 16 + q * 8 + 2 * tq] = acc[q][2];
      rw[(gq + 8) * 16 + q * 8 + 2 * tq + 1] = acc[q][3];
    }
    __syncthreads();
    {
      const int r = threadIdx.x >> 4, tt = threadIdx.x & 15;
      const int64_t nn2 = rt * kVRows + r;
      if (tt < T && tt < NT * 8 && nn2 < w.N) {
        float sum = 0.f;
#pragma unroll
        for (int ww = 0; ww < kVWarps; ++ww) sum += red[ww * 256 + r * 16 + tt];
        atomicAdd(a.Y + (int64_t)tt * w.N + nn2, sum);
      }
      if (threadIdx.x == 0) s_bad = 0u;
    }
    __syncthreads();
  }
}

template <int NT>
int launch_block(const GemmArgs& a, cudaStream_t st) {
  const size_t smem = (size_t)kVTile * 2 + kVWarps * sizeof(VerifyStage);
  auto kern = verify_gemm_block_kernel<NT>;
  const int per_sm = occupancy((const void*)kern, kVThreads, smem);
  if (per_sm < 1) return CAS_ERR_CUDA;
  const int64_t ntasks = (a.w.N + kVRows - 1) / kVRows * a.w.nsr;
  if (ntasks + (int64_t)sm_count() * per_sm >= (int64_t)1 << 32) return CAS_ERR_INVALID;  // 32-bit task indices
  const int g = (int)std::max<int64_t>(1, std::min<int64_t>(ntasks, (int64_t)sm_count() * per_sm));
  return launch_k(kern, g, kVThreads, smem, st, a);
}

}  // namespace

int corrupt_status_gemm(bool clear) {
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
}  // namespace cas

using namespace cas;

namespace {
int verify_gemm_call(const cas_weights* W, const uint16_t* X, int T, float* Y, bool accumulate, cudaStream_t st) {
  int s = check_weights(W);
  if (s) return s;
  if (T < 1 || T > 16) return CAS_ERR_INVALID;
  if (W->N == 0) return CAS_OK;  // nothing to write (Y may be an empty tensor)
  if (!X || !Y || !aligned16(X) || !aligned16(Y)) return CAS_ERR_INVALID;
  if (!accumulate)
    if (const int e = zero_f32(Y, (int64_t)T * W->N, st)) return e;
  if (W->K == 0) return CAS_OK;
  GemmArgs a;
  a.w = make_view(W);
  for (int i = 0; i < 256; ++i) a.lut.v[i] = W->exp_of_rank[i];
  a.X = X;
  a.Y = Y;
  a.T = T;
  bool v1 = W->p.variant == 1;
  const bool whole = a.w.nbr % CAS_SB == 0;
  const bool fast = v1 && a.w.k == 64 && a.w.m == 3 && whole;
  if (T <= 8) {
    if (fast) return launch_block<1>(a, st);
    if (whole) return v1 ? launch<1, 1, 2>(a, st) : launch<2, 1, 2>(a, st);
    return v1 ? launch<1, 1, 0>(a, st) : launch<2, 1, 0>(a, st);
  }
  if (fast) return launch_block<2>(a, st);
  if (whole) return v1 ? launch<1, 2, 2>(a, st) : launch<2, 2, 2>(a, st);
  return v1 ? launch<1, 2, 0>(a, st) : launch<2, 2, 0>(a, st);
}
}  // namespace

extern "C" int cas_verify_gemm(const cas_weights* W, const uint16_t* X, int T, float* Y, void* stream) {
  return verify_gemm_call(W, X, T, Y, false, (cudaStream_t)stream);
}

extern "C" int cas_verify_gemm_accumulate(const cas_weights* W, const uint16_t* X, int T, float* Y, void* stream) {
  return verify_gemm_call(W, X, T, Y, true, (cudaStream_t)stream);
}
