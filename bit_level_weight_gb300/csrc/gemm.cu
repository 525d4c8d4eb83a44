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
// atomics; Y is cleared first. The row-superblocks are rebuilt by the
// per-lane decoders of lanedec.cuh (k = 64, m = 3; any k, m on rows of whole
// superblocks, both variants) or, for rows ending in a partial superblock, by
// the generic warp decoder of sbdecode.cuh.
#include <cuda_runtime.h>

#include <algorithm>

#include "lanedec.cuh"
#include "mma.cuh"
#include "sbdecode.cuh"
#include "wordlane.cuh"

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
static_assert(scratch_warp<1>() >= (int)sizeof(WordTileStage), "word decoder stage fits");
static_assert(scratch_warp<2>() >= (int)sizeof(TileStage2) && alignof(TileStage2) <= 16, "Cassandra-2 stage fits");
static_assert(kWarps * scratch_warp<1>() >= kWarps * 256 * 4, "warp partials fit in the scratch");

// FAST: Cassandra-1, k = 64, m = 3, whole superblocks (per-lane cursors, lane_sb_tile).
// MODE 1: Cassandra-1, k = 64, m = 3 (lane_sb_tile); MODE 2: rows of whole
// superblocks, any k, m (runs_sb_tile, Cassandra-2: runs_sb_tile_c2);
// MODE 0: generic.
template <int VAR, int NT, int MODE>
__global__ void __launch_bounds__(kThreads, 4) verify_gemm_kernel(GemmArgs a) {
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
        } else if (MODE == 1) {
          uint32_t a0, a1;
          stream_range(w.sidx, s, w.lim_sexp, a0, a1);
          done = word_tile<true>(w.mask + gb0 * 4, w.ssm + gb0 * 8, w.vlo + gb0 * 8, w.vpr + gb0 * 16,
                                 w.sexp + a0, (int)(a1 - a0), w.vexp + v0, (int)(v1 - v0), s_lut,
                                 *reinterpret_cast<WordTileStage*>(wscr), tile + r * kTileStride, kBlkStride, lane);
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
  kern<<<g, kThreads, smem, st>>>(a);
  return launch_status();
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

extern "C" int cas_verify_gemm(const cas_weights* W, const uint16_t* X, int T, float* Y, void* stream) {
  int s = check_weights(W);
  if (s) return s;
  if (T < 1 || T > 16) return CAS_ERR_INVALID;
  if (W->N == 0) return CAS_OK;  // nothing to write (Y may be an empty tensor)
  if (!X || !Y || !aligned16(X) || !aligned16(Y)) return CAS_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(Y, 0, sizeof(float) * T * W->N, st) != cudaSuccess) return CAS_ERR_CUDA;
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
    if (fast) return launch<1, 1, 1>(a, st);
    if (whole) return v1 ? launch<1, 1, 2>(a, st) : launch<2, 1, 2>(a, st);
    return v1 ? launch<1, 1, 0>(a, st) : launch<2, 1, 0>(a, st);
  }
  if (fast) return launch<1, 2, 1>(a, st);
  if (whole) return v1 ? launch<1, 2, 2>(a, st) : launch<2, 2, 2>(a, st);
  return v1 ? launch<1, 2, 0>(a, st) : launch<2, 2, 0>(a, st);
}
