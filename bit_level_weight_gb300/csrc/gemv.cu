// gemv.cu - fused draft decode + GEMV: y[v][n] = sum_k D(W)[n][k] x[v][k].
//
// Reads only the speculation sections (mask, sign/mantissa records, unary
// exponent stream and its superblock index; Cassandra-2: shared exponents and
// q records). The draft does full-size FLOPs and saves bandwidth (Cassandra
// blog review, section 3.1), so the kernel is bound by the HBM read of the
// speculation stream and by the integer work of decoding it.
//
// Mapping: one warp per superblock (row n, 8 blocks); lane L owns mask word L,
// i.e. 32 positions of block L>>2. The lane walks only its kept positions:
// the sign/mantissa field comes from the block record, the exponent from the
// superblock's unary codes decoded into shared memory, x from shared memory
// (staged once per CTA by a TMA bulk copy). Partial sums go to y with one
// fp32 atomic per (superblock, vector); y is cleared first.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"

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
};

// Set when a bounded wait on the x staging copy gave up (read by
// cas_device_status).
__device__ int g_gemv_wait_status = 0;

template <int VAR, int NV>
__global__ void __launch_bounds__(kThreads) draft_gemv_kernel(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const WView& w = a.w;
  const int K = (int)w.K;
  const int xbytes = NV * K * 2;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + xbytes);
  uint8_t* s_lut = smem + xbytes + 16;
  uint8_t* s_code = s_lut + 256 + (threadIdx.x >> 5) * 1024;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_tx(bar, (uint32_t)xbytes);
    bulk_g2s(xs, a.x, (uint32_t)xbytes, bar);
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) s_lut[i] = a.lut.v[i];
  bool ok = mbar_wait_bounded(bar, 0);
  if (!__syncthreads_and(ok)) {
    if (threadIdx.x == 0) atomicExch(&g_gemv_wait_status, CAS_ERR_TIMEOUT);
    mbar_wait_bounded(bar, 0);  // let an in-flight copy land before the CTA exits
    return;
  }

  const int k = w.k, m = w.m;
  for (int64_t s = blockIdx.x * (int64_t)kWarps + warp; s < w.nsb; s += (int64_t)gridDim.x * kWarps) {
    int64_t n = s / w.nsr;
    int j = (int)(s % w.nsr);
    int nb = min(CAS_SB, w.nbr - CAS_SB * j);
    int64_t gb0 = n * w.nbr + CAS_SB * j;
    uint32_t mw = lane < 4 * nb ? __ldg(w.mask + gb0 * 4 + lane) : 0u;
    int cnt = __popc(mw);
    int o = warp_incl_add(cnt, lane) - cnt;
    if (VAR == 1) {
      uint32_t b0 = __ldg(w.sidx + s), b1 = __ldg(w.sidx + s + 1);
      warp_decode_unary(w.sexp + b0, (int)(b1 - b0), s_lut, s_code, nb * k, lane);
      __syncwarp();
    }
    float acc[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[v] = 0.f;
    if (mw) {
      int blk = lane >> 2, g = lane & 3;
      int64_t gb = gb0 + blk;
      int t = o - k * blk;
      const uint16_t* xr = xs + CAS_BLK * CAS_SB * j + CAS_BLK * blk + 32 * g;
      if (VAR == 1) {
        const uint32_t* rs = w.ssm + gb * w.rec_sm;
        const uint32_t fmask = (1u << m) - 1u;
        while (mw) {
          int p = __ffs(mw) - 1;
          mw &= mw - 1;
          uint32_t fld = get_field(rs, t * (m + 1), m + 1);
          uint32_t bits = ((fld >> m) << 31) | ((uint32_t)s_code[o] << 23) | ((fld & fmask) << (23 - m));
          float val = __uint_as_float(bits);
#pragma unroll
          for (int v = 0; v < NV; ++v) acc[v] = fmaf(val, bf2f(xr[v * K + p]), acc[v]);
          ++t;
          ++o;
        }
      } else {
        const uint32_t* rs = w.sq + gb * w.rec_q;
        float scale = pow2_biased(max((int)__ldg(w.smx + gb * 4 + g), 1) - m);
        const uint32_t qmask = (1u << (m + 1)) - 1u;
        while (mw) {
          int p = __ffs(mw) - 1;
          mw &= mw - 1;
          uint32_t fld = get_field(rs, t * (m + 2), m + 2);
          float val = (float)(fld & qmask) * scale;
          val = (fld >> (m + 1)) & 1u ? -val : val;
#pragma unroll
          for (int v = 0; v < NV; ++v) acc[v] = fmaf(val, bf2f(xr[v * K + p]), acc[v]);
          ++t;
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

template <int VAR, int NV>
int launch(const GemvArgs& a, cudaStream_t st) {
  size_t smem = (size_t)NV * a.w.K * 2 + 16 + 256 + kWarps * 1024;
  auto kern = draft_gemv_kernel<VAR, NV>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return CAS_ERR_CUDA;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  per_sm = std::max(per_sm, 1);
  int64_t need = (a.w.nsb + kWarps - 1) / kWarps;
  int g = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sm_count() * per_sm));
  kern<<<g, kThreads, smem, st>>>(a);
  return launch_status();
}

template <int VAR>
int dispatch(const GemvArgs& a, int nvec, cudaStream_t st) {
  switch (nvec) {
    case 1: return launch<VAR, 1>(a, st);
    case 2: return launch<VAR, 2>(a, st);
    case 3: return launch<VAR, 3>(a, st);
    default: return launch<VAR, 4>(a, st);
  }
}

}  // namespace

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

extern "C" int cas_draft_gemv(const cas_weights* W, const uint16_t* x, int nvec, float* y, void* stream) {
  int s = check_weights(W);
  if (s) return s;
  if (nvec < 1 || nvec > kMaxVec) return CAS_ERR_INVALID;
  if ((int64_t)nvec * W->K * 2 > 200 * 1024) return CAS_ERR_INVALID;  // x must fit in shared memory
  if (W->N == 0) return CAS_OK;  // nothing to write (y may be an empty tensor)
  if (!x || !y || !aligned16(x) || !aligned16(y)) return CAS_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(y, 0, sizeof(float) * nvec * W->N, st) != cudaSuccess) return CAS_ERR_CUDA;
  if (W->K == 0) return CAS_OK;
  GemvArgs a;
  a.w = make_view(W);
  for (int i = 0; i < 256; ++i) a.lut.v[i] = W->exp_of_rank[i];
  a.x = x;
  a.y = y;
  return W->p.variant == 1 ? dispatch<1>(a, nvec, st) : dispatch<2>(a, nvec, st);
}
