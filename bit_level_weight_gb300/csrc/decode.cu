// decode.cu - materialise the draft values or the original bits of an encoded
// tensor as bf16 [N][K] (test path of the speculation / verification split).
#include <cuda_runtime.h>

#include <algorithm>

#include "sbdecode.cuh"

namespace cas {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int VAR, bool FULL>
__global__ void __launch_bounds__(kThreads) decode_kernel(WView w, Lut lut, uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint8_t s_lut[256];
  __shared__ uint8_t s_code[kWarps][1024];
  __shared__ uint8_t s_vcode[kWarps][1024];
  __shared__ uint32_t s_res[kWarps][kResWords];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) s_lut[i] = lut.v[i];
  __syncthreads();
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  SbScratch sc{s_code[warp], s_vcode[warp], s_res[warp]};
  for (int64_t s = blockIdx.x * (int64_t)kWarps + warp; s < w.nsb; s += (int64_t)gridDim.x * kWarps) {
    SbInfo in = sb_prepare<VAR, FULL>(w, s, s_lut, sc, lane);
    if (lane < 4 * in.nb) {
      uint32_t v[16];
      sb_rebuild_word<VAR, FULL>(w, in, sc, lane, v);
      uint4* dst = reinterpret_cast<uint4*>(out + in.n * w.K + (int64_t)CAS_BLK * CAS_SB * in.j + 32 * lane);
      dst[0] = make_uint4(v[0], v[1], v[2], v[3]);
      dst[1] = make_uint4(v[4], v[5], v[6], v[7]);
      dst[2] = make_uint4(v[8], v[9], v[10], v[11]);
      dst[3] = make_uint4(v[12], v[13], v[14], v[15]);
    }
    __syncwarp();
  }
}

template <bool FULL>
int run_decode(const cas_weights* W, uint16_t* out, void* stream) {
  int s = check_weights(W);
  if (s) return s;
  WView v = make_view(W);
  if (v.nsb == 0) return CAS_OK;
  if (!out || !aligned16(out)) return CAS_ERR_INVALID;
  Lut lut;
  for (int i = 0; i < 256; ++i) lut.v[i] = W->exp_of_rank[i];
  int64_t g = std::min<int64_t>((v.nsb + kWarps - 1) / kWarps, (int64_t)sm_count() * 8);
  cudaStream_t st = (cudaStream_t)stream;
  return v.variant == 1 ? launch_k(decode_kernel<1, FULL>, (int)g, kThreads, 0, st, v, lut, out)
                        : launch_k(decode_kernel<2, FULL>, (int)g, kThreads, 0, st, v, lut, out);
}

}  // namespace

int corrupt_status_decode(bool clear) {
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

extern "C" int cas_decode_draft(const cas_weights* W, uint16_t* out, void* stream) {
  return cas::run_decode<false>(W, out, stream);
}
extern "C" int cas_reconstruct(const cas_weights* W, uint16_t* out, void* stream) {
  return cas::run_decode<true>(W, out, stream);
}
