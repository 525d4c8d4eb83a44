// api.cu - status strings, argument checks and descriptor views of libcas.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "common.cuh"

extern "C" const char* cas_status_str(int s) {
  switch (s) {
    case CAS_OK: return "ok";
    case CAS_ERR_INVALID: return "invalid argument";
    case CAS_ERR_SHAPE: return "K (or head_dim) is not a multiple of 128";
    case CAS_ERR_NONFINITE: return "NaN or Inf in a tensor to encode";
    case CAS_ERR_CAPACITY: return "KV cache capacity exhausted";
    case CAS_ERR_CUDA: return "CUDA error";
    case CAS_ERR_BUFFER: return "buffer or workspace too small";
    case CAS_ERR_CORRUPT: return "encoded data inconsistent";
    case CAS_ERR_TIMEOUT: return "bounded device wait gave up";
    default: return "unknown status";
  }
}

extern "C" int32_t cas_keep_from_ratio(double r) {
  if (!(r >= 0.0)) return 0;
  if (r >= 1.0) return CAS_BLK;
  return (int32_t)std::floor(128.0 * r + 0.5);
}

namespace cas {
int gemv_wait_status(bool clear);
int set_first_wait_spins(uint32_t spins);
void set_launch_overlap(bool on);
}  // namespace cas

extern "C" int cas_test_first_wait_spins(uint32_t spins) {
  if (cudaDeviceSynchronize() != cudaSuccess) return CAS_ERR_CUDA;
  return cas::set_first_wait_spins(spins == 0xFFFFFFFFu ? cas::kSpinLimit : spins);
}

extern "C" int cas_set_launch_overlap(int on) {
  cas::set_launch_overlap(on != 0);
  return CAS_OK;
}

extern "C" int cas_device_status(void* stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CAS_ERR_CUDA;
  int s = cas::gemv_wait_status(true);
  const int c[3] = {cas::corrupt_status_gemv(true), cas::corrupt_status_gemm(true), cas::corrupt_status_decode(true)};
  for (int v : c)
    if (!s) s = v;
  return s;
}

namespace cas {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int sm_count() {
  static int cached = 0;
  if (!cached) {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached = n > 0 ? n : 1;
  }
  return cached;
}

int occupancy(const void* func, int threads, size_t smem) {
  struct Key {
    const void* f;
    int t;
    size_t s;
    bool operator==(const Key& o) const { return f == o.f && t == o.t && s == o.s; }
  };
  struct Hash {
    size_t operator()(const Key& k) const { return (size_t)k.f ^ ((size_t)k.t << 20) ^ (k.s << 1); }
  };
  static std::mutex mu;
  static std::unordered_map<Key, int, Hash> cache;
  static std::unordered_map<const void*, size_t> smem_set;
  std::lock_guard<std::mutex> g(mu);
  Key k{func, threads, smem};
  auto it = cache.find(k);
  if (it != cache.end()) return it->second;
  auto s = smem_set.find(func);
  if (smem > 48 * 1024 && (s == smem_set.end() || s->second < smem)) {
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    smem_set[func] = smem;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem) != cudaSuccess) n = 0;
  cache[k] = n;
  return n;
}

namespace {
std::atomic<int> g_launch_overlap{0};
}
bool launch_overlap() { return g_launch_overlap.load(std::memory_order_relaxed) != 0; }
void set_launch_overlap(bool on) { g_launch_overlap.store(on ? 1 : 0, std::memory_order_relaxed); }

int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CAS_OK : CAS_ERR_CUDA;
}

int check_weights(const cas_weights* W) {
  if (!W || !W->base) return CAS_ERR_INVALID;
  if (W->N < 0 || W->K < 0 || (W->K % CAS_BLK)) return CAS_ERR_SHAPE;
  if (W->p.variant != 1 && W->p.variant != 2) return CAS_ERR_INVALID;
  if (W->p.keep_per_block < 0 || W->p.keep_per_block > CAS_BLK) return CAS_ERR_INVALID;
  if (W->p.mant_bits < 0 || W->p.mant_bits > 7) return CAS_ERR_INVALID;
  return CAS_OK;
}

WView make_view(const cas_weights* W) {
  WView v{};
  const uint8_t* b = (const uint8_t*)W->base;
  auto w32 = [&](int s) { return (const uint32_t*)(b + W->off[s]); };
  v.mask = w32(CAS_SEC_MASK);
  v.ssm = w32(CAS_SEC_SPEC_SM);
  v.sexp = w32(CAS_SEC_SPEC_EXP);
  v.sidx = w32(CAS_SEC_SPEC_SBIDX);
  v.smx = b + W->off[CAS_SEC_SPEC_MX];
  v.sq = w32(CAS_SEC_SPEC_Q);
  v.vlo = w32(CAS_SEC_VER_LO);
  v.vd = w32(CAS_SEC_VER_D);
  v.vdidx = w32(CAS_SEC_VER_D_SBIDX);
  v.vres = w32(CAS_SEC_VER_RES);
  v.vresidx = w32(CAS_SEC_VER_RES_SBIDX);
  v.vpr = w32(CAS_SEC_VER_PR);
  v.vexp = w32(CAS_SEC_VER_EXP);
  v.vidx = w32(CAS_SEC_VER_SBIDX);
  v.N = W->N;
  v.K = W->K;
  v.nbr = (int)(W->K / CAS_BLK);
  v.nsr = (v.nbr + CAS_SB - 1) / CAS_SB;
  v.nsb = W->N * v.nsr;
  v.variant = W->p.variant;
  v.k = W->p.keep_per_block;
  v.m = W->p.mant_bits;
  v.rec_sm = rec_words(v.k, v.m + 1);
  v.rec_q = rec_words(v.k, v.m + 2);
  v.rec_lo = rec_words(v.k, 7 - v.m);
  v.rec_pr = rec_words(CAS_BLK - v.k, 8);
  auto words = [&](int sec) { return (uint32_t)std::min<uint64_t>(W->len[sec] / 4, 0xFFFFFFFFull); };
  v.lim_sexp = words(CAS_SEC_SPEC_EXP);
  v.lim_vexp = words(CAS_SEC_VER_EXP);
  v.lim_vd = words(CAS_SEC_VER_D);
  v.lim_vres = words(CAS_SEC_VER_RES);
  return v;
}

}  // namespace cas
