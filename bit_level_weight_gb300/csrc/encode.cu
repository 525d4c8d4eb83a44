// encode.cu - offline weight encoding: exponent histogram, rank table,
// per-superblock stream lengths, exclusive scan, section writer.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "blockenc.cuh"

namespace cas {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Workspace layout (byte offsets), sized for nsb superblocks.
struct WsLayout {
  uint64_t counts, roe, totals, lens, idx, bytes;
};
WsLayout ws_layout(int64_t nsb) {
  WsLayout L;
  uint64_t o = 0;
  L.counts = o; o += 256 * 8;                      // u64 histogram
  L.roe = o; o += 256;                             // rank_of_exp
  L.totals = o; o += 4 * 8;                        // u64 stream totals (words)
  L.lens = o; o += 4 * (uint64_t)(nsb + 1) * 4;    // u32 words per superblock, 4 streams
  o = (o + 255) & ~255ull;
  L.idx = o; o += 4 * (uint64_t)(nsb + 1) * 4;     // u32 exclusive scans
  L.bytes = (o + 255) & ~255ull;
  return L;
}

// 256-bin histogram of the biased exponent (8 values per thread per step).
__global__ void hist_kernel(const uint16_t* __restrict__ W, int64_t n, unsigned long long* counts) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned int h[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
  __syncthreads();
  int64_t n8 = n / 8;
  const uint4* W4 = reinterpret_cast<const uint4*>(W);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    uint4 r = __ldg(W4 + i);
    uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      atomicAdd(&h[(w[j] >> 7) & 0xFF], 1u);
      atomicAdd(&h[(w[j] >> 23) & 0xFF], 1u);
    }
  }
  for (int64_t i = n8 * 8 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    atomicAdd(&h[(W[i] >> 7) & 0xFF], 1u);
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (h[i]) atomicAdd(counts + i, (unsigned long long)h[i]);
}

// Pass 1: words of each variable-length stream of every superblock.
template <int VAR>
__global__ void __launch_bounds__(kThreads) lengths_kernel(const uint16_t* __restrict__ W, int64_t K, int nbr,
                                                          int nsr, int64_t nsb, int k, int m,
                                                          const uint8_t* __restrict__ roe_g, uint32_t* lens,
                                                          int64_t stride) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint8_t roe[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) roe[i] = roe_g[i];
  __syncthreads();
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t s = blockIdx.x * (int64_t)kWarps + warp; s < nsb; s += (int64_t)gridDim.x * kWarps) {
    int64_t n = s / nsr;
    int j = (int)(s % nsr);
    int b1 = min(nbr, 8 * j + 8);
    int a_s = 0, a_v = 0, a_d = 0, a_r = 0;
    for (int b = 8 * j; b < b1; ++b) {
      uint32_t v[4];
      load_block4(W + n * K + (int64_t)b * CAS_BLK, lane, v);
      uint32_t key[4] = {v[0] & 0x7FFFu, v[1] & 0x7FFFu, v[2] & 0x7FFFu, v[3] & 0x7FFFu};
      uint32_t kept = select_block4(key, k, lane);
      int E = VAR == 2 ? group_shared_exp(v, kept) : 0;
      BlockBits lb = block_lane_bits<VAR>(v, kept, E, m, roe);
      a_s += lb.sexp;
      a_v += lb.vexp;
      a_d += lb.vd;
      a_r += lb.vres;
    }
    a_s = warp_sum(a_s);
    a_v = warp_sum(a_v);
    a_d = warp_sum(a_d);
    a_r = warp_sum(a_r);
    if (lane == 0) {
      lens[0 * stride + s] = (uint32_t)((a_s + 31) / 32);
      lens[1 * stride + s] = (uint32_t)((a_v + 31) / 32);
      lens[2 * stride + s] = (uint32_t)((a_d + 31) / 32);
      lens[3 * stride + s] = (uint32_t)((a_r + 31) / 32);
    }
  }
}

// Exclusive scan of up to 4 arrays of n words (one CTA per array). out[n]
// receives the total; totals[i] as well (u64, to detect 32-bit overflow).
struct ScanArgs {
  const uint32_t* in[4];
  uint32_t* out[4];
  unsigned long long* totals;
  int64_t n;
};
__global__ void __launch_bounds__(1024) scan_kernel(ScanArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned long long sh[1024];
  int which = blockIdx.x;
  const uint32_t* in = a.in[which];
  uint32_t* out = a.out[which];
  if (!in) return;
  int64_t n = a.n;
  int T = blockDim.x, tid = threadIdx.x;
  int64_t per = (n + T - 1) / T;
  int64_t s0 = tid * per, s1 = min(n, s0 + per);
  unsigned long long sum = 0;
  for (int64_t i = s0; i < s1; ++i) sum += in[i];
  sh[tid] = sum;
  __syncthreads();
  for (int d = 1; d < T; d <<= 1) {
    unsigned long long t = tid >= d ? sh[tid - d] : 0ull;
    __syncthreads();
    sh[tid] += t;
    __syncthreads();
  }
  unsigned long long run = sh[tid] - sum;
  if (out)
    for (int64_t i = s0; i < s1; ++i) {
      out[i] = (uint32_t)run;
      run += in[i];
    }
  if (tid == T - 1) {
    if (out) out[n] = (uint32_t)sh[tid];
    a.totals[which] = sh[tid];
  }
}

struct WriteArgs {
  const uint16_t* W;
  int64_t K, nsb;
  int nbr, nsr, k, m;
  int rec_s, rec_lo, rec_pr;
  const uint8_t* roe;
  uint32_t* mask;
  uint32_t* rec_s_base;
  uint32_t* rec_lo_base;
  uint32_t* rec_pr_base;
  uint8_t* mx;
  uint32_t* sexp;
  const uint32_t* sidx;
  uint64_t sexp_words;
  uint32_t* vexp;
  const uint32_t* vidx;
  uint64_t vexp_words;
  uint32_t* vd;
  const uint32_t* vdidx;
  uint64_t vd_words;
  uint32_t* vres;
  const uint32_t* vresidx;
  uint64_t vres_words;
};

// Pass 2: one warp per superblock writes every section.
template <int VAR>
__global__ void __launch_bounds__(kThreads) write_kernel(WriteArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint8_t roe[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) roe[i] = a.roe[i];
  __syncthreads();
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t s = blockIdx.x * (int64_t)kWarps + warp; s < a.nsb; s += (int64_t)gridDim.x * kWarps) {
    int64_t n = s / a.nsr;
    int j = (int)(s % a.nsr);
    int b1 = min(a.nbr, 8 * j + 8);
    Stream sexp{a.sexp, VAR == 1 ? (uint64_t)a.sidx[s] * 32 : 0, a.sexp_words};
    Stream vexp{a.vexp, (uint64_t)a.vidx[s] * 32, a.vexp_words};
    Stream vd{a.vd, VAR == 2 ? (uint64_t)a.vdidx[s] * 32 : 0, a.vd_words};
    Stream vres{a.vres, VAR == 2 ? (uint64_t)a.vresidx[s] * 32 : 0, a.vres_words};
    for (int b = 8 * j; b < b1; ++b) {
      int64_t gb = n * a.nbr + b;
      uint32_t v[4];
      load_block4(a.W + n * a.K + (int64_t)b * CAS_BLK, lane, v);
      BlockDst dst;
      dst.mask = a.mask + gb * 4;
      dst.rec_s = a.rec_s_base + gb * a.rec_s;
      dst.rec_lo = a.rec_lo_base + gb * a.rec_lo;
      dst.rec_pr = a.rec_pr_base + gb * a.rec_pr;
      dst.mx = a.mx + gb * 4;
      encode_block<VAR>(v, a.k, a.m, roe, dst, sexp, vexp, vd, vres, lane, ~0ull);
    }
  }
}

int grid_for(int64_t units, int per_cta) {
  int64_t g = (units + per_cta - 1) / per_cta;
  int64_t cap = (int64_t)sm_count() * 8;
  return (int)std::max<int64_t>(1, std::min(g, cap));
}

bool params_ok(const cas_params& p) {
  return (p.variant == 1 || p.variant == 2) && p.keep_per_block >= 0 && p.keep_per_block <= CAS_BLK &&
         p.mant_bits >= 0 && p.mant_bits <= 7;
}

// lengths + scan into `idx_out` pointers (4 arrays of nsb+1 words or null).
int run_lengths_scan(const uint16_t* W, const cas_weights* d, uint8_t* ws, const WsLayout& L,
                     uint32_t* const idx_out[4], cudaStream_t st) {
  int nbr = (int)(d->K / CAS_BLK), nsr = (nbr + 7) / 8;
  int64_t nsb = d->N * nsr;
  if (nsb == 0) return CAS_OK;
  uint32_t* lens = (uint32_t*)(ws + L.lens);
  int g = grid_for(nsb, kWarps);
  {
    const int e_ = d->p.variant == 1 ? launch_plain(lengths_kernel<1>, g, kThreads, 0, st, W, d->K, nbr, nsr, nsb,
                                                    d->p.keep_per_block, d->p.mant_bits, ws + L.roe, lens, nsb + 1)
                                     : launch_plain(lengths_kernel<2>, g, kThreads, 0, st, W, d->K, nbr, nsr, nsb,
                                                    d->p.keep_per_block, d->p.mant_bits, ws + L.roe, lens, nsb + 1);
    if (e_) return e_;
  }
  ScanArgs sa{};
  for (int i = 0; i < 4; ++i) {
    sa.in[i] = lens + i * (nsb + 1);
    sa.out[i] = idx_out[i];
  }
  sa.totals = (unsigned long long*)(ws + L.totals);
  sa.n = nsb;
  return launch_plain(scan_kernel, 4, 1024, 0, st, sa);
}

void fill_sections(cas_weights* d, const uint64_t words[4]) {
  int64_t nbr = d->K / CAS_BLK, nsr = (nbr + 7) / 8, nblk = d->N * nbr, nsb = d->N * nsr;
  int k = d->p.keep_per_block, m = d->p.mant_bits;
  uint64_t* len = d->len;
  for (int i = 0; i < CAS_NSECT; ++i) len[i] = 0;
  uint64_t nb = (uint64_t)nblk, nsbi = (uint64_t)nsb + 1;
  len[CAS_SEC_MASK] = nb * 16;
  len[CAS_SEC_VER_PR] = nb * rec_words(CAS_BLK - k, 8) * 4;
  len[CAS_SEC_VER_EXP] = words[1] * 4;
  len[CAS_SEC_VER_SBIDX] = nsbi * 4;
  if (d->p.variant == 1) {
    len[CAS_SEC_SPEC_SM] = nb * rec_words(k, m + 1) * 4;
    len[CAS_SEC_SPEC_EXP] = words[0] * 4;
    len[CAS_SEC_SPEC_SBIDX] = nsbi * 4;
    len[CAS_SEC_VER_LO] = nb * rec_words(k, 7 - m) * 4;
  } else {
    len[CAS_SEC_SPEC_MX] = nb * 4;
    len[CAS_SEC_SPEC_Q] = nb * rec_words(k, m + 2) * 4;
    len[CAS_SEC_VER_D] = words[2] * 4;
    len[CAS_SEC_VER_D_SBIDX] = nsbi * 4;
    len[CAS_SEC_VER_RES] = words[3] * 4;
    len[CAS_SEC_VER_RES_SBIDX] = nsbi * 4;
  }
  uint64_t run = 0;
  for (int i = 0; i < CAS_NSECT; ++i) {
    d->off[i] = (run + 255) & ~255ull;
    run = d->off[i] + len[i];
  }
  d->bytes = (run + 255) & ~255ull;
}

}  // namespace
}  // namespace cas

using namespace cas;

extern "C" uint64_t cas_encode_workspace_bytes(int64_t N, int64_t K) {
  if (N < 0 || K < 0) return 0;
  int64_t nsr = (K / CAS_BLK + 7) / 8;
  return ws_layout(N * nsr).bytes;
}

extern "C" int cas_encode_weights_plan(const uint16_t* W, int64_t N, int64_t K, cas_params p, cas_weights* d,
                                       uint64_t* bytes_needed, void* workspace, uint64_t workspace_bytes,
                                       void* stream) {
  if (!d || !bytes_needed || N < 0 || K < 0 || !params_ok(p)) return CAS_ERR_INVALID;
  if (K % CAS_BLK) return CAS_ERR_SHAPE;
  if (N * K > 0 && (!W || !aligned16(W))) return CAS_ERR_INVALID;
  int64_t nsr = (K / CAS_BLK + 7) / 8, nsb = N * nsr;
  WsLayout L = ws_layout(nsb);
  if (!workspace || workspace_bytes < L.bytes || !aligned16(workspace)) return CAS_ERR_BUFFER;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  std::memset(d, 0, sizeof(*d));
  d->N = N;
  d->K = K;
  d->p = p;

  std::vector<unsigned long long> counts(256, 0);
  if (cudaMemsetAsync(ws + L.counts, 0, 256 * 8, st) != cudaSuccess) return CAS_ERR_CUDA;
  if (N * K > 0) {
    if (const int e_ = launch_plain(hist_kernel, sm_count() * 4, 256, 0, st, W, N * K,
                                    (unsigned long long*)(ws + L.counts)))
      return e_;
  }
  if (cudaMemcpyAsync(counts.data(), ws + L.counts, 256 * 8, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return CAS_ERR_CUDA;
  if (counts[255]) return CAS_ERR_NONFINITE;
  // rank table: exponents by (count desc, exponent asc)
  std::vector<int> order(256);
  for (int e = 0; e < 256; ++e) order[e] = e;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return counts[a] > counts[b]; });
  for (int r = 0; r < 256; ++r) {
    d->exp_of_rank[r] = (uint8_t)order[r];
    d->rank_of_exp[order[r]] = (uint8_t)r;
  }
  uint64_t words[4] = {0, 0, 0, 0};
  if (nsb > 0) {
    if (cudaMemcpyAsync(ws + L.roe, d->rank_of_exp, 256, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return CAS_ERR_CUDA;
    uint32_t* idx_out[4] = {nullptr, nullptr, nullptr, nullptr};
    int s = run_lengths_scan(W, d, ws, L, idx_out, st);
    if (s) return s;
    unsigned long long tot[4];
    if (cudaMemcpyAsync(tot, ws + L.totals, sizeof(tot), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return CAS_ERR_CUDA;
    for (int i = 0; i < 4; ++i) {
      if (tot[i] > 0xFFFFFFFFull) return CAS_ERR_INVALID;
      words[i] = tot[i];
    }
  }
  fill_sections(d, words);
  *bytes_needed = d->bytes;
  return CAS_OK;
}

extern "C" int cas_encode_weights(const uint16_t* W, cas_weights* d, void* buf, uint64_t buf_bytes, void* workspace,
                                  uint64_t workspace_bytes, void* stream) {
  if (!d || !buf || ((uintptr_t)buf & 255u) || d->N < 0 || d->K < 0 || !params_ok(d->p)) return CAS_ERR_INVALID;
  if (d->K % CAS_BLK) return CAS_ERR_SHAPE;
  if (d->N * d->K > 0 && (!W || !aligned16(W))) return CAS_ERR_INVALID;
  if (buf_bytes < d->bytes) return CAS_ERR_BUFFER;
  int nbr = (int)(d->K / CAS_BLK), nsr = (nbr + 7) / 8;
  int64_t nsb = d->N * nsr;
  WsLayout L = ws_layout(nsb);
  if (!workspace || workspace_bytes < L.bytes || !aligned16(workspace)) return CAS_ERR_BUFFER;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  uint8_t* b = (uint8_t*)buf;
  if (cudaMemsetAsync(buf, 0, d->bytes, st) != cudaSuccess) return CAS_ERR_CUDA;
  d->base = buf;
  if (nsb == 0) return CAS_OK;
  if (cudaMemcpyAsync(ws + L.roe, d->rank_of_exp, 256, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return CAS_ERR_CUDA;
  auto sec = [&](int i) { return (uint32_t*)(b + d->off[i]); };
  bool v1 = d->p.variant == 1;
  uint32_t* idx_out[4] = {v1 ? sec(CAS_SEC_SPEC_SBIDX) : nullptr, sec(CAS_SEC_VER_SBIDX),
                          v1 ? nullptr : sec(CAS_SEC_VER_D_SBIDX), v1 ? nullptr : sec(CAS_SEC_VER_RES_SBIDX)};
  int s = run_lengths_scan(W, d, ws, L, idx_out, st);
  if (s) return s;
  WriteArgs a{};
  a.W = W;
  a.K = d->K;
  a.nsb = nsb;
  a.nbr = nbr;
  a.nsr = nsr;
  a.k = d->p.keep_per_block;
  a.m = d->p.mant_bits;
  a.rec_s = v1 ? rec_words(a.k, a.m + 1) : rec_words(a.k, a.m + 2);
  a.rec_lo = rec_words(a.k, 7 - a.m);
  a.rec_pr = rec_words(CAS_BLK - a.k, 8);
  a.roe = ws + L.roe;
  a.mask = sec(CAS_SEC_MASK);
  a.rec_s_base = v1 ? sec(CAS_SEC_SPEC_SM) : sec(CAS_SEC_SPEC_Q);
  a.rec_lo_base = sec(CAS_SEC_VER_LO);
  a.rec_pr_base = sec(CAS_SEC_VER_PR);
  a.mx = b + d->off[CAS_SEC_SPEC_MX];
  a.sexp = sec(CAS_SEC_SPEC_EXP);
  a.sidx = sec(CAS_SEC_SPEC_SBIDX);
  a.sexp_words = d->len[CAS_SEC_SPEC_EXP] / 4;
  a.vexp = sec(CAS_SEC_VER_EXP);
  a.vidx = sec(CAS_SEC_VER_SBIDX);
  a.vexp_words = d->len[CAS_SEC_VER_EXP] / 4;
  a.vd = sec(CAS_SEC_VER_D);
  a.vdidx = sec(CAS_SEC_VER_D_SBIDX);
  a.vd_words = d->len[CAS_SEC_VER_D] / 4;
  a.vres = sec(CAS_SEC_VER_RES);
  a.vresidx = sec(CAS_SEC_VER_RES_SBIDX);
  a.vres_words = d->len[CAS_SEC_VER_RES] / 4;
  int g = grid_for(nsb, kWarps);
  return v1 ? launch_plain(write_kernel<1>, g, kThreads, 0, st, a) : launch_plain(write_kernel<2>, g, kThreads, 0, st, a);
}

extern "C" int cas_choose_variant(const uint16_t* W, int64_t N, int64_t K, int keep_per_block, int mant_bits,
                                  void* workspace, uint64_t workspace_bytes, int* variant, uint64_t* spec_bytes,
                                  void* stream) {
  if (!variant) return CAS_ERR_INVALID;
  uint64_t sb[2] = {0, 0};
  for (int v = 1; v <= 2; ++v) {
    cas_weights d;
    uint64_t need = 0;
    const cas_params p{v, keep_per_block, mant_bits};
    const int s = cas_encode_weights_plan(W, N, K, p, &d, &need, workspace, workspace_bytes, stream);
    if (s) return s;
    for (int sec : {CAS_SEC_MASK, CAS_SEC_SPEC_SM, CAS_SEC_SPEC_EXP, CAS_SEC_SPEC_SBIDX, CAS_SEC_SPEC_MX,
                    CAS_SEC_SPEC_Q})
      sb[v - 1] += d.len[sec];
  }
  *variant = sb[1] < sb[0] ? 2 : 1;
  if (spec_bytes) {
    spec_bytes[0] = sb[0];
    spec_bytes[1] = sb[1];
  }
  return CAS_OK;
}
