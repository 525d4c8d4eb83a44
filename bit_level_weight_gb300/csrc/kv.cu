// kv.cu - compressed KV cache: layout, calibration (rank tables), online
// append (Cassandra blog review, section 3.3: the KV cache is produced during
// inference and encoded online), truncation (rejected draft tokens) and the
// device status.
//
// Append runs two kernels with one CTA per (head, K|V) stream: the first
// computes every new token's code lengths and checks capacity and finiteness
// (a failure sets a per-call flag and the sticky status); the second, unless
// the flag is set, clears the stream words it will fill and encodes the tokens
// (one warp per token). The CTA that finishes last advances n_tokens and
// resets the per-call counters. No CTA waits on another.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "blockenc.cuh"
#include "kvview.cuh"

namespace cas {

KvDev make_kv_dev(const cas_kv* kv) {
  KvDev d{};
  d.base = (uint8_t*)kv->base;
  for (int i = 0; i < CAS_KV_NSECT; ++i) {
    d.off[i] = kv->off[i];
    d.stride[i] = kv->stride[i];
  }
  d.H = kv->n_kv_heads;
  d.k = kv->p.keep_per_block;
  d.m = kv->p.mant_bits;
  d.rec_sm = rec_words(d.k, d.m + 1);
  d.rec_lo = rec_words(d.k, 7 - d.m);
  d.rec_pr = rec_words(CAS_BLK - d.k, 8);
  d.max_tokens = kv->max_tokens;
  d.cap_spec = kv->cap_spec_words;
  d.cap_ver = kv->cap_ver_words;
  return d;
}

int check_kv(const cas_kv* kv) {
  if (!kv || !kv->base || kv->n_kv_heads < 1 || kv->head_dim != CAS_BLK || kv->p.variant != 1 ||
      kv->p.keep_per_block < 0 || kv->p.keep_per_block > CAS_BLK || kv->p.mant_bits < 0 || kv->p.mant_bits > 7)
    return CAS_ERR_INVALID;
  return CAS_OK;
}

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 256;  // tokens whose starts are computed per round

uint64_t a256(uint64_t x) { return (x + 255) & ~255ull; }

struct KvLayout {
  uint64_t off[16], stride[16], bytes, cap_spec, cap_ver;
};

bool kv_layout(int H, int64_t Tm, cas_params p, double est, KvLayout* L) {
  if (H < 1 || Tm < 1 || p.variant != 1 || p.keep_per_block < 0 || p.keep_per_block > CAS_BLK || p.mant_bits < 0 ||
      p.mant_bits > 7 || !(est > 0.0) || est > 256.0)
    return false;
  int k = p.keep_per_block, m = p.mant_bits;
  uint64_t S = 2ull * H, nsbm = (uint64_t)(Tm + 7) / 8;
  L->cap_spec = (uint64_t)std::ceil((double)Tm * k * est / 32.0) + nsbm + 2;
  L->cap_ver = (uint64_t)std::ceil((double)Tm * (CAS_BLK - k) * est / 32.0) + nsbm + 2;
  std::memset(L->off, 0, sizeof(L->off));
  std::memset(L->stride, 0, sizeof(L->stride));
  uint64_t state_bytes = 32 + 16 * S;
  L->stride[CAS_KV_TABLES] = 512;
  L->stride[CAS_KV_MASK] = a256((uint64_t)Tm * 16);
  L->stride[CAS_KV_SPEC_SM] = a256((uint64_t)Tm * rec_words(k, m + 1) * 4);
  L->stride[CAS_KV_SPEC_EXP] = a256(L->cap_spec * 4);
  L->stride[CAS_KV_SPEC_SBIDX] = a256((nsbm + 1) * 4);
  L->stride[CAS_KV_VER_LO] = a256((uint64_t)Tm * rec_words(k, 7 - m) * 4);
  L->stride[CAS_KV_VER_PR] = a256((uint64_t)Tm * rec_words(CAS_BLK - k, 8) * 4);
  L->stride[CAS_KV_VER_EXP] = a256(L->cap_ver * 4);
  L->stride[CAS_KV_VER_SBIDX] = a256((nsbm + 1) * 4);
  uint64_t run = 0;
  for (int i = 0; i < CAS_KV_NSECT; ++i) {
    L->off[i] = a256(run);
    run = L->off[i] + (i == CAS_KV_STATE ? state_bytes : L->stride[i] * S);
  }
  L->bytes = a256(run);
  return true;
}

// Exponent histogram of each stream's calibration tokens (u32 counts).
__global__ void kv_hist_kernel(const uint16_t* __restrict__ ck, const uint16_t* __restrict__ cv, int64_t n, int H,
                               unsigned int* hist) {
  __shared__ unsigned int h[256];
  int st = blockIdx.y;
  const uint16_t* src = st < H ? ck : cv;
  int head = st % H;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
  __syncthreads();
  int64_t total = n * CAS_BLK;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    int64_t t = i / CAS_BLK, d = i % CAS_BLK;
    atomicAdd(&h[(src[(t * H + head) * CAS_BLK + d] >> 7) & 0xFF], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (h[i]) atomicAdd(hist + st * 256 + i, h[i]);
}

// Code bits of one token block (warp): spec = kept codes, ver = pruned codes.
// Also reports whether any value is NaN/Inf.
__device__ __forceinline__ void token_bits(const uint16_t* blk, int k, const uint8_t* roe, int lane, int* bs, int* bv,
                                           bool* nonfinite) {
  uint32_t v[4];
  load_block4(blk, lane, v);
  uint32_t key[4] = {v[0] & 0x7FFFu, v[1] & 0x7FFFu, v[2] & 0x7FFFu, v[3] & 0x7FFFu};
  uint32_t kept = select_block4(key, k, lane);
  int s = 0, u = 0;
  bool nf = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int e = (v[j] >> 7) & 0xFF;
    nf |= e == 255;
    if ((kept >> j) & 1) s += roe[e] + 1;
    else u += roe[e] + 1;
  }
  *bs = warp_sum(s);
  *bv = warp_sum(u);
  *nonfinite = __any_sync(CAS_FULL, nf);
}

struct AppendArgs {
  KvDev d;
  const uint16_t* knew;
  const uint16_t* vnew;
  int T;
};

// Shared per-round state of the append kernels.
struct RoundSmem {
  int bits_s[kChunk], bits_v[kChunk];
  uint64_t start_s[kChunk], start_v[kChunk];
  int nonfinite;
};

// Computes the starts of tokens [r0, r0+cnt) given the cursors before them;
// returns updated cursors in cur_s / cur_v (thread 0 only). Token t starting
// a superblock aligns its streams to a word and records the superblock index.
__device__ void round_starts(RoundSmem& sm, int64_t t0, int cnt, uint64_t* cur_s, uint64_t* cur_v, uint32_t* sidx,
                             uint32_t* vidx, bool write_idx) {
  uint64_t cs = *cur_s, cv = *cur_v;
  for (int i = 0; i < cnt; ++i) {
    int64_t t = t0 + i;
    if ((t & 7) == 0) {
      cs = (cs + 31) & ~31ull;
      cv = (cv + 31) & ~31ull;
      if (write_idx) {
        sidx[t >> 3] = (uint32_t)(cs >> 5);
        vidx[t >> 3] = (uint32_t)(cv >> 5);
      }
    }
    sm.start_s[i] = cs;
    sm.start_v[i] = cv;
    cs += sm.bits_s[i];
    cv += sm.bits_v[i];
  }
  *cur_s = cs;
  *cur_v = cv;
}

template <bool WRITE>
__global__ void __launch_bounds__(kThreads) kv_append_kernel(AppendArgs a) {
  __shared__ RoundSmem sm;
  __shared__ uint8_t roe[256];
  __shared__ uint64_t cur_s, cur_v;
  __shared__ int skip;
  const KvDev& d = a.d;
  const int st = blockIdx.x, H = d.H, head = st % H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  KvState* S = kv_state(d);
  const uint16_t* src = st < H ? a.knew : a.vnew;
  for (int i = threadIdx.x; i < 256; i += kThreads) roe[i] = kv_rank_of_exp(d, st)[i];
  const int64_t n0 = *(volatile int64_t*)&S->n_tokens;
  if (threadIdx.x == 0) {
    cur_s = kv_tail_spec(d)[st];
    cur_v = kv_tail_ver(d)[st];
    sm.nonfinite = 0;
    skip = WRITE ? *(volatile int32_t*)&S->call_fail : 0;
  }
  __syncthreads();
  uint32_t* sidx = (uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, st);
  uint32_t* vidx = (uint32_t*)kv_sec(d, CAS_KV_VER_SBIDX, st);
  bool fail = !WRITE && n0 + a.T > d.max_tokens;
  if (!skip && !fail) {
    for (int r0 = 0; r0 < a.T; r0 += kChunk) {
      int cnt = min(kChunk, a.T - r0);
      for (int i = warp; i < cnt; i += kWarps) {
        int bs, bv;
        bool nf;
        token_bits(src + ((int64_t)(r0 + i) * H + head) * CAS_BLK, d.k, roe, lane, &bs, &bv, &nf);
        if (lane == 0) {
          sm.bits_s[i] = bs;
          sm.bits_v[i] = bv;
          if (nf) sm.nonfinite = 1;
        }
      }
      __syncthreads();
      uint64_t before_s = cur_s, before_v = cur_v;
      __syncthreads();
      if (threadIdx.x == 0) {
        uint64_t cs = cur_s, cv = cur_v;
        round_starts(sm, n0 + r0, cnt, &cs, &cv, sidx, vidx, WRITE);
        cur_s = cs;
        cur_v = cv;
      }
      __syncthreads();
      if (WRITE) {
        // clear [before, end) of both streams: partial first word keeps its old bits
        uint32_t* ws = (uint32_t*)kv_sec(d, CAS_KV_SPEC_EXP, st);
        uint32_t* wv = (uint32_t*)kv_sec(d, CAS_KV_VER_EXP, st);
        uint64_t e_s = (cur_s + 31) >> 5, e_v = (cur_v + 31) >> 5;
        for (uint64_t i = (before_s >> 5) + threadIdx.x; i < e_s; i += kThreads) {
          uint32_t keep = (i == (before_s >> 5) && (before_s & 31)) ? ~(0xFFFFFFFFu >> (before_s & 31)) : 0u;
          if (i < d.cap_spec) ws[i] &= keep;
        }
        for (uint64_t i = (before_v >> 5) + threadIdx.x; i < e_v; i += kThreads) {
          uint32_t keep = (i == (before_v >> 5) && (before_v & 31)) ? ~(0xFFFFFFFFu >> (before_v & 31)) : 0u;
          if (i < d.cap_ver) wv[i] &= keep;
        }
        __syncthreads();
        for (int i = warp; i < cnt; i += kWarps) {
          int64_t t = n0 + r0 + i;
          uint32_t* mask = (uint32_t*)kv_sec(d, CAS_KV_MASK, st) + t * 4;
          uint32_t* rs = (uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, st) + t * d.rec_sm;
          uint32_t* rl = (uint32_t*)kv_sec(d, CAS_KV_VER_LO, st) + t * d.rec_lo;
          uint32_t* rp = (uint32_t*)kv_sec(d, CAS_KV_VER_PR, st) + t * d.rec_pr;
          for (int q = lane; q < d.rec_sm; q += 32) rs[q] = 0u;
          for (int q = lane; q < d.rec_lo; q += 32) rl[q] = 0u;
          for (int q = lane; q < d.rec_pr; q += 32) rp[q] = 0u;
          __syncwarp();
          uint32_t v[4];
          load_block4(src + ((int64_t)(r0 + i) * H + head) * CAS_BLK, lane, v);
          BlockDst dst{mask, rs, rl, rp, nullptr};
          Stream ss{ws, sm.start_s[i], d.cap_spec};
          Stream sv{wv, sm.start_v[i], d.cap_ver};
          Stream dummy{nullptr, 0, 0};
          Stream dummy2{nullptr, 0, 0};
          encode_block<1>(v, d.k, d.m, roe, dst, ss, sv, dummy, dummy2, lane, ~0ull);
        }
      }
      __syncthreads();
    }
  }
  if (threadIdx.x == 0) {
    if (!WRITE) {
      bool cap = fail || ((cur_s + 31) >> 5) > d.cap_spec || ((cur_v + 31) >> 5) > d.cap_ver;
      int err = sm.nonfinite ? CAS_ERR_NONFINITE : (cap ? CAS_ERR_CAPACITY : CAS_OK);
      if (err) {
        atomicExch(&S->call_fail, 1);
        atomicCAS(&S->status, 0, err);
      }
    } else {
      if (!skip) {
        int64_t n1 = n0 + a.T;
        kv_tail_spec(d)[st] = cur_s;
        kv_tail_ver(d)[st] = cur_v;
        sidx[(n1 + 7) >> 3] = (uint32_t)((cur_s + 31) >> 5);
        vidx[(n1 + 7) >> 3] = (uint32_t)((cur_v + 31) >> 5);
      }
      __threadfence();
      unsigned int prev = atomicAdd(&S->done, 1u);
      if (prev == gridDim.x - 1) {
        if (!skip) S->n_tokens = n0 + a.T;
        S->call_fail = 0;
        S->done = 0;
        __threadfence();
      }
    }
  }
}

// Position just past the c-th '1' (c >= 1) of an MSB-first stream starting at
// word w0 (warp); returns w0 * 32 when c == 0.
__device__ uint64_t after_nth_one(const uint32_t* words, uint64_t w0, uint64_t wend, int64_t c, int lane) {
  if (c <= 0) return w0 * 32;
  int64_t seen = 0;
  for (uint64_t b = w0; b < wend; b += 32) {
    uint64_t wi = b + lane;
    uint32_t w = wi < wend ? words[wi] : 0u;
    int ones = __popc(w);
    int incl = warp_incl_add(ones, lane);
    int64_t before = seen + incl - ones;
    bool here = before < c && before + ones >= c;
    unsigned ball = __ballot_sync(CAS_FULL, here);
    if (ball) {
      int src = __ffs(ball) - 1;
      uint64_t pos = 0;
      if (lane == src) {
        int need = (int)(c - before);
        uint32_t x = w;
        int i = 0;
        for (int q = 0; q < need; ++q) {
          i = __clz(x);
          x &= 0x7FFFFFFFu >> i;
        }
        pos = wi * 32 + i + 1;
      }
      return __shfl_sync(CAS_FULL, pos, src);
    }
    seen += __shfl_sync(CAS_FULL, incl, 31);
  }
  return wend * 32;
}

__global__ void kv_truncate_kernel(KvDev d, int64_t n_req) {
  const int st = blockIdx.x, lane = threadIdx.x & 31;
  KvState* S = kv_state(d);
  const int64_t n0 = *(volatile int64_t*)&S->n_tokens;
  const int64_t n = n_req < n0 ? n_req : n0;
  if (n < n0) {
    const uint32_t* ws = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_EXP, st);
    const uint32_t* wv = (const uint32_t*)kv_sec(d, CAS_KV_VER_EXP, st);
    uint32_t* sidx = (uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, st);
    uint32_t* vidx = (uint32_t*)kv_sec(d, CAS_KV_VER_SBIDX, st);
    uint64_t ts = 0, tv = 0;
    if (n > 0) {
      int64_t sb = (n - 1) >> 3, r = n - 8 * sb;
      uint64_t end_s = min((uint64_t)d.cap_spec, (kv_tail_spec(d)[st] + 31) >> 5);
      uint64_t end_v = min((uint64_t)d.cap_ver, (kv_tail_ver(d)[st] + 31) >> 5);
      ts = after_nth_one(ws, sidx[sb], end_s, r * d.k, lane);
      tv = after_nth_one(wv, vidx[sb], end_v, r * (CAS_BLK - d.k), lane);
    }
    if (lane == 0) {
      kv_tail_spec(d)[st] = ts;
      kv_tail_ver(d)[st] = tv;
      sidx[(n + 7) >> 3] = (uint32_t)((ts + 31) >> 5);
      vidx[(n + 7) >> 3] = (uint32_t)((tv + 31) >> 5);
    }
  }
  if (lane == 0) {
    __threadfence();
    unsigned int prev = atomicAdd(&S->done, 1u);
    if (prev == gridDim.x - 1) {
      S->n_tokens = n;
      S->done = 0;
      __threadfence();
    }
  }
}

}  // namespace
}  // namespace cas

using namespace cas;

extern "C" int cas_kv_plan(int H, int64_t Tm, cas_params p, double est, uint64_t* bytes) {
  KvLayout L;
  if (!bytes || !kv_layout(H, Tm, p, est, &L)) return CAS_ERR_INVALID;
  *bytes = L.bytes;
  return CAS_OK;
}

extern "C" int cas_kv_init(cas_kv* kv, void* buf, uint64_t bytes, int H, int64_t Tm, cas_params p, double est,
                           const uint16_t* ck, const uint16_t* cv, int64_t n_calib, void* stream) {
  KvLayout L;
  if (!kv || !buf || ((uintptr_t)buf & 255u) || !kv_layout(H, Tm, p, est, &L)) return CAS_ERR_INVALID;
  if (n_calib < 0 || (n_calib > 0 && (!ck || !cv || !aligned16(ck) || !aligned16(cv)))) return CAS_ERR_INVALID;
  if (bytes < L.bytes) return CAS_ERR_BUFFER;
  cudaStream_t st = (cudaStream_t)stream;
  std::memset(kv, 0, sizeof(*kv));
  kv->n_kv_heads = H;
  kv->head_dim = CAS_BLK;
  kv->p = p;
  kv->max_tokens = Tm;
  kv->cap_spec_words = L.cap_spec;
  kv->cap_ver_words = L.cap_ver;
  kv->base = buf;
  kv->bytes = L.bytes;
  for (int i = 0; i < CAS_KV_NSECT; ++i) {
    kv->off[i] = L.off[i];
    kv->stride[i] = L.stride[i];
  }
  int S = 2 * H;
  uint8_t* b = (uint8_t*)buf;
  if (cudaMemsetAsync(buf, 0, L.bytes, st) != cudaSuccess) return CAS_ERR_CUDA;
  // histogram scratch: the region after the tables (zeroed again below)
  unsigned int* hist = (unsigned int*)(b + L.off[CAS_KV_MASK]);
  std::vector<unsigned int> h((size_t)S * 256, 0);
  if (n_calib > 0) {
    dim3 grid((unsigned)std::min<int64_t>((n_calib * CAS_BLK + 255) / 256, 64), S);
    kv_hist_kernel<<<grid, 256, 0, st>>>(ck, cv, n_calib, H, hist);
    if (launch_status()) return CAS_ERR_CUDA;
    if (cudaMemcpyAsync(h.data(), hist, h.size() * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return CAS_ERR_CUDA;
  }
  std::vector<uint8_t> tables((size_t)S * 512);
  for (int s = 0; s < S; ++s) {
    const unsigned int* c = h.data() + (size_t)s * 256;
    if (c[255]) return CAS_ERR_NONFINITE;
    std::vector<int> order(256);
    for (int e = 0; e < 256; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return c[x] > c[y]; });
    for (int r = 0; r < 256; ++r) {
      tables[(size_t)s * 512 + r] = (uint8_t)order[r];
      tables[(size_t)s * 512 + 256 + order[r]] = (uint8_t)r;
    }
  }
  if (cudaMemsetAsync(hist, 0, (size_t)S * 256 * 4, st) != cudaSuccess ||
      cudaMemcpyAsync(b + L.off[CAS_KV_TABLES], tables.data(), tables.size(), cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return CAS_ERR_CUDA;
  return CAS_OK;
}

extern "C" int cas_encode_kv_append(cas_kv* kv, const uint16_t* knew, const uint16_t* vnew, int T, void* stream) {
  int s = check_kv(kv);
  if (s) return s;
  if (T < 0 || (T > 0 && (!knew || !vnew || !aligned16(knew) || !aligned16(vnew)))) return CAS_ERR_INVALID;
  if (T == 0) return CAS_OK;
  AppendArgs a{make_kv_dev(kv), knew, vnew, T};
  cudaStream_t st = (cudaStream_t)stream;
  int S = 2 * kv->n_kv_heads;
  kv_append_kernel<false><<<S, kThreads, 0, st>>>(a);
  kv_append_kernel<true><<<S, kThreads, 0, st>>>(a);
  return launch_status();
}

extern "C" int cas_kv_truncate(cas_kv* kv, int64_t n, void* stream) {
  int s = check_kv(kv);
  if (s) return s;
  if (n < 0) return CAS_ERR_INVALID;
  kv_truncate_kernel<<<2 * kv->n_kv_heads, 32, 0, (cudaStream_t)stream>>>(make_kv_dev(kv), n);
  return launch_status();
}

extern "C" int cas_kv_status(const cas_kv* kv, int64_t* n_tokens, void* stream) {
  int s = check_kv(kv);
  if (s) return s;
  KvState h;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&h, (uint8_t*)kv->base + kv->off[CAS_KV_STATE], sizeof(h), cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return CAS_ERR_CUDA;
  if (n_tokens) *n_tokens = h.n_tokens;
  return h.status;
}

extern "C" int cas_kv_clear_status(cas_kv* kv, void* stream) {
  int s = check_kv(kv);
  if (s) return s;
  if (cudaMemsetAsync((uint8_t*)kv->base + kv->off[CAS_KV_STATE] + 8, 0, 4, (cudaStream_t)stream) != cudaSuccess)
    return CAS_ERR_CUDA;
  return CAS_OK;
}
