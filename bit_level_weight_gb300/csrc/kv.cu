// kv.cu - compressed KV cache: layout, calibration (rank tables), online
// append (Cassandra blog review, section 3.3: the KV cache is produced during
// inference and encoded online), truncation (rejected draft tokens) and the
// device status. Both variants: Cassandra-1 (unary exponent codes) and
// Cassandra-2 (MX shared exponent per 32 positions).
//
// Every (head, K|V) stream has up to three variable-length code streams:
//   A: unary codes of kept values (C-1 exponent ranks, C-2 distances d);
//   B: unary codes of pruned exponents (both variants);
//   C: C-2 residual significand bits (fixed widths min(8, 7-m+d)).
// Each is word-aligned per superblock (8 tokens) with a u32 index of word
// offsets; the device state keeps the bit tail of every stream.
//
// Append runs two kernels with one CTA per stream: the first computes every
// new token's code lengths and checks capacity and finiteness (a failure sets
// a per-call flag and the sticky status); the second, unless the flag is set,
// clears the stream words it will fill and encodes the tokens (one warp per
// token). The CTA that finishes last advances n_tokens and resets the
// per-call counters. No CTA waits on another.
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
  d.variant = kv->p.variant;
  d.k = kv->p.keep_per_block;
  d.m = kv->p.mant_bits;
  d.rec_sm = rec_words(d.k, d.m + 1);
  d.rec_q = rec_words(d.k, d.m + 2);
  d.rec_lo = rec_words(d.k, 7 - d.m);
  d.rec_pr = rec_words(CAS_BLK - d.k, 8);
  d.max_tokens = kv->max_tokens;
  d.cap_a = kv->cap_spec_words;
  d.cap_b = kv->cap_ver_words;
  d.cap_c = kv->stride[CAS_KV_VER_RES] / 4;
  return d;
}

int check_kv(const cas_kv* kv) {
  if (!kv || !kv->base || kv->n_kv_heads < 1 || kv->head_dim != CAS_BLK || kv->max_tokens < 1 ||
      (kv->p.variant != 1 && kv->p.variant != 2) || kv->p.keep_per_block < 0 || kv->p.keep_per_block > CAS_BLK ||
      kv->p.mant_bits < 0 || kv->p.mant_bits > 7)
    return CAS_ERR_INVALID;
  return CAS_OK;
}

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 256;  // tokens whose starts are computed per round

uint64_t a256(uint64_t x) { return (x + 255) & ~255ull; }

struct KvLayout {
  uint64_t off[16], stride[16], bytes, cap_a, cap_b;
};

bool kv_layout(int H, int64_t Tm, cas_params p, double est, KvLayout* L) {
  if (H < 1 || Tm < 1 || (p.variant != 1 && p.variant != 2) || p.keep_per_block < 0 ||
      p.keep_per_block > CAS_BLK || p.mant_bits < 0 || p.mant_bits > 7 || !(est > 0.0) || est > 256.0)
    return false;
  const int k = p.keep_per_block, m = p.mant_bits;
  const bool v1 = p.variant == 1;
  const uint64_t S = 2ull * H, nsbm = (uint64_t)(Tm + 7) / 8, T = (uint64_t)Tm;
  L->cap_a = (uint64_t)std::ceil((double)Tm * k * est / 32.0) + nsbm + 2;
  L->cap_b = (uint64_t)std::ceil((double)Tm * (CAS_BLK - k) * est / 32.0) + nsbm + 2;
  const uint64_t cap_c = v1 ? 0 : nsbm * (2ull * k + 1) + 2;  // 8 tokens x k x 8 bits per superblock
  std::memset(L->off, 0, sizeof(L->off));
  std::memset(L->stride, 0, sizeof(L->stride));
  const uint64_t state_bytes = 32 + 24 * S;
  const uint64_t idx = a256((nsbm + 1) * 4);
  L->stride[CAS_KV_TABLES] = 512;
  L->stride[CAS_KV_MASK] = a256(T * 16);
  L->stride[CAS_KV_VER_PR] = a256(T * rec_words(CAS_BLK - k, 8) * 4);
  L->stride[CAS_KV_VER_EXP] = a256(L->cap_b * 4);
  L->stride[CAS_KV_VER_SBIDX] = idx;
  if (v1) {
    L->stride[CAS_KV_SPEC_SM] = a256(T * rec_words(k, m + 1) * 4);
    L->stride[CAS_KV_SPEC_EXP] = a256(L->cap_a * 4);
    L->stride[CAS_KV_SPEC_SBIDX] = idx;
    L->stride[CAS_KV_VER_LO] = a256(T * rec_words(k, 7 - m) * 4);
  } else {
    L->stride[CAS_KV_SPEC_MX] = a256(T * 4);
    L->stride[CAS_KV_SPEC_Q] = a256(T * rec_words(k, m + 2) * 4);
    L->stride[CAS_KV_VER_D] = a256(L->cap_a * 4);
    L->stride[CAS_KV_VER_D_SBIDX] = idx;
    L->stride[CAS_KV_VER_RES] = a256(cap_c * 4);
    L->stride[CAS_KV_VER_RES_SBIDX] = idx;
  }
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
  pdl_wait();
  pdl_trigger();
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

// Code bits of one token block (warp) for streams A, B, C; also reports
// whether any value is NaN/Inf.
template <int VAR>
__device__ __forceinline__ void token_bits(const uint16_t* blk, int k, int m, const uint8_t* roe, int lane,
                                           int bits[3], bool* nonfinite) {
  uint32_t v[4];
  load_block4(blk, lane, v);
  uint32_t key[4] = {v[0] & 0x7FFFu, v[1] & 0x7FFFu, v[2] & 0x7FFFu, v[3] & 0x7FFFu};
  uint32_t kept = select_block4(key, k, lane);
  bool nf = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) nf |= ((v[j] >> 7) & 0xFF) == 255;
  const int E = VAR == 2 ? group_shared_exp(v, kept) : 0;
  const BlockBits b = block_lane_bits<VAR>(v, kept, E, m, roe);
  bits[0] = warp_sum(VAR == 1 ? b.sexp : b.vd);
  bits[1] = warp_sum(b.vexp);
  bits[2] = warp_sum(b.vres);
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
  int bits[3][kChunk];
  uint64_t start[3][kChunk];
  int nonfinite;
};

template <int VAR, bool WRITE>
__global__ void __launch_bounds__(kThreads) kv_append_kernel(AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ RoundSmem sm;
  __shared__ uint8_t roe[256];
  __shared__ uint64_t cur[3];
  __shared__ int skip;
  const KvDev& d = a.d;
  const int st = blockIdx.x, H = d.H, head = st % H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nstreams = VAR == 1 ? 2 : 3;
  KvState* S = kv_state(d);
  const uint16_t* src = st < H ? a.knew : a.vnew;
  for (int i = threadIdx.x; i < 256; i += kThreads) roe[i] = kv_rank_of_exp(d, st)[i];
  const int64_t n0 = *(volatile int64_t*)&S->n_tokens;
  if (threadIdx.x == 0) {
    for (int q = 0; q < 3; ++q) cur[q] = q < nstreams ? kv_tail(d, q)[st] : 0ull;
    sm.nonfinite = 0;
    skip = WRITE ? *(volatile int32_t*)&S->call_fail : 0;
  }
  __syncthreads();
  uint32_t* words[3];
  uint32_t* idx[3];
  uint64_t cap[3] = {d.cap_a, d.cap_b, d.cap_c};
  for (int q = 0; q < 3; ++q) {
    words[q] = (uint32_t*)kv_sec(d, kv_stream_sec(VAR, q), st);
    idx[q] = (uint32_t*)kv_sec(d, kv_index_sec(VAR, q), st);
  }
  const bool fail = !WRITE && n0 + a.T > d.max_tokens;
  if (!skip && !fail) {
    for (int r0 = 0; r0 < a.T; r0 += kChunk) {
      const int cnt = min(kChunk, a.T - r0);
      for (int i = warp; i < cnt; i += kWarps) {
        int bits[3];
        bool nf;
        token_bits<VAR>(src + ((int64_t)(r0 + i) * H + head) * CAS_BLK, d.k, d.m, roe, lane, bits, &nf);
        if (lane == 0) {
          for (int q = 0; q < 3; ++q) sm.bits[q][i] = bits[q];
          if (nf) sm.nonfinite = 1;
        }
      }
      __syncthreads();
      uint64_t before[3] = {cur[0], cur[1], cur[2]};
      __syncthreads();
      if (threadIdx.x == 0) {
        // token t starting a superblock aligns every stream to a word and
        // records the superblock's word offsets
        uint64_t c[3] = {cur[0], cur[1], cur[2]};
        for (int i = 0; i < cnt; ++i) {
          const int64_t t = n0 + r0 + i;
          for (int q = 0; q < nstreams; ++q) {
            if ((t & 7) == 0) {
              c[q] = (c[q] + 31) & ~31ull;
              if (WRITE) idx[q][t >> 3] = (uint32_t)(c[q] >> 5);
            }
            sm.start[q][i] = c[q];
            c[q] += sm.bits[q][i];
          }
        }
        for (int q = 0; q < 3; ++q) cur[q] = c[q];
      }
      __syncthreads();
      if (WRITE) {
        // clear [before, end) of every stream; a partial first word keeps its old bits
        for (int q = 0; q < nstreams; ++q) {
          const uint64_t b0 = before[q], e = (cur[q] + 31) >> 5;
          for (uint64_t i = (b0 >> 5) + threadIdx.x; i < e; i += kThreads) {
            uint32_t keep = 0u;
            if (i == (b0 >> 5) && (b0 & 31)) keep = q == 2 ? (0xFFFFFFFFu >> (32 - (b0 & 31))) : ~(0xFFFFFFFFu >> (b0 & 31));
            if (i < cap[q]) words[q][i] &= keep;
          }
        }
        __syncthreads();
        for (int i = warp; i < cnt; i += kWarps) {
          const int64_t t = n0 + r0 + i;
          uint32_t* mask = (uint32_t*)kv_sec(d, CAS_KV_MASK, st) + t * 4;
          uint32_t* rp = (uint32_t*)kv_sec(d, CAS_KV_VER_PR, st) + t * d.rec_pr;
          uint32_t* rs;
          uint32_t* rl = nullptr;
          uint8_t* mx = nullptr;
          int rs_words, rl_words = 0;
          if (VAR == 1) {
            rs = (uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, st) + t * d.rec_sm;
            rs_words = d.rec_sm;
            rl = (uint32_t*)kv_sec(d, CAS_KV_VER_LO, st) + t * d.rec_lo;
            rl_words = d.rec_lo;
          } else {
            rs = (uint32_t*)kv_sec(d, CAS_KV_SPEC_Q, st) + t * d.rec_q;
            rs_words = d.rec_q;
            mx = kv_sec(d, CAS_KV_SPEC_MX, st) + t * 4;
          }
          for (int q = lane; q < rs_words; q += 32) rs[q] = 0u;
          for (int q = lane; q < rl_words; q += 32) rl[q] = 0u;
          for (int q = lane; q < d.rec_pr; q += 32) rp[q] = 0u;
          __syncwarp();
          uint32_t v[4];
          load_block4(src + ((int64_t)(r0 + i) * H + head) * CAS_BLK, lane, v);
          BlockDst dst{mask, rs, rl, rp, mx};
          Stream sa{words[0], sm.start[0][i], cap[0]};
          Stream sb{words[1], sm.start[1][i], cap[1]};
          Stream sc{words[2], VAR == 2 ? sm.start[2][i] : 0ull, cap[2]};
          Stream none{nullptr, 0, 0};
          if (VAR == 1)
            encode_block<1>(v, d.k, d.m, roe, dst, sa, sb, none, none, lane, ~0ull);
          else
            encode_block<2>(v, d.k, d.m, roe, dst, none, sb, sa, sc, lane, ~0ull);
        }
      }
      __syncthreads();
    }
  }
  if (threadIdx.x == 0) {
    if (!WRITE) {
      bool over = fail;
      for (int q = 0; q < nstreams; ++q) over |= ((cur[q] + 31) >> 5) > cap[q];
      const int err = sm.nonfinite ? CAS_ERR_NONFINITE : (over ? CAS_ERR_CAPACITY : CAS_OK);
      if (err) {
        atomicExch(&S->call_fail, 1);
        atomicCAS(&S->status, 0, err);
      }
    } else {
      if (!skip) {
        const int64_t n1 = n0 + a.T;
        for (int q = 0; q < nstreams; ++q) {
          kv_tail(d, q)[st] = cur[q];
          idx[q][(n1 + 7) >> 3] = (uint32_t)((cur[q] + 31) >> 5);
        }
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

// Truncation: the new tail of each stream is found inside the superblock of
// the last kept token - after its r*k kept codes (stream A), r*(128-k) pruned
// codes (stream B) and, for Cassandra-2, after the residual widths of those r*k
// kept values, which are read from their d codes (stream C).
// One warp per stream st of the cache; the last of its 2H warps to finish
// publishes the new token count.
template <int VAR>
__device__ __forceinline__ void kv_truncate_stream(const KvDev& d, int64_t n_req, int st, uint8_t* s_d) {
  const int lane = threadIdx.x & 31;
  KvState* S = kv_state(d);
  const int64_t n0 = *(volatile int64_t*)&S->n_tokens;
  const int64_t n = n_req < n0 ? n_req : n0;
  const int nstreams = VAR == 1 ? 2 : 3;
  if (n < n0) {
    uint64_t tail[3] = {0, 0, 0};
    const uint64_t cap[3] = {d.cap_a, d.cap_b, d.cap_c};
    const int64_t sb = n > 0 ? (n - 1) >> 3 : 0;
    if (n > 0) {
      const int64_t r = n - 8 * sb;
      const int64_t cnt[2] = {r * d.k, r * (CAS_BLK - d.k)};
      for (int q = 0; q < 2; ++q) {
        const uint32_t* w = (const uint32_t*)kv_sec(d, kv_stream_sec(VAR, q), st);
        const uint32_t* ix = (const uint32_t*)kv_sec(d, kv_index_sec(VAR, q), st);
        const uint64_t end = min(cap[q], (kv_tail(d, q)[st] + 31) >> 5);
        tail[q] = after_nth_one(w, ix[sb], end, cnt[q], lane);
      }
      if (VAR == 2) {
        const uint32_t* w = (const uint32_t*)kv_sec(d, CAS_KV_VER_D, st);
        const uint32_t* ix = (const uint32_t*)kv_sec(d, CAS_KV_VER_D_SBIDX, st);
        const uint32_t* rix = (const uint32_t*)kv_sec(d, CAS_KV_VER_RES_SBIDX, st);
        const int ncodes = (int)cnt[0];
        const int nw = (int)(min(cap[0], (kv_tail(d, 0)[st] + 31) >> 5) - ix[sb]);
        warp_decode_unary_raw(w + ix[sb], nw, s_d, ncodes, lane);
        __syncwarp();
        int sum = 0;
        for (int i = lane; i < ncodes; i += 32) sum += min(8, 7 - d.m + (int)s_d[i]);
        sum = warp_sum(sum);
        tail[2] = (uint64_t)rix[sb] * 32 + sum;
      }
    }
    if (lane == 0) {
      for (int q = 0; q < nstreams; ++q) {
        kv_tail(d, q)[st] = tail[q];
        uint32_t* ix = (uint32_t*)kv_sec(d, kv_index_sec(VAR, q), st);
        ix[(n + 7) >> 3] = (uint32_t)((tail[q] + 31) >> 5);
      }
    }
  }
  if (lane == 0) {
    __threadfence();
    unsigned int prev = atomicAdd(&S->done, 1u);
    if (prev == 2u * (unsigned)d.H - 1u) {
      S->n_tokens = n;
      S->done = 0;
      __threadfence();
    }
  }
}

template <int VAR>
__global__ void kv_truncate_kernel(KvDev d, int64_t n_req) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint8_t s_d[CAS_SB * CAS_BLK];
  kv_truncate_stream<VAR>(d, n_req, blockIdx.x, s_d);
}

// Several caches of one variant in one launch: blockIdx.y picks the cache,
// blockIdx.x its stream (caches with fewer heads leave the rest idle).
constexpr int kTruncBatch = 80;  // descriptors per launch (kernel parameters stay under 32 KB)
struct TruncBatch {
  KvDev d[kTruncBatch];
};
template <int VAR>
__global__ void kv_truncate_many_kernel(const __grid_constant__ TruncBatch b, int64_t n_req) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint8_t s_d[CAS_SB * CAS_BLK];
  const KvDev& d = b.d[blockIdx.y];
  if ((int)blockIdx.x < 2 * d.H) kv_truncate_stream<VAR>(d, n_req, blockIdx.x, s_d);
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
  kv->cap_spec_words = L.cap_a;
  kv->cap_ver_words = L.cap_b;
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
    if (const int e_ = launch_plain(kv_hist_kernel, grid, 256, 0, st, ck, cv, n_calib, H, hist)) return e_;
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
  if (kv->p.variant == 1) {
    if (const int e_ = launch_k(kv_append_kernel<1, false>, S, kThreads, 0, st, a)) return e_;
    if (const int e_ = launch_k(kv_append_kernel<1, true>, S, kThreads, 0, st, a)) return e_;
  } else {
    if (const int e_ = launch_k(kv_append_kernel<2, false>, S, kThreads, 0, st, a)) return e_;
    if (const int e_ = launch_k(kv_append_kernel<2, true>, S, kThreads, 0, st, a)) return e_;
  }
  return launch_status();
}

extern "C" int cas_kv_truncate(cas_kv* kv, int64_t n, void* stream) {
  int s = check_kv(kv);
  if (s) return s;
  if (n < 0) return CAS_ERR_INVALID;
  const cudaStream_t st = (cudaStream_t)stream;
  return kv->p.variant == 1 ? launch_k(kv_truncate_kernel<1>, 2 * kv->n_kv_heads, 32, 0, st, make_kv_dev(kv), n)
                            : launch_k(kv_truncate_kernel<2>, 2 * kv->n_kv_heads, 32, 0, st, make_kv_dev(kv), n);
}

extern "C" int cas_kv_truncate_many(cas_kv* const* kvs, int count, int64_t n, void* stream) {
  if (count < 0 || (count > 0 && !kvs) || n < 0) return CAS_ERR_INVALID;
  for (int i = 0; i < count; ++i) {
    const int s = check_kv(kvs[i]);
    if (s) return s;
  }
  const cudaStream_t st = (cudaStream_t)stream;
  // one launch per variant and per kTruncBatch caches
  for (int var = 1; var <= 2; ++var) {
    TruncBatch b;
    int m = 0, hmax = 0;
    for (int i = 0; i <= count; ++i) {
      if (i < count && kvs[i]->p.variant == var) {
        b.d[m++] = make_kv_dev(kvs[i]);
        hmax = std::max(hmax, kvs[i]->n_kv_heads);
      }
      if (m > 0 && (m == kTruncBatch || i == count)) {
        const dim3 grid((unsigned)(2 * hmax), (unsigned)m);
        const int e = var == 1 ? launch_k(kv_truncate_many_kernel<1>, grid, 32, 0, st, b, n)
                               : launch_k(kv_truncate_many_kernel<2>, grid, 32, 0, st, b, n);
        if (e) return e;
        m = hmax = 0;
      }
    }
  }
  return CAS_OK;
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
