// glue.cu - the transformer operations between the split's matrix products in
// one decode step of the evaluated models (Llama-3-8B, Qwen3-8B: Cassandra
// paper, evaluation; Cassandra blog review, section 4): residual add fused with
// RMSNorm, the split of the fused QKV product with rotary position embedding,
// SiLU(gate) * up, fp32 -> bf16, greedy argmax and the embedding lookup.
// They turn the per-matrix entry points into a data-dependent forward: every
// kernel reads what the previous one wrote.
//
// Numerics: fp32 arithmetic, bf16 outputs rounded to nearest even; the rotary
// angle p * theta^(-2i/D) is formed and reduced in double precision and its
// sine and cosine taken in double, so long contexts lose no accuracy there.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"

namespace cas {
namespace {

__device__ __forceinline__ uint16_t to_bf16(float f) { return f2bf(f); }

// ---------------------------------------------------------------- add + RMSNorm
// x[r] += y[r] (when y is given), then out[r] = bf16(x[r] / sqrt(mean(x[r]^2) + eps) * gamma).
// One CTA of 1024 threads per row; a thread keeps its <= kNormVpt values in
// registers, so the row is read and written once.
constexpr int kNormThreads = 1024;
constexpr int kNormVpt = 16;  // dim <= 16384
__global__ void __launch_bounds__(kNormThreads) add_rmsnorm_kernel(float* __restrict__ x, const float* __restrict__ y,
                                                                   int dim, const uint16_t* __restrict__ gamma,
                                                                   float eps, uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[kNormThreads / 32];
  const int64_t r = blockIdx.x;
  float* xr = x + r * dim;
  const float* yr = y ? y + r * dim : nullptr;
  float v[kNormVpt];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kNormVpt; ++k) {
    const int i = threadIdx.x + k * kNormThreads;
    v[k] = 0.f;
    if (i < dim) {
      v[k] = xr[i];
      if (yr) {
        v[k] += yr[i];
        xr[i] = v[k];
      }
    }
    ss = fmaf(v[k], v[k], ss);
  }
  ss = warp_sumf(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = (threadIdx.x & 31) < kNormThreads / 32 ? red[threadIdx.x & 31] : 0.f;
  tot = warp_sumf(tot);
  const float inv = rsqrtf(tot / (float)dim + eps);
#pragma unroll
  for (int k = 0; k < kNormVpt; ++k) {
    const int i = threadIdx.x + k * kNormThreads;
    if (i < dim) out[r * dim + i] = to_bf16(v[k] * inv * bf2f(gamma[i]));
  }
}

// ---------------------------------------------------------------- QKV split + rotary embedding
// qkv: fp32 [rows][(Hq + 2 Hkv) * 128] (q heads, then k heads, then v heads).
// Pairs (i, i + 64) of a q or k head rotate by angle p * theta^(-i/64):
// (a, b) -> (a cos - b sin, b cos + a sin); p = pos0 + row % rows_per_seq.
// The 64 sines and cosines of the row's position are taken once per block.
__global__ void rope_split_kernel(const float* __restrict__ qkv, int Hq, int Hkv, int64_t pos0, int rows_per_seq,
                                  double log_theta, uint16_t* __restrict__ q, uint16_t* __restrict__ k,
                                  int64_t k_stride, uint16_t* __restrict__ v, int64_t v_stride) {
  pdl_wait();
  pdl_trigger();
  __shared__ float cs[64], sn[64];
  const int r = blockIdx.y;
  if (threadIdx.x < 64) {
    const double p = (double)(pos0 + r % rows_per_seq);
    const double ang = p * exp(-log_theta * (double)threadIdx.x / 64.0);
    double sd, cd;
    sincos(fmod(ang, 6.283185307179586476925286766559), &sd, &cd);
    cs[threadIdx.x] = (float)cd;
    sn[threadIdx.x] = (float)sd;
  }
  __syncthreads();
  const int H = Hq + 2 * Hkv;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;  // (head, pair)
  if (t >= H * 64) return;
  const int h = t >> 6, i = t & 63;
  const float* src = qkv + ((int64_t)r * H + h) * CAS_BLK;
  const float a = src[i], b = src[i + 64];
  if (h >= Hq + Hkv) {  // v: no rotation
    uint16_t* d = v + (int64_t)r * v_stride + (int64_t)(h - Hq - Hkv) * CAS_BLK;
    d[i] = to_bf16(a);
    d[i + 64] = to_bf16(b);
    return;
  }
  const float s = sn[i], c = cs[i];
  uint16_t* d = h < Hq ? q + ((int64_t)r * Hq + h) * CAS_BLK : k + (int64_t)r * k_stride + (int64_t)(h - Hq) * CAS_BLK;
  d[i] = to_bf16(fmaf(a, c, -b * s));
  d[i + 64] = to_bf16(fmaf(b, c, a * s));
}

// ---------------------------------------------------------------- SiLU(gate) * up
__global__ void silu_mul_kernel(const float* __restrict__ gu, int F, int64_t n, uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / F;
    const int j = (int)(t - r * F);
    const float g = gu[r * 2 * F + j], u = gu[r * 2 * F + F + j];
    out[t] = to_bf16(silu_mul_f(g, u));
  }
}

__global__ void to_bf16_kernel(const float* __restrict__ in, int64_t n, uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x)
    out[t] = to_bf16(in[t]);
}

// ---------------------------------------------------------------- greedy argmax (ties to the lower index)
constexpr int kArgThreads = 1024;
__global__ void __launch_bounds__(kArgThreads) argmax_kernel(const float* __restrict__ logits, int64_t V,
                                                             int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ float bv[kArgThreads / 32];
  __shared__ int64_t bi[kArgThreads / 32];
  const float* lr = logits + (int64_t)blockIdx.x * V;
  float best = -INFINITY;
  int64_t idx = V;  // none yet
  for (int64_t i = threadIdx.x; i < V; i += kArgThreads) {
    const float v = lr[i];
    if (v > best) {  // strictly greater: the first (lowest) index of a tie stays
      best = v;
      idx = i;
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const float ov = __shfl_xor_sync(CAS_FULL, best, d);
    const int64_t oi = __shfl_xor_sync(CAS_FULL, idx, d);
    if (ov > best || (ov == best && oi < idx)) {
      best = ov;
      idx = oi;
    }
  }
  if ((threadIdx.x & 31) == 0) {
    bv[threadIdx.x >> 5] = best;
    bi[threadIdx.x >> 5] = idx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kArgThreads / 32; ++w)
      if (bv[w] > best || (bv[w] == best && bi[w] < idx)) {
        best = bv[w];
        idx = bi[w];
      }
    out[blockIdx.x] = (int32_t)(idx < V ? idx : 0);
  }
}

// ---------------------------------------------------------------- embedding lookup
__global__ void embed_kernel(const int32_t* __restrict__ tok, const uint16_t* __restrict__ table, int64_t V, int dim,
                             float* __restrict__ x) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  const int64_t id = tok[r];
  const int64_t row = id < 0 ? 0 : (id >= V ? V - 1 : id);  // an invalid id reads a valid row
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < dim; i += gridDim.x * blockDim.x)
    x[(int64_t)r * dim + i] = bf2f(table[row * dim + i]);
}

int grid1d(int64_t n, int threads) {
  const int64_t g = (n + threads - 1) / threads;
  return (int)std::min<int64_t>(std::max<int64_t>(g, 1), (int64_t)sm_count() * 8);
}

// ---------------------------------------------------------------- zero fill
// Clears an fp32 output before kernels that add into it with atomics: as a
// kernel (not a memset) it keeps the chain of kernels that launch overlap
// relies on unbroken.
__global__ void zero_f32_kernel(float4* __restrict__ p4, int64_t n4, float* __restrict__ tail, int nt) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x)
    p4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (blockIdx.x == 0 && (int)threadIdx.x < nt) tail[threadIdx.x] = 0.f;
}

}  // namespace

int zero_f32(float* p, int64_t n, cudaStream_t st) {
  if (n <= 0) return CAS_OK;
  const int64_t n4 = n / 4;  // p is 16-byte aligned
  return launch_k(zero_f32_kernel, grid1d(std::max<int64_t>(n4, 1), 256), 256, 0, st, reinterpret_cast<float4*>(p),
                  n4, p + 4 * n4, (int)(n - 4 * n4));
}
}  // namespace cas

using namespace cas;

extern "C" int cas_add_rmsnorm(float* x, const float* y, int rows, int dim, const uint16_t* gamma, float eps,
                               uint16_t* out, void* stream) {
  if (rows < 0 || dim < 1 || dim > kNormThreads * kNormVpt || !(eps >= 0.f)) return CAS_ERR_INVALID;
  if (rows == 0) return CAS_OK;
  if (!x || !gamma || !out) return CAS_ERR_INVALID;
  return launch_k(add_rmsnorm_kernel, rows, kNormThreads, 0, (cudaStream_t)stream, x, y, dim, gamma, eps, out);
}

extern "C" int cas_rope_split(const float* qkv, int rows, int n_q_heads, int n_kv_heads, int64_t pos0,
                              int rows_per_seq, double theta, uint16_t* q, uint16_t* k, int64_t k_row_stride,
                              uint16_t* v, int64_t v_row_stride, void* stream) {
  if (rows < 0 || n_q_heads < 1 || n_kv_heads < 1 || pos0 < 0 || rows_per_seq < 1 || !(theta > 1.0))
    return CAS_ERR_INVALID;
  if (rows == 0) return CAS_OK;
  if (!qkv || !q || !k || !v || k_row_stride < (int64_t)n_kv_heads * CAS_BLK ||
      v_row_stride < (int64_t)n_kv_heads * CAS_BLK)
    return CAS_ERR_INVALID;
  const int pairs = (n_q_heads + 2 * n_kv_heads) * 64;
  dim3 g((pairs + 255) / 256, rows);
  return launch_k(rope_split_kernel, g, 256, 0, (cudaStream_t)stream, qkv, n_q_heads, n_kv_heads, pos0, rows_per_seq,
                                                         std::log(theta), q, k, k_row_stride, v, v_row_stride);
}

extern "C" int cas_silu_mul(const float* gate_up, int rows, int ffn, uint16_t* out, void* stream) {
  if (rows < 0 || ffn < 1) return CAS_ERR_INVALID;
  if (rows == 0) return CAS_OK;
  if (!gate_up || !out) return CAS_ERR_INVALID;
  const int64_t n = (int64_t)rows * ffn;
  return launch_k(silu_mul_kernel, grid1d(n, 256), 256, 0, (cudaStream_t)stream, gate_up, ffn, n, out);
}

extern "C" int cas_f32_to_bf16(const float* in, int64_t n, uint16_t* out, void* stream) {
  if (n < 0) return CAS_ERR_INVALID;
  if (n == 0) return CAS_OK;
  if (!in || !out) return CAS_ERR_INVALID;
  return launch_k(to_bf16_kernel, grid1d(n, 256), 256, 0, (cudaStream_t)stream, in, n, out);
}

extern "C" int cas_argmax(const float* logits, int rows, int64_t vocab, int32_t* out, void* stream) {
  if (rows < 0 || vocab < 1 || vocab > 0x7FFFFFFF) return CAS_ERR_INVALID;
  if (rows == 0) return CAS_OK;
  if (!logits || !out) return CAS_ERR_INVALID;
  return launch_k(argmax_kernel, rows, kArgThreads, 0, (cudaStream_t)stream, logits, vocab, out);
}

extern "C" int cas_embed(const int32_t* tokens, int rows, const uint16_t* table, int64_t vocab, int dim, float* x,
                         void* stream) {
  if (rows < 0 || vocab < 1 || dim < 1) return CAS_ERR_INVALID;
  if (rows == 0) return CAS_OK;
  if (!tokens || !table || !x) return CAS_ERR_INVALID;
  dim3 g((dim + 255) / 256, rows);
  return launch_k(embed_kernel, g, 256, 0, (cudaStream_t)stream, tokens, table, vocab, dim, x);
}
