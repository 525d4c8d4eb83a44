// common.cuh - device helpers shared by the libcas kernels (sm_103a).
//
// Format (restated from the method; see include/cas.h for the section list):
//   block      = 128 consecutive elements of a row (value-pruning granule);
//   superblock = 8 consecutive blocks of one row (Cassandra paper, Fig. 11);
//   unary code of rank r = r zero bits then a one bit, MSB-first in u32 words
//   (Cassandra blog review, section 3.2: "count zeros until a one");
//   fixed-width fields are LSB-first in u32 words.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/cas.h"

#define CAS_FULL 0xFFFFFFFFu
#define CAS_BLK 128
#define CAS_SB 8

namespace cas {

// ------------------------------------------------------------------ views
// Device view of an encoded weight tensor, passed by value to kernels.
struct WView {
  const uint32_t* mask;
  const uint32_t* ssm;
  const uint32_t* sexp;
  const uint32_t* sidx;
  const uint8_t* smx;
  const uint32_t* sq;
  const uint32_t* vlo;
  const uint32_t* vd;
  const uint32_t* vdidx;
  const uint32_t* vres;
  const uint32_t* vresidx;
  const uint32_t* vpr;
  const uint32_t* vexp;
  const uint32_t* vidx;
  int64_t N, K, nsb;
  int nbr, nsr;
  int variant, k, m;
  int rec_sm, rec_q, rec_lo, rec_pr;
  // words of each variable-length stream section (reads stay below these)
  uint32_t lim_sexp, lim_vexp, lim_vd, lim_vres;
};

struct Lut {
  uint8_t v[256];
};

inline int rec_words(int nfields, int width) { return (nfields * width + 31) / 32; }

// ------------------------------------------------------------------ warp primitives
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

__device__ __forceinline__ int warp_incl_add(int v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int t = __shfl_up_sync(CAS_FULL, v, d);
    if (lane >= d) v += t;
  }
  return v;
}
__device__ __forceinline__ int warp_incl_max(int v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int t = __shfl_up_sync(CAS_FULL, v, d);
    if (lane >= d) v = max(v, t);
  }
  return v;
}
__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(CAS_FULL, v, d);
  return v;
}
__device__ __forceinline__ float warp_sumf(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(CAS_FULL, v, d);
  return v;
}

// Bit field of `width` (<= 25) bits at bit offset `bit` of an LSB-first word
// array. Reads words bit>>5 and (bit>>5)+1; callers pad arrays by one word.
__device__ __forceinline__ uint32_t get_field(const uint32_t* w, int bit, int width) {
  int i = bit >> 5;
  uint32_t v = __funnelshift_r(w[i], w[i + 1], bit & 31);
  return v & ((1u << width) - 1u);
}

// Position (0..31, from the LSB) of the r-th set bit of m (r 0-based,
// r < popc(m)): five popcount steps.
__device__ __forceinline__ int nth_set_bit(uint32_t m, int r) {
  int pos = 0;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    int c = __popc(m & ((1u << w) - 1u));
    if (r >= c) {
      r -= c;
      m >>= w;
      pos += w;
    }
  }
  return pos;
}

// Number of lanes whose non-decreasing value `v` is <= target (binary lifting
// over the warp with shuffles); when v[31] > target this is the first lane
// with v > target.
__device__ __forceinline__ int warp_count_le(int v, int target) {
  int lo = 0;
#pragma unroll
  for (int step = 16; step >= 1; step >>= 1) {
    int u = __shfl_sync(CAS_FULL, v, lo + step - 1);
    if (u <= target) lo += step;
  }
  return lo;
}

// ------------------------------------------------------------------ unary decoding
// Warp-cooperative decode of the first `ncodes` unary codes of an MSB-first
// stream of `nwords` words. Code i (rank r) is written as lut[r] to out[i].
// Each lane takes one word per round: a popcount prefix gives the ordinal of
// the first code ending in the word, a max-scan of the last '1' position gives
// where the previous code ended, and the lane walks its '1' bits with clz.
// Stream words are read with the read-only path; out and lut are shared memory.
__device__ __forceinline__ void warp_decode_unary(const uint32_t* __restrict__ words, int nwords,
                                                  const uint8_t* __restrict__ lut,
                                                  uint8_t* __restrict__ out, int ncodes, int lane) {
  int done = 0;   // codes completed before this round
  int prev = -1;  // stream bit index of the last '1' before this round
  for (int c0 = 0; c0 < nwords && done < ncodes; c0 += 32) {
    int wi = c0 + lane;
    uint32_t w = wi < nwords ? __ldg(words + wi) : 0u;
    int ones = __popc(w);
    int incl = warp_incl_add(ones, lane);
    int ord = done + incl - ones;
    int last = w ? (wi * 32 + 32 - __ffs(w)) : -1;
    int mx = warp_incl_max(last, lane);
    int pv = __shfl_up_sync(CAS_FULL, mx, 1);
    if (lane == 0) pv = -1;
    pv = max(pv, prev);
    int base = wi * 32;
    while (w) {
      int i = __clz(w);
      int pos = base + i;
      if (ord < ncodes) out[ord] = lut[(pos - pv - 1) & 255];
      pv = pos;
      ++ord;
      w &= 0x7FFFFFFFu >> i;
    }
    done += __shfl_sync(CAS_FULL, incl, 31);
    prev = max(prev, __shfl_sync(CAS_FULL, mx, 31));
  }
}

// Same, but writes the raw code value (the unary count) instead of a table
// lookup; used for the Cassandra-2 exponent distances.
__device__ __forceinline__ void warp_decode_unary_raw(const uint32_t* __restrict__ words, int nwords,
                                                      uint8_t* __restrict__ out, int ncodes, int lane) {
  int done = 0, prev = -1;
  for (int c0 = 0; c0 < nwords && done < ncodes; c0 += 32) {
    int wi = c0 + lane;
    uint32_t w = wi < nwords ? __ldg(words + wi) : 0u;
    int ones = __popc(w);
    int incl = warp_incl_add(ones, lane);
    int ord = done + incl - ones;
    int last = w ? (wi * 32 + 32 - __ffs(w)) : -1;
    int mx = warp_incl_max(last, lane);
    int pv = __shfl_up_sync(CAS_FULL, mx, 1);
    if (lane == 0) pv = -1;
    pv = max(pv, prev);
    int base = wi * 32;
    while (w) {
      int i = __clz(w);
      int pos = base + i;
      if (ord < ncodes) out[ord] = (uint8_t)min(pos - pv - 1, 255);
      pv = pos;
      ++ord;
      w &= 0x7FFFFFFFu >> i;
    }
    done += __shfl_sync(CAS_FULL, incl, 31);
    prev = max(prev, __shfl_sync(CAS_FULL, mx, 31));
  }
}

// ------------------------------------------------------------------ value pruning
// Block of 128 values held 4 per lane (lane L: positions 4L..4L+3, in order).
// Returns a 4-bit mask of kept positions: the k largest keys (bits & 0x7FFF),
// ties to the lower position (Cassandra blog review, section 3.1: keep the most
// salient values). tau = largest key with count(key >= tau) >= k, found by a
// 15-step bisection with ballots.
__device__ __forceinline__ uint32_t select_block4(const uint32_t key[4], int k, int lane) {
  if (k <= 0) return 0u;
  if (k >= CAS_BLK) return 0xFu;
  int lo = 0, hi = 0x7FFF;  // invariant: count(key >= lo) >= k
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    int c = __popc(__ballot_sync(CAS_FULL, key[0] >= (uint32_t)mid)) +
            __popc(__ballot_sync(CAS_FULL, key[1] >= (uint32_t)mid)) +
            __popc(__ballot_sync(CAS_FULL, key[2] >= (uint32_t)mid)) +
            __popc(__ballot_sync(CAS_FULL, key[3] >= (uint32_t)mid));
    if (c >= k) lo = mid; else hi = mid - 1;
  }
  uint32_t tau = (uint32_t)lo;
  int gt = __popc(__ballot_sync(CAS_FULL, key[0] > tau)) + __popc(__ballot_sync(CAS_FULL, key[1] > tau)) +
           __popc(__ballot_sync(CAS_FULL, key[2] > tau)) + __popc(__ballot_sync(CAS_FULL, key[3] > tau));
  int need = k - gt;  // equal keys to keep, lowest positions first
  int eq = (key[0] == tau) + (key[1] == tau) + (key[2] == tau) + (key[3] == tau);
  int before = warp_incl_add(eq, lane) - eq;
  uint32_t kept = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    bool keep = key[j] > tau;
    if (key[j] == tau) {
      keep = before < need;
      ++before;
    }
    kept |= (uint32_t)keep << j;
  }
  return kept;
}

// Mask word w (positions 32w..32w+31) of a block whose kept nibbles are spread
// 4 per lane. Valid in lanes 0..3 (lane = w).
__device__ __forceinline__ uint32_t gather_mask_word(uint32_t nib, int lane) {
  uint32_t word = 0;
#pragma unroll
  for (int l = 0; l < 8; ++l) {
    uint32_t v = __shfl_sync(CAS_FULL, nib, ((lane & 3) << 3) + l);
    word |= v << (4 * l);
  }
  return word;
}

// ------------------------------------------------------------------ stream indices
#ifdef CAS_DEBUG
// Debug builds: set when a superblock index is not non-decreasing or points
// past its section (one flag per translation unit, read by cas_device_status).
static __device__ int g_corrupt_status = 0;
#endif

// Word range [a, b) of superblock s of a variable-length stream whose index
// is idx and whose section holds lim words. A corrupted index cannot move a
// read outside the section: b is clamped to lim and a to b.
__device__ __forceinline__ void stream_clamp(uint32_t a0, uint32_t b0, uint32_t lim, uint32_t& a, uint32_t& b) {
  b = min(b0, lim);
  a = min(a0, b);
#ifdef CAS_DEBUG
  if (a0 > b0 || b0 > lim) atomicExch(&g_corrupt_status, CAS_ERR_CORRUPT);
#endif
}
__device__ __forceinline__ void stream_range(const uint32_t* __restrict__ idx, int64_t s, uint32_t lim, uint32_t& a,
                                             uint32_t& b) {
  stream_clamp(__ldg(idx + s), __ldg(idx + s + 1), lim, a, b);
}

// ------------------------------------------------------------------ bounded waits
// Spin limits: a wait that runs out returns false; the caller records a status
// and leaves the kernel instead of hanging the GPU.
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(a), "r"(phase)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, phase)) return true;
  return false;
}
// 1-D bulk copy global -> shared through the TMA unit, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  uint32_t b = (uint32_t)__cvta_generic_to_shared(bar);
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(d),
               "l"(src), "r"(bytes), "r"(b)
               : "memory");
}

// bf16 bits -> float
__device__ __forceinline__ float bf2f(uint32_t b) { return __uint_as_float(b << 16); }
// float -> bf16 bits, round to nearest even (the glue kernels' rounding)
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
// SiLU(g) * u in fp32, one expression shared by every kernel that forms it
__device__ __forceinline__ float silu_mul_f(float g, float u) { return g / (1.f + expf(-g)) * u; }

// 2^(be - 127) as a float for be in [-22, 254] (subnormal below 1).
__device__ __forceinline__ float pow2_biased(int be) {
  return be >= 1 ? __uint_as_float((uint32_t)be << 23) : __uint_as_float(1u << (22 + be));
}

}  // namespace cas

// ------------------------------------------------------------------ launches
// Launch overlap (cas_set_launch_overlap, off by default): kernels are then
// launched with programmatic stream serialization, so a kernel's CTAs may
// become resident while the kernel before it in the stream is still running.
// Every kernel starts with pdl_wait(), which returns once that kernel has
// completed and its writes are visible (at once without such a kernel):
// nothing global is read or written before it, so what overlaps is the launch
// and the CTA start-up. pdl_trigger() lets the next kernel's CTAs launch into
// the SM slots this kernel frees. A kernel that a call enqueues right after
// its own memset or copy is launched plainly (launch_plain).
namespace cas {
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

bool launch_overlap();

template <class... P, class... A>
inline int launch_with(bool overlap, void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       A... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, args...) == cudaSuccess ? CAS_OK : CAS_ERR_CUDA;
}
template <class... P, class... A>
inline int launch_k(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A... args) {
  return launch_with(launch_overlap(), k, grid, block, smem, st, args...);
}
template <class... P, class... A>
inline int launch_plain(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A... args) {
  return launch_with(false, k, grid, block, smem, st, args...);
}
}  // namespace cas

// host-side helpers shared by the translation units
namespace cas {
WView make_view(const cas_weights* W);
bool aligned16(const void* p);
int check_weights(const cas_weights* W);
// Reads (and with clear, resets) the debug build's corrupt-index flag of the
// translation unit that defines it; 0 in other builds.
int corrupt_status_gemv(bool clear);
int corrupt_status_gemm(bool clear);
int corrupt_status_decode(bool clear);
int sm_count();
int launch_status();
// Clears n floats at p (16-byte aligned) with a kernel on st.
int zero_f32(float* p, int64_t n, cudaStream_t st);
// Resident CTAs per SM of `func` with `threads` threads and `smem` dynamic
// shared bytes; raises the kernel's dynamic shared-memory limit on first use.
// Cached per (func, threads, smem), so repeated launches make no query.
int occupancy(const void* func, int threads, size_t smem);
}  // namespace cas
