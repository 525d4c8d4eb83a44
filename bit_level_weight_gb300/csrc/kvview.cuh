// kvview.cuh - device view of a compressed KV cache (one sequence, one layer).
//
// Stream st = kv * H + head holds one 128-element block per token; a
// superblock is 8 consecutive tokens of a stream, so the stream is encoded
// exactly like a weight tensor of one row whose blocks are the tokens.
#pragma once
#include "common.cuh"

namespace cas {

struct KvDev {
  uint8_t* base;
  uint64_t off[CAS_KV_NSECT];
  uint64_t stride[CAS_KV_NSECT];
  int H, variant, k, m;
  int rec_sm, rec_q, rec_lo, rec_pr;
  int64_t max_tokens;
  uint64_t cap_a, cap_b, cap_c;  // words of the three code streams (per stream)
};

// device state (STATE section)
struct KvState {
  int64_t n_tokens;
  int32_t status;
  int32_t call_fail;
  uint32_t done;
  uint32_t pad[3];
  // followed by uint64 tails[3][S]: kept-value unary stream (A), pruned
  // exponents (B), Cassandra-2 residuals (C)
};
static_assert(sizeof(KvState) == 32, "state header");

__host__ __device__ inline KvState* kv_state(const KvDev& d) { return (KvState*)(d.base + d.off[CAS_KV_STATE]); }
__host__ __device__ inline uint64_t* kv_tail(const KvDev& d, int which) {
  return (uint64_t*)(d.base + d.off[CAS_KV_STATE] + sizeof(KvState)) + which * 2 * d.H;
}
// sections of the three code streams and their superblock indices
__host__ __device__ inline int kv_stream_sec(int variant, int which) {
  return which == 0 ? (variant == 1 ? CAS_KV_SPEC_EXP : CAS_KV_VER_D) : which == 1 ? CAS_KV_VER_EXP : CAS_KV_VER_RES;
}
__host__ __device__ inline int kv_index_sec(int variant, int which) {
  return which == 0 ? (variant == 1 ? CAS_KV_SPEC_SBIDX : CAS_KV_VER_D_SBIDX)
                    : which == 1 ? CAS_KV_VER_SBIDX : CAS_KV_VER_RES_SBIDX;
}
__host__ __device__ inline uint8_t* kv_sec(const KvDev& d, int sec, int st) {
  return d.base + d.off[sec] + (uint64_t)st * d.stride[sec];
}
__host__ __device__ inline const uint8_t* kv_exp_of_rank(const KvDev& d, int st) { return kv_sec(d, CAS_KV_TABLES, st); }
__host__ __device__ inline const uint8_t* kv_rank_of_exp(const KvDev& d, int st) {
  return kv_sec(d, CAS_KV_TABLES, st) + 256;
}

// Weight-style view of stream st holding n tokens.
__device__ inline WView kv_stream_view(const KvDev& d, int st, int64_t n) {
  WView w{};
  w.mask = (const uint32_t*)kv_sec(d, CAS_KV_MASK, st);
  w.ssm = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SM, st);
  w.sexp = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_EXP, st);
  w.sidx = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_SBIDX, st);
  w.vlo = (const uint32_t*)kv_sec(d, CAS_KV_VER_LO, st);
  w.vpr = (const uint32_t*)kv_sec(d, CAS_KV_VER_PR, st);
  w.vexp = (const uint32_t*)kv_sec(d, CAS_KV_VER_EXP, st);
  w.vidx = (const uint32_t*)kv_sec(d, CAS_KV_VER_SBIDX, st);
  w.smx = kv_sec(d, CAS_KV_SPEC_MX, st);
  w.sq = (const uint32_t*)kv_sec(d, CAS_KV_SPEC_Q, st);
  w.vd = (const uint32_t*)kv_sec(d, CAS_KV_VER_D, st);
  w.vdidx = (const uint32_t*)kv_sec(d, CAS_KV_VER_D_SBIDX, st);
  w.vres = (const uint32_t*)kv_sec(d, CAS_KV_VER_RES, st);
  w.vresidx = (const uint32_t*)kv_sec(d, CAS_KV_VER_RES_SBIDX, st);
  w.N = 1;
  w.K = n * CAS_BLK;
  w.nbr = (int)n;
  w.nsr = (int)((n + CAS_SB - 1) / CAS_SB);
  w.nsb = w.nsr;
  w.variant = d.variant;
  w.k = d.k;
  w.m = d.m;
  w.rec_sm = d.rec_sm;
  w.rec_q = d.rec_q;
  w.rec_lo = d.rec_lo;
  w.rec_pr = d.rec_pr;
  w.lim_sexp = (uint32_t)(d.variant == 1 ? d.cap_a : 0);
  w.lim_vd = (uint32_t)(d.variant == 2 ? d.cap_a : 0);
  w.lim_vexp = (uint32_t)d.cap_b;
  w.lim_vres = (uint32_t)d.cap_c;
  return w;
}

KvDev make_kv_dev(const cas_kv* kv);
int check_kv(const cas_kv* kv);

}  // namespace cas
