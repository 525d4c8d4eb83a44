/*
 * cas.h - C ABI of libcas, a GB300 (sm_103a) implementation of the Cassandra
 * bit-level split of bf16 weights and KV cache into speculation data (read by
 * the draft) and verification data (which completes the value).
 *
 * Method sources, cited per entry point below:
 *   [B3.1] Cassandra blog review (marsggbo.github.io/blog/2026/20260722-cassandra),
 *          section 3.1 - value pruning and mantissa truncation split every value
 *          into speculation and verification data; the draft zero-fills, the
 *          target merges both losslessly; the draft runs full-size FLOPs and
 *          saves only bandwidth.
 *   [B3.2] same page, section 3.2 - exponent coding: frequency-ranked unary codes
 *          (Cassandra-1, lossless) or MX shared exponents (Cassandra-2).
 *   [B3.3] same page, section 3.3 - the KV cache is produced at inference time
 *          and encoded online.
 *   [F11]  Cassandra paper (arXiv 2605.26558), Fig. 11 - superblock-based data
 *          management.
 *   [ABS]  Cassandra paper abstract - draft built from the most salient values
 *          of weights and KV cache, verified at full precision.
 *
 * Conventions for every entry point:
 *   - Tensors are DEVICE pointers unless stated. bf16 values travel as uint16_t
 *     bit patterns. Row-major. Pointers to bf16 / float data must be 16-byte
 *     aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - The library never allocates or frees device memory. Buffers and
 *     workspaces are owned by the caller; their sizes come from the *_plan /
 *     *_workspace_bytes calls.
 *   - Entry points are asynchronous on `stream` unless marked "synchronises".
 *   - Argument errors return at once and launch nothing. CAS_ERR_CUDA reports a
 *     launch or runtime error. Data errors found on the device while the KV
 *     cache is appended (capacity, non-finite input) are sticky and are read
 *     back by cas_kv_status.
 */
#ifndef CAS_H_
#define CAS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CAS_OK = 0,
  CAS_ERR_INVALID = -1,   /* bad argument (null pointer, range, alignment) */
  CAS_ERR_SHAPE = -2,     /* K (or head_dim) not a multiple of 128          */
  CAS_ERR_NONFINITE = -3, /* NaN or Inf in a tensor to encode               */
  CAS_ERR_CAPACITY = -4,  /* KV cache full (tokens or code stream words)    */
  CAS_ERR_CUDA = -5,      /* CUDA launch / runtime error                     */
  CAS_ERR_BUFFER = -6,    /* buffer or workspace smaller than required       */
  CAS_ERR_CORRUPT = -7,   /* encoded data inconsistent (debug builds)        */
  CAS_ERR_TIMEOUT = -8    /* a bounded device-side wait gave up              */
} cas_status;

/* Encoding parameters of one tensor.
 *   variant        1 = Cassandra-1 (unary exponent codes), 2 = Cassandra-2
 *                  (MX shared exponent per 32 positions) [B3.2]
 *   keep_per_block k in [0,128]: values kept per 128-element block by magnitude
 *                  [B3.1]; cas_keep_from_ratio(r) = floor(128 r + 0.5)
 *   mant_bits      m in [0,7]: mantissa bits the draft keeps [B3.1]          */
typedef struct {
  int32_t variant;
  int32_t keep_per_block;
  int32_t mant_bits;
} cas_params;

/* Section indices of an encoded tensor (one buffer, each section 256-byte
 * aligned, speculation sections first so the draft reads a compact prefix). */
enum {
  CAS_SEC_MASK = 0,        /* u32[nblk][4]: bit p set when position p is kept        */
  CAS_SEC_SPEC_SM,         /* C-1: per block ceil(k(m+1)/32) words, field (s<<m)|f_hi */
  CAS_SEC_SPEC_EXP,        /* C-1: unary codes of kept exponents, MSB-first words     */
  CAS_SEC_SPEC_SBIDX,      /* C-1: u32[nsb+1] word offsets of superblocks             */
  CAS_SEC_SPEC_MX,         /* C-2: u8[nblk][4] shared exponent per 32-position group  */
  CAS_SEC_SPEC_Q,          /* C-2: per block ceil(k(m+2)/32) words, (s<<(m+1))|q      */
  CAS_SEC_VER_LO,          /* C-1: per block ceil(k(7-m)/32) words, cut mantissa bits */
  CAS_SEC_VER_D,           /* C-2: unary codes of exponent distance d, MSB-first      */
  CAS_SEC_VER_D_SBIDX,     /* C-2: u32[nsb+1]                                         */
  CAS_SEC_VER_RES,         /* C-2: residual significand bits, LSB-first               */
  CAS_SEC_VER_RES_SBIDX,   /* C-2: u32[nsb+1]                                         */
  CAS_SEC_VER_PR,          /* both: per block ceil((128-k)/4) words, bytes (s<<7)|f   */
  CAS_SEC_VER_EXP,         /* both: unary codes of pruned exponents, MSB-first        */
  CAS_SEC_VER_SBIDX,       /* both: u32[nsb+1]                                        */
  CAS_NSECT
};

/* Descriptor of one encoded weight tensor W[N][K] (K % 128 == 0). Plain old
 * data, owned by the caller, filled by cas_encode_weights_plan; `base` points
 * into the caller's device buffer once cas_encode_weights has run. A block is
 * 128 consecutive elements of a row; a superblock is 8 consecutive blocks of
 * one row (the last one of a row may be shorter) [F11]. */
typedef struct cas_weights {
  int64_t N, K;
  cas_params p;
  int32_t reserved0;
  uint8_t exp_of_rank[256]; /* rank table, exponents by (count desc, exp asc) */
  uint8_t rank_of_exp[256];
  void* base;               /* device buffer holding every section            */
  uint64_t bytes;           /* bytes of the buffer the sections occupy        */
  uint64_t off[CAS_NSECT];  /* section byte offsets from base                 */
  uint64_t len[CAS_NSECT];  /* section byte lengths                           */
} cas_weights;

const char* cas_status_str(int status);

/* Reads and clears the flags that device code sets: a bounded wait that gave
 * up (a TMA staging copy that did not complete within its spin limit:
 * CAS_ERR_TIMEOUT) and, in a library built with CAS_DEBUG, a superblock index
 * of an encoded tensor that decreases or points past its section
 * (CAS_ERR_CORRUPT; every build clamps such reads to the section, so corrupt
 * data gives wrong values but no read outside the buffer). Synchronises
 * `stream`. Returns CAS_OK, the first flag set, or CAS_ERR_CUDA on a runtime
 * error. */
int cas_device_status(void* stream);
/* Failure-detection test hook, not for production use. The draft GEMV
 * kernels that stage x in shared memory by a bulk copy wait for that copy
 * with a spin limit; on expiry they record CAS_ERR_TIMEOUT (read by
 * cas_device_status), wait once more with the normal limit so the copy lands
 * before the block exits, and write no output. This sets the limit of that
 * first wait for later launches: 0 makes it give up at once, 0xFFFFFFFF
 * restores the normal limit. Synchronises the device; returns CAS_OK or
 * CAS_ERR_CUDA. */
int cas_test_first_wait_spins(uint32_t spins);
/* Launch overlap, process-wide, off by default. When on, the kernels of later
 * calls are launched with programmatic stream serialization: a kernel's
 * thread blocks may start while the previous kernel in the stream is still
 * running, and wait on the device (before touching any global memory) until
 * that kernel has completed and its writes are visible. This hides the gap
 * between back-to-back kernels, e.g. in a captured decode step. Contract while
 * on: the operation enqueued on a stream directly before a libcas call must be
 * a kernel (any kernel) or a libcas call, not a copy, memset or event wait
 * issued by the caller; libcas's own memsets and copies are always followed by
 * plainly launched kernels. Affects launches only (captured graphs keep what
 * they recorded). Returns CAS_OK. */
int cas_set_launch_overlap(int on);
int32_t cas_keep_from_ratio(double ratio);
/* Device-side scratch that cas_encode_weights_plan / cas_encode_weights need
 * for a tensor of N x K (histogram, per-superblock lengths, scan). */
uint64_t cas_encode_workspace_bytes(int64_t N, int64_t K);

/* Plans the encoding of W [B3.1][B3.2]: counts the exponent histogram on the
 * device, builds the rank table (count desc, exponent asc; unseen exponents
 * last), selects the kept values of every block and sizes every section.
 * Fills *desc (base = NULL) and *bytes_needed. Synchronises `stream`.
 * Errors: CAS_ERR_SHAPE if K % 128, CAS_ERR_NONFINITE if W holds NaN/Inf,
 * CAS_ERR_BUFFER if workspace_bytes < cas_encode_workspace_bytes(N, K). */
int cas_encode_weights_plan(const uint16_t* W, int64_t N, int64_t K, cas_params p,
                            cas_weights* desc, uint64_t* bytes_needed, void* workspace,
                            uint64_t workspace_bytes, void* stream);

/* Writes every section of W into buf (>= desc->bytes bytes, 256-byte aligned)
 * with the rank table in *desc, sets desc->base = buf. Asynchronous. The same
 * W and workspace as the plan must be passed. Output is byte-identical to the
 * format definition (padding bits zero). */
int cas_encode_weights(const uint16_t* W, cas_weights* desc, void* buf, uint64_t buf_bytes,
                       void* workspace, uint64_t workspace_bytes, void* stream);

/* Per-tensor choice between Cassandra-1 and Cassandra-2 [B3.2]: plans W under
 * both variants with the same k and m (as cas_encode_weights_plan, which it
 * calls twice; synchronises `stream`) and sets *variant to the one whose
 * speculation sections (mask, records, exponent codes or shared exponents,
 * index) are smaller; ties go to Cassandra-1, whose draft keeps every kept
 * value's own exponent. spec_bytes (NULL or 2 entries) receives both sizes,
 * Cassandra-1 first. Errors: those of cas_encode_weights_plan;
 * CAS_ERR_INVALID if variant is NULL. */
int cas_choose_variant(const uint16_t* W, int64_t N, int64_t K, int keep_per_block, int mant_bits,
                       void* workspace, uint64_t workspace_bytes, int* variant, uint64_t* spec_bytes,
                       void* stream);

/* Draft GEMV [B3.1]: y[v][n] = sum_k D(W)[n][k] * x[v][k] for v < nvec (1..4),
 * where D(W) is the zero-filled speculation value (pruned -> 0, kept ->
 * mantissa truncated, Cassandra-2 -> shared-exponent grid). Reads only the
 * speculation sections. x: bf16 [nvec][K]; y: fp32 [nvec][N], overwritten.
 * fp32 accumulation; summation order is unspecified. Errors: those of the
 * descriptor check (CAS_ERR_INVALID, CAS_ERR_SHAPE); CAS_ERR_INVALID if nvec
 * is outside 1..4, x or y is null or not 16-byte aligned, nvec * K * 2 bytes
 * exceed 200 KiB (x is staged whole in shared memory) or the tensor has 2^30
 * superblocks or more; CAS_ERR_CUDA on a launch error. N = 0 writes nothing. */
int cas_draft_gemv(const cas_weights* W, const uint16_t* x, int nvec, float* y, void* stream);

/* Draft GEMV that adds into y: y[v][n] += sum_k D(W)[n][k] * x[v][k], y not
 * cleared (a residual stream can be y). Same arguments and errors as
 * cas_draft_gemv. */
int cas_draft_gemv_accumulate(const cas_weights* W, const uint16_t* x, int nvec, float* y, void* stream);

/* Draft GEMV of a normalised input [B3.1]: xn[v] = bf16(x[v] / sqrt(mean(x[v]^2)
 * + eps) * gamma) (RMSNorm, as cas_add_rmsnorm without the add; the mean of
 * squares is reduced in an unspecified order) and y[v][n] = sum_k
 * D(W)[n][k] * xn[v][k], overwriting y. x: fp32 [nvec][K], 16-byte aligned,
 * not written; gamma: bf16 [K]; xn: bf16 [nvec][K] out, 16-byte aligned,
 * written by the call (the normalisation runs inside the GEMV's staging of
 * x where the lane-per-block kernel takes the tensor, else as a separate
 * kernel first). Errors: those of cas_draft_gemv; CAS_ERR_INVALID if x,
 * gamma or xn is null or misaligned, eps is negative or NaN, or K exceeds
 * 16384. N = 0 still writes xn. */
int cas_draft_gemv_rmsnorm(const cas_weights* W, const float* x, int nvec, const uint16_t* gamma, float eps,
                           uint16_t* xn, float* y, void* stream);

/* Input transforms of cas_draft_gemv_f32 (the forward operation that produces
 * a matrix product's bf16 input in the evaluated models). */
enum {
  CAS_X_ROUND = 0,    /* xn = bf16(x), as cas_f32_to_bf16; x: fp32 [nvec][K]            */
  CAS_X_RMSNORM = 1,  /* xn = bf16(rmsnorm(x) * gamma), as cas_draft_gemv_rmsnorm       */
  CAS_X_SILU_MUL = 2  /* xn = bf16(silu(g) * u), as cas_silu_mul; x: fp32 [nvec][2K], g
                         the first K and u the last K values of a row (fused gate|up)  */
};
/* Draft GEMV of an fp32 input [B3.1] with the transform `op` applied while
 * the GEMV stages x (where the lane-per-block kernel takes the tensor; else a
 * separate glue kernel writes xn first): xn[v] = the transformed bf16 input,
 * written by the call (bit-identical to the glue kernel's output for
 * CAS_X_ROUND and CAS_X_SILU_MUL), and y[v][n] = sum_k D(W)[n][k] * xn[v][k],
 * overwriting y, or added to y when `accumulate` is non-zero (y not cleared;
 * a residual stream can be y). gamma: bf16 [K], used by CAS_X_RMSNORM only
 * (may be NULL otherwise). x, xn, y 16-byte aligned; x is not written.
 * Errors: those of cas_draft_gemv; CAS_ERR_INVALID for an unknown op, a null
 * or misaligned x or xn, a missing gamma or a negative / NaN eps with
 * CAS_X_RMSNORM, or K above 16384. N = 0 still writes xn. */
int cas_draft_gemv_f32(const cas_weights* W, const float* x, int nvec, int op, const uint16_t* gamma, float eps,
                       uint16_t* xn, float* y, int accumulate, void* stream);

/* Verify GEMM [B3.1]: Y[t][n] = sum_k W[n][k] * X[t][k] for t < T (1..16)
 * with W rebuilt bit-exactly from both streams, on tensor cores with fp32
 * accumulation. X: bf16 [T][K]; Y: fp32 [T][N], overwritten. Errors: those
 * of the descriptor check (CAS_ERR_INVALID, CAS_ERR_SHAPE); CAS_ERR_INVALID if
 * T is outside 1..16 or X or Y is null or not 16-byte aligned; CAS_ERR_CUDA on
 * a launch error. N = 0 writes nothing. */
int cas_verify_gemm(const cas_weights* W, const uint16_t* X, int T, float* Y, void* stream);
/* Verify GEMM that adds into Y: Y[t][n] += sum_k W[n][k] * X[t][k], Y not
 * cleared (a residual stream can be Y). Same arguments and errors as
 * cas_verify_gemm. */
int cas_verify_gemm_accumulate(const cas_weights* W, const uint16_t* X, int T, float* Y, void* stream);

/* Materialises the draft values D(W) as bf16 [N][K] (test path) [B3.1].
 * Errors: those of the descriptor check; CAS_ERR_INVALID if out is null or
 * not 16-byte aligned (an empty tensor writes nothing); CAS_ERR_CUDA. */
int cas_decode_draft(const cas_weights* W, uint16_t* out, void* stream);
/* Rebuilds the original bf16 bits of W [N][K] from both streams [B3.1].
 * Errors as cas_decode_draft. */
int cas_reconstruct(const cas_weights* W, uint16_t* out, void* stream);

/* ------------------------------------------------------------------ KV cache
 * One cas_kv holds the K and V cache of one (sequence, layer): n_kv_heads
 * heads of head_dim 128, one 128-element block per token, head and K|V.
 * Each (head, K|V) stream has its own rank table, counted over calibration
 * tokens and then frozen [B3.3]. A KV superblock is 8 consecutive tokens of
 * one stream. Either variant: Cassandra-1 (unary exponent codes) or
 * Cassandra-2 (shared exponent per 32 dimensions of a token).
 * Every KV entry point first checks the descriptor: CAS_ERR_INVALID for a
 * null kv or base, n_kv_heads < 1, head_dim != 128 or parameters out of
 * range.
 * The device state (n_tokens, per-stream code tails, sticky status) lives in
 * the caller's buffer, so appends, truncations and attention calls need no
 * host round trip. */
/* Sections of a KV buffer. Streams are numbered kv * n_kv_heads + head
 * (kv 0 = K, 1 = V); section i of stream st starts at off[i] + st * stride[i].
 * STATE holds the device state: int64 n_tokens, int32 sticky status, two
 * internal counters, then three u64 code tails per stream, [3][S] with
 * S = 2 * n_kv_heads: the kept-value unary stream (Cassandra-1 exponents,
 * Cassandra-2 distances d), the pruned-exponent unary stream and the
 * Cassandra-2 residual stream. TABLES holds per stream exp_of_rank[256] then
 * rank_of_exp[256]. The other sections are those of an encoded weight tensor
 * with one row per stream and one block per token, sized for max_tokens;
 * sections the variant does not use have stride 0. */
enum {
  CAS_KV_STATE = 0,
  CAS_KV_TABLES,
  CAS_KV_MASK,
  CAS_KV_SPEC_SM,
  CAS_KV_SPEC_EXP,
  CAS_KV_SPEC_SBIDX,
  CAS_KV_VER_LO,
  CAS_KV_VER_PR,
  CAS_KV_VER_EXP,
  CAS_KV_VER_SBIDX,
  CAS_KV_SPEC_MX,
  CAS_KV_SPEC_Q,
  CAS_KV_VER_D,
  CAS_KV_VER_D_SBIDX,
  CAS_KV_VER_RES,
  CAS_KV_VER_RES_SBIDX,
  CAS_KV_NSECT
};

typedef struct cas_kv {
  int32_t n_kv_heads, head_dim;
  cas_params p;
  int64_t max_tokens;
  uint64_t cap_spec_words;  /* kept-value unary stream capacity per stream, u32 words */
  uint64_t cap_ver_words;   /* pruned-exponent unary stream capacity per stream */
  void* base;               /* device buffer */
  uint64_t bytes;
  uint64_t off[16];         /* section offsets (see cas_kv_plan)          */
  uint64_t stride[16];      /* bytes between consecutive streams          */
} cas_kv;

/* Bytes of device buffer one cas_kv needs: est_bits_per_code is the planned
 * mean unary code length of the unary streams; each stream gets that many bits
 * per code plus one word of alignment slack per superblock (the Cassandra-2
 * residual stream is sized for its worst case, 8 bits per kept value). Pruned (small)
 * values have more spread exponents and longer codes than kept ones: on
 * N(0,1) x LogNormal(0,0.5) K/V with k = 64 they average about 4 to 5 bits,
 * so 6.0 leaves room; an append that would overflow sets CAS_ERR_CAPACITY.
 * Errors: CAS_ERR_INVALID for a null bytes, n_kv_heads < 1, max_tokens < 1,
 * parameters out of range or an estimate outside (0, 256] bits. */
int cas_kv_plan(int n_kv_heads, int64_t max_tokens, cas_params p, double est_bits_per_code,
                uint64_t* bytes);

/* Lays out *kv in buf and builds the rank table of each (head, K|V) stream from
 * the n_calib calibration tokens calib_k / calib_v (bf16 [n_calib][H][128]).
 * The cache starts empty (n_tokens = 0); calibration tokens are not appended.
 * Synchronises `stream`. Errors: CAS_ERR_INVALID for bad layout arguments (as
 * cas_kv_plan), a buf not 256-byte aligned, n_calib < 0 or null / misaligned
 * calibration tokens; CAS_ERR_BUFFER if bytes is below the plan;
 * CAS_ERR_NONFINITE for NaN/Inf calibration; CAS_ERR_CUDA. */
int cas_kv_init(cas_kv* kv, void* buf, uint64_t bytes, int n_kv_heads, int64_t max_tokens,
                cas_params p, double est_bits_per_code, const uint16_t* calib_k,
                const uint16_t* calib_v, int64_t n_calib, void* stream);

/* Online KV encoding [B3.3]: appends T tokens, k_new / v_new bf16 [T][H][128],
 * in order. On the device: if the tokens or code words would exceed capacity,
 * or a value is NaN/Inf, nothing is written and the sticky status is set.
 * Errors at the call: CAS_ERR_INVALID for T < 0 or null / misaligned tokens
 * (T = 0 does nothing); CAS_ERR_CUDA. */
int cas_encode_kv_append(cas_kv* kv, const uint16_t* k_new, const uint16_t* v_new, int T,
                         void* stream);

/* Rolls the cache back to its first n_tokens tokens (rejected draft tokens).
 * n_tokens larger than the current count leaves the cache unchanged.
 * Errors: CAS_ERR_INVALID for n_tokens < 0; CAS_ERR_CUDA. */
int cas_kv_truncate(cas_kv* kv, int64_t n_tokens, void* stream);
/* cas_kv_truncate of every cache kvs[0..count) to n_tokens, in one launch per
 * variant (up to 80 caches a launch), e.g. the rollback of all layers at the
 * end of a decode step. The caches must be distinct. Errors: CAS_ERR_INVALID
 * for count < 0, a null array with count > 0 or n_tokens < 0; the
 * descriptor check's errors for any cache; CAS_ERR_CUDA. count = 0 does
 * nothing. */
int cas_kv_truncate_many(cas_kv* const* kvs, int count, int64_t n_tokens, void* stream);

/* Reads the device state. Synchronises `stream`. Returns the sticky device
 * status (CAS_OK, CAS_ERR_CAPACITY or CAS_ERR_NONFINITE) and the token count. */
int cas_kv_status(const cas_kv* kv, int64_t* n_tokens, void* stream);

/* Clears the sticky device status. Errors: CAS_ERR_CUDA. */
int cas_kv_clear_status(cas_kv* kv, void* stream);

/* Workspace bytes of cas_draft_attn_decode / cas_verify_attn for a batch. */
uint64_t cas_attn_workspace_bytes(int batch, int n_q_heads, int T, int64_t max_tokens);

/* Draft attention decode [B3.1][B3.3]: for each sequence b and query head h,
 * o = softmax(q K~^T / sqrt(128)) V~ over the speculation KV of kv[b] (pruned
 * entries zero, kept mantissas truncated) followed by n_tail exact bf16 tail
 * tokens (the draft tokens of this step). GQA: head h reads kv head
 * h / (n_q_heads / n_kv_heads). q: bf16 [batch][n_q_heads][128];
 * tail_k, tail_v: bf16 [batch][n_tail][n_kv_heads][128] (NULL when n_tail = 0);
 * o: fp32 [batch][n_q_heads][128]. Softmax in fp32. Errors: CAS_ERR_INVALID
 * for batch outside 1..8, null or misaligned q / o, n_tail outside 0..16 (or
 * null tails with n_tail > 0), caches that differ in n_kv_heads, k or m, or
 * n_q_heads not a multiple of n_kv_heads with at most 64 query vectors per kv
 * head; CAS_ERR_BUFFER if the workspace is null, misaligned or smaller than
 * cas_attn_workspace_bytes; CAS_ERR_CUDA. */
int cas_draft_attn_decode(const cas_kv* const* kv, int batch, const uint16_t* q, int n_q_heads,
                          const uint16_t* tail_k, const uint16_t* tail_v, int n_tail, float* o,
                          void* workspace, uint64_t workspace_bytes, void* stream);

/* Draft attention decode that allocates nothing and takes no workspace. The
 * paper has no counterpart: this entry point is for callers that cannot
 * allocate device memory when they decode (a runtime whose memory plan is
 * fixed at start-up, or an application that owns every allocation and passes
 * only inputs and outputs). Arguments and result are those of
 * cas_draft_attn_decode. The chunk partials live in one fixed 8 MiB array in
 * the library's device image (held by every GPU that loads the library until
 * the process exits); the call returns CAS_ERR_BUFFER, without launching, when
 * batch * n_q_heads * ceil(max_tokens / 256) * 520 bytes exceeds 8 MiB (e.g.
 * batch 1 with 32 query heads reaches 128K tokens). Every call looks up the
 * array's device address in the calling thread's current context (the device
 * and context the caller has made current), so a rebuilt context is
 * followed; the first call in a context may load the library's device code,
 * so make it before any stream capture. Every call uses the same array, so
 * calls that overlap on the GPU (on different streams, or on streams not
 * ordered with each other) race; calls ordered on one stream do not. The
 * array keeps the last call's partials; each call writes every partial it
 * reads, so no clearing is needed. */
int cas_draft_attn_decode_noalloc(const cas_kv* const* kv, int batch, const uint16_t* q, int n_q_heads,
                                  const uint16_t* tail_k, const uint16_t* tail_v, int n_tail, float* o,
                                  void* stream);

/* Verify attention [B3.1]: T query tokens per sequence over the exact KV
 * (both streams merged), the T queries being the last T tokens of the cache:
 * query j sees every earlier token and the new tokens 0..j.
 * q: bf16 [batch][T][n_q_heads][128]; o: fp32 [batch][T][n_q_heads][128].
 * Errors as cas_draft_attn_decode, with T outside 1..16 also CAS_ERR_INVALID
 * and T * n_q_heads / n_kv_heads at most 64. */
int cas_verify_attn(const cas_kv* const* kv, int batch, const uint16_t* q, int T, int n_q_heads,
                    float* o, void* workspace, uint64_t workspace_bytes, void* stream);

/* ---- Forward-pass glue. The operations between the matrix products of one
 * decode step of the models the method is evaluated on (Llama-3-8B,
 * Qwen3-8B: Cassandra paper, evaluation; Cassandra blog review, section 4),
 * so that a step runs as a data-dependent forward through this library. All
 * asynchronous on `stream`; fp32 arithmetic; bf16 outputs rounded to nearest
 * even; CAS_ERR_INVALID for a null pointer or a size out of range (nothing
 * launched), CAS_ERR_CUDA for a launch error; rows == 0 does nothing. */

/* Residual add fused with RMSNorm: for each of `rows` rows of dim fp32,
 * x += y (skipped when y is NULL), then
 * out = bf16(x / sqrt(mean(x^2) + eps) * gamma). x: fp32 [rows][dim], updated
 * in place; y: fp32 [rows][dim] or NULL; gamma: bf16 [dim]; out: bf16
 * [rows][dim]; dim at most 16384. */
int cas_add_rmsnorm(float* x, const float* y, int rows, int dim, const uint16_t* gamma, float eps,
                    uint16_t* out, void* stream);

/* Split of a fused QKV product with rotary position embedding (head_dim
 * 128). qkv: fp32 [rows][(n_q_heads + 2 n_kv_heads) * 128], q heads then k
 * heads then v heads. Row r has position p = pos0 + r % rows_per_seq; in
 * every q and k head the pair (i, i + 64), i < 64, turns by the angle
 * p * theta^(-i/64): (a, b) -> (a cos - b sin, b cos + a sin), the angle
 * formed in double precision. Outputs bf16: q [rows][n_q_heads][128]; k and v
 * rows of n_kv_heads * 128 values at strides k_row_stride / v_row_stride
 * elements (at least n_kv_heads * 128), so rows can land in a KV tail buffer.
 * theta must exceed 1. */
int cas_rope_split(const float* qkv, int rows, int n_q_heads, int n_kv_heads, int64_t pos0, int rows_per_seq,
                   double theta, uint16_t* q, uint16_t* k, int64_t k_row_stride, uint16_t* v,
                   int64_t v_row_stride, void* stream);

/* out = bf16(silu(gate) * up) with silu(g) = g / (1 + exp(-g)); gate_up:
 * fp32 [rows][2 ffn] (gate then up, the fused gate|up product); out: bf16
 * [rows][ffn]. */
int cas_silu_mul(const float* gate_up, int rows, int ffn, uint16_t* out, void* stream);

/* out = bf16(in) for n values (e.g. an attention output before the output
 * projection). */
int cas_f32_to_bf16(const float* in, int64_t n, uint16_t* out, void* stream);

/* Greedy decoding: out[r] = the lowest index of the largest of the `vocab`
 * fp32 logits of row r (NaN never wins). logits: [rows][vocab]; out: int32
 * [rows]. vocab at most 2^31 - 1. */
int cas_argmax(const float* logits, int rows, int64_t vocab, int32_t* out, void* stream);

/* Embedding lookup: x[r] = fp32(table[tokens[r]]); table: bf16 [vocab][dim];
 * x: fp32 [rows][dim]. A token id outside [0, vocab) reads the nearest valid
 * row (the device cannot report it). */
int cas_embed(const int32_t* tokens, int rows, const uint16_t* table, int64_t vocab, int dim, float* x,
              void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CAS_H_ */
