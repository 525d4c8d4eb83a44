"""CPU oracle of the Cassandra bit-level weight / KV split.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package. The
product library (``bit_level_weight_gb300``) never imports it, and this package
never imports the product library; the two share no code.

The bit-level parts (rank table, value pruning, encode, decode, draft values,
matrix-vector products) are plain C in ``cas_oracle.c``, compiled here with gcc
on first use. Attention and the statistics are plain numpy in float64.

Sources: the Cassandra blog review (marsggbo.github.io/blog/2026/20260722-
cassandra), sections 3.1 (value pruning, mantissa truncation, lossless split,
zero-filled draft) and 3.2 (exponent entropy, unary code, MX shared exponent);
the Cassandra paper (arXiv 2605.26558), Fig. 6 (exponent entropy) and Fig. 11
(superblock data management).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cas_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libcas_oracle.so")
_lock = threading.Lock()
_lib = None

BLK = 128
NSEC = 14
# section names, in buffer order (format definition)
SECTIONS = (
    "mask", "spec_sm", "spec_exp", "spec_sbidx", "spec_mx", "spec_q", "ver_lo",
    "ver_d", "ver_d_sbidx", "ver_res", "ver_res_sbidx", "ver_pr", "ver_exp", "ver_sbidx",
)
SPEC_SECTIONS = ("mask", "spec_sm", "spec_exp", "spec_sbidx", "spec_mx", "spec_q")
ORC_OK, ORC_INVALID, ORC_SHAPE, ORC_NONFINITE, ORC_CORRUPT = 0, -1, -2, -3, -7


def build(force: bool = False) -> str:
    """Compile the C oracle (plain -O2, single thread) and return the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int
            lib.orc_exp_hist.argtypes = [P, i64, P]
            lib.orc_rank_table.argtypes = [P, P, P]
            lib.orc_select_block.argtypes = [P, i32, i32, P]
            lib.orc_encode.argtypes = [P, i64, i64, i32, i32, i32, P, P, P, P, P]
            lib.orc_encode.restype = i32
            lib.orc_draft_values.argtypes = [P, i64, i64, i32, i32, i32, P]
            lib.orc_draft_values.restype = i32
            lib.orc_decode.argtypes = [P, P, i64, i64, i32, i32, i32, P, i32, P]
            lib.orc_decode.restype = i32
            lib.orc_matvec.argtypes = [P, i64, i64, P, i32, P, P]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        a = a.view(np.uint16) if a.dtype == np.int16 else a.astype(np.uint16)
    return a


class OracleError(RuntimeError):
    pass


def _check(st: int, what: str):
    if st != ORC_OK:
        raise OracleError(f"{what}: oracle status {st}")


# ------------------------------------------------------------------ exponent statistics
def exp_hist(w) -> np.ndarray:
    """256-bin count of the biased bf16 exponent over every element."""
    w = _u16(w)
    counts = np.zeros(256, np.uint64)
    _L().orc_exp_hist(_p(w), w.size, _p(counts))
    return counts


def rank_table(counts) -> tuple[np.ndarray, np.ndarray]:
    """(exp_of_rank, rank_of_exp): exponents sorted by (count desc, exponent asc)."""
    counts = np.ascontiguousarray(counts, np.uint64)
    eor = np.zeros(256, np.uint8)
    roe = np.zeros(256, np.uint8)
    _L().orc_rank_table(_p(counts), _p(eor), _p(roe))
    return eor, roe


def exp_entropy(counts) -> float:
    """Shannon entropy (bits) of the exponent distribution (blog section 3.2)."""
    c = np.asarray(counts, np.float64)
    p = c[c > 0] / c.sum()
    return float(-(p * np.log2(p)).sum())


def unary_mean_len(counts, rank_of_exp) -> float:
    """Average unary code length sum_e p(e) * (rank(e) + 1) (blog section 3.2)."""
    c = np.asarray(counts, np.float64)
    r = np.asarray(rank_of_exp, np.float64)
    return float((c * (r + 1)).sum() / c.sum())


# ------------------------------------------------------------------ value pruning
def select_block(blk, k: int) -> np.ndarray:
    """Keep mask of one block of any length B (tests use tiny B)."""
    blk = _u16(blk).ravel()
    keep = np.zeros(blk.size, np.uint8)
    _L().orc_select_block(_p(blk), blk.size, k, _p(keep))
    return keep.astype(bool)


# ------------------------------------------------------------------ encode / decode
class Encoded:
    """An oracle-encoded tensor: the whole buffer plus the section table."""

    def __init__(self, buf, off, length, N, K, variant, k, m, exp_of_rank, rank_of_exp):
        self.buf, self.off, self.len = buf, off, length
        self.N, self.K, self.variant, self.k, self.m = N, K, variant, k, m
        self.exp_of_rank, self.rank_of_exp = exp_of_rank, rank_of_exp

    def section(self, name: str) -> np.ndarray:
        i = SECTIONS.index(name)
        return self.buf[self.off[i]: self.off[i] + self.len[i]]

    def spec_bytes(self) -> int:
        return int(sum(self.len[SECTIONS.index(s)] for s in SPEC_SECTIONS))

    def all_bytes(self) -> int:
        return int(sum(self.len))


def encode(W, variant: int, k: int, m: int, rank_of_exp=None, exp_of_rank=None) -> Encoded:
    """Encode a [N][K] bf16 tensor. The rank table defaults to the tensor's own."""
    W = _u16(W)
    if W.ndim != 2:
        raise ValueError("W must be 2-D")
    N, K = W.shape
    if rank_of_exp is None:
        exp_of_rank, rank_of_exp = rank_table(exp_hist(W))
    roe = np.ascontiguousarray(rank_of_exp, np.uint8)
    off = np.zeros(NSEC, np.uint64)
    ln = np.zeros(NSEC, np.uint64)
    total = np.zeros(1, np.uint64)
    L = _L()
    _check(L.orc_encode(_p(W), N, K, variant, k, m, _p(roe), None, _p(off), _p(ln), _p(total)), "encode plan")
    buf = np.zeros(int(total[0]), np.uint8)
    _check(L.orc_encode(_p(W), N, K, variant, k, m, _p(roe), _p(buf), _p(off), _p(ln), _p(total)), "encode")
    return Encoded(buf, off.astype(np.int64), ln.astype(np.int64), N, K, variant, k, m,
                   np.ascontiguousarray(exp_of_rank, np.uint8), roe)


def draft_values(W, variant: int, k: int, m: int) -> np.ndarray:
    """Speculation value of every element, straight from the definition."""
    W = _u16(W)
    N, K = W.shape
    out = np.zeros_like(W)
    _check(_L().orc_draft_values(_p(W), N, K, variant, k, m, _p(out)), "draft_values")
    return out


def decode(enc: Encoded, full: bool) -> np.ndarray:
    """Parse an encoded buffer: draft (full=False) or lossless original (full=True)."""
    out = np.zeros((enc.N, enc.K), np.uint16)
    off = np.ascontiguousarray(enc.off, np.uint64)
    eor = np.ascontiguousarray(enc.exp_of_rank, np.uint8)
    buf = np.ascontiguousarray(enc.buf, np.uint8)
    st = _L().orc_decode(_p(buf), _p(off), enc.N, enc.K, enc.variant, enc.k, enc.m, _p(eor), int(full), _p(out))
    _check(st, "decode")
    return out


# ------------------------------------------------------------------ products
def bf16_to_f64(a) -> np.ndarray:
    a = _u16(a)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def matvec(A, x) -> tuple[np.ndarray, np.ndarray]:
    """y[v][n] = sum_k A[n][k] x[v][k] in double, plus sum_k |A[n][k] x[v][k]|.

    The draft GEMV is matvec(draft_values(W), x); the verify GEMM is matvec(W, X).
    """
    A = _u16(A)
    x = _u16(x)
    if x.ndim == 1:
        x = x[None, :]
    N, K = A.shape
    nvec = x.shape[0]
    assert x.shape[1] == K
    y = np.zeros((nvec, N), np.float64)
    ad = np.zeros((nvec, N), np.float64)
    _L().orc_matvec(_p(A), N, K, _p(np.ascontiguousarray(x)), nvec, _p(y), _p(ad))
    return y, ad


def attention(q, Kc, Vc, causal_new: int = 0):
    """Scaled dot-product attention in float64 with GQA, for one sequence.

    q  : [Tq][Hq][D] bf16 bits (Tq query tokens),
    Kc : [T][Hkv][D] bf16 bits, Vc likewise (T cached tokens, oldest first).
    causal_new = Tq means the last Tq cached tokens are the queries' own tokens:
    query j sees every earlier token and new tokens 0..j. causal_new = 0 means
    every query sees all T tokens.
    Returns (o [Tq][Hq][D] float64, norm [Tq][Hq][D] = sum_t p_t |v_t|).
    Query head h reads kv head h // (Hq / Hkv); scale 1/sqrt(D).
    """
    qf = bf16_to_f64(q)
    Kf = bf16_to_f64(Kc)
    Vf = bf16_to_f64(Vc)
    Tq, Hq, D = qf.shape
    T, Hkv, _ = Kf.shape
    G = Hq // Hkv
    o = np.zeros((Tq, Hq, D))
    nrm = np.zeros((Tq, Hq, D))
    for j in range(Tq):
        visible = T if causal_new == 0 else T - causal_new + j + 1
        for h in range(Hq):
            kh = h // G
            s = Kf[:visible, kh, :] @ qf[j, h, :] / np.sqrt(D)
            s = s - s.max()
            p = np.exp(s)
            p = p / p.sum()
            o[j, h] = p @ Vf[:visible, kh, :]
            nrm[j, h] = p @ np.abs(Vf[:visible, kh, :])
    return o, nrm


# ------------------------------------------------------------------ KV cache
def kv_stream_encode(tokens, variant: int, k: int, m: int, rank_of_exp, exp_of_rank) -> Encoded:
    """One (head, K|V) stream of the KV cache: token t is block t of a single
    row, so a superblock holds 8 consecutive tokens."""
    t = _u16(tokens)
    T, D = t.shape
    assert D == BLK
    return encode(t.reshape(1, T * D), variant, k, m, rank_of_exp, exp_of_rank)


# ------------------------------------------------------------------ exponent code ablation
def huffman_code_lengths(counts) -> np.ndarray:
    """Huffman code length of every exponent with a nonzero count (0 for the
    others): the optimal prefix code the blog review (section 3.2) weighs the
    unary code against - shorter on average, but decoding needs a table over
    2^N bit patterns or a serial parse."""
    import heapq
    c = np.asarray(counts, np.float64)
    lens = np.zeros(c.size, np.int64)
    syms = [i for i in range(c.size) if c[i] > 0]
    if len(syms) == 1:
        lens[syms[0]] = 1
        return lens
    heap = [(c[i], k, [i]) for k, i in enumerate(syms)]
    heapq.heapify(heap)
    tie = len(heap)
    while len(heap) > 1:
        a = heapq.heappop(heap)
        b = heapq.heappop(heap)
        for i in a[2] + b[2]:
            lens[i] += 1
        heapq.heappush(heap, (a[0] + b[0], tie, a[2] + b[2]))
        tie += 1
    return lens


def huffman_mean_len(counts) -> float:
    c = np.asarray(counts, np.float64)
    return float((c * huffman_code_lengths(c)).sum() / c.sum())
