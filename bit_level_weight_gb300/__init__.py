"""bit_level_weight_gb300 - Python binding of libcas (Cassandra bit-level split on GB300).

Thin ctypes marshalling over the C ABI declared in ``include/cas.h``: every
function here has the name of the C entry point it calls, converts torch
tensors to device pointers and the current torch stream to a cudaStream_t,
and raises ``CasError`` on a non-zero status. All computation happens in the
CUDA kernels of ``libcas.so``; there is no Python or CPU fallback, and a
missing library is an error.

PyTorch is used only for device memory (buffers, workspaces) and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcas.so")

NSECT = 14
SECTIONS = (
    "mask", "spec_sm", "spec_exp", "spec_sbidx", "spec_mx", "spec_q", "ver_lo",
    "ver_d", "ver_d_sbidx", "ver_res", "ver_res_sbidx", "ver_pr", "ver_exp", "ver_sbidx",
)
SPEC_SECTIONS = ("mask", "spec_sm", "spec_exp", "spec_sbidx", "spec_mx", "spec_q")
KV_SECTIONS = ("state", "tables", "mask", "spec_sm", "spec_exp", "spec_sbidx", "ver_lo", "ver_pr",
               "ver_exp", "ver_sbidx", "spec_mx", "spec_q", "ver_d", "ver_d_sbidx", "ver_res", "ver_res_sbidx")

CAS_OK = 0


class CasError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status})")


class cas_params(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("keep_per_block", ctypes.c_int32), ("mant_bits", ctypes.c_int32)]


class cas_weights(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("p", cas_params), ("reserved0", ctypes.c_int32),
        ("exp_of_rank", ctypes.c_uint8 * 256), ("rank_of_exp", ctypes.c_uint8 * 256),
        ("base", ctypes.c_void_p), ("bytes", ctypes.c_uint64),
        ("off", ctypes.c_uint64 * NSECT), ("len", ctypes.c_uint64 * NSECT),
    ]


class cas_kv(ctypes.Structure):
    _fields_ = [
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("p", cas_params),
        ("max_tokens", ctypes.c_int64), ("cap_spec_words", ctypes.c_uint64), ("cap_ver_words", ctypes.c_uint64),
        ("base", ctypes.c_void_p), ("bytes", ctypes.c_uint64),
        ("off", ctypes.c_uint64 * 16), ("stride", ctypes.c_uint64 * 16),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libcas.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libcas.so not built at {LIB_PATH}; run bit_level_weight_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
        sig = {
            "cas_status_str": ([i32], ctypes.c_char_p),
            "cas_keep_from_ratio": ([ctypes.c_double], ctypes.c_int32),
            "cas_encode_workspace_bytes": ([i64, i64], u64),
            "cas_encode_weights_plan": ([P, i64, i64, cas_params, P, P, P, u64, P], i32),
            "cas_encode_weights": ([P, P, P, u64, P, u64, P], i32),
            "cas_choose_variant": ([P, i64, i64, i32, i32, P, u64, P, P, P], i32),
            "cas_draft_gemv": ([P, P, i32, P, P], i32),
            "cas_draft_gemv_accumulate": ([P, P, i32, P, P], i32),
            "cas_draft_gemv_rmsnorm": ([P, P, i32, P, ctypes.c_float, P, P, P], i32),
            "cas_draft_gemv_f32": ([P, P, i32, i32, P, ctypes.c_float, P, P, i32, P], i32),
            "cas_verify_gemm": ([P, P, i32, P, P], i32),
            "cas_verify_gemm_accumulate": ([P, P, i32, P, P], i32),
            "cas_decode_draft": ([P, P, P], i32),
            "cas_reconstruct": ([P, P, P], i32),
            "cas_kv_plan": ([i32, i64, cas_params, ctypes.c_double, P], i32),
            "cas_kv_init": ([P, P, u64, i32, i64, cas_params, ctypes.c_double, P, P, i64, P], i32),
            "cas_encode_kv_append": ([P, P, P, i32, P], i32),
            "cas_kv_truncate": ([P, i64, P], i32),
            "cas_kv_truncate_many": ([P, i32, i64, P], i32),
            "cas_kv_status": ([P, P, P], i32),
            "cas_kv_clear_status": ([P, P], i32),
            "cas_attn_workspace_bytes": ([i32, i32, i32, i64], u64),
            "cas_draft_attn_decode": ([P, i32, P, i32, P, P, i32, P, P, u64, P], i32),
            "cas_verify_attn": ([P, i32, P, i32, i32, P, P, u64, P], i32),
            "cas_device_status": ([P], i32),
            "cas_test_first_wait_spins": ([ctypes.c_uint32], i32),
            "cas_set_launch_overlap": ([i32], i32),
            "cas_add_rmsnorm": ([P, P, i32, i32, P, ctypes.c_float, P, P], i32),
            "cas_rope_split": ([P, i32, i32, i32, i64, i32, ctypes.c_double, P, P, i64, P, i64, P], i32),
            "cas_silu_mul": ([P, i32, i32, P, P], i32),
            "cas_f32_to_bf16": ([P, i64, P, P], i32),
            "cas_argmax": ([P, i32, i64, P, P], i32),
            "cas_embed": ([P, i32, P, i64, i32, P, P], i32),
            "cas_draft_attn_decode_noalloc": ([P, i32, P, i32, P, P, i32, P, P], i32),
        }
        for name, (args, res) in sig.items():
            if hasattr(L, name):
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
        _lib = L
    return _lib


def status_str(s: int) -> str:
    try:
        return lib().cas_status_str(int(s)).decode()
    except Exception:  # noqa: BLE001
        return "status"


def _check(s: int, what: str):
    if s != CAS_OK:
        raise CasError(s, what)


def _stream(stream=None) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_cuda:
        raise ValueError("libcas takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libcas takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _bits(t: torch.Tensor) -> torch.Tensor:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype not in (torch.int16, torch.uint16):
        raise ValueError("bf16 data must be bfloat16 or int16 bit patterns")
    return t


def _shape(t: torch.Tensor, shape: tuple, what: str):
    """Raises unless t has exactly `shape` (the C ABI takes sizes on trust)."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _out(t: torch.Tensor, n: int, dtypes: tuple, what: str):
    """Raises unless the output t holds exactly n elements of one of dtypes."""
    if t.dtype not in dtypes:
        raise ValueError(f"{what}: dtype {t.dtype}, expected one of {dtypes}")
    if t.numel() != n:
        raise ValueError(f"{what}: {t.numel()} elements, expected {n}")


def params(variant: int = 1, keep_per_block: int = 64, mant_bits: int = 3) -> cas_params:
    return cas_params(variant, keep_per_block, mant_bits)


def cas_keep_from_ratio(r: float) -> int:
    return int(lib().cas_keep_from_ratio(float(r)))


# ------------------------------------------------------------------ weights
class EncodedWeights:
    """An encoded tensor: the descriptor plus the torch buffer it points into."""

    def __init__(self, desc: cas_weights, buf: torch.Tensor):
        self.desc, self.buf = desc, buf

    @property
    def N(self):
        return self.desc.N

    @property
    def K(self):
        return self.desc.K

    def section(self, name: str) -> torch.Tensor:
        i = SECTIONS.index(name)
        o, n = int(self.desc.off[i]), int(self.desc.len[i])
        return self.buf[o:o + n]

    def spec_bytes(self) -> int:
        return sum(int(self.desc.len[SECTIONS.index(s)]) for s in SPEC_SECTIONS)

    def all_bytes(self) -> int:
        return sum(int(self.desc.len[i]) for i in range(NSECT))

    def exp_of_rank(self):
        return bytes(self.desc.exp_of_rank)


def cas_encode_workspace_bytes(N: int, K: int) -> int:
    return int(lib().cas_encode_workspace_bytes(N, K))


def cas_encode_weights_plan(W: torch.Tensor, p: cas_params, workspace: torch.Tensor, stream=None):
    """Returns (desc, bytes_needed). Synchronises the stream."""
    W = _bits(W)
    N, K = W.shape
    desc = cas_weights()
    need = ctypes.c_uint64(0)
    _check(lib().cas_encode_weights_plan(_ptr(W), N, K, p, ctypes.byref(desc), ctypes.byref(need),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream)), "cas_encode_weights_plan")
    return desc, int(need.value)


def cas_encode_weights(W: torch.Tensor, desc: cas_weights, buf: torch.Tensor, workspace: torch.Tensor, stream=None):
    W = _bits(W)
    _check(lib().cas_encode_weights(_ptr(W), ctypes.byref(desc), _ptr(buf), buf.numel() * buf.element_size(),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "cas_encode_weights")


def cas_choose_variant(W: torch.Tensor, keep_per_block: int = 64, mant_bits: int = 3, stream=None):
    """(variant, (cassandra1_spec_bytes, cassandra2_spec_bytes)) for W [N][K]."""
    W = _bits(W).contiguous()
    N, K = W.shape
    ws = torch.empty(max(cas_encode_workspace_bytes(N, K), 256), dtype=torch.uint8, device=W.device)
    v = ctypes.c_int(0)
    sb = (ctypes.c_uint64 * 2)()
    _check(lib().cas_choose_variant(_ptr(W), N, K, keep_per_block, mant_bits, _ptr(ws), ws.numel(),
                                    ctypes.byref(v), sb, _stream(stream)), "cas_choose_variant")
    return int(v.value), (int(sb[0]), int(sb[1]))


def encode_weights(W: torch.Tensor, variant: int = 1, keep_per_block: int = 64, mant_bits: int = 3,
                   stream=None) -> EncodedWeights:
    """Plan, allocate (torch) and encode W [N][K] on its device."""
    W = _bits(W).contiguous()
    N, K = W.shape
    ws = torch.empty(max(cas_encode_workspace_bytes(N, K), 256), dtype=torch.uint8, device=W.device)
    desc, need = cas_encode_weights_plan(W, params(variant, keep_per_block, mant_bits), ws, stream)
    buf = torch.empty(max(need, 256), dtype=torch.uint8, device=W.device)
    cas_encode_weights(W, desc, buf, ws, stream)
    return EncodedWeights(desc, buf)


def cas_draft_gemv(W: EncodedWeights, x: torch.Tensor, y: torch.Tensor, stream=None):
    x = _bits(x)
    nvec = 1 if x.dim() == 1 else x.shape[0]
    _shape(x, (W.K,) if x.dim() == 1 else (nvec, W.K), "x")
    _out(y, nvec * W.N, (torch.float32,), "y")
    _check(lib().cas_draft_gemv(ctypes.byref(W.desc), _ptr(x), nvec, _ptr(y), _stream(stream)), "cas_draft_gemv")
    return y


def cas_draft_gemv_accumulate(W: EncodedWeights, x: torch.Tensor, y: torch.Tensor, stream=None):
    """y += D(W) x (y not cleared)."""
    x = _bits(x)
    nvec = 1 if x.dim() == 1 else x.shape[0]
    _shape(x, (W.K,) if x.dim() == 1 else (nvec, W.K), "x")
    _out(y, nvec * W.N, (torch.float32,), "y")
    _check(lib().cas_draft_gemv_accumulate(ctypes.byref(W.desc), _ptr(x), nvec, _ptr(y), _stream(stream)),
           "cas_draft_gemv_accumulate")
    return y


def draft_gemv_rmsnorm(W: EncodedWeights, x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-5,
                       xn: torch.Tensor | None = None, y: torch.Tensor | None = None, stream=None):
    """xn = bf16 rmsnorm(x) * gamma, y = D(W) xn; x: fp32 [nvec][K]. Returns (xn, y)."""
    if x.dtype != torch.float32 or x.dim() != 2 or x.shape[1] != W.K:
        raise ValueError("draft_gemv_rmsnorm: x must be fp32 [nvec][K]")
    nvec = x.shape[0]
    gamma = _bits(gamma)
    _shape(gamma, (W.K,), "gamma")
    if xn is None:
        xn = torch.empty(nvec, W.K, dtype=torch.int16, device=x.device)
    if y is None:
        y = torch.empty(nvec, W.N, dtype=torch.float32, device=x.device)
    _out(xn, nvec * W.K, (torch.int16, torch.bfloat16), "xn")
    _out(y, nvec * W.N, (torch.float32,), "y")
    _check(lib().cas_draft_gemv_rmsnorm(ctypes.byref(W.desc), _ptr(x), nvec, _ptr(gamma), float(eps), _ptr(xn),
                                        _ptr(y), _stream(stream)), "cas_draft_gemv_rmsnorm")
    return xn, y


X_ROUND, X_RMSNORM, X_SILU_MUL = 0, 1, 2  # input transforms of cas_draft_gemv_f32


def draft_gemv_f32(W: EncodedWeights, x: torch.Tensor, op: int, gamma: torch.Tensor | None = None,
                   eps: float = 1e-5, xn: torch.Tensor | None = None, y: torch.Tensor | None = None,
                   accumulate: bool = False, stream=None):
    """xn = the bf16 input made from fp32 x by `op` (X_ROUND: bf16(x); X_RMSNORM:
    bf16(rmsnorm(x) * gamma); X_SILU_MUL: bf16(silu(g) * u) of rows [g | u] of
    2K values), y = D(W) xn (added to y with accumulate). Returns (xn, y)."""
    if op not in (X_ROUND, X_RMSNORM, X_SILU_MUL):
        raise ValueError("draft_gemv_f32: unknown op")
    width = 2 * W.K if op == X_SILU_MUL else W.K
    if x.dtype != torch.float32 or x.dim() != 2 or x.shape[1] != width or not x.is_contiguous():
        raise ValueError(f"draft_gemv_f32: x must be contiguous fp32 [nvec][{width}]")
    nvec = x.shape[0]
    if op == X_RMSNORM:
        if gamma is None:
            raise ValueError("draft_gemv_f32: X_RMSNORM needs gamma")
        gamma = _bits(gamma)
        _shape(gamma, (W.K,), "gamma")
    if xn is None:
        xn = torch.empty(nvec, W.K, dtype=torch.int16, device=x.device)
    if y is None:
        if accumulate:
            raise ValueError("draft_gemv_f32: accumulate needs y")
        y = torch.empty(nvec, W.N, dtype=torch.float32, device=x.device)
    _out(xn, nvec * W.K, (torch.int16, torch.bfloat16), "xn")
    _out(y, nvec * W.N, (torch.float32,), "y")
    _check(lib().cas_draft_gemv_f32(ctypes.byref(W.desc), _ptr(x), nvec, op, _ptr(gamma) if op == X_RMSNORM else None,
                                    float(eps), _ptr(xn), _ptr(y), 1 if accumulate else 0, _stream(stream)),
           "cas_draft_gemv_f32")
    return xn, y


def cas_verify_gemm(W: EncodedWeights, X: torch.Tensor, Y: torch.Tensor, stream=None):
    X = _bits(X)
    T = 1 if X.dim() == 1 else X.shape[0]
    _shape(X, (W.K,) if X.dim() == 1 else (T, W.K), "X")
    _out(Y, T * W.N, (torch.float32,), "Y")
    _check(lib().cas_verify_gemm(ctypes.byref(W.desc), _ptr(X), T, _ptr(Y), _stream(stream)), "cas_verify_gemm")
    return Y


def cas_decode_draft(W: EncodedWeights, out: torch.Tensor, stream=None):
    _out(out, W.N * W.K, (torch.int16, torch.uint16, torch.bfloat16), "out")
    _check(lib().cas_decode_draft(ctypes.byref(W.desc), _ptr(out), _stream(stream)), "cas_decode_draft")
    return out


def cas_reconstruct(W: EncodedWeights, out: torch.Tensor, stream=None):
    _out(out, W.N * W.K, (torch.int16, torch.uint16, torch.bfloat16), "out")
    _check(lib().cas_reconstruct(ctypes.byref(W.desc), _ptr(out), _stream(stream)), "cas_reconstruct")
    return out


def draft_gemv(W: EncodedWeights, x: torch.Tensor) -> torch.Tensor:
    nvec = 1 if x.dim() == 1 else x.shape[0]
    y = torch.empty(nvec, W.N, dtype=torch.float32, device=x.device)
    return cas_draft_gemv(W, x, y)


def cas_verify_gemm_accumulate(W: EncodedWeights, X: torch.Tensor, Y: torch.Tensor, stream=None):
    """Y += W X (Y not cleared)."""
    X = _bits(X)
    T = 1 if X.dim() == 1 else X.shape[0]
    _shape(X, (W.K,) if X.dim() == 1 else (T, W.K), "X")
    _out(Y, T * W.N, (torch.float32,), "Y")
    _check(lib().cas_verify_gemm_accumulate(ctypes.byref(W.desc), _ptr(X), T, _ptr(Y), _stream(stream)),
           "cas_verify_gemm_accumulate")
    return Y


def verify_gemm(W: EncodedWeights, X: torch.Tensor) -> torch.Tensor:
    T = 1 if X.dim() == 1 else X.shape[0]
    Y = torch.empty(T, W.N, dtype=torch.float32, device=X.device)
    return cas_verify_gemm(W, X, Y)


def decode_draft(W: EncodedWeights) -> torch.Tensor:
    out = torch.empty(W.N, W.K, dtype=torch.int16, device=W.buf.device)
    return cas_decode_draft(W, out)


def reconstruct(W: EncodedWeights) -> torch.Tensor:
    out = torch.empty(W.N, W.K, dtype=torch.int16, device=W.buf.device)
    return cas_reconstruct(W, out)


def set_launch_overlap(on: bool) -> None:
    """Launch later kernels with programmatic stream serialization (see
    cas_set_launch_overlap): back-to-back libcas kernels overlap their launch
    with the previous kernel's tail. The caller must not enqueue its own copy
    or memset directly before a libcas call while this is on."""
    _check(lib().cas_set_launch_overlap(1 if on else 0), "cas_set_launch_overlap")


def cas_device_status(stream=None) -> int:
    """Reads and clears the flags that bounded device waits set (syncs)."""
    return int(lib().cas_device_status(_stream(stream)))


# ------------------------------------------------------------------ prepared calls
def prepare(fn_name: str, *args):
    """Returns a zero-argument callable that re-issues one C entry point with
    arguments already converted to ctypes (for launch loops); raises on error."""
    f = getattr(lib(), fn_name)
    conv = []
    for a in args:
        if a is None:
            conv.append(ctypes.c_void_p(0))
        elif isinstance(a, torch.Tensor):
            conv.append(_ptr(a))
        elif isinstance(a, (EncodedWeights,)):
            conv.append(ctypes.byref(a.desc))
        elif isinstance(a, torch.cuda.Stream):
            conv.append(ctypes.c_void_p(a.cuda_stream))
        else:
            conv.append(a)
    conv = tuple(conv)

    def call():
        s = f(*conv)
        if s != CAS_OK:
            raise CasError(s, fn_name)
    return call


# ------------------------------------------------------------------ KV cache
def cas_kv_plan(n_kv_heads: int, max_tokens: int, p: cas_params, est_bits_per_code: float = 6.0) -> int:
    n = ctypes.c_uint64(0)
    _check(lib().cas_kv_plan(n_kv_heads, max_tokens, p, est_bits_per_code, ctypes.byref(n)), "cas_kv_plan")
    return int(n.value)


class KVCache:
    """One (sequence, layer) compressed KV cache in a torch-owned device buffer."""

    def __init__(self, n_kv_heads: int, max_tokens: int, p: cas_params, calib_k: torch.Tensor,
                 calib_v: torch.Tensor, est_bits_per_code: float = 6.0, stream=None):
        calib_k, calib_v = _bits(calib_k).contiguous(), _bits(calib_v).contiguous()
        _shape(calib_k, (calib_k.shape[0], n_kv_heads, 128), "calib_k")
        _shape(calib_v, tuple(calib_k.shape), "calib_v")
        dev = calib_k.device
        self.buf = torch.empty(cas_kv_plan(n_kv_heads, max_tokens, p, est_bits_per_code), dtype=torch.uint8,
                               device=dev)
        self.desc = cas_kv()
        _check(lib().cas_kv_init(ctypes.byref(self.desc), _ptr(self.buf), self.buf.numel(), n_kv_heads, max_tokens,
                                 p, est_bits_per_code, _ptr(calib_k), _ptr(calib_v), calib_k.shape[0],
                                 _stream(stream)), "cas_kv_init")

    @property
    def H(self):
        return self.desc.n_kv_heads

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        k_new, v_new = _bits(k_new).contiguous(), _bits(v_new).contiguous()
        _shape(k_new, (k_new.shape[0], self.H, 128), "k_new")
        _shape(v_new, tuple(k_new.shape), "v_new")
        _check(lib().cas_encode_kv_append(ctypes.byref(self.desc), _ptr(k_new), _ptr(v_new), k_new.shape[0],
                                          _stream(stream)), "cas_encode_kv_append")

    def truncate(self, n_tokens: int, stream=None):
        _check(lib().cas_kv_truncate(ctypes.byref(self.desc), n_tokens, _stream(stream)), "cas_kv_truncate")

    def status(self, stream=None) -> tuple[int, int]:
        n = ctypes.c_int64(0)
        s = lib().cas_kv_status(ctypes.byref(self.desc), ctypes.byref(n), _stream(stream))
        return int(n.value), int(s)

    def clear_status(self, stream=None):
        _check(lib().cas_kv_clear_status(ctypes.byref(self.desc), _stream(stream)), "cas_kv_clear_status")

    def section(self, name: str, stream_index: int) -> torch.Tensor:
        i = KV_SECTIONS.index(name)
        o = int(self.desc.off[i]) + stream_index * int(self.desc.stride[i])
        return self.buf[o:o + int(self.desc.stride[i])]

    def tables(self, kv: int, head: int):
        """(rank_of_exp, exp_of_rank) of the K (kv=0) or V (kv=1) stream of a head, as numpy."""
        t = self.section("tables", kv * self.H + head).cpu().numpy()
        return t[256:512].copy(), t[:256].copy()

    def prepare_append(self, k_new, v_new, stream=None):
        return prepare("cas_encode_kv_append", ctypes.byref(self.desc), _bits(k_new), _bits(v_new),
                       int(k_new.shape[0]), stream or torch.cuda.current_stream())

    def prepare_truncate(self, n_tokens: int, stream=None):
        return prepare("cas_kv_truncate", ctypes.byref(self.desc), ctypes.c_int64(n_tokens),
                       stream or torch.cuda.current_stream())


class _KvArray:
    """C array of cas_kv pointers; keeps the descriptors alive."""

    def __init__(self, kvs):
        self.kvs = list(kvs)
        self.arr = (ctypes.POINTER(cas_kv) * len(self.kvs))(*[ctypes.pointer(k.desc) for k in self.kvs])
        self.ptr = ctypes.c_void_p(ctypes.addressof(self.arr))


def _kv_array(kvs):
    return _KvArray(kvs)


def kv_truncate_many(kvs, n_tokens: int, stream=None):
    """Rolls every cache in kvs back to n_tokens tokens (one launch per variant)."""
    arr = _kv_array(kvs)
    _check(lib().cas_kv_truncate_many(arr.ptr, len(arr.kvs), n_tokens, _stream(stream)), "cas_kv_truncate_many")


def prepare_truncate_many(kvs, n_tokens: int, stream=None):
    """Zero-argument callable of kv_truncate_many (for launch loops and graphs)."""
    arr = _kv_array(kvs)
    f = lib().cas_kv_truncate_many
    st = _stream(stream or torch.cuda.current_stream())

    def call():
        _check(f(arr.ptr, len(arr.kvs), n_tokens, st), "cas_kv_truncate_many")
    call.keep = arr
    return call


def cas_attn_workspace_bytes(batch: int, n_q_heads: int, T: int, max_tokens: int) -> int:
    return int(lib().cas_attn_workspace_bytes(batch, n_q_heads, T, max_tokens))


def _check_draft_args(kvs, q, tail_k, tail_v) -> int:
    """Shape checks of a draft attention call; returns n_tail."""
    _shape(q, (len(kvs), q.shape[1], 128), "q")
    if (tail_k is None) != (tail_v is None):
        raise ValueError("tail_k and tail_v: both or neither")
    if tail_k is None:
        return 0
    _shape(tail_k, (len(kvs), tail_k.shape[1], kvs[0].H, 128), "tail_k")
    _shape(tail_v, tuple(tail_k.shape), "tail_v")
    return int(tail_k.shape[1])


def draft_attn_decode(kvs, q: torch.Tensor, tail_k=None, tail_v=None, out=None, workspace=None, stream=None):
    """q [B][Hq][128] -> o [B][Hq][128] fp32 over the speculation KV plus bf16 tail tokens."""
    q = _bits(q).contiguous()
    B, Hq, _ = q.shape
    n_tail = _check_draft_args(kvs, q, tail_k, tail_v)
    if out is None:
        out = torch.empty(B, Hq, 128, dtype=torch.float32, device=q.device)
    _out(out, B * Hq * 128, (torch.float32,), "out")
    if workspace is None:
        workspace = torch.empty(cas_attn_workspace_bytes(B, Hq, 1, max(k.desc.max_tokens for k in kvs)),
                                dtype=torch.uint8, device=q.device)
    tk = None if tail_k is None else _bits(tail_k).contiguous()
    tv = None if tail_v is None else _bits(tail_v).contiguous()
    arr = _kv_array(kvs)
    _check(lib().cas_draft_attn_decode(arr.ptr, B, _ptr(q), Hq, _ptr(tk), _ptr(tv), n_tail, _ptr(out), _ptr(workspace),
                                       workspace.numel(), _stream(stream)), "cas_draft_attn_decode")
    return out


def cas_draft_attn_decode_noalloc(kvs, q: torch.Tensor, tail_k=None, tail_v=None, out=None, stream=None):
    """Draft attention without a workspace: for callers that cannot allocate
    device memory when they decode. The library keeps the partials in one
    fixed 8 MiB device array shared by every call (see include/cas.h)."""
    q = _bits(q).contiguous()
    B, Hq, _ = q.shape
    n_tail = _check_draft_args(kvs, q, tail_k, tail_v)
    if out is None:
        out = torch.empty(B, Hq, 128, dtype=torch.float32, device=q.device)
    _out(out, B * Hq * 128, (torch.float32,), "out")
    tk = None if tail_k is None else _bits(tail_k).contiguous()
    tv = None if tail_v is None else _bits(tail_v).contiguous()
    arr = _kv_array(kvs)
    _check(lib().cas_draft_attn_decode_noalloc(arr.ptr, B, _ptr(q), Hq, _ptr(tk), _ptr(tv), n_tail, _ptr(out),
                                               _stream(stream)), "cas_draft_attn_decode_noalloc")
    return out


def verify_attn(kvs, q: torch.Tensor, out=None, workspace=None, stream=None):
    """q [B][T][Hq][128] -> o [B][T][Hq][128] fp32 over the exact KV (causal in the last T)."""
    q = _bits(q).contiguous()
    B, T, Hq, _ = q.shape
    _shape(q, (len(kvs), T, Hq, 128), "q")
    if out is None:
        out = torch.empty(B, T, Hq, 128, dtype=torch.float32, device=q.device)
    _out(out, B * T * Hq * 128, (torch.float32,), "out")
    if workspace is None:
        workspace = torch.empty(cas_attn_workspace_bytes(B, Hq, T, max(k.desc.max_tokens for k in kvs)),
                                dtype=torch.uint8, device=q.device)
    arr = _kv_array(kvs)
    _check(lib().cas_verify_attn(arr.ptr, B, _ptr(q), T, Hq, _ptr(out), _ptr(workspace), workspace.numel(),
                                 _stream(stream)), "cas_verify_attn")
    return out


def prepare_draft_attn(kvs, q, tail_k, tail_v, out, workspace, stream=None):
    arr = _kv_array(kvs)
    B, Hq, _ = q.shape
    n_tail = 0 if tail_k is None else int(tail_k.shape[1])
    call = prepare("cas_draft_attn_decode", arr.ptr, B, _bits(q), Hq, tail_k, tail_v, n_tail, out, workspace,
                   workspace.numel(), stream or torch.cuda.current_stream())
    call.keep = (arr, kvs, q, tail_k, tail_v, out, workspace)
    return call


def prepare_verify_attn(kvs, q, out, workspace, stream=None):
    arr = _kv_array(kvs)
    B, T, Hq, _ = q.shape
    call = prepare("cas_verify_attn", arr.ptr, B, _bits(q), T, Hq, out, workspace, workspace.numel(),
                   stream or torch.cuda.current_stream())
    call.keep = (arr, kvs, q, out, workspace)
    return call


# ------------------------------------------------------------------ forward-pass glue
def add_rmsnorm(x: torch.Tensor, y: torch.Tensor | None, gamma: torch.Tensor, eps: float = 1e-5,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """x += y (if given), returns bf16 rmsnorm(x) * gamma. x, y: fp32 [rows][dim]."""
    rows, dim = x.shape
    if x.dtype != torch.float32 or (y is not None and (y.dtype != torch.float32 or tuple(y.shape) != (rows, dim))):
        raise ValueError("add_rmsnorm: x and y must be fp32 of one shape")
    gamma = _bits(gamma)
    _shape(gamma, (dim,), "gamma")
    if out is None:
        out = torch.empty(rows, dim, dtype=torch.int16, device=x.device)
    _out(out, rows * dim, (torch.int16, torch.bfloat16), "out")
    _check(lib().cas_add_rmsnorm(_ptr(x), _ptr(y), rows, dim, _ptr(gamma), float(eps), _ptr(out), _stream(stream)),
           "cas_add_rmsnorm")
    return out


def rope_split(qkv: torch.Tensor, n_q_heads: int, n_kv_heads: int, pos0: int, rows_per_seq: int | None = None,
               theta: float = 500000.0, stream=None):
    """Returns (q, k, v) bf16 bit patterns [rows][H][128] from fp32 qkv [rows][(Hq+2Hkv)*128]."""
    rows = qkv.shape[0]
    _shape(qkv, (rows, (n_q_heads + 2 * n_kv_heads) * 128), "qkv")
    if qkv.dtype != torch.float32:
        raise ValueError("rope_split: qkv must be fp32")
    dev = qkv.device
    q = torch.empty(rows, n_q_heads, 128, dtype=torch.int16, device=dev)
    k = torch.empty(rows, n_kv_heads, 128, dtype=torch.int16, device=dev)
    v = torch.empty(rows, n_kv_heads, 128, dtype=torch.int16, device=dev)
    _check(lib().cas_rope_split(_ptr(qkv), rows, n_q_heads, n_kv_heads, pos0, rows_per_seq or rows, float(theta),
                                _ptr(q), _ptr(k), n_kv_heads * 128, _ptr(v), n_kv_heads * 128, _stream(stream)),
           "cas_rope_split")
    return q, k, v


def silu_mul(gate_up: torch.Tensor, stream=None) -> torch.Tensor:
    rows, two_f = gate_up.shape
    if gate_up.dtype != torch.float32 or two_f % 2:
        raise ValueError("silu_mul: fp32 [rows][2 ffn] expected")
    out = torch.empty(rows, two_f // 2, dtype=torch.int16, device=gate_up.device)
    _check(lib().cas_silu_mul(_ptr(gate_up), rows, two_f // 2, _ptr(out), _stream(stream)), "cas_silu_mul")
    return out


def f32_to_bf16(x: torch.Tensor, stream=None) -> torch.Tensor:
    if x.dtype != torch.float32:
        raise ValueError("f32_to_bf16: fp32 input expected")
    out = torch.empty(x.shape, dtype=torch.int16, device=x.device)
    _check(lib().cas_f32_to_bf16(_ptr(x), x.numel(), _ptr(out), _stream(stream)), "cas_f32_to_bf16")
    return out


def argmax(logits: torch.Tensor, stream=None) -> torch.Tensor:
    rows, V = logits.shape
    if logits.dtype != torch.float32:
        raise ValueError("argmax: fp32 logits expected")
    out = torch.empty(rows, dtype=torch.int32, device=logits.device)
    _check(lib().cas_argmax(_ptr(logits), rows, V, _ptr(out), _stream(stream)), "cas_argmax")
    return out


def embed(tokens: torch.Tensor, table: torch.Tensor, stream=None) -> torch.Tensor:
    if tokens.dtype != torch.int32:
        raise ValueError("embed: int32 token ids expected")
    table = _bits(table)
    V, dim = table.shape
    x = torch.empty(tokens.numel(), dim, dtype=torch.float32, device=table.device)
    _check(lib().cas_embed(_ptr(tokens), tokens.numel(), _ptr(table), V, dim, _ptr(x), _stream(stream)), "cas_embed")
    return x
