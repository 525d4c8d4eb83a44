"""The draft attention entry point that allocates nothing.

Some callers cannot allocate device memory when they decode (a runtime whose
memory plan is fixed at start-up, or an application that owns every
allocation and passes the library only inputs and outputs).
cas_draft_attn_decode_noalloc serves them with a fixed device array inside
the library instead of a workspace. This test calls it through the C ABI and
checks it against cas_draft_attn_decode on two calls in a row (the second
with other inputs, so a stale partial from the first call would show).

Kept in a file of its own that sorts last, so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu
TOL = 2e-3
D = 128


@pytest.fixture(scope="module")
def cas():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_level_weight_gb300 as cas
    from bit_level_weight_gb300 import build
    build.build()
    return cas


def _caches(cas, lens, H, seed, max_tokens=None):
    """One cache per entry of lens holding that many tokens (0 allowed),
    sized for max_tokens (default: its length + 64)."""
    caches = []
    for b, T in enumerate(lens):
        sk, sv = synthetic.kv_scales(b, H, 0), synthetic.kv_scales(b, H, 1)
        K = synthetic.kv_tokens(max(T, 16), H, seed=seed + 2 * b, scales=sk).cuda()
        V = synthetic.kv_tokens(max(T, 16), H, seed=seed + 2 * b + 1, scales=sv).cuda()
        cap = max_tokens if max_tokens is not None else T + 64
        kv = cas.KVCache(H, cap, cas.params(1, 64, 3), K[:16].contiguous(), V[:16].contiguous())
        if T:
            kv.append(K[:T].contiguous(), V[:T].contiguous())
        assert kv.status() == (T, 0)
        caches.append(kv)
    return caches


def _check_against_workspace_version(cas, caches, Hq, H, seed, what):
    B = len(caches)
    q = synthetic.activations(B, Hq * D, seed=seed).view(B, Hq, D).cuda()
    tk = synthetic.activations(B * 3, H * D, seed=seed + 10).view(B, 3, H, D).cuda()
    tv = synthetic.activations(B * 3, H * D, seed=seed + 20).view(B, 3, H, D).cuda()
    ref = cas.draft_attn_decode(caches, q, tk, tv)
    out = torch.full_like(ref, float("nan"))
    assert _noalloc_abi(cas, caches, q, tk, tv, out) == 0
    torch.cuda.synchronize()
    r, o = ref.double().cpu().numpy(), out.double().cpu().numpy()
    assert np.isfinite(o).all(), what
    err = np.abs(o - r)
    assert (err <= TOL * np.abs(r) + 1e-6).all(), f"{what}: worst {err.max():.3g}"


def _noalloc_abi(cas, caches, q, tk, tv, out):
    """Direct C-ABI call of cas_draft_attn_decode_noalloc."""
    f = cas.lib().cas_draft_attn_decode_noalloc
    P = ctypes.c_void_p
    f.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, P, ctypes.c_int, P, P]
    f.restype = ctypes.c_int
    arr = (ctypes.POINTER(cas.cas_kv) * len(caches))(*[ctypes.pointer(k.desc) for k in caches])
    B, Hq, _ = q.shape
    n_tail = 0 if tk is None else tk.shape[1]
    st = torch.cuda.current_stream().cuda_stream
    return f(ctypes.addressof(arr), B, q.data_ptr(), Hq, tk.data_ptr() if tk is not None else None,
             tv.data_ptr() if tv is not None else None, n_tail, out.data_ptr(), st)


def test_noalloc_matches_workspace_version_two_calls(cas):
    H, Hq = 8, 32
    caches = _caches(cas, (700, 1500), H, seed=90)
    for call, seed in enumerate((5, 6)):
        q = synthetic.activations(2, Hq * D, seed=seed).view(2, Hq, D).cuda()
        tk = synthetic.activations(2 * 3, H * D, seed=seed + 10).view(2, 3, H, D).cuda()
        tv = synthetic.activations(2 * 3, H * D, seed=seed + 20).view(2, 3, H, D).cuda()
        ref = cas.draft_attn_decode(caches, q, tk, tv)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_abi(cas, caches, q, tk, tv, out) == 0
        torch.cuda.synchronize()
        r, o = ref.double().cpu().numpy(), out.double().cpu().numpy()
        assert np.isfinite(o).all(), f"call {call}"
        err = np.abs(o - r)
        assert (err <= TOL * np.abs(r) + 1e-6).all(), f"call {call}: worst {err.max():.3g}"


def test_noalloc_large_call_then_smaller_layout(cas):
    """A call that fills much of the array (batch 2, 24 chunks per head) and
    then one with another chunk count and stride, one of whose sequences has
    no cached tokens: the second call must read none of the first call's
    partials."""
    H, Hq = 8, 32
    big = _caches(cas, (5000, 4100), H, seed=70, max_tokens=6000)
    _check_against_workspace_version(cas, big, Hq, H, seed=11, what="large call")
    small = _caches(cas, (0, 200), H, seed=80, max_tokens=300)
    _check_against_workspace_version(cas, small, Hq, H, seed=12, what="smaller call after it")
    one = _caches(cas, (130,), H, seed=85)
    _check_against_workspace_version(cas, one, 16, H, seed=13, what="batch 1, 16 query heads")


def test_noalloc_rejects_invalid_descriptor_like_workspace_version(cas):
    H = 8
    good = _caches(cas, (40,), H, seed=3)[0]
    bad = cas.cas_kv.from_buffer_copy(bytes(good.desc))
    bad.max_tokens = 0
    q = torch.zeros(1, 32, D, dtype=torch.int16, device="cuda")
    out = torch.zeros(1, 32, D, dtype=torch.float32, device="cuda")
    f = cas.lib().cas_draft_attn_decode_noalloc
    P = ctypes.c_void_p
    f.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, P, ctypes.c_int, P, P]
    f.restype = ctypes.c_int
    arr = (ctypes.POINTER(cas.cas_kv) * 1)(ctypes.pointer(bad))
    st = torch.cuda.current_stream().cuda_stream
    got = f(ctypes.addressof(arr), 1, q.data_ptr(), 32, None, None, 0, out.data_ptr(), st)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    g = cas.lib().cas_draft_attn_decode
    g.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, P, ctypes.c_int, P, P, ctypes.c_uint64, P]
    g.restype = ctypes.c_int
    want = g(ctypes.addressof(arr), 1, q.data_ptr(), 32, None, None, 0, out.data_ptr(), ws.data_ptr(), ws.numel(), st)
    assert got == want == -1  # CAS_ERR_INVALID


def test_noalloc_rejects_oversized_request(cas):
    H = 8
    sk, sv = synthetic.kv_scales(0, H, 0), synthetic.kv_scales(0, H, 1)
    K = synthetic.kv_tokens(16, H, seed=1, scales=sk).cuda()
    V = synthetic.kv_tokens(16, H, seed=2, scales=sv).cuda()
    # 2 sequences x 256 query heads x ceil(20000 / 256) chunks x 520 B = 20.8 MB > 8 MiB
    big = [cas.KVCache(H, 20000, cas.params(1, 64, 3), K, V) for _ in range(2)]
    q = torch.zeros(2, 256, D, dtype=torch.int16, device="cuda")
    out = torch.full((2, 256, D), 7.0, dtype=torch.float32, device="cuda")
    assert _noalloc_abi(cas, big, q, None, None, out) == -6  # CAS_ERR_BUFFER, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
