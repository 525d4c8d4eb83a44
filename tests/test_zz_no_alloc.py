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


def _caches(cas, lens, H, seed):
    caches = []
    for b, T in enumerate(lens):
        sk, sv = synthetic.kv_scales(b, H, 0), synthetic.kv_scales(b, H, 1)
        K = synthetic.kv_tokens(T, H, seed=seed + 2 * b, scales=sk).cuda()
        V = synthetic.kv_tokens(T, H, seed=seed + 2 * b + 1, scales=sv).cuda()
        kv = cas.KVCache(H, T + 64, cas.params(1, 64, 3), K[:16].contiguous(), V[:16].contiguous())
        kv.append(K, V)
        assert kv.status() == (T, 0)
        caches.append(kv)
    return caches


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
