"""Checkpoint and resume: an encoded tensor or KV cache is a plain descriptor
plus one device buffer, so saving both bytes and restoring them into a fresh
buffer (with the descriptor's base moved to it) gives back the same tensor
without re-encoding."""
import ctypes
import io

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module")
def cas():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_level_weight_gb300 as cas
    from bit_level_weight_gb300 import build
    build.build()
    return cas


def np16(t):
    return t.cpu().numpy().view(np.uint16)


def save(buf, desc):
    f = io.BytesIO()
    torch.save({"buf": buf.cpu(), "desc": bytes(desc)}, f)
    return f.getvalue()


@pytest.mark.parametrize("variant", [1, 2])
def test_weights_save_reload_without_reencoding(cas, orc, variant):
    N, K = 40, 2048
    W = synthetic.t4_weight(N, K, seed=17 + variant)
    enc = cas.encode_weights(W.cuda(), variant, 64, 3)
    blob = save(enc.buf, enc.desc)
    x = synthetic.activations(1, K, seed=5).cuda()
    y0 = cas.draft_gemv(enc, x)
    del enc
    torch.cuda.empty_cache()
    st = torch.load(io.BytesIO(blob))
    pad = torch.empty(4096, dtype=torch.uint8, device="cuda")  # a different address
    buf = st["buf"].cuda()
    desc = cas.cas_weights.from_buffer_copy(st["desc"])
    desc.base = buf.data_ptr()
    enc2 = cas.EncodedWeights(desc, buf)
    assert np.array_equal(np16(cas.reconstruct(enc2)), np16(W))
    assert np.array_equal(np16(cas.decode_draft(enc2)), orc.draft_values(np16(W), variant, 64, 3))
    y1 = cas.draft_gemv(enc2, x)
    ref, norm = orc.matvec(orc.draft_values(np16(W), variant, 64, 3), np16(x.cpu()))
    for y in (y0, y1):
        assert (np.abs(y.double().cpu().numpy() - ref) <= 2e-3 * norm).all()
    del pad


def test_kv_cache_save_reload_and_continue(cas):
    H, Hq, T0 = 2, 8, 300
    sk, sv = synthetic.kv_scales(0, H, 0), synthetic.kv_scales(0, H, 1)
    Kt = synthetic.kv_tokens(T0 + 8, H, seed=4, scales=sk).cuda()
    Vt = synthetic.kv_tokens(T0 + 8, H, seed=5, scales=sv).cuda()
    kv = cas.KVCache(H, 512, cas.params(1, 64, 3), Kt[:16].contiguous(), Vt[:16].contiguous())
    kv.append(Kt[:T0].contiguous(), Vt[:T0].contiguous())
    torch.cuda.synchronize()
    blob = save(kv.buf, kv.desc)
    q = synthetic.activations(1, Hq * D, seed=6).view(1, Hq, D).cuda()
    o0 = cas.draft_attn_decode([kv], q)
    st = torch.load(io.BytesIO(blob))
    kv2 = cas.KVCache.__new__(cas.KVCache)
    kv2.buf = st["buf"].cuda()
    kv2.desc = cas.cas_kv.from_buffer_copy(st["desc"])
    kv2.desc.base = kv2.buf.data_ptr()
    assert kv2.status() == (T0, 0)
    o1 = cas.draft_attn_decode([kv2], q)
    assert torch.equal(o0, o1)
    # both continue identically: append the same tokens to each
    kv.append(Kt[T0:].contiguous(), Vt[T0:].contiguous())
    kv2.append(Kt[T0:].contiguous(), Vt[T0:].contiguous())
    assert kv.status() == kv2.status() == (T0 + 8, 0)
    torch.cuda.synchronize()
    assert torch.equal(kv.buf, kv2.buf)
