"""Shape and dtype checks of the Python binding (no GPU): the C ABI takes
sizes on trust, so a tensor of the wrong shape must be refused before any
call reaches the library."""
import types

import pytest
import torch

import bit_level_weight_gb300 as cas


def fake_weights(N, K):
    d = cas.cas_weights()
    d.N, d.K = N, K
    return cas.EncodedWeights(d, torch.empty(0, dtype=torch.uint8))


def fake_kv(H=8, max_tokens=64):
    return types.SimpleNamespace(H=H, desc=types.SimpleNamespace(max_tokens=max_tokens))


W = fake_weights(6, 256)


@pytest.mark.parametrize("x,y,what", [
    (torch.zeros(1, 128, dtype=torch.int16), torch.zeros(1, 6), "x"),
    (torch.zeros(2, 256, dtype=torch.int16), torch.zeros(1, 6), "y"),
    (torch.zeros(256, dtype=torch.int16), torch.zeros(6, dtype=torch.float64), "y"),
])
def test_draft_gemv_shapes(x, y, what):
    with pytest.raises(ValueError, match=what):
        cas.cas_draft_gemv(W, x, y)


@pytest.mark.parametrize("X,Y,what", [
    (torch.zeros(5, 255, dtype=torch.int16), torch.zeros(5, 6), "X"),
    (torch.zeros(5, 256, dtype=torch.int16), torch.zeros(4, 6), "Y"),
])
def test_verify_gemm_shapes(X, Y, what):
    with pytest.raises(ValueError, match=what):
        cas.cas_verify_gemm(W, X, Y)


def test_materialise_shapes():
    with pytest.raises(ValueError, match="out"):
        cas.cas_decode_draft(W, torch.zeros(6, 128, dtype=torch.int16))
    with pytest.raises(ValueError, match="out"):
        cas.cas_reconstruct(W, torch.zeros(6, 256, dtype=torch.float32))


def test_draft_attention_shapes():
    kvs = [fake_kv(), fake_kv()]
    q = torch.zeros(2, 32, 128, dtype=torch.int16)
    with pytest.raises(ValueError, match="q"):
        cas.draft_attn_decode(kvs[:1], q)
    tk = torch.zeros(2, 3, 8, 128, dtype=torch.int16)
    with pytest.raises(ValueError, match="tail_k and tail_v"):
        cas.draft_attn_decode(kvs, q, tk, None)
    with pytest.raises(ValueError, match="tail_k"):
        cas.draft_attn_decode(kvs, q, tk[:, :, :4], tk[:, :, :4])
    with pytest.raises(ValueError, match="tail_v"):
        cas.draft_attn_decode(kvs, q, tk, tk[:, :2])
    with pytest.raises(ValueError, match="out"):
        cas.draft_attn_decode(kvs, q, out=torch.zeros(2, 32, 64))
    with pytest.raises(ValueError, match="q"):
        cas.cas_draft_attn_decode_noalloc(kvs, q[:1])


def test_verify_attention_shapes():
    kvs = [fake_kv()]
    with pytest.raises(ValueError, match="q"):
        cas.verify_attn(kvs, torch.zeros(2, 5, 32, 128, dtype=torch.int16))
    with pytest.raises(ValueError, match="out"):
        cas.verify_attn(kvs, torch.zeros(1, 5, 32, 128, dtype=torch.int16), out=torch.zeros(1, 5, 32, 127))


def test_kv_append_shapes():
    kv = object.__new__(cas.KVCache)
    kv.desc = cas.cas_kv()
    kv.desc.n_kv_heads = 8
    k = torch.zeros(3, 8, 128, dtype=torch.int16)
    with pytest.raises(ValueError, match="k_new"):
        kv.append(torch.zeros(3, 4, 128, dtype=torch.int16), k)
    with pytest.raises(ValueError, match="v_new"):
        kv.append(k, k[:2])


@pytest.mark.parametrize("x,op,kw,what", [
    (torch.zeros(1, 256), 7, {}, "unknown op"),
    (torch.zeros(1, 256, dtype=torch.float64), 0, {}, "fp32"),
    (torch.zeros(1, 256), 2, {}, "fp32 \\[nvec\\]\\[512\\]"),       # SiLU*mul reads rows of 2K
    (torch.zeros(1, 512), 0, {}, "fp32 \\[nvec\\]\\[256\\]"),
    (torch.zeros(1, 256), 1, {}, "gamma"),                         # RMSNorm without gamma
    (torch.zeros(1, 256), 0, {"accumulate": True}, "accumulate needs y"),
    (torch.zeros(1, 256), 0, {"y": torch.zeros(1, 5)}, "y"),
    (torch.zeros(1, 256), 0, {"xn": torch.zeros(1, 255, dtype=torch.int16)}, "xn"),
])
def test_draft_gemv_f32_checks(x, op, kw, what):
    with pytest.raises(ValueError, match=what):
        cas.draft_gemv_f32(W, x, op, **kw)
