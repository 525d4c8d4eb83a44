"""Launch overlap (programmatic stream serialization) changes no result.

A chain of libcas calls - draft GEMV of a normalised fp32 input, SiLU*mul,
accumulating draft GEMV into the residual, to_bf16, argmax, and a draft GEMV
whose rows span several chunks (fp32 atomics after a memset) - runs three
times with overlap off, with overlap on, and as a CUDA graph captured with
overlap on. Every kernel waits on the device for the one before it, so the
outputs that one writer produces (rows of one chunk, glue) are bit-identical
and the atomically summed ones agree to fp32 rounding.
"""
import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cas():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_level_weight_gb300 as m
    from bit_level_weight_gb300 import build
    build.build()
    return m


def test_overlap_chain_matches(cas):
    dev = torch.device("cuda", 0)
    K, F, Nq, Nb = 4096, 4096, 1024, 2048
    Wg = cas.encode_weights(synthetic.t4_weight(2 * F, K, seed=41).to(dev), 1, 64, 3)
    Wd = cas.encode_weights(synthetic.t4_weight(K, F, seed=42).to(dev), 1, 64, 3)
    Wq = cas.encode_weights(synthetic.t4_weight(Nq, K, seed=43).to(dev), 1, 64, 3)
    Wb = cas.encode_weights(synthetic.t4_weight(Nb, 2 * K, seed=44).to(dev), 1, 64, 3)  # 64 blocks a row
    gamma = synthetic.to_bits(1.0 + 0.1 * torch.randn(K, generator=torch.Generator().manual_seed(45))).to(dev)
    x0 = (torch.randn(1, K, generator=torch.Generator().manual_seed(46)) * 2.0).to(dev)
    x = torch.empty_like(x0)
    xn = torch.empty(1, K, dtype=torch.int16, device=dev)
    gu = torch.empty(1, 2 * F, dtype=torch.float32, device=dev)
    hh = torch.empty(1, F, dtype=torch.int16, device=dev)
    q = torch.empty(1, Nq, dtype=torch.float32, device=dev)
    qb = torch.empty(1, Nq, dtype=torch.int16, device=dev)
    tok = torch.empty(3, dtype=torch.int32, device=dev)
    xb2 = torch.empty(1, 2 * K, dtype=torch.int16, device=dev)
    yb = torch.empty(1, Nb, dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(device=dev)
    P = cas.prepare
    chain = []
    for it in range(3):
        chain += [P("cas_draft_gemv_rmsnorm", Wg, x, 1, gamma, 1e-5, xn, gu, st),
                  P("cas_silu_mul", gu, 1, F, hh, st),
                  P("cas_draft_gemv_accumulate", Wd, hh, 1, x, st),
                  P("cas_draft_gemv_rmsnorm", Wq, x, 1, gamma, 1e-5, xn, q, st),
                  P("cas_f32_to_bf16", q, Nq, qb, st),
                  P("cas_argmax", q, 1, Nq, tok[it:it + 1], st),
                  P("cas_f32_to_bf16", gu, 2 * K, xb2, st),
                  P("cas_draft_gemv", Wb, xb2, 1, yb, st)]

    def run():
        x.copy_(x0)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            for f in chain:
                f()
        torch.cuda.synchronize()
        return [t.clone() for t in (x, xn, gu, hh, q, qb, tok, yb)]

    cas.set_launch_overlap(False)
    ref = run()
    cas.set_launch_overlap(True)
    try:
        on = run()
        g = torch.cuda.CUDAGraph()
        x.copy_(x0)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=st):
            for f in chain:
                f()
    finally:
        cas.set_launch_overlap(False)
    x.copy_(x0)
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        g.replay()
    torch.cuda.synchronize()
    graph = [t.clone() for t in (x, xn, gu, hh, q, qb, tok, yb)]
    names = ("x", "xn", "gu", "hh", "q", "qb", "tok", "yb")
    for got in (on, graph):
        for name, a, b in zip(names[:-1], ref[:-1], got[:-1]):
            assert torch.equal(a, b), name
        r, o = ref[-1].double().cpu().numpy(), got[-1].double().cpu().numpy()
        assert np.allclose(o, r, rtol=1e-5, atol=1e-5 * np.abs(r).max())
