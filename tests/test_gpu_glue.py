"""GPU parity of the forward-pass glue kernels against the float64 oracle
(oracle/glue.py), through the C ABI. bf16 outputs: within one bf16 rounding
(2^-8 relative) of the float64 value, plus fp32 arithmetic; the rotary outputs
relative to the magnitude of their input pair. argmax and embed: exact."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import glue

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cas():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_level_weight_gb300 as cas
    from bit_level_weight_gb300 import build
    build.build()
    return cas


def f64(bits):
    return glue._f64_of_bf16(bits.cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("rows,dim,with_y", [(1, 4096, True), (14, 4096, True), (5, 1152, False), (2, 12288, True)])
def test_add_rmsnorm(cas, rows, dim, with_y):
    g = torch.Generator().manual_seed(rows + dim)
    x = torch.randn(rows, dim, generator=g) * 3.0
    y = torch.randn(rows, dim, generator=g) if with_y else None
    gamma = synthetic.to_bits(1.0 + 0.1 * torch.randn(dim, generator=g))
    xd = x.cuda()
    out = cas.add_rmsnorm(xd, y.cuda() if with_y else None, gamma.cuda(), 1e-5)
    xs = x.double().numpy() + (y.double().numpy() if with_y else 0.0)
    ref = glue.rmsnorm(xs, gamma.numpy().view(np.uint16), 1e-5)
    assert np.allclose(xd.double().cpu().numpy(), xs, rtol=1e-6, atol=1e-6)  # x updated in place
    got = f64(out)
    assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6).all()


@pytest.mark.parametrize("Hq,Hkv,rows,rps,pos0", [(32, 8, 1, 1, 0), (32, 8, 5, 5, 32768), (32, 8, 14, 7, 16384),
                                                  (8, 2, 3, 3, 131000)])
def test_rope_split(cas, Hq, Hkv, rows, rps, pos0):
    g = torch.Generator().manual_seed(Hq + rows + pos0)
    qkv = torch.randn(rows, (Hq + 2 * Hkv) * 128, generator=g) * 2.0
    theta = 500000.0
    q, k, v = cas.rope_split(qkv.cuda(), Hq, Hkv, pos0, rps, theta)
    rq, rk, rv = glue.rope_split(qkv.double().numpy(), Hq, Hkv, pos0, rps, theta)
    h = qkv.double().numpy().reshape(rows, Hq + 2 * Hkv, 128)
    for got, ref, src in ((q, rq, h[:, :Hq]), (k, rk, h[:, Hq:Hq + Hkv])):
        mag = np.sqrt(src[..., :64] ** 2 + src[..., 64:] ** 2)
        mag = np.concatenate([mag, mag], axis=-1)
        assert (np.abs(f64(got) - ref) <= 2.0 ** -8 * mag + 1e-6).all()
    assert (np.abs(f64(v) - rv) <= 2.0 ** -8 * np.abs(rv)).all()


def test_silu_mul(cas):
    g = torch.Generator().manual_seed(3)
    gu = torch.randn(5, 2 * 14336, generator=g) * 3.0
    out = cas.silu_mul(gu.cuda())
    ref = glue.silu_mul(gu.double().numpy())
    assert (np.abs(f64(out) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6).all()


def test_argmax_exact_with_ties(cas):
    g = torch.Generator().manual_seed(4)
    lg = torch.randn(3, 151936, generator=g)
    lg[0, 70000] = lg[0, 900] = 50.0      # tie: the lower index wins
    lg[1, 151935] = 60.0                  # maximum at the last index
    lg[2, :] = -1.0
    lg[2, 5] = lg[2, 6] = 0.0
    out = cas.argmax(lg.cuda()).cpu().numpy()
    assert list(out) == list(glue.argmax(lg.double().numpy())) == [900, 151935, 5]


def test_embed_exact(cas):
    table = synthetic.normal_weight(1000, 4096, seed=5)
    tok = torch.tensor([0, 999, 17, 17], dtype=torch.int32)
    x = cas.embed(tok.cuda(), table.cuda()).double().cpu().numpy()
    assert np.array_equal(x, glue.embed(tok.numpy(), table.numpy().view(np.uint16)))


@pytest.mark.parametrize("keep", [64, 38])
@pytest.mark.parametrize("N,K,nvec", [(40, 4096, 1), (24, 14336, 2), (20, 1152, 1), (33, 4096, 2)])
def test_draft_gemv_rmsnorm_and_accumulate(cas, N, K, nvec, keep):
    """The draft GEMV of a normalised fp32 input (RMSNorm in the GEMV's x
    staging where the lane-per-block kernel takes the tensor, K = 4096 and
    14336; a separate normalisation for K = 1152) against the float64
    statements, and the accumulating GEMV (y += D(W) x) on top of a given y."""
    import oracle
    g = torch.Generator().manual_seed(N + K + nvec + keep)
    W = synthetic.t4_weight(N, K, seed=N + K)
    enc = cas.encode_weights(W.cuda(), 1, keep, 3)
    Wd = oracle.draft_values(W.numpy().view(np.uint16), 1, keep, 3)
    x = torch.randn(nvec, K, generator=g) * 2.0
    gamma = synthetic.to_bits(1.0 + 0.1 * torch.randn(K, generator=g))
    xn, y = cas.draft_gemv_rmsnorm(enc, x.cuda(), gamma.cuda(), 1e-5)
    ref_xn = glue.rmsnorm(x.double().numpy(), gamma.numpy().view(np.uint16), 1e-5)
    got_xn = f64(xn)
    assert (np.abs(got_xn - ref_xn) <= 2.0 ** -8 * np.abs(ref_xn) + 1e-6).all()
    ref, nrm = oracle.matvec(Wd, xn.cpu().numpy().view(np.uint16))  # y against the xn the call wrote
    assert (np.abs(y.double().cpu().numpy() - ref) <= 2e-3 * nrm + 1e-30).all()
    y0 = torch.randn(nvec, N, generator=g)
    ya = cas.cas_draft_gemv_accumulate(enc, xn, y0.clone().cuda())
    assert (np.abs(ya.double().cpu().numpy() - (y0.double().numpy() + ref)) <= 2e-3 * nrm + 1e-5).all()


@pytest.mark.parametrize("op", ["round", "silu_mul"])
@pytest.mark.parametrize("N,K,nvec", [(40, 4096, 1), (24, 14336, 2), (20, 1152, 1), (33, 4096, 2)])
def test_draft_gemv_f32_inputs(cas, N, K, nvec, op):
    """The draft GEMV of an fp32 input rounded to bf16, or of SiLU(gate) * up
    of a fused fp32 gate|up row, formed in the GEMV's x staging (K = 4096 and
    14336) or by the glue kernel first (K = 1152): xn is bit-identical to
    cas_f32_to_bf16 / cas_silu_mul, y matches the float64 statements on xn,
    and the accumulating call adds the same product to a given y."""
    import oracle
    g = torch.Generator().manual_seed(N + K + nvec + len(op))
    W = synthetic.t4_weight(N, K, seed=N + K + 1)
    enc = cas.encode_weights(W.cuda(), 1, 64, 3)
    Wd = oracle.draft_values(W.numpy().view(np.uint16), 1, 64, 3)
    width = 2 * K if op == "silu_mul" else K
    x = (torch.randn(nvec, width, generator=g) * 3.0).cuda()
    code = cas.X_SILU_MUL if op == "silu_mul" else cas.X_ROUND
    xn, y = cas.draft_gemv_f32(enc, x, code)
    want = cas.silu_mul(x) if op == "silu_mul" else cas.f32_to_bf16(x)
    assert torch.equal(xn.cpu(), want.cpu())
    ref, nrm = oracle.matvec(Wd, xn.cpu().numpy().view(np.uint16))
    assert (np.abs(y.double().cpu().numpy() - ref) <= 2e-3 * nrm + 1e-30).all()
    y0 = torch.randn(nvec, N, generator=g)
    xn2, ya = cas.draft_gemv_f32(enc, x, code, y=y0.clone().cuda(), accumulate=True)
    assert torch.equal(xn2.cpu(), want.cpu())
    assert (np.abs(ya.double().cpu().numpy() - (y0.double().numpy() + ref)) <= 2e-3 * nrm + 1e-5).all()
