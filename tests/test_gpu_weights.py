"""GPU parity of the weight path against the CPU oracle, through the C ABI.

Encode / decode_draft / reconstruct: byte-exact. Draft GEMV and verify GEMM:
|y - y_ref| <= 2e-3 * sum_k |w_k x_k| per output (y_ref in float64 over the
oracle's draft values, resp. the original values).
"""
import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu
TOL = 2e-3


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


def check_close(y, ref, norm, what):
    y = y.double().cpu().numpy()
    err = np.abs(y - ref)
    bound = TOL * norm + 1e-30
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside 2e-3 bound; worst ratio {(err / bound).max():.3g}"


CASES = [
    # (N, K, variant, k, m)
    (64, 1024, 1, 64, 3),
    (37, 1152, 1, 38, 3),    # ragged superblock tail (9 blocks per row), odd N
    (16, 384, 1, 0, 3),
    (16, 256, 1, 128, 7),
    (24, 640, 1, 77, 2),     # fields straddle words
    (8, 128, 1, 1, 0),
    (64, 1024, 2, 64, 3),
    (37, 1152, 2, 38, 1),
    (16, 256, 2, 128, 5),
    (24, 640, 2, 90, 0),
    (16, 384, 2, 0, 4),
]


@pytest.mark.parametrize("N,K,variant,k,m", CASES)
def test_encode_decode_bit_exact(cas, orc, N, K, variant, k, m):
    W = synthetic.normal_weight(N, K, seed=N * 1000 + K + variant, outlier_frac=0.01)
    Wn = np16(W)
    ref = orc.encode(Wn, variant, k, m)
    enc = cas.encode_weights(W.cuda(), variant, k, m)
    d = enc.desc
    assert bytes(d.exp_of_rank) == ref.exp_of_rank.tobytes()
    assert list(d.off) == list(ref.off) and list(d.len) == list(ref.len)
    assert int(d.bytes) == ref.buf.size
    got = enc.buf[: ref.buf.size].cpu().numpy()
    for i, name in enumerate(orc.SECTIONS):
        a, b = int(d.off[i]), int(d.off[i]) + int(d.len[i])
        assert np.array_equal(got[a:b], ref.buf[a:b]), name
    assert np.array_equal(got, ref.buf)  # padding bytes too
    assert np.array_equal(np16(cas.decode_draft(enc)), orc.draft_values(Wn, variant, k, m))
    assert np.array_equal(np16(cas.reconstruct(enc)), Wn)


@pytest.mark.parametrize("N,K,variant,k,m", CASES)
@pytest.mark.parametrize("nvec", [1, 2, 4])
def test_draft_gemv(cas, orc, N, K, variant, k, m, nvec):
    W = synthetic.normal_weight(N, K, seed=7 + N + K, outlier_frac=0.01)
    x = synthetic.activations(nvec, K, seed=99 + nvec)
    enc = cas.encode_weights(W.cuda(), variant, k, m)
    y = cas.draft_gemv(enc, x.cuda())
    ref, norm = orc.matvec(orc.draft_values(np16(W), variant, k, m), np16(x))
    check_close(y, ref, norm, "draft_gemv")


@pytest.mark.parametrize("k,m", [(64, 3), (26, 1), (102, 5), (38, 3)])
def test_choose_variant_matches_oracle_sizes(cas, orc, k, m):
    W = synthetic.normal_weight(48, 2048, seed=k + m, outlier_frac=0.001)
    v, (b1, b2) = cas.cas_choose_variant(W.cuda(), k, m)
    r1 = orc.encode(np16(W), 1, k, m).spec_bytes()
    r2 = orc.encode(np16(W), 2, k, m).spec_bytes()
    assert (b1, b2) == (r1, r2)
    assert v == (2 if r2 < r1 else 1)


def wide_exponent_rows(N, K, n_wide, seed):
    """Normal rows, then n_wide rows whose exponents spread over ~200 values:
    their unary codes are long (tens to hundreds of bits) and their
    superblock streams exceed a few hundred words. Row 0 gets a few long codes
    inside otherwise short streams."""
    Wn = np16(synthetic.normal_weight(N, K, seed=seed)).copy()
    rng = np.random.default_rng(seed)
    e = rng.integers(-100, 100, size=(n_wide, K)).astype(np.float64)
    v = rng.choice([-1.0, 1.0], size=(n_wide, K)) * rng.uniform(1.0, 2.0, size=(n_wide, K)) * 2.0 ** e
    Wn[N - n_wide:] = np16(synthetic.to_bits(torch.from_numpy(v.astype(np.float32))))
    spikes = 2.0 ** rng.integers(-60, 60, size=Wn[0, ::97].size)
    Wn[0, ::97] = np16(synthetic.to_bits(torch.from_numpy(spikes.astype(np.float32))))
    return torch.from_numpy(Wn.view(np.int16))


RUN_CASES = [
    # rows of whole superblocks (K % 1024 == 0) with k, m off the k = 64, m = 3 path
    (32, 2048, 1, 38, 3), (16, 1024, 1, 0, 3), (16, 2048, 1, 128, 7), (24, 1024, 1, 77, 2),
    (8, 1024, 1, 1, 0), (16, 1024, 1, 26, 5), (32, 2048, 2, 38, 1), (16, 1024, 2, 128, 7),
    (24, 2048, 2, 90, 0), (16, 1024, 2, 0, 4), (16, 1024, 2, 51, 3),
]


@pytest.mark.parametrize("N,K,variant,k,m", RUN_CASES)
@pytest.mark.parametrize("nvec", [1, 2, 3, 4])
def test_draft_gemv_any_k_m(cas, orc, N, K, variant, k, m, nvec):
    W = synthetic.normal_weight(N, K, seed=3 * N + K + k, outlier_frac=0.01)
    x = synthetic.activations(nvec, K, seed=7 + nvec)
    enc = cas.encode_weights(W.cuda(), variant, k, m)
    y = cas.draft_gemv(enc, x.cuda())
    ref, norm = orc.matvec(orc.draft_values(np16(W), variant, k, m), np16(x))
    check_close(y, ref, norm, "draft_gemv any k, m")


@pytest.mark.parametrize("N,K,variant,k,m", RUN_CASES)
@pytest.mark.parametrize("T", [5, 14])
def test_verify_gemm_any_k_m(cas, orc, N, K, variant, k, m, T):
    W = synthetic.normal_weight(N, K, seed=5 * N + K + k + m, outlier_frac=0.01)
    X = synthetic.activations(T, K, seed=31 + T)
    enc = cas.encode_weights(W.cuda(), variant, k, m)
    Y = cas.verify_gemm(enc, X.cuda())
    ref, norm = orc.matvec(np16(W), np16(X))
    check_close(Y, ref, norm, "verify_gemm any k, m")


@pytest.mark.parametrize("variant,k,m", [(1, 38, 3), (1, 90, 5), (2, 38, 3)])
def test_draft_gemv_any_k_m_long_codes(cas, orc, variant, k, m):
    N, K = 48, 2048
    W = wide_exponent_rows(N, K, 8, seed=9)
    x = synthetic.activations(2, K, seed=19)
    enc = cas.encode_weights(W.cuda(), variant, k, m)
    y = cas.draft_gemv(enc, x.cuda())
    ref, norm = orc.matvec(orc.draft_values(np16(W), variant, k, m), np16(x))
    check_close(y, ref, norm, "draft_gemv any k, m, long codes")
    X = synthetic.activations(5, K, seed=20)
    Y = cas.verify_gemm(enc, X.cuda())
    ref, norm = orc.matvec(np16(W), np16(X))
    check_close(Y, ref, norm, "verify_gemm any k, m, long codes")


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("nvec", [1, 3])
def test_draft_gemv_long_codes(cas, orc, variant, nvec):
    N, K = 48, 2048
    W = wide_exponent_rows(N, K, 8, seed=5)
    x = synthetic.activations(nvec, K, seed=17)
    enc = cas.encode_weights(W.cuda(), variant, 64, 3)
    y = cas.draft_gemv(enc, x.cuda())
    ref, norm = orc.matvec(orc.draft_values(np16(W), variant, 64, 3), np16(x))
    check_close(y, ref, norm, "draft_gemv long codes")


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("T", [5, 14])
def test_verify_gemm_long_codes(cas, orc, variant, T):
    N, K = 48, 2048
    W = wide_exponent_rows(N, K, 8, seed=6)
    X = synthetic.activations(T, K, seed=18)
    enc = cas.encode_weights(W.cuda(), variant, 64, 3)
    Y = cas.verify_gemm(enc, X.cuda())
    ref, norm = orc.matvec(np16(W), np16(X))
    check_close(Y, ref, norm, "verify_gemm long codes")
    assert np.array_equal(np16(cas.reconstruct(enc)), np16(W))


@pytest.mark.parametrize("N,K,variant,k,m", CASES)
@pytest.mark.parametrize("T", [1, 5, 8, 9, 14, 16])
def test_verify_gemm(cas, orc, N, K, variant, k, m, T):
    W = synthetic.normal_weight(N, K, seed=11 + N + K, outlier_frac=0.01)
    X = synthetic.activations(T, K, seed=123 + T)
    enc = cas.encode_weights(W.cuda(), variant, k, m)
    Y = cas.verify_gemm(enc, X.cuda())
    ref, norm = orc.matvec(np16(W), np16(X))
    check_close(Y, ref, norm, "verify_gemm")


def test_all_finite_patterns_roundtrip(cas):
    v = np.arange(65536, dtype=np.uint32)
    v = v[((v >> 7) & 0xFF) != 255].astype(np.uint16)
    rng = np.random.default_rng(4)
    W = rng.permutation(np.concatenate([v, rng.choice(v, 65536 - v.size)])).reshape(64, 1024)
    Wt = torch.from_numpy(W.view(np.int16)).cuda()
    for variant in (1, 2):
        for k, m in ((64, 3), (128, 0), (0, 7), (101, 1)):
            enc = cas.encode_weights(Wt, variant, k, m)
            assert np.array_equal(np16(cas.reconstruct(enc)), W)


def test_errors(cas):
    W = torch.zeros(4, 200, dtype=torch.int16, device="cuda")
    with pytest.raises(cas.CasError) as e:
        cas.encode_weights(W)
    assert e.value.status == -2
    W = torch.zeros(4, 256, dtype=torch.int16, device="cuda")
    W[1, 3] = 0x7F80  # +inf
    with pytest.raises(cas.CasError) as e:
        cas.encode_weights(W)
    assert e.value.status == -3
    W = synthetic.normal_weight(8, 256, seed=1).cuda()
    enc = cas.encode_weights(W)
    x = torch.zeros(5, 256, dtype=torch.int16, device="cuda")
    with pytest.raises(cas.CasError):
        cas.draft_gemv(enc, x)  # nvec > 4
    X = torch.zeros(17, 256, dtype=torch.int16, device="cuda")
    with pytest.raises(cas.CasError):
        cas.verify_gemm(enc, X)  # T > 16
    assert cas.cas_device_status() == 0


def test_empty_tensor(cas):
    W = torch.zeros(0, 256, dtype=torch.int16, device="cuda")
    enc = cas.encode_weights(W)
    y = cas.draft_gemv(enc, torch.zeros(1, 256, dtype=torch.int16, device="cuda"))
    assert y.shape == (1, 0)


def test_cfg0_full_size(cas, orc):
    """The 4096x4096 workload: encode byte-exact, GEMV and GEMM (T=5) in tolerance."""
    W = synthetic.cfg0_weight()
    Wn = np16(W)
    ref = orc.encode(Wn, 1, 64, 3)
    enc = cas.encode_weights(W.cuda(), 1, 64, 3)
    assert np.array_equal(enc.buf[: ref.buf.size].cpu().numpy(), ref.buf)
    x = synthetic.activations(1, 4096, seed=1)
    y = cas.draft_gemv(enc, x.cuda())
    yr, nr = orc.matvec(orc.decode(ref, False), np16(x))
    check_close(y, yr, nr, "cfg0 draft gemv")
    X = synthetic.activations(5, 4096, seed=2)
    Y = cas.verify_gemm(enc, X.cuda())
    Yr, Nr = orc.matvec(Wn, np16(X))
    check_close(Y, Yr, Nr, "cfg0 verify gemm")


@pytest.mark.parametrize("variant,k", [(1, 64), (1, 38), (2, 64)])
def test_llama_ffn_full_size_sampled(cas, orc, variant, k):
    """A 14336x4096 Student-t(4) FFN matrix: lossless reconstruct of the whole
    tensor; sampled rows of the encoding byte-exact and of the GEMV / GEMM in
    tolerance (rows are independent given the tensor's rank table)."""
    N, K, m = 14336, 4096, 3
    W = synthetic.t4_weight(N, K, seed=4)
    Wd = W.cuda()
    enc = cas.encode_weights(Wd, variant, k, m)
    assert torch.equal(cas.reconstruct(enc), Wd)
    Wn = np16(W)
    eor, roe = orc.rank_table(orc.exp_hist(Wn))
    assert bytes(enc.desc.exp_of_rank) == eor.tobytes()
    rows = np.array([0, 1, 777, 8191, 14335])
    sub = orc.encode(Wn[rows], variant, k, m, roe, eor)
    nbr, nsr = K // 128, (K // 128 + 7) // 8
    for name in ("mask", "spec_sm", "spec_q", "spec_mx", "ver_lo", "ver_pr"):
        full, part = enc.section(name).cpu().numpy(), sub.section(name)
        if part.size == 0:
            continue
        per_row = part.size // len(rows)
        for i, r in enumerate(rows):
            assert np.array_equal(full[r * per_row:(r + 1) * per_row], part[i * per_row:(i + 1) * per_row]), name
    for sname, iname in (("spec_exp", "spec_sbidx"), ("ver_exp", "ver_sbidx"), ("ver_d", "ver_d_sbidx"),
                         ("ver_res", "ver_res_sbidx")):
        part_idx = sub.section(iname).view(np.uint32)
        if part_idx.size == 0:
            continue
        full_idx = enc.section(iname).cpu().numpy().view(np.uint32)
        full_w = enc.section(sname).cpu().numpy().view(np.uint32)
        part_w = sub.section(sname).view(np.uint32)
        for i, r in enumerate(rows):
            for j in range(nsr):
                s, ps = r * nsr + j, i * nsr + j
                a = full_w[full_idx[s]:full_idx[s + 1]]
                b = part_w[part_idx[ps]:part_idx[ps + 1]]
                assert np.array_equal(a, b), (sname, r, j)
    x = synthetic.activations(1, K, seed=5)
    y = cas.draft_gemv(enc, x.cuda())[:, rows]
    yr, nr = orc.matvec(orc.draft_values(Wn[rows], variant, k, m), np16(x))
    check_close(y, yr, nr, "ffn draft gemv rows")
    X = synthetic.activations(5, K, seed=6)
    Y = cas.verify_gemm(enc, X.cuda())[:, rows]
    Yr, Nr = orc.matvec(Wn[rows], np16(X))
    check_close(Y, Yr, Nr, "ffn verify gemm rows")


def clustered_rows(N, K, seed):
    """Rows whose kept values sit in chosen mask words of every block, so the
    per-word counts of one superblock range from 0 to 32: row r of a group of
    four keeps positions [0, 64), [64, 128), [32, 96) or every other position
    of each block; the magnitudes of kept values are spread over many
    exponents in the last rows, which makes their code runs long."""
    rng = np.random.default_rng(seed)
    base = rng.standard_normal((N, K)) * 0.02
    big = rng.standard_normal((N, K)) * 0.5 + np.sign(rng.standard_normal((N, K))) * 0.6
    keep = np.zeros((N, K // 128, 128), dtype=bool)
    for r in range(N):
        kind = r % 4
        if kind == 0:
            keep[r, :, :64] = True
        elif kind == 1:
            keep[r, :, 64:] = True
        elif kind == 2:
            keep[r, :, 32:96] = True
        else:
            keep[r, :, ::2] = True
    v = np.where(keep.reshape(N, K), big, base)
    wide = max(1, N // 8)
    v[-wide:] = np.where(keep.reshape(N, K)[-wide:], v[-wide:] * 2.0 ** rng.integers(-40, 40, size=(wide, K)),
                         v[-wide:])
    return synthetic.to_bits(torch.from_numpy(v.astype(np.float32)))


@pytest.mark.parametrize("nvec", [1, 2])
@pytest.mark.parametrize("N,K", [(32, 2048), (24, 4096)])
def test_draft_gemv_clustered_masks(cas, orc, N, K, nvec):
    W = clustered_rows(N, K, seed=N + K)
    x = synthetic.activations(nvec, K, seed=41 + nvec)
    enc = cas.encode_weights(W.cuda(), 1, 64, 3)
    y = cas.draft_gemv(enc, x.cuda())
    ref, norm = orc.matvec(orc.draft_values(np16(W), 1, 64, 3), np16(x))
    check_close(y, ref, norm, "draft_gemv clustered masks")


@pytest.mark.parametrize("keep", [64, 38])
@pytest.mark.parametrize("nvec", [1, 2])
@pytest.mark.parametrize("N,K,kind", [(3, 4096, "t4"), (5, 14336, "t4"), (7, 5120, "t4"), (9, 8192, "t4"),
                                       (6, 5120, "clustered"), (11, 14336, "clustered")])
def test_draft_gemv_block_chunks(cas, orc, N, K, kind, nvec, keep):
    """Rows of 32 or more blocks: a warp decodes 32 consecutive blocks (four
    superblocks) at once, for keep 64 and 38 of 128, so chunks span two rows
    (K = 5120, 14336), the last
    chunk of a matrix can hold fewer than four superblocks (N * K / 1024 not a
    multiple of 4), and chunks with long codes or long runs of pruned
    positions (clustered rows) go to the generic decoder."""
    W = synthetic.t4_weight(N, K, seed=N + K) if kind == "t4" else clustered_rows(N, K, seed=2 * N + K)
    x = synthetic.activations(nvec, K, seed=17 + nvec)
    enc = cas.encode_weights(W.cuda(), 1, keep, 3)
    y = cas.draft_gemv(enc, x.cuda())
    ref, norm = orc.matvec(orc.draft_values(np16(W), 1, keep, 3), np16(x))
    check_close(y, ref, norm, "draft_gemv block chunks")


@pytest.mark.parametrize("T", [1, 5, 13])
@pytest.mark.parametrize("N,K,kind", [(3, 1024, "t4"), (21, 4096, "t4"), (35, 5120, "t4"), (18, 2048, "clustered"),
                                       (40, 1024, "wide")])
def test_verify_gemm_block_tiles(cas, orc, N, K, kind, T):
    """The verify GEMM rebuilds 16-row tiles with one lane per block: row
    counts that leave the last tile partly empty, clustered masks whose long
    runs of kept or pruned positions and rows whose long codes send a warp's
    row-superblocks to the generic decoder, against the exact product."""
    if kind == "t4":
        W = synthetic.t4_weight(N, K, seed=N + K + T)
    elif kind == "clustered":
        W = clustered_rows(N, K, seed=N + K)
    else:
        W = wide_exponent_rows(N, K, 6, seed=N + T)
    X = synthetic.activations(T, K, seed=23 + T)
    enc = cas.encode_weights(W.cuda(), 1, 64, 3)
    Y = cas.verify_gemm(enc, X.cuda())
    ref, norm = orc.matvec(np16(W), np16(X))
    check_close(Y, ref, norm, "verify_gemm block tiles")


@pytest.mark.parametrize("nvec", [1, 2])
@pytest.mark.parametrize("kind", ["t4", "wide", "clustered"])
def test_draft_gemv_rows_of_one_chunk(cas, orc, kind, nvec):
    """Rows of exactly 32 blocks (K = 4096): one warp owns each row, so the
    lane-per-block kernel stores the row sum (y is not cleared first) or adds
    it to y (the accumulating call), also for rows whose long codes send the
    chunk to the generic decoder or whose clustered masks make a lane scan its
    block again. y starts as NaN (plain call) or random (accumulating call)."""
    N, K = 24, 4096
    if kind == "t4":
        W = synthetic.t4_weight(N, K, seed=31)
    elif kind == "wide":
        W = wide_exponent_rows(N, K, 5, seed=32)
    else:
        W = clustered_rows(N, K, seed=33)
    x = synthetic.activations(nvec, K, seed=34 + nvec).cuda()
    enc = cas.encode_weights(W.cuda(), 1, 64, 3)
    ref, norm = orc.matvec(orc.draft_values(np16(W), 1, 64, 3), np16(x.cpu()))
    y = torch.full((nvec, N), float("nan"), dtype=torch.float32, device="cuda")
    cas.cas_draft_gemv(enc, x, y)
    check_close(y, ref, norm, "draft_gemv rows of one chunk")
    g = torch.Generator().manual_seed(35)
    y0 = torch.randn(nvec, N, generator=g)
    ya = cas.cas_draft_gemv_accumulate(enc, x, y0.clone().cuda())
    check_close(ya - y0.cuda(), ref, norm, "draft_gemv_accumulate rows of one chunk")


@pytest.mark.parametrize("N,K,T", [(24, 4096, 5), (40, 2048, 3), (17, 1152, 9)])
def test_verify_gemm_accumulate(cas, orc, N, K, T):
    """The accumulating verify GEMM adds W X to a given Y (for the block-walk
    kernel and the other tile decoders), and the plain one overwrites it."""
    W = synthetic.t4_weight(N, K, seed=N + K + T)
    X = synthetic.activations(T, K, seed=T + 3)
    enc = cas.encode_weights(W.cuda(), 1, 64, 3)
    ref, norm = orc.matvec(np16(W), np16(X))
    g = torch.Generator().manual_seed(N)
    Y0 = torch.randn(T, N, generator=g)
    Ya = cas.cas_verify_gemm_accumulate(enc, X.cuda(), Y0.clone().cuda())
    check_close(Ya - Y0.cuda(), ref, norm, "verify_gemm_accumulate")
    Yp = cas.cas_verify_gemm(enc, X.cuda(), Y0.clone().cuda())
    check_close(Yp, ref, norm, "verify_gemm over a given Y")
