"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these checks re-types the oracle's own code: value pruning is checked by
brute force over subsets, the draft values by float64 arithmetic on the decoded
magnitude, the rank table by a Counter sort, the byte layout by a string-of-bits
restatement and a hand-derived block, the products by exact rational sums and
library routines.
"""
import itertools
import math
from collections import Counter
from fractions import Fraction

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.filterwarnings("ignore")


def bits_to_f64(a):
    a = np.asarray(a, np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- value pruning
def _brute_keep(blk, k):
    """The unique k-subset S whose every member outranks every non-member, where
    i outranks j when |x_i| > |x_j|, or equal magnitude bits and i < j."""
    B = len(blk)
    key = [int(v) & 0x7FFF for v in blk]
    found = []
    for S in itertools.combinations(range(B), k):
        s = set(S)
        ok = all((key[i] > key[j]) or (key[i] == key[j] and i < j)
                 for i in s for j in range(B) if j not in s)
        if ok:
            found.append(s)
    assert len(found) == 1
    keep = np.zeros(B, bool)
    keep[list(found[0])] = True
    return keep


@pytest.mark.parametrize("B", [6, 8])
def test_select_block_brute_force(orc, B):
    rng = np.random.default_rng(1)
    for trial in range(60):
        if trial % 3 == 0:   # many ties, signs that must not matter
            blk = rng.choice(np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x3F00], np.uint16), B)
        else:
            blk = rng.integers(0, 0x7F80, B).astype(np.uint16) | (rng.integers(0, 2, B).astype(np.uint16) << 15)
        for k in range(B + 1):
            assert (orc.select_block(blk, k) == _brute_keep(blk, k)).all(), (blk, k)


def test_select_block_128_matches_lexsort(orc):
    rng = np.random.default_rng(2)
    for _ in range(20):
        blk = rng.integers(0, 0x7F80, 128).astype(np.uint16)
        blk[rng.integers(0, 128, 30)] = blk[0]  # ties
        for k in (0, 1, 26, 38, 64, 77, 127, 128):
            order = np.lexsort((np.arange(128), -(blk.astype(np.int64) & 0x7FFF)))
            ref = np.zeros(128, bool)
            ref[order[:k]] = True
            assert (orc.select_block(blk, k) == ref).all()


# ---------------------------------------------------------------- rank table
def test_rank_table_counter_sort(orc):
    rng = np.random.default_rng(3)
    for _ in range(5):
        w = (rng.integers(100, 140, 5000).astype(np.uint16) << 7) | rng.integers(0, 128, 5000).astype(np.uint16)
        cnt = Counter(int((v >> 7) & 0xFF) for v in w)
        ref = sorted(range(256), key=lambda e: (-cnt.get(e, 0), e))
        c = orc.exp_hist(w)
        eor, roe = orc.rank_table(c)
        assert list(eor) == ref
        assert all(roe[e] == r for r, e in enumerate(ref))
        assert sorted(eor) == list(range(256))


def test_unary_ranking_is_optimal_among_unary_codes(orc):
    """A unary code of rank r costs r+1 bits, so sorting by count descending is
    the best assignment of ranks: no permutation gives a shorter mean."""
    w = synthetic.normal_weight(256, 512, seed=5, outlier_frac=0.001).numpy().view(np.uint16)
    c = orc.exp_hist(w)
    _, roe = orc.rank_table(c)
    best = orc.unary_mean_len(c, roe)
    rng = np.random.default_rng(0)
    assert best <= orc.unary_mean_len(c, np.arange(256)) + 1e-12
    assert best <= orc.unary_mean_len(c, 255 - np.arange(256)) + 1e-12
    for _ in range(20):
        assert best <= orc.unary_mean_len(c, rng.permutation(256)) + 1e-12


# ---------------------------------------------------------------- entropy (blog 3.2 / Fig. 6)
def test_exponent_stats_weights(orc):
    """Weight exponents carry about 2.6 bits of entropy and the unary code costs
    about 2.85 bits (blog section 3.2). Shannon bound: mean length >= entropy."""
    w = synthetic.cfg0_weight().numpy().view(np.uint16)
    c = orc.exp_hist(w)
    _, roe = orc.rank_table(c)
    H, u = orc.exp_entropy(c), orc.unary_mean_len(c, roe)
    assert 2.45 <= H <= 2.8
    assert abs(u - 2.85) <= 0.25
    assert u >= H
    # entropy of a uniform exponent histogram is exactly log2 of its support
    flat = np.zeros(256, np.uint64)
    flat[100:108] = 10
    assert orc.exp_entropy(flat) == pytest.approx(3.0)


def test_exponent_stats_kv(orc):
    """KV exponents: about 2.7-2.8 bits of entropy (blog section 3.2)."""
    sc = synthetic.kv_scales(0, 8, 0)
    kv = synthetic.kv_tokens(2048, 8, seed=11, scales=sc).numpy().view(np.uint16)
    c = orc.exp_hist(kv)
    _, roe = orc.rank_table(c)
    H, u = orc.exp_entropy(c), orc.unary_mean_len(c, roe)
    assert 2.6 <= H <= 2.9
    assert u >= H
    assert abs(u - 2.85) <= 0.35


# ---------------------------------------------------------------- draft values (blog 3.1 / 3.2)
def _kept_mask(orc, W, k):
    N, K = W.shape
    return np.stack([orc.select_block(W.reshape(-1, 128)[b], k) for b in range(N * K // 128)]).reshape(N, K)


@pytest.mark.parametrize("k,m", [(64, 3), (38, 3), (128, 0), (1, 7), (90, 5)])
def test_c1_draft_is_truncated_subset(orc, k, m):
    """Cassandra-1 draft: pruned values are zero, kept values are the original
    truncated toward zero to m mantissa bits, i.e. floor(|x|/u)*u with u one unit
    of the m-th mantissa bit of x's binade."""
    W = synthetic.normal_weight(8, 512, seed=7, outlier_frac=0.01).numpy().view(np.uint16).copy()
    W[0, :128] = np.arange(128, dtype=np.uint16)          # subnormals and +0
    W[1, :128] = np.arange(128, dtype=np.uint16) | 0x8000  # negative subnormals and -0
    d = orc.draft_values(W, 1, k, m)
    keep = _kept_mask(orc, W, k)
    x = bits_to_f64(W)
    e = ((W >> 7) & 0xFF).astype(np.int64)
    u = np.ldexp(1.0, np.maximum(e, 1) - 127 - m)
    ref = np.where(keep, np.sign(x) * np.floor(np.abs(x) / u) * u, 0.0)
    got = bits_to_f64(d)
    assert np.array_equal(got, ref)
    # pruned slots are +0 bit patterns; kept slots keep the sign bit
    assert (d[~keep] == 0).all()
    assert ((d[keep] >> 15) == (W[keep] >> 15)).all()
    assert keep.sum() == k * W.size // 128


@pytest.mark.parametrize("k,m", [(64, 3), (38, 1), (128, 5), (26, 0), (96, 7)])
def test_c2_draft_properties(orc, k, m):
    """Cassandra-2 (MX shared exponent per 32 values): every kept draft value is a
    multiple of the group grid u = 2^(E'-127-m) no larger in magnitude than x and
    within one grid step of it; a value whose exponent is the group maximum gets
    exactly its Cassandra-1 draft; pruned values are zero."""
    W = synthetic.normal_weight(6, 1024, seed=9, outlier_frac=0.02).numpy().view(np.uint16).copy()
    W[0, :64] = np.arange(64, dtype=np.uint16) * 2  # subnormal group
    d2 = orc.draft_values(W, 2, k, m)
    d1 = orc.draft_values(W, 1, k, m)
    keep = _kept_mask(orc, W, k)
    x, y = bits_to_f64(W), bits_to_f64(d2)
    e = ((W >> 7) & 0xFF).astype(np.int64)
    eg = np.where(keep, e, 0).reshape(-1, 32)
    E = np.maximum(eg.max(1, keepdims=True), 1)
    u = np.broadcast_to(np.ldexp(1.0, E - 127 - m), eg.shape).reshape(W.shape)
    assert (d2[~keep] == 0).all()
    xs, ys, us = np.abs(x[keep]), np.abs(y[keep]), u[keep]
    assert (ys <= xs).all()
    assert (xs - ys < us).all()
    assert np.array_equal(np.mod(ys, us), np.zeros_like(ys))
    assert ((d2[keep] >> 15) == (W[keep] >> 15)).all()
    top = keep & (e.reshape(-1, 32) == np.where(eg.max(1, keepdims=True) == 0, -1, eg.max(1, keepdims=True))).reshape(W.shape)
    top &= e > 0
    assert top.sum() > 0
    assert np.array_equal(d2[top], d1[top])


# ---------------------------------------------------------------- lossless split (blog 3.1)
def _all_finite_patterns():
    v = np.arange(65536, dtype=np.uint32)
    v = v[((v >> 7) & 0xFF) != 255].astype(np.uint16)
    assert v.size == 65280
    rng = np.random.default_rng(4)
    pad = rng.choice(v, 65536 - v.size)
    return rng.permutation(np.concatenate([v, pad])).reshape(64, 1024)


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("k,m", [(64, 3), (0, 3), (128, 0), (128, 7), (38, 5), (101, 1)])
def test_lossless_all_finite_patterns(orc, variant, k, m):
    """Verification data united with speculation data rebuilds every finite bf16
    value bit for bit (blog section 3.1: the target merges both losslessly), and
    the speculation data alone decodes to the draft values."""
    W = _all_finite_patterns()
    enc = orc.encode(W, variant, k, m)
    assert np.array_equal(orc.decode(enc, True), W)
    assert np.array_equal(orc.decode(enc, False), orc.draft_values(W, variant, k, m))


@pytest.mark.parametrize("variant", [1, 2])
def test_lossless_adversarial_blocks(orc, variant):
    W = np.zeros((4, 1152), np.uint16)       # 9 blocks per row: a ragged superblock tail
    W[1] = 0x3F80                            # 128 equal values per block
    W[2, ::2] = 0x8000                       # -0 / +0 mix
    W[3] = np.tile(np.array([0x0001, 0x807F, 0x7F7F, 0xFF7F], np.uint16), 288)  # extremes
    for k, m in ((64, 3), (1, 0), (127, 6)):
        enc = orc.encode(W, variant, k, m)
        assert np.array_equal(orc.decode(enc, True), W)
        assert np.array_equal(orc.decode(enc, False), orc.draft_values(W, variant, k, m))


def test_nonfinite_and_shape_rejected(orc):
    W = np.zeros((2, 256), np.uint16)
    W[1, 5] = 0x7F80  # +inf
    with pytest.raises(orc.OracleError):
        orc.encode(W, 1, 64, 3)
    W[1, 5] = 0x7FC1  # nan
    with pytest.raises(orc.OracleError):
        orc.encode(W, 2, 64, 3)
    with pytest.raises(orc.OracleError):
        orc.encode(np.zeros((2, 200), np.uint16), 1, 64, 3)


# ---------------------------------------------------------------- byte layout
def test_layout_hand_derived_block(orc):
    """One block: positions 0..63 hold +1.5 (0x3FC0: e=127, f=0x40), positions
    64..127 hold -0.25 (0xBE80: e=125, f=0). k=64, m=3, Cassandra-1.
    Worked by hand from the format definition:
      keys 0x3FC0 > 0x3E80 -> positions 0..63 kept  -> mask words FFFFFFFF FFFFFFFF 0 0
      counts e127:64, e125:64, tie -> lower exponent first: rank(125)=0, rank(127)=1
      kept field (s<<3)|f>>4 = 4, 64 fields of 4 bits LSB-first -> 8 words 0x44444444
      kept codes rank 1 = '01', 64 of them MSB-first -> 4 words 0x55555555, index [0, 4]
      cut bits f & 15 = 0 -> 8 zero words
      pruned bytes (1<<7)|0 = 0x80 -> 16 words 0x80808080
      pruned codes rank 0 = '1' x 64 -> 2 words 0xFFFFFFFF, index [0, 2]
    """
    W = np.array([[0x3FC0] * 64 + [0xBE80] * 64], np.uint16)
    enc = orc.encode(W, 1, 64, 3)
    w32 = lambda n: enc.section(n).view(np.uint32).tolist()  # noqa: E731
    assert w32("mask") == [0xFFFFFFFF, 0xFFFFFFFF, 0, 0]
    assert w32("spec_sm") == [0x44444444] * 8
    assert w32("spec_exp") == [0x55555555] * 4
    assert w32("spec_sbidx") == [0, 4]
    assert w32("ver_lo") == [0] * 8
    assert w32("ver_pr") == [0x80808080] * 16
    assert w32("ver_exp") == [0xFFFFFFFF] * 2
    assert w32("ver_sbidx") == [0, 2]
    assert all(o % 256 == 0 for o in enc.off)


def _pack(bitstr, msb_first):
    """'0'/'1' string -> u32 words, zero padded to a word."""
    bitstr = bitstr + "0" * (-len(bitstr) % 32)
    out = []
    for i in range(0, len(bitstr), 32):
        chunk = bitstr[i:i + 32]
        out.append(int(chunk, 2) if msb_first else int(chunk[::-1], 2))
    return out


def _fields(vals, width):
    return "".join(format(v, f"0{width}b")[::-1] for v in vals) if width else ""


def _restate(W, variant, k, m, roe, keep):
    """Independent restatement of the sections from the format definition,
    building each stream as a string of bits."""
    N, K = W.shape
    nbr = K // 128
    nsr = -(-nbr // 8)
    sec = {n: [] for n in ("mask", "spec_sm", "spec_exp", "spec_sbidx", "spec_mx", "spec_q", "ver_lo",
                           "ver_d", "ver_d_sbidx", "ver_res", "ver_res_sbidx", "ver_pr", "ver_exp", "ver_sbidx")}
    idx = {"spec_exp": [0], "ver_exp": [0], "ver_d": [0], "ver_res": [0]}
    for n in range(N):
        for j in range(nsr):
            streams = {"spec_exp": "", "ver_exp": "", "ver_d": "", "ver_res": ""}
            for b in range(j * 8, min(j * 8 + 8, nbr)):
                x = [int(v) for v in W[n, b * 128:(b + 1) * 128]]
                kp = keep[n, b * 128:(b + 1) * 128]
                sec["mask"] += _pack("".join("1" if t else "0" for t in kp), False)
                kept = [v for v, t in zip(x, kp) if t]
                pruned = [v for v, t in zip(x, kp) if not t]
                sec["ver_pr"] += _pack(_fields([((v >> 15) << 7) | (v & 0x7F) for v in pruned], 8), False) \
                    if 128 - k else []
                streams["ver_exp"] += "".join("0" * int(roe[(v >> 7) & 0xFF]) + "1" for v in pruned)
                if variant == 1:
                    if k:
                        sec["spec_sm"] += _pack(_fields([((v >> 15) << m) | ((v & 0x7F) >> (7 - m)) for v in kept], m + 1), False)
                    if k and m < 7:
                        sec["ver_lo"] += _pack(_fields([v & ((1 << (7 - m)) - 1) for v in kept], 7 - m), False)
                    streams["spec_exp"] += "".join("0" * int(roe[(v >> 7) & 0xFF]) + "1" for v in kept)
                else:
                    E = []
                    for g in range(4):
                        es = [(x[p] >> 7) & 0xFF for p in range(32 * g, 32 * g + 32) if kp[p]]
                        E.append(max(es) if es else 0)
                    sec["spec_mx"].append(bytes(E))
                    qs = []
                    t = 0
                    for p in range(128):
                        if not kp[p]:
                            continue
                        v = x[p]
                        e = (v >> 7) & 0xFF
                        sig = (0x80 if e else 0) | (v & 0x7F)
                        d = max(E[p // 32], 1) - max(e, 1)
                        sh = 7 - m + d
                        qs.append(((v >> 15) << (m + 1)) | (sig >> sh if sh < 8 else 0))
                        streams["ver_d"] += "0" * d + "1"
                        w = min(sh, 8)
                        streams["ver_res"] += format(sig & ((1 << w) - 1), f"0{w}b")[::-1] if w else ""
                        t += 1
                    if k:
                        sec["spec_q"] += _pack(_fields(qs, m + 2), False)
            for s, msb in (("spec_exp", True), ("ver_exp", True), ("ver_d", True), ("ver_res", False)):
                words = _pack(streams[s], msb) if streams[s] else []
                sec[s] += words
                idx[s].append(idx[s][-1] + len(words))
    out = {}
    for name, val in sec.items():
        if name == "spec_mx":
            out[name] = b"".join(val)
        else:
            out[name] = np.array(val, np.uint32).tobytes()
    if variant == 1:
        out["spec_sbidx"] = np.array(idx["spec_exp"], np.uint32).tobytes()
    else:
        out["ver_d_sbidx"] = np.array(idx["ver_d"], np.uint32).tobytes()
        out["ver_res_sbidx"] = np.array(idx["ver_res"], np.uint32).tobytes()
    out["ver_sbidx"] = np.array(idx["ver_exp"], np.uint32).tobytes()
    return out


@pytest.mark.parametrize("variant,k,m,shape", [
    (1, 64, 3, (1, 128)), (1, 38, 3, (2, 1152)), (1, 77, 2, (1, 512)), (1, 128, 7, (1, 256)),
    (2, 64, 3, (1, 128)), (2, 38, 1, (2, 1152)), (2, 90, 5, (1, 512)), (2, 0, 4, (1, 256)),
])
def test_layout_matches_bitstring_restatement(orc, variant, k, m, shape):
    W = synthetic.normal_weight(*shape, seed=13, outlier_frac=0.02).numpy().view(np.uint16)
    c = orc.exp_hist(W)
    eor, roe = orc.rank_table(c)
    enc = orc.encode(W, variant, k, m, roe, eor)
    keep = np.stack([orc.select_block(W.reshape(-1, 128)[b], k) for b in range(W.size // 128)]).reshape(W.shape)
    ref = _restate(W, variant, k, m, roe, keep)
    for name, want in ref.items():
        got = enc.section(name).tobytes()
        assert got == want, name


# ---------------------------------------------------------------- products
def test_matvec_exact_rational(orc):
    """Double-precision sums of bf16 products against exact rational sums."""
    A = synthetic.normal_weight(5, 256, seed=21).numpy().view(np.uint16)
    x = synthetic.activations(2, 256, seed=22).numpy().view(np.uint16)
    y, ad = orc.matvec(A, x)
    Af, xf = bits_to_f64(A), bits_to_f64(x)
    for v in range(2):
        for n in range(5):
            exact = sum(Fraction(float(Af[n, i])) * Fraction(float(xf[v, i])) for i in range(256))
            mag = sum(abs(Fraction(float(Af[n, i])) * Fraction(float(xf[v, i]))) for i in range(256))
            assert abs(Fraction(y[v, n]) - exact) <= Fraction(1, 10**12) * mag
            assert ad[v, n] == pytest.approx(float(mag), rel=1e-12)
    # non-square shapes: the rows of A pair with the rows of x, not a transpose
    A2 = synthetic.normal_weight(3, 384, seed=23).numpy().view(np.uint16)
    x2 = synthetic.activations(4, 384, seed=24).numpy().view(np.uint16)
    y2, _ = orc.matvec(A2, x2)
    assert y2.shape == (4, 3)
    assert np.allclose(y2, bits_to_f64(x2) @ bits_to_f64(A2).T, rtol=1e-12, atol=1e-12)


def test_attention_matches_sdpa(orc):
    """float64 GQA attention against torch's scaled_dot_product_attention."""
    T, Hq, Hkv, D = 37, 8, 2, 128
    q = synthetic.activations(1, Hq * D, seed=31).numpy().view(np.uint16).reshape(1, Hq, D)
    Kc = synthetic.activations(T, Hkv * D, seed=32).numpy().view(np.uint16).reshape(T, Hkv, D)
    Vc = synthetic.activations(T, Hkv * D, seed=33).numpy().view(np.uint16).reshape(T, Hkv, D)
    o, nrm = orc.attention(q, Kc, Vc)
    qt = torch.from_numpy(bits_to_f64(q)).permute(1, 0, 2)           # [Hq][1][D]
    kt = torch.from_numpy(bits_to_f64(Kc)).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    vt = torch.from_numpy(bits_to_f64(Vc)).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).permute(1, 0, 2).numpy()
    assert np.allclose(o, ref, rtol=1e-10, atol=1e-12)
    assert (nrm >= np.abs(o) - 1e-12).all()
    # causal verify: Tq queries are the last Tq tokens
    Tq = 5
    q5 = synthetic.activations(Tq, Hq * D, seed=34).numpy().view(np.uint16).reshape(Tq, Hq, D)
    o5, _ = orc.attention(q5, Kc, Vc, causal_new=Tq)
    for j in range(Tq):
        vis = T - Tq + j + 1
        qj = torch.from_numpy(bits_to_f64(q5[j:j + 1])).permute(1, 0, 2)
        r = torch.nn.functional.scaled_dot_product_attention(qj, kt[:, :vis], vt[:, :vis]).permute(1, 0, 2).numpy()
        assert np.allclose(o5[j:j + 1], r, rtol=1e-10, atol=1e-12)
