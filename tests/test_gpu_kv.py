"""GPU parity of the compressed KV cache and the attention kernels, both
variants (Cassandra-1 unary exponent codes, Cassandra-2 shared exponents).

Online append: every stream byte-exact with the oracle's encoding of the same
tokens (a stream = one row whose blocks are the tokens); chunked appends equal
token-by-token appends; truncate + re-append equals a direct append; data
faults set the sticky status and write nothing. Attention: within
2e-3 * sum_t p_t |v_t| of the float64 oracle over the oracle's draft (resp.
exact) K and V.
"""
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


def np16(t):
    return t.cpu().numpy().view(np.uint16)


def make_tokens(T, H, layer=0, seed=0):
    K = synthetic.kv_tokens(T, H, seed=seed, scales=synthetic.kv_scales(layer, H, 0))
    V = synthetic.kv_tokens(T, H, seed=seed + 1, scales=synthetic.kv_scales(layer, H, 1))
    return K, V


def new_cache(cas, H, Tm, K, V, k=64, m=3, calib=16, est=6.0, variant=1):
    return cas.KVCache(H, Tm, cas.params(variant, k, m), K[:calib].cuda(), V[:calib].cuda(), est)


def stream_sections(kv, st, n):
    """Valid bytes of every section of stream st holding n tokens."""
    k, m = kv.desc.p.keep_per_block, kv.desc.p.mant_bits
    rec = lambda f, w: -(-(f * w) // 32)  # noqa: E731
    nsb = -(-n // 8)
    sec = lambda name: kv.section(name, st).cpu().numpy()  # noqa: E731
    out = {"mask": sec("mask")[:n * 16], "ver_pr": sec("ver_pr")[:n * rec(128 - k, 8) * 4]}

    def stream(words, index):
        ix = sec(index).view(np.uint32)[:nsb + 1]
        out[index] = ix.tobytes()
        out[words] = sec(words)[:int(ix[-1]) * 4]

    stream("ver_exp", "ver_sbidx")
    if kv.desc.p.variant == 1:
        out["spec_sm"] = sec("spec_sm")[:n * rec(k, m + 1) * 4]
        out["ver_lo"] = sec("ver_lo")[:n * rec(k, 7 - m) * 4]
        stream("spec_exp", "spec_sbidx")
    else:
        out["spec_mx"] = sec("spec_mx")[:n * 4]
        out["spec_q"] = sec("spec_q")[:n * rec(k, m + 2) * 4]
        stream("ver_d", "ver_d_sbidx")
        stream("ver_res", "ver_res_sbidx")
    return out


def state_bytes(kv):
    o = int(kv.desc.off[0])
    return kv.buf[o:o + 32 + 24 * 2 * kv.H].cpu()


def assert_streams_equal(a, b):
    for key in a:
        x, y = a[key], b[key]
        x = x.tobytes() if hasattr(x, "tobytes") else x
        y = y.tobytes() if hasattr(y, "tobytes") else y
        assert x == y, key


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("T,k,m", [(37, 64, 3), (8, 64, 3), (64, 38, 3), (19, 128, 7), (11, 0, 2), (29, 77, 5),
                                   (21, 128, 0)])
def test_append_matches_oracle(cas, orc, T, k, m, variant):
    H = 3
    K, V = make_tokens(T, H, seed=T)
    kv = new_cache(cas, H, 100, K, V, k, m, calib=min(16, T), variant=variant)
    kv.append(K.cuda(), V.cuda())
    n, st = kv.status()
    assert (n, st) == (T, 0)
    for kvi, src in ((0, K), (1, V)):
        calib = np16(src[:min(16, T)])
        for h in range(H):
            s = kvi * H + h
            roe, eor = kv.tables(kvi, h)
            c = orc.exp_hist(calib[:, h])
            eor_ref, roe_ref = orc.rank_table(c)
            assert np.array_equal(eor, eor_ref) and np.array_equal(roe, roe_ref)
            ref = orc.kv_stream_encode(np16(src[:, h]), variant, k, m, roe, eor)
            got = stream_sections(kv, s, T)
            for name, val in got.items():
                want = ref.section(name).tobytes()
                val = val if isinstance(val, bytes) else val.tobytes()
                assert val == want, (name, kvi, h)


@pytest.mark.parametrize("variant", [1, 2])
def test_chunked_equals_token_by_token(cas, variant):
    H, T = 2, 45
    K, V = make_tokens(T, H, seed=5)
    a = new_cache(cas, H, 64, K, V, variant=variant)
    b = new_cache(cas, H, 64, K, V, variant=variant)
    a.append(K.cuda(), V.cuda())
    for t in range(T):
        b.append(K[t:t + 1].cuda(), V[t:t + 1].cuda())
    for chunks in ((3, 17, 25), ):
        c = new_cache(cas, H, 64, K, V, variant=variant)
        p = 0
        for e in chunks + (T,):
            c.append(K[p:e].cuda(), V[p:e].cuda())
            p = e
        for s in range(2 * H):
            assert_streams_equal(stream_sections(a, s, T), stream_sections(c, s, T))
    for s in range(2 * H):
        assert_streams_equal(stream_sections(a, s, T), stream_sections(b, s, T))
    assert torch.equal(state_bytes(a), state_bytes(b))


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("cut", [0, 1, 7, 8, 9, 30, 40])
def test_truncate_then_append(cas, cut, variant):
    H, T = 2, 40
    K, V = make_tokens(T, H, seed=9)
    K2, V2 = make_tokens(T, H, seed=77)
    ref = new_cache(cas, H, 96, K, V, variant=variant)
    ref.append(K[:cut].cuda(), V[:cut].cuda())
    ref.append(K2.cuda(), V2.cuda())
    kv = new_cache(cas, H, 96, K, V, variant=variant)
    kv.append(K.cuda(), V.cuda())
    kv.truncate(cut)
    assert kv.status() == (cut, 0)
    kv.append(K2.cuda(), V2.cuda())
    assert kv.status() == (cut + T, 0)
    for s in range(2 * H):
        assert_streams_equal(stream_sections(ref, s, cut + T), stream_sections(kv, s, cut + T))
    assert torch.equal(state_bytes(ref), state_bytes(kv))
    kv.truncate(10**9)  # larger than the count: unchanged
    assert kv.status() == (cut + T, 0)


@pytest.mark.parametrize("variant", [1, 2])
def test_capacity_and_nonfinite_write_nothing(cas, variant):
    H = 2
    K, V = make_tokens(24, H, seed=3)
    kv = new_cache(cas, H, 16, K, V, variant=variant)
    kv.append(K[:10].cuda(), V[:10].cuda())
    before = kv.buf.clone()
    kv.append(K[10:24].cuda(), V[10:24].cuda())  # 24 > 16 tokens
    n, st = kv.status()
    assert (n, st) == (10, -4)
    so = int(kv.desc.off[0])
    assert torch.equal(kv.buf[:so + 8], before[:so + 8])
    assert torch.equal(kv.buf[so + 12:], before[so + 12:])
    kv.clear_status()
    assert kv.status() == (10, 0)
    Kb = K[10:12].clone()
    Kb[1, 1, 5] = 0x7FC1  # NaN
    kv.append(Kb.cuda(), V[10:12].cuda())
    assert kv.status() == (10, -3)
    assert torch.equal(kv.buf[so + 12:], before[so + 12:])
    kv.clear_status()
    kv.append(K[10:12].cuda(), V[10:12].cuda())
    assert kv.status() == (12, 0)
    # code-stream capacity: a tiny estimate of bits per code overflows the stream
    small = new_cache(cas, H, 64, K, V, est=0.05, variant=variant)
    small.append(K.cuda(), V.cuda())
    assert small.status() == (0, -4)


def oracle_draft_kv(orc, toks, k, m, variant=1):
    T, H, _ = toks.shape
    a = np16(toks)
    return np.stack([orc.draft_values(a[:, h].reshape(1, T * D), variant, k, m).reshape(T, D) for h in range(H)], 1)


def check_attn(o, ref, nrm, what):
    o = o.double().cpu().numpy()
    bound = TOL * nrm + 1e-6
    bad = np.abs(o - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} bad, worst {(np.abs(o - ref) / bound).max():.3g}"


@pytest.mark.parametrize("lens,n_tail,variant,k,m", [
    ((300,), 0, 1, 64, 3), ((1, ), 1, 1, 64, 3), ((517, 64), 3, 1, 64, 3), ((0,), 2, 1, 64, 3),
    ((256, 1000), 4, 1, 64, 3), ((300,), 0, 2, 64, 3), ((517, 64), 3, 2, 64, 3), ((777,), 1, 2, 48, 4),
    ((99,), 2, 1, 40, 2)])
def test_draft_attention(cas, orc, lens, n_tail, variant, k, m):
    H, Hq = 8, 32
    B = len(lens)
    caches, Ks, Vs = [], [], []
    for b, T in enumerate(lens):
        K, V = make_tokens(max(T, 16), H, layer=b, seed=31 + b)
        kv = new_cache(cas, H, 1100, K, V, k, m, variant=variant)
        if T:
            kv.append(K[:T].cuda(), V[:T].cuda())
        assert kv.status() == (T, 0)
        caches.append(kv)
        Ks.append(K[:T])
        Vs.append(V[:T])
    q = synthetic.activations(B, Hq * D, seed=40).view(B, Hq, D)
    tk = synthetic.activations(B * max(n_tail, 1), H * D, seed=41).view(B, max(n_tail, 1), H, D)[:, :n_tail]
    tv = synthetic.activations(B * max(n_tail, 1), H * D, seed=42).view(B, max(n_tail, 1), H, D)[:, :n_tail]
    o = cas.draft_attn_decode(caches, q.cuda(), tk.contiguous().cuda() if n_tail else None,
                              tv.contiguous().cuda() if n_tail else None)
    for b in range(B):
        Kd = oracle_draft_kv(orc, Ks[b], k, m, variant) if lens[b] else np.zeros((0, H, D), np.uint16)
        Vd = oracle_draft_kv(orc, Vs[b], k, m, variant) if lens[b] else np.zeros((0, H, D), np.uint16)
        Kall = np.concatenate([Kd, np16(tk[b])], 0)
        Vall = np.concatenate([Vd, np16(tv[b])], 0)
        if Kall.shape[0] == 0:
            assert torch.all(o[b] == 0)
            continue
        ref, nrm = orc.attention(np16(q[b:b + 1]), Kall, Vall)
        check_attn(o[b:b + 1], ref, nrm, f"draft attention b={b}")


@pytest.mark.parametrize("Hq", [8, 16, 64])
def test_draft_attention_gqa_ratios(cas, orc, Hq):
    """1, 2 and 8 query heads per kv head (the fused kernel takes up to 4 query
    vectors per kv head, the chunk kernel more)."""
    H, T = 8, 600
    K, V = make_tokens(T, H, layer=2, seed=71)
    kv = new_cache(cas, H, 700, K, V)
    kv.append(K.cuda(), V.cuda())
    assert kv.status() == (T, 0)
    q = synthetic.activations(1, Hq * D, seed=72).view(1, Hq, D)
    tk = synthetic.activations(2, H * D, seed=73).view(1, 2, H, D)
    tv = synthetic.activations(2, H * D, seed=74).view(1, 2, H, D)
    o = cas.draft_attn_decode([kv], q.cuda(), tk.contiguous().cuda(), tv.contiguous().cuda())
    Kall = np.concatenate([oracle_draft_kv(orc, K, 64, 3), np16(tk[0])], 0)
    Vall = np.concatenate([oracle_draft_kv(orc, V, 64, 3), np16(tv[0])], 0)
    ref, nrm = orc.attention(np16(q), Kall, Vall)
    check_attn(o, ref, nrm, f"draft attention Hq={Hq}")


@pytest.mark.parametrize("lens,T,variant", [((300,), 5, 1), ((5,), 5, 1), ((517, 40), 7, 1), ((1024,), 14, 1),
                                            ((260,), 16, 1), ((9,), 1, 1), ((517, 40), 7, 2), ((1024,), 14, 2),
                                            ((9,), 1, 2)])
def test_verify_attention(cas, orc, lens, T, variant):
    H, Hq = 8, 32
    B = len(lens)
    caches, Ks, Vs = [], [], []
    for b, n in enumerate(lens):
        K, V = make_tokens(max(n, 16), H, layer=b, seed=51 + b)
        kv = new_cache(cas, H, 1100, K, V, variant=variant)
        kv.append(K[:n].cuda(), V[:n].cuda())
        assert kv.status() == (n, 0)
        caches.append(kv)
        Ks.append(K[:n])
        Vs.append(V[:n])
    q = synthetic.activations(B * T, Hq * D, seed=60).view(B, T, Hq, D)
    o = cas.verify_attn(caches, q.cuda())
    for b in range(B):
        ref, nrm = orc.attention(np16(q[b]), np16(Ks[b]), np16(Vs[b]), causal_new=T)
        check_attn(o[b], ref, nrm, f"verify attention b={b}")


@pytest.mark.parametrize("variant,k,m", [(1, 38, 3), (2, 38, 2), (1, 100, 6), (2, 77, 5), (1, 128, 7), (2, 0, 3),
                                         (1, 0, 0), (2, 128, 7)])
def test_attention_any_k_m(cas, orc, variant, k, m):
    """Draft and verify attention over caches with k, m off the 64 / 3 path."""
    H, Hq, n, T = 8, 32, 523, 5
    K, V = make_tokens(n, H, layer=3, seed=91)
    kv = new_cache(cas, H, 600, K, V, k, m, variant=variant)
    kv.append(K.cuda(), V.cuda())
    assert kv.status() == (n, 0)
    q = synthetic.activations(1, Hq * D, seed=92).view(1, Hq, D)
    o = cas.draft_attn_decode([kv], q.cuda())
    ref, nrm = orc.attention(np16(q), oracle_draft_kv(orc, K, k, m, variant), oracle_draft_kv(orc, V, k, m, variant))
    check_attn(o, ref, nrm, f"draft attention k={k} m={m} v={variant}")
    qv = synthetic.activations(T, Hq * D, seed=93).view(1, T, Hq, D)
    ov = cas.verify_attn([kv], qv.cuda())
    ref, nrm = orc.attention(np16(qv[0]), np16(K), np16(V), causal_new=T)
    check_attn(ov[0], ref, nrm, f"verify attention k={k} m={m} v={variant}")


def test_attention_errors(cas):
    H = 8
    K, V = make_tokens(16, H, seed=1)
    kv = new_cache(cas, H, 64, K, V)
    q = torch.zeros(1, 30, D, dtype=torch.int16, device="cuda")  # 30 q heads not a multiple of 8
    with pytest.raises(cas.CasError):
        cas.draft_attn_decode([kv], q)
    q = torch.zeros(1, 17, 32, D, dtype=torch.int16, device="cuda")  # T > 16
    with pytest.raises(cas.CasError):
        cas.verify_attn([kv], q)


# Caches sized for 20000 tokens hold ceil(20000 / 256) = 79 token chunks; with
# 2 kv heads and one sequence every resident-CTA budget keeps at least 76 of
# them, so each of the combine kernel's 32 warps merges two or more chunks
# (the rescale of its running maximum is exercised). Live lengths leave many
# chunks empty.
MULTI_CHUNK_CAP = 20000


def _long_cache(cas, H, n, variant, seed):
    K, V = make_tokens(n, H, layer=4, seed=seed)
    kv = new_cache(cas, H, MULTI_CHUNK_CAP, K, V, variant=variant)
    for t0 in range(0, n, 2048):
        kv.append(K[t0:t0 + 2048].cuda(), V[t0:t0 + 2048].cuda())
    assert kv.status() == (n, 0)
    return kv, K, V


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("Hq,n,n_tail", [(8, 4000, 3), (16, 1600, 0), (8, 9000, 1)])
def test_draft_attention_multi_chunk_combine(cas, orc, variant, Hq, n, n_tail):
    H = 2
    kv, K, V = _long_cache(cas, H, n, variant, seed=200 + n)
    q = synthetic.activations(1, Hq * D, seed=201).view(1, Hq, D)
    tk = synthetic.activations(max(n_tail, 1), H * D, seed=202).view(1, max(n_tail, 1), H, D)[:, :n_tail]
    tv = synthetic.activations(max(n_tail, 1), H * D, seed=203).view(1, max(n_tail, 1), H, D)[:, :n_tail]
    o = cas.draft_attn_decode([kv], q.cuda(), tk.contiguous().cuda() if n_tail else None,
                              tv.contiguous().cuda() if n_tail else None)
    Kall = np.concatenate([oracle_draft_kv(orc, K, 64, 3, variant), np16(tk[0])], 0)
    Vall = np.concatenate([oracle_draft_kv(orc, V, 64, 3, variant), np16(tv[0])], 0)
    ref, nrm = orc.attention(np16(q), Kall, Vall)
    check_attn(o, ref, nrm, f"draft attention, {n} tokens in a {MULTI_CHUNK_CAP}-token cache, v={variant}")


@pytest.mark.parametrize("variant", [1, 2])
def test_draft_attention_tail_holds_the_maximum(cas, orc, variant):
    """The bf16 draft tail scores far above every cached token, so the running
    maximum comes from the tail and every chunk partial is rescaled by it."""
    H, Hq, n = 2, 8, 3000
    kv, K, V = _long_cache(cas, H, n, variant, seed=300)
    q = synthetic.activations(1, Hq * D, seed=301).view(1, Hq, D)
    qf = q.view(torch.int16).to(torch.int32).__lshift__(16).view(torch.float32)  # bf16 -> fp32
    G = Hq // H
    tail = torch.stack([qf[0, h * G:(h + 1) * G].sum(0) for h in range(H)])  # [H][D]
    tk = synthetic.to_bits((2.0 * tail)[None, None])                       # [1][1][H][D]
    tv = synthetic.activations(H, D, seed=302).view(1, 1, H, D)
    o = cas.draft_attn_decode([kv], q.cuda(), tk.contiguous().cuda(), tv.contiguous().cuda())
    Kall = np.concatenate([oracle_draft_kv(orc, K, 64, 3, variant), np16(tk[0])], 0)
    Vall = np.concatenate([oracle_draft_kv(orc, V, 64, 3, variant), np16(tv[0])], 0)
    ref, nrm = orc.attention(np16(q), Kall, Vall)
    s_tail = (np.asarray(orc.bf16_to_f64(np16(q)))[0].reshape(H, G, D) *
              np.asarray(orc.bf16_to_f64(np16(tk)))[0, 0][:, None, :]).sum(-1)
    s_cache = np.einsum("thd,hgd->thg", orc.bf16_to_f64(Kall[:-1]), orc.bf16_to_f64(np16(q))[0].reshape(H, G, D))
    assert (s_tail > s_cache.max(0)).all()  # the tail really holds the maximum
    check_attn(o, ref, nrm, f"draft attention with a dominant tail, v={variant}")


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("n,T", [(5000, 5), (2100, 14)])
def test_verify_attention_multi_chunk_combine(cas, orc, variant, n, T):
    H, Hq = 2, 8
    kv, K, V = _long_cache(cas, H, n, variant, seed=400 + n)
    q = synthetic.activations(T, Hq * D, seed=401).view(1, T, Hq, D)
    o = cas.verify_attn([kv], q.cuda())
    ref, nrm = orc.attention(np16(q[0]), np16(K), np16(V), causal_new=T)
    check_attn(o[0], ref, nrm, f"verify attention, {n} tokens in a {MULTI_CHUNK_CAP}-token cache, v={variant}")


def _wild_tokens(n, H, seed):
    """Tokens the calibrated tables rank badly: in a third of them 6 dims hold
    values of 2^-20 .. 2^7 (exponents unseen in calibration, so codes of rank
    31 and more, longer than a window), a third whose large values fill dims
    32 .. 95 only (kept positions start after a gap of 32, pruned ones have a
    gap of 64), the rest ordinary."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, H, D))
    kind = np.arange(n) % 3
    spread = rng.choice([-1.0, 1.0], size=(n, H, D)) * 2.0 ** rng.uniform(-20, 7, size=(n, H, D))
    pick = np.zeros((n, H, D), dtype=bool)
    for t in range(n):
        for h in range(H):
            pick[t, h, rng.choice(D, 6, replace=False)] = True
    x = np.where((kind == 0)[:, None, None] & pick, spread, x)
    band = np.zeros(D, dtype=bool)
    band[32:96] = True
    sign = rng.choice([-1.0, 1.0], size=(n, H, D))
    banded = sign * np.where(band, rng.uniform(1.0, 2.0, size=(n, H, D)), rng.uniform(0.125, 0.25, size=(n, H, D)))
    x = np.where((kind == 1)[:, None, None], banded, x)
    return synthetic.to_bits(torch.from_numpy(x.astype(np.float32)))


def test_attention_long_codes_and_gaps(cas, orc):
    """Draft and verify attention over a cache whose tokens defeat the 64-bit
    windows of the block walk (codes longer than a window, gaps of 32 or more
    positions), so the per-group scans and the whole-token rescans run."""
    H, Hq, n, T = 2, 8, 700, 5
    K0, V0 = make_tokens(16, H, seed=500)
    K = torch.cat([K0, _wild_tokens(n - 16, H, seed=501)])
    V = torch.cat([V0, _wild_tokens(n - 16, H, seed=502)])
    kv = new_cache(cas, H, n + 64, K, V, est=16.0)  # long codes: room for ~16 bits per code
    kv.append(K[:n - T].cuda(), V[:n - T].cuda())
    assert kv.status() == (n - T, 0)
    q = synthetic.activations(1, Hq * D, seed=503).view(1, Hq, D)
    tk = synthetic.activations(2, H * D, seed=504).view(1, 2, H, D)
    tv = synthetic.activations(2, H * D, seed=505).view(1, 2, H, D)
    o = cas.draft_attn_decode([kv], q.cuda(), tk.cuda(), tv.cuda())
    Kall = np.concatenate([oracle_draft_kv(orc, K[:n - T], 64, 3, 1), np16(tk[0])], 0)
    Vall = np.concatenate([oracle_draft_kv(orc, V[:n - T], 64, 3, 1), np16(tv[0])], 0)
    ref, nrm = orc.attention(np16(q), Kall, Vall)
    check_attn(o, ref, nrm, "draft attention, long codes and gaps")
    kv.append(K[n - T:].cuda(), V[n - T:].cuda())
    qv = synthetic.activations(T, Hq * D, seed=506).view(1, T, Hq, D)
    ov = cas.verify_attn([kv], qv.cuda())
    ref, nrm = orc.attention(np16(qv[0]), np16(K), np16(V), causal_new=T)
    check_attn(ov[0], ref, nrm, "verify attention, long codes and gaps")


@pytest.mark.parametrize("cut", [0, 9, 30])
def test_truncate_many_equals_truncate(cas, cut):
    """cas_kv_truncate_many over caches of both variants and of 1, 2 and 4
    heads (one launch per variant, idle warps for the smaller caches) leaves
    every stream section and the state exactly as cas_kv_truncate does, and
    appends after it continue the same way."""
    T = 40
    specs = [(2, 1), (1, 2), (4, 1), (2, 2), (1, 1)]  # (heads, variant)
    made = []
    for i, (H, var) in enumerate(specs):
        K, V = make_tokens(T, H, seed=100 + i)
        K2, V2 = make_tokens(8, H, seed=200 + i)
        a = new_cache(cas, H, 96, K, V, variant=var)
        b = new_cache(cas, H, 96, K, V, variant=var)
        a.append(K.cuda(), V.cuda())
        b.append(K.cuda(), V.cuda())
        made.append((H, a, b, K2, V2))
    for _, a, _, _, _ in made:
        a.truncate(cut)
    cas.kv_truncate_many([b for _, _, b, _, _ in made], cut)
    for H, a, b, K2, V2 in made:
        assert b.status() == (cut, 0)
        a.append(K2.cuda(), V2.cuda())
        b.append(K2.cuda(), V2.cuda())
        for s in range(2 * H):
            assert_streams_equal(stream_sections(a, s, cut + 8), stream_sections(b, s, cut + 8))
        assert torch.equal(state_bytes(a), state_bytes(b))
    cas.kv_truncate_many([], 0)  # nothing to do
