#!/usr/bin/env python
"""Benchmark of the Cassandra bit-split hot path on GB300.

One step = one self-speculative decode step of a Llama-3-8B-shaped model (32
layers, hidden 4096, FFN 14336, GQA 32q/8kv, head_dim 128, 128256-row LM head)
with random-init Student-t(4) bf16 weights split at keep 50% / 3 mantissa bits
(Cassandra-1), batch 1, draft length 4, and a compressed KV cache of 32K tokens
(bf16 K/V ~ N(0,1) x LogNormal(0,0.5) channel scales), run as a data-dependent
forward through the library's C ABI:
  4 draft forwards : embedding of the previous token; per layer draft GEMV
                     Wqkv of the RMSNorm of the residual (the norm runs in the
                     GEMV's x staging), RoPE into the bf16 draft tail, draft
                     attention over the speculation KV + tail, draft GEMV Wo
                     added into the residual, draft GEMV Wgate|up of its
                     RMSNorm, SiLU*mul, draft GEMV Wdown added into the
                     residual; final RMSNorm + draft LM head, argmax = the
                     next token;
  1 verify forward : the same over the exact weights for the 5 tokens (verify
                     GEMMs, online KV append of the 5 tokens, verify attention);
  then the caches are rolled back to the context (fixed schedule: acceptance
  has no meaning on random weights); the verify's last token starts the next
  step.

Headline value: draft decode+GEMV GB/s over the algorithmic bytes of the
speculation streams read (plus x read and y written), timed with CUDA events on
the launching stream around the draft-GEMV launches of the timed steps.
Also reported: verify GEMM GB/s, microseconds per decode step (the whole step
replayed as one CUDA graph), roofline of the draft GEMV against the measured
HBM copy bandwidth, the end-to-end number through the C ABI with host buffers,
a dense bf16 GEMV of the same shape next to the draft GEMV (the break-even of
reading fewer bytes), the other configurations of the workload table, and the
CPU oracle as a reported baseline.

--impl reference times the CPU oracle (the plain C restatement) on the host
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft decode+GEMV GB/s (% of HBM peak); verify GEMM GB/s; µs per decode step"
WORKLOADS = {"llama3-8b": "llama3-8b-stack speculative decode step",
             "qwen3-8b": "qwen3-8b full speculative decode step (with LM head)"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="cas", choices=["cas", "reference"])
    ap.add_argument("--workload", default="llama3-8b", choices=["llama3-8b", "qwen3-8b"])
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--ctx", type=int, default=None)
    ap.add_argument("--keep", type=int, default=64)
    ap.add_argument("--mant", type=int, default=3)
    ap.add_argument("--draft-len", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--capacity", action="store_true",
                    help="max context at a fixed HBM budget from measured encoded sizes")
    ap.add_argument("--sweep", action="store_true",
                    help="Cassandra-1 vs -2 over keep 20-60%% x mantissa 1-5 on the FFN matrices")
    ap.add_argument("--no-attn", action="store_true", help="weights only (no KV cache)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other configurations (keep 30%%, Qwen3-8B step, 128K attention)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--micro", default=None,
                    choices=["draft_gemv", "verify_gemm", "draft_attn", "verify_attn", "kv_append", "encode"],
                    help="time one kernel on one tensor (for profiling)")
    ap.add_argument("--N", type=int, default=28672)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--variant", type=int, default=1)
    ap.add_argument("--nvec", type=int, default=1)
    ap.add_argument("--T", type=int, default=5)
    ap.add_argument("--reps", type=int, default=20)
    a = ap.parse_args()
    # workload defaults: Llama-3-8B stack at batch 1, draft length 4, 32K
    # context; Qwen3-8B step at batch 2, draft length 6, 16K context
    dflt = {"llama3-8b": dict(layers=32, ctx=32768, draft_len=4, batch=1),
            "qwen3-8b": dict(layers=36, ctx=16384, draft_len=6, batch=2)}[a.workload]
    for key, val in dflt.items():
        if getattr(a, key) is None:
            setattr(a, key, val)
    return a


# ---------------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during timing."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:  # noqa: BLE001
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if len(r) > 8 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 8 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows if len(r) > 8 for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ---------------------------------------------------------------------- CPU oracle baseline
def cpu_baseline(seconds: float, keep: int, mant: int, variant: int = 1):
    """The oracle's draft decode + float64 GEMV (plain C) timed on the host
    cores on a bounded sample of the same workload: a 1024x4096 Student-t(4)
    matrix of the stack, split into one 1024/n-row slice per thread (each
    slice encoded as its own tensor), repeated for about `seconds` - half the
    time on one thread, half on every host core. value = speculation bytes
    decoded per second with all cores; the one-thread figure is reported too."""
    import concurrent.futures as cf

    import numpy as np

    import oracle
    import synthetic
    oracle.build()
    N, K = 1024, 4096
    W = synthetic.t4_weight(N, K, seed=0).numpy().view(np.uint16)
    x = synthetic.activations(1, K, seed=1).numpy().view(np.uint16)
    host = os.cpu_count() or 1

    def timed(nthreads, budget):
        rows = N // nthreads
        parts = [oracle.encode(np.ascontiguousarray(W[i * rows:(i + 1) * rows]), variant, keep, mant)
                 for i in range(nthreads)]
        spec = sum(p.spec_bytes() + K * 2 + rows * 4 for p in parts)

        def work(p):
            oracle.matvec(oracle.decode(p, False), x)

        reps, t0 = 0, time.perf_counter()
        with cf.ThreadPoolExecutor(nthreads) as ex:
            while True:
                list(ex.map(work, parts))
                reps += 1
                if time.perf_counter() - t0 >= budget:
                    break
        dt = time.perf_counter() - t0
        return spec * reps / dt / 1e9, reps, dt

    one, r1, t1 = timed(1, seconds / 2)
    nt = max(1, min(host, 64))
    while N % nt:
        nt -= 1
    allc, rn, tn = timed(nt, seconds / 2)
    return {"value": allc, "unit": "GB/s", "cores": nt, "host_cores": host, "kind": "oracle",
            "single_thread_value": one,
            "sample": f"oracle draft decode + float64 GEMV of one 1024x4096 t4 matrix (keep {keep}/128, m={mant}, "
                      f"Cassandra-{variant}): {r1} passes on 1 thread in {t1:.1f} s, {rn} passes with the rows "
                      f"split over {nt} threads in {tn:.1f} s"}


# ---------------------------------------------------------------------- workload
class Stack:
    """Encoded decoder stack of one model shape (Student-t(4) bf16 weights,
    Wq|Wk|Wv and Wgate|Wup fused), its RMSNorm weights, LM head, embedding
    table and compressed KV caches filled to `ctx` tokens per sequence."""

    def __init__(self, cas, dev, workload, layers, variant, keep, mant, ctx, batch, attn=True):
        import torch

        import synthetic
        self.cas, self.dev = cas, dev
        shp = dict(synthetic.LLAMA3_8B if workload == "llama3-8b" else synthetic.QWEN3_8B)
        self.L, self.ctx, self.B = layers, ctx, batch
        self.variant, self.keep, self.mant = variant, keep, mant
        h, f = shp["hidden"], shp["ffn"]
        self.hidden, self.ffn, self.nq, self.nkv, self.hd = h, f, shp["n_q"], shp["n_kv"], shp["head_dim"]
        self.vocab, self.theta = shp["vocab"], shp["rope_theta"]
        self.mats, self.g1, self.g2 = [], [], []
        t0 = time.time()
        for layer in range(self.L):
            raw = {nm: synthetic.t4_weight(N, K, seed=layer * 16 + idx, device=dev)
                   for idx, (nm, N, K) in enumerate(synthetic.layer_matrices(shp))}
            fused = {"qkv": torch.cat([raw["wq"], raw["wk"], raw["wv"]], 0), "o": raw["wo"],
                     "gateup": torch.cat([raw["wgate"], raw["wup"]], 0), "down": raw["wdown"]}
            del raw
            self.mats.append({nm: cas.encode_weights(W, variant, keep, mant) for nm, W in fused.items()})
            del fused
            self.g1.append(synthetic.norm_weight(h, seed=layer * 16 + 8, device=dev))
            self.g2.append(synthetic.norm_weight(h, seed=layer * 16 + 9, device=dev))
        self.gf = synthetic.norm_weight(h, seed=999_981, device=dev)
        Wl = synthetic.t4_weight(self.vocab, h, seed=999_983, device=dev)
        self.lm = cas.encode_weights(Wl, variant, keep, mant)
        del Wl
        self.emb = synthetic.normal_weight(self.vocab, h, seed=999_979, device=dev)
        torch.cuda.synchronize()
        self.encode_s = time.time() - t0
        self.kv = self._fill_kv() if attn else None

    def _fill_kv(self):
        import torch

        import synthetic
        cas, dev, T = self.cas, self.dev, self.ctx
        p = cas.params(self.variant, self.keep, self.mant)
        kvs = []
        for layer in range(self.L):
            layer_kv = []
            for b in range(self.B):
                sk = synthetic.kv_scales(layer, self.nkv, 0, device=dev)
                sv = synthetic.kv_scales(layer, self.nkv, 1, device=dev)
                Kc = synthetic.kv_tokens(T, self.nkv, seed=100 * layer + 2 * b, scales=sk, device=dev)
                Vc = synthetic.kv_tokens(T, self.nkv, seed=100 * layer + 2 * b + 1, scales=sv, device=dev)
                kv = cas.KVCache(self.nkv, T + 64, p, Kc[:128], Vc[:128])
                for t0 in range(0, T, 2048):
                    kv.append(Kc[t0:t0 + 2048], Vc[t0:t0 + 2048])
                layer_kv.append(kv)
                del Kc, Vc
            kvs.append(layer_kv)
        torch.cuda.synchronize()
        for layer_kv in kvs:
            for kv in layer_kv:
                n, s = kv.status()
                assert s == 0 and n == T, (n, s)
        return kvs


# kernels of ours each call launches (the y / Y clear of the matrix products
# is a memset node, not a kernel)
KERNELS_PER_CALL = {"gemv": 1, "gemm": 2, "gemm_acc": 1, "draft_attn": 2, "verify_attn": 2, "append": 2, "truncate": 1, "glue": 1}


class Step:
    """One self-speculative decode step as a data-dependent forward through
    the C ABI: D draft tokens, each a forward of every layer over the
    speculation data (embedding, draft GEMV Wqkv of the RMSNorm of the
    residual, RoPE into a bf16 draft tail, draft attention over the compressed
    KV + tail, Wo of its bf16-rounded output added into the residual, Wgate|up
    of the RMSNorm (the rounding and the norm inside the GEMV's staging of x),
    SiLU*mul, Wdown added into the residual, ..., final RMSNorm, LM head, argmax
    -> next draft token), then one verify forward of the T = D + 1 tokens over
    the exact weights (verify GEMMs, online KV append, verify attention, LM
    head, argmax), then a rollback of the KV caches to the context (fixed
    schedule: acceptance has no meaning on random weights). The verify's last
    token is the next step's first token, so successive steps chain."""

    def __init__(self, cas, stk, st, D):
        import torch
        self.cas, self.stk, self.st, self.D = cas, stk, st, D
        B, T, dev = stk.B, D + 1, stk.dev
        self.T = T
        h, F, Hq, Hkv, hd, V = stk.hidden, stk.ffn, stk.nq, stk.nkv, stk.hd, stk.vocab
        f32, i16 = torch.float32, torch.int16
        E = lambda *s, dt=f32: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        self.vtok = torch.zeros(B * T, dtype=torch.int32, device=dev)  # per sequence: [t_last, d_1 .. d_D]
        x, xn, qkv, q = E(B, h), E(B, h, dt=i16), E(B, (Hq + 2 * Hkv) * hd), E(B, Hq, hd, dt=i16)
        tk, tv, o, ob = E(B, D, Hkv, hd, dt=i16), E(B, D, Hkv, hd, dt=i16), E(B, Hq, hd), E(B, Hq * hd, dt=i16)
        gu, hh, lg = E(B, 2 * F), E(B, F, dt=i16), E(B, V)
        tk.zero_()
        tv.zero_()
        X, Xn, QKV = E(B * T, h), E(B * T, h, dt=i16), E(B * T, (Hq + 2 * Hkv) * hd)
        Q, Kn, Vn = E(B * T, Hq, hd, dt=i16), E(B * T, Hkv, hd, dt=i16), E(B * T, Hkv, hd, dt=i16)
        O, Ob = E(B, T, Hq, hd), E(B * T, Hq * hd, dt=i16)
        GU, HH, LG = E(B * T, 2 * F), E(B * T, F, dt=i16), E(B * T, V)
        self.vout = torch.zeros(B * T, dtype=torch.int32, device=dev)
        attn = stk.kv is not None
        ws = E(cas.cas_attn_workspace_bytes(B, Hq, T, stk.ctx + 64), dt=torch.uint8) if attn else None
        self.keep = [x, xn, qkv, q, tk, tv, o, ob, gu, hh, lg, X, Xn, QKV, Q, Kn, Vn, O, Ob, GU, HH,
                     LG, ws]
        P, eps = cas.prepare, 1e-5
        segs, self.kernels = [], {"gemv": 0, "gemm": 0, "other": 0}
        self.draft_bytes, self.verify_bytes = 0, 0

        def add(kind, fns, what):
            segs.append((kind, fns))
            self.kernels["other" if kind == "other" else kind] += sum(KERNELS_PER_CALL[w] for w in what)

        def gemv_norm(W, xres, gamma, xout, y):
            # y = D(W) bf16(rmsnorm(xres) * gamma): the norm runs in the GEMV's x staging
            self.draft_bytes += W.spec_bytes() + B * W.K * 4 + W.K * 2 + B * W.K * 2 + B * W.N * 4
            add("gemv", [P("cas_draft_gemv_rmsnorm", W, xres, B, gamma, eps, xout, y, st)], ["gemv"])

        def gemv_acc(W, xin, y):
            # y += D(W) xin: the residual add happens in the GEMV's row writes
            self.draft_bytes += W.spec_bytes() + B * W.K * 2 + B * W.N * 8
            add("gemv", [P("cas_draft_gemv_accumulate", W, xin, B, y, st)], ["gemv"])

        def gemv_f32(W, src, op, width, xout, y):
            # y += D(W) bf16(op(src)): rounding or SiLU*mul of the fp32 input in the GEMV's x staging
            self.draft_bytes += W.spec_bytes() + B * width * 4 + B * W.K * 2 + B * W.N * 8
            add("gemv", [P("cas_draft_gemv_f32", W, src, B, op, None, 0.0, xout, y, 1, st)], ["gemv"])

        def gemm(W, Xin, Y):
            self.verify_bytes += W.all_bytes() + B * T * W.K * 2 + B * T * W.N * 4
            add("gemm", [P("cas_verify_gemm", W, Xin, B * T, Y, st)], ["gemm"])

        def gemm_acc(W, Xin, Y):
            # Y += W Xin: the residual add happens in the GEMM's atomics
            self.verify_bytes += W.all_bytes() + B * T * W.K * 2 + B * T * W.N * 8
            add("gemm", [P("cas_verify_gemm_accumulate", W, Xin, B * T, Y, st)], ["gemm_acc"])

        for d in range(D):
            add("other", [P("cas_embed", self.vtok[b * T + d:b * T + d + 1], 1, stk.emb, V, h, x[b:b + 1], st)
                          for b in range(B)], ["glue"] * B)
            for layer in range(stk.L):
                M = stk.mats[layer]
                gemv_norm(M["qkv"], x, stk.g1[layer], xn, qkv)
                fns = [P("cas_rope_split", qkv, B, Hq, Hkv, stk.ctx + d, 1, stk.theta, q, tk[0, d], D * Hkv * hd,
                         tv[0, d], D * Hkv * hd, st)]
                what = ["glue"]
                if attn:
                    for b in range(B):
                        fns.append(cas.prepare_draft_attn([stk.kv[layer][b]], q[b:b + 1], tk[b:b + 1, :d + 1],
                                                          tv[b:b + 1, :d + 1], o[b:b + 1], ws, st))
                        what.append("draft_attn")
                add("other", fns, what)
                gemv_f32(M["o"], o, cas.X_ROUND, Hq * hd, ob, x)
                gemv_norm(M["gateup"], x, stk.g2[layer], xn, gu)
                # SiLU*mul stays a kernel of its own: formed in every CTA's staging it
                # reads the 2F fp32 gate|up row once per CTA, more than it saves
                add("other", [P("cas_silu_mul", gu, B, F, hh, st)], ["glue"])
                gemv_acc(M["down"], hh, x)
            gemv_norm(stk.lm, x, stk.gf, xn, lg)
            add("other", [P("cas_argmax", lg[b:b + 1], 1, V, self.vtok[b * T + 1 + d:b * T + 2 + d], st)
                          for b in range(B)], ["glue"] * B)
        # verify forward of the T tokens of every sequence
        add("other", [P("cas_embed", self.vtok, B * T, stk.emb, V, h, X, st)], ["glue"])
        for layer in range(stk.L):
            M = stk.mats[layer]
            add("other", [P("cas_add_rmsnorm", X, None, B * T, h, stk.g1[layer], eps, Xn, st)], ["glue"])
            gemm(M["qkv"], Xn, QKV)
            fns = [P("cas_rope_split", QKV, B * T, Hq, Hkv, stk.ctx, T, stk.theta, Q, Kn, Hkv * hd, Vn, Hkv * hd, st)]
            what = ["glue"]
            if attn:
                for b in range(B):
                    fns.append(stk.kv[layer][b].prepare_append(Kn[b * T:(b + 1) * T], Vn[b * T:(b + 1) * T], st))
                    what.append("append")
                fns.append(cas.prepare_verify_attn(stk.kv[layer], Q.view(B, T, Hq, hd), O, ws, st))
                what.append("verify_attn")
            fns.append(P("cas_f32_to_bf16", O, B * T * Hq * hd, Ob, st))
            what.append("glue")
            add("other", fns, what)
            gemm_acc(M["o"], Ob, X)
            add("other", [P("cas_add_rmsnorm", X, None, B * T, h, stk.g2[layer], eps, Xn, st)], ["glue"])
            gemm(M["gateup"], Xn, GU)
            add("other", [P("cas_silu_mul", GU, B * T, F, HH, st)], ["glue"])
            gemm_acc(M["down"], HH, X)
        add("other", [P("cas_add_rmsnorm", X, None, B * T, h, stk.gf, eps, Xn, st)], ["glue"])
        gemm(stk.lm, Xn, LG)
        fns = [P("cas_argmax", LG, B * T, V, self.vout, st)]
        fns += [P("cas_argmax", LG[b * T + T - 1:b * T + T], 1, V, self.vtok[b * T:b * T + 1], st) for b in range(B)]
        what = ["glue"] * (1 + B)
        if attn:  # rollback: every cache back to the context, one launch for all of them
            fns.append(cas.prepare_truncate_many([kv for layer_kv in stk.kv for kv in layer_kv], stk.ctx, st))
            what.append("truncate")
        add("other", fns, what)
        self.segs = segs
        self.launches = sum(self.kernels.values())

    def eager(self):
        for _, fns in self.segs:
            for f in fns:
                f()

    def eager_overlapped(self):
        """The step call by call with launch overlap: the first segment (the
        embedding) follows the caller's copy of the first token and is
        launched plainly; every later call follows a libcas kernel."""
        self.segs_run(self.segs[:1])
        self.cas.set_launch_overlap(True)
        try:
            self.segs_run(self.segs[1:])
        finally:
            self.cas.set_launch_overlap(False)

    @staticmethod
    def segs_run(segs):
        for _, fns in segs:
            for f in fns:
                f()

    def capture(self):
        """The whole step as one CUDA graph (how it runs), and one graph per
        segment (so the matrix products can be timed on their own), captured
        with launch overlap on: the step holds only libcas calls, so each
        kernel may launch while the one before it drains."""
        import torch
        self.cas.set_launch_overlap(True)
        try:
            self.full = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.full, stream=self.st):
                for _, fns in self.segs:
                    for f in fns:
                        f()
            self.graphs = []
            for kind, fns in self.segs:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.st):
                    for f in fns:
                        f()
                self.graphs.append((kind, g))
        finally:
            self.cas.set_launch_overlap(False)

    def replay(self, ev=None):
        """One step from the graphs; with `ev`, events around every matrix-product segment."""
        e = 0
        for kind, g in self.graphs:
            if ev is not None and kind != "other":
                ev[e].record(self.st)
                g.replay()
                ev[e + 1].record(self.st)
                e += 2
            else:
                g.replay()


def time_step(step, steps, warmup, clocks=None):
    """Steps timed with CUDA events on the step's stream: the whole-step graph
    replayed `steps` times (total ms), then the per-segment graphs replayed
    `steps` times with events around every matrix-product segment (draft GEMV
    ms, verify GEMM ms per step). Returns (total ms, draft GEMV ms, verify GEMM
    ms) over `steps` steps."""
    import torch
    st = step.st
    with torch.cuda.stream(st):
        for _ in range(max(warmup, 3)):
            step.eager()
    torch.cuda.synchronize()
    step.capture()
    torch.cuda.synchronize()
    kinds = [k for k, _ in step.graphs if k != "other"]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(kinds))] for _ in range(steps)]
    with torch.cuda.stream(st):
        for _ in range(max(warmup, 3)):
            step.full.replay()
        for _ in range(2):
            step.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx = clocks if clocks is not None else _Null()
    with ctx, torch.cuda.stream(st):
        torch.cuda.nvtx.range_push("timed")  # lets a profiler select the timed launches
        a.record(st)
        for i in range(steps):
            step.full.replay()
        b.record(st)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        for i in range(steps):
            step.replay(evs[i])
        torch.cuda.synchronize()
    gemv_ms = gemm_ms = 0.0
    for ev in evs:
        for i, kind in enumerate(kinds):
            ms = ev[2 * i].elapsed_time(ev[2 * i + 1])
            if kind == "gemv":
                gemv_ms += ms
            else:
                gemm_ms += ms
    return a.elapsed_time(b), gemv_ms, gemm_ms


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def e2e_step(step, steps):
    """The whole step through the C ABI, launched call by call as a user would
    (no graphs, launch overlap after the first call), with each step's first
    token copied in from pinned host memory and its verified tokens copied back
    and read on the host."""
    import torch
    st, B, T = step.st, step.stk.B, step.T
    host_in = step.vtok.view(B, T)[:, 0].cpu().pin_memory()
    host_out = torch.empty(B * T, dtype=torch.int32).pin_memory()
    first = [step.vtok[b * T:b * T + 1] for b in range(B)]

    def one():
        for b in range(B):
            first[b].copy_(host_in[b:b + 1], non_blocking=True)
        step.eager_overlapped()
        host_out.copy_(step.vout, non_blocking=True)
        st.synchronize()
        host_in.copy_(host_out.view(B, T)[:, -1])

    with torch.cuda.stream(st):
        for _ in range(2):
            one()
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
        dt = (time.perf_counter() - t0) / steps
    return dt * 1e3, B * 4, B * T * 4


def run_cas(args):
    import torch
    import torch.distributed as dist

    import bit_level_weight_gb300 as cas

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from bit_level_weight_gb300 import build as _b
    _b.build()

    stk = Stack(cas, dev, args.workload, args.layers, args.variant, args.keep, args.mant, args.ctx, args.batch,
                attn=not args.no_attn)
    st = torch.cuda.Stream(device=dev)  # every call of the step is bound to this stream
    step = Step(cas, stk, st, args.draft_len)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        total_ms, gemv_ms, gemm_ms = time_step(step, args.steps, args.warmup)
    if world > 1:
        dist.barrier()
    steps, D = args.steps, args.draft_len
    d_bytes = step.draft_bytes * steps
    v_bytes = step.verify_bytes * steps
    gemv_gbs = d_bytes / (gemv_ms * 1e-3) / 1e9
    gemm_gbs = v_bytes / (gemm_ms * 1e-3) / 1e9
    ms_per_step = total_ms / steps
    e2e_ms, h2d, d2h = e2e_step(step, max(3, steps // 2))
    status = cas.cas_device_status(st)
    assert status == 0, f"device status {status}"

    if world > 1:
        agg = replica_aggregate(gather_stats((d_bytes, gemv_ms, v_bytes, gemm_ms, ms_per_step, e2e_ms), world))
        gemv_gbs, gemm_gbs, ms_per_step, e2e_ms = agg["gemv_gbs"], agg["gemm_gbs"], agg["ms_per_step"], agg["e2e_ms"]
    launches = step.launches
    ctx_used = args.ctx if stk.kv is not None else 0
    extra = {}
    if rank == 0 and not args.no_extra and world == 1:
        del step
        extra = extra_configs(cas, args, dev, stk)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = peaks()
    n_gemv = 4 * stk.L + 1  # per draft token
    per_launch_bytes = step_draft_bytes = d_bytes / steps
    per_launch_bytes = step_draft_bytes / (D * n_gemv)
    per_launch_ms = gemv_ms / (steps * D * n_gemv)
    achieved = per_launch_bytes / (per_launch_ms * 1e-3) / 1e9
    kern = gemv_kernel_name(args, args.batch)
    rec = profiled_record(kern)
    out = {
        "metric": METRIC,
        "value": round(gemv_gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": WORKLOADS[args.workload],
            "layers": stk.L, "lm_head_rows": stk.vocab, "hidden": stk.hidden, "ffn": stk.ffn,
            "heads": f"{stk.nq}q/{stk.nkv}kv x {stk.hd}", "batch": args.batch, "draft_len": D,
            "verify_tokens": args.batch * (D + 1), "ctx": ctx_used,
            "keep_per_block": args.keep, "mant_bits": args.mant, "variant": f"Cassandra-{args.variant}",
            "weights": "Student-t(4) x 0.02/sqrt(2), fused qkv and gate|up; embedding N(0, 0.02)",
            "forward": "data-dependent: embedding, RMSNorm, RoPE, SiLU*mul, residual adds, LM head, argmax chain",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": f"inputs larger than L2 ({step_draft_bytes / D / 1e9:.2f} GB speculation stream per draft pass)",
        },
        "verify_gemm_gbs": round(gemm_gbs, 1),
        "us_per_decode_step": round(ms_per_step * 1e3, 1),
        "draft_gemv_frac_of_hbm": round(gemv_gbs / world / peak, 4),
        "draft_gemv_frac_of_8tbs_nominal": round(gemv_gbs / world / 8000.0, 4),
        "verify_gemm_frac_of_hbm": round(gemm_gbs / world / peak, 4),
        "draft_gemv_ms_per_step": round(gemv_ms / steps, 3),
        "verify_gemm_ms_per_step": round(gemm_ms / steps, 3),
        "roofline": {"kernel": kern, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                     "traffic": (round(rec["traffic_ratio"] * per_launch_bytes) if rec else None),
                     "traffic_note": ("per launch: ncu dram bytes / algorithmic bytes of one profiled launch of "
                                      f"this kernel ({rec['shape']}) x algorithmic bytes per launch of this step"
                                      if rec else "null: the kernel's source changed since its counters were taken"),
                     "algorithmic_bytes_per_launch": int(per_launch_bytes)},
        "alu_roof": (alu_roof(achieved, clk, rec) if args.variant == 1 and args.keep == 64 and args.mant == 3
                     and args.batch <= 2 else None),
        "e2e": {"value": round(step_draft_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "us_per_step": round(e2e_ms * 1e3, 1),
                "what": "the whole step (draft forwards, verify forward, KV append and rollback) called entry point "
                        "by entry point through the C ABI without graphs (launch overlap on after the first call), the "
                        "first token copied in from pinned host memory and the verified tokens copied out and read "
                        "each step; value = the step's "
                        "speculation bytes over its end-to-end time"},
        "gpu_launches": launches * steps,
        "encode_s": round(stk.encode_s, 2),
    }
    out.update(extra)
    out["clocks"] = clk.summary()
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds, args.keep, args.mant, args.variant)
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def extra_configs(cas, args, dev, main_stk):
    """The other configurations of the workload table, each timed on this
    GPU after the main line: the 30%-keep stack (k = 38), the Qwen3-8B-shaped
    full step (36 layers + 151936-row LM head, batch 2, 16K, draft 6) and the
    attention of a 128K-token cache (batch 1 and 2)."""
    import gc

    import torch
    out = {}
    if args.workload == "llama3-8b" and args.variant == 1:
        out["dense_bf16_gemv"] = dense_vs_draft(cas, dev, main_stk)
    for kv in (main_stk.kv or []):
        del kv
    main_stk.kv = None
    gc.collect()
    torch.cuda.empty_cache()

    def step_ms(workload, layers, keep, ctx, batch, D):
        stk = Stack(cas, dev, workload, layers, args.variant, keep, args.mant, ctx, batch)
        st = torch.cuda.Stream(device=dev)
        s = Step(cas, stk, st, D)
        total, gv, gm = time_step(s, 3, 3)
        r = {"ms_per_step": round(total / 3, 3), "draft_gemv_gbs": round(s.draft_bytes * 3 / (gv * 1e-3) / 1e9, 1),
             "verify_gemm_gbs": round(s.verify_bytes * 3 / (gm * 1e-3) / 1e9, 1)}
        del s, stk
        gc.collect()
        torch.cuda.empty_cache()
        return r

    if args.workload == "llama3-8b":
        out["keep30"] = dict(step_ms("llama3-8b", 32, cas.cas_keep_from_ratio(0.3), 32768, 1, 4),
                             config="llama3-8b stack, keep 38/128, m = 3, batch 1, draft 4, 32K")
        out["qwen3_step"] = dict(step_ms("qwen3-8b", 36, args.keep, 16384, 2, 6),
                                 config="qwen3-8b full step, 36 layers + 151936-row LM head, batch 2, 16K, draft 6")
        out["keep30_step_ms"] = out["keep30"]["ms_per_step"]
        out["qwen3_step_ms"] = out["qwen3_step"]["ms_per_step"]
    out.update(attn_128k(cas, args, dev))
    return out


def dense_vs_draft(cas, dev, stk):
    """The break-even of the draft: a dense bf16 GEMV (cuBLAS through
    torch.mv) of the fused gate|up shape, 28672 x 4096, against the draft
    decode + GEMV of the same shape from the stack's encoded matrices. Both
    rotate over matrices that together exceed L2 (2 dense, 8 encoded); CUDA
    events, 24 calls each after 6 warm-up calls."""
    import torch

    import synthetic
    mats = [stk.mats[i]["gateup"] for i in range(min(8, len(stk.mats)))]
    N, K = mats[0].N, mats[0].K
    st = torch.cuda.Stream(device=dev)
    x = synthetic.activations(1, K, seed=71, device=dev)
    y = torch.empty(1, N, dtype=torch.float32, device=dev)
    draft = [cas.prepare("cas_draft_gemv", m, x, 1, y, st) for m in mats]
    gen = torch.Generator(device=dev).manual_seed(72)
    dense = [(torch.randn(N, K, device=dev, generator=gen) * 0.02).to(torch.bfloat16) for _ in range(2)]
    xd = x.view(torch.bfloat16).view(K)

    def timed(calls):
        with torch.cuda.stream(st):
            for i in range(6):
                calls[i % len(calls)]()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            for i in range(24):
                calls[i % len(calls)]()
            b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / 24

    dense_us = timed([lambda W=W: torch.mv(W, xd) for W in dense])
    draft_us = timed(draft)
    spec = sum(m.spec_bytes() for m in mats) / len(mats)
    del dense
    torch.cuda.empty_cache()
    return {"shape": f"{N} x {K}", "dense_us": round(dense_us, 2),
            "dense_gbs": round(N * K * 2 / (dense_us * 1e-6) / 1e9, 1), "draft_us": round(draft_us, 2),
            "draft_gbs": round((spec + K * 2 + N * 4) / (draft_us * 1e-6) / 1e9, 1),
            "draft_speedup_over_dense": round(dense_us / draft_us, 3)}


def attn_128k(cas, args, dev):
    """Draft and verify attention of one layer over 128K-token compressed
    caches (8 kv heads, 32 query heads), batch 1 and 2: CUDA-event time of 10
    calls each; the 32-layer figure is 32 x this."""
    import torch

    import synthetic
    H, Hq, T, n = 8, 32, 5, 131072
    p = cas.params(args.variant, args.keep, args.mant)
    res = {}
    caches = []
    for b in range(2):
        sk, sv = synthetic.kv_scales(0, H, 0, device=dev), synthetic.kv_scales(0, H, 1, device=dev)
        kv = cas.KVCache(H, n + 64, p, synthetic.kv_tokens(128, H, seed=7 + b, scales=sk, device=dev),
                         synthetic.kv_tokens(128, H, seed=9 + b, scales=sv, device=dev))
        for t0 in range(0, n, 4096):
            Kc = synthetic.kv_tokens(4096, H, seed=1000 + 2 * t0 + b, scales=sk, device=dev)
            Vc = synthetic.kv_tokens(4096, H, seed=1001 + 2 * t0 + b, scales=sv, device=dev)
            kv.append(Kc, Vc)
        caches.append(kv)
    st = torch.cuda.Stream(device=dev)
    for B in (1, 2):
        kvs = caches[:B]
        ws = torch.empty(cas.cas_attn_workspace_bytes(B, Hq, T, n + 64), dtype=torch.uint8, device=dev)
        q = synthetic.activations(B, Hq * 128, seed=3, device=dev).view(B, Hq, 128)
        tk = synthetic.activations(B * 4, H * 128, seed=4, device=dev).view(B, 4, H, 128)
        tv = synthetic.activations(B * 4, H * 128, seed=5, device=dev).view(B, 4, H, 128)
        o = torch.empty(B, Hq, 128, dtype=torch.float32, device=dev)
        d = cas.prepare_draft_attn(kvs, q, tk, tv, o, ws, st)
        for kv in kvs:
            kv.truncate(n - T)
        newk = synthetic.activations(T, H * 128, seed=6, device=dev).view(T, H, 128)
        newv = synthetic.activations(T, H * 128, seed=8, device=dev).view(T, H, 128)
        for kv in kvs:
            kv.append(newk, newv)
        qv = synthetic.activations(B * T, Hq * 128, seed=7, device=dev).view(B, T, Hq, 128)
        ov = torch.empty(B, T, Hq, 128, dtype=torch.float32, device=dev)
        v = cas.prepare_verify_attn(kvs, qv, ov, ws, st)
        for name, f in (("draft", d), ("verify", v)):
            with torch.cuda.stream(st):
                for _ in range(3):
                    f()
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(st)
                for _ in range(10):
                    f()
                b_.record(st)
                torch.cuda.synchronize()
            res[f"{name}_attn_128k_b{B}_us"] = round(a.elapsed_time(b_) / 10 * 1e3, 1)
    res["draft_attn_128k_us"] = res["draft_attn_128k_b1_us"]
    res["verify_attn_128k_us"] = res["verify_attn_128k_b1_us"]
    res["attn_128k_note"] = "one layer (8 kv heads, 32 query heads) over a 131072-token cache; x 32 for a stack"
    return res


# ncu counters of one profiled launch of each draft GEMV kernel, stored with a
# hash of the sources the kernel is built from; a record whose hash no longer
# matches the tree is not used (the kernel changed since it was profiled).
PROFILED = {
    # ncu --set full on the 28672 x 4096 Student-t(4) matrix, one vector
    # (bench.py --micro draft_gemv --N 28672): dram read + write 61.809 + 0.129 MB
    # for 61.853 MB algorithmic, 46525966 warp instructions
    "draft_gemv_block_kernel<1>": {"source_sha16": "c53408e41b703cc8", "shape": "28672 x 4096, keep 64, m = 3",
                                   "traffic_ratio": (61.80864 + 0.129024) / 61.85268,
                                   "lane_instr_per_elem": 46525966 * 32 / (28672 * 4096),
                                   "spec_bits_per_elem": 4.205},
}
PROFILED_SOURCES = ("bit_level_weight_gb300/csrc/gemv.cu", "bit_level_weight_gb300/csrc/blockwalk.cuh",
                    "bit_level_weight_gb300/csrc/wordlane.cuh", "bit_level_weight_gb300/csrc/common.cuh",
                    "bit_level_weight_gb300/csrc/sbdecode.cuh")
SMS, LANES_PER_SM_CLK = 152, 128  # 4 schedulers x 32 lanes issue per SM clock


def source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in PROFILED_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_record(kernel: str):
    rec = PROFILED.get(kernel)
    return rec if rec and rec["source_sha16"] == source_hash() else None


def gemv_kernel_name(args, nvec: int) -> str:
    """The draft GEMV kernel the stack's matrices (rows of whole superblocks) run."""
    if args.keep == 64 and args.mant == 3:
        if args.variant == 1:
            return f"draft_gemv_block_kernel<{nvec}>" if nvec <= 2 else f"draft_gemv_fast_kernel<{nvec}>"
        if nvec <= 2:
            return f"draft_gemv_fast2_kernel<{nvec}>"
    return f"draft_gemv_runs_kernel<{args.variant},{nvec}>"


def alu_roof(achieved_gbs: float, clk, rec) -> dict:
    """The draft GEMV is bound by instruction issue (integer decode), so its
    second roof is the lane-instruction issue peak: SMs x 128 x SM clock.
    achieved = profiled lane instructions per element x elements per second."""
    if not rec:
        return None
    mhz = (clk.summary() or {}).get("sm_mhz") or 2070.0
    peak = SMS * LANES_PER_SM_CLK * mhz * 1e6
    bytes_per_elem = rec["spec_bits_per_elem"] / 8
    elems = achieved_gbs * 1e9 / bytes_per_elem
    achieved = rec["lane_instr_per_elem"] * elems
    budget = peak / (0.75 * peaks()[0] * 1e9 / bytes_per_elem)
    return {"bound": "alu", "achieved": round(achieved / 1e12, 2), "peak": round(peak / 1e12, 2),
            "unit": "T lane-instr/s", "frac": round(achieved / peak, 4),
            "lane_instr_per_elem": round(rec["lane_instr_per_elem"], 2),
            "budget_at_75pct_hbm": round(budget, 2),
            "note": f"lane instructions per element from ncu smsp__inst_executed.sum on {rec['shape']}; "
                    "peak = 152 SMs x 128 lanes x median SM clock"}


def gather_stats(local: tuple, world: int) -> list:
    """All ranks' (draft bytes, draft ms, verify bytes, verify ms, ms/step, e2e ms)."""
    import torch.distributed as dist
    out = [None] * world
    dist.all_gather_object(out, tuple(float(v) for v in local))
    return out


def replica_aggregate(stats: list) -> dict:
    """Whole-job numbers of N independent replicas (weak scaling): bytes all
    ranks processed over the slowest rank's time; the step time is the max."""
    d_bytes = sum(s[0] for s in stats)
    v_bytes = sum(s[2] for s in stats)
    gemv_ms = max(s[1] for s in stats)
    gemm_ms = max(s[3] for s in stats)
    return {"gemv_gbs": d_bytes / (gemv_ms * 1e-3) / 1e9, "gemm_gbs": v_bytes / (gemm_ms * 1e-3) / 1e9,
            "ms_per_step": max(s[4] for s in stats), "e2e_ms": max(s[5] for s in stats) if len(stats[0]) > 5 else 0.0}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    K, W = args.steps, max(args.warmup, 3)
    per = max(1.0, min(args.cpu_seconds, 90.0 / (K + W)))
    for _ in range(W):
        cpu_baseline(per / 4, args.keep, args.mant, args.variant)
    vals = [cpu_baseline(per, args.keep, args.mant, args.variant) for _ in range(K)]
    v = statistics.median(x["value"] for x in vals)
    import synthetic
    shp = synthetic.LLAMA3_8B if args.workload == "llama3-8b" else synthetic.QWEN3_8B
    out = {
        "impl": "reference",
        "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "layers": args.layers, "hidden": shp["hidden"], "ffn": shp["ffn"],
                   "batch": args.batch, "draft_len": args.draft_len, "keep_per_block": args.keep,
                   "mant_bits": args.mant, "variant": f"Cassandra-{args.variant}"},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": vals[0]["cores"],
                         "host_cores": vals[0]["host_cores"], "kind": "oracle",
                         "single_thread_value": round(statistics.median(x["single_thread_value"] for x in vals), 4),
                         "sample": vals[0]["sample"]},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "CPU oracle (plain C) timed on the host cores on a bounded sample of the draft GEMV workload; "
                "value = speculation bytes decoded per second with every core",
    }
    print(json.dumps(out), flush=True)


def run_micro(args):
    """One kernel on one tensor: reps launches timed with CUDA events, bytes
    per launch from the encoded section lengths."""
    import torch

    import bit_level_weight_gb300 as cas
    import synthetic
    from bit_level_weight_gb300 import build as _b
    _b.build()
    dev = torch.device("cuda", 0)
    st = torch.cuda.Stream(device=dev)
    out = {"micro": args.micro}
    if args.micro in ("draft_gemv", "verify_gemm", "encode"):
        W = synthetic.t4_weight(args.N, args.K, seed=1, device=dev)
        enc = cas.encode_weights(W, args.variant, args.keep, args.mant)
        if args.micro == "draft_gemv":
            x = synthetic.activations(args.nvec, args.K, seed=2, device=dev)
            y = torch.empty(args.nvec, args.N, dtype=torch.float32, device=dev)
            call = cas.prepare("cas_draft_gemv", enc, x, args.nvec, y, st)
            nbytes = enc.spec_bytes() + args.nvec * args.K * 2 + args.nvec * args.N * 4
        elif args.micro == "verify_gemm":
            X = synthetic.activations(args.T, args.K, seed=3, device=dev)
            Y = torch.empty(args.T, args.N, dtype=torch.float32, device=dev)
            call = cas.prepare("cas_verify_gemm", enc, X, args.T, Y, st)
            nbytes = enc.all_bytes() + args.T * args.K * 2 + args.T * args.N * 4
        else:
            ws = torch.empty(cas.cas_encode_workspace_bytes(args.N, args.K), dtype=torch.uint8, device=dev)
            buf = torch.empty_like(enc.buf)

            def call():
                cas.cas_encode_weights(W, enc.desc, buf, ws, st)
            nbytes = args.N * args.K * 2 + enc.all_bytes()
        out.update(N=args.N, K=args.K, variant=args.variant, keep=args.keep, mant=args.mant,
                   spec_bits_per_elem=enc.spec_bytes() * 8 / (args.N * args.K),
                   all_bits_per_elem=enc.all_bytes() * 8 / (args.N * args.K))
    else:
        H, Hq = 8, 32
        sk, sv = synthetic.kv_scales(0, H, 0, device=dev), synthetic.kv_scales(0, H, 1, device=dev)
        Kc = synthetic.kv_tokens(args.ctx, H, seed=5, scales=sk, device=dev)
        Vc = synthetic.kv_tokens(args.ctx, H, seed=6, scales=sv, device=dev)
        kv = cas.KVCache(H, args.ctx + 64, cas.params(args.variant, args.keep, args.mant), Kc[:128], Vc[:128])
        for t0 in range(0, args.ctx, 2048):
            kv.append(Kc[t0:t0 + 2048], Vc[t0:t0 + 2048])
        assert kv.status() == (args.ctx, 0)
        spec, full = kv_section_bytes(kv, args.ctx, args.variant, args.keep, args.mant)
        if args.micro == "draft_attn":
            q = synthetic.activations(1, Hq * 128, seed=7, device=dev).view(1, Hq, 128)
            tk = synthetic.activations(1, H * 128, seed=8, device=dev).view(1, 1, H, 128)
            tv = synthetic.activations(1, H * 128, seed=9, device=dev).view(1, 1, H, 128)
            o = torch.empty(1, Hq, 128, dtype=torch.float32, device=dev)
            ws = torch.empty(cas.cas_attn_workspace_bytes(1, Hq, 1, args.ctx + 64), dtype=torch.uint8, device=dev)
            call = cas.prepare_draft_attn([kv], q, tk, tv, o, ws, st)
            nbytes = spec
        elif args.micro == "verify_attn":
            kv.truncate(args.ctx - args.T)
            kv.append(Kc[-args.T:], Vc[-args.T:])
            q = synthetic.activations(args.T, Hq * 128, seed=7, device=dev).view(1, args.T, Hq, 128)
            o = torch.empty(1, args.T, Hq, 128, dtype=torch.float32, device=dev)
            ws = torch.empty(cas.cas_attn_workspace_bytes(1, Hq, args.T, args.ctx + 64), dtype=torch.uint8, device=dev)
            call = cas.prepare_verify_attn([kv], q, o, ws, st)
            nbytes = full
        else:
            newk = Kc[-args.T:].contiguous()
            newv = Vc[-args.T:].contiguous()
            app = kv.prepare_append(newk, newv, st)
            tr = kv.prepare_truncate(args.ctx, st)

            def call():
                app()
                tr()
            nbytes = 2 * args.T * H * 128 * 2
        out.update(ctx=args.ctx, T=args.T, kv_spec_bytes=spec, kv_all_bytes=full)
    with torch.cuda.stream(st):
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(args.reps):
            call()
        b.record(st)
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.reps
    peak, _ = peaks()
    out.update(us_per_call=round(ms * 1e3, 2), bytes_per_call=int(nbytes),
               gbs=round(nbytes / (ms * 1e-3) / 1e9, 1), frac_of_hbm=round(nbytes / (ms * 1e-3) / 1e9 / peak, 4))
    print(json.dumps(out), flush=True)


def kv_section_bytes(kv, n: int, variant: int, k: int, m: int) -> tuple:
    """(speculation bytes, all bytes) of the KV cache's 2H streams holding n
    tokens: fixed per-token records plus the words of every variable-length
    stream and its superblock index."""
    words = lambda f, w: -(-(f * w) // 32) * 4  # noqa: E731
    nsb = (n + 7) // 8
    idx = (nsb + 1) * 4

    def stream(name, s_):
        return 4 * int(kv.section(name, s_).cpu().numpy().view("uint32")[nsb]) + idx
    spec = full = 0
    for s_ in range(2 * kv.H):
        if variant == 1:
            sp = n * (16 + words(k, m + 1)) + stream("spec_sbidx", s_)
            vr = n * (words(k, 7 - m) + words(128 - k, 8)) + stream("ver_sbidx", s_)
        else:
            sp = n * (16 + 4 + words(k, m + 2))
            vr = (n * words(128 - k, 8) + stream("ver_sbidx", s_) + stream("ver_d_sbidx", s_)
                  + stream("ver_res_sbidx", s_))
        spec += sp
        full += sp + vr
    return spec, full


def run_sweep(args):
    """Cassandra-1 vs Cassandra-2 on the two FFN matrix shapes, keep 20..60 %
    x mantissa 1..5: compression ratio CR = 1 - speculation bytes / bf16 bytes
    (sections, index and padding included) and draft GEMV GB/s. One JSON line
    per point; the points with CR in [40, 80] % are the pages' usable range."""
    import torch

    import bit_level_weight_gb300 as cas
    import synthetic
    from bit_level_weight_gb300 import build as _b
    _b.build()
    dev = torch.device("cuda", 0)
    st = torch.cuda.Stream(device=dev)
    for (N, K) in ((4096, 14336), (14336, 4096)):
        W = synthetic.normal_weight(N, K, seed=N + K, std=0.02, device=dev)
        x = synthetic.activations(1, K, seed=3, device=dev)
        y = torch.empty(1, N, dtype=torch.float32, device=dev)
        for keep in (0.2, 0.3, 0.4, 0.5, 0.6):
            k = cas.cas_keep_from_ratio(keep)
            for m in range(1, 6):
                chosen, _ = cas.cas_choose_variant(W, k, m)  # per-tensor choice: fewer speculation bytes
                for variant in (1, 2):
                    enc = cas.encode_weights(W, variant, k, m)
                    call = cas.prepare("cas_draft_gemv", enc, x, 1, y, st)
                    with torch.cuda.stream(st):
                        for _ in range(3):
                            call()
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record(st)
                        for _ in range(10):
                            call()
                        b.record(st)
                        torch.cuda.synchronize()
                    ms = a.elapsed_time(b) / 10
                    nbytes = enc.spec_bytes() + K * 2 + N * 4
                    cr = 1.0 - enc.spec_bytes() / (2.0 * N * K)
                    print(json.dumps({"sweep": "cassandra-1 vs -2", "N": N, "K": K, "keep": keep, "k": k, "m": m,
                                      "variant": variant, "chosen": variant == chosen,
                                      "cr": round(cr, 4), "in_40_80": 0.4 <= cr <= 0.8,
                                      "spec_bits_per_elem": round(enc.spec_bytes() * 8 / (N * K), 3),
                                      "all_bits_per_elem": round(enc.all_bytes() * 8 / (N * K), 3),
                                      "draft_gemv_us": round(ms * 1e3, 1),
                                      "draft_gemv_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}), flush=True)
                    del enc


def run_capacity(args):
    """Memory-capacity model (the pages' 24 GB / Llama 3 8B comparison, Fig. 14):
    model bytes and KV bytes per token measured from this library's encodings
    (one decoder layer of weights, 4096 appended KV tokens), then the longest
    context that fits a budget, bf16 vs Cassandra (both streams stored, as
    the verification needs them). EAGLE-3 is modelled as bf16 plus one extra
    bf16 decoder layer and its KV (a reading: the pages give no size)."""
    import torch

    import bit_level_weight_gb300 as cas
    import synthetic
    from bit_level_weight_gb300 import build as _b
    _b.build()
    dev = torch.device("cuda", 0)
    shp = dict(synthetic.LLAMA3_8B)
    L, h, nkv, hd = shp["layers"], shp["hidden"], shp["n_kv"], shp["head_dim"]
    vocab = 128256  # Llama 3 embedding and LM head rows
    layer_params, layer_bytes, layer_spec = 0, 0, 0
    for idx, (nm, N, K) in enumerate(synthetic.layer_matrices(shp)):
        W = synthetic.t4_weight(N, K, seed=idx, device=dev)
        enc = cas.encode_weights(W, 1, args.keep, args.mant)
        layer_params += N * K
        layer_bytes += enc.all_bytes()
        layer_spec += enc.spec_bytes()
        del W, enc
    bits_per_param = layer_bytes * 8 / layer_params
    T = 4096
    sk, sv = synthetic.kv_scales(0, nkv, 0, device=dev), synthetic.kv_scales(0, nkv, 1, device=dev)
    Kc = synthetic.kv_tokens(T, nkv, seed=5, scales=sk, device=dev)
    Vc = synthetic.kv_tokens(T, nkv, seed=6, scales=sv, device=dev)
    kv = cas.KVCache(nkv, T, cas.params(1, args.keep, args.mant), Kc[:128], Vc[:128])
    kv.append(Kc, Vc)
    assert kv.status() == (T, 0)
    k, m = args.keep, args.mant
    rec = lambda f, w: -(-(f * w) // 32) * 4  # noqa: E731
    per_tok_fixed = 16 + rec(k, m + 1) + rec(k, 7 - m) + rec(128 - k, 8)
    nsb = (T + 7) // 8
    code_bytes = 0
    for st in range(2 * nkv):
        code_bytes += 4 * int(kv.section("spec_sbidx", st).cpu().numpy().view("uint32")[nsb])
        code_bytes += 4 * int(kv.section("ver_sbidx", st).cpu().numpy().view("uint32")[nsb])
        code_bytes += 2 * 4 * (nsb + 1)
    kv_layer_bytes = 2 * nkv * T * per_tok_fixed + code_bytes
    kv_bits_per_elem = kv_layer_bytes * 8 / (T * 2 * nkv * hd)
    params = L * layer_params + 2 * vocab * h
    kv_bf16_tok = L * 2 * nkv * hd * 2
    kv_cas_tok = kv_bf16_tok * kv_bits_per_elem / 16
    embed_bytes = 2 * vocab * h * 2  # embedding and LM head kept bf16 in this model
    schemes = {
        "bf16": (params * 2, kv_bf16_tok),
        "eagle3 (bf16 + one bf16 draft layer)": (params * 2 + layer_params * 2, kv_bf16_tok * (L + 1) / L),
        "cassandra": (L * layer_params * bits_per_param / 8 + embed_bytes, kv_cas_tok),
    }
    for budget_name, budget in (("24 GB (RTX 4090 in the pages)", 24e9), ("GB300 HBM 284208 MiB", 284208 * 2**20)):
        base = None
        for name, (wbytes, tok) in schemes.items():
            ctx = max(0.0, (budget - wbytes) / tok)
            base = base or ctx
            print(json.dumps({"capacity": budget_name, "scheme": name, "weights_gb": round(wbytes / 1e9, 3),
                              "kv_bytes_per_token": round(tok), "max_context_tokens": int(ctx),
                              "vs_bf16": round(ctx / base, 3) if base else None,
                              "weight_bits_per_param": round(bits_per_param, 3) if name == "cassandra" else 16,
                              "kv_bits_per_elem": round(kv_bits_per_elem, 3) if name == "cassandra" else 16}),
                  flush=True)


def main():
    args = parse()
    if args.capacity:
        run_capacity(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.micro:
        run_micro(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cas(args)


if __name__ == "__main__":
    main()
