#!/usr/bin/env python
"""Benchmark of the Cassandra bit-split hot path on GB300.

One step = one self-speculative decode step of a Llama-3-8B-shaped decoder
stack (32 layers, hidden 4096, FFN 14336, GQA 32q/8kv, head_dim 128) with
random-init Student-t(4) bf16 weights split at keep 50% / 3 mantissa bits
(Cassandra-1), batch 1, draft length 4, and a compressed KV cache of 32K tokens
(bf16 K/V ~ N(0,1) x LogNormal(0,0.5) channel scales):
  4 draft forwards  : per layer draft GEMV (Wqkv), draft attention over the
                      speculation KV + bf16 tail, draft GEMV (Wo, Wgate|up, Wdown);
  1 verify forward  : per layer verify GEMM (T=5), online KV append of the 5
                      tokens, verify attention, verify GEMMs;
  then the 5 tokens are rolled back (fixed schedule: acceptance has no meaning
  on random weights).
Activations fed to each kernel are synthetic device vectors (the norm / RoPE /
activation glue between kernels is not part of the measured path).

Headline value: draft decode+GEMV GB/s over the algorithmic bytes of the
speculation streams read (plus x read and y written), timed with CUDA events on
the launching stream around the draft-GEMV launches of the timed steps.
Also reported: verify GEMM GB/s, microseconds per decode step, roofline of the
draft GEMV against the measured HBM copy bandwidth, the end-to-end number
through the C ABI with host buffers, and the CPU oracle as a reported baseline.

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
    """Oracle draft decode + GEMV (plain C, one thread) on a bounded sample: one
    1024x4096 Student-t(4) matrix of the same stack, repeated for ~`seconds`."""
    import numpy as np

    import oracle
    import synthetic
    N, K = 1024, 4096
    W = synthetic.t4_weight(N, K, seed=0).numpy().view(np.uint16)
    x = synthetic.activations(1, K, seed=1).numpy().view(np.uint16)
    enc = oracle.encode(W, variant, keep, mant)
    spec = enc.spec_bytes() + K * 2 + N * 4
    reps, t0 = 0, time.perf_counter()
    while True:
        d = oracle.decode(enc, False)
        oracle.matvec(d, x)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": spec * reps / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} x oracle draft decode + float64 GEMV of one 1024x4096 t4 matrix "
                      f"(keep {keep}/128, m={mant}, Cassandra-{variant}), {dt:.1f} s"}


# ---------------------------------------------------------------------- workload
class Stack:
    """Encoded Llama-3-8B-shaped stack plus its compressed KV caches."""

    def __init__(self, cas, args, dev):
        import torch

        import synthetic
        self.cas, self.args, self.dev = cas, args, dev
        shp = dict(synthetic.LLAMA3_8B if args.workload == "llama3-8b" else synthetic.QWEN3_8B)
        self.L = args.layers
        self.vocab = shp.get("vocab", 0)
        h, f = shp["hidden"], shp["ffn"]
        self.hidden, self.ffn, self.nq, self.nkv, self.hd = h, f, shp["n_q"], shp["n_kv"], shp["head_dim"]
        self.mats = []  # per layer: dict name -> EncodedWeights
        t0 = time.time()
        for layer in range(self.L):
            names = synthetic.layer_matrices(shp)
            raw = {}
            for idx, (nm, N, K) in enumerate(names):
                raw[nm] = synthetic.t4_weight(N, K, seed=layer * 16 + idx, device=dev)
            fused = {
                "qkv": torch.cat([raw["wq"], raw["wk"], raw["wv"]], 0),
                "o": raw["wo"],
                "gateup": torch.cat([raw["wgate"], raw["wup"]], 0),
                "down": raw["wdown"],
            }
            del raw
            enc = {nm: cas.encode_weights(W, args.variant, args.keep, args.mant) for nm, W in fused.items()}
            del fused
            self.mats.append(enc)
        self.lm = None
        if self.vocab:
            Wl = synthetic.t4_weight(self.vocab, h, seed=999_983, device=dev)
            self.lm = cas.encode_weights(Wl, args.variant, args.keep, args.mant)
            del Wl
        torch.cuda.synchronize()
        self.encode_s = time.time() - t0
        self.kv = None
        if not args.no_attn and hasattr(cas, "KVCache"):
            self._fill_kv()

    def _fill_kv(self):
        import torch

        import synthetic
        cas, args, dev = self.cas, self.args, self.dev
        T = args.ctx
        self.kv = []
        p = cas.params(args.variant, args.keep, args.mant)
        chunk = 2048
        for layer in range(self.L):
            layer_kv = []
            for b in range(args.batch):
                sk = synthetic.kv_scales(layer, self.nkv, 0, device=dev)
                sv = synthetic.kv_scales(layer, self.nkv, 1, device=dev)
                Kc = synthetic.kv_tokens(T, self.nkv, seed=100 * layer + 2 * b, scales=sk, device=dev)
                Vc = synthetic.kv_tokens(T, self.nkv, seed=100 * layer + 2 * b + 1, scales=sv, device=dev)
                kv = cas.KVCache(self.nkv, T + 64, p, Kc[:128], Vc[:128])
                for t0 in range(0, T, chunk):
                    kv.append(Kc[t0:t0 + chunk], Vc[t0:t0 + chunk])
                layer_kv.append(kv)
                del Kc, Vc
            self.kv.append(layer_kv)
        torch.cuda.synchronize()
        for layer_kv in self.kv:
            for kv in layer_kv:
                n, st = kv.status()
                assert st == 0 and n == T, (n, st)


def run_cas(args):
    import torch
    import torch.distributed as dist

    import bit_level_weight_gb300 as cas
    import synthetic

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from bit_level_weight_gb300 import build as _b
    _b.build()

    stk = Stack(cas, args, dev)
    st = torch.cuda.Stream(device=dev)  # every call of the step is bound to this stream
    D, B = args.draft_len, args.batch
    nvec = B
    xs = {"qkv": synthetic.activations(nvec, stk.hidden, seed=1, device=dev),
          "o": synthetic.activations(nvec, stk.hidden, seed=2, device=dev),
          "gateup": synthetic.activations(nvec, stk.hidden, seed=3, device=dev),
          "down": synthetic.activations(nvec, stk.ffn, seed=4, device=dev)}
    T = B * (D + 1)
    Xs = {"qkv": synthetic.activations(T, stk.hidden, seed=5, device=dev),
          "o": synthetic.activations(T, stk.hidden, seed=6, device=dev),
          "gateup": synthetic.activations(T, stk.hidden, seed=7, device=dev),
          "down": synthetic.activations(T, stk.ffn, seed=8, device=dev)}
    ys = {nm: torch.empty(nvec, stk.mats[0][nm].N, dtype=torch.float32, device=dev) for nm in xs}
    Ys = {nm: torch.empty(T, stk.mats[0][nm].N, dtype=torch.float32, device=dev) for nm in Xs}

    gemv = [{nm: cas.prepare("cas_draft_gemv", stk.mats[l][nm], xs[nm], nvec, ys[nm], st) for nm in xs}
            for l in range(stk.L)]
    gemm = [{nm: cas.prepare("cas_verify_gemm", stk.mats[l][nm], Xs[nm], T, Ys[nm], st) for nm in Xs}
            for l in range(stk.L)]
    draft_bytes = {nm: sum(stk.mats[l][nm].spec_bytes() + nvec * stk.mats[l][nm].K * 2 + nvec * stk.mats[l][nm].N * 4
                           for l in range(stk.L)) for nm in xs}
    verify_bytes = {nm: sum(stk.mats[l][nm].all_bytes() + T * stk.mats[l][nm].K * 2 + T * stk.mats[l][nm].N * 4
                            for l in range(stk.L)) for nm in Xs}
    lm_gemv = lm_gemm = None
    if stk.lm is not None:
        y_lm = torch.empty(nvec, stk.vocab, dtype=torch.float32, device=dev)
        Y_lm = torch.empty(T, stk.vocab, dtype=torch.float32, device=dev)
        lm_gemv = cas.prepare("cas_draft_gemv", stk.lm, xs["qkv"], nvec, y_lm, st)
        lm_gemm = cas.prepare("cas_verify_gemm", stk.lm, Xs["qkv"], T, Y_lm, st)
        draft_bytes["lm_head"] = stk.lm.spec_bytes() + nvec * stk.hidden * 2 + nvec * stk.vocab * 4
        verify_bytes["lm_head"] = stk.lm.all_bytes() + T * stk.hidden * 2 + T * stk.vocab * 4

    attn = stk.kv is not None
    if attn:
        q_d = synthetic.activations(B, stk.nq * stk.hd, seed=20, device=dev).view(B, stk.nq, stk.hd)
        tail_k = synthetic.activations(B * D, stk.nkv * stk.hd, seed=21, device=dev).view(B, D, stk.nkv, stk.hd)
        tail_v = synthetic.activations(B * D, stk.nkv * stk.hd, seed=22, device=dev).view(B, D, stk.nkv, stk.hd)
        q_v = synthetic.activations(B * (D + 1), stk.nq * stk.hd, seed=23, device=dev).view(B, D + 1, stk.nq, stk.hd)
        newk = synthetic.activations(D + 1, stk.nkv * stk.hd, seed=24, device=dev).view(D + 1, stk.nkv, stk.hd)
        newv = synthetic.activations(D + 1, stk.nkv * stk.hd, seed=25, device=dev).view(D + 1, stk.nkv, stk.hd)
        ws = torch.empty(cas.cas_attn_workspace_bytes(B, stk.nq, D + 1, args.ctx + 64), dtype=torch.uint8, device=dev)
        o_d = torch.empty(B, stk.nq, stk.hd, dtype=torch.float32, device=dev)
        o_v = torch.empty(B, D + 1, stk.nq, stk.hd, dtype=torch.float32, device=dev)
        tails = [(tail_k[:, :d + 1].contiguous(), tail_v[:, :d + 1].contiguous()) for d in range(D)]
        dattn = [[cas.prepare_draft_attn(stk.kv[l], q_d, tails[d][0], tails[d][1], o_d, ws, st) for d in range(D)]
                 for l in range(stk.L)]
        vattn = [cas.prepare_verify_attn(stk.kv[l], q_v, o_v, ws, st) for l in range(stk.L)]
        appends = [[kv.prepare_append(newk, newv, st) for kv in stk.kv[l]] for l in range(stk.L)]
        truncs = [[kv.prepare_truncate(args.ctx, st) for kv in stk.kv[l]] for l in range(stk.L)]

    # The step as an ordered list of segments; GEMV / GEMM segments are timed.
    def seq(*fns):
        def run():
            for f in fns:
                f()
        return run
    segs = []  # (kind, callable)
    for d in range(D):
        for l in range(stk.L):
            g = gemv[l]
            segs.append(("gemv", g["qkv"]))
            if attn:
                segs.append(("attn", dattn[l][d]))
            segs.append(("gemv", seq(g["o"], g["gateup"], g["down"])))
        if lm_gemv is not None:
            segs.append(("gemv", lm_gemv))
    for l in range(stk.L):
        g = gemm[l]
        segs.append(("gemm", g["qkv"]))
        if attn:
            segs.append(("attn", seq(*appends[l], vattn[l])))
        segs.append(("gemm", seq(g["o"], g["gateup"], g["down"])))
    if lm_gemm is not None:
        segs.append(("gemm", lm_gemm))
    if attn:
        segs.append(("attn", seq(*[t for l in range(stk.L) for t in truncs[l]])))

    launches_per_step = D * stk.L * 4 + stk.L * 4 + (D + 1 if lm_gemv is not None else 0)
    if attn:
        launches_per_step += D * stk.L * 2 + stk.L * (2 * B + 2) + stk.L * B

    # eager warm-up (also caches every launch configuration), then one CUDA
    # graph per segment so the timed region has no host gaps inside a segment
    with torch.cuda.stream(st):
        for _ in range(max(args.warmup, 3)):
            for _, f in segs:
                f()
    torch.cuda.synchronize()
    graphs = []
    for kind, f in segs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            f()
        graphs.append((kind, g))
    torch.cuda.synchronize()
    n_timed = sum(1 for k, _ in graphs if k != "attn")
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * n_timed)] for _ in range(args.steps)]

    def step(ev=None):
        e = 0
        for kind, g in graphs:
            if ev is not None and kind != "attn":
                ev[e].record(st)
                g.replay()
                ev[e + 1].record(st)
                e += 2
            else:
                g.replay()

    with torch.cuda.stream(st):
        for _ in range(max(args.warmup, 3)):
            step()
    torch.cuda.synchronize()

    # ---- timed region
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    gemv_ms, gemm_ms = 0.0, 0.0
    kinds = [k for k, _ in graphs if k != "attn"]
    with ClockSampler(local) as clk, torch.cuda.stream(st):
        torch.cuda.nvtx.range_push("timed")  # lets a profiler select the timed launches
        t_start.record(st)
        for i in range(args.steps):
            step(evsets[i])
        t_end.record(st)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    for ev in evsets:
        for i, kind in enumerate(kinds):
            ms = ev[2 * i].elapsed_time(ev[2 * i + 1])
            if kind == "gemv":
                gemv_ms += ms
            else:
                gemm_ms += ms
    total_ms = t_start.elapsed_time(t_end)
    if world > 1:
        dist.barrier()

    steps = args.steps
    d_bytes = sum(draft_bytes.values()) * D * steps
    v_bytes = sum(verify_bytes.values()) * steps
    gemv_gbs = d_bytes / (gemv_ms * 1e-3) / 1e9
    gemm_gbs = v_bytes / (gemm_ms * 1e-3) / 1e9
    ms_per_step = total_ms / steps

    # ---- e2e: draft GEMV pass of the whole stack through the C ABI with the
    # activation in pinned host memory (H2D) and every output read back (D2H)
    with torch.cuda.stream(st):
        e2e = e2e_draft_pass(cas, stk, xs, ys, nvec, st, steps=max(3, steps))

    if world > 1:
        agg = replica_aggregate(gather_stats((d_bytes, gemv_ms, v_bytes, gemm_ms, ms_per_step), world))
        gemv_gbs, gemm_gbs, ms_per_step = agg["gemv_gbs"], agg["gemm_gbs"], agg["ms_per_step"]
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = peaks()
    n_gemv = 4 * stk.L + (1 if lm_gemv is not None else 0)
    per_launch_bytes = sum(draft_bytes.values()) / n_gemv
    per_launch_ms = gemv_ms / (steps * D * n_gemv)
    achieved = per_launch_bytes / (per_launch_ms * 1e-3) / 1e9
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
            "layers": stk.L, "lm_head_rows": stk.vocab or None, "hidden": stk.hidden, "ffn": stk.ffn, "heads": f"{stk.nq}q/{stk.nkv}kv x {stk.hd}",
            "batch": B, "draft_len": D, "verify_tokens": T, "ctx": args.ctx if attn else 0,
            "keep_per_block": args.keep, "mant_bits": args.mant, "variant": f"Cassandra-{args.variant}",
            "weights": "Student-t(4) x 0.02/sqrt(2), fused qkv and gate|up",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": f"inputs larger than L2 ({sum(draft_bytes.values()) / 1e9:.2f} GB speculation stream per draft pass)",
        },
        "verify_gemm_gbs": round(gemm_gbs, 1),
        "us_per_decode_step": round(ms_per_step * 1e3, 1),
        "draft_gemv_frac_of_hbm": round(gemv_gbs / world / peak, 4),
        "draft_gemv_frac_of_8tbs_nominal": round(gemv_gbs / world / 8000.0, 4),
        "verify_gemm_frac_of_hbm": round(gemm_gbs / world / peak, 4),
        "roofline": {"kernel": gemv_kernel_name(args, B), "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                     "traffic": (round(PROFILED_TRAFFIC_RATIO * per_launch_bytes) if PROFILED_TRAFFIC_RATIO
                                 else None),
                     "traffic_note": "per launch: (ncu dram bytes / algorithmic bytes of a 28672x4096 launch, "
                                     "profiles/draft_gemv_28672x4096.md) x algorithmic bytes per launch of this step",
                     "algorithmic_bytes_per_launch": int(per_launch_bytes)},
        "alu_roof": (alu_roof(achieved, clk) if args.variant == 1 and args.keep == 64 and args.mant == 3 and B == 1
                     else None),
        "e2e": e2e,
        "gpu_launches": launches_per_step * steps,
        "encode_s": round(stk.encode_s, 2),
    }
    out["clocks"] = clk.summary()
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds, args.keep, args.mant, args.variant)
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


# dram bytes read + written / algorithmic bytes of one draft_gemv_fast_kernel<1>
# launch on the 28672 x 4096 matrix (ncu: 62.04 MB for 61.85 MB algorithmic,
# profiles/draft_gemv_28672x4096.md); set to None whenever that kernel changes
# until it is captured again
PROFILED_TRAFFIC_RATIO = (61.904384 + 0.135168) / 61.85268


# warp instructions x 32 / elements of one draft_gemv_fast_kernel<1> launch on
# the 28672 x 4096 matrix (ncu smsp__inst_executed.sum,
# profiles/draft_gemv_28672x4096.md); None whenever that kernel changes
PROFILED_LANE_INSTR_PER_ELEM = 107314082 * 32 / (28672 * 4096)
SMS, LANES_PER_SM_CLK = 152, 128  # 4 schedulers x 32 lanes issue per SM clock


def gemv_kernel_name(args, nvec: int) -> str:
    """The draft GEMV kernel the stack's matrices (rows of whole superblocks) run."""
    if args.keep == 64 and args.mant == 3:
        if args.variant == 1:
            return f"draft_gemv_fast_kernel<{nvec}>"
        if nvec <= 2:
            return f"draft_gemv_fast2_kernel<{nvec}>"
    return f"draft_gemv_runs_kernel<{args.variant},{nvec}>"


def alu_roof(achieved_gbs: float, clk) -> dict:
    """The draft GEMV is bound by instruction issue (integer decode), so its
    second roof is the lane-instruction issue peak: SMs x 128 x SM clock.
    achieved = profiled lane instructions per element x elements per second."""
    if PROFILED_LANE_INSTR_PER_ELEM is None:
        return None
    mhz = (clk.summary() or {}).get("sm_mhz") or 2070.0
    peak = SMS * LANES_PER_SM_CLK * mhz * 1e6
    bytes_per_elem = 4.205 / 8  # speculation bits per element of the Student-t matrices (k = 64, m = 3)
    elems = achieved_gbs * 1e9 / bytes_per_elem
    achieved = PROFILED_LANE_INSTR_PER_ELEM * elems
    budget = peak / (0.75 * peaks()[0] * 1e9 / bytes_per_elem)
    return {"bound": "alu", "achieved": round(achieved / 1e12, 2), "peak": round(peak / 1e12, 2),
            "unit": "T lane-instr/s", "frac": round(achieved / peak, 4),
            "lane_instr_per_elem": round(PROFILED_LANE_INSTR_PER_ELEM, 2),
            "budget_at_75pct_hbm": round(budget, 2),
            "note": "lane instructions per element from ncu (profiles/draft_gemv_28672x4096.md); "
                    "peak = 152 SMs x 128 lanes x median SM clock"}


def gather_stats(local: tuple, world: int) -> list:
    """All ranks' (draft bytes, draft ms, verify bytes, verify ms, ms/step)."""
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
            "ms_per_step": max(s[4] for s in stats)}


def e2e_draft_pass(cas, stk, xs, ys, nvec, st, steps):
    import torch
    host_x = {nm: x.cpu().pin_memory() for nm, x in xs.items()}
    host_y = {nm: torch.empty(stk.L, *y.shape, dtype=torch.float32).pin_memory() for nm, y in ys.items()}
    dev_y = {nm: torch.empty(stk.L, *y.shape, dtype=torch.float32, device=y.device) for nm, y in ys.items()}
    calls = [{nm: cas.prepare("cas_draft_gemv", stk.mats[l][nm], xs[nm], nvec, dev_y[nm][l], st) for nm in xs}
             for l in range(stk.L)]
    h2d = sum(t.numel() * t.element_size() for t in host_x.values())
    d2h = sum(t.numel() * t.element_size() for t in host_y.values())
    spec = sum(stk.mats[l][nm].spec_bytes() + nvec * stk.mats[l][nm].K * 2 + nvec * stk.mats[l][nm].N * 4
               for l in range(stk.L) for nm in xs)

    def one():
        for nm in xs:
            xs[nm].copy_(host_x[nm], non_blocking=True)
        for l in range(stk.L):
            c = calls[l]
            c["qkv"](); c["o"](); c["gateup"](); c["down"]()
        for nm in ys:
            host_y[nm].copy_(dev_y[nm], non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(steps):
        one()
    b.record(st)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"value": round(spec / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "what": f"one draft GEMV pass over all {stk.L} layers' matrices via "
            "cas_draft_gemv, x copied in from pinned host memory and all outputs copied out, per step"}


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
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": vals[0]["sample"]},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "CPU oracle (plain C, one thread) timed on a bounded sample of the draft GEMV workload; "
                "value = speculation bytes decoded per second",
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
