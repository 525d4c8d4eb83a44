"""Host-side arithmetic of bench.py (no GPU): kernel naming, the ALU issue
roof and the KV section byte count."""
import types

import numpy as np
import pytest
import torch

import bench


def args(variant=1, keep=64, mant=3):
    return types.SimpleNamespace(variant=variant, keep=keep, mant=mant)


@pytest.mark.parametrize("a,nvec,name", [
    (args(), 1, "draft_gemv_block_kernel<1>"), (args(), 2, "draft_gemv_block_kernel<2>"),
    (args(), 3, "draft_gemv_fast_kernel<3>"),
    (args(2), 2, "draft_gemv_fast2_kernel<2>"), (args(2), 3, "draft_gemv_runs_kernel<2,3>"),
    (args(1, 38), 1, "draft_gemv_runs_kernel<1,1>"), (args(2, 64, 4), 1, "draft_gemv_runs_kernel<2,1>"),
])
def test_gemv_kernel_name(a, nvec, name):
    assert bench.gemv_kernel_name(a, nvec) == name


def test_alu_roof_arithmetic():
    clk = types.SimpleNamespace(summary=lambda: {"sm_mhz": 2000.0})
    rec = {"lane_instr_per_elem": 23.0, "spec_bits_per_elem": 4.205, "shape": "28672 x 4096"}
    r = bench.alu_roof(500.0, clk, rec)
    peak = 152 * 128 * 2000e6
    elems = 500e9 / (4.205 / 8)
    assert r["bound"] == "alu"
    assert r["peak"] == pytest.approx(peak / 1e12, abs=0.01)
    assert r["achieved"] == pytest.approx(23.0 * elems / 1e12, abs=0.01)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], abs=1e-3)
    budget = peak / (0.75 * bench.peaks()[0] * 1e9 / (4.205 / 8))
    assert r["budget_at_75pct_hbm"] == pytest.approx(budget, abs=0.01)
    assert bench.alu_roof(500.0, clk, None) is None


def test_profiled_record_needs_matching_source_hash(monkeypatch):
    h = bench.source_hash()
    rec = {"source_sha16": h, "traffic_ratio": 1.0, "lane_instr_per_elem": 1.0, "spec_bits_per_elem": 4.2,
           "shape": "x"}
    monkeypatch.setitem(bench.PROFILED, "k<1>", rec)
    assert bench.profiled_record("k<1>") is rec
    monkeypatch.setitem(bench.PROFILED, "k<1>", dict(rec, source_sha16="0" * 16))
    assert bench.profiled_record("k<1>") is None
    assert bench.profiled_record("absent<1>") is None


class FakeKV:
    """Two streams (H = 1) with known superblock indices."""
    H = 1

    def __init__(self, n):
        nsb = (n + 7) // 8
        self.idx = {"spec_sbidx": [10, 20], "ver_sbidx": [30, 40], "ver_d_sbidx": [5, 6],
                    "ver_res_sbidx": [7, 8]}
        self.nsb = nsb

    def section(self, name, s):
        a = np.zeros(self.nsb + 1, np.uint32)
        a[self.nsb] = self.idx[name][s]
        return torch.from_numpy(a.view(np.uint8))


@pytest.mark.parametrize("variant", [1, 2])
def test_kv_section_bytes(variant):
    n, k, m = 20, 38, 3
    kv = FakeKV(n)
    spec, full = bench.kv_section_bytes(kv, n, variant, k, m)
    words = lambda f, w: -(-(f * w) // 32) * 4  # noqa: E731
    idx = (3 + 1) * 4  # 3 superblocks + 1 index entries
    if variant == 1:
        sp = [n * (16 + words(k, m + 1)) + 4 * w + idx for w in (10, 20)]
        vr = [n * (words(k, 7 - m) + words(128 - k, 8)) + 4 * w + idx for w in (30, 40)]
    else:
        sp = [n * (20 + words(k, m + 2))] * 2
        vr = [n * words(128 - k, 8) + 4 * (a + b + c) + 3 * idx for a, b, c in ((30, 5, 7), (40, 6, 8))]
    assert spec == sum(sp)
    assert full == sum(sp) + sum(vr)
