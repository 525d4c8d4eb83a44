"""Writes tests/golden/exponent_stats.json: exponent entropy, unary mean code
length and Huffman mean code length of the synthetic workloads, from the CPU
oracle only (blog review section 3.2: entropy about 2.6 bits for weights and
2.7-2.8 for the KV cache; unary about 2.85 bits, slightly above Huffman)."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synthetic  # noqa: E402


def row(w, k=64):
    c = oracle.exp_hist(w)
    _, roe = oracle.rank_table(c)
    keep = np.concatenate([oracle.select_block(b, k) for b in w.reshape(-1, 128)[:20000]])
    flat = w.reshape(-1)[: keep.size]
    ck, cp = oracle.exp_hist(flat[keep]), oracle.exp_hist(flat[~keep])
    return {"entropy_bits": oracle.exp_entropy(c), "unary_mean_bits": oracle.unary_mean_len(c, roe),
            "huffman_mean_bits": oracle.huffman_mean_len(c), "distinct_exponents": int((c > 0).sum()),
            "unary_mean_bits_kept": oracle.unary_mean_len(ck, roe),
            "unary_mean_bits_pruned": oracle.unary_mean_len(cp, roe)}


def main():
    out = {}
    out["cfg0_4096x4096_normal_outliers"] = row(synthetic.cfg0_weight().numpy().view(np.uint16))
    out["t4_14336x4096_llama_ffn"] = row(synthetic.t4_weight(14336, 4096, seed=4).numpy().view(np.uint16))
    sc = synthetic.kv_scales(0, 8, 0)
    out["kv_4096x8x128_lognormal_channels"] = row(
        synthetic.kv_tokens(4096, 8, seed=11, scales=sc).numpy().view(np.uint16).reshape(-1, 128))
    with open(os.path.join(HERE, "exponent_stats.json"), "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
    print(json.dumps(out, indent=1, sort_keys=True))


if __name__ == "__main__":
    main()
