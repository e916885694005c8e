"""Writes the fixtures in this directory. Calls only oracle/ (and the seeded
input generators of synthetic/): the pages print no worked example of the
layer, so these files freeze the oracle's own results on small seeded cases.
A later change to the oracle's arithmetic that alters them must say, in its
commit message, which passage (or reading of it) justifies the change.

Run from the repository root: python tests/golden/make_golden.py
"""
import dataclasses
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import moe_oracle as O  # noqa: E402
from synthetic import CONFIGS, get_config, make_inputs  # noqa: E402
from synthetic.gen import normal_f32  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def f32_hex(a):
    return [float(v).hex() for v in np.asarray(a, dtype=np.float32).ravel()]


def routing_case():
    """Softmax, Top-K, weights and capacity drops on 48 tokens, 6 experts,
    top-2, CF 0.75 over sub-sequences of 16 tokens, with repeated logit rows
    (ties between tokens) and a tie between experts inside one token."""
    cfg = dataclasses.replace(get_config("tiny_f32"), T=48, E=6, K=2, drop=True, cf=0.75, S=16)
    logits = normal_f32(7, 10, (cfg.T, cfg.E), std=2.0)
    logits[5] = logits[4]                 # token tie
    logits[9, 2] = logits[9, 4]           # expert tie inside one token
    r = O.route(cfg, None, logits=logits.astype(np.float64))
    counts, offsets, row_of, src_of, n = O.build_map(r["topk_idx"], r["keep"], cfg.E)
    return {"T": cfg.T, "E": cfg.E, "K": cfg.K, "cf": cfg.cf, "S": cfg.S,
            "logits_f32_hex": f32_hex(logits),
            "topk_idx": r["topk_idx"].ravel().tolist(),
            "topk_prob_f32_hex": f32_hex(r["topk_prob"]),
            "topk_w_f32_hex": f32_hex(r["topk_w"]),
            "keep": r["keep"].ravel().tolist(),
            "counts": counts.tolist(), "row_of": row_of.ravel().tolist()}


def layer_case():
    """The tiny fp32 workload's layer output on its first 8 tokens."""
    cfg = get_config("tiny_f32")
    inp = make_inputs(cfg)
    f = O.layer_forward(cfg, inp)
    return {"config": "tiny_f32", "tokens": 8, "out_f32_hex": f32_hex(f["out"][:8])}


def capacities():
    """Capacity per (sub-sequence, expert) and padded rows per expert of the
    token-dropping workloads."""
    out = {}
    for name, c in CONFIGS.items():
        if c.drop:
            S = c.S if 0 < c.S < c.T else c.T
            out[name] = {"cap_full_subseq": O.capacity(c.cf, S, c.K, c.E),
                         "padded_rows_per_expert": O.padded_capacity(c.T, c.S, c.K, c.E, c.cf)}
    return out


if __name__ == "__main__":
    for fname, fn in (("routing_tiny.json", routing_case), ("layer_tiny_f32.json", layer_case),
                      ("capacities.json", capacities)):
        with open(os.path.join(HERE, fname), "w") as f:
            json.dump(fn(), f, indent=0)
            f.write("\n")
        print("wrote", fname)
