"""The oracle against its frozen fixtures (tests/golden/, written by
tests/golden/make_golden.py from the oracle alone): routing decisions, the
weights' fp32 bits, the capacity drops, the map and a small layer output must
not change unless the oracle's arithmetic is changed on purpose. The GPU test
feeds the fixture's logits to moe_route_topk and expects the same bits."""
import dataclasses
import json
import os

import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import CONFIGS, get_config, make_inputs

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def _f32(hexes):
    return np.array([float.fromhex(h) for h in hexes], dtype=np.float32)


def _routing_cfg(g):
    return dataclasses.replace(get_config("tiny_f32"), T=g["T"], E=g["E"], K=g["K"], drop=True,
                               cf=g["cf"], S=g["S"])


def test_routing_fixture():
    g = _load("routing_tiny.json")
    cfg = _routing_cfg(g)
    logits = _f32(g["logits_f32_hex"]).reshape(cfg.T, cfg.E)
    r = O.route(cfg, None, logits=logits.astype(np.float64))
    assert r["topk_idx"].ravel().tolist() == g["topk_idx"]
    assert np.array_equal(np.asarray(r["topk_prob"], np.float32).view(np.uint32),
                          _f32(g["topk_prob_f32_hex"]).view(np.uint32).reshape(cfg.T, cfg.K))
    assert np.array_equal(np.asarray(r["topk_w"], np.float32).view(np.uint32),
                          _f32(g["topk_w_f32_hex"]).view(np.uint32).reshape(cfg.T, cfg.K))
    assert r["keep"].ravel().tolist() == g["keep"]
    counts, _, row_of, _, _ = O.build_map(r["topk_idx"], r["keep"], cfg.E)
    assert counts.tolist() == g["counts"] and row_of.ravel().tolist() == g["row_of"]
    # the fixture exercises both tie rules and actually drops
    assert 0 < sum(g["keep"]) < cfg.T * cfg.K


def test_layer_fixture():
    g = _load("layer_tiny_f32.json")
    cfg = get_config(g["config"])
    out = O.layer_forward(cfg, make_inputs(cfg))["out"][: g["tokens"]]
    assert np.array_equal(np.asarray(out, np.float32).ravel().view(np.uint32),
                          _f32(g["out_f32_hex"]).view(np.uint32))


def test_capacity_fixture():
    g = _load("capacities.json")
    for name, v in g.items():
        c = CONFIGS[name]
        S = c.S if 0 < c.S < c.T else c.T
        assert O.capacity(c.cf, S, c.K, c.E) == v["cap_full_subseq"]
        assert O.padded_capacity(c.T, c.S, c.K, c.E, c.cf) == v["padded_rows_per_expert"]


@pytest.mark.gpu
def test_gpu_routing_matches_fixture():
    from tests.gpu_util import dev, empty, host, lib, torch
    L = lib()
    g = _load("routing_tiny.json")
    cfg = _routing_cfg(g)
    logits = _f32(g["logits_f32_hex"]).reshape(cfg.T, cfg.E)
    s = L.shape_of(cfg)
    ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
    o = dict(topk_idx=empty((cfg.T, cfg.K), torch.int32), topk_prob=empty((cfg.T, cfg.K), torch.float32),
             topk_w=empty((cfg.T, cfg.K), torch.float32), keep=empty((cfg.T, cfg.K), torch.uint8))
    L.moe_route_topk(s, dev(logits), o["topk_idx"], o["topk_prob"], o["topk_w"], o["keep"], ws)
    rc, info = L.moe_get_status(ws)
    assert rc == 0, (rc, hex(info))
    assert host(o["topk_idx"]).ravel().tolist() == g["topk_idx"]
    assert np.array_equal(host(o["topk_prob"]).view(np.uint32).ravel(), _f32(g["topk_prob_f32_hex"]).view(np.uint32))
    assert np.array_equal(host(o["topk_w"]).view(np.uint32).ravel(), _f32(g["topk_w_f32_hex"]).view(np.uint32))
    assert host(o["keep"]).ravel().tolist() == g["keep"]
