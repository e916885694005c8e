"""GShard-style padded layout (moe_permute_padded) on the GPU: the fixed
[E, C] map, counts, offsets and copied rows bit-exact against the oracle's
padded map (padding rows zero, src_of -1), on the drop workloads' routing and
on edge cases (one expert taking every kept slot, everything dropped, a
capacity above the sub-sequence length, a ragged last sub-sequence); and the
whole layer with the padded layout, forward and backward, against the
oracle layer (the layout changes where rows live, not what is computed)."""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs
from tests.gpu_util import act_dtype, assert_close, bf16_bits, dev, empty, host, inputs, lib, torch

pytestmark = pytest.mark.gpu


def _check_padded(L, cfg, x, idx, keep):
    T, K, d, E = cfg.T, cfg.K, cfg.d, cfg.E
    s = L.shape_of(cfg)
    C = L.moe_padded_capacity(s)
    assert C == O.padded_capacity(T, cfg.S, K, E, cfg.cf)
    ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
    o = dict(Xp=torch.full((E * C, d), 7.0, dtype=act_dtype(cfg), device="cuda"),
             row_of=empty((T, K), torch.int32), src_of=torch.full((E * C,), 7, dtype=torch.int32,
                                                                  device="cuda"),
             counts=empty((E,), torch.int32), offsets=empty((E + 1,), torch.int32))
    L.moe_permute_padded(s, dev(x), dev(idx), dev(keep), o["Xp"], o["row_of"], o["src_of"],
                         o["counts"], o["offsets"], ws)
    rc, info = L.moe_get_status(ws)
    assert rc == 0, (rc, hex(info))
    counts, offsets, row_of, src_of = O.build_map_padded(idx, keep, E, C)
    assert np.array_equal(host(o["counts"]), counts)
    assert np.array_equal(host(o["offsets"]), offsets)
    assert np.array_equal(host(o["row_of"]), row_of)
    assert np.array_equal(host(o["src_of"]), src_of)
    Xp_ref = O.permute_padded(x, src_of, K)
    if cfg.dtype == "bf16":
        assert np.array_equal(bf16_bits(o["Xp"]), Xp_ref)
    else:
        assert np.array_equal(host(o["Xp"]), Xp_ref)


@pytest.mark.parametrize("name", ["mixtral_8x22b@small", "mixtral_8x22b_g8t8@small"])
def test_permute_padded(name):
    L = lib()
    cfg = get_config(name)
    inp = inputs(cfg, need_backward=False)
    r = O.route(cfg, inp)
    _check_padded(L, cfg, inp["x"], r["topk_idx"], r["keep"])


@pytest.mark.parametrize("case", ["one_expert", "all_dropped", "cap_above_subseq", "ragged_subseq"])
def test_permute_padded_edge_cases(case):
    L = lib()
    cfg = dataclasses.replace(get_config("mixtral_8x22b@small"), T=1000, d=256, S=256)
    rng = np.random.default_rng(5)
    idx = np.stack([rng.permutation(cfg.E)[:cfg.K] for _ in range(cfg.T)]).astype(np.int32)
    if case == "one_expert":        # expert 3 in every token's first slot, kept up to capacity
        idx[:, 0] = 3
        idx[:, 1] = np.where(idx[:, 1] == 3, 4, idx[:, 1])
        p = np.sort(rng.random((cfg.T, cfg.K)).astype(np.float32), axis=1)[:, ::-1]
        keep = O.capacity_keep(idx, p, cfg.E, cfg.cf, cfg.S)
    elif case == "all_dropped":
        keep = np.zeros((cfg.T, cfg.K), np.uint8)
    elif case == "cap_above_subseq":   # CF 8: cap = ceil(8*256*2/8) = 512 > 256 tokens
        cfg = dataclasses.replace(cfg, cf=8.0)
        keep = np.ones((cfg.T, cfg.K), np.uint8)
    else:                             # T = 1000 = 3 * 300 + 100
        cfg = dataclasses.replace(cfg, S=300)
        p = rng.random((cfg.T, cfg.K)).astype(np.float32)
        keep = O.capacity_keep(idx, p, cfg.E, cfg.cf, cfg.S)
    x = make_inputs(cfg, need_backward=False)["x"]
    _check_padded(L, cfg, x, idx, keep)


@pytest.mark.parametrize("name,etp", [("mixtral_8x22b@small", 1), ("mixtral_8x22b_g8t8@small", 1),
                                      ("mixtral_8x22b_g8t8@small", 2)])
def test_layer_padded_matches_oracle(name, etp):
    L = lib()
    from token_dispatch_expert_moe_gb300.layer import MoELayer
    cfg = dataclasses.replace(get_config(name), backward=True)
    inp = make_inputs(cfg, need_backward=True)
    w = {k: dev(v) for k, v in inp.items() if k not in ("x", "dout")}
    layer = MoELayer(cfg, w, backward=True, layout="padded", etp=etp)
    x, dout = dev(inp["x"]), dev(inp["dout"])
    for _ in range(2):   # the second step runs on padding rows the first step left behind
        out = layer.forward(x)
        g = layer.backward(dout)
    rc, info = L.moe_get_status(layer.ws)
    assert rc == 0, (rc, hex(info))
    f = O.layer_forward(cfg, inp, etp=etp)
    assert np.array_equal(host(layer.counts), f["counts"])
    assert_close("out", host(out), f["out"], cfg.dtype)
    gr = O.layer_backward(cfg, inp, f, etp=etp)
    for k in ("dx", "dW_r"):
        assert_close(k, host(g[k]), gr[k], cfg.dtype)
    if etp == 1:
        dW_gu, dW_down = g["dW_gu"], g["dW_down"]
    else:   # per-shard weight gradients back to the full layouts
        Fl = g["dW_gu"][0].shape[1] // 2
        dW_gu = torch.cat([torch.cat([s_[:, :Fl] for s_ in g["dW_gu"]], 1),
                           torch.cat([s_[:, Fl:] for s_ in g["dW_gu"]], 1)], 1)
        dW_down = torch.cat(g["dW_down"], 2)
    assert_close("dW_gu", host(dW_gu), gr["dW_gu"], cfg.dtype)
    assert_close("dW_down", host(dW_down), gr["dW_down"], cfg.dtype)
