"""The whole layer through the C ABI (MoELayer) vs the oracle layer, forward
and backward, on the reduced workloads; determinism across runs; status word
clean after every run."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs
from tests.gpu_util import SMALL, assert_close, dev, host, lib, torch

pytestmark = pytest.mark.gpu


def _layer(cfg, inp, backward):
    from token_dispatch_expert_moe_gb300.layer import MoELayer
    w = {k: dev(v) for k, v in inp.items() if k not in ("x", "dout")}
    return MoELayer(cfg, w, backward=backward)


@pytest.mark.parametrize("name", SMALL)
def test_layer_forward_backward(name):
    L = lib()
    cfg = get_config(name)
    bwd = cfg.backward or cfg.dtype == "bf16"
    inp = make_inputs(cfg, need_backward=bwd)
    layer = _layer(cfg, inp, bwd)
    x = dev(inp["x"])
    out = layer.forward(x)
    rc, info = L.moe_get_status(layer.ws)
    assert rc == 0, (rc, hex(info))
    f = O.layer_forward(cfg, inp)
    assert np.array_equal(host(layer.topk_idx), f["topk_idx"])
    assert np.array_equal(host(layer.keep), f["keep"])
    assert np.array_equal(host(layer.offsets), f["offsets"])
    assert_close("out", host(out), f["out"], cfg.dtype)
    if not bwd:
        return
    g = layer.backward(dev(inp["dout"]))
    rc, info = L.moe_get_status(layer.ws)
    assert rc == 0, (rc, hex(info))
    gr = O.layer_backward(cfg, inp, f)
    for k in ("dx", "dW_r", "dW_gu", "dW_down", "db_r", "dWs_gu", "dWs_down", "dw_sg"):
        if k in g:
            assert_close(k, host(g[k]), gr[k], cfg.dtype)


@pytest.mark.parametrize("name", SMALL)
def test_layer_deterministic(name):
    lib()
    cfg = get_config(name)
    inp = make_inputs(cfg, need_backward=True)
    bwd = cfg.backward or cfg.dtype == "bf16"
    layer = _layer(cfg, inp, bwd)
    x, dout = dev(inp["x"]), dev(inp["dout"])
    runs = []
    for _ in range(2):
        out = layer.forward(x).clone()
        g = {k: v.clone() for k, v in layer.backward(dout).items()} if bwd else {}
        runs.append((out, g))
    assert torch.equal(runs[0][0], runs[1][0])
    for k in runs[0][1]:
        assert torch.equal(runs[0][1][k], runs[1][1][k]), k


# degenerate cases of the method, through the whole layer (forward + backward)
DEGENERATE = {
    # one expert takes every token: softmax over one logit is 1, dlogits = 0
    "single_expert": ("mixtral_8x22b@small", dict(E=1, K=1, drop=False)),
    # Top-K = E: every token goes to every expert (a dense mixture)
    "all_experts": ("mixtral_8x22b_g8t8@small", dict(E=8, K=8, drop=False)),
    # a capacity of 4 per (sub-sequence, expert): most slots dropped, tokens
    # with every slot dropped output 0
    "tiny_capacity": ("mixtral_8x22b_g8t8@small", dict(cf=0.05)),
    # one token
    "single_token": ("mixtral_8x22b@small", dict(T=1, S=0)),
}


@pytest.mark.parametrize("case", sorted(DEGENERATE))
def test_layer_degenerate_cases(case):
    import dataclasses
    L = lib()
    base, kw = DEGENERATE[case]
    cfg = dataclasses.replace(get_config(base), name=f"{base}@{case}", **kw)
    inp = make_inputs(cfg, need_backward=True)
    layer = _layer(cfg, inp, True)
    out = layer.forward(dev(inp["x"]))
    g = layer.backward(dev(inp["dout"]))
    rc, info = L.moe_get_status(layer.ws)
    assert rc == 0, (rc, hex(info))
    f = O.layer_forward(cfg, inp)
    assert np.array_equal(host(layer.topk_idx), f["topk_idx"])
    assert np.array_equal(host(layer.keep), f["keep"])
    assert np.array_equal(host(layer.offsets), f["offsets"])
    assert_close("out", host(out), f["out"], cfg.dtype)
    gr = O.layer_backward(cfg, inp, f)
    for k in ("dx", "dW_r", "dW_gu", "dW_down"):
        assert_close(k, host(g[k]), gr[k], cfg.dtype)
