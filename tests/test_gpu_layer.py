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


@pytest.mark.parametrize("name", ["qwen2_57b_a14b@small", "mixtral_8x22b_g8t8@small"])
def test_layer_deterministic(name):
    lib()
    cfg = get_config(name)
    inp = make_inputs(cfg, need_backward=True)
    layer = _layer(cfg, inp, True)
    x, dout = dev(inp["x"]), dev(inp["dout"])
    runs = []
    for _ in range(2):
        out = layer.forward(x).clone()
        g = {k: v.clone() for k, v in layer.backward(dout).items()}
        runs.append((out, g))
    assert torch.equal(runs[0][0], runs[1][0])
    for k in runs[0][1]:
        assert torch.equal(runs[0][1][k], runs[1][1][k]), k
