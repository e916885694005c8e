"""Expert-tensor-parallel F-split on one GPU: moe_sum_partials bit for bit
against an fp32 in-order sum on the host, and MoELayer(etp=2/4) forward and
backward against the oracle layer with the same F-split (each shard's partial
output stored in the activation dtype, the partials added in shard order in
fp32, as a ReduceScatter-V of partials would)."""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs
from synthetic.gen import normal_bf16, normal_f32
from tests.gpu_util import assert_close, dev, host, lib, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n_parts", [1, 2, 3])
def test_sum_partials_bit_exact(dtype, n_parts):
    L = lib()
    rows, d = 1037, 264
    gen = normal_bf16 if dtype == "bf16" else normal_f32
    parts = gen(31, 1, (n_parts, rows, d))
    acc = O.decode(parts[0]).astype(np.float32)
    for p in range(1, n_parts):
        acc = (acc + O.decode(parts[p]).astype(np.float32)).astype(np.float32)
    code = L.MOE_BF16 if dtype == "bf16" else L.MOE_F32
    out = torch.empty((rows, d), dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                      device="cuda")
    L.moe_sum_partials(code, n_parts, rows, d, dev(parts), out)
    torch.cuda.synchronize()
    if dtype == "bf16":   # bf16 values are exact in fp32: compare them there
        ref = O.round_bf16(acc.astype(np.float64)).astype(np.float32)
        assert np.array_equal(host(out).view(np.uint32), ref.view(np.uint32))
    else:
        assert np.array_equal(host(out).view(np.uint32), acc.view(np.uint32))


def _full_grads(g, etp):
    """Per-shard weight gradients -> the full [E,2F,d] and [E,d,F] layouts."""
    gu, dn = g["dW_gu"], g["dW_down"]
    Fl = gu[0].shape[1] // 2
    dW_gu = torch.cat([torch.cat([s[:, :Fl] for s in gu], 1), torch.cat([s[:, Fl:] for s in gu], 1)], 1)
    dW_down = torch.cat(dn, 2)
    return dW_gu, dW_down


@pytest.mark.parametrize("name,etp", [("mixtral_8x22b_g8t8@small", 2), ("qwen2_57b_a14b@small", 2),
                                      ("tiny_f32", 2), ("tiny_f32", 4)])
def test_layer_etp_matches_oracle(name, etp):
    L = lib()
    from token_dispatch_expert_moe_gb300.layer import MoELayer
    cfg = dataclasses.replace(get_config(name), backward=True)
    inp = make_inputs(cfg, need_backward=True)
    w = {k: dev(v) for k, v in inp.items() if k not in ("x", "dout")}
    layer = MoELayer(cfg, w, backward=True, etp=etp)
    out = layer.forward(dev(inp["x"]))
    g = layer.backward(dev(inp["dout"]))
    rc, info = L.moe_get_status(layer.ws)
    assert rc == 0, (rc, hex(info))
    f = O.layer_forward(cfg, inp, etp=etp)
    assert np.array_equal(host(layer.offsets), f["offsets"])
    assert_close("out", host(out), f["out"], cfg.dtype)
    gr = O.layer_backward(cfg, inp, f, etp=etp)
    dW_gu, dW_down = _full_grads(g, etp)
    assert_close("dW_gu", host(dW_gu), gr["dW_gu"], cfg.dtype)
    assert_close("dW_down", host(dW_down), gr["dW_down"], cfg.dtype)
    for k in ("dx", "dW_r", "db_r", "dWs_gu", "dWs_down", "dw_sg"):
        if k in g:
            assert_close(k, host(g[k]), gr[k], cfg.dtype)
