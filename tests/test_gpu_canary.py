"""Guard canaries around every device buffer the layer holds (workspace,
routing outputs, permuted buffers, activations, gradients): each buffer is
placed between two 4 KB guards filled with a byte pattern, the layer runs
forward and backward, and the guards must be intact. An out-of-bounds write by
any kernel into its neighbour's memory shows up here even when the result
happens to stay within tolerance. The guarded run is also checked against the
oracle, so the test sees real work."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs
from tests.gpu_util import assert_close, dev, host, lib, torch

pytestmark = pytest.mark.gpu

GUARD = 4096      # bytes on each side (keeps every buffer 256-byte aligned)
PATTERN = 0xA5


def _guard_buffers(layer):
    bases = {}
    for name, t in list(vars(layer).items()):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.numel() == 0:
            continue
        nbytes = t.numel() * t.element_size()
        base = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=t.device)
        body = base[GUARD:GUARD + nbytes]
        body.copy_(t.contiguous().reshape(-1).view(torch.uint8))
        setattr(layer, name, body.view(t.dtype).view(t.shape))
        bases[name] = base
    return bases


@pytest.mark.parametrize("name,layout", [("qwen2_57b_a14b@small", "compact"),
                                         ("mixtral_8x22b_g8t8@small", "compact"),
                                         ("mixtral_8x22b_g8t8@small", "padded")])
def test_no_write_outside_any_buffer(name, layout):
    from token_dispatch_expert_moe_gb300.layer import MoELayer
    L = lib()
    cfg = get_config(name)
    inp = make_inputs(cfg, need_backward=True)
    w = {k: dev(v) for k, v in inp.items() if k not in ("x", "dout")}
    layer = MoELayer(cfg, w, backward=True, layout=layout)
    bases = _guard_buffers(layer)
    assert {"ws", "Xp", "Yp", "out", "dXp", "dW_gu", "dW_r", "dx"} <= set(bases)
    out = layer.forward(dev(inp["x"]))
    g = layer.backward(dev(inp["dout"]))
    rc, info = L.moe_get_status(layer.ws)
    assert rc == 0, (rc, hex(info))
    torch.cuda.synchronize()
    for buf, base in bases.items():
        assert bool((base[:GUARD] == PATTERN).all()), f"write below {buf}"
        assert bool((base[-GUARD:] == PATTERN).all()), f"write past the end of {buf}"
    f = O.layer_forward(cfg, inp)
    assert_close("out", host(out), f["out"], cfg.dtype)
    gr = O.layer_backward(cfg, inp, f)
    assert_close("dx", host(g["dx"]), gr["dx"], cfg.dtype)
