"""The parity tolerances separate rounding from mistakes (CPU, oracle only).

Not too tight: an F-split of the experts (partial outputs rounded to bf16 and
added in fp32, a different set of rounding points than the unsplit layer, and a
larger perturbation than a change of fp32 summation order on the GPU) stays
within them. Not vacuous: mistakes of the size a wrong kernel makes (an
expert's rows lost, two tokens' rows exchanged, a combine weight off by 2 %, the
shared expert missing, one expert's weight gradient lost) fall outside them, at
the reduced sizes the GPU parity tests use."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs
from tests.gpu_util import assert_close


def _fails(name, got, ref, dtype):
    with pytest.raises(AssertionError):
        assert_close(name, got, ref, dtype)


@pytest.mark.parametrize("name", ["mixtral_8x22b@small", "qwen2_57b_a14b@small",
                                  "mixtral_8x22b_g8t8@small"])
def test_tolerance_passes_rounding_and_fails_mistakes(name):
    cfg = get_config(name)
    inp = make_inputs(cfg, need_backward=True)
    f = O.layer_forward(cfg, inp)
    out = f["out"]
    # a different set of rounding points passes
    fs = O.layer_forward(cfg, inp, etp=2)
    assert not np.array_equal(fs["out"], out)
    assert_close("out (F-split)", fs["out"], out, cfg.dtype)
    # an expert's rows lost
    Yp = f["Yp"].copy()
    e = int(np.argmax(np.diff(f["offsets"])))
    Yp[f["offsets"][e]:f["offsets"][e + 1]] = 0.0
    Ys, z = f.get("Ys"), f.get("gate_logit")
    _fails("out (expert lost)", O.unpermute(Yp, f["row_of"], f["topk_w"], Ys, z, cfg.dtype),
           out, cfg.dtype)
    # two tokens' rows exchanged
    sw = out.copy()
    sw[[3, 700]] = sw[[700, 3]]
    _fails("out (tokens exchanged)", sw, out, cfg.dtype)
    # the first slot's combine weight off by 2 %
    w = np.array(f["topk_w"], dtype=np.float64)
    w[:, 0] *= 1.02
    _fails("out (weight 2 %)", O.unpermute(f["Yp"], f["row_of"], w, Ys, z, cfg.dtype),
           out, cfg.dtype)
    if cfg.Fs:   # the shared expert missing
        _fails("out (no shared expert)", O.unpermute(f["Yp"], f["row_of"], f["topk_w"],
                                                     dtype=cfg.dtype), out, cfg.dtype)
    if not cfg.backward:
        return
    g = O.layer_backward(cfg, inp, f)
    gs = O.layer_backward(cfg, inp, fs, etp=2)
    assert_close("dx (F-split)", gs["dx"], g["dx"], cfg.dtype)
    dW = g["dW_gu"].copy()
    dW[e] = 0.0
    _fails("dW_gu (expert lost)", dW, g["dW_gu"], cfg.dtype)
