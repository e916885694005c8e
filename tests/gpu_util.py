"""Helpers of the GPU parity tests: device transfer, tolerances, configs.

Tolerances: bf16 layers, relative Frobenius error <= 5e-3 and max-abs <= 3e-2
on outputs and gradients, the max-abs bound scaled by max(1, RMS of the
reference): gradients that sum over thousands of tokens (dW_r, dW_gu, dW_down
reach 1e2..1e3) carry the bf16 rounding noise of the activations they are
built from in proportion to their size, so a fixed 3e-2 only has meaning at
unit scale, where the scaled and the fixed bounds coincide; fp32 layers, relative Frobenius <= 1e-5 and max-abs
<= 1e-5 * max(1, max|ref|) (fp32 accumulation over the reduction depths used
here keeps the error a few ulp of the largest value); router logits,
relative Frobenius <= 1e-5; every index, mask, map and count bit-exact.
Stored bf16 intermediates (A = [G|U], H, Yp, dA) are checked with the same
relative Frobenius bound and a per-element bound of max(3e-2, one bf16 ulp of
the reference): an fp32 accumulator and an fp64 value that straddle a bf16
rounding boundary round one ulp apart, and above |v| = 4 one ulp exceeds 3e-2.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

SMALL = ["tiny_f32", "mixtral_8x22b@small", "qwen2_57b_a14b@small",
         "mixtral_8x22b_g8t8@small", "llama3_8x70b@small"]
FULL = ["mixtral_8x22b", "qwen2_57b_a14b", "mixtral_8x22b_g8t8", "llama3_8x70b"]


_INPUT_CACHE = {}


def inputs(cfg, need_backward=None):
    """make_inputs with a one-entry cache (full-size weights take seconds)."""
    key = (cfg, need_backward)
    if key not in _INPUT_CACHE:
        _INPUT_CACHE.clear()
        from synthetic import make_inputs
        _INPUT_CACHE[key] = make_inputs(cfg, need_backward=need_backward)
    return _INPUT_CACHE[key]


def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_dispatch_expert_moe_gb300 import _lib
    return _lib


def dev(a: np.ndarray) -> "torch.Tensor":
    from token_dispatch_expert_moe_gb300.layer import to_device
    return to_device(a)


def host(t: "torch.Tensor") -> np.ndarray:
    t = t.detach()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    return t.cpu().numpy()


def bf16_bits(t: "torch.Tensor") -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def empty(shape, dtype):
    return torch.empty(shape, dtype=dtype, device="cuda")


def act_dtype(cfg):
    return torch.bfloat16 if cfg.dtype == "bf16" else torch.float32


def rel_frob(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


def bf16_ulp(v):
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0**-126)))
    return 2.0 ** (e - 7)


def assert_close(name, got, ref, dtype, kind="output"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    rf = rel_frob(got, ref)
    ma = float(np.abs(got - ref).max()) if got.size else 0.0
    mref = float(np.abs(ref).max()) if ref.size else 0.0
    if dtype == "bf16" and kind == "act":
        ok = rf <= 5e-3 and bool(np.all(np.abs(got - ref) <= np.maximum(3e-2, bf16_ulp(ref))))
    elif dtype == "bf16":
        rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
        ok = rf <= 5e-3 and ma <= 3e-2 * max(1.0, rms)
    else:
        ok = rf <= 1e-5 and ma <= 1e-5 * max(1.0, mref)
    assert ok, f"{name}: rel_frob {rf:.3e} max_abs {ma:.3e} (max|ref| {mref:.3g}, {dtype})"
    return rf, ma
