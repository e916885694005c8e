"""The permutation fused into the gate/up GEMM (moe_expert_ffn_gather): the
GEMM gathers permuted row R from x as x[src_of[R] / K] instead of reading
Xp. It must give exactly what moe_permute followed by moe_expert_ffn gives
(the tensor cores see the same operand bits in the same order), so A_save, H
and Yp are compared bit for bit, and against the oracle's expert FFN within
the bf16 tolerance. Cases: the routing of every bf16 workload at its reduced
size, routings with empty experts, one-row experts and one expert taking
every slot, a single token, the padded [E, C] layout (padding rows gather
zeros), map-only moe_permute (Xp = NULL) giving the same map, and the
full-size workloads (all rows bit for bit)."""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs
from tests.gpu_util import FULL, SMALL, assert_close, bf16_bits, dev, empty, host, inputs, lib, torch

pytestmark = pytest.mark.gpu


def _bits(t, n):
    return t[:n].contiguous().view(torch.int16)


def _both_paths(L, cfg, x, idx, keep, W_gu, W_down, padded=False):
    """(reference: permute + moe_expert_ffn, fused: map-only permute +
    moe_expert_ffn_gather), each a dict of device tensors, and n rows."""
    T, K, d, E, F = cfg.T, cfg.K, cfg.d, cfg.E, cfg.F
    s = L.shape_of(cfg)
    ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
    rows = E * L.moe_padded_capacity(s) if padded else T * K
    permute = L.moe_permute_padded if padded else L.moe_permute
    x_d, idx_d, keep_d = dev(x), dev(idx), dev(keep)
    out = {}
    for name in ("ref", "fused"):
        o = dict(Xp=empty((rows, d), torch.bfloat16) if name == "ref" else None,
                 row_of=empty((T, K), torch.int32),
                 src_of=torch.full((rows,), -7, dtype=torch.int32, device="cuda"),
                 counts=empty((E,), torch.int32), offsets=empty((E + 1,), torch.int32),
                 A=torch.full((rows, 2 * F), 3.0, dtype=torch.bfloat16, device="cuda"),
                 H=torch.full((rows, F), 3.0, dtype=torch.bfloat16, device="cuda"),
                 Y=torch.full((rows, d), 3.0, dtype=torch.bfloat16, device="cuda"))
        permute(s, x_d, idx_d, keep_d, o["Xp"], o["row_of"], o["src_of"], o["counts"],
                o["offsets"], ws)
        if name == "ref":
            L.moe_expert_ffn(L.MOE_BF16, rows, d, F, E, o["offsets"], o["Xp"], W_gu, W_down,
                             o["A"], o["H"], o["Y"], ws)
        else:
            L.moe_expert_ffn_gather(rows, d, F, E, o["offsets"], x_d, T, K, o["src_of"], W_gu,
                                    W_down, o["A"], o["H"], o["Y"], ws)
        out[name] = o
    rc, info = L.moe_get_status(ws)
    assert rc == 0, (rc, hex(info))
    n = int(out["ref"]["offsets"][-1].item())
    return out["ref"], out["fused"], n


def _assert_same(ref, fused, n):
    for k in ("row_of", "counts", "offsets"):
        assert torch.equal(ref[k], fused[k]), k
    assert torch.equal(ref["src_of"][:n], fused["src_of"][:n])
    for k in ("A", "H", "Y"):
        assert torch.equal(_bits(ref[k], n), _bits(fused[k], n)), k


@pytest.mark.parametrize("name", [n for n in SMALL if get_config(n).dtype == "bf16"])
def test_gather_matches_permute_then_ffn(name):
    L = lib()
    cfg = get_config(name)
    inp = inputs(cfg, need_backward=False)
    r = O.route(cfg, inp)
    W_gu, W_down = dev(inp["W_gu"]), dev(inp["W_down"])
    ref, fused, n = _both_paths(L, cfg, inp["x"], r["topk_idx"], r["keep"], W_gu, W_down)
    _assert_same(ref, fused, n)
    _, offsets, _, src_of, n_o = O.build_map(r["topk_idx"], r["keep"], cfg.E)
    assert n == n_o
    Ar, Hr, Yr = O.expert_ffn(O.permute(inp["x"], src_of, cfg.K), offsets, inp["W_gu"],
                              inp["W_down"], "bf16")
    assert_close("A_save", host(fused["A"])[:n], Ar, "bf16")
    assert_close("H", host(fused["H"])[:n], Hr, "bf16")
    assert_close("Yp", host(fused["Y"])[:n], Yr, "bf16")


def _routing(T, E, K, experts, seed, keep_frac=1.0):
    """Top-K routing whose slots use only the given experts (others empty)."""
    rng = np.random.default_rng(seed)
    ex = np.asarray(experts)
    idx = np.stack([rng.permutation(ex)[:K] for _ in range(T)]).astype(np.int32)
    keep = (rng.random((T, K)) < keep_frac).astype(np.uint8)
    return idx, keep


@pytest.mark.parametrize("case", ["two_of_eight", "one_expert", "single_token", "ragged_drop"])
def test_gather_edge_cases(case):
    L = lib()
    base = dataclasses.replace(get_config("mixtral_8x22b@small"), drop=False)
    if case == "two_of_eight":      # six empty experts, two large ones
        cfg = dataclasses.replace(base, T=700)
        idx, keep = _routing(cfg.T, cfg.E, cfg.K, [1, 6], 3)
    elif case == "one_expert":      # K = 1, every token to expert 4
        cfg = dataclasses.replace(base, T=513, K=1)
        idx, keep = np.full((cfg.T, 1), 4, np.int32), np.ones((cfg.T, 1), np.uint8)
    elif case == "single_token":
        cfg = dataclasses.replace(base, T=1)
        idx, keep = np.array([[5, 2]], np.int32), np.ones((1, 2), np.uint8)
    else:                           # a few rows per expert, some slots dropped
        cfg = dataclasses.replace(base, T=93)
        idx, keep = _routing(cfg.T, cfg.E, cfg.K, range(cfg.E), 4, keep_frac=0.8)
    inp = make_inputs(cfg, need_backward=False)
    ref, fused, n = _both_paths(L, cfg, inp["x"], idx, keep, dev(inp["W_gu"]), dev(inp["W_down"]))
    assert n == int(keep.sum())
    _assert_same(ref, fused, n)


def test_gather_padded_layout():
    L = lib()
    cfg = get_config("mixtral_8x22b_g8t8@small")
    inp = inputs(cfg, need_backward=False)
    r = O.route(cfg, inp)
    ref, fused, n = _both_paths(L, cfg, inp["x"], r["topk_idx"], r["keep"], dev(inp["W_gu"]),
                                dev(inp["W_down"]), padded=True)
    _assert_same(ref, fused, n)
    # padding rows are zero rows: H = silu(0) * 0 = 0 and Y = 0 there
    pad = host(fused["src_of"]) < 0
    assert pad.any()
    assert not host(fused["H"])[pad].any() and not host(fused["Y"])[pad].any()


@pytest.mark.parametrize("name", ["mixtral_8x22b", "mixtral_8x22b_g8t8"])
def test_gather_full_size(name):
    L = lib()
    cfg = get_config(name)
    inp = inputs(cfg, need_backward=False)
    from token_dispatch_expert_moe_gb300.layer import MoELayer
    w = {k: dev(v) for k, v in inp.items() if k not in ("x", "dout")}
    layer = MoELayer(cfg, w, backward=False)
    x = dev(inp["x"])
    layer.forward(x)   # the GPU's own routing
    idx, keep = host(layer.topk_idx), host(layer.keep)
    ref, fused, n = _both_paths(L, cfg, inp["x"], idx, keep, w["W_gu"], w["W_down"])
    _assert_same(ref, fused, n)
