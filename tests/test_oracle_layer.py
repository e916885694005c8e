"""Pins for the oracle's permute / FFN / combine / backward.

Special cases reduce the layer to a library routine (torch's SwiGLU MLP in
float64), invariants that any correct layer keeps, and central finite
differences in fp64 for every gradient."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synthetic import MoEConfig, make_inputs


def _f64_inputs(cfg, rng, with_dout=True):
    T, d, E, F = cfg.T, cfg.d, cfg.E, cfg.F
    inp = {"x": rng.standard_normal((T, d)),
           "W_r": rng.standard_normal((E, d)) * cfg.router_scale / np.sqrt(d),
           "W_gu": rng.standard_normal((E, 2 * F, d)) / np.sqrt(d),
           "W_down": rng.standard_normal((E, d, F)) / np.sqrt(F)}
    if cfg.bias:
        inp["b_r"] = rng.standard_normal(E)
    if cfg.Fs:
        inp["w_sg"] = rng.standard_normal(d) / np.sqrt(d)
        inp["Ws_gu"] = rng.standard_normal((2 * cfg.Fs, d)) / np.sqrt(d)
        inp["Ws_down"] = rng.standard_normal((d, cfg.Fs)) / np.sqrt(cfg.Fs)
    if with_dout:
        inp["dout"] = rng.standard_normal((T, d))
    return inp


def _torch_swiglu(x, Wgu, Wd):
    x, Wgu, Wd = (torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (x, Wgu, Wd))
    F = Wgu.shape[0] // 2
    h = torch.nn.functional.silu(x @ Wgu[:F].T) * (x @ Wgu[F:].T)
    return (h @ Wd.T).numpy()


@pytest.mark.parametrize("K", [2, 8])
def test_identity_experts_give_k_times_x(K):
    cfg = MoEConfig("t", T=300, d=64, E=16, K=K, F=8, dtype="bf16", drop=False)
    inp = make_inputs(cfg)
    r = O.route(cfg, inp)
    counts, offsets, row_of, src_of, n = O.build_map(r["topk_idx"], r["keep"], cfg.E)
    Xp = O.permute(inp["x"], src_of, K)
    Yp = O.decode(Xp)                        # identity experts
    out = O.unpermute(Yp, row_of, np.ones((cfg.T, K), np.float32), dtype="bf16")
    assert np.array_equal(out, K * O.decode(inp["x"]))   # exact in bf16
    # renormalised weights on identity experts give x back (dropless)
    out_w = O.unpermute(Yp, row_of, r["topk_w"], dtype="bf16")
    assert np.array_equal(out_w, O.decode(inp["x"]))


def test_identity_experts_with_drop():
    cfg = MoEConfig("t", T=300, d=32, E=8, K=2, F=8, dtype="bf16", drop=True, cf=0.7, S=100)
    inp = make_inputs(cfg)
    r = O.route(cfg, inp)
    assert 0 < r["keep"].sum() < cfg.T * cfg.K
    counts, offsets, row_of, src_of, n = O.build_map(r["topk_idx"], r["keep"], cfg.E)
    Yp = O.decode(O.permute(inp["x"], src_of, cfg.K))
    out = O.unpermute(Yp, row_of, np.ones((cfg.T, cfg.K), np.float32), dtype="bf16")
    nk = r["keep"].sum(axis=1).astype(np.float64)
    assert np.array_equal(out, O.round_bf16(nk[:, None] * O.decode(inp["x"])))


def test_single_expert_is_dense_swiglu():
    cfg = MoEConfig("t", T=64, d=32, E=1, K=1, F=48, dtype="f32", drop=False)
    inp = _f64_inputs(cfg, np.random.default_rng(0), with_dout=False)
    f = O.layer_forward(cfg, inp, mirror=False)
    ref = _torch_swiglu(inp["x"], inp["W_gu"][0], inp["W_down"][0])
    assert np.allclose(f["out"], ref, rtol=1e-12, atol=1e-12)


def test_all_experts_is_dense_mixture():
    cfg = MoEConfig("t", T=64, d=32, E=4, K=4, F=16, dtype="f32", drop=False, bias=True)
    inp = _f64_inputs(cfg, np.random.default_rng(1), with_dout=False)
    f = O.layer_forward(cfg, inp, mirror=False)
    logits = inp["x"] @ inp["W_r"].T + inp["b_r"]
    p = torch.softmax(torch.from_numpy(logits), dim=1).numpy()
    ref = sum(p[:, e:e + 1] * _torch_swiglu(inp["x"], inp["W_gu"][e], inp["W_down"][e])
              for e in range(cfg.E))
    assert np.allclose(f["out"], ref, rtol=1e-12, atol=1e-12)


def test_shared_expert_adds_gated_dense_ffn():
    cfg = MoEConfig("t", T=40, d=16, E=4, K=1, F=8, dtype="f32", drop=False, Fs=24)
    inp = _f64_inputs(cfg, np.random.default_rng(2), with_dout=False)
    f = O.layer_forward(cfg, inp, mirror=False)
    base = dataclasses.replace(cfg, Fs=0)
    f0 = O.layer_forward(base, inp, mirror=False)
    gate = torch.sigmoid(torch.from_numpy(inp["x"] @ inp["w_sg"])).numpy()[:, None]
    ref = f0["out"] + gate * _torch_swiglu(inp["x"], inp["Ws_gu"], inp["Ws_down"])
    assert np.allclose(f["out"], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("drop", [False, True])
def test_expert_relabelling_invariance(drop):
    cfg = MoEConfig("t", T=96, d=16, E=6, K=2, F=8, dtype="f32", drop=drop, cf=0.8, S=32,
                    bias=True)
    inp = _f64_inputs(cfg, np.random.default_rng(3), with_dout=False)
    sigma = np.array([3, 0, 5, 1, 4, 2])
    inp2 = dict(inp, W_r=inp["W_r"][sigma], b_r=inp["b_r"][sigma],
                W_gu=inp["W_gu"][sigma], W_down=inp["W_down"][sigma])
    a = O.layer_forward(cfg, inp, mirror=False)["out"]
    b = O.layer_forward(cfg, inp2, mirror=False)["out"]
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("drop", [False, True])
def test_token_permutation_equivariance(drop):
    cfg = MoEConfig("t", T=96, d=16, E=4, K=2, F=8, dtype="f32", drop=drop, cf=0.8, S=32)
    inp = _f64_inputs(cfg, np.random.default_rng(4), with_dout=False)
    rng = np.random.default_rng(9)
    perm = np.concatenate([lo + rng.permutation(32) for lo in range(0, 96, 32)])
    a = O.layer_forward(cfg, inp, mirror=False)["out"]
    b = O.layer_forward(cfg, dict(inp, x=inp["x"][perm]), mirror=False)["out"]
    assert np.allclose(a[perm], b, rtol=1e-13, atol=1e-13)


def _loss(cfg, inp):
    return float((O.layer_forward(cfg, inp, mirror=False)["out"] * inp["dout"]).sum())


def _margins_ok(cfg, inp):
    """Routing must be locally constant for finite differences: a clear gap
    between the K-th and (K+1)-th probability, and between kept and dropped
    capacity keys."""
    r = O.route(cfg, inp, mirror=False)
    ps = -np.sort(-r["p"], axis=1)
    if cfg.K < cfg.E and (ps[:, cfg.K - 1] - ps[:, cfg.K]).min() < 1e-3:
        return False
    if cfg.drop:
        S = cfg.subseq
        for lo in range(0, cfg.T, S):
            sub = slice(lo, min(cfg.T, lo + S))
            for e in range(cfg.E):
                m = r["topk_idx"][sub] == e
                kp = r["topk_prob"][sub][m & (r["keep"][sub] == 1)]
                dp = r["topk_prob"][sub][m & (r["keep"][sub] == 0)]
                if dp.size and kp.size and kp.min() - dp.max() < 1e-3:
                    return False
    return True


@pytest.mark.parametrize("variant", ["dropless_shared_bias", "drop_renorm", "no_renorm"])
def test_backward_matches_finite_differences(variant):
    if variant == "dropless_shared_bias":
        cfg = MoEConfig("fd", T=12, d=8, E=4, K=2, F=6, dtype="f32", drop=False,
                        Fs=5, bias=True)
    elif variant == "drop_renorm":
        cfg = MoEConfig("fd", T=16, d=8, E=4, K=2, F=6, dtype="f32", drop=True, cf=0.5, S=8)
    else:
        cfg = MoEConfig("fd", T=12, d=8, E=4, K=2, F=6, dtype="f32", drop=False, renorm=False)
    for seed in range(200):
        inp = _f64_inputs(cfg, np.random.default_rng(seed))
        if _margins_ok(cfg, inp):
            break
    else:
        pytest.fail("no input with clear routing margins")
    f = O.layer_forward(cfg, inp, mirror=False)
    if cfg.drop:
        assert 0 < f["keep"].sum() < cfg.T * cfg.K
    g = O.layer_backward(cfg, inp, f, mirror=False)
    names = {"x": "dx", "W_r": "dW_r", "W_gu": "dW_gu", "W_down": "dW_down"}
    if cfg.bias:
        names["b_r"] = "db_r"
    if cfg.Fs:
        names.update(w_sg="dw_sg", Ws_gu="dWs_gu", Ws_down="dWs_down")
    rng = np.random.default_rng(123)
    h = 1e-6
    for pname, gname in names.items():
        arr = inp[pname]
        flat_idx = rng.choice(arr.size, size=min(arr.size, 12), replace=False)
        for fi in flat_idx:
            i = np.unravel_index(fi, arr.shape)
            old = arr[i]
            arr[i] = old + h
            lp = _loss(cfg, inp)
            arr[i] = old - h
            lm = _loss(cfg, inp)
            arr[i] = old
            num = (lp - lm) / (2 * h)
            ana = g[gname][i]
            assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), (pname, i, num, ana)


# ---- expert F-split over an expert-tensor-parallel group (f4) ----

@pytest.mark.parametrize("shards", [2, 3])
def test_fsplit_is_the_unsplit_ffn_in_exact_arithmetic(shards):
    """Without rounding (fp64), the F-split FFN equals the unsplit one: the
    down projection is linear in the hidden units, and SwiGLU acts per unit.
    A wrong gate/up row pairing or W_down column choice breaks this."""
    rng = np.random.default_rng(7)
    E, n, d, F = 3, 40, 10, 12
    Xp = rng.standard_normal((n, d))
    offsets = np.array([0, 17, 17, 40], dtype=np.int32)
    W_gu = rng.standard_normal((E, 2 * F, d)) / np.sqrt(d)
    W_down = rng.standard_normal((E, d, F)) / np.sqrt(F)
    A, H, Y = O.expert_ffn(Xp, offsets, W_gu, W_down, "f32", mirror=False)
    As, Hs, Ys = O.expert_ffn_fsplit(Xp, offsets, W_gu, W_down, shards, "f32", mirror=False)
    assert np.array_equal(As, A) and np.array_equal(Hs, H)
    assert np.abs(Ys - Y).max() <= 1e-12 * np.abs(Y).max()
    dYp = rng.standard_normal((n, d))
    dX, dWgu, dWd, dA = O.expert_ffn_bwd(dYp, Xp, A, H, offsets, W_gu, W_down, "f32", mirror=False)
    sX, sWgu, sWd, sA = O.expert_ffn_bwd_fsplit(dYp, Xp, A, H, offsets, W_gu, W_down, shards,
                                                "f32", mirror=False)
    assert np.array_equal(sA, dA) and np.array_equal(sWgu, dWgu) and np.array_equal(sWd, dWd)
    assert np.abs(sX - dX).max() <= 1e-12 * np.abs(dX).max()


def test_fsplit_one_shard_is_expert_ffn():
    rng = np.random.default_rng(8)
    Xp = rng.standard_normal((20, 8)).astype(np.float32)
    offsets = np.array([0, 9, 20], dtype=np.int32)
    W_gu = (rng.standard_normal((2, 12, 8)) / 3).astype(np.float32)
    W_down = (rng.standard_normal((2, 8, 6)) / 3).astype(np.float32)
    a = O.expert_ffn(Xp, offsets, W_gu, W_down, "bf16")
    b = O.expert_ffn_fsplit(Xp, offsets, W_gu, W_down, 1, "bf16")
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_sum_partials_adds_in_shard_order_in_fp32():
    """(a + b) + c differs from a + (b + c) in fp32 here: the oracle must take
    the shard order with an fp32 rounding after every addition."""
    a, b, c = np.float64(1.0), np.float64(2.0 ** -24), np.float64(2.0 ** -24)
    left = O.sum_partials([np.array([a]), np.array([b]), np.array([c])])
    assert left[0] == 1.0                         # each tiny addend is rounded away
    right = O.sum_partials([np.array([b]), np.array([c]), np.array([a])])
    assert right[0] == 1.0 + 2.0 ** -23           # the two tiny addends first survive
    assert O.sum_partials([np.array([a]), np.array([b])], mirror=False)[0] == 1.0 + 2.0 ** -24
