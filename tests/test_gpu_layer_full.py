"""The whole layer at the workloads' full sizes, through the C ABI in the
launch configuration the benchmark times (MoELayer), checked on outputs the
oracle can compute one by one:

- routing: the GPU's decisions agree with the oracle's on >= 99.9 % of tokens
  (the rest are near ties of the fp32 logits; decisions from identical logits
  are compared bit for bit elsewhere);
- out[t] and dx[t] for 16 sampled tokens (routing agreed), each recomputed by
  the oracle from that token's own rows;
- dW_down[e][:, j] and dW_gu[e][j | F+j, :] for 3 sampled experts and 8
  hidden units j: the SwiGLU FFN separates over hidden units, so the
  oracle's own group functions run on a sub-expert made of the sampled units
  over all of the expert's rows;
- the router backward, element by element over every token: dW_r, db_r,
  dw_sg and dx_router against the oracle's router backward fed the GPU's own
  logits, Top-K outputs, combine-weight gradient dw and gate gradient dz.
  The router runs in fp32 arithmetic on identical inputs, so besides the
  layer's bf16 tolerance its error is held to an fp32 accumulation bound,
  rel-Frobenius <= max(1e-5, 10 * 2^-24 * sqrt(T)).
"""
import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config
from tests.gpu_util import FULL, assert_close, dev, host, inputs, lib, torch

pytestmark = pytest.mark.gpu


def _run_layer(cfg, inp):
    from token_dispatch_expert_moe_gb300.layer import MoELayer
    w = {k: dev(v) for k, v in inp.items() if k not in ("x", "dout")}
    layer = MoELayer(cfg, w, backward=cfg.backward)
    out = layer.forward(dev(inp["x"]))
    g = layer.backward(dev(inp["dout"])) if cfg.backward else None
    return layer, out, g


@pytest.mark.parametrize("name", FULL)
def test_layer_full_size_sampled(name):
    L = lib()
    cfg = get_config(name)
    inp = inputs(cfg, need_backward=cfg.backward)
    layer, out, g = _run_layer(cfg, inp)
    rc, info = L.moe_get_status(layer.ws)
    assert rc == 0, (rc, hex(info))
    T, K, E, F = cfg.T, cfg.K, cfg.E, cfg.F
    rnd = O.act_rounder(cfg.dtype, True)
    r32 = O.f32_rounder(True)

    # routing decisions
    r = O.route(cfg, inp)
    gi, gk = host(layer.topk_idx), host(layer.keep)
    agree = np.all(gi == r["topk_idx"], axis=1) & np.all(gk == r["keep"], axis=1)
    assert agree.mean() >= 0.999, agree.mean()

    rng = np.random.default_rng(1)
    toks = np.sort(rng.choice(np.nonzero(agree)[0], size=16, replace=False))
    # forward and backward rows of every sampled (token, slot), one expert at a time
    fwd_rows, bwd_rows = {}, {}
    needed = sorted({int(r["topk_idx"][t, k]) for t in toks for k in range(K) if r["keep"][t, k]})
    for e in needed:
        Wgu, Wd = O.decode(inp["W_gu"][e]), O.decode(inp["W_down"][e])
        for t in toks:
            for k in range(K):
                if r["keep"][t, k] and r["topk_idx"][t, k] == e:
                    X = O.decode(inp["x"][t:t + 1])
                    A_r, H_r, Y_r = O.swiglu_group(X, Wgu, Wd, rnd)
                    fwd_rows[(t, k)] = (A_r, H_r, Y_r)
                    if g is not None:   # dYp of this slot needs only w and dout
                        ub = O.unpermute_bwd(inp["dout"][t:t + 1], Y_r,
                                             np.array([[0]], np.int32), r["topk_w"][t:t + 1, k:k + 1],
                                             dtype=cfg.dtype)
                        bwd_rows[(t, k)] = O.swiglu_group_bwd(ub["dYp"], X, A_r, H_r, Wgu, Wd,
                                                              rnd, r32)[0][0]
        del Wgu, Wd
    shared = None
    if cfg.Fs:
        shared = (O.decode(inp["Ws_gu"]), O.decode(inp["Ws_down"]))
    out_h = host(out)
    dx_h = host(g["dx"]) if g is not None else None
    for t in toks:
        x_t = inp["x"][t:t + 1]
        X = O.decode(x_t)
        kept = [k for k in range(K) if r["keep"][t, k]]
        row_of_t = np.full((1, K), -1, np.int32)
        for i, k in enumerate(kept):
            row_of_t[0, k] = i
        Yp_t = (np.concatenate([fwd_rows[(t, k)][2] for k in kept]) if kept
                else np.zeros((0, cfg.d)))
        Ys_t = z_t = None
        if shared is not None:
            As_t, Hs_t, Ys_t = O.swiglu_group(X, shared[0], shared[1], rnd)
            z_t = O.gate_logit(x_t, inp["w_sg"])
        ref = O.unpermute(Yp_t, row_of_t, r["topk_w"][t:t + 1], Ys_t, z_t, cfg.dtype)
        assert_close(f"out[{t}]", out_h[t:t + 1], ref, cfg.dtype)
        if g is None:
            continue
        ub = O.unpermute_bwd(inp["dout"][t:t + 1], Yp_t, row_of_t, r["topk_w"][t:t + 1], Ys_t,
                             z_t, cfg.dtype)
        dXp_t = (np.stack([bwd_rows[(t, k)] for k in kept]) if kept else np.zeros((0, cfg.d)))
        dx_add = None
        if shared is not None:
            dx_add = O.swiglu_group_bwd(ub["dYs"], X, As_t, Hs_t, shared[0], shared[1], rnd, r32)[0]
        rb = O.route_bwd(x_t, inp["W_r"], r["p"][t:t + 1], r["topk_idx"][t:t + 1],
                         r["topk_prob"][t:t + 1], r["topk_w"][t:t + 1], ub["dw"], cfg.renorm,
                         inp.get("w_sg"), ub.get("dz"))
        dx_add = rb["dx_router"] if dx_add is None else dx_add + rb["dx_router"]
        ref_dx = O.permute_bwd(dXp_t, row_of_t, dx_add)
        assert_close(f"dx[{t}]", dx_h[t:t + 1], ref_dx, cfg.dtype)

    if g is None:
        return
    # weight gradients of sampled experts whose rows match the oracle's exactly
    counts, offsets, row_of, src_of, n_kept = O.build_map(r["topk_idx"], r["keep"], E)
    g_src = host(layer.src_of)
    g_off = host(layer.offsets)
    same = [e for e in range(E) if offsets[e + 1] > offsets[e]
            and np.array_equal(g_src[g_off[e]:g_off[e + 1]], src_of[offsets[e]:offsets[e + 1]])]
    assert len(same) >= min(2, E)
    dWd_h, dWgu_h = g["dW_down"], g["dW_gu"]
    for e in rng.choice(same, size=min(3, len(same)), replace=False):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        t_r, k_r = src_of[lo:hi] // K, src_of[lo:hi] % K
        Xp_e = O.decode(inp["x"][t_r])
        row_of_e = np.full((T, K), -1, np.int32)
        row_of_e[t_r, k_r] = np.arange(hi - lo, dtype=np.int32)
        dYp_e = O.unpermute_bwd(inp["dout"], np.zeros((hi - lo, cfg.d)), row_of_e,
                                r["topk_w"], dtype=cfg.dtype)["dYp"]
        js = np.sort(rng.choice(F, size=8, replace=False))
        Wgu_sub = O.decode(np.concatenate([inp["W_gu"][e][js], inp["W_gu"][e][F + js]]))
        Wd_sub = O.decode(inp["W_down"][e][:, js])
        A_s, H_s, _ = O.swiglu_group(Xp_e, Wgu_sub, Wd_sub, rnd)
        _, dWd_ref, dWgu_ref, _ = O.swiglu_group_bwd(dYp_e, Xp_e, A_s, H_s, Wgu_sub, Wd_sub, rnd, r32)
        got_dWd = dWd_h[int(e)][:, torch.as_tensor(js, device="cuda")].cpu().numpy()
        assert_close(f"dW_down[{e}][:, js]", got_dWd, dWd_ref, cfg.dtype)
        sel = torch.as_tensor(np.concatenate([js, F + js]), device="cuda")
        got_dWgu = dWgu_h[int(e)][sel].cpu().numpy()
        assert_close(f"dW_gu[{e}][js]", got_dWgu, dWgu_ref, cfg.dtype)

    # router backward over every token, fed the GPU's own routing and gradients
    p = O.softmax_f32(host(layer.logits).astype(np.float32))
    sh = cfg.Fs > 0
    rb = O.route_bwd(inp["x"], inp["W_r"], p, host(layer.topk_idx), host(layer.topk_prob),
                     host(layer.topk_w), host(layer.dw), cfg.renorm, inp.get("w_sg"),
                     host(layer.dz) if sh else None)
    fp32_bound = max(1e-5, 10 * 2.0 ** -24 * np.sqrt(T))
    checks = [("dW_r", g["dW_r"], rb["dW_r"])]
    if "db_r" in g:
        checks.append(("db_r", g["db_r"], rb["db_r"]))
    if sh:
        checks.append(("dw_sg", g["dw_sg"], rb["dw_sg"]))
    dx_in = host(layer.dXs).astype(np.float64) if sh else 0.0   # the call's own addend
    checks.append(("dx_router", layer.dx_router, rb["dx_router"] + dx_in))
    for nm, got, ref in checks:
        rf, _ = assert_close(nm, host(got), ref, cfg.dtype)
        assert rf <= fp32_bound, (nm, rf, fp32_bound)
