"""GPU permutation map, permute and un-permute/combine vs oracle, on the
oracle's routing decisions: maps, counts and copied rows bit-exact; combined
outputs within tolerance. Edge cases: everything dropped, one expert taking
every token, empty experts, ragged token blocks, a single token."""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs
from tests.gpu_util import inputs, FULL, SMALL, act_dtype, assert_close, bf16_bits, dev, empty, host, lib, torch

pytestmark = pytest.mark.gpu


def _permute_gpu(L, cfg, x, idx, keep):
    T, K, d, E = cfg.T, cfg.K, cfg.d, cfg.E
    s = L.shape_of(cfg)
    ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
    o = dict(Xp=empty((T * K, d), act_dtype(cfg)), row_of=empty((T, K), torch.int32),
             src_of=empty((T * K,), torch.int32), counts=empty((E,), torch.int32),
             offsets=empty((E + 1,), torch.int32))
    L.moe_permute(s, dev(x), dev(idx), dev(keep), o["Xp"], o["row_of"], o["src_of"], o["counts"],
                  o["offsets"], ws)
    rc, info = L.moe_get_status(ws)
    assert rc == 0, (rc, hex(info))
    return o


def _check_permute(L, cfg, x, idx, keep):
    o = _permute_gpu(L, cfg, x, idx, keep)
    counts, offsets, row_of, src_of, n = O.build_map(idx, keep, cfg.E)
    assert np.array_equal(host(o["counts"]), counts)
    assert np.array_equal(host(o["offsets"]), offsets)
    assert np.array_equal(host(o["row_of"]), row_of)
    assert np.array_equal(host(o["src_of"])[:n], src_of)
    Xp_ref = O.permute(x, src_of, cfg.K)
    if cfg.dtype == "bf16":
        assert np.array_equal(bf16_bits(o["Xp"][:n]), Xp_ref)
    else:
        assert np.array_equal(host(o["Xp"][:n]), Xp_ref)
    return o, n


@pytest.mark.parametrize("name", SMALL + FULL)
def test_permute(name):
    L = lib()
    cfg = get_config(name)
    inp = inputs(cfg, need_backward=False)
    r = O.route(cfg, inp)
    _check_permute(L, cfg, inp["x"], r["topk_idx"], r["keep"])


@pytest.mark.parametrize("case", ["all_dropped", "one_expert", "empty_experts", "ragged_T", "T1"])
def test_permute_edge_cases(case):
    L = lib()
    base = dataclasses.replace(get_config("mixtral_8x22b@small"), T=1000, d=256)
    rng = np.random.default_rng(3)
    cfg = base
    if case == "T1":
        cfg = dataclasses.replace(base, T=1)
    if case == "ragged_T":
        cfg = dataclasses.replace(base, T=257)
    inp = inputs(cfg, need_backward=False)
    T, K, E = cfg.T, cfg.K, cfg.E
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    keep = (rng.random((T, K)) < 0.8).astype(np.uint8)
    if case == "all_dropped":
        keep[:] = 0
    if case == "one_expert":
        idx[:, 0], idx[:, 1] = 3, 5
        keep[:] = 1
    if case == "empty_experts":
        idx = np.where(idx % 3 == 0, (idx + 1) % E, idx)
        for t in range(T):   # keep slots distinct
            if idx[t, 0] == idx[t, 1]:
                idx[t, 1] = (idx[t, 1] + 1) % E
                if idx[t, 1] % 3 == 0:
                    idx[t, 1] = (idx[t, 1] + 1) % E
    _check_permute(L, cfg, inp["x"], idx, keep)


def _unpermute_gpu(L, cfg, Yp, row_of, w, Ys=None, z=None):
    s = L.shape_of(cfg)
    out = empty((cfg.T, cfg.d), act_dtype(cfg))
    L.moe_unpermute(s, Yp, dev(row_of), dev(w), Ys, None if z is None else dev(z), out)
    torch.cuda.synchronize()
    return host(out)


def _as_act(cfg, v):
    """fp64 activation values (already rounded) -> device tensor of the layer dtype."""
    t = torch.from_numpy(np.asarray(v, np.float32))
    return t.to(act_dtype(cfg)).cuda()


@pytest.mark.parametrize("name", SMALL)
def test_unpermute(name):
    L = lib()
    cfg = get_config(name)
    inp = inputs(cfg, need_backward=False)
    f = O.layer_forward(cfg, inp)
    Ys = _as_act(cfg, f["Ys"]) if cfg.Fs else None
    z = f["gate_logit"].astype(np.float32) if cfg.Fs else None
    got = _unpermute_gpu(L, cfg, _as_act(cfg, f["Yp"]), f["row_of"], f["topk_w"].astype(np.float32), Ys, z)
    assert_close("out", got, f["out"], cfg.dtype)


def test_unpermute_dropped_tokens_output_zero():
    L = lib()
    cfg = dataclasses.replace(get_config("mixtral_8x22b@small"), T=300, d=256)
    rng = np.random.default_rng(4)
    row_of = np.full((cfg.T, cfg.K), -1, np.int32)
    kept = rng.random((cfg.T, cfg.K)) < 0.5
    row_of[kept] = np.arange(kept.sum(), dtype=np.int32)
    Yp = rng.standard_normal((cfg.T * cfg.K, cfg.d))
    w = rng.random((cfg.T, cfg.K)).astype(np.float32)
    got = _unpermute_gpu(L, cfg, _as_act(cfg, O.round_bf16(Yp)), row_of, w)
    ref = O.unpermute(O.round_bf16(Yp), row_of, w)
    assert_close("out", got, ref, "bf16")
    none = ~kept.any(axis=1)
    assert none.any() and np.all(got[none] == 0)


def test_identity_experts_round_trip():
    """Permute then un-permute with identity experts and unit weights gives
    K x exactly in bf16 (dropless)."""
    L = lib()
    cfg = dataclasses.replace(get_config("qwen2_57b_a14b@small"), T=640, Fs=0)
    inp = inputs(cfg, need_backward=False)
    r = O.route(cfg, inp)
    o, n = _check_permute(L, cfg, inp["x"], r["topk_idx"], r["keep"])
    got = _unpermute_gpu(L, cfg, o["Xp"], host(o["row_of"]), np.ones((cfg.T, cfg.K), np.float32))
    assert np.array_equal(got, cfg.K * O.decode(inp["x"]))


@pytest.mark.parametrize("K", [1, 3, 4, 5, 8])
@pytest.mark.parametrize("shared", [False, True])
def test_unpermute_and_backward_every_slot_bound(K, shared):
    """The un-permute kernels are compiled for slot bounds 1, 2, 4 and 8 (the
    smallest at or above K): every bound, K below its bound (3, 5), dropped
    slots and the shared expert, forward and backward, against the oracle."""
    L = lib()
    base = get_config("mixtral_8x22b@small")
    cfg = dataclasses.replace(base, T=333, d=512, E=8, K=K, Fs=256 if shared else 0)
    rng = np.random.default_rng(10 + K)
    row_of = np.full((cfg.T, K), -1, np.int32)
    kept = rng.random((cfg.T, K)) < 0.85
    row_of[kept] = rng.permutation(int(kept.sum())).astype(np.int32)
    n = int(kept.sum())
    Yp = O.round_bf16(rng.standard_normal((n, cfg.d)))
    w = rng.random((cfg.T, K)).astype(np.float32)
    dout = O.round_bf16(rng.standard_normal((cfg.T, cfg.d)))
    Ys = O.round_bf16(rng.standard_normal((cfg.T, cfg.d))) if shared else None
    z = rng.standard_normal(cfg.T).astype(np.float32) if shared else None
    s = L.shape_of(cfg)
    bf = torch.bfloat16
    Yp_d = torch.as_tensor(Yp, dtype=bf).cuda()
    Ys_d = torch.as_tensor(Ys, dtype=bf).cuda() if shared else None
    z_d = torch.as_tensor(z).cuda() if shared else None
    out = empty((cfg.T, cfg.d), bf)
    L.moe_unpermute(s, Yp_d, dev(row_of), dev(w), Ys_d, z_d, out)
    ref = O.unpermute(Yp, row_of, w, Ys, z)
    assert_close("out", host(out), ref, "bf16")
    dYp = empty((max(n, 1), cfg.d), bf)
    dw = empty((cfg.T, K), torch.float32)
    dYs = empty((cfg.T, cfg.d), bf) if shared else None
    dz = empty((cfg.T,), torch.float32) if shared else None
    L.moe_unpermute_bwd(s, torch.as_tensor(dout, dtype=bf).cuda(), Yp_d, dev(row_of), dev(w),
                        Ys_d, z_d, dYp, dw, dYs, dz)
    ub = O.unpermute_bwd(O.round_bf16(dout), Yp, row_of, w, Ys, z)
    # the oracle's dout argument is bf16 bits or values: it decodes arrays of values as is
    assert_close("dYp", host(dYp)[:n], ub["dYp"], "bf16")
    assert_close("dw", host(dw), ub["dw"], "bf16")
    if shared:
        assert_close("dYs", host(dYs), ub["dYs"], "bf16")
        assert_close("dz", host(dz), ub["dz"], "bf16")
