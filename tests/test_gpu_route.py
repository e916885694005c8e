"""GPU router vs oracle: decisions bit-exact on identical fp32 logits; the
fused router's logits within 1e-5 relative Frobenius, and its decisions equal
to the logits-in path applied to its own logits."""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs
from synthetic.gen import TID, normal_f32
from tests.gpu_util import inputs, FULL, SMALL, bf16_bits, dev, empty, host, lib, rel_frob, torch

pytestmark = pytest.mark.gpu


def _logits(cfg, ties: bool):
    l = normal_f32(cfg.seed, TID["logits"], (cfg.T, cfg.E), std=2.0 * cfg.router_scale)
    if ties:   # every 7th token repeats its predecessor: equal capacity keys
        l[7::7] = l[6:-1:7][: l[7::7].shape[0]]
    return l


def _route_topk_gpu(L, cfg, logits):
    T, K = cfg.T, cfg.K
    s = L.shape_of(cfg)
    ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
    out = dict(topk_idx=empty((T, K), torch.int32), topk_prob=empty((T, K), torch.float32),
               topk_w=empty((T, K), torch.float32), keep=empty((T, K), torch.uint8))
    L.moe_route_topk(s, dev(logits), out["topk_idx"], out["topk_prob"], out["topk_w"],
                     out["keep"], ws)
    L.moe_clear_status(ws)
    torch.cuda.synchronize()
    return {k: host(v) for k, v in out.items()}


def _assert_same_decisions(g, r):
    assert np.array_equal(g["topk_idx"], r["topk_idx"])
    assert np.array_equal(g["topk_prob"].view(np.uint32), np.asarray(r["topk_prob"], np.float32).view(np.uint32))
    assert np.array_equal(g["topk_w"].view(np.uint32), np.asarray(r["topk_w"], np.float32).view(np.uint32))
    assert np.array_equal(g["keep"], r["keep"])


@pytest.mark.parametrize("name", SMALL + FULL)
@pytest.mark.parametrize("ties", [False, True])
def test_route_topk_bit_exact(name, ties):
    L = lib()
    cfg = get_config(name)
    logits = _logits(cfg, ties)
    g = _route_topk_gpu(L, cfg, logits)
    r = O.route(cfg, None, logits=logits.astype(np.float64))
    _assert_same_decisions(g, r)


@pytest.mark.parametrize("variant", ["full_seq_drop", "no_renorm", "ragged_subseq", "k1", "e64k8_cf",
                                     "full_seq_drop_global_keys"])
def test_route_topk_variants(variant):
    L = lib()
    base = get_config("mixtral_8x22b_g8t8@small")
    cfg = {
        "full_seq_drop": dataclasses.replace(base, S=0),
        # a sub-sequence longer than the capacity kernel's shared-memory key
        # buffer (16384 candidates): the keys go to the workspace
        "full_seq_drop_global_keys": dataclasses.replace(base, T=20000, S=0),
        "no_renorm": dataclasses.replace(base, renorm=False),
        "ragged_subseq": dataclasses.replace(base, T=1000, S=300),
        "k1": dataclasses.replace(base, K=1, E=16, cf=0.5),
        "e64k8_cf": dataclasses.replace(base, cf=1.37),
    }[variant]
    logits = _logits(cfg, True)
    _assert_same_decisions(_route_topk_gpu(L, cfg, logits),
                           O.route(cfg, None, logits=logits.astype(np.float64)))


def test_exp_and_softmax_bits_over_a_wide_range():
    """E = 2: p0 = e^0 / (e^0 + e^u) with u = l1 - l0 swept over [-90, 0]: the
    GPU probabilities equal the oracle's fp32 arithmetic bit for bit."""
    L = lib()
    T = 1 << 18
    u = np.linspace(-90.0, 0.0, T).astype(np.float32)
    logits = np.stack([np.zeros(T, np.float32), u], axis=1)
    cfg = dataclasses.replace(get_config("tiny_f32"), T=T, E=2, K=2, drop=False)
    g = _route_topk_gpu(L, cfg, logits)
    r = O.route(cfg, None, logits=logits.astype(np.float64))
    _assert_same_decisions(g, r)


@pytest.mark.parametrize("name", SMALL + FULL)
def test_route_fused(name):
    _check_route(get_config(name))


# bf16 shapes whose row tiles (T / 128) leave SMs idle, so the tensor-core
# logits split their K loop over a cluster of CTAs (the even CTA adds the
# parts in order and routes): 4 parts of 8 K blocks with E = 8; 3 parts with
# the gate logit and bias riding along (E = 64 + 1 columns: the even CTA's
# exchange buffer holds two other parts); 3 parts over 3 ragged row tiles;
# 2 parts of 8 K blocks
SPLIT_K = {
    "split4_e8": ("mixtral_8x22b", dict(T=1000, d=2048, F=128, S=250)),
    "split4_gate_bias": ("qwen2_57b_a14b", dict(T=1000, d=2048, F=128, Fs=128)),
    "split3_ragged": ("mixtral_8x22b", dict(T=300, d=1536, F=128, S=100)),
    "split2_e64": ("mixtral_8x22b_g8t8", dict(T=2000, d=1024, F=128, S=500)),
    # the exchange and logits paths for rows that are not four contiguous
    # floats at a time: the gate column away from the experts (E = 8 padded
    # to 16), and E = 9
    "split4_gate_e8": ("qwen2_57b_a14b", dict(T=1000, d=2048, F=128, E=8, K=2, Fs=128)),
    "split4_e9": ("mixtral_8x22b", dict(T=1000, d=2048, F=128, E=9, S=250)),
}


# shapes whose router GEMM routes in its epilogue (no K split, E <= 16):
# E = 16 with K = 4, and E = 9 (padded to 16 experts) with the bias
FUSED = {
    "e16_k4": ("mixtral_8x22b", dict(T=1500, d=512, F=128, E=16, K=4, S=500)),
    "e9_bias": ("qwen2_57b_a14b", dict(T=700, d=512, F=128, E=9, K=3, Fs=0)),
}


@pytest.mark.parametrize("case", sorted(FUSED))
def test_route_fused_epilogue(case):
    base, kw = FUSED[case]
    _check_route(dataclasses.replace(get_config(base), name=f"{base}@{case}", **kw))


@pytest.mark.parametrize("case", sorted(SPLIT_K))
def test_route_split_k(case):
    base, kw = SPLIT_K[case]
    _check_route(dataclasses.replace(get_config(base), name=f"{base}@{case}", **kw))


def _check_route(cfg):
    L = lib()
    inp = inputs(cfg, need_backward=False)
    T, E, K = cfg.T, cfg.E, cfg.K
    s = L.shape_of(cfg)
    ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
    o = dict(logits=empty((T, E), torch.float32), topk_idx=empty((T, K), torch.int32),
             topk_prob=empty((T, K), torch.float32), topk_w=empty((T, K), torch.float32),
             keep=empty((T, K), torch.uint8))
    gl = empty((T,), torch.float32) if cfg.Fs else None
    L.moe_route(s, dev(inp["x"]), dev(inp["W_r"]), dev(inp["b_r"]) if cfg.bias else None,
                dev(inp["w_sg"]) if cfg.Fs else None, o["logits"], gl, o["topk_idx"],
                o["topk_prob"], o["topk_w"], o["keep"], ws)
    rc, info = L.moe_get_status(ws)
    assert rc == 0, (rc, hex(info))
    got = {k: host(v) for k, v in o.items()}
    ref_l = O.router_logits(inp["x"], inp["W_r"], inp.get("b_r"))
    assert rel_frob(got["logits"], ref_l) <= 1e-5
    if cfg.Fs:
        assert rel_frob(host(gl), O.gate_logit(inp["x"], inp["w_sg"])) <= 1e-5
    # decisions are the logits-in path applied to the fused path's own logits
    _assert_same_decisions(got, _route_topk_gpu(L, cfg, got["logits"]))
    # and agree with the oracle except on tokens whose decision is a near tie
    r = O.route(cfg, inp)
    same = np.all(got["topk_idx"] == r["topk_idx"], axis=1) & np.all(got["keep"] == r["keep"], axis=1)
    assert same.mean() >= 0.999, same.mean()
