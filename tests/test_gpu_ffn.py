"""GPU grouped SwiGLU FFN (tcgen05 path for bf16, CUDA-core path for fp32)
and its backward vs the oracle, on the oracle's permuted rows. Group layouts
include empty groups, groups of one row, groups spanning many 128-row tiles
with ragged tails, and a single group (the shared-expert call)."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs
from synthetic.gen import normal_bf16, normal_f32
from tests.gpu_util import inputs, FULL, SMALL, act_dtype, assert_close, dev, empty, host, lib, torch

pytestmark = pytest.mark.gpu


def _ffn_gpu(L, dtype, Xp, offsets, W_gu, W_down, max_rows, d, F, with_A=True):
    G = W_gu.shape[0]
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    code = L.MOE_BF16 if dtype == "bf16" else L.MOE_F32
    A = empty((max_rows, 2 * F), tdt) if with_A else None
    H = empty((max_rows, F), tdt)
    Y = empty((max_rows, d), tdt)
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    L.moe_expert_ffn(code, max_rows, d, F, G, dev(offsets), Xp, dev(W_gu), dev(W_down), A, H, Y, ws)
    rc, info = L.moe_get_status(ws)
    assert rc == 0, (rc, hex(info))
    return A, H, Y


def _check_fwd(L, dtype, Xp_host, offsets, W_gu, W_down, d, F, rows=None):
    n = int(offsets[-1])
    max_rows = max(n, 1)
    Xp = dev(Xp_host) if n else empty((1, d), torch.bfloat16 if dtype == "bf16" else torch.float32)
    A, H, Y = _ffn_gpu(L, dtype, Xp, offsets, W_gu, W_down, max_rows, d, F)
    Ar, Hr, Yr = O.expert_ffn(Xp_host, offsets, W_gu, W_down, dtype, rows=rows)
    sel = np.arange(n) if rows is None else rows
    assert_close("A_save", host(A)[sel], Ar[sel], dtype, "act")
    assert_close("H", host(H)[sel], Hr[sel], dtype, "act")
    assert_close("Yp", host(Y)[sel], Yr[sel], dtype, "act")
    return A, H, Y


@pytest.mark.parametrize("name", SMALL)
def test_ffn_forward(name):
    L = lib()
    cfg = get_config(name)
    inp = inputs(cfg, need_backward=False)
    r = O.route(cfg, inp)
    _, offsets, _, src_of, n = O.build_map(r["topk_idx"], r["keep"], cfg.E)
    Xp = O.permute(inp["x"], src_of, cfg.K)
    _check_fwd(L, cfg.dtype, Xp, offsets, inp["W_gu"], inp["W_down"], cfg.d, cfg.F)


@pytest.mark.parametrize("rows", [[0, 300, 1, 129, 0, 256, 2, 0], [0, 0, 0, 0], [517]])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ffn_group_layouts(rows, dtype):
    L = lib()
    d, F, G = 256, 384, len(rows)
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    n = int(offsets[-1])
    gen = normal_bf16 if dtype == "bf16" else normal_f32
    Xp = gen(5, 101, (max(n, 1), d))[:n]
    W_gu = gen(5, 102, (G, 2 * F, d), 1 / np.sqrt(d))
    W_down = gen(5, 103, (G, d, F), 1 / np.sqrt(F))
    if n == 0:
        return   # nothing to compare; the call must still succeed
    _check_fwd(L, dtype, Xp, offsets, W_gu, W_down, d, F)


@pytest.mark.parametrize("rows,d,F", [
    ([300, 129, 1, 0, 700], 4096, 256),   # gate/up with K = d = 4096 (two N tiles per pair tile)
    ([300, 0, 200], 512, 8192),           # down projection with K = F = 8192 (two N tiles)
])
def test_ffn_forward_long_k(rows, d, F):
    """The forward shapes that switch the gate/up and down GEMMs to two N
    tiles per pair tile, on ragged groups (a one-row group, an empty one, last
    tiles of at most 128 rows for the tail kernel), every element against the
    oracle."""
    L = lib()
    G = len(rows)
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    n = int(offsets[-1])
    Xp = normal_bf16(8, 101, (n, d))
    W_gu = normal_bf16(8, 102, (G, 2 * F, d), 1 / np.sqrt(d))
    W_down = normal_bf16(8, 103, (G, d, F), 1 / np.sqrt(F))
    _check_fwd(L, "bf16", Xp, offsets, W_gu, W_down, d, F)


@pytest.mark.parametrize("name", FULL)
def test_ffn_forward_full_size_sampled(name):
    """Full-size grouped GEMM on the workload's routing; 3 sampled rows per
    expert (first, middle, last) checked against the oracle row by row."""
    L = lib()
    cfg = get_config(name)
    inp = inputs(cfg, need_backward=False)
    r = O.route(cfg, inp)
    _, offsets, _, src_of, n = O.build_map(r["topk_idx"], r["keep"], cfg.E)
    Xp = O.permute(inp["x"], src_of, cfg.K)
    rows = sorted({int(v) for e in range(cfg.E) for v in
                   (offsets[e], (offsets[e] + offsets[e + 1]) // 2, offsets[e + 1] - 1)
                   if offsets[e + 1] > offsets[e]})
    _check_fwd(L, cfg.dtype, Xp, offsets, inp["W_gu"], inp["W_down"], cfg.d, cfg.F,
               rows=np.array(rows))


def _check_bwd(L, dtype, Xp, offsets, W_gu, W_down, dYp, d, F):
    n = int(offsets[-1])
    Ar, Hr, Yr = O.expert_ffn(Xp, offsets, W_gu, W_down, dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    code = L.MOE_BF16 if dtype == "bf16" else L.MOE_F32
    G = W_gu.shape[0]
    A = torch.from_numpy(Ar.astype(np.float32)).to(tdt).cuda()
    H = torch.from_numpy(Hr.astype(np.float32)).to(tdt).cuda()
    dY = torch.from_numpy(dYp.astype(np.float32)).to(tdt).cuda()
    dA = empty((n, 2 * F), tdt)
    dX = empty((n, d), torch.float32)
    dWgu = empty((G, 2 * F, d), torch.float32)
    dWd = empty((G, d, F), torch.float32)
    ws = torch.zeros(L.MOE_FFN_BWD_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    L.moe_expert_ffn_bwd(code, n, d, F, G, dev(offsets), dY, dev(Xp), A, H, dev(W_gu), dev(W_down),
                         dA, dX, dWgu, dWd, ws)
    rc, info = L.moe_get_status(ws)
    assert rc == 0, (rc, hex(info))
    dXr, dWgur, dWdr, dAr = O.expert_ffn_bwd(dYp, Xp, Ar, Hr, offsets, W_gu, W_down, dtype)
    assert_close("dA", host(dA), dAr, dtype, "act")
    assert_close("dXp", host(dX), dXr, dtype)
    assert_close("dW_down", host(dWd), dWdr, dtype)
    assert_close("dW_gu", host(dWgu), dWgur, dtype)


@pytest.mark.parametrize("rows", [[0, 300, 1, 129, 0, 256, 2, 70], [1000], [5, 0, 0, 64]])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ffn_backward_group_layouts(rows, dtype):
    L = lib()
    d, F, G = 256, 384, len(rows)
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    n = int(offsets[-1])
    gen = normal_bf16 if dtype == "bf16" else normal_f32
    Xp = gen(6, 101, (n, d))
    W_gu = gen(6, 102, (G, 2 * F, d), 1 / np.sqrt(d))
    W_down = gen(6, 103, (G, d, F), 1 / np.sqrt(F))
    rnd = O.act_rounder(dtype, True)
    dYp = rnd(O.decode(gen(6, 104, (n, d))) * 0.5)
    _check_bwd(L, dtype, Xp, offsets, W_gu, W_down, dYp, d, F)


@pytest.mark.parametrize("pair", ["0", "1"])
def test_single_cta_and_pair_kernels_agree(pair):
    """The CTA-pair and single-CTA grouped GEMMs both match the oracle (each
    run in its own process with the test build of the library, whose
    MOE_GEMM_PAIR switch selects the kernels and is read once)."""
    import os
    import subprocess
    import sys
    lib()
    from token_dispatch_expert_moe_gb300 import build
    code = ("import sys; sys.argv=['x']; import pytest; "
            "sys.exit(pytest.main(['-q', '-p', 'no:cacheprovider', '-k', "
            "'group_layouts and bf16', 'tests/test_gpu_ffn.py']))")
    env = dict(os.environ, MOE_GEMM_PAIR=pair, MOE_LIBRARY=build.TEST_LIB)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=root, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]


@pytest.mark.parametrize("rows,d,F", [
    ([8300, 8100], 512, 512),   # weight gradients: >= 8192 rows per group (two N tiles per pair tile)
    ([300, 0, 200], 8192, 512),  # dH with K = d = 8192 (two N tiles per pair tile)
    ([300, 200], 512, 4096),     # dXp with K = 2F = 8192 (two N tiles per pair tile)
    ([300, 129, 1], 512, 2048),  # dXp at the two-tile threshold, K = 2F = 4096, with tail tiles
])
def test_ffn_backward_long_k(rows, d, F):
    """The long-K shapes that switch the CTA-pair GEMMs to two N tiles per
    pair tile, against the oracle."""
    L = lib()
    G = len(rows)
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    n = int(offsets[-1])
    Xp = normal_bf16(7, 101, (n, d))
    W_gu = normal_bf16(7, 102, (G, 2 * F, d), 1 / np.sqrt(d))
    W_down = normal_bf16(7, 103, (G, d, F), 1 / np.sqrt(F))
    rnd = O.act_rounder("bf16", True)
    dYp = rnd(O.decode(normal_bf16(7, 104, (n, d))) * 0.5)
    _check_bwd(L, "bf16", Xp, offsets, W_gu, W_down, dYp, d, F)
