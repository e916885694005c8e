"""The bandwidth-bound calls of the layer at the workloads' full sizes, checked
element by element against the oracle: moe_unpermute (weighted Top-K
combine), moe_unpermute_bwd (dYp, dw and the shared expert's dYs, dz) and
moe_permute_bwd (dx), on every bf16 workload at its full T and d.

Inputs are seeded synthetic tensors of the workload's shape: the routing is
the oracle's own (softmax, Top-K, capacity dropping) on synthetic fp32 logits,
and Yp, Ys, gate logits, dout, dXp and the dx addend are normal draws. The
oracle evaluates the same calls on chunks of tokens (each call is independent
per token), with the chunk's permuted rows renumbered locally, so every
output element of the GPU call is compared.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, normal_bf16, normal_f32
from synthetic.gen import TID
from tests.gpu_util import FULL, assert_close, bf16_bits, dev, host, lib, torch

pytestmark = pytest.mark.gpu

CHUNK = 2048   # tokens per oracle evaluation


def _routing(cfg):
    logits = normal_f32(cfg.seed, TID["logits"], (cfg.T, cfg.E), 2.0)
    r = O.route(cfg, {}, logits=logits)
    _, _, row_of, _, n_kept = O.build_map(r["topk_idx"], r["keep"], cfg.E)
    return r, row_of, n_kept


def _local(row_of_chunk):
    """The chunk's kept rows (ascending) and row_of renumbered into them."""
    rows = np.unique(row_of_chunk[row_of_chunk >= 0])
    loc = np.full_like(row_of_chunk, -1)
    m = row_of_chunk >= 0
    loc[m] = np.searchsorted(rows, row_of_chunk[m])
    return rows, loc


def _bf16(t):
    return O.decode(bf16_bits(t))


@pytest.mark.parametrize("name", FULL)
def test_unpermute_and_backward_full_size(name):
    L = lib()
    cfg = get_config(name)
    assert cfg.dtype == "bf16"
    T, d, K, s = cfg.T, cfg.d, cfg.K, cfg.seed
    r, row_of, n_kept = _routing(cfg)
    Yp = normal_bf16(s, TID["Yp"], (n_kept, d))
    dout = normal_bf16(s, TID["dout"], (T, d))
    Ys = normal_bf16(s, TID["Ys"], (T, d)) if cfg.Fs else None
    z = normal_f32(s, TID["gate_logit"], (T,)) if cfg.Fs else None
    shape = L.shape_of(cfg)
    row_of_d, w_d, Yp_d = dev(row_of), dev(r["topk_w"]), dev(Yp)
    Ys_d = dev(Ys) if Ys is not None else None
    z_d = dev(z) if z is not None else None
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    L.moe_unpermute(shape, Yp_d, row_of_d, w_d, Ys_d, z_d, out)
    dYp = torch.empty((max(n_kept, 1), d), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((T, K), dtype=torch.float32, device="cuda")
    dYs = torch.empty((T, d), dtype=torch.bfloat16, device="cuda") if cfg.Fs else None
    dz = torch.empty((T,), dtype=torch.float32, device="cuda") if cfg.Fs else None
    L.moe_unpermute_bwd(shape, dev(dout), Yp_d, row_of_d, w_d, Ys_d, z_d, dYp, dw, dYs, dz)
    torch.cuda.synchronize()
    out_h, dYp_h, dw_h = _bf16(out), _bf16(dYp), host(dw)
    dYs_h = _bf16(dYs) if dYs is not None else None
    dz_h = host(dz) if dz is not None else None
    for lo in range(0, T, CHUNK):
        hi = min(T, lo + CHUNK)
        rows, loc = _local(row_of[lo:hi])
        Yl = O.decode(Yp[rows])
        Ysl = O.decode(Ys[lo:hi]) if Ys is not None else None
        zl = z[lo:hi] if z is not None else None
        w = r["topk_w"][lo:hi]
        ref = O.unpermute(Yl, loc, w, Ysl, zl, dtype="bf16")
        assert_close(f"out[{lo}:{hi}]", out_h[lo:hi], ref, "bf16")
        ub = O.unpermute_bwd(dout[lo:hi], Yl, loc, w, Ysl, zl, dtype="bf16")
        if rows.size:
            assert_close(f"dYp[{lo}:{hi}]", dYp_h[rows], ub["dYp"], "bf16")
        assert_close(f"dw[{lo}:{hi}]", dw_h[lo:hi], ub["dw"], "bf16")
        if Ys is not None:
            assert_close(f"dYs[{lo}:{hi}]", dYs_h[lo:hi], ub["dYs"], "bf16")
            assert_close(f"dz[{lo}:{hi}]", dz_h[lo:hi], ub["dz"], "bf16")


@pytest.mark.parametrize("name", FULL)
def test_permute_bwd_full_size(name):
    L = lib()
    cfg = get_config(name)
    T, d, s = cfg.T, cfg.d, cfg.seed
    r, row_of, n_kept = _routing(cfg)
    dXp = normal_f32(s, TID["dXp"], (n_kept, d))
    dx_add = normal_f32(s, TID["dx_add"], (T, d))
    dx = torch.empty((T, d), dtype=torch.float32, device="cuda")
    L.moe_permute_bwd(L.shape_of(cfg), dev(dXp), dev(row_of), dev(dx_add), dx)
    torch.cuda.synchronize()
    dx_h = host(dx)
    for lo in range(0, T, CHUNK):
        hi = min(T, lo + CHUNK)
        rows, loc = _local(row_of[lo:hi])
        ref = O.permute_bwd(dXp[rows].astype(np.float64), loc, dx_add[lo:hi].astype(np.float64))
        # fp32 sums of at most K + 1 terms: equal to the oracle's fp32 rounding
        # of the exact sum up to the rounding of the partial sums
        assert_close(f"dx[{lo}:{hi}]", dx_h[lo:hi], ref, "bf16")
        assert np.abs(dx_h[lo:hi] - ref).max() <= 4 * (cfg.K + 1) * 2.0 ** -24 * max(
            1.0, np.abs(ref).max())
