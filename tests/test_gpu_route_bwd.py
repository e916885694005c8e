"""GPU router backward (moe_route_bwd) vs the oracle's route_bwd on seeded
inputs, one case per register-tile width of the CUDA kernels (rows of dl
padded to 8, 16, 32, 64 and 72), with ragged token counts (not multiples of
the 128-token tile) and hidden sizes that end inside a 64-column tile and a
256-column tile, plus the tensor-core path (bf16, d a multiple of 256: dl as
three bf16 planes through the grouped-GEMM kernels; with a dx_in addend the
dx part stays on the CUDA cores). Outputs are fp32 sums of exactly representable inputs, so
every case is held to the fp32 tolerance (relative Frobenius and max-abs
1e-5)."""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config
from synthetic.gen import normal_bf16, normal_f32
from tests.gpu_util import assert_close, dev, empty, host, lib, torch

pytestmark = pytest.mark.gpu

# (dtype, T, d, E, K, shared-expert gate, renorm, dx_in given)
CASES = [
    ("f32", 300, 64, 4, 2, False, True, False),      # 8 rows
    ("bf16", 300, 200, 12, 2, False, False, True),   # 16 rows; d ends inside a 64-col tile
    ("bf16", 257, 384, 24, 4, True, True, True),     # 25 rows -> 32
    ("bf16", 1000, 520, 64, 8, False, True, False),  # 64 rows
    ("bf16", 129, 256, 64, 8, True, True, True),     # 65 rows -> 72
    ("f32", 77, 36, 5, 1, True, False, True),        # tiny, d not a multiple of 64
    # bf16 with d % 256 == 0: the tensor-core path (dl split into three bf16 planes)
    ("bf16", 1000, 512, 64, 8, False, True, False),  # 128-wide planes, dx GEMM
    ("bf16", 3000, 768, 8, 2, True, True, False),    # gate row, 64-wide planes, dx GEMM
    ("bf16", 2000, 256, 24, 4, False, False, False), # no renorm
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-T{c[1]}-d{c[2]}-E{c[3]}" for c in CASES])
def test_route_bwd_matches_oracle(case):
    L = lib()
    dtype, T, d, E, K, gate, renorm, with_dx_in = case
    cfg = dataclasses.replace(get_config("mixtral_8x22b@small"), T=T, d=d, E=E, K=K, dtype=dtype,
                              drop=False, renorm=renorm, Fs=128 if gate else 0, seed=3)
    gen = normal_bf16 if dtype == "bf16" else normal_f32
    x = gen(21, 1, (T, d))
    W_r = gen(21, 2, (E, d), 1 / np.sqrt(d))
    w_sg = gen(21, 3, (d,), 1 / np.sqrt(d)) if gate else None
    logits = normal_f32(21, 4, (T, E), std=2.0)
    dw = normal_f32(21, 5, (T, K))
    dz = normal_f32(21, 6, (T,)) if gate else None
    dx_in = normal_f32(21, 7, (T, d)) if with_dx_in else None
    r = O.route(cfg, None, logits=logits.astype(np.float64))
    ref = O.route_bwd(x, W_r, r["p"], r["topk_idx"], r["topk_prob"], r["topk_w"], dw, renorm,
                      w_sg, dz)
    s = L.shape_of(cfg)
    ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
    out = dict(dW_r=empty((E, d), torch.float32), db_r=empty((E,), torch.float32),
               dx_router=empty((T, d), torch.float32))
    if gate:
        out["dw_sg"] = empty((d,), torch.float32)
    L.moe_route_bwd(s, dev(x), dev(W_r), dev(w_sg) if gate else None, dev(logits),
                    dev(r["topk_idx"].astype(np.int32)), dev(np.asarray(r["topk_prob"], np.float32)),
                    dev(np.asarray(r["topk_w"], np.float32)), dev(dw), dev(dz) if gate else None,
                    dev(dx_in) if with_dx_in else None, out["dW_r"], out["db_r"],
                    out.get("dw_sg"), out["dx_router"], ws)
    rc, info = L.moe_get_status(ws)
    assert rc == 0, (rc, hex(info))
    ref_dx = ref["dx_router"] + (dx_in.astype(np.float64) if with_dx_in else 0.0)
    assert_close("dx_router", host(out["dx_router"]), ref_dx, "f32")
    assert_close("dW_r", host(out["dW_r"]), ref["dW_r"], "f32")
    assert_close("db_r", host(out["db_r"]), ref["db_r"], "f32")
    if gate:
        assert_close("dw_sg", host(out["dw_sg"]), ref["dw_sg"], "f32")
