"""Expert-parallel and expert-tensor-parallel exchange bookkeeping
(token_dispatch_expert_moe_gb300.ep) with gloo ranks on CPU.

Each rank holds its own tokens (its own seeded x) and the same weights. It
routes, builds the map and permutes with the oracle, exchanges rows with the
module under test, runs only its own experts (EP) or its own F-shard of every
expert (ETP) with the oracle's FFN, exchanges back, un-permutes, and compares
with the oracle layer run on that rank's tokens with every expert local. The
dispatch/combine round trip with identity experts must return the permuted
rows bit for bit. fp32 workloads: the only differences allowed are fp64
summation-order effects rounded to fp32 (1e-6 relative)."""
import dataclasses
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cfg(drop):
    from synthetic import get_config
    return dataclasses.replace(get_config("tiny_f32"), T=96, d=32, E=8, K=2, F=48, drop=drop,
                               cf=1.0, S=32, seed=5)


def _rank_inputs(cfg, rank):
    from synthetic import make_inputs
    from synthetic.gen import TID, normal_f32
    inp = make_inputs(cfg)                       # weights shared by every rank
    inp["x"] = normal_f32(100 + rank, TID["x"], (cfg.T, cfg.d))   # tokens of this rank
    return inp


def _close(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    rf = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)
    return rf <= 1e-6 and np.abs(a - b).max() <= 1e-6 * max(1.0, np.abs(b).max())


def _worker(rank, world, port, mode, drop, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import moe_oracle as O
        from token_dispatch_expert_moe_gb300 import ep
        cfg = _cfg(drop)
        inp = _rank_inputs(cfg, rank)
        E, K, F = cfg.E, cfg.K, cfg.F
        ref = O.layer_forward(cfg, inp)
        r = O.route(cfg, inp)
        counts, offsets, row_of, src_of, n = O.build_map(r["topk_idx"], r["keep"], E)
        Xp = O.permute(inp["x"], src_of, K)
        res = {}
        if mode == "ep":
            plan = ep.ep_plan(torch.from_numpy(counts.astype(np.int64)))
            recv = ep.ep_dispatch(torch.from_numpy(Xp), plan)
            # identity experts: the round trip is exact
            back = ep.ep_combine(recv, plan)
            res["roundtrip"] = bool(torch.equal(back, torch.from_numpy(Xp)))
            # bookkeeping
            El = E // world
            res["splits"] = (sum(plan.send_splits) == n and
                             int(plan.local_offsets[-1]) == recv.shape[0] and
                             plan.local_counts.sum().item() == sum(plan.recv_splits))
            lo = rank * El
            _, _, Y = O.expert_ffn(recv.numpy(), plan.local_offsets.numpy(), inp["W_gu"][lo:lo + El],
                                   inp["W_down"][lo:lo + El], cfg.dtype)
            Yp = ep.ep_combine(torch.from_numpy(Y), plan).numpy()
        else:   # etp: every rank holds every expert's F-shard [rank*F/world, (rank+1)*F/world)
            g, allc, order = ep.etp_allgather_v(torch.from_numpy(Xp), torch.from_numpy(counts))
            res["splits"] = int(allc.sum()) == g.shape[0] and int(allc[rank].sum()) == n
            goffs = np.zeros(E + 1, np.int32)
            goffs[1:] = np.cumsum(allc.sum(0).numpy())
            Fl = F // world
            cols = np.arange(rank * Fl, (rank + 1) * Fl)
            W_gu = np.concatenate([inp["W_gu"][:, cols], inp["W_gu"][:, F + cols]], axis=1)
            W_dn = inp["W_down"][:, :, cols]
            # partial outputs unrounded (fp64): the ReduceScatter-V sums them first
            _, _, Yh = O.expert_ffn(g.numpy(), goffs, W_gu, W_dn, cfg.dtype, mirror=False)
            Ysum = ep.etp_reduce_scatter_v(torch.from_numpy(Yh), allc, order).numpy()
            Yp = O.act_rounder(cfg.dtype, True)(Ysum)
            res["roundtrip"] = True
        out = O.unpermute(Yp, row_of, r["topk_w"], None, None, cfg.dtype)
        res["out"] = _close(out, ref["out"])
        q.put((rank, res))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("mode", ["ep", "etp"])
@pytest.mark.parametrize("drop", [False, True])
def test_exchange_matches_single_rank_layer(world, mode, drop):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, mode, drop, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r in sorted(res.items()):
        assert r["roundtrip"], rank
        assert r["splits"], rank
        assert r["out"], rank


def test_chunk_order():
    from token_dispatch_expert_moe_gb300.ep import chunk_order
    sizes = torch.tensor([[2, 0, 1], [1, 3, 0]])     # rows: a-major chunks (0,0)(0,1)(0,2)(1,0)...
    # a-major layout: [0,1] (0,0) | - (0,1) | [2] (0,2) | [3] (1,0) | [4,5,6] (1,1) | - (1,2)
    assert chunk_order(sizes).tolist() == [0, 1, 3, 4, 5, 6, 2]
    assert chunk_order(torch.zeros((2, 2), dtype=torch.int64)).tolist() == []
