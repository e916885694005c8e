"""Counter-style seeded normal draws and the per-workload input set.

Element i of tensor `tid` under seed `seed` is taken from an independent
Philox-4x32 stream keyed by (seed, tid, i // CHUNK), so any range of any tensor
can be regenerated alone, in parallel, on any host, with the same values.
bf16 tensors are fp32 draws rounded to the nearest bf16 (ties to even) and are
returned as their uint16 bit patterns.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import MoEConfig

CHUNK = 1 << 22

# Tensor ids: one per named input, fixed for all workloads.
TID = {"x": 1, "W_r": 2, "b_r": 3, "w_sg": 4, "W_gu": 5, "W_down": 6,
       "Ws_gu": 7, "Ws_down": 8, "dout": 9, "logits": 10,
       # stand-alone inputs of single calls (the stage tests at full size)
       "Yp": 11, "Ys": 12, "gate_logit": 13, "dXp": 14, "dx_add": 15}

_THREADS = max(1, min(32, len(os.sched_getaffinity(0))))


def _chunk_f32(seed: int, tid: int, c: int, n: int, std: float) -> np.ndarray:
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, tid, c])))
    a = g.standard_normal(n, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    u = a.view(np.uint32)
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (u >> np.uint32(16)).astype(np.uint16)


def _fill(seed: int, tid: int, n: int, std: float, bf16: bool) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16 if bf16 else np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c: int) -> None:
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        a = _chunk_f32(seed, tid, c, hi - lo, std)
        out[lo:hi] = _to_bf16_bits(a) if bf16 else a

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal_f32(seed: int, tid: int, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return _fill(seed, tid, n, std, False).reshape(shape)


def normal_bf16(seed: int, tid: int, shape, std: float = 1.0) -> np.ndarray:
    """uint16 bf16 bit patterns of N(0, std^2) draws."""
    n = int(np.prod(shape))
    return _fill(seed, tid, n, std, True).reshape(shape)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_inputs(cfg: MoEConfig, need_backward: bool | None = None) -> dict:
    """All inputs of one workload as host arrays.

    Distributions: x ~ N(0,1); W_r ~ N(0, (router_scale)^2/d); b_r ~ N(0,1);
    w_sg ~ N(0, 1/d); W_gu, Ws_gu ~ N(0, 1/d); W_down ~ N(0, 1/F);
    Ws_down ~ N(0, 1/Fs); upstream gradient dout ~ N(0,1).
    Layouts: x [T,d]; W_r [E,d]; W_gu [E,2F,d] (rows [0,F) gate, [F,2F) up);
    W_down [E,d,F]; Ws_gu [2Fs,d]; Ws_down [d,Fs]; dout [T,d].
    bf16 tensors are uint16 bit arrays; fp32 workloads give float32 arrays.
    b_r, when present, is always float32.
    """
    s, T, d, E, F = cfg.seed, cfg.T, cfg.d, cfg.E, cfg.F
    bf = cfg.dtype == "bf16"
    gen = normal_bf16 if bf else normal_f32
    inp = {
        "x": gen(s, TID["x"], (T, d)),
        "W_r": gen(s, TID["W_r"], (E, d), cfg.router_scale / np.sqrt(d)),
        "W_gu": gen(s, TID["W_gu"], (E, 2 * F, d), 1.0 / np.sqrt(d)),
        "W_down": gen(s, TID["W_down"], (E, d, F), 1.0 / np.sqrt(F)),
    }
    if cfg.bias:
        inp["b_r"] = normal_f32(s, TID["b_r"], (E,))
    if cfg.Fs:
        Fs = cfg.Fs
        inp["w_sg"] = gen(s, TID["w_sg"], (d,), 1.0 / np.sqrt(d))
        inp["Ws_gu"] = gen(s, TID["Ws_gu"], (2 * Fs, d), 1.0 / np.sqrt(d))
        inp["Ws_down"] = gen(s, TID["Ws_down"], (d, Fs), 1.0 / np.sqrt(Fs))
    if cfg.backward if need_backward is None else need_backward:
        inp["dout"] = gen(s, TID["dout"], (T, d))
    return inp
