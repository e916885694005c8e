"""MoELayer: the whole layer through the C ABI, buffers held in torch tensors.

Forward: moe_route -> moe_permute -> moe_expert_ffn (routed experts)
[-> moe_expert_ffn (shared expert: one group, offsets {0, T})] -> moe_unpermute.
Backward: moe_unpermute_bwd -> moe_expert_ffn_bwd (routed [, shared]) ->
moe_route_bwd -> moe_permute_bwd.
torch only allocates device memory and supplies the stream; every step runs
in libmoe.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib as L


def to_device(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Host array -> device tensor; uint16 arrays are bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class MoELayer:
    """One MoE layer of configuration `cfg` (a synthetic.MoEConfig-like object)
    with device weights W_r, W_gu, W_down (+ b_r, w_sg, Ws_gu, Ws_down).

    etp > 1 runs the routed experts F-split the way an expert-tensor-parallel
    group of `etp` ranks would (MoE Parallel Folding study notes, "method
    overview": the expert's FFN dimension is sharded and a ReduceScatter-V
    sums the partial outputs): shard s holds gate and up rows
    [s*F/etp, (s+1)*F/etp) and the matching W_down columns, each shard is one
    moe_expert_ffn call, and moe_sum_partials adds the partial Yp (and, in the
    backward, the partial dXp) in shard order. Weight gradients stay per shard.

    layout="padded" (token dropping only) uses the fixed GShard-style layout of
    moe_permute_padded: expert e owns rows [e*C, (e+1)*C), zero rows after its
    kept ones, and the grouped GEMMs run every padded row.

    gather=True (bf16, forward only, etp = 1) fuses the permutation into the
    routed experts' gate/up GEMM: moe_permute builds the map alone (Xp NULL)
    and moe_expert_ffn_gather reads each permuted row from x through src_of,
    so the permuted copy of the tokens is never written."""

    def __init__(self, cfg, weights: dict, device="cuda", backward=None, etp: int = 1,
                 layout: str = "compact", gather: bool = False):
        self.cfg = cfg
        self.etp = etp
        self.layout = layout
        self.gather = gather
        if gather and (etp != 1 or cfg.dtype != "bf16"
                       or (cfg.backward if backward is None else backward)):
            raise ValueError("gather=True serves the bf16 forward-only layer with etp = 1")
        self.shape = L.shape_of(cfg)
        self.backward_enabled = cfg.backward if backward is None else backward
        self.w = weights
        T, d, E, K, F = cfg.T, cfg.d, cfg.E, cfg.K, cfg.F
        dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        self.dt = dt
        self.dtype_code = L.MOE_BF16 if cfg.dtype == "bf16" else L.MOE_F32
        if layout == "padded":
            C = L.moe_padded_capacity(L.shape_of(cfg))
            if C <= 0:
                raise ValueError("the padded layout needs token dropping (a fixed capacity)")
            N = E * C
        elif layout == "compact":
            N = T * K
        else:
            raise ValueError(f"unknown layout {layout!r}")
        self.rows = N   # rows of the permuted buffers
        z = lambda *s, dtype=dt: torch.empty(*s, dtype=dtype, device=device)  # noqa: E731
        self.ws = torch.zeros(L.moe_workspace_size(self.shape), dtype=torch.uint8, device=device)
        self.logits = z(T, E, dtype=torch.float32)
        self.topk_idx = z(T, K, dtype=torch.int32)
        self.topk_prob = z(T, K, dtype=torch.float32)
        self.topk_w = z(T, K, dtype=torch.float32)
        self.keep = z(T, K, dtype=torch.uint8)
        self.Xp = None if gather else z(N, d)
        self.row_of = z(T, K, dtype=torch.int32)
        self.src_of = z(N, dtype=torch.int32)
        self.counts = z(E, dtype=torch.int32)
        self.offsets = z(E + 1, dtype=torch.int32)
        self.A_save = z(N, 2 * F) if self.backward_enabled and etp == 1 else None
        self.H = z(N, F) if etp == 1 else None
        self.Yp = z(N, d)
        if etp > 1:
            if F % etp != 0:
                raise ValueError(f"F={F} does not split into {etp} shards")
            Fl = F // etp
            self.Fl = Fl
            Wgu, Wdn = weights["W_gu"], weights["W_down"]
            self.W_gu_s = [torch.cat([Wgu[:, s * Fl:(s + 1) * Fl], Wgu[:, F + s * Fl:F + (s + 1) * Fl]],
                                     dim=1).contiguous() for s in range(etp)]
            self.W_down_s = [Wdn[:, :, s * Fl:(s + 1) * Fl].contiguous() for s in range(etp)]
            self.A_s = [z(N, 2 * Fl) if self.backward_enabled else None for _ in range(etp)]
            self.H_s = [z(N, Fl) for _ in range(etp)]
            self.Y_parts = z(etp, N, d)
        self.out = z(T, d)
        self.shared = cfg.Fs > 0
        if self.shared:
            Fs = cfg.Fs
            self.gate_logit = z(T, dtype=torch.float32)
            self.off1 = torch.tensor([0, T], dtype=torch.int32, device=device)
            self.As = z(T, 2 * Fs) if self.backward_enabled else None
            self.Hs = z(T, Fs)
            self.Ys = z(T, d)
        else:
            self.gate_logit = self.Ys = None
        if self.backward_enabled:
            # zeros: in the padded layout the padding rows of dYp are never
            # written, and the weight gradients read them (times zero activations)
            self.dYp = torch.zeros((N, d), dtype=dt, device=device)
            self.dw = z(T, K, dtype=torch.float32)
            self.dXp = z(N, d, dtype=torch.float32)
            if etp == 1:
                self.dA = z(N, 2 * F)
                self.dW_gu = z(E, 2 * F, d, dtype=torch.float32)
                self.dW_down = z(E, d, F, dtype=torch.float32)
            else:
                Fl = self.Fl
                self.dA_s = z(N, 2 * Fl)   # reused shard after shard
                self.dX_parts = z(etp, N, d, dtype=torch.float32)
                self.dW_gu = [z(E, 2 * Fl, d, dtype=torch.float32) for _ in range(etp)]
                self.dW_down = [z(E, d, Fl, dtype=torch.float32) for _ in range(etp)]
            self.dW_r = z(E, d, dtype=torch.float32)
            self.db_r = z(E, dtype=torch.float32)
            self.dx_router = z(T, d, dtype=torch.float32)
            self.dx = z(T, d, dtype=torch.float32)
            if self.shared:
                Fs = cfg.Fs
                self.dYs = z(T, d)
                self.dz = z(T, dtype=torch.float32)
                self.dAs = z(T, 2 * Fs)
                self.dXs = z(T, d, dtype=torch.float32)
                self.dWs_gu = z(2 * Fs, d, dtype=torch.float32)
                self.dWs_down = z(d, Fs, dtype=torch.float32)
                self.dw_sg = z(d, dtype=torch.float32)

    def forward(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        c, s, w = self.cfg, self.shape, self.w
        self.x = x
        L.moe_route(s, x, w["W_r"], w.get("b_r"), w.get("w_sg"), self.logits, self.gate_logit,
                    self.topk_idx, self.topk_prob, self.topk_w, self.keep, self.ws, stream)
        permute = L.moe_permute_padded if self.layout == "padded" else L.moe_permute
        permute(s, x, self.topk_idx, self.keep, self.Xp, self.row_of, self.src_of,
                self.counts, self.offsets, self.ws, stream)
        self.routed_ffn(stream)
        if self.shared:
            L.moe_expert_ffn(self.dtype_code, c.T, c.d, c.Fs, 1, self.off1, x, w["Ws_gu"],
                             w["Ws_down"], self.As, self.Hs, self.Ys, self.ws, stream)
        L.moe_unpermute(s, self.Yp, self.row_of, self.topk_w, self.Ys, self.gate_logit, self.out,
                        stream)
        return self.out

    def routed_ffn(self, stream=None):
        c, w = self.cfg, self.w
        if self.gather:
            L.moe_expert_ffn_gather(self.rows, c.d, c.F, c.E, self.offsets, self.x, c.T, c.K,
                                    self.src_of, w["W_gu"], w["W_down"], self.A_save, self.H,
                                    self.Yp, self.ws, stream)
            return
        if self.etp == 1:
            L.moe_expert_ffn(self.dtype_code, self.rows, c.d, c.F, c.E, self.offsets, self.Xp,
                             w["W_gu"], w["W_down"], self.A_save, self.H, self.Yp, self.ws, stream)
            return
        for s in range(self.etp):
            L.moe_expert_ffn(self.dtype_code, self.rows, c.d, self.Fl, c.E, self.offsets, self.Xp,
                             self.W_gu_s[s], self.W_down_s[s], self.A_s[s], self.H_s[s],
                             self.Y_parts[s], self.ws, stream)
        L.moe_sum_partials(self.dtype_code, self.etp, self.rows, c.d, self.Y_parts, self.Yp, stream)

    def routed_ffn_bwd(self, stream=None):
        c, w = self.cfg, self.w
        if self.etp == 1:
            L.moe_expert_ffn_bwd(self.dtype_code, self.rows, c.d, c.F, c.E, self.offsets, self.dYp,
                                 self.Xp, self.A_save, self.H, w["W_gu"], w["W_down"], self.dA,
                                 self.dXp, self.dW_gu, self.dW_down, self.ws, stream)
            return
        for s in range(self.etp):
            L.moe_expert_ffn_bwd(self.dtype_code, self.rows, c.d, self.Fl, c.E, self.offsets,
                                 self.dYp, self.Xp, self.A_s[s], self.H_s[s], self.W_gu_s[s],
                                 self.W_down_s[s], self.dA_s, self.dX_parts[s], self.dW_gu[s],
                                 self.dW_down[s], self.ws, stream)
        L.moe_sum_partials(L.MOE_F32, self.etp, self.rows, c.d, self.dX_parts, self.dXp, stream)

    def backward(self, dout: torch.Tensor, stream=None, marks=None) -> dict:
        """marks: optional dict of (start, end) CUDA event pairs, keyed by
        "unpermute_bwd", "ffn_bwd" (routed experts), "shared_ffn_bwd",
        "route_bwd" and "permute_bwd"; each present pair is recorded on the
        current stream around that call."""
        c, s, w = self.cfg, self.shape, self.w
        marks = marks or {}

        def mark(name, i):
            if name in marks:
                marks[name][i].record()

        mark("unpermute_bwd", 0)
        L.moe_unpermute_bwd(s, dout, self.Yp, self.row_of, self.topk_w, self.Ys, self.gate_logit,
                            self.dYp, self.dw, self.dYs if self.shared else None,
                            self.dz if self.shared else None, stream)
        mark("unpermute_bwd", 1)
        mark("ffn_bwd", 0)
        self.routed_ffn_bwd(stream)
        mark("ffn_bwd", 1)
        dx_in = None
        if self.shared:
            mark("shared_ffn_bwd", 0)
            L.moe_expert_ffn_bwd(self.dtype_code, c.T, c.d, c.Fs, 1, self.off1, self.dYs, self.x,
                                 self.As, self.Hs, w["Ws_gu"], w["Ws_down"], self.dAs, self.dXs,
                                 self.dWs_gu, self.dWs_down, self.ws, stream)
            mark("shared_ffn_bwd", 1)
            dx_in = self.dXs
        mark("route_bwd", 0)
        L.moe_route_bwd(s, self.x, w["W_r"], w.get("w_sg"), self.logits, self.topk_idx,
                        self.topk_prob, self.topk_w, self.dw, self.dz if self.shared else None,
                        dx_in, self.dW_r, self.db_r if "b_r" in w else None,
                        self.dw_sg if self.shared else None, self.dx_router, self.ws, stream)
        mark("route_bwd", 1)
        mark("permute_bwd", 0)
        L.moe_permute_bwd(s, self.dXp, self.row_of, self.dx_router, self.dx, stream)
        mark("permute_bwd", 1)
        g = {"dx": self.dx, "dW_r": self.dW_r, "dW_gu": self.dW_gu, "dW_down": self.dW_down}
        if "b_r" in w:
            g["db_r"] = self.db_r
        if self.shared:
            g.update(dWs_gu=self.dWs_gu, dWs_down=self.dWs_down, dw_sg=self.dw_sg)
        return g
