"""ctypes binding of libmoe.so (argument marshalling only).

Each function has the name and argument order of the C entry point declared in
include/moe.h. Tensor arguments are torch tensors (or None for NULL); they are
passed as raw device pointers. `stream` defaults to torch's current CUDA
stream. A non-OK status raises MoEError. There is no fallback: if libmoe.so is
missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_LIBRARY selects another build of the library (the tests point it at
# libmoe_testhooks.so, the build with the failure-injection hooks)
LIB_PATH = os.environ.get("MOE_LIBRARY") or os.path.join(PKG, "libmoe.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_FFN_BWD_WORKSPACE_BYTES = 33280   # include/moe.h
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_DEVICE"}


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {STATUS.get(code, code)}")
        self.code = code


class MoEShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("F", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("drop", ctypes.c_int32), ("capacity_factor", ctypes.c_float),
                ("subseq_len", ctypes.c_int64), ("renorm", ctypes.c_int32), ("Fs", ctypes.c_int32)]


def shape_of(cfg) -> MoEShape:
    """moe_shape_t of a synthetic.MoEConfig-like object."""
    return MoEShape(T=cfg.T, d=cfg.d, E=cfg.E, K=cfg.K, F=cfg.F,
                    dtype=MOE_BF16 if cfg.dtype == "bf16" else MOE_F32,
                    drop=int(cfg.drop), capacity_factor=float(cfg.cf),
                    subseq_len=int(cfg.S), renorm=int(cfg.renorm), Fs=int(cfg.Fs))


if not os.path.exists(LIB_PATH):
    raise ImportError(f"the library is not built ({LIB_PATH}); run "
                      "`python -m token_dispatch_expert_moe_gb300.build`")
lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_S = ctypes.POINTER(MoEShape)
_I32, _I64 = ctypes.c_int32, ctypes.c_int64

_SIGS = {
    "moe_route": [_S, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_route_topk": [_S, _P, _P, _P, _P, _P, _P, _P],
    "moe_permute": [_S, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_permute_noalloc": [_S, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_permute_padded": [_S, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_expert_ffn": [_I32, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_expert_ffn_gather": [_I64, _I32, _I32, _I32, _P, _P, _I64, _I32, _P, _P, _P, _P, _P, _P,
                              _P, _P],
    "moe_unpermute": [_S, _P, _P, _P, _P, _P, _P, _P],
    "moe_unpermute_bwd": [_S, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_expert_ffn_bwd": [_I32, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                           _P, _P, _P, ctypes.c_size_t, _P],
    "moe_permute_bwd": [_S, _P, _P, _P, _P, _P],
    "moe_sum_partials": [_I32, _I32, _I64, _I32, _P, _P, _P],
    "moe_route_bwd": [_S, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_clear_status": [_P, _P],
    "moe_get_status": [_P, _P, ctypes.POINTER(ctypes.c_uint32)],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
lib.moe_workspace_size.argtypes = [_S]
lib.moe_workspace_size.restype = ctypes.c_size_t
lib.moe_padded_capacity.argtypes = [_S]
lib.moe_padded_capacity.restype = ctypes.c_int64
lib.moe_version.restype = ctypes.c_char_p
lib.moe_status_string.argtypes = [ctypes.c_int]
lib.moe_status_string.restype = ctypes.c_char_p

EXPORTED = sorted(list(_SIGS) + ["moe_workspace_size", "moe_version", "moe_status_string",
                                  "moe_padded_capacity"])


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name, *args):
    rc = getattr(lib, name)(*args)
    if rc != 0:
        raise MoEError(name, rc)


def version() -> str:
    return lib.moe_version().decode()


def moe_workspace_size(shape: MoEShape) -> int:
    return int(lib.moe_workspace_size(ctypes.byref(shape)))


def moe_clear_status(ws, stream=None):
    _call("moe_clear_status", _ptr(ws), _stream(stream))


def moe_get_status(ws, stream=None):
    info = ctypes.c_uint32(0)
    rc = lib.moe_get_status(_ptr(ws), _stream(stream), ctypes.byref(info))
    return rc, info.value


def moe_route(shape, x, W_r, b_r, w_sg, logits, gate_logit, topk_idx, topk_prob, topk_w, keep,
              ws, stream=None):
    _call("moe_route", ctypes.byref(shape), _ptr(x), _ptr(W_r), _ptr(b_r), _ptr(w_sg),
          _ptr(logits), _ptr(gate_logit), _ptr(topk_idx), _ptr(topk_prob), _ptr(topk_w),
          _ptr(keep), _ptr(ws), _stream(stream))


def moe_route_topk(shape, logits, topk_idx, topk_prob, topk_w, keep, ws, stream=None):
    _call("moe_route_topk", ctypes.byref(shape), _ptr(logits), _ptr(topk_idx), _ptr(topk_prob),
          _ptr(topk_w), _ptr(keep), _ptr(ws), _stream(stream))


def moe_permute(shape, x, topk_idx, keep, Xp, row_of, src_of, counts, offsets, ws, stream=None):
    _call("moe_permute", ctypes.byref(shape), _ptr(x), _ptr(topk_idx), _ptr(keep), _ptr(Xp),
          _ptr(row_of), _ptr(src_of), _ptr(counts), _ptr(offsets), _ptr(ws), _stream(stream))


def moe_padded_capacity(shape: MoEShape) -> int:
    return int(lib.moe_padded_capacity(ctypes.byref(shape)))


def moe_permute_padded(shape, x, topk_idx, keep, Xp, row_of, src_of, counts, offsets, ws,
                       stream=None):
    _call("moe_permute_padded", ctypes.byref(shape), _ptr(x), _ptr(topk_idx), _ptr(keep),
          _ptr(Xp), _ptr(row_of), _ptr(src_of), _ptr(counts), _ptr(offsets), _ptr(ws),
          _stream(stream))


def moe_permute_noalloc(shape, x, topk_idx, keep, Xp, row_of, src_of, counts, offsets,
                        stream=None):
    """moe_permute without a workspace (scratch inside libmoe.so); see moe.h."""
    _call("moe_permute_noalloc", ctypes.byref(shape), _ptr(x), _ptr(topk_idx), _ptr(keep),
          _ptr(Xp), _ptr(row_of), _ptr(src_of), _ptr(counts), _ptr(offsets), _stream(stream))


def moe_expert_ffn(dtype, max_rows, d, F, n_groups, offsets, Xp, W_gu, W_down, A_save, H_save,
                   Yp, ws, stream=None):
    _call("moe_expert_ffn", dtype, max_rows, d, F, n_groups, _ptr(offsets), _ptr(Xp), _ptr(W_gu),
          _ptr(W_down), _ptr(A_save), _ptr(H_save), _ptr(Yp), _ptr(ws), _stream(stream))


def moe_expert_ffn_gather(max_rows, d, F, n_groups, offsets, x, T, K, src_of, W_gu, W_down,
                          A_save, H_save, Yp, ws, stream=None):
    _call("moe_expert_ffn_gather", max_rows, d, F, n_groups, _ptr(offsets), _ptr(x), T, K,
          _ptr(src_of), _ptr(W_gu), _ptr(W_down), _ptr(A_save), _ptr(H_save), _ptr(Yp), _ptr(ws),
          _stream(stream))


def moe_unpermute(shape, Yp, row_of, topk_w, Ys, gate_logit, out, stream=None):
    _call("moe_unpermute", ctypes.byref(shape), _ptr(Yp), _ptr(row_of), _ptr(topk_w), _ptr(Ys),
          _ptr(gate_logit), _ptr(out), _stream(stream))


def moe_unpermute_bwd(shape, dout, Yp, row_of, topk_w, Ys, gate_logit, dYp, dw, dYs, dz,
                      stream=None):
    _call("moe_unpermute_bwd", ctypes.byref(shape), _ptr(dout), _ptr(Yp), _ptr(row_of),
          _ptr(topk_w), _ptr(Ys), _ptr(gate_logit), _ptr(dYp), _ptr(dw), _ptr(dYs), _ptr(dz),
          _stream(stream))


def moe_expert_ffn_bwd(dtype, max_rows, d, F, n_groups, offsets, dYp, Xp, A_save, H_save, W_gu,
                       W_down, dA, dXp, dW_gu, dW_down, ws, stream=None, ws_bytes=None):
    """ws: a device tensor (its size becomes ws_bytes) or a pointer with ws_bytes."""
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _call("moe_expert_ffn_bwd", dtype, max_rows, d, F, n_groups, _ptr(offsets), _ptr(dYp),
          _ptr(Xp), _ptr(A_save), _ptr(H_save), _ptr(W_gu), _ptr(W_down), _ptr(dA), _ptr(dXp),
          _ptr(dW_gu), _ptr(dW_down), _ptr(ws), ws_bytes, _stream(stream))


def moe_permute_bwd(shape, dXp, row_of, dx_add, dx, stream=None):
    _call("moe_permute_bwd", ctypes.byref(shape), _ptr(dXp), _ptr(row_of), _ptr(dx_add), _ptr(dx),
          _stream(stream))


def moe_sum_partials(dtype, n_parts, rows, d, partials, out, stream=None):
    _call("moe_sum_partials", dtype, n_parts, rows, d, _ptr(partials), _ptr(out), _stream(stream))


def moe_route_bwd(shape, x, W_r, w_sg, logits, topk_idx, topk_prob, topk_w, dw, dz, dx_in, dW_r,
                  db_r, dw_sg, dx_router, ws, stream=None):
    _call("moe_route_bwd", ctypes.byref(shape), _ptr(x), _ptr(W_r), _ptr(w_sg), _ptr(logits),
          _ptr(topk_idx), _ptr(topk_prob), _ptr(topk_w), _ptr(dw), _ptr(dz), _ptr(dx_in),
          _ptr(dW_r), _ptr(db_r), _ptr(dw_sg), _ptr(dx_router), _ptr(ws), _stream(stream))
