"""The oracle's pins are sharp: each plausible mistake planted in the oracle
(on the CPU, through monkeypatch, for one test only) makes one of its pins
fail. Every mutant below is a slip a reader of the method could make (a
dropped term, a wrong sign, a swapped operand, a wrong index or tie rule, the
wrong summation order), and the pin named beside it is the one that catches it.
"""
import math

import numpy as np
import pytest

from oracle import moe_oracle as O
from tests import test_oracle_layer as PL
from tests import test_oracle_rounding_points as PRP
from tests import test_oracle_routing as PR
from tests import test_oracle_softmax as PS
from tests import test_oracle_values as PV

_orig = {n: getattr(O, n) for n in (
    "silu", "swiglu_group", "route_bwd", "sigmoid", "capacity", "unpermute", "unpermute_bwd",
    "permute_bwd", "sum_partials", "router_logits", "padded_capacity", "route", "expert_ffn",
    "swiglu_group_bwd")}


# ---- mutants ----

def _swiglu_gate_up_swapped(X, Wgu, Wdown, rnd):
    F = Wgu.shape[0] // 2
    return _orig["swiglu_group"](X, np.concatenate([Wgu[F:], Wgu[:F]]), Wdown, rnd)


def _swiglu_bwd(sign_dg=1.0, keep_g_in_du=True):
    def f(dY, X, A, H, Wgu, Wdown, rnd, r32):
        F = Wgu.shape[0] // 2
        dH = dY @ Wdown
        G, U = A[:, :F], A[:, F:]
        sg = 1.0 / (1.0 + np.exp(-G))
        dG = dH * U * sg * (1.0 + sign_dg * G * (1.0 - sg))
        dU = dH * (G if keep_g_in_du else 1.0) * sg
        dA = rnd(np.concatenate([dG, dU], axis=1))
        return r32(dA @ Wgu), r32(dY.T @ H), r32(dA.T @ X), dA
    return f


def _route_bwd_without_renorm_term(*a, **k):
    return _orig["route_bwd"](*a[:7], False, *a[8:], **k)


def _route_bwd_without_gate_term_in_dx(*a, **k):
    r = _orig["route_bwd"](*a, **k)
    if len(a) > 9 and a[9] is not None:
        r["dx_router"] = _orig["route_bwd"](*a[:9], None, **k)["dx_router"]
    return r


def _route_bwd_jacobian_sign(x, W_r, p, idx, prob, w, dw, renorm, w_sg=None, dz=None,
                             mirror=True):
    """dl = p (dp + sum p dp): the softmax Jacobian's minus sign turned."""
    r = _orig["route_bwd"](x, W_r, p, idx, prob, w, dw, renorm, w_sg, dz, mirror=mirror)
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(dw, dtype=np.float64)
    if renorm:
        Z = np.asarray(prob, dtype=np.float64).sum(axis=1, keepdims=True)
        dpk = (g - (g * np.asarray(w, dtype=np.float64)).sum(axis=1, keepdims=True)) / Z
    else:
        dpk = g
    dp = np.zeros_like(p)
    np.put_along_axis(dp, idx.astype(np.int64), dpk, axis=1)
    dl = p * (dp + (p * dp).sum(axis=1, keepdims=True))
    r32 = O.f32_rounder(mirror)
    X, Wr = O.decode(x), O.decode(W_r)
    dxr = dl @ Wr
    if dz is not None:
        dxr = dxr + np.asarray(dz, dtype=np.float64)[:, None] * O.decode(w_sg)[None, :]
    r.update(dlogits=dl, dW_r=r32(dl.T @ X), db_r=r32(dl.sum(axis=0)), dx_router=r32(dxr))
    return r


def _topk_ties_to_higher_index(p, K):
    work = np.array(p, copy=True)[:, ::-1].copy()
    E = work.shape[1]
    T = work.shape[0]
    idx = np.empty((T, K), dtype=np.int32)
    rows = np.arange(T)
    for k in range(K):
        j = np.argmax(work, axis=1)
        idx[:, k] = E - 1 - j
        work[rows, j] = -np.inf
    return idx, np.take_along_axis(np.asarray(p), idx.astype(np.int64), axis=1)


def _capacity_keep(ties_to_higher_token=False, full_cap_for_short_block=False):
    def f(idx, prob, E, cf, S):
        T, K = idx.shape
        keep = np.zeros((T, K), dtype=np.uint8)
        S = S if S > 0 else T
        for lo in range(0, T, S):
            hi = min(T, lo + S)
            cap = O.capacity(cf, S if full_cap_for_short_block else hi - lo, K, E)
            sub_idx, sub_p = idx[lo:hi], prob[lo:hi]
            for e in range(E):
                t_loc, k = np.nonzero(sub_idx == e)
                if t_loc.size == 0:
                    continue
                pe = sub_p[t_loc, k].astype(np.float64)
                order = np.lexsort(((-t_loc if ties_to_higher_token else t_loc), -pe))
                chosen = order[:cap]
                keep[lo + t_loc[chosen], k[chosen]] = 1
        return keep
    return f


def _build_map_tokens_descending(idx, keep, E):
    T, K = idx.shape
    t, k = np.nonzero(keep)
    e = idx[t, k]
    order = np.lexsort((-t, e))
    t, k, e = t[order], k[order], e[order]
    counts = np.bincount(e, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    n_kept = int(offsets[E])
    row_of = np.full((T, K), -1, dtype=np.int32)
    row_of[t, k] = np.arange(n_kept, dtype=np.int32)
    return counts, offsets, row_of, (t * K + k).astype(np.int32), n_kept


def _route_ranks_capacity_by_weight(cfg, inp, mirror=True, logits=None):
    """route() with the capacity keys taken from the renormalised weights."""
    r = _orig["route"](cfg, inp, mirror=mirror, logits=logits)
    if cfg.drop:
        r["keep"] = O.capacity_keep(r["topk_idx"], r["topk_w"], cfg.E, cfg.cf, cfg.subseq)
    return r


def _expert_rows_one_late(Xp, offsets, W_gu, W_down, dtype="bf16", mirror=True, rows=None):
    off = np.array(offsets, copy=True)
    off[:-1] = np.minimum(off[:-1] + 1, off[1:])
    return _orig["expert_ffn"](Xp, off, W_gu, W_down, dtype, mirror, rows)


def _unpermute_bwd_dw_from_next_slot(dout, Yp, row_of, w, *a, **k):
    """dw[t, k] = <dout[t], Yp[row_of[t, k + 1]]>: an off-by-one slot index."""
    r = _orig["unpermute_bwd"](dout, Yp, row_of, w, *a, **k)
    r["dw"] = _orig["unpermute_bwd"](dout, Yp, np.roll(row_of, -1, axis=1), w, *a, **k)["dw"]
    return r


def _softmax_without_max(logits):
    l = np.asarray(logits, dtype=np.float32)
    q = O.exp_f32(l)
    s = O.pairwise_sum_f32(q)[..., None]
    return (q / s).astype(np.float32)


def _round_bf16_truncating(v):
    m, e = np.frexp(np.asarray(v, dtype=np.float64))
    return np.ldexp(np.trunc(m * 256.0) / 256.0, e)


def _round_bf16_ties_away(v):
    m, e = np.frexp(np.asarray(v, dtype=np.float64))
    return np.ldexp(np.sign(m) * np.floor(np.abs(m) * 256.0 + 0.5) / 256.0, e)


def _route_bwd_db_from_dp(x, W_r, p, idx, prob, w, dw, renorm, w_sg=None, dz=None, mirror=True):
    """db_r summed from dp (before the softmax Jacobian) instead of dl."""
    r = _orig["route_bwd"](x, W_r, p, idx, prob, w, dw, renorm, w_sg, dz, mirror=mirror)
    dp = np.zeros_like(np.asarray(p, dtype=np.float64))
    np.put_along_axis(dp, idx.astype(np.int64), np.asarray(dw, dtype=np.float64), axis=1)
    r["db_r"] = O.f32_rounder(mirror)(dp.sum(axis=0))
    return r


def _unpermute_bwd_dz_without_sigmoid_slope(dout, Yp, row_of, w, Ys=None, z=None, *a, **k):
    r = _orig["unpermute_bwd"](dout, Yp, row_of, w, Ys, z, *a, **k)
    if Ys is not None:
        s = _orig["sigmoid"](z)
        r["dz"] = r["dz"] / (s * (1.0 - s))
    return r


def _build_map_padded_tokens_descending(idx, keep, E, C):
    T, K = idx.shape
    counts = np.zeros(E, dtype=np.int32)
    row_of = np.full((T, K), -1, dtype=np.int32)
    src_of = np.full(E * C, -1, dtype=np.int32)
    for t in range(T - 1, -1, -1):
        for k in range(K):
            if keep[t, k]:
                e = int(idx[t, k])
                row = e * C + int(counts[e])
                row_of[t, k] = row
                src_of[row] = t * K + k
                counts[e] += 1
    return counts, (np.arange(E + 1) * C).astype(np.int32), row_of, src_of


def _permute_padded_without_zero_fill(x, src_of, K):
    return x[np.maximum(src_of, 0) // K]


def _pairwise_sum_sequential(q):
    q = np.asarray(q, dtype=np.float32)
    acc = np.zeros(q.shape[:-1], dtype=np.float32)
    for i in range(q.shape[-1]):
        acc = (acc + q[..., i]).astype(np.float32)
    return acc


def _fsplit_gate_rows_twice(W_gu, W_down, shards, s):
    F = W_gu.shape[1] // 2
    Fl = F // shards
    cols = np.arange(s * Fl, (s + 1) * Fl)
    return W_gu[:, np.concatenate([cols, cols])], W_down[:, :, cols]


def _padded_capacity_unclipped(T, S, K, E, cf):
    S = S if 0 < S < T else T
    return sum(O.capacity(cf, min(S, T - lo), K, E) for lo in range(0, T, S))


def _swiglu_h_from_rounded_gu(X, Wgu, Wdown, rnd):
    F = Wgu.shape[0] // 2
    Acc = X @ Wgu.T
    G, U = rnd(Acc[:, :F]), rnd(Acc[:, F:])
    H = rnd(O.silu(G) * U)
    return rnd(Acc), H, rnd(H @ Wdown.T)


def _swiglu_y_from_unrounded_h(X, Wgu, Wdown, rnd):
    F = Wgu.shape[0] // 2
    Acc = X @ Wgu.T
    h = O.silu(Acc[:, :F]) * Acc[:, F:]
    return rnd(Acc), rnd(h), rnd(h @ Wdown.T)


def _swiglu_bwd_rounding(round_dh=False, dx_from_unrounded=False):
    def f(dY, X, A, H, Wgu, Wdown, rnd, r32):
        F = Wgu.shape[0] // 2
        dH = dY @ Wdown
        if round_dh:
            dH = rnd(dH)
        G, U = A[:, :F], A[:, F:]
        sg = 1.0 / (1.0 + np.exp(-G))
        dA_raw = np.concatenate([dH * U * sg * (1.0 + G * (1.0 - sg)), dH * G * sg], axis=1)
        dA = rnd(dA_raw)
        dX = r32((dA_raw if dx_from_unrounded else dA) @ Wgu)
        return dX, r32(dY.T @ H), r32(dA.T @ X), dA
    return f


def _unpermute_rounds_each_term(Yp, row_of, w, Ys=None, z=None, dtype="bf16", mirror=True,
                                tokens=None):
    rnd = O.act_rounder(dtype, mirror)
    T, K = row_of.shape
    acc = np.zeros((T, Yp.shape[1]))
    for k in range(K):
        r = row_of[:, k]
        m = r >= 0
        acc[m] += rnd(np.asarray(w, dtype=np.float64)[m, k][:, None] * Yp[r[m]])
    return rnd(acc)


def _unpermute_bwd_dyp_unrounded(dout, Yp, row_of, w, *a, **k):
    r = _orig["unpermute_bwd"](dout, Yp, row_of, w, *a, **dict(k, mirror=False))
    ref = _orig["unpermute_bwd"](dout, Yp, row_of, w, *a, **k)
    return dict(ref, dYp=r["dYp"])


# name: (attribute -> replacement, the pin that must fail)
MUTANTS = {
    "silu dropped (H = G*U)": (
        {"silu": lambda g: g}, PL.test_single_expert_is_dense_swiglu),
    "gate and up rows swapped": (
        {"swiglu_group": _swiglu_gate_up_swapped}, PL.test_single_expert_is_dense_swiglu),
    "SwiGLU backward: sign of the G(1-s) term": (
        {"swiglu_group_bwd": _swiglu_bwd(sign_dg=-1.0)},
        lambda: PL.test_backward_matches_finite_differences("drop_renorm")),
    "SwiGLU backward: dU without the factor G": (
        {"swiglu_group_bwd": _swiglu_bwd(keep_g_in_du=False)},
        lambda: PL.test_backward_matches_finite_differences("no_renorm")),
    "router backward: renormalisation term dropped": (
        {"route_bwd": _route_bwd_without_renorm_term},
        lambda: PL.test_backward_matches_finite_differences("drop_renorm")),
    "router backward: softmax Jacobian sign": (
        {"route_bwd": _route_bwd_jacobian_sign},
        lambda: PL.test_backward_matches_finite_differences("no_renorm")),
    "router backward: shared gate term missing from dx": (
        {"route_bwd": _route_bwd_without_gate_term_in_dx},
        lambda: PL.test_backward_matches_finite_differences("dropless_shared_bias")),
    "un-permute backward: dYp not weighted by w": (
        {"unpermute_bwd": lambda dout, Yp, row_of, w, *a, **k: dict(
            _orig["unpermute_bwd"](dout, Yp, row_of, np.ones_like(np.asarray(w)), *a, **k),
            dw=_orig["unpermute_bwd"](dout, Yp, row_of, w, *a, **k)["dw"])},
        lambda: PL.test_backward_matches_finite_differences("no_renorm")),
    "permute backward: router dx addend dropped": (
        {"permute_bwd": lambda dXp, row_of, dx_add=None, mirror=True:
            _orig["permute_bwd"](dXp, row_of, None, mirror)},
        lambda: PL.test_backward_matches_finite_differences("no_renorm")),
    "shared gate: 1 - sigmoid": (
        {"sigmoid": lambda z: 1.0 - _orig["sigmoid"](z)}, PL.test_shared_expert_adds_gated_dense_ffn),
    "router bias dropped": (
        {"router_logits": lambda x, W_r, b_r=None, mirror=True, chunk=4096:
            _orig["router_logits"](x, W_r, None, mirror, chunk)},
        PL.test_all_experts_is_dense_mixture),
    "combine ignores the weights": (
        {"unpermute": lambda Yp, row_of, w, *a, **k:
            _orig["unpermute"](Yp, row_of, np.ones_like(np.asarray(w)), *a, **k)},
        lambda: PL.test_identity_experts_give_k_times_x(2)),
    "no renormalisation": (
        {"renorm_weights": lambda prob, renorm: np.array(prob, copy=True)}, PR.test_renorm_weights),
    "Top-K ties to the higher expert": (
        {"topk": _topk_ties_to_higher_index}, lambda: PR.test_topk_brute_force(8, 2, True)),
    "capacity: floor for ceil": (
        {"capacity": lambda cf, S_j, K, E: int(math.floor(float(np.float32(cf)) * S_j * K / E))},
        PR.test_capacity_formula),
    "capacity: ties to the higher token": (
        {"capacity_keep": _capacity_keep(ties_to_higher_token=True)},
        lambda: PR.test_capacity_brute_force(48, 4, 2, 16, 1.0, True)),
    "capacity: short last sub-sequence gets the full cap": (
        {"capacity_keep": _capacity_keep(full_cap_for_short_block=True)},
        PR.test_capacity_short_last_subsequence_uses_its_own_length),
    "capacity ranked by the renormalised weight": (
        {"route": _route_ranks_capacity_by_weight}, PR.test_route_composes_the_pinned_steps),
    "map: tokens descending inside an expert": (
        {"build_map": _build_map_tokens_descending}, lambda: PR.test_map_invariants(False)),
    "padded capacity not clipped to the sub-sequence": (
        {"padded_capacity": _padded_capacity_unclipped}, PR.test_padded_capacity_formula),
    "exp: Cody-Waite low part dropped": (
        {"LN2_LO": np.float32(0.0)}, PS.test_exp_within_two_ulp_of_double_exp),
    "exp: polynomial truncated after r^5": (
        {"TAYLOR": O.TAYLOR[:6] + [np.float32(0.0), np.float32(0.0)]},
        PS.test_exp_within_two_ulp_of_double_exp),
    "expert rows start one row late": (
        {"expert_ffn": _expert_rows_one_late}, PL.test_single_expert_is_dense_swiglu),
    "un-permute backward: dw from the neighbouring slot's row": (
        {"unpermute_bwd": _unpermute_bwd_dw_from_next_slot},
        lambda: PL.test_backward_matches_finite_differences("no_renorm")),
    "softmax without the max subtraction": (
        {"softmax_f32": _softmax_without_max}, PS.test_softmax_bits_invariant_under_a_shift_of_the_logits),
    "bf16 decode shifted by 15 bits": (
        {"decode": lambda a: ((a.astype(np.uint32) << np.uint32(15)).view(np.float32).astype(np.float64)
                              if a.dtype == np.uint16 else np.asarray(a, dtype=np.float64))},
        PV.test_decode_bf16_bits_matches_torch),
    "bf16 rounding truncates": (
        {"round_bf16": _round_bf16_truncating}, PV.test_round_bf16_matches_torch_rne),
    "bf16 rounding ties away from zero": (
        {"round_bf16": _round_bf16_ties_away}, PV.test_round_bf16_matches_torch_rne),
    "capacity from the double, not the fp32, capacity factor": (
        {"capacity": lambda cf, S_j, K, E: int(math.ceil(float(cf) * S_j * K / E))},
        PV.test_capacity_takes_the_fp32_capacity_factor),
    "router backward: db_r summed before the softmax Jacobian": (
        {"route_bwd": _route_bwd_db_from_dp},
        lambda: PL.test_backward_matches_finite_differences("dropless_shared_bias")),
    "shared gate backward: dz without the sigmoid slope": (
        {"unpermute_bwd": _unpermute_bwd_dz_without_sigmoid_slope},
        lambda: PL.test_backward_matches_finite_differences("dropless_shared_bias")),
    "padded map: tokens descending inside an expert": (
        {"build_map_padded": _build_map_padded_tokens_descending},
        PR.test_padded_map_is_the_compact_map_with_fixed_strides),
    "padded permute: padding rows not zeroed": (
        {"permute_padded": _permute_padded_without_zero_fill},
        PR.test_padded_map_is_the_compact_map_with_fixed_strides),
    "softmax sum left to right": (
        {"pairwise_sum_f32": _pairwise_sum_sequential}, PS.test_pairwise_sum_order),
    "ETP shard: gate rows used for up": (
        {"fsplit_weights": _fsplit_gate_rows_twice},
        lambda: PL.test_fsplit_is_the_unsplit_ffn_in_exact_arithmetic(2)),
    "SwiGLU: H from the bf16-rounded G and U": (
        {"swiglu_group": _swiglu_h_from_rounded_gu}, PRP.test_forward_rounding_points),
    "SwiGLU: Yp from the unrounded H": (
        {"swiglu_group": _swiglu_y_from_unrounded_h}, PRP.test_forward_rounding_points),
    "SwiGLU backward: dH rounded to bf16 before dA": (
        {"swiglu_group_bwd": _swiglu_bwd_rounding(round_dh=True)}, PRP.test_backward_rounding_points),
    "SwiGLU backward: dXp from the unrounded dA": (
        {"swiglu_group_bwd": _swiglu_bwd_rounding(dx_from_unrounded=True)},
        PRP.test_backward_rounding_points),
    "combine: every weighted term rounded": (
        {"unpermute": _unpermute_rounds_each_term}, PRP.test_combine_rounds_once_after_the_sum),
    "un-permute backward: dYp not rounded": (
        {"unpermute_bwd": _unpermute_bwd_dyp_unrounded},
        PRP.test_unpermute_bwd_rounds_dyp_to_bf16_and_keeps_dw_fp32),
    "permute backward: dx rounded to bf16": (
        {"permute_bwd": lambda dXp, row_of, dx_add=None, mirror=True:
            O.round_bf16(_orig["permute_bwd"](dXp, row_of, dx_add, mirror))},
        PRP.test_permute_bwd_sums_in_fp32),
    "ETP partials summed in reverse shard order": (
        {"sum_partials": lambda parts, mirror=True: _orig["sum_partials"](parts[::-1], mirror)},
        PL.test_sum_partials_adds_in_shard_order_in_fp32),
}


@pytest.mark.filterwarnings("ignore::RuntimeWarning")   # mutants may overflow
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pin_catches_planted_mistake(name, monkeypatch):
    patches, pin = MUTANTS[name]
    for attr, value in patches.items():
        assert hasattr(O, attr), attr
        monkeypatch.setattr(O, attr, value)
    with pytest.raises(AssertionError):
        pin()
