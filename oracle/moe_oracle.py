"""CPU oracle: a plain, slow, obviously correct MoE layer in numpy (fp64).

TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's CPU
baseline are the only callers. It shares no code with the CUDA library.

Sources. The method is the token-level dispatcher of "MoE Parallel Folding:
Heterogeneous Parallelism Mappings for Efficient Large-Scale MoE Model Training
with Megatron Core" (arXiv 2504.14960), as described by its study-notes page:
  [notes/prereq]   prerequisites: Top-K gating and the capacity factor;
  [notes/method]   method overview: the router assigns each token its Top-K
                   experts, a permutation makes each expert's tokens
                   contiguous, the experts' FFN runs, an un-permutation
                   restores token order; drop and dropless routing; the
                   backward swaps each step for its counterpart;
  [notes/modules]  key modules: the dispatcher handles token dropping and
                   dropless routing and dynamic shapes; sub-sequence dropping
                   decides drops inside the local sub-sequence;
  [notes/setup]    setup and metrics: BF16, capacity factor 1 for the
                   token-drop benchmarks;
  [notes/qa]       Q&A: full- vs sub-sequence dropping;
  [quote 3.3]      quote of the paper's section 3.3 (Token Dispatcher):
                   sub-sequence dropping is the default;
and the paper's abstract (mlsanity paper page, "Abstract"), which states the
dispatcher supports token-dropping and dropless training.

The pages fix none of: the gating function, the FFN type, the capacity
formula, tie rules, rounding points. The readings used here are:
  * softmax over the E experts, then Top-K on the probabilities, ties to the
    lower expert index; combine weights renormalised over the K (optional);
  * SwiGLU experts: H = silu(x W_g^T) * (x W_u^T), y = H W_down^T, with
    W_gu = [W_g; W_u] stacked on rows;
  * capacity per (sub-sequence, expert) = ceil(CF * S_j * K / E), S_j the
    sub-sequence's actual length; sub-sequences are contiguous blocks of the
    flat token order; keep the highest-probability assignments (raw softmax p),
    ties to the lower token index; kept weights are not renormalised again;
  * permuted order: expert-major, token-ascending inside an expert, compact;
  * an optional shared expert adds sigmoid(x . w_sg) * SwiGLU_shared(x);
  * expert tensor parallelism (the F-split of an expert over a group, whose
    partial outputs a ReduceScatter-V sums): each shard's partial output is
    stored in the activation dtype, the partials are added in shard order
    with fp32 additions and rounded once; in the backward each shard's fp32
    dXp partial is added the same way.

Precision. Arithmetic is fp64 everywhere except the routing decision chain,
which both sides must take on identical bits: the softmax below is specified
operation by operation in fp32 (own exp from Cody-Waite range reduction and the
degree-7 Taylor polynomial, a fixed pairwise sum, IEEE division) and Top-K,
renormalisation and capacity work on those fp32 values. With mirror=True the
oracle also rounds to the activation dtype where the layer stores an
activation (A = [G|U], H, Yp, out, dYp, dA; fp32 for dXp, dx and weight
gradients); mirror=False keeps every value in fp64 and uses an fp64 softmax,
for finite-difference checks.
"""
from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# value helpers

def decode(a: np.ndarray) -> np.ndarray:
    """Input array -> float64. uint16 arrays hold bf16 bit patterns."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (8 significant bits), ties to
    even; returned as float64."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                  # v = m * 2**e, |m| in [0.5, 1)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def round_f32(v: np.ndarray) -> np.ndarray:
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


def act_rounder(dtype: str, mirror: bool):
    """Rounding applied where the layer stores an activation."""
    if not mirror:
        return lambda v: np.asarray(v, dtype=np.float64)
    return round_bf16 if dtype == "bf16" else round_f32


def f32_rounder(mirror: bool):
    if not mirror:
        return lambda v: np.asarray(v, dtype=np.float64)
    return round_f32


# --------------------------------------------------------------------------
# a1: router logits  [notes/method: the router assigns Top-K experts]

def router_logits(x, W_r, b_r=None, mirror=True, chunk=4096):
    """l[t,e] = sum_j x[t,j] W_r[e,j] (+ b_r[e]), accumulated in fp64 and
    stored as fp32 (mirror) or kept in fp64."""
    Wr = decode(W_r)
    T = x.shape[0]
    out = np.empty((T, Wr.shape[0]), dtype=np.float64)
    for lo in range(0, T, chunk):
        out[lo:lo + chunk] = decode(x[lo:lo + chunk]) @ Wr.T
    if b_r is not None:
        out += np.asarray(b_r, dtype=np.float64)[None, :]
    return f32_rounder(mirror)(out)


def gate_logit(x, w_sg, mirror=True, chunk=4096):
    """Shared-expert gate logit z[t] = x[t] . w_sg (fp64 -> fp32)."""
    w = decode(w_sg)
    T = x.shape[0]
    z = np.empty(T, dtype=np.float64)
    for lo in range(0, T, chunk):
        z[lo:lo + chunk] = decode(x[lo:lo + chunk]) @ w
    return f32_rounder(mirror)(z)


# --------------------------------------------------------------------------
# a2: softmax, specified in fp32 so that two implementations agree bit for bit

_F = np.float32
LOG2E = _F(1.4426950408889634)          # log2(e) rounded to fp32
LN2_HI = _F(0.693359375)                # 355/512: n*LN2_HI is exact for |n| < 2**15
LN2_LO = _F(math.log(2.0) - 0.693359375)  # ln2 - LN2_HI, rounded to fp32
TAYLOR = [_F(1.0 / math.factorial(k)) for k in range(8)]   # 1/k!, k = 0..7


def exp_f32(u: np.ndarray) -> np.ndarray:
    """e**u for fp32 u <= 0, every operation an fp32 rounding (no fused
    multiply-add):  n = rint(u*log2e);  r = (u - n*LN2_HI) - n*LN2_LO;
    P = Horner of sum_{k<=7} r**k/k! (multiply, then add);  result P * 2**n,
    or 0 when n < -125 (below the normal range)."""
    u = np.asarray(u, dtype=np.float32)
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        n = np.rint(u * LOG2E).astype(np.float32)
        r = (u - n * LN2_HI) - n * LN2_LO
        p = TAYLOR[7]
        for k in range(6, -1, -1):
            p = (p * r).astype(np.float32) + TAYLOR[k]
        p = np.asarray(p, dtype=np.float32)
        ni = n.astype(np.int32)
        scale = ((np.clip(ni, -125, 127) + 127).astype(np.uint32) << np.uint32(23)).view(np.float32)
        out = (p * scale).astype(np.float32)
    return np.where(ni < -125, np.float32(0.0), out).astype(np.float32)


def pairwise_sum_f32(q: np.ndarray) -> np.ndarray:
    """Sum over the last axis: pad to a power of two with zeros, then
    v[i] += v[i + h] for h = P/2, P/4, ..., 1 (fp32)."""
    q = np.asarray(q, dtype=np.float32)
    E = q.shape[-1]
    P = 1
    while P < E:
        P *= 2
    v = np.zeros(q.shape[:-1] + (P,), dtype=np.float32)
    v[..., :E] = q
    h = P // 2
    while h >= 1:
        v[..., :h] = v[..., :h] + v[..., h:2 * h]
        h //= 2
    return v[..., 0]


def softmax_f32(logits: np.ndarray) -> np.ndarray:
    """p = q / s with m = max_e l, q_e = exp_f32(l_e - m), s = pairwise sum of
    q, each step in fp32 (division correctly rounded)."""
    l = np.asarray(logits, dtype=np.float32)
    m = l.max(axis=-1, keepdims=True)
    q = exp_f32((l - m).astype(np.float32))
    s = pairwise_sum_f32(q)[..., None]
    return (q / s).astype(np.float32)


def softmax_f64(logits: np.ndarray) -> np.ndarray:
    l = np.asarray(logits, dtype=np.float64)
    q = np.exp(l - l.max(axis=-1, keepdims=True))
    return q / q.sum(axis=-1, keepdims=True)


# --------------------------------------------------------------------------
# a2: Top-K and renormalisation  [notes/prereq, notes/method: Top-K gating]

def topk(p: np.ndarray, K: int):
    """K rounds of arg-max over the not-yet-chosen experts; ties go to the
    lower expert index (argmax returns the first maximum). Returns
    (idx [T,K] int32 in selection order, prob [T,K] = p at idx)."""
    work = np.array(p, copy=True)
    T = work.shape[0]
    idx = np.empty((T, K), dtype=np.int32)
    rows = np.arange(T)
    for k in range(K):
        j = np.argmax(work, axis=1)
        idx[:, k] = j
        work[rows, j] = -np.inf
    prob = np.take_along_axis(np.asarray(p), idx.astype(np.int64), axis=1)
    return idx, prob


def renorm_weights(prob: np.ndarray, renorm: bool) -> np.ndarray:
    """w_k = prob_k / Z with Z = prob_0 + prob_1 + ... in slot order, in the
    dtype of prob (fp32 ops for the fp32 chain); w = prob without renorm."""
    if not renorm:
        return np.array(prob, copy=True)
    Z = prob[:, 0].copy()
    for k in range(1, prob.shape[1]):
        Z = Z + prob[:, k]
    return prob / Z[:, None]


# --------------------------------------------------------------------------
# a3: capacity-factor dropping per sub-sequence
# [notes/prereq: capacity factor; notes/modules, notes/qa, quote 3.3:
#  drops are decided inside each local sub-sequence]

def capacity(cf: float, S_j: int, K: int, E: int) -> int:
    """ceil(CF * S_j * K / E), evaluated in double from the fp32 CF, left to
    right."""
    return int(math.ceil(float(np.float32(cf)) * S_j * K / E))


def capacity_keep(idx: np.ndarray, prob: np.ndarray, E: int, cf: float, S: int):
    """keep[t,k] = 1 when assignment (t,k) is among the top-cap assignments of
    its (sub-sequence, expert) under the order (prob descending, token index
    ascending); sub-sequence j is tokens [jS, min((j+1)S, T))."""
    T, K = idx.shape
    keep = np.zeros((T, K), dtype=np.uint8)
    S = S if S > 0 else T
    for lo in range(0, T, S):
        hi = min(T, lo + S)
        cap = capacity(cf, hi - lo, K, E)
        sub_idx = idx[lo:hi]
        sub_p = prob[lo:hi]
        for e in range(E):
            t_loc, k = np.nonzero(sub_idx == e)
            if t_loc.size == 0:
                continue
            pe = sub_p[t_loc, k]
            order = np.lexsort((t_loc, -pe.astype(np.float64)))
            chosen = order[:cap]
            keep[lo + t_loc[chosen], k[chosen]] = 1
    return keep


# --------------------------------------------------------------------------
# a4: the permutation map  [notes/method: permutation makes each expert's
# tokens contiguous; notes/modules: dynamic shapes]

def build_map(idx: np.ndarray, keep: np.ndarray, E: int):
    """Expert-major, token-ascending order of the kept assignments.
    Returns counts [E], offsets [E+1], row_of [T,K] (-1 when dropped),
    src_of [n_kept] (= t*K + k of each permuted row), n_kept."""
    T, K = idx.shape
    t, k = np.nonzero(keep)
    e = idx[t, k]
    order = np.lexsort((t, e))
    t, k, e = t[order], k[order], e[order]
    counts = np.bincount(e, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    n_kept = int(offsets[E])
    row_of = np.full((T, K), -1, dtype=np.int32)
    row_of[t, k] = np.arange(n_kept, dtype=np.int32)
    src_of = (t * K + k).astype(np.int32)
    return counts, offsets, row_of, src_of, n_kept


# --------------------------------------------------------------------------
# a5: permute  [notes/method]

def padded_capacity(T: int, S: int, K: int, E: int, cf: float) -> int:
    """Rows per expert of the GShard-style fixed layout: the most the
    capacity rule can keep for one expert, summed over the sub-sequences;
    an expert takes at most one slot per token, so min(cap_j, S_j)."""
    S = S if 0 < S < T else T
    return sum(min(capacity(cf, min(S, T - lo), K, E), min(S, T - lo)) for lo in range(0, T, S))


def build_map_padded(idx: np.ndarray, keep: np.ndarray, E: int, C: int):
    """Fixed [E, C] layout [notes/modules, Q&A: capacity bounds each expert's
    tokens, so buffers can be fixed-size]: expert e owns rows [eC, (e+1)C),
    its kept assignments first in token order, padding after.
    Returns counts [E], offsets [E+1] = e*C, row_of [T,K] (-1 dropped),
    src_of [E*C] (-1 on padding rows)."""
    T, K = idx.shape
    counts = np.zeros(E, dtype=np.int32)
    row_of = np.full((T, K), -1, dtype=np.int32)
    src_of = np.full(E * C, -1, dtype=np.int32)
    for t in range(T):
        for k in range(K):
            if keep[t, k]:
                e = int(idx[t, k])
                if counts[e] >= C:
                    raise ValueError("more kept rows than the padded capacity")
                row = e * C + int(counts[e])
                row_of[t, k] = row
                src_of[row] = t * K + k
                counts[e] += 1
    offsets = (np.arange(E + 1) * C).astype(np.int32)
    return counts, offsets, row_of, src_of


def permute_padded(x: np.ndarray, src_of: np.ndarray, K: int) -> np.ndarray:
    """Xp[row] = x[src_of[row] // K], zero on padding rows (src_of < 0)."""
    Xp = np.zeros((src_of.shape[0],) + x.shape[1:], dtype=x.dtype)
    m = src_of >= 0
    Xp[m] = x[src_of[m] // K]
    return Xp


def permute(x: np.ndarray, src_of: np.ndarray, K: int) -> np.ndarray:
    """Xp[row] = x[src_of[row] // K] (an exact copy; same dtype as x)."""
    return x[src_of // K]


# --------------------------------------------------------------------------
# a6/a7: SwiGLU expert FFN per expert group  [notes/method: expert FFN]

def silu(g):
    return g / (1.0 + np.exp(-g))


def swiglu_group(X, Wgu, Wdown, rnd):
    """One expert on its rows: G|U = X Wgu^T, H = silu(G)*U, Y = H Wdown^T.
    X, Wgu, Wdown are fp64 values; rnd is the activation rounding.
    Returns (A = rnd([G|U]), H = rnd(silu(G)*U from unrounded G, U),
    Y = rnd(H Wdown^T))."""
    F = Wgu.shape[0] // 2
    Acc = X @ Wgu.T
    G, U = Acc[:, :F], Acc[:, F:]
    H = rnd(silu(G) * U)
    Y = rnd(H @ Wdown.T)
    return rnd(Acc), H, Y


def expert_ffn(Xp, offsets, W_gu, W_down, dtype="bf16", mirror=True, rows=None):
    """Grouped SwiGLU FFN over the permuted rows.
    Xp [n,d] (input dtype), offsets [E+1]; W_gu [E,2F,d]; W_down [E,d,F].
    rows: optional sorted array of permuted-row indices to evaluate (the
    others are left as NaN) for sampled checks of large layers.
    Returns A_save [n,2F], H [n,F], Yp [n,d] as fp64 values."""
    rnd = act_rounder(dtype, mirror)
    n = Xp.shape[0]
    E = W_gu.shape[0]
    F = W_gu.shape[1] // 2
    d = W_gu.shape[2]
    A = np.full((n, 2 * F), np.nan)
    H = np.full((n, F), np.nan)
    Y = np.full((n, d), np.nan)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        r = np.arange(lo, hi) if rows is None else rows[(rows >= lo) & (rows < hi)]
        if r.size == 0:
            continue
        a, h, y = swiglu_group(decode(Xp[r]), decode(W_gu[e]), decode(W_down[e]), rnd)
        A[r], H[r], Y[r] = a, h, y
    return A, H, Y


# --------------------------------------------------------------------------
# f4: the expert FFN F-split over an expert-tensor-parallel group
#     [notes/method: ETP shards the expert's FFN dimension over ranks; a
#      ReduceScatter-V sums the partial outputs]

def fsplit_weights(W_gu, W_down, shards: int, s: int):
    """Shard s of `shards`: gate rows [s F/P, (s+1) F/P) and the same up rows
    of W_gu [E,2F,d] (stacked gate then up, as in the full layout), and the
    matching columns of W_down [E,d,F]."""
    F = W_gu.shape[1] // 2
    Fl = F // shards
    cols = np.arange(s * Fl, (s + 1) * Fl)
    return W_gu[:, np.concatenate([cols, F + cols])], W_down[:, :, cols]


def sum_partials(parts, mirror=True):
    """Sum of shard partials in shard order; with mirror every addition is an
    fp32 addition (the partials are fp32-representable values)."""
    r32 = f32_rounder(mirror)
    acc = np.asarray(parts[0], dtype=np.float64)
    for p in parts[1:]:
        acc = r32(acc + np.asarray(p, dtype=np.float64))
    return acc


def expert_ffn_fsplit(Xp, offsets, W_gu, W_down, shards: int, dtype="bf16", mirror=True):
    """Grouped SwiGLU FFN with F split into `shards`: every shard is a full
    grouped FFN on its gate/up rows and W_down columns; its partial output
    is stored in the activation dtype (the partials a ReduceScatter-V adds);
    Yp = rnd(sum of the partials in shard order, fp32 additions). A_save and
    H are the shards' columns put back in the full layout (SwiGLU acts per
    column, so they equal the unsplit ones)."""
    rnd = act_rounder(dtype, mirror)
    F = W_gu.shape[1] // 2
    Fl = F // shards
    n = Xp.shape[0]
    A = np.full((n, 2 * F), np.nan)
    H = np.full((n, F), np.nan)
    parts = []
    for s in range(shards):
        Wg, Wd = fsplit_weights(W_gu, W_down, shards, s)
        a, h, y = expert_ffn(Xp, offsets, Wg, Wd, dtype, mirror)
        cols = np.arange(s * Fl, (s + 1) * Fl)
        A[:, cols], A[:, F + cols], H[:, cols] = a[:, :Fl], a[:, Fl:], h
        parts.append(y)
    return A, H, rnd(sum_partials(parts, mirror))


# --------------------------------------------------------------------------
# a9: un-permute and combine  [notes/method: un-permutation restores order]

def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))


def unpermute(Yp, row_of, w, Ys=None, z=None, dtype="bf16", mirror=True, tokens=None):
    """out[t] = rnd( sum_{kept k, slot order} w[t,k] * Yp[row_of[t,k]]
    (+ sigmoid(z[t]) * Ys[t]) ), summed in fp64. Dropped slots add nothing;
    a token with no kept slot and no shared expert outputs 0.
    Yp, Ys are fp64 values; tokens selects a subset of tokens."""
    rnd = act_rounder(dtype, mirror)
    T, K = row_of.shape
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    d = Yp.shape[1]
    acc = np.zeros((tok.size, d))
    for k in range(K):
        r = row_of[tok, k]
        m = r >= 0
        acc[m] += np.asarray(w, dtype=np.float64)[tok[m], k][:, None] * Yp[r[m]]
    if Ys is not None:
        acc += sigmoid(z[tok])[:, None] * Ys[tok]
    return rnd(acc)


# --------------------------------------------------------------------------
# backward  [notes/method: the backward pass mirrors the forward chain]

def unpermute_bwd(dout, Yp, row_of, w, Ys=None, z=None, dtype="bf16", mirror=True):
    """a10. dYp[row_of[t,k]] = rnd(w[t,k] * dout[t]);
    dw[t,k] = <dout[t], Yp[row_of[t,k]]> (0 when dropped), fp32;
    shared: dYs = rnd(sigmoid(z) * dout), dz = s(1-s) <dout, Ys>, fp32."""
    rnd = act_rounder(dtype, mirror)
    r32 = f32_rounder(mirror)
    g = decode(dout)
    T, K = row_of.shape
    n = int(row_of.max()) + 1 if row_of.size and row_of.max() >= 0 else 0
    dYp = np.zeros((n, g.shape[1]))
    dw = np.zeros((T, K))
    w64 = np.asarray(w, dtype=np.float64)
    for k in range(K):
        r = row_of[:, k]
        m = r >= 0
        dYp[r[m]] = rnd(w64[m, k][:, None] * g[m])
        dw[m, k] = np.einsum("ij,ij->i", g[m], Yp[r[m]])
    out = {"dYp": dYp, "dw": r32(dw)}
    if Ys is not None:
        s = sigmoid(z)
        out["dYs"] = rnd(s[:, None] * g)
        out["dz"] = r32(s * (1.0 - s) * np.einsum("ij,ij->i", g, Ys))
    return out


def swiglu_group_bwd(dY, X, A, H, Wgu, Wdown, rnd, r32):
    """One expert's backward on its rows (fp64 values in, rounded outputs):
    dH = dY Wdown; with G|U = A and sg = sigmoid(G):
    dG = dH * U * sg * (1 + G (1 - sg)), dU = dH * G * sg, dA = rnd([dG|dU]);
    dX = r32(dA Wgu); dWdown = r32(dY^T H); dWgu = r32(dA^T X)."""
    F = Wgu.shape[0] // 2
    dH = dY @ Wdown
    G, U = A[:, :F], A[:, F:]
    sg = 1.0 / (1.0 + np.exp(-G))
    dG = dH * U * sg * (1.0 + G * (1.0 - sg))
    dU = dH * G * sg
    dA = rnd(np.concatenate([dG, dU], axis=1))
    return r32(dA @ Wgu), r32(dY.T @ H), r32(dA.T @ X), dA


def expert_ffn_bwd(dYp, Xp, A_save, H_save, offsets, W_gu, W_down,
                   dtype="bf16", mirror=True):
    """a11/a12 over all experts. dYp, A_save, H_save are fp64 values; Xp,
    W_gu, W_down are inputs. Returns dXp [n,d], dW_gu [E,2F,d],
    dW_down [E,d,F] (fp32 values), dA [n,2F]. An expert with no rows has
    zero weight gradients."""
    rnd = act_rounder(dtype, mirror)
    r32 = f32_rounder(mirror)
    E, twoF, d = W_gu.shape
    n = Xp.shape[0]
    dXp = np.zeros((n, d))
    dA = np.zeros((n, twoF))
    dWgu = np.zeros((E, twoF, d))
    dWd = np.zeros((E, d, twoF // 2))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        dX, dwd, dwgu, da = swiglu_group_bwd(dYp[lo:hi], decode(Xp[lo:hi]), A_save[lo:hi],
                                             H_save[lo:hi], decode(W_gu[e]),
                                             decode(W_down[e]), rnd, r32)
        dXp[lo:hi], dWd[e], dWgu[e], dA[lo:hi] = dX, dwd, dwgu, da
    return dXp, dWgu, dWd, dA


def expert_ffn_bwd_fsplit(dYp, Xp, A_save, H_save, offsets, W_gu, W_down, shards: int,
                         dtype="bf16", mirror=True):
    """Backward of expert_ffn_fsplit: every shard sees the whole dYp (the
    backward of the ReduceScatter-V is a gather); each shard's dXp partial is
    fp32 and dXp is their sum in shard order (fp32 additions); the weight
    gradients and dA are per shard, put back in the full layout."""
    E, twoF, d = W_gu.shape
    F = twoF // 2
    Fl = F // shards
    n = Xp.shape[0]
    dWgu = np.zeros((E, twoF, d))
    dWd = np.zeros((E, d, F))
    dA = np.zeros((n, twoF))
    parts = []
    for s in range(shards):
        cols = np.arange(s * Fl, (s + 1) * Fl)
        Wg, Wd = fsplit_weights(W_gu, W_down, shards, s)
        A_s = np.concatenate([A_save[:, cols], A_save[:, F + cols]], axis=1)
        dX, dwgu, dwd, da = expert_ffn_bwd(dYp, Xp, A_s, H_save[:, cols], offsets, Wg, Wd,
                                           dtype, mirror)
        parts.append(dX)
        dWgu[:, cols], dWgu[:, F + cols], dWd[:, :, cols] = dwgu[:, :Fl], dwgu[:, Fl:], dwd
        dA[:, cols], dA[:, F + cols] = da[:, :Fl], da[:, Fl:]
    return sum_partials(parts, mirror), dWgu, dWd, dA


def permute_bwd(dXp, row_of, dx_add=None, mirror=True):
    """a13. dx[t] = sum_{kept k} dXp[row_of[t,k]] (+ dx_add[t]), fp32."""
    T, K = row_of.shape
    dx = np.zeros((T, dXp.shape[1]))
    for k in range(K):
        r = row_of[:, k]
        m = r >= 0
        dx[m] += dXp[r[m]]
    if dx_add is not None:
        dx += dx_add
    return f32_rounder(mirror)(dx)


def route_bwd(x, W_r, p, idx, prob, w, dw, renorm, w_sg=None, dz=None, mirror=True):
    """a14. Gradient through renormalisation, softmax and the router GEMV.
    g = dw; with renorm (Z = sum_k prob_k): dp_j = (g_j - sum_k g_k w_k) / Z for
    j in the Top-K, else dp = g on the Top-K; dp = 0 off the Top-K.
    Softmax: dl_i = p_i (dp_i - sum_j p_j dp_j) over all E experts.
    dW_r = dl^T x; db_r = sum_t dl; dx_router = dl W_r (+ dz w_sg);
    dw_sg = dz^T x. All fp64, returned rounded to fp32 (mirror)."""
    r32 = f32_rounder(mirror)
    T, K = idx.shape
    p = np.asarray(p, dtype=np.float64)
    prob = np.asarray(prob, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    g = np.asarray(dw, dtype=np.float64)
    if renorm:
        Z = prob.sum(axis=1, keepdims=True)
        dpk = (g - (g * w).sum(axis=1, keepdims=True)) / Z
    else:
        dpk = g
    dp = np.zeros_like(p)
    np.put_along_axis(dp, idx.astype(np.int64), dpk, axis=1)
    dl = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    X = decode(x)
    Wr = decode(W_r)
    out = {"dlogits": dl, "dW_r": r32(dl.T @ X), "db_r": r32(dl.sum(axis=0))}
    dxr = dl @ Wr
    if dz is not None:
        dzv = np.asarray(dz, dtype=np.float64)
        dxr = dxr + dzv[:, None] * decode(w_sg)[None, :]
        out["dw_sg"] = r32(dzv @ X)
    out["dx_router"] = r32(dxr)
    return out


# --------------------------------------------------------------------------
# the whole layer

def route(cfg, inp, mirror=True, logits=None):
    """a1-a3: logits (or the given fp32 logits), softmax, Top-K, weights, keep."""
    if logits is None:
        logits = router_logits(inp["x"], inp["W_r"], inp.get("b_r"), mirror=mirror)
    if mirror:
        p = softmax_f32(logits.astype(np.float32))
    else:
        p = softmax_f64(logits)
    idx, prob = topk(p, cfg.K)
    w = renorm_weights(prob, cfg.renorm)
    if cfg.drop:
        keep = capacity_keep(idx, prob, cfg.E, cfg.cf, cfg.subseq)
    else:
        keep = np.ones_like(idx, dtype=np.uint8)
    return {"logits": logits, "p": p, "topk_idx": idx, "topk_prob": prob,
            "topk_w": w, "keep": keep}


def layer_forward(cfg, inp, mirror=True, logits=None, etp=1):
    """Full forward: route, drop, map, permute, expert FFN, (shared expert),
    un-permute with the weighted Top-K combine. etp > 1: the routed experts
    F-split into etp shards (expert_ffn_fsplit)."""
    r = route(cfg, inp, mirror=mirror, logits=logits)
    counts, offsets, row_of, src_of, n_kept = build_map(r["topk_idx"], r["keep"], cfg.E)
    Xp = permute(inp["x"], src_of, cfg.K)
    if etp > 1:
        A, H, Yp = expert_ffn_fsplit(Xp, offsets, inp["W_gu"], inp["W_down"], etp, cfg.dtype,
                                     mirror)
    else:
        A, H, Yp = expert_ffn(Xp, offsets, inp["W_gu"], inp["W_down"], cfg.dtype, mirror)
    out = dict(r, counts=counts, offsets=offsets, row_of=row_of, src_of=src_of,
               n_kept=n_kept, Xp=Xp, A_save=A, H_save=H, Yp=Yp)
    Ys = z = None
    if cfg.Fs:
        z = gate_logit(inp["x"], inp["w_sg"], mirror=mirror)
        off1 = np.array([0, cfg.T], dtype=np.int32)
        As, Hs, Ys = expert_ffn(inp["x"], off1, inp["Ws_gu"][None], inp["Ws_down"][None],
                                cfg.dtype, mirror)
        out.update(gate_logit=z, As_save=As, Hs_save=Hs, Ys=Ys)
    out["out"] = unpermute(Yp, row_of, r["topk_w"], Ys, z, cfg.dtype, mirror)
    return out


def layer_backward(cfg, inp, fwd, mirror=True, etp=1):
    """Full backward for upstream gradient inp['dout'] (etp as in layer_forward)."""
    ub = unpermute_bwd(inp["dout"], fwd["Yp"], fwd["row_of"], fwd["topk_w"],
                       fwd.get("Ys"), fwd.get("gate_logit"), cfg.dtype, mirror)
    if etp > 1:
        dXp, dWgu, dWd, dA = expert_ffn_bwd_fsplit(ub["dYp"], fwd["Xp"], fwd["A_save"],
                                                   fwd["H_save"], fwd["offsets"], inp["W_gu"],
                                                   inp["W_down"], etp, cfg.dtype, mirror)
    else:
        dXp, dWgu, dWd, dA = expert_ffn_bwd(ub["dYp"], fwd["Xp"], fwd["A_save"], fwd["H_save"],
                                            fwd["offsets"], inp["W_gu"], inp["W_down"],
                                            cfg.dtype, mirror)
    g = {"dYp": ub["dYp"], "dw": ub["dw"], "dXp": dXp, "dA": dA,
         "dW_gu": dWgu, "dW_down": dWd}
    dx_add = None
    if cfg.Fs:
        off1 = np.array([0, cfg.T], dtype=np.int32)
        dXs, dWsgu, dWsd, _ = expert_ffn_bwd(ub["dYs"], inp["x"], fwd["As_save"], fwd["Hs_save"],
                                             off1, inp["Ws_gu"][None], inp["Ws_down"][None],
                                             cfg.dtype, mirror)
        g.update(dYs=ub["dYs"], dz=ub["dz"], dXs=dXs, dWs_gu=dWsgu[0], dWs_down=dWsd[0])
        dx_add = dXs
    rb = route_bwd(inp["x"], inp["W_r"], fwd["p"], fwd["topk_idx"], fwd["topk_prob"],
                   fwd["topk_w"], ub["dw"], cfg.renorm, inp.get("w_sg"), ub.get("dz"),
                   mirror=mirror)
    g.update(dlogits=rb["dlogits"], dW_r=rb["dW_r"], db_r=rb["db_r"],
             dx_router=rb["dx_router"])
    if "dw_sg" in rb:
        g["dw_sg"] = rb["dw_sg"]
    dx_add = rb["dx_router"] if dx_add is None else dx_add + rb["dx_router"]
    g["dx"] = permute_bwd(dXp, fwd["row_of"], dx_add, mirror)
    return g


__all__ = [n for n in dir() if not n.startswith("_")]
