"""Benchmark of the single-GPU MoE layer (tokens/s) on synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

A step is one pass of the layer's hot path over one batch: route (logits,
softmax, Top-K, capacity), permute, grouped SwiGLU FFN, un-permute, and for
workloads that train the backward chain (un-permute backward, the experts'
dgrad and wgrad, router backward, permute backward). The default workload is
the Llama3-8x70B-shaped training layer, forward + backward: T=32768 tokens
(one 32K-token sequence), d=8192, E=8, Top-2, SwiGLU ffn 28672, dropless,
router logits scaled x3. `--config mixtral_8x22b` runs the forward-only
Mixtral-8x22B shape (T=8192, d=6144, E=8, Top-2, ffn 16384, capacity factor 1
per 4096-token sub-sequence).

Timing: W untimed warm-up steps, then K steps in one region bracketed by a
barrier and cudaDeviceSynchronize, timed with CUDA events on the launching
stream; the max over ranks is reported. Each step streams every expert weight
(11.3 GB on the default workload, 4.9 GB on the Mixtral-8x22B shape) through
the 129 MB L2, so no step starts with its inputs in L2. SM clocks and
throttle reasons are sampled with nvidia-smi during the timed region.
`roofline` is the routed experts' grouped GEMMs (forward, plus backward when
the workload trains) against the measured dense bf16 peak; `stages` gives
every call's event-timed duration and its fraction of its own roofline.

`e2e` repeats the measurement through the C ABI with host buffers: each step
copies its tokens (and, when it trains, the upstream gradient) from pinned
host memory to the device and its output (and dx) back, inside the timed
region; the copies run on a second stream with double buffers, overlapping
the neighbouring steps' compute.

`--impl reference` times the CPU oracle (the plain numpy definition of the
layer) on the host cores instead, on the same bounded sample as the
`cpu_baseline` of the GPU arm, extrapolated to the whole workload.

With N > 1 (under torchrun) every rank runs an independent replica on its
own batch (weak scaling); `value` is the tokens of all ranks / the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time


def _reference_arm_rank0_under_torchrun() -> bool:
    argv = sys.argv[1:]
    ref = "--impl=reference" in argv or any(
        a == "--impl" and i + 1 < len(argv) and argv[i + 1] == "reference" for i, a in enumerate(argv))
    return (ref and os.environ.get("RANK", "0") == "0"
            and int(os.environ.get("LOCAL_WORLD_SIZE", "1")) > 1)


# The reference arm's CPU oracle runs on rank 0 alone (the other ranks exit),
# so it may use every core of the process's affinity mask, although torchrun
# sets OMP_NUM_THREADS=1 for each rank; BLAS reads these when numpy loads.
if _reference_arm_rank0_under_torchrun():
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        os.environ[_v] = str(len(os.sched_getaffinity(0)))

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "llama3_8x70b"
METRIC = "MoE layer fwd+bwd tokens/s on 1 GB300; grouped-GEMM % BF16 peak; permute % HBM"


# ---------------------------------------------------------------------------
# multi-rank bookkeeping (host logic; also exercised by CPU tests with gloo)

def host_threads() -> int:
    """Threads the oracle's BLAS uses: the affinity mask, unless a thread
    count variable (read by BLAS when numpy loads) lowers it."""
    n = len(os.sched_getaffinity(0))
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return max(1, min(n, int(os.environ[v])))
    return n


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(tokens_per_rank: float, seconds_per_rank: float, world: int, dist=None) -> dict:
    """Whole-job throughput: all ranks' tokens / the slowest rank's time."""
    secs = seconds_per_rank
    toks = tokens_per_rank
    if world > 1 and dist is not None:
        import torch
        t = torch.tensor([secs], dtype=torch.float64)
        n = torch.tensor([toks], dtype=torch.float64)
        if dist.get_backend() == "nccl":
            t, n = t.cuda(), n.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        secs, toks = float(t.item()), float(n.item())
    else:
        toks = toks * world
    return {"seconds": secs, "tokens": toks, "value": toks / secs}


# ---------------------------------------------------------------------------
# clocks

SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + SMI_FIELDS,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)

ORACLE_TOKEN_SAMPLE = 4096       # tokens routed, mapped, permuted and combined
ORACLE_FFN_FLOP_BUDGET = 1e12    # fp64 work of the expert-FFN sample (fwd [+ bwd])


def oracle_throughput(cfg, inp) -> dict:
    """Time the oracle as it stands on a bounded sample of the workload and
    extrapolate to tokens/s of the whole workload.

    Sample: the routing (logits, softmax, Top-K, capacity), map, permute and
    combine on the first ORACLE_TOKEN_SAMPLE tokens (whole sub-sequences);
    the expert FFN (its weight decode and the per-expert group routine,
    forward and, for training workloads, the backward group routine: dgrad
    and wgrad) on the first rows of expert 0 (and 1, ...) up to
    ORACLE_FFN_FLOP_BUDGET of fp64 work; for training workloads the oracle's
    un-permute backward, router backward and permute backward on the token
    sample too. Each timed part is scaled by its own unit count (tokens,
    kept rows, experts' weight decode) to the whole workload. The same
    function serves the benchmark's `cpu_baseline` and `--impl reference`."""
    import dataclasses
    from oracle import moe_oracle as O
    T = min(cfg.T, max(ORACLE_TOKEN_SAMPLE, cfg.subseq if cfg.drop else 0))
    c = dataclasses.replace(cfg, T=T)
    sub = {k: (v[:T] if k in ("x", "dout") else v) for k, v in inp.items()}
    wall0 = time.perf_counter()
    t0 = time.perf_counter()
    r = O.route(c, sub)
    counts, offsets, row_of, src_of, n_kept = O.build_map(r["topk_idx"], r["keep"], c.E)
    Xp = O.permute(sub["x"], src_of, c.K)
    t_tok = time.perf_counter() - t0
    # expert FFN sample: fwd (+ bwd) group routines on rows of experts 0, 1, ...
    rnd, r32 = O.act_rounder(cfg.dtype, True), O.f32_rounder(True)
    row_flop = (18.0 if cfg.backward else 6.0) * cfg.d * cfg.F
    cap = max(16, int(ORACLE_FFN_FLOP_BUDGET / row_flop))
    t_decode, t_rows, n_rows, experts = 0.0, 0.0, 0, 0
    Yp = np.zeros((n_kept, c.d))
    for e in range(c.E):
        left = cap - n_rows
        rows = np.arange(min(left, int(counts[e])))
        if rows.size == 0:
            if left <= 0:
                break
            continue
        t1 = time.perf_counter()
        Wgu = O.decode(inp["W_gu"][e])
        Wd = O.decode(inp["W_down"][e])
        t2 = time.perf_counter()
        Xe = O.decode(Xp[rows + offsets[e]])
        A, H, Y = O.swiglu_group(Xe, Wgu, Wd, rnd)
        if cfg.backward:
            dY = rnd(O.decode(sub["dout"][src_of[rows + offsets[e]] // c.K]))
            O.swiglu_group_bwd(dY, Xe, A, H, Wgu, Wd, rnd, r32)
        t_rows += time.perf_counter() - t2
        t_decode += t2 - t1
        Yp[rows + offsets[e]] = Y
        n_rows += rows.size
        experts += 1
        del Wgu, Wd
    t3 = time.perf_counter()
    Ys = z = None
    if cfg.Fs:   # the shared expert's gate (its FFN is counted with the rows below)
        z = O.gate_logit(sub["x"], inp["w_sg"])
        Ys = np.zeros((T, c.d))
    O.unpermute(Yp, row_of, r["topk_w"], Ys, z, dtype=c.dtype)
    if cfg.backward:
        ub = O.unpermute_bwd(sub["dout"], Yp, row_of, r["topk_w"], Ys, z, dtype=c.dtype)
        rb = O.route_bwd(sub["x"], inp["W_r"], r["p"], r["topk_idx"], r["topk_prob"], r["topk_w"],
                         ub["dw"], c.renorm, inp.get("w_sg"), ub.get("dz"))
        O.permute_bwd(np.zeros((n_kept, c.d)), row_of, rb["dx_router"])
    t_tok += time.perf_counter() - t3
    wall = time.perf_counter() - wall0
    n_full = n_kept * cfg.T / T          # kept rows of the whole workload
    per_row = t_rows / n_rows
    total = (t_tok * cfg.T / T + cfg.E * t_decode / experts + per_row * n_full
             + (per_row * cfg.T * cfg.Fs / cfg.F if cfg.Fs else 0.0))
    busy = int(np.count_nonzero(counts))   # experts with rows in the token sample
    extrapolated = bool(T < cfg.T or n_rows < n_kept or experts < busy or cfg.Fs)
    return {"value": cfg.T / total, "unit": "tokens/s", "cores": host_threads(),
            "kind": "oracle", "extrapolated": extrapolated,
            "sample": (f"routing, map, permute and combine"
                       + (", un-permute, router and permute backward" if cfg.backward else "")
                       + f" on {T} of {cfg.T} tokens; expert FFN "
                       + ("forward + backward (dgrad, wgrad) " if cfg.backward else "forward ")
                       + f"on {n_rows} rows of {experts} expert(s) with their weight decode; "
                       f"each part scaled by its own units to {cfg.E} experts, {int(n_full)} "
                       f"kept rows and {cfg.T} tokens"
                       + (f" (the shared expert as {cfg.T} rows of width {cfg.Fs})" if cfg.Fs else "")),
            "sample_seconds": round(wall, 2),
            "blas": "numpy's BLAS for the oracle's fp64 matrix products"}


# ---------------------------------------------------------------------------

def code_text(path: str) -> str:
    """A source file without its // comments and blank lines: the key under
    which profiles/traffic.json records the counters of that code."""
    out = []
    for line in open(path):
        line = line.split("//", 1)[0].strip()
        if line:
            out.append(line)
    return "\n".join(out)


def route_algorithmic_bytes(cfg) -> int:
    """HBM bytes moe_route must move: x and the router weights (and the gate
    vector) read once; logits (and gate logits) written; Top-K index, prob,
    weight and keep flag written per slot."""
    b = 2 if cfg.dtype == "bf16" else 4
    n = cfg.T * cfg.d * b + cfg.E * cfg.d * b + cfg.T * cfg.E * 4
    if cfg.Fs:
        n += cfg.d * b + cfg.T * 4
    return n + cfg.T * cfg.K * (4 + 4 + 4 + 1)


def launches_per_step(cfg, etp: int = 1, gather: bool = False) -> int:
    """Kernels of this library launched per step (bf16 row-grouped GEMMs are a
    CTA-pair launch plus the single-CTA launch for half-empty last tiles)."""
    bf16 = cfg.dtype == "bf16"
    tc = bf16 and cfg.d % 64 == 0
    n = 1 if tc and (cfg.E > 16 or router_splits(cfg) > 1) else 0   # Top-K kernel after the router GEMM
    n += 1                                 # router GEMM (fp32: the fused router kernel)
    n += 2 if cfg.drop else 0              # capacity: bucket + select
    n += 3 if not gather else 2            # map count, map scatter, row copy (fused: no copy)
    fwd_gemm = (4 if bf16 else 2)          # gate/up and down, each pair + tails
    if gather:
        fwd_gemm = 3                       # gathered gate/up (no tails) + down + tails
    n += fwd_gemm * etp + (1 if etp > 1 else 0)   # routed experts per F-shard [+ partial sum]
    n += (4 if bf16 else 2) if cfg.Fs else 0      # shared expert
    n += 1                                 # un-permute
    if cfg.backward:
        gm = 2 if bf16 else 0              # group tensor maps of the two weight-gradient GEMMs
        # dH and dXp with their tail launches, dW_down, dW_gu
        bwd_gemm = (6 if bf16 else 4) + gm
        n += 1                             # un-permute backward
        n += bwd_gemm * etp + (1 if etp > 1 else 0)
        n += bwd_gemm if cfg.Fs else 0
        if bf16 and cfg.d % 256 == 0:      # router backward on the tensor cores:
            # dl, dl planes, [W_r planes + dx GEMM (+ tails) | dx kernel with the
            # shared-expert addend], group maps, dW_r GEMM, plane sum
            n += 6 + (0 if cfg.Fs else 2)
        else:
            n += 4                         # dl, dx, dW_r partials, reduce
        n += 1 if cfg.bias else 0          # db_r
        n += 1                             # permute backward
    return n


def router_splits(cfg) -> int:
    """K parts of the tensor-core router GEMM (as libmoe.so chooses them: as
    many as leave no SM idle on a 152-SM GB300, at most 4, >= 8 K blocks each,
    and at most what the even CTA's exchange buffer holds)."""
    mtiles = (cfg.T + 127) // 128
    kb = cfg.d // 64
    s = max(1, min(4, 152 // mtiles if mtiles else 1, kb // 8))
    per = (kb + s - 1) // s
    s = (kb + per - 1) // per
    gate = 1 if cfg.Fs else 0
    n = (cfg.E + 15) // 16 * 16 + 16 * gate
    stage = 16384 + (n * 128 + 1023) // 1024 * 1024
    room = 4 * 49152 + 32768 - 6 * stage
    return min(s, 1 + room // (128 * (cfg.E + gate) * 4))


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return
    from synthetic import make_inputs
    inp = make_inputs(cfg, need_backward=cfg.backward)
    vals = []
    for i in range(args.warmup + args.steps):
        r = oracle_throughput(cfg, inp)
        if i >= args.warmup:
            vals.append(r["value"])
    v = statistics.median(vals)
    cpu = dict(r, value=v)
    line = {"impl": "reference", "metric": metric_name(cfg), "value": v, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * cfg.T / v, "extrapolated": cpu["extrapolated"],
            "ms_per_step_note": ("the whole workload's time extrapolated from the timed sample"
                                 if cpu["extrapolated"] else "timed"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(cfg), "cpu_baseline": cpu,
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def metric_name(cfg) -> str:
    if cfg.backward:
        return METRIC
    return "MoE layer fwd tokens/s on 1 GB300; grouped-GEMM % BF16 peak; permute % HBM"


def workload_config(cfg) -> dict:
    return {"workload": (f"{cfg.name} MoE layer {'fwd+bwd' if cfg.backward else 'fwd'}: T={cfg.T}, "
                         f"d={cfg.d}, E={cfg.E}, top-{cfg.K}, SwiGLU ffn={cfg.F}"
                         + (f", shared ffn={cfg.Fs}" if cfg.Fs else "")
                         + (f", capacity factor {cfg.cf} per {cfg.subseq}-token sub-sequence"
                            if cfg.drop else ", dropless")),
            "tokens_per_step": cfg.T, "l2": "inputs larger than L2 (all expert weights stream every step)",
            "parallelism": "replicas"}


def stage_bytes(cfg, n_kept: int) -> dict:
    """Algorithmic HBM bytes of the bandwidth-bound calls (each tensor read or
    written once): activations b bytes per element, dXp / dx / dx_router fp32,
    row_of and topk_w 4 bytes per slot, keep 1."""
    b = 2 if cfg.dtype == "bf16" else 4
    T, d, K = cfg.T, cfg.d, cfg.K
    shared = (2 * T * d * b + 2 * T * 4) if cfg.Fs else 0   # Ys, dYs (or Ys twice); z, dz
    return {
        # x read, Xp written; topk_idx, keep read, row_of, src_of written
        "permute": T * d * b + n_kept * d * b + T * K * 9 + n_kept * 4,
        # Yp read, out written, row_of + topk_w read (+ Ys, z read)
        "unpermute": n_kept * d * b + T * d * b + T * K * 8 + ((T * d * b + T * 4) if cfg.Fs else 0),
        # dout read, Yp read, dYp written, row_of + topk_w read, dw written (+ Ys read, dYs written)
        "unpermute_bwd": T * d * b + 2 * n_kept * d * b + T * K * 12 + shared,
        # dXp read, dx_router read, dx written (fp32), row_of read
        "permute_bwd": n_kept * d * 4 + 2 * T * d * 4 + T * K * 4,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layout", default="compact", choices=["compact", "padded"],
                    help="permuted-row layout: compact (default) or the fixed [E, capacity] "
                         "layout (token-dropping workloads)")
    ap.add_argument("--etp", type=int, default=1,
                    help="run the routed experts F-split into this many shards (the arithmetic "
                         "of an expert-tensor-parallel group, on one GPU)")
    ap.add_argument("--gather", action="store_true",
                    help="forward-only bf16 workloads: fuse the permutation into the gate/up "
                         "GEMM (map-only moe_permute + moe_expert_ffn_gather)")
    ap.add_argument("--override", default="",
                    help="profiling cases only: comma-separated field=value changes to the "
                         "workload, e.g. T=4096,E=16 (the JSON line then names the changed shape)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    from synthetic import get_config, make_inputs
    cfg = get_config(args.config)
    if args.override:
        import dataclasses
        kv = dict(item.split("=", 1) for item in args.override.split(","))

        def cast(k, v):
            t = type(getattr(cfg, k))
            if t is bool:   # bool("False") is True: read the word
                if v.lower() not in ("0", "1", "false", "true"):
                    raise ValueError(f"{k}={v}: expected true/false")
                return v.lower() in ("1", "true")
            return t(v)
        typed = {k: cast(k, v) for k, v in kv.items()}
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}[{args.override}]", **typed)
    rank, world, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl != "reference" else "gloo")
    if args.impl == "reference":
        run_reference(args, cfg, rank, world)
        if dist is not None:
            dist.destroy_process_group()
        return

    import torch
    torch.cuda.set_device(local)
    from token_dispatch_expert_moe_gb300 import _lib as L
    from token_dispatch_expert_moe_gb300.layer import MoELayer, to_device
    import dataclasses
    cfg_r = dataclasses.replace(cfg, seed=cfg.seed + rank)   # each replica its own batch
    inp = make_inputs(cfg_r)
    w = {k: to_device(v) for k, v in inp.items() if k not in ("x", "dout")}
    layer = MoELayer(cfg_r, w, etp=args.etp, layout=args.layout, gather=args.gather)
    x = to_device(inp["x"])
    layer.x = x   # the backward reads the forward's tokens
    dout = to_device(inp["dout"]) if cfg.backward else None
    stream = torch.cuda.current_stream()

    FWD = ("route", "permute", "ffn", "shared_ffn", "unpermute")
    BWD = ("unpermute_bwd", "ffn_bwd", "shared_ffn_bwd", "route_bwd", "permute_bwd")
    recorded = []   # per timed step: {stage: (start event, end event)}

    def step(x, out, dout=None, dx=None, record=False):
        c, s, ws = cfg_r, layer.shape, layer.ws
        ev = {n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for n in FWD + BWD} if record else {}

        def mark(name, i):
            if record:
                ev[name][i].record(stream)

        layer.x = x
        mark("route", 0)
        L.moe_route(s, x, w["W_r"], w.get("b_r"), w.get("w_sg"), layer.logits, layer.gate_logit,
                    layer.topk_idx, layer.topk_prob, layer.topk_w, layer.keep, ws)
        mark("route", 1)
        mark("permute", 0)
        permute = L.moe_permute_padded if args.layout == "padded" else L.moe_permute
        permute(s, x, layer.topk_idx, layer.keep, layer.Xp, layer.row_of, layer.src_of,
                layer.counts, layer.offsets, ws)
        mark("permute", 1)
        mark("ffn", 0)
        layer.routed_ffn()
        mark("ffn", 1)
        if c.Fs:
            mark("shared_ffn", 0)
            L.moe_expert_ffn(layer.dtype_code, c.T, c.d, c.Fs, 1, layer.off1, x, w["Ws_gu"],
                             w["Ws_down"], layer.As, layer.Hs, layer.Ys, ws)
            mark("shared_ffn", 1)
        mark("unpermute", 0)
        L.moe_unpermute(s, layer.Yp, layer.row_of, layer.topk_w, layer.Ys, layer.gate_logit, out)
        mark("unpermute", 1)
        if c.backward:
            if dx is not None:
                layer.dx = dx
            layer.backward(dout, marks={n: ev[n] for n in BWD if n in ev})
        if record:
            recorded.append(ev)

    for _ in range(args.warmup):
        step(x, layer.out, dout)
    torch.cuda.synchronize()
    rc, info = L.moe_get_status(layer.ws)
    assert rc == 0, f"device status {rc} info {info:#x}"

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.4)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step(x, layer.out, dout, record=True)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    secs = t_start.elapsed_time(t_end) / 1e3
    agg = aggregate(cfg.T * args.steps, secs, world, dist)
    rc, info = L.moe_get_status(layer.ws)
    assert rc == 0, f"device status {rc} info {info:#x}"

    def stage_ms(name, skip_first=False):
        evs = [r[name] for r in recorded if name in r]
        if skip_first and len(evs) > 1:
            evs = evs[1:]
        vals = [a.elapsed_time(b) for a, b in evs]
        return statistics.mean(vals) if vals else None

    n_kept = int(layer.counts.sum().item())   # kept rows (the padded layout computes more)
    peaks = {}
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        peaks = json.load(open(pk_path))
    # a kernel timed inside a region of more than a second runs under the
    # power cap: the sustained peak; otherwise the burst figure
    long_region = secs > 1.0
    if "bf16_tflops" in peaks:
        bf16_peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
        peak_src = "measured, " + ("sustained" if long_region else "burst")
    else:
        bf16_peak = 1700.0 if long_region else 1900.0
        peak_src = "fallback, " + ("sustained" if long_region else "burst")
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    ffn_ms = stage_ms("ffn")
    ffn_bwd_ms = stage_ms("ffn_bwd") if cfg.backward else 0.0
    gemm_flops = (18.0 if cfg.backward else 6.0) * n_kept * cfg.d * cfg.F
    gemm_ms = ffn_ms + ffn_bwd_ms
    achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12
    sb = stage_bytes(cfg, n_kept)
    if args.gather:   # the permute call builds the map only; the GEMM reads x
        sb["permute"] = cfg.T * cfg.K * 9 + n_kept * 4
    route_bytes = route_algorithmic_bytes(cfg)
    traffic = None
    tr_key = f"{cfg.name}:grouped_gemm" + (":fwd_bwd" if cfg.backward else "")
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tr_path) and args.etp == 1 and args.layout == "compact":
        import hashlib
        ent = json.load(open(tr_path)).get(tr_key)
        src = os.path.join(ROOT, "token_dispatch_expert_moe_gb300", "csrc", "gemm_tc.cu")
        sha = hashlib.sha256(code_text(src).encode()).hexdigest()[:16]
        if ent is not None and ent.get("source_sha") == sha:   # counters of this very kernel
            traffic = ent["bytes"]

    # e2e through the C ABI with host buffers: every step copies its tokens
    # (and, when it trains, the upstream gradient) from pinned host memory and
    # reads its output (and dx) back; the copies run on a second stream,
    # double-buffered, so that they overlap the neighbouring steps' compute
    # (step i+1's inputs and step i-1's outputs move during step i).
    copy_stream = torch.cuda.Stream()
    ins = [("x", x)] + ([("dout", dout)] if cfg.backward else [])
    outs = [("out", layer.out)] + ([("dx", layer.dx)] if cfg.backward else [])
    dev_in = {n: [t, torch.empty_like(t)] for n, t in ins}
    dev_out = {n: [t, torch.empty_like(t)] for n, t in outs}
    host_in = {n: [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for _ in range(2)]
               for n, t in ins}
    for n, t in ins:
        for hb in host_in[n]:
            hb.copy_(t)
    host_out = {n: [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for _ in range(2)]
                for n, t in outs}
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(nsteps, start_event=None):
        if start_event is not None:
            copy_stream.wait_event(start_event)
        with torch.cuda.stream(copy_stream):
            for n in dev_in:
                dev_in[n][0].copy_(host_in[n][0], non_blocking=True)
            h2d_done[0].record(copy_stream)
        for i in range(nsteps):
            b = i % 2
            stream.wait_event(h2d_done[b])
            if i >= 2:
                stream.wait_event(d2h_done[b])   # buffers b read back two steps ago
            step(dev_in["x"][b], dev_out["out"][b],
                 dev_in["dout"][b] if cfg.backward else None,
                 dev_out["dx"][b] if cfg.backward else None)
            comp_done[b].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < nsteps:
                    nb = (i + 1) % 2
                    if i >= 1:
                        copy_stream.wait_event(comp_done[nb])   # step i-1 done with buffers nb
                    for n in dev_in:
                        dev_in[n][nb].copy_(host_in[n][nb], non_blocking=True)
                    h2d_done[nb].record(copy_stream)
                copy_stream.wait_event(comp_done[b])
                for n in dev_out:
                    host_out[n][b].copy_(dev_out[n][b], non_blocking=True)
                d2h_done[b].record(copy_stream)
        stream.wait_stream(copy_stream)

    e2e_run(2)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps, start_event=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e = aggregate(cfg.T * args.steps, e0.elapsed_time(e1) / 1e3, world, dist)
    h2d = sum(t.numel() * t.element_size() for _, t in ins)
    d2h = sum(t.numel() * t.element_size() for _, t in outs)

    if rank == 0:
        stages = {"n_kept": n_kept, "hbm_peak_GBps": hbm_peak, "bf16_peak_TFLOPs": bf16_peak}

        def hbm_stage(name, nbytes, ms):
            if ms is None:
                return
            stages[f"{name}_ms"] = ms
            stages[f"{name}_GBps"] = nbytes / ms / 1e6
            stages[f"{name}_hbm_frac"] = nbytes / ms / 1e6 / hbm_peak
            stages[f"{name}_bytes"] = nbytes

        # the stream is idle when the timed region starts, so the first
        # step's route also waits for the host's launches: later steps only
        hbm_stage("route", route_bytes, stage_ms("route", skip_first=True))
        hbm_stage("permute", sb["permute"], stage_ms("permute"))
        hbm_stage("unpermute", sb["unpermute"], stage_ms("unpermute"))
        fwd_tf = 6.0 * n_kept * cfg.d * cfg.F / (ffn_ms * 1e-3) / 1e12
        stages.update(ffn_ms=ffn_ms, ffn_tflops=fwd_tf, ffn_frac=fwd_tf / bf16_peak)
        if cfg.Fs:
            sh_ms = stage_ms("shared_ffn")
            stages.update(shared_ffn_ms=sh_ms,
                          shared_ffn_frac=6.0 * cfg.T * cfg.d * cfg.Fs / (sh_ms * 1e-3) / 1e12 / bf16_peak)
        if cfg.backward:
            bwd_tf = 12.0 * n_kept * cfg.d * cfg.F / (ffn_bwd_ms * 1e-3) / 1e12
            stages.update(ffn_bwd_ms=ffn_bwd_ms, ffn_bwd_tflops=bwd_tf, ffn_bwd_frac=bwd_tf / bf16_peak)
            hbm_stage("unpermute_bwd", sb["unpermute_bwd"], stage_ms("unpermute_bwd"))
            hbm_stage("permute_bwd", sb["permute_bwd"], stage_ms("permute_bwd"))
            stages["route_bwd_ms"] = stage_ms("route_bwd")
            if cfg.Fs:
                sh_ms = stage_ms("shared_ffn_bwd")
                stages.update(shared_ffn_bwd_ms=sh_ms,
                              shared_ffn_bwd_frac=12.0 * cfg.T * cfg.d * cfg.Fs / (sh_ms * 1e-3) / 1e12
                              / bf16_peak)
        line = {
            "metric": metric_name(cfg), "value": agg["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * agg["seconds"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic (seeded normal inputs, random-init weights)",
            "config": dict(workload_config(cfg), **({"etp_shards": args.etp} if args.etp > 1 else {}),
                           **({"layout": "padded"} if args.layout == "padded" else {}),
                           **({"permute": "fused into the gate/up GEMM"} if args.gather else {})),
            "clocks": clk,
            "e2e": {"value": e2e["value"], "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": (launches_per_step(cfg, args.etp, args.gather)
                             + (1 if args.layout == "padded" else 0)) * args.steps,
            "roofline": {"kernel": ("routed experts' grouped GEMMs, forward + backward (moe_expert_ffn: "
                                    "gate/up + down; moe_expert_ffn_bwd: dH, dXp, dW_down, dW_gu)"
                                    if cfg.backward else
                                    "routed experts' grouped GEMMs (moe_expert_ffn: gate/up + down)"),
                         "bound": "tensor", "achieved": achieved, "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": achieved / bf16_peak, "traffic": traffic,
                         "peak_source": peak_src,
                         "flops_per_launch": gemm_flops, "ms_per_launch": gemm_ms,
                         "launch": "one moe_expert_ffn call" + (" + one moe_expert_ffn_bwd call"
                                                                if cfg.backward else "")},
            "stages": stages,
        }
        if not args.no_cpu_baseline and world == 1:   # rank 0 at N = 1 only
            line["cpu_baseline"] = oracle_throughput(cfg, inp)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
