"""Benchmark of the single-GPU MoE layer (tokens/s) on synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

A step is one pass of the layer's hot path over one batch: route (logits,
softmax, Top-K, capacity), permute, grouped SwiGLU FFN, un-permute (+ the
backward chain for workloads that train). The default workload is the
Mixtral-8x22B-shaped layer: T=8192 tokens (2 x 4096), d=6144, E=8, Top-2,
SwiGLU ffn 16384, capacity factor 1 per 4096-token sub-sequence, forward.

Timing: W untimed warm-up steps, then K steps in one region bracketed by a
barrier and cudaDeviceSynchronize, timed with CUDA events on the launching
stream; the max over ranks is reported. Each step streams every expert weight
(4.9 GB for the default workload) through the 129 MB L2, so no step starts
with its inputs in L2. SM clocks and throttle reasons are sampled with
nvidia-smi during the timed region.

`e2e` repeats the measurement through the C ABI with host buffers: each step
copies its tokens from pinned host memory to the device and its output back,
inside the timed region; the copies run on a second stream with double
buffers, overlapping the neighbouring steps' compute.

`--impl reference` times the CPU oracle (the plain numpy definition of the
layer) on the host cores instead, on a bounded sample of the same workload.

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

DEFAULT_CONFIG = "mixtral_8x22b"
METRIC = "MoE layer tokens/s on 1 GB300"


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

ORACLE_FFN_FLOP_BUDGET = 4e12   # fp64 work of the CPU baseline's FFN sample


def oracle_throughput(cfg, inp, ffn_rows: int | None = None, token_cap: int | None = None) -> dict:
    """Time the oracle as it stands on a bounded sample and scale to tokens/s.

    Routing, map, permute and combine run on `token_cap` tokens (all T by
    default). The expert FFN runs the oracle's per-expert group routine
    (weight decode + the rows' GEMMs) on whole experts 0, 1, ... while their
    work (6 d F FLOP per row) fits ORACLE_FFN_FLOP_BUDGET, at least on the
    first ORACLE_FFN_FLOP_BUDGET's worth of expert 0's rows; `ffn_rows` caps
    the rows per expert instead. The times are scaled to every expert's
    decode and all kept rows."""
    from oracle import moe_oracle as O
    T = cfg.T if token_cap is None else min(cfg.T, token_cap)
    sub = dict(inp)
    sub["x"] = inp["x"][:T]
    import dataclasses
    c = dataclasses.replace(cfg, T=T)
    t0 = time.perf_counter()
    r = O.route(c, sub)
    counts, offsets, row_of, src_of, n_kept = O.build_map(r["topk_idx"], r["keep"], c.E)
    Xp = O.permute(sub["x"], src_of, c.K)
    t_route = time.perf_counter() - t0
    row_flop = 6.0 * cfg.d * cfg.F
    cap = ffn_rows if ffn_rows is not None else max(64, int(ORACLE_FFN_FLOP_BUDGET / row_flop))
    t_decode, t_rows, n_rows, experts = 0.0, 0.0, 0, 0
    for e in range(c.E):
        rows = np.arange(min(cap, int(counts[e])))
        if rows.size == 0:
            continue
        if experts and (ffn_rows is not None or (n_rows + rows.size) * row_flop > ORACLE_FFN_FLOP_BUDGET):
            break
        t1 = time.perf_counter()
        Wgu = O.decode(inp["W_gu"][e])
        Wd = O.decode(inp["W_down"][e])
        t2 = time.perf_counter()
        O.swiglu_group(O.decode(Xp[rows + offsets[e]]), Wgu, Wd, O.act_rounder(cfg.dtype, True))
        t_rows += time.perf_counter() - t2
        t_decode += t2 - t1
        n_rows += rows.size
        experts += 1
    Yp = np.zeros((n_kept, c.d))
    t3 = time.perf_counter()
    O.unpermute(Yp, row_of, r["topk_w"], dtype=c.dtype)
    t_comb = time.perf_counter() - t3
    n_full = n_kept * cfg.T / T
    total = (t_route + t_comb) * cfg.T / T + cfg.E * t_decode / experts + t_rows * n_full / n_rows
    if cfg.Fs:
        total += t_rows * cfg.T / n_rows * cfg.Fs / cfg.F
    if cfg.backward:
        total *= 3.0   # backward: two GEMMs per forward GEMM (dgrad + wgrad)
    wall = time.perf_counter() - t0
    return {"value": cfg.T / total, "unit": "tokens/s", "cores": host_threads(),
            "kind": "oracle",
            "sample": (f"routing, map, permute and combine on {T} of {cfg.T} tokens; expert FFN "
                       f"on {n_rows} rows of {experts} expert(s) with their weight decode, "
                       f"scaled to {cfg.E} experts and {int(n_full)} kept rows"
                       + ("; backward counted as 2x the forward GEMMs" if cfg.backward else "")),
            "sample_seconds": round(wall, 2)}


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


def launches_per_step(cfg, etp: int = 1) -> int:
    bf16 = cfg.dtype == "bf16"
    n = 2 if bf16 else 1                   # router: logits GEMM + Top-K (fp32: one fused kernel)
    n += 1 if cfg.drop else 0             # capacity
    n += 3                                 # map count, map scatter, row copy
    n += 2 * etp + (1 if etp > 1 else 0)   # routed grouped GEMMs per F-shard [+ partial sum]
    n += 2 if cfg.Fs else 0                # shared expert
    n += 1                                 # un-permute
    if cfg.backward:
        gm = 2 if bf16 else 0              # group tensor maps of the two weight-gradient GEMMs
        n += 1                             # un-permute backward
        n += (4 + gm) * etp + (1 if etp > 1 else 0)   # dH, dX, dW_down, dW_gu per shard [+ dXp sum]
        n += (4 + gm) if cfg.Fs else 0
        if bf16 and cfg.d % 256 == 0:      # router backward on the tensor cores:
            # dl, dl planes, [W_r planes + dx GEMM | dx kernel with the shared-expert addend],
            # group maps, dW_r GEMM, plane sum
            n += 6 + (0 if cfg.Fs else 1)
        else:
            n += 4                         # dl, dx, dW_r partials, reduce
        n += 1 if cfg.bias else 0          # db_r
        n += 1                             # permute backward
    return n


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return
    from synthetic import make_inputs
    inp = make_inputs(cfg, need_backward=False)
    vals = []
    for i in range(args.warmup + args.steps):
        r = oracle_throughput(cfg, inp, ffn_rows=64, token_cap=1024)
        if i >= args.warmup:
            vals.append(r["value"])
    v = statistics.median(vals)
    cpu = dict(r, value=v)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * cfg.T / v,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(cfg), "cpu_baseline": cpu,
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(cfg) -> dict:
    return {"workload": (f"{cfg.name} MoE layer {'fwd+bwd' if cfg.backward else 'fwd'}: T={cfg.T}, "
                         f"d={cfg.d}, E={cfg.E}, top-{cfg.K}, SwiGLU ffn={cfg.F}"
                         + (f", shared ffn={cfg.Fs}" if cfg.Fs else "")
                         + (f", capacity factor {cfg.cf} per {cfg.subseq}-token sub-sequence"
                            if cfg.drop else ", dropless")),
            "tokens_per_step": cfg.T, "l2": "inputs larger than L2 (all expert weights stream every step)",
            "parallelism": "replicas"}


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
        typed = {k: type(getattr(cfg, k))(v) for k, v in kv.items()}
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
    layer = MoELayer(cfg_r, w, etp=args.etp, layout=args.layout)
    x = to_device(inp["x"])
    layer.x = x   # the backward reads the forward's tokens
    dout = to_device(inp["dout"]) if cfg.backward else None
    stream = torch.cuda.current_stream()

    ffn_ev, perm_ev, unperm_ev, ffn_bwd_ev, route_ev = [], [], [], [], []

    def step(x, out, record=False):
        c, s, ws = cfg_r, layer.shape, layer.ws
        layer.x = x
        e = [torch.cuda.Event(enable_timing=True) for _ in range(8)] if record else None
        if record: e[6].record(stream)
        L.moe_route(s, x, w["W_r"], w.get("b_r"), w.get("w_sg"), layer.logits, layer.gate_logit,
                    layer.topk_idx, layer.topk_prob, layer.topk_w, layer.keep, ws)
        if record: e[7].record(stream)
        if record: e[0].record(stream)
        permute = L.moe_permute_padded if args.layout == "padded" else L.moe_permute
        permute(s, x, layer.topk_idx, layer.keep, layer.Xp, layer.row_of, layer.src_of,
                layer.counts, layer.offsets, ws)
        if record: e[1].record(stream)
        if record: e[2].record(stream)
        layer.routed_ffn()
        if record: e[3].record(stream)
        if c.Fs:
            L.moe_expert_ffn(layer.dtype_code, c.T, c.d, c.Fs, 1, layer.off1, x, w["Ws_gu"],
                             w["Ws_down"], layer.As, layer.Hs, layer.Ys, ws)
        if record: e[4].record(stream)
        L.moe_unpermute(s, layer.Yp, layer.row_of, layer.topk_w, layer.Ys, layer.gate_logit, out)
        if record: e[5].record(stream)
        if c.backward:
            eb = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) if record else None
            layer.backward(dout, ffn_events=eb)
            if record:
                ffn_bwd_ev.append(eb)
        if record:
            perm_ev.append((e[0], e[1]))
            ffn_ev.append((e[2], e[3]))
            unperm_ev.append((e[4], e[5]))
            route_ev.append((e[6], e[7]))

    for _ in range(args.warmup):
        step(x, layer.out)
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
        step(x, layer.out, record=True)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    secs = t_start.elapsed_time(t_end) / 1e3
    agg = aggregate(cfg.T * args.steps, secs, world, dist)

    n_kept = int(layer.counts.sum().item())   # kept rows (the padded layout computes more)
    ffn_ms = statistics.mean(a.elapsed_time(b) for a, b in ffn_ev)
    perm_ms = statistics.mean(a.elapsed_time(b) for a, b in perm_ev)
    unperm_ms = statistics.mean(a.elapsed_time(b) for a, b in unperm_ev)
    # the stream is idle when the timed region starts, so the first step's
    # route also waits for the host's launches: average the later steps
    route_ms = statistics.mean(a.elapsed_time(b) for a, b in (route_ev[1:] or route_ev))
    peaks = {}
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        peaks = json.load(open(pk_path))
    bf16_peak = peaks.get("bf16_tflops", 1900.0)
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured (burst)" if "bf16_tflops" in peaks else "fallback"
    flops = 6.0 * n_kept * cfg.d * cfg.F
    achieved = flops / (ffn_ms * 1e-3) / 1e12
    b = 2 if cfg.dtype == "bf16" else 4
    perm_bytes = cfg.T * cfg.d * b + n_kept * cfg.d * b + cfg.T * cfg.K * 9
    unperm_bytes = n_kept * cfg.d * b + cfg.T * cfg.d * b + cfg.T * cfg.K * 8
    route_bytes = route_algorithmic_bytes(cfg)
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tr_path):
        import hashlib
        ent = json.load(open(tr_path)).get(f"{cfg.name}:grouped_gemm")
        src = os.path.join(ROOT, "token_dispatch_expert_moe_gb300", "csrc", "gemm_tc.cu")
        sha = hashlib.sha256(code_text(src).encode()).hexdigest()[:16]
        if ent is not None and ent.get("source_sha") == sha:   # counters of this very kernel
            traffic = ent["bytes"]

    # e2e through the C ABI with host buffers: every step copies its tokens from
    # pinned host memory and reads its output back; the copies run on a second
    # stream, double-buffered, so that they overlap the neighbouring steps'
    # compute (step i+1's input and step i-1's output move during step i).
    copy_stream = torch.cuda.Stream()
    x_dev = [x, torch.empty_like(x)]
    out_dev = [layer.out, torch.empty_like(layer.out)]
    x_host = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for _ in range(2)]
    for hb in x_host:
        hb.copy_(x)
    out_host = [torch.empty(layer.out.shape, dtype=layer.out.dtype, pin_memory=True)
                for _ in range(2)]
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(nsteps, start_event=None):
        if start_event is not None:
            copy_stream.wait_event(start_event)
        with torch.cuda.stream(copy_stream):
            x_dev[0].copy_(x_host[0], non_blocking=True)
            h2d_done[0].record(copy_stream)
        for i in range(nsteps):
            b = i % 2
            stream.wait_event(h2d_done[b])
            if i >= 2:
                stream.wait_event(d2h_done[b])   # out_dev[b] read back two steps ago
            step(x_dev[b], out_dev[b])
            comp_done[b].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < nsteps:
                    nb = (i + 1) % 2
                    if i >= 1:
                        copy_stream.wait_event(comp_done[nb])   # step i-1 done with x_dev[nb]
                    x_dev[nb].copy_(x_host[nb], non_blocking=True)
                    h2d_done[nb].record(copy_stream)
                copy_stream.wait_event(comp_done[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
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
    h2d = x.numel() * x.element_size()
    d2h = layer.out.numel() * layer.out.element_size()

    if rank == 0:
        line = {
            "metric": METRIC, "value": agg["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * agg["seconds"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic (seeded normal inputs, random-init weights)",
            "config": dict(workload_config(cfg), **({"etp_shards": args.etp} if args.etp > 1 else {}),
                           **({"layout": "padded"} if args.layout == "padded" else {})),
            "clocks": clk,
            "e2e": {"value": e2e["value"], "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": (launches_per_step(cfg, args.etp)
                             + (1 if args.layout == "padded" else 0)) * args.steps,
            "roofline": {"kernel": "grouped SwiGLU GEMM (moe_expert_ffn: gate/up + down)",
                         "bound": "tensor", "achieved": achieved, "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": achieved / bf16_peak, "traffic": traffic,
                         "peak_source": peak_src,
                         "flops_per_launch": flops, "ms_per_launch": ffn_ms},
            "stages": {
                "n_kept": n_kept,
                "permute_ms": perm_ms, "permute_GBps": perm_bytes / perm_ms / 1e6,
                "permute_hbm_frac": perm_bytes / perm_ms / 1e6 / hbm_peak,
                "unpermute_ms": unperm_ms, "unpermute_GBps": unperm_bytes / unperm_ms / 1e6,
                "unpermute_hbm_frac": unperm_bytes / unperm_ms / 1e6 / hbm_peak,
                "route_ms": route_ms, "route_GBps": route_bytes / route_ms / 1e6,
                "route_hbm_frac": route_bytes / route_ms / 1e6 / hbm_peak,
                "hbm_peak_GBps": hbm_peak,
            },
        }
        if ffn_bwd_ev:   # routed experts' dgrad + wgrad: 12 N d F FLOP per call
            bwd_ms = statistics.mean(a.elapsed_time(b) for a, b in ffn_bwd_ev)
            bwd_tf = 12.0 * n_kept * cfg.d * cfg.F / (bwd_ms * 1e-3) / 1e12
            line["stages"].update(ffn_bwd_ms=bwd_ms, ffn_bwd_tflops=bwd_tf,
                                  ffn_bwd_frac=bwd_tf / bf16_peak)
        if not args.no_cpu_baseline and world == 1:   # rank 0 at N = 1 only
            line["cpu_baseline"] = oracle_throughput(cfg, inp)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
