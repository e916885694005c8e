"""bench.py host logic without a GPU: whole-job aggregation over ranks
(tokens summed, slowest rank's time) with two gloo ranks, and the launch
count per step."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r = bench.aggregate(tokens_per_rank=1000.0 * (rank + 1), seconds_per_rank=0.5 + rank,
                        world=world, dist=dist)
    q.put((rank, r))
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in res.values():
        assert r["tokens"] == 3000.0 and r["seconds"] == 1.5
        assert abs(r["value"] - 2000.0) < 1e-9


def test_aggregate_single_rank():
    import bench
    r = bench.aggregate(8192.0, 2.0, 1)
    assert r["value"] == 4096.0


def test_launch_counts():
    import bench
    from synthetic import get_config
    # mixtral fwd: router GEMM + Top-K (K split in two), bucket + select, map count,
    # scatter, row copy, gate/up and down (pair + tail launch each), un-permute
    assert bench.launches_per_step(get_config("mixtral_8x22b")) == 12
    assert bench.launches_per_step(get_config("mixtral_8x22b"), gather=True) == 10
    # llama: fwd 9 (routing in the router GEMM's epilogue); bwd: un-permute 1,
    # FFN 6 + 2 maps, router 8 (dl, planes, W_r planes, dx pair + tail, maps,
    # dW_r, plane sum), permute 1
    assert bench.launches_per_step(get_config("llama3_8x70b")) == 9 + 18
    # qwen: fwd 14 (shared expert 4); bwd: 1 + (8 + 8) + router 6 + db 1 + permute 1
    assert bench.launches_per_step(get_config("qwen2_57b_a14b")) == 14 + 25
    # g8t8: fwd 12; bwd 1 + 8 + 8 + 1
    assert bench.launches_per_step(get_config("mixtral_8x22b_g8t8")) == 12 + 18
    assert bench.launches_per_step(get_config("tiny_f32")) == 7


def test_router_split_matches_the_library():
    """bench.router_splits restates libmoe.so's choice of K parts (it sizes the
    launch count); the library's router_k_split is exercised on the GPU."""
    import bench
    from synthetic import get_config
    assert [bench.router_splits(get_config(n)) for n in
            ("mixtral_8x22b", "qwen2_57b_a14b", "mixtral_8x22b_g8t8", "llama3_8x70b")] == [2, 2, 1, 1]


def test_traffic_key_ignores_comments_only(tmp_path):
    import bench
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text("int f() {\n  return 1;  // one\n}\n")
    b.write_text("// header\nint f() {\n\n  return 1;\n}\n")
    c.write_text("int f() {\n  return 2;\n}\n")
    assert bench.code_text(str(a)) == bench.code_text(str(b))
    assert bench.code_text(str(a)) != bench.code_text(str(c))



def test_route_bytes():
    import bench
    from synthetic import get_config
    # Mixtral-8x22B shape: x 8192 x 6144 bf16, W_r 8 x 6144 bf16, logits
    # 8192 x 8 fp32, 8192 x 2 slots of (index, prob, weight, keep)
    assert bench.route_algorithmic_bytes(get_config("mixtral_8x22b")) == (
        100663296 + 98304 + 262144 + 212992)
    # Qwen2 shape adds the gate vector (3584 bf16) and 8192 fp32 gate logits
    q = get_config("qwen2_57b_a14b")
    assert bench.route_algorithmic_bytes(q) == (
        8192 * 3584 * 2 + 64 * 3584 * 2 + 8192 * 64 * 4 + 3584 * 2 + 8192 * 4 + 8192 * 8 * 13)


def test_oracle_thread_count(monkeypatch):
    import bench
    n = len(os.sched_getaffinity(0))
    monkeypatch.delenv("OPENBLAS_NUM_THREADS", raising=False)
    monkeypatch.delenv("OMP_NUM_THREADS", raising=False)
    assert bench.host_threads() == n
    monkeypatch.setenv("OMP_NUM_THREADS", "1")      # what torchrun sets per rank
    assert bench.host_threads() == 1
    monkeypatch.setenv("OPENBLAS_NUM_THREADS", str(n + 7))
    assert bench.host_threads() == n


def test_reference_arm_rank0_detection(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_WORLD_SIZE", "2")
    for argv, want in ([["bench.py", "--impl", "reference"], True],
                       [["bench.py", "--impl=reference", "--gpus", "2"], True],
                       [["bench.py", "--gpus", "2"], False]):
        monkeypatch.setattr("sys.argv", argv)
        assert bench._reference_arm_rank0_under_torchrun() is want
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference"])
    monkeypatch.setenv("RANK", "1")
    assert not bench._reference_arm_rank0_under_torchrun()
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_WORLD_SIZE", "1")
    assert not bench._reference_arm_rank0_under_torchrun()


def test_oracle_baseline_sample_is_bounded():
    import bench
    from synthetic import get_config, make_inputs
    cfg = get_config("mixtral_8x22b@small")
    r = bench.oracle_throughput(cfg, make_inputs(cfg))
    assert r["kind"] == "oracle" and r["value"] > 0 and r["cores"] >= 1
    assert "expert(s) with their weight decode" in r["sample"]
    # the FFN sample is sized by its fp64 work: one Llama3-8x70B row is 1.4 GFLOP,
    # so its sample stops well short of the 8192 rows of one expert
    big = get_config("llama3_8x70b")
    assert int(bench.ORACLE_FFN_FLOP_BUDGET / (6.0 * big.d * big.F)) < 4096
