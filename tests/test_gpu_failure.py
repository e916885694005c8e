"""Failure detection without a GPU fault: the grouped GEMM's pipeline waits
are bounded. The test build of the library (libmoe_testhooks.so, the same
kernels with a fault-injection hook compiled in) runs in a process of its
own: with MOE_FAULT_INJECT_STALL=1 the TMA producer issues no loads, so the
MMA warp waits on a barrier that nothing will complete; after about two
seconds the kernel records MOE_ERR_TIMEOUT in the status word, stops every
warp role, releases its tensor memory and returns. The test reads the status
on the host and then checks that the same context still computes correct
results. The product library (libmoe.so) has no such hook."""
import os
import subprocess
import sys
import time

import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic.gen import normal_bf16
from tests.gpu_util import assert_close, dev, empty, host, lib, torch

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 4
INFO_GEMM_TIMEOUT = 0x1000


def _case():
    d, F = 256, 256
    offsets = np.array([0, 100, 400], dtype=np.int32)
    n = int(offsets[-1])
    Xp = normal_bf16(7, 101, (n, d))
    W_gu = normal_bf16(7, 102, (2, 2 * F, d), 1 / np.sqrt(d))
    W_down = normal_bf16(7, 103, (2, d, F), 1 / np.sqrt(F))
    return d, F, offsets, n, Xp, W_gu, W_down


def _run(L, d, F, offsets, n, Xp, W_gu, W_down, ws):
    H = empty((n, F), torch.bfloat16)
    Y = empty((n, d), torch.bfloat16)
    L.moe_expert_ffn(L.MOE_BF16, n, d, F, 2, dev(offsets), dev(Xp), dev(W_gu), dev(W_down), None,
                     H, Y, ws)
    return H, Y


def _under_test_build():
    return os.environ.get("MOE_LIBRARY", "").endswith("libmoe_testhooks.so")


def test_timeout_case(monkeypatch):
    """Runs only inside the test build's process (see the two tests below)."""
    if not _under_test_build():
        pytest.skip("needs the test build of the library (run by the tests below)")
    L = lib()
    d, F, offsets, n, Xp, W_gu, W_down = _case()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    monkeypatch.setenv("MOE_FAULT_INJECT_STALL", "1")
    t0 = time.time()
    _run(L, d, F, offsets, n, Xp, W_gu, W_down, ws)
    rc, info = L.moe_get_status(ws)
    elapsed = time.time() - t0
    assert rc == MOE_ERR_TIMEOUT, (rc, hex(info))
    assert info & 0xF000 == INFO_GEMM_TIMEOUT, hex(info)
    assert elapsed < 60, elapsed
    # the context is intact: the same call without the stall is correct
    monkeypatch.delenv("MOE_FAULT_INJECT_STALL")
    L.moe_clear_status(ws)
    H, Y = _run(L, d, F, offsets, n, Xp, W_gu, W_down, ws)
    rc, info = L.moe_get_status(ws)
    assert rc == 0, (rc, hex(info))
    _, Hr, Yr = O.expert_ffn(Xp, offsets, W_gu, W_down, "bf16")
    assert_close("H", host(H), Hr, "bf16", "act")
    assert_close("Yp", host(Y), Yr, "bf16", "act")


def _in_test_build(extra_env):
    lib()
    from token_dispatch_expert_moe_gb300 import build
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys, pytest; sys.exit(pytest.main(['-q', '-p', 'no:cacheprovider', "
            "'tests/test_gpu_failure.py::test_timeout_case']))")
    env = dict(os.environ, MOE_LIBRARY=build.TEST_LIB, **extra_env)
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=root, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "1 passed" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


def test_pair_kernel_timeout():
    _in_test_build({})


def test_single_cta_kernel_timeout():
    _in_test_build({"MOE_GEMM_PAIR": "0"})
