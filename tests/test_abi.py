"""The C ABI without a GPU: libmoe.so loads, exports every entry point that
include/moe.h declares, sizes workspaces, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from token_dispatch_expert_moe_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from token_dispatch_expert_moe_gb300 import _lib
    return _lib


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"\b(moe_\w+)\s*\(", txt)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert "moe_route" in declared and "moe_expert_ffn_bwd" in declared
    for name in declared:
        assert hasattr(L.lib, name), name
    assert set(declared) == set(L.EXPORTED)


def test_version_and_status_strings(L):
    assert L.version().count(".") == 2
    for code in range(6):
        assert L.lib.moe_status_string(code)


def test_workspace_size(L):
    from synthetic import CONFIGS
    for cfg in CONFIGS.values():
        n = L.moe_workspace_size(L.shape_of(cfg))
        assert n > 0 and n % 256 == 0
    bad = L.MoEShape(T=10, d=64, E=65, K=2, F=128, dtype=1)
    assert L.moe_workspace_size(bad) == 0
    bad = L.MoEShape(T=10, d=64, E=8, K=9, F=128, dtype=1)
    assert L.moe_workspace_size(bad) == 0
    bad = L.MoEShape(T=10, d=60, E=8, K=2, F=128, dtype=1)   # d % 8 for bf16
    assert L.moe_workspace_size(bad) == 0
    bad = L.MoEShape(T=0, d=64, E=8, K=2, F=128, dtype=1)    # an empty batch
    assert L.moe_workspace_size(bad) == 0
    bad = L.MoEShape(T=1 << 28, d=64, E=8, K=8, F=128, dtype=1)   # T*K rows overflow int32
    assert L.moe_workspace_size(bad) == 0
    # the tensor-core router adds its K-split parts in shared memory (a
    # cluster of CTAs), so the workspace does not depend on the dtype
    b16 = L.moe_workspace_size(L.MoEShape(T=4096, d=512, E=8, K=2, F=128, dtype=1))
    f32 = L.moe_workspace_size(L.MoEShape(T=4096, d=512, E=8, K=2, F=128, dtype=0))
    assert b16 == f32


def test_invalid_arguments_rejected_on_host(L):
    s = L.MoEShape(T=16, d=64, E=4, K=2, F=128, dtype=1)
    fake = 1 << 20   # never dereferenced: validation fails first
    with pytest.raises(L.MoEError) as e:
        L.moe_route(s, None, fake, None, None, fake, None, fake, fake, fake, fake, fake, 0)
    assert e.value.code == 1
    with pytest.raises(L.MoEError) as e:   # misaligned x
        L.moe_route(s, fake + 2, fake, None, None, fake, None, fake, fake, fake, fake, fake, 0)
    assert e.value.code == 1
    with pytest.raises(L.MoEError) as e:   # w_sg without gate_logit
        L.moe_route(s, fake, fake, None, fake, fake, None, fake, fake, fake, fake, fake, 0)
    assert e.value.code == 1
    with pytest.raises(L.MoEError) as e:   # bf16 FFN needs d, F multiples of 128
        L.moe_expert_ffn(1, 32, 96, 128, 4, fake, fake, fake, fake, None, fake, fake, fake, 0)
    assert e.value.code == 2
    with pytest.raises(L.MoEError) as e:   # H_save is required
        L.moe_expert_ffn(1, 32, 128, 128, 4, fake, fake, fake, fake, None, None, fake, fake, 0)
    assert e.value.code == 1
    with pytest.raises(L.MoEError) as e:   # unpermute: Ys without gate_logit
        L.moe_unpermute(s, fake, fake, fake, fake, None, fake, 0)
    assert e.value.code == 1
    with pytest.raises(L.MoEError) as e:
        L.moe_route_bwd(s, fake, fake, fake, fake, fake, fake, fake, fake, None, None, fake, None,
                        None, fake, fake, 0)
    assert e.value.code == 1
    with pytest.raises(L.MoEError) as e:   # route_bwd: misaligned dx_router
        L.moe_route_bwd(s, fake, fake, None, fake, fake, fake, fake, fake, None, None, fake, None,
                        None, fake + 4, fake, 0)
    assert e.value.code == 1
    for args in [(3, 2, 8, 64, fake, fake + (1 << 16)),      # unknown dtype
                 (1, 0, 8, 64, fake, fake + (1 << 16)),      # no parts
                 (1, 17, 8, 64, fake, fake + (1 << 16)),     # too many parts
                 (1, 2, 8, 60, fake, fake + (1 << 16)),      # d % 8 for bf16
                 (1, 2, 8, 64, fake + 2, fake + (1 << 16)),  # misaligned partials
                 (1, 2, 8, 64, fake, fake + 1024)]:          # out inside partials
        with pytest.raises(L.MoEError) as e:
            L.moe_sum_partials(*args, 0)
        assert e.value.code == 1, args
    L.moe_sum_partials(1, 2, 0, 64, None, None, 0)   # zero rows: nothing to do
    with pytest.raises(L.MoEError) as e:   # ffn backward: workspace too small for the group maps
        L.moe_expert_ffn_bwd(1, 32, 128, 128, 4, fake, fake, fake, fake, fake, fake, fake, fake,
                             fake, fake, fake, fake, 0, ws_bytes=L.MOE_FFN_BWD_WORKSPACE_BYTES - 256)
    assert e.value.code == 1


def test_plain_c_caller(L, tmp_path):
    """The header is plain C: a C program compiled against include/moe.h
    alone links libmoe.so and runs its host-side checks (no device access)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from token_dispatch_expert_moe_gb300 import build
    exe = str(tmp_path / "c_abi_probe")
    libdir = os.path.dirname(build.LIB)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_abi_probe.c"), "-o", exe,
                        build.LIB, "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi probe ok" in r.stdout


def test_binding_constants_match_header(L):
    txt = open(os.path.join(ROOT, "include", "moe.h")).read()
    m = re.search(r"#define\s+MOE_FFN_BWD_WORKSPACE_BYTES\s+(\d+)u?", txt)
    assert m and int(m.group(1)) == L.MOE_FFN_BWD_WORKSPACE_BYTES
    m = re.search(r"#define\s+MOE_PERMUTE_NOALLOC_MAX_TOKENS\s+(\d+)", txt)
    assert m and int(m.group(1)) == 131072
    assert re.search(r"MOE_F32\s*=\s*0", txt) and re.search(r"MOE_BF16\s*=\s*1", txt)
    assert (L.MOE_F32, L.MOE_BF16) == (0, 1)
