"""moe_permute_noalloc: the workspace-free variant of moe_permute.

It serves callers that may not allocate device memory where they call the
layer (inside an allocator callback, under a fixed memory budget reserved at
start-up, or on a path that must not risk the device synchronisation an
allocation can cause). Its scratch lives in a fixed array inside libmoe.so.

The GPU test calls it through the C ABI twice in a row, on two different
routings, and checks each result against moe_permute on the same inputs, bit
for bit (maps, counts, offsets and copied rows are integer/byte work). The
second call also shows that the scratch left by the first call does not leak
into the next result. The file sorts last so that a stop-at-first-failure run
has already run every other test; it also passes alone in a fresh process.
"""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from synthetic import get_config, make_inputs


def _routing(cfg, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(cfg.E)[:cfg.K] for _ in range(cfg.T)]).astype(np.int32)
    keep = (rng.random((cfg.T, cfg.K)) < 0.9).astype(np.uint8)
    return idx, keep


@pytest.mark.gpu
def test_noalloc_matches_moe_permute_on_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_dispatch_expert_moe_gb300 import _lib as L
    from token_dispatch_expert_moe_gb300.layer import to_device

    cases = [
        dataclasses.replace(get_config("mixtral_8x22b_g8t8@small"), T=3000, d=256),
        dataclasses.replace(get_config("mixtral_8x22b@small"), T=777, d=512),
    ]
    for call, cfg in enumerate(cases):
        inp = make_inputs(cfg, need_backward=False)
        if call == 0:
            r = O.route(cfg, inp)
            idx, keep = r["topk_idx"], r["keep"]
        else:
            idx, keep = _routing(cfg, 11)
        s = L.shape_of(cfg)
        x, idx_d, keep_d = to_device(inp["x"]), to_device(idx), to_device(keep)
        T, K, E, d = cfg.T, cfg.K, cfg.E, cfg.d

        def outputs():
            return dict(Xp=torch.zeros((T * K, d), dtype=torch.bfloat16, device="cuda"),
                        row_of=torch.full((T, K), 7, dtype=torch.int32, device="cuda"),
                        src_of=torch.full((T * K,), 7, dtype=torch.int32, device="cuda"),
                        counts=torch.full((E,), 7, dtype=torch.int32, device="cuda"),
                        offsets=torch.full((E + 1,), 7, dtype=torch.int32, device="cuda"))

        ref = outputs()
        ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
        L.moe_permute(s, x, idx_d, keep_d, ref["Xp"], ref["row_of"], ref["src_of"],
                      ref["counts"], ref["offsets"], ws)
        got = outputs()
        L.moe_permute_noalloc(s, x, idx_d, keep_d, got["Xp"], got["row_of"], got["src_of"],
                              got["counts"], got["offsets"])
        torch.cuda.synchronize()
        n = int(ref["offsets"][-1].item())
        assert 0 < n <= T * K
        for k in ("row_of", "counts", "offsets"):
            assert torch.equal(got[k], ref[k]), (call, k)
        assert torch.equal(got["src_of"][:n], ref["src_of"][:n]), call
        assert torch.equal(got["Xp"][:n].view(torch.int16), ref["Xp"][:n].view(torch.int16)), call


@pytest.mark.gpu
def test_noalloc_at_its_token_limit():
    """T = MOE_PERMUTE_NOALLOC_MAX_TOKENS with E = 64 fills every word of the
    fixed scratch (512 map blocks x 64 experts); the result still equals
    moe_permute's bit for bit, the last block's rows included."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_dispatch_expert_moe_gb300 import _lib as L
    from token_dispatch_expert_moe_gb300.layer import to_device
    cfg = dataclasses.replace(get_config("mixtral_8x22b_g8t8@small"), T=131072, d=64, drop=False)
    assert cfg.E == 64 and cfg.K == 8
    idx, keep = _routing(cfg, 12)
    x = make_inputs(cfg, need_backward=False)["x"]
    s = L.shape_of(cfg)
    T, K, E, d = cfg.T, cfg.K, cfg.E, cfg.d
    x_d, idx_d, keep_d = to_device(x), to_device(idx), to_device(keep)

    def outputs():
        return dict(Xp=torch.zeros((T * K, d), dtype=torch.bfloat16, device="cuda"),
                    row_of=torch.full((T, K), 7, dtype=torch.int32, device="cuda"),
                    src_of=torch.full((T * K,), 7, dtype=torch.int32, device="cuda"),
                    counts=torch.full((E,), 7, dtype=torch.int32, device="cuda"),
                    offsets=torch.full((E + 1,), 7, dtype=torch.int32, device="cuda"))

    ref, got = outputs(), outputs()
    ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
    L.moe_permute(s, x_d, idx_d, keep_d, ref["Xp"], ref["row_of"], ref["src_of"], ref["counts"],
                  ref["offsets"], ws)
    L.moe_permute_noalloc(s, x_d, idx_d, keep_d, got["Xp"], got["row_of"], got["src_of"],
                          got["counts"], got["offsets"])
    torch.cuda.synchronize()
    n = int(ref["offsets"][-1].item())
    assert n == int(keep.sum())
    for k in ("row_of", "counts", "offsets"):
        assert torch.equal(got[k], ref[k]), k
    assert torch.equal(got["src_of"][:n], ref["src_of"][:n])
    assert torch.equal(got["Xp"][:n].view(torch.int16), ref["Xp"][:n].view(torch.int16))
    # the last 256-token block's kept slots land where the oracle's map puts them
    _, _, row_of, _, _ = O.build_map(idx, keep, E)
    assert np.array_equal(got["row_of"][-256:].cpu().numpy(), row_of[-256:])


def test_noalloc_rejects_more_tokens_than_its_scratch_holds():
    pytest.importorskip("torch")
    from token_dispatch_expert_moe_gb300 import build
    import os
    if not os.path.exists(build.LIB):
        build.build()
    from token_dispatch_expert_moe_gb300 import _lib as L
    s = L.MoEShape(T=131072 + 1, d=256, E=8, K=2, F=256, dtype=1)
    fake = 1 << 20   # never dereferenced: the size check fails first
    with pytest.raises(L.MoEError) as e:
        L.moe_permute_noalloc(s, fake, fake, fake, fake, fake, fake, fake, fake, 0)
    assert e.value.code == 2   # MOE_ERR_UNSUPPORTED
