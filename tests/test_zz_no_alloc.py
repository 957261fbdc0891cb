"""moe_permute_noalloc: the permutation for callers that cannot allocate device memory.

Some callers only ever receive their input and output buffers (for example a plugin
inside a framework that owns all device memory), so they cannot hand moe_permute a
workspace.  moe_permute_noalloc keeps that scratch in a fixed array inside the library.
This file is collected last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_scores_b300 import build, moe, synth


def test_noalloc_limit_is_stated_and_enforced():
    build.build()
    L = moe.load()
    cap = L.moe_permute_noalloc_max_scratch_bytes()
    assert cap == 256 * 1024
    # Sizes whose scratch exceeds the array are rejected on the host before any launch (and
    # before any pointer is looked at: every pointer here is NULL).  With at most 128 token
    # chunks of E int32 counters each, every N fits while E <= 512; at E = 1024 the largest
    # accepted batch is N = 64 (64 one-token chunks, exactly 256 KiB).
    for N, k, E in ((1 << 16, 2, 1024), (65, 8, 1024)):
        assert L.moe_permute_workspace_bytes(N, k, E) > cap
        assert L.moe_permute_noalloc(None, 1, N, 64, None, k, E, None, None, None, None, None, None) == -2
    assert L.moe_permute_workspace_bytes(64, 8, 1024) == cap
    for N in (1, 100, 1 << 20):
        assert L.moe_permute_workspace_bytes(N, 16, 512) <= cap


@pytest.mark.gpu
@pytest.mark.parametrize("N,E,k", [(777, 64, 8), (64, 1024, 8)], ids=["N777-E64", "N64-E1024-full-scratch"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(N, E, k):
    """Bit-exact agreement with moe_permute on two calls in a row (the second with other
    routing, so stale scratch from the first call cannot leak into it), at a small size and
    at the largest size the array holds (E = 1024, N = 64: all 256 KiB in use)."""
    cfg = synth.scaled(synth.CONFIGS["handbook"], N=N, D=256, E=E, F=128, k=k)
    xn, _ = synth.make_tokens(cfg, "cuda")
    rng = np.random.default_rng(9)
    for call in range(2):
        idx = np.stack([rng.choice(cfg.E, cfg.k, replace=False) for _ in range(cfg.N)])
        idx = torch.from_numpy(idx.astype(np.int32)).cuda()
        ref = moe.moe_permute(xn, idx, cfg.E)
        out = (torch.full((cfg.E,), -7, dtype=torch.int32, device="cuda"),
               torch.full((cfg.E + 1,), -7, dtype=torch.int32, device="cuda"),
               torch.full((cfg.N, cfg.k), -7, dtype=torch.int32, device="cuda"),
               torch.full((cfg.N * cfg.k,), -7, dtype=torch.int32, device="cuda"),
               torch.zeros(cfg.N * cfg.k, cfg.D, dtype=torch.bfloat16, device="cuda"))
        got = moe.moe_permute_noalloc(xn, idx, cfg.E, *out)
        torch.cuda.synchronize()
        assert moe.last_device_status() == 0
        for name, a, b in zip(("counts", "offsets", "row_map", "perm_token", "x_perm"), got, ref):
            assert torch.equal(a, b), (call, name)
