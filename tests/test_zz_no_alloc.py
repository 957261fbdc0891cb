"""moe_permute_noalloc: the permutation for callers that cannot allocate device memory.

Some callers only ever receive their input and output buffers (for example a plugin
inside a framework that owns all device memory), so they cannot hand moe_permute a
workspace.  moe_permute_noalloc keeps that scratch in a fixed array inside the library.
This file is collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_scores_b300 import build, moe, synth


def test_noalloc_limit_is_stated_and_enforced():
    build.build()
    L = moe.load()
    cap = L.moe_permute_noalloc_max_scratch_bytes()
    assert cap == 256 * 1024
    # (N, k, E) whose scratch exceeds the array: rejected on the host before any launch
    N, k, E = 1 << 16, 2, 1024
    assert L.moe_permute_workspace_bytes(N, k, E) > cap
    vp = ctypes.c_void_p
    assert L.moe_permute_noalloc(vp(16), 1, N, 64, vp(16), k, E, vp(16), vp(16), vp(16), vp(16),
                                 vp(16), None) == -2


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    """Bit-exact agreement with moe_permute on two calls in a row (the second with other
    routing, so stale scratch from the first call cannot leak into it)."""
    cfg = synth.scaled(synth.CONFIGS["handbook"], N=777, D=256, E=64, F=128, k=8)
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
