"""Failure detection on the device, without faulting it.

* A bounded pipeline wait that runs out: moe_selftest_bounded_wait waits, with the code every
  tensor-core kernel uses, on a barrier nothing arrives on.  The kernel must give up within
  its short limit, record MOE_ERR_TIMEOUT, let its in-flight copy land, free its tensor
  memory and return; the device then runs a layer that still matches the oracle.
* Non-finite router logits (NaN or infinite inputs) are reported as MOE_ERR_NAN_INPUT by both
  routers, and the other tokens' routing is unchanged.
"""
import time

import numpy as np
import pytest
import torch

from mixture_experts_layer_scores_b300 import moe, synth
from oracle import moe_oracle
from tests import parity as P

pytestmark = pytest.mark.gpu

TIMEOUT, NAN_INPUT = -4, -5


def _small_layer_matches_oracle():
    cfg = synth.scaled(synth.CONFIGS["handbook"], N=300, D=256, E=16, F=128, k=4)
    inp = P.make_inputs(cfg, "cuda")
    g = P.gpu_layer(cfg, inp)
    assert moe.last_device_status() == 0
    o = P.oracle_layer(cfg, P.make_inputs(cfg, "cpu"))
    P.compare_layer(cfg, g, o)


def test_bounded_wait_runs_out_and_the_device_stays_usable():
    assert moe.last_device_status() == 0
    src = torch.arange(1024, dtype=torch.int32, device="cuda")   # 4 KB copied while the wait runs out
    steps = torch.zeros(1, dtype=torch.int32, device="cuda")
    limit = 2_000_000                                               # about 1 ms of SM cycles
    t0 = time.perf_counter()
    moe.selftest_bounded_wait(src, steps, limit)
    st = moe.last_device_status()                                   # waits for the kernel
    dt = time.perf_counter() - t0
    assert st == TIMEOUT, moe.STATUS.get(st, st)
    assert int(steps.item()) == 15, int(steps.item())               # copy landed, gave up, left, freed
    assert dt < 1.0, dt                                             # the short limit, not the 2 s one
    assert moe.last_device_status() == 0                            # reading cleared the word
    _small_layer_matches_oracle()
    # and once more: the path is repeatable
    moe.selftest_bounded_wait(src, steps, limit)
    assert moe.last_device_status() == TIMEOUT and int(steps.item()) == 15


def test_selftest_rejects_bad_arguments_before_launch():
    src = torch.zeros(1024, dtype=torch.int32, device="cuda")
    steps = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = moe.load()
    s = moe._stream()
    assert L.moe_selftest_bounded_wait(None, 2_000_000, moe._p(steps), s) == -1
    assert L.moe_selftest_bounded_wait(moe._p(src), 10, moe._p(steps), s) == -1          # limit too short
    assert L.moe_selftest_bounded_wait(moe._p(src), 1 << 40, moe._p(steps), s) == -1     # above the normal limit
    assert moe.last_device_status() == 0


@pytest.mark.parametrize("path", ["tensor_core", "cuda_core"])
def test_nonfinite_logits_are_reported(path):
    cfg = synth.scaled(synth.CONFIGS["handbook"], N=200, D=256, E=32, k=4)
    xn, _ = synth.make_tokens(cfg, "cuda")
    w, _ = synth.make_router(cfg, "cuda")
    b = synth.gaussian(cfg.seed, "bias", (cfg.E,), 0.05, device="cuda")
    if path == "tensor_core":
        ws = moe.moe_router_split(w)
        run = lambda x: moe.moe_router_topk_split(x, ws, b, cfg.k)
    else:
        run = lambda x: moe.moe_router_topk(x, w, b, cfg.k)
    _, idx0, gate0, _ = run(xn)
    assert moe.last_device_status() == 0
    for bad in (float("nan"), float("inf")):
        x = xn.clone()
        x[7, 3] = bad                                   # token 7: every logit non-finite
        _, idx, gate, _ = run(x)
        assert moe.last_device_status() == NAN_INPUT
        keep = torch.ones(cfg.N, dtype=torch.bool, device="cuda")
        keep[7] = False
        assert torch.equal(idx[keep], idx0[keep]) and torch.equal(gate[keep], gate0[keep])
        ids = idx[7].tolist()
        assert len(set(ids)) == cfg.k and all(0 <= e < cfg.E for e in ids)
    _, idx, _, _ = run(xn)                              # clean input: clean status again
    assert moe.last_device_status() == 0 and torch.equal(idx, idx0)


def test_shared_call_rejects_rows_to_gather_without_tokens():
    """moe_grouped_swiglu_shared asked to gather routed rows (perm_token given) from N = 0 tokens
    returns MOE_ERR_INVALID_ARG on the host: nothing is launched, nothing is read."""
    G, D, F, M = 4, 128, 128, 64
    z = lambda *sh: torch.zeros(*sh, dtype=torch.bfloat16, device="cuda")
    wg, wu, wd = z(G, F, D), z(G, F, D), z(G, D, F)
    offsets = torch.tensor([0, 16, 32, 48, 64], dtype=torch.int32, device="cuda")
    perm = torch.zeros(M, dtype=torch.int32, device="cuda")
    h, y, xn = z(M, F), z(M, D), z(8, D)
    L = moe.load()
    p = moe._p
    assert L.moe_grouped_swiglu_shared(None, p(perm), p(offsets), G, M, D, F, p(wg), p(wu), p(wd), p(h), p(y), p(xn),
                                       0, None, None, None, None, None, moe._stream()) == -1
    torch.cuda.synchronize()
    assert moe.last_device_status() == 0
