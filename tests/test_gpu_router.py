"""Router parity at the full router shapes of every layer configuration, both paths.

The tensor-core router (split fp32 weights) and the CUDA-core fp32 router must both give
logits within 1e-5 relative Frobenius of the oracle and bit-exact expert ids outside the
1e-6 near-tie band.  Also: the weight split is exact, and (handbook article, router
precision) a router with bf16-rounded weights does change winners where these do not.
"""
import math

import numpy as np
import pytest
import torch

from mixture_experts_layer_scores_b300 import moe, synth
from oracle import moe_oracle
from tests import parity as P

pytestmark = pytest.mark.gpu

FULL = {name: synth.CONFIGS[name] for name in ("handbook", "mixtral", "deepseek_v3", "skewed")}


def _route_inputs(cfg, bias_scale=0.0):
    xg, _ = synth.make_tokens(cfg, "cuda")
    wg, _ = synth.make_router(cfg, "cuda")
    xc, _ = synth.make_tokens(cfg, "cpu")
    wc, _ = synth.make_router(cfg, "cpu")
    b = synth.gaussian(cfg.seed, "bias", (cfg.E,), bias_scale) if bias_scale else torch.zeros(cfg.E)
    return xg, wg, b.cuda(), xc, wc, b


def _check(cfg, g, o):
    gi = {"idx": g[1].cpu(), "gate": g[2].cpu(), "logits": g[0].cpu(), "near_tie": g[3].cpu()}
    rep = P.compare_routing(gi, o, cfg.k)
    err = np.abs(gi["logits"].numpy().astype(np.float64) - o["logits"].astype(np.float64))
    rep["logit_max_abs"] = float(err.max())
    rep["logit_rms_err"] = float(np.sqrt((err ** 2).mean()))
    return rep


@pytest.mark.parametrize("name", list(FULL))
def test_router_full_size_both_paths(name):
    cfg = FULL[name]
    scale = 0.02 if cfg.score_fn == "sigmoid" else 0.1
    xg, wg, bg, xc, wc, bc = _route_inputs(cfg, scale)
    o = moe_oracle.route(P.np64(xc), wc.numpy(), bc.numpy(), cfg.k, cfg.score_fn)
    split = moe.moe_router_split(wg)
    tc = moe.moe_router_topk_split(xg, split, bg, cfg.k, cfg.score_fn)
    torch.cuda.synchronize()
    rep_tc = _check(cfg, tc, o)
    simt = moe.moe_router_topk(xg, wg, bg, cfg.k, cfg.score_fn)
    torch.cuda.synchronize()
    rep_simt = _check(cfg, simt, o)
    print(name, "tensor-core", rep_tc)
    print(name, "cuda-core", rep_simt)
    assert moe.last_device_status() == 0


def test_split_is_exact():
    E, D = 64, 256
    w = synth.gaussian(3, "misc", (E, D), 0.02).cuda()
    w[0, :8] = torch.tensor([0.0, -0.0, 1.0, -3.0e-30, 1.0e30, 2.0 ** -100, 1.0 + 2.0 ** -23, -7.123456])
    sp = moe.moe_router_split(w)
    torch.cuda.synchronize()
    total = sp.double().sum(0)
    assert torch.equal(total, w.double())


def test_ragged_router_shapes():
    """Token counts off the 128-row tile, E off the 16/32/64-column tiles, k at both ends."""
    for N, D, E, k, fn in [(1, 64, 3, 1, "softmax"), (129, 128, 17, 5, "softmax"),
                           (300, 192, 48, 16, "sigmoid"), (257, 256, 200, 8, "sigmoid"),
                           (64, 64, 256, 1, "softmax")]:
        cfg = synth.scaled(synth.CONFIGS["handbook"], N=N, D=D, E=E, k=k, score_fn=fn)
        xg, wg, bg, xc, wc, bc = _route_inputs(cfg, 0.05 if fn == "softmax" else 0.01)
        o = moe_oracle.route(P.np64(xc), wc.numpy(), bc.numpy(), k, fn)
        tc = moe.moe_router_topk_split(xg, moe.moe_router_split(wg), bg, k, fn)
        torch.cuda.synchronize()
        _check(cfg, tc, o)


def test_bf16_router_flips_winners_fp32_does_not():
    """Handbook article, router precision: rounding the router to bf16 merges close
    logits and changes the chosen experts; the fp32-accurate routers do not."""
    cfg = synth.CONFIGS["handbook"]
    xg, wg, bg, xc, wc, bc = _route_inputs(cfg)
    o = moe_oracle.route(P.np64(xc), wc.numpy(), None, cfg.k)
    w_bf16 = wg.to(torch.bfloat16).float()
    bf = moe.moe_router_topk(xg, w_bf16, None, cfg.k)
    tc = moe.moe_router_topk_split(xg, moe.moe_router_split(wg), None, cfg.k)
    torch.cuda.synchronize()
    flips_bf16 = int(((bf[1].cpu().numpy() != o["idx"]).any(1) & (o["gap"] >= P.GAP)).sum())
    flips_tc = int(((tc[1].cpu().numpy() != o["idx"]).any(1) & (o["gap"] >= P.GAP)).sum())
    print("tokens whose experts change outside the near-tie band: bf16 router", flips_bf16,
          "fp32 (split) router", flips_tc)
    assert flips_bf16 > 0 and flips_tc == 0


def test_special_scores_order():
    """Equal scores (including -0 vs +0) keep ascending ids; NaN and -inf rank last, by id."""
    D, E, k = 64, 12, 12
    vals = [0.5, -0.0, 0.0, float("nan"), float("-inf"), 0.5, 0.25, 0.0, -1.0, float("nan"), 2.0, -0.0]
    w = torch.zeros(E, D)
    w[:, 0] = torch.tensor(vals)
    x = torch.zeros(1, D, dtype=torch.bfloat16)
    x[0, 0] = 1.0
    r = moe_oracle.route(x.double().numpy(), w.numpy(), None, k)
    expect = [10, 0, 5, 6, 1, 2, 7, 11, 8, 3, 4, 9]
    assert r["idx"][0].tolist() == expect
    _, idx, _, _ = moe.moe_router_topk(x.cuda(), w.cuda(), None, k)
    torch.cuda.synchronize()
    assert idx[0].cpu().tolist() == expect
    assert moe.last_device_status() == -5  # NaN and -inf logits: reported, routed by the order rule
    # tensor-core path with finite weights only (the split needs finite weights)
    wf = w.clone()
    wf[3, 0], wf[4, 0], wf[9, 0] = -3.0, -3.0, -5.0
    r = moe_oracle.route(x.double().numpy(), wf.numpy(), None, 8)
    _, idx, _, _ = moe.moe_router_topk_split(x.cuda(), moe.moe_router_split(wf.cuda()), None, 8)
    torch.cuda.synchronize()
    assert idx[0].cpu().tolist() == r["idx"][0].tolist()
    assert moe.last_device_status() == 0


@pytest.mark.parametrize("N,D,E,k,fn", [(4096, 1024, 896, 16, "sigmoid"), (8192, 2048, 64, 8, "sqrt_softplus"),
                                        (2048, 512, 1024, 8, "softmax")])
def test_router_large_E_and_sqrt_softplus(N, D, E, k, fn):
    """Routers beyond 256 experts (16 of 896, as the handbook article's Kimi example) and the
    sqrt(softplus) score function, on the tensor-core path."""
    cfg = synth.scaled(synth.CONFIGS["handbook"], N=N, D=D, E=E, k=k, score_fn=fn)
    xg, wg, bg, xc, wc, bc = _route_inputs(cfg, 0.02)
    o = moe_oracle.route(P.np64(xc), wc.numpy(), bc.numpy(), k, fn)
    tc = moe.moe_router_topk_split(xg, moe.moe_router_split(wg), bg, k, fn)
    torch.cuda.synchronize()
    print(N, D, E, k, fn, _check(cfg, tc, o))
