"""Full-size layers, in the launch configuration bench.py times (MoELayer, same buffers).

The oracle checks, at each configuration's real size:
* routing of every token (logits, ids outside the near-tie band, gates);
* counts, offsets, row map and token permutation, bit for bit;
* the permuted rows, bit for bit, and the expert outputs of the row-gathering GEMM against
  those of the GEMM over the permuted copy, bit for bit;
* the expert outputs and the layer output of a seeded sample of tokens that together visit
  every expert (so every expert's GEMM tiles are checked somewhere), computed one expert at a
  time on the CPU from regenerated weights (bf16 tolerance of tests/parity.py), and, where
  the weights fit comfortably in host memory, the same layer outputs through the oracle's
  token_outputs;
* the bias step, bit for bit;
and one property that holds at any size checks the combine over every token:
out = h + shared + sum_j gate * Y[row_map], evaluated in float64 from the kernel's inputs.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_scores_b300 import moe, synth
from oracle import moe_oracle
from tests import parity as P

pytestmark = pytest.mark.gpu

# (config, k, gather): gather None is the layer's own choice; the DeepSeek-V3 layer also runs
# with its routed rows gathered (the shared expert's tiles then ride in the gathering launch)
CASES = [("handbook", None, None), ("mixtral", None, None), ("deepseek_v3", None, None),
         ("deepseek_v3", None, True), ("skewed", 8, None), ("skewed", 4, None)]
SAMPLE = 6


def _layer(cfg, k, gather=None):
    dev = "cuda"
    xn, h = synth.make_tokens(cfg, dev)
    w_r, b = synth.make_router(cfg, dev)
    b = synth.gaussian(cfg.seed, "bias", (cfg.E,), 0.02 if cfg.score_fn == "sigmoid" else 0.1, device=dev)
    wg, wu, wd = synth.make_experts(cfg, dev)
    sh = synth.make_shared(cfg, dev)
    b0 = b.clone()
    layer = moe.MoELayer(moe.LayerWeights(w_r, b, wg, wu, wd, sh), cfg.N, k, cfg.score_fn, cfg.gamma,
                         gather=gather)
    assert gather is None or layer.gather == gather
    out = layer.forward(xn, h)
    torch.cuda.synchronize()
    assert moe.last_device_status() == 0
    return layer, xn, h, b0, out


@pytest.mark.parametrize("name,k,gather", CASES,
                         ids=[f"{n}-k{k or synth.CONFIGS[n].k}" + ("-gather" if g else "") for n, k, g in CASES])
def test_full_size_layer(name, k, gather):
    cfg = synth.CONFIGS[name]
    k = cfg.k if k is None else k
    layer, xn, h, b0, out = _layer(cfg, k, gather)

    # --- routing, every token -------------------------------------------------------
    xc, hc = synth.make_tokens(cfg, "cpu")
    wc, _ = synth.make_router(cfg, "cpu")
    assert torch.equal(xc, xn.cpu()) and torch.equal(hc, h.cpu())   # same generator bits
    r = moe_oracle.route(P.np64(xc), wc.numpy(), b0.cpu().numpy(), k, cfg.score_fn)
    g = {"idx": layer.idx.cpu(), "gate": layer.gate.cpu(), "logits": layer.logits.cpu(),
         "near_tie": layer.near_tie.cpu()}
    rep = P.compare_routing(g, r, k)
    print(name, k, rep)

    idx = g["idx"].numpy()
    same = ~(idx != r["idx"]).any(1)
    # --- histogram, scan, permutation ------------------------------------------------
    if rep["identical"]:
        counts = moe_oracle.expert_counts(r["idx"], cfg.E)
        offsets = moe_oracle.exclusive_scan(counts)
        row_map, perm = moe_oracle.stable_permutation(r["idx"], offsets)
        assert np.array_equal(layer.counts.cpu().numpy(), counts)
        assert np.array_equal(layer.offsets.cpu().numpy(), offsets)
        assert np.array_equal(layer.row_map.cpu().numpy(), row_map)
        assert np.array_equal(layer.perm_token.cpu().numpy(), perm)
        new_b, mom = moe_oracle.bias_update(b0.cpu().numpy(), counts, cfg.N * k, cfg.gamma)
        assert np.array_equal(layer.w.bias.cpu().numpy(), new_b)
        assert abs(layer.mom.item() - mom) <= 1e-6 * mom
    else:
        P.check_permutation_properties({"idx": g["idx"], "counts": layer.counts.cpu(),
                                        "offsets": layer.offsets.cpu(), "row_map": layer.row_map.cpu(),
                                        "perm_token": layer.perm_token.cpu()}, cfg.E, k)
    perm_t = layer.perm_token.long()
    # the GEMM over the permuted copy and the GEMM gathering its rows from xn through
    # perm_token (whichever the layer ran): the same bits
    w = layer.w
    x_perm = layer.x_perm if layer.x_perm is not None else xn[perm_t]
    assert torch.equal(x_perm, xn[perm_t])                            # permuted rows exact
    if layer.x_perm is None:
        y_other = moe.moe_grouped_swiglu(x_perm, layer.offsets, w.w_gate, w.w_up, w.w_down)
    else:
        y_other = moe.moe_grouped_swiglu_gather(xn, layer.perm_token, layer.offsets, w.w_gate, w.w_up,
                                                w.w_down)
    torch.cuda.synchronize()
    assert moe.last_device_status() == 0
    assert torch.equal(y_other, layer.y_perm)
    del y_other, x_perm

    # --- the combine, every token (property) -------------------------------------------
    rm = layer.row_map.long()
    ref = h.double() + (layer.sh_y.double() if layer.sh_y is not None else 0.0)
    ref = ref + (layer.gate.double()[:, :, None] * layer.y_perm.double()[rm]).sum(1)
    err = (out.double() - ref).abs()
    half_ulp = torch.ldexp(torch.ones_like(ref), torch.frexp(ref.abs())[1] - 9)
    assert bool((err <= half_ulp * 1.0001 + 1e-6).all()), float((err - half_ulp).max())

    # --- expert outputs and layer output of sampled tokens ----------------------------
    tokens = _covering_sample(r["idx"], np.where(same)[0], cfg.E, cfg.seed)
    assert set(r["idx"][tokens].ravel().tolist()) == set(r["idx"][same].ravel().tolist())  # every routed expert
    x_s = P.np64(xc[tokens])
    want_y = {}                            # (token position, slot) -> oracle expert output
    for e in sorted({int(v) for v in r["idx"][tokens].ravel()}):
        wg, wu, wd = (P.np64(t) for t in synth.make_expert(cfg, e, "cpu"))
        pairs = [(i, j) for i, t in enumerate(tokens) for j in np.where(r["idx"][t] == e)[0]]
        ys = moe_oracle.swiglu_expert(x_s[[i for i, _ in pairs]], wg, wu, wd)  # one call per expert
        for (i, j), y in zip(pairs, ys):
            want_y[(i, j)] = y
    y_gpu = layer.y_perm.cpu()
    got_rows, want_rows = [], []
    for (i, j), y in want_y.items():
        got_rows.append(P.np64(y_gpu[int(layer.row_map[tokens[i], j])]))
        want_rows.append(y)
    P.assert_close("y_perm (sampled rows)", np.stack(got_rows), np.stack(want_rows))
    want_out = P.np64(hc[tokens]).copy()
    if cfg.shared:
        sg, su, sd = synth.make_expert(cfg, 0, "cpu", shared=True)
        ysh = moe_oracle.swiglu_expert(x_s, P.np64(sg), P.np64(su), P.np64(sd))
        P.assert_close("shared_y (sampled)", P.np64(layer.sh_y.cpu()[tokens]), ysh)
        want_out += ysh
    for (i, j), y in want_y.items():
        want_out[i] += r["gate"][tokens[i], j] * y
    P.assert_close("out (sampled)", P.np64(out.cpu()[tokens]), want_out)
    P.delta_close("out - h (sampled)", P.np64(out.cpu()[tokens]), want_out, P.np64(hc[tokens]))
    if 3 * cfg.E * cfg.D * cfg.F * 2 <= 2e9:  # the oracle's per-token formula, weights cached per expert
        sh = None
        if cfg.shared:
            sh = tuple(P.np64(t) for t in synth.make_expert(cfg, 0, "cpu", shared=True))
        via = moe_oracle.token_outputs(tokens, x_s, P.np64(hc[tokens]), r["idx"][tokens], r["gate"][tokens],
                                       lambda e: tuple(t.float().numpy() for t in synth.make_expert(cfg, e, "cpu")),
                                       sh)
        P.assert_close("out (sampled, token_outputs)", P.np64(out.cpu()[tokens]), via)


def _covering_sample(idx, candidates, E, seed, at_least=SAMPLE):
    """Seeded tokens, drawn in random order, kept while they visit an expert no kept token
    visits yet, until every expert is visited (or the candidates run out); at least
    `at_least` tokens."""
    rng = np.random.default_rng(seed)
    order = rng.permutation(candidates)
    seen, kept = set(), []
    for t in order:
        new = set(idx[t].tolist()) - seen
        if new or len(kept) < at_least:
            kept.append(int(t))
            seen |= set(idx[t].tolist())
        if len(seen) == E and len(kept) >= at_least:
            break
    return np.array(kept)


def test_generator_bits_equal_on_gpu_and_cpu():
    for name in ("handbook", "deepseek_v3"):
        cfg = synth.CONFIGS[name]
        idx = torch.arange(0, cfg.E * cfg.F * cfg.D, 9973, dtype=torch.int64)
        for stream in ("w_gate", "w_down", "xn"):
            a = synth.gaussian_at(cfg.seed, stream, idx.cuda(), 0.1, torch.bfloat16).cpu()
            b = synth.gaussian_at(cfg.seed, stream, idx, 0.1, torch.bfloat16)
            assert torch.equal(a, b)


def test_sustained_gemm_mode_runs_its_three_inputs():
    """bench.py --sustained-gemm on a small layer: three loops, the same bits as before for the
    layer afterwards (the mode restores the offsets and the permuted rows it changes)."""
    import bench
    cfg = synth.scaled(synth.CONFIGS["deepseek_v3"], N=512, D=256, E=32, F=128, k=8, F_shared=128)
    wl = bench.Workload(cfg, cfg.k, torch.device("cuda"))
    b0 = wl.layer.w.bias.clone()  # every forward steps the bias: each run below starts from b0
    out0 = wl.run().clone()
    r = bench.sustained_gemm(wl, calls=2, reps=2)
    assert set(r) == {"routed counts", "balanced counts", "zero activations"}
    assert r["balanced counts"]["row_tiles"] == cfg.E and r["balanced counts"]["half_tiles"] == 0
    assert all(v["ms_per_call"] > 0 for v in r.values())
    wl.layer.w.bias.copy_(b0)
    out1 = wl.run()
    torch.cuda.synchronize()
    assert moe.last_device_status() == 0
    assert torch.equal(out0, out1)


def test_full_size_router_launch_with_the_shared_first_gemm():
    """DeepSeek-V3-shaped layer with the shared expert's first GEMM in the router's launch: the
    default layer's routing, shared H and output, bit for bit, at full size."""
    cfg = synth.CONFIGS["deepseek_v3"]
    layer, xn, h, b0, out = _layer(cfg, cfg.k)
    out_ref = out.clone()
    w = layer.w
    lw = moe.LayerWeights(w.w_router, b0.clone(), w.w_gate, w.w_up, w.w_down, w.shared)
    got = moe.MoELayer(lw, cfg.N, cfg.k, cfg.score_fn, cfg.gamma, router_shared=True)
    o = got.forward(xn, h)
    torch.cuda.synchronize()
    assert moe.last_device_status() == 0
    assert torch.equal(got.idx, layer.idx) and torch.equal(got.logits, layer.logits)
    assert torch.equal(got.sh_h, layer.sh_h) and torch.equal(got.sh_y, layer.sh_y)
    assert torch.equal(o, out_ref)
