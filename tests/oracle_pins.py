"""Checks that pin the CPU oracle to facts fixed outside it.

Each ``check_*`` takes the oracle module (so a mutation test can hand in a copy
with a planted mistake) and raises AssertionError when the oracle disagrees with
the pages, a closed form, an invariant, a library routine or brute force.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _arr(v, dt=np.float32):
    return np.array([[float(x) for x in row] for row in v], dtype=dt) if isinstance(v[0], list) \
        else np.array([float(x) for x in v], dtype=dt)


# ---- worked examples ------------------------------------------------------------------

def check_route_golden(o):
    """Hand-worked router examples (lesson 'Build it' step 1; sigmoid reading)."""
    for c in _load("route_examples.json")["cases"]:
        x = np.array([c["hidden"]], dtype=np.float32)
        w = _arr(c["w_router"])
        b = np.array(c["bias"], dtype=np.float32)
        r = o.route(x, w, b, c["k"], c["score_fn"])
        assert r["idx"][0].tolist() == c["idx"], (c["name"], r["idx"][0].tolist())
        assert np.allclose(r["gate"][0], c["gate"], rtol=0, atol=1e-7), (c["name"], r["gate"][0])


def check_layer_golden(o):
    """Hand-worked one-token layers (lesson 'Concept' and 'Shared experts')."""
    for c in _load("layer_example.json")["cases"]:
        sh = None
        if c["shared"]:
            s = c["shared"]
            sh = (np.array(s["w_gate"]), np.array(s["w_up"]), np.array(s["w_down"]))
        r = o.moe_layer(np.array(c["xn"]), np.array(c["h"]), np.array(c["w_router"], np.float32),
                        np.array(c["bias"], np.float32), np.array(c["w_gate"]),
                        np.array(c["w_up"]), np.array(c["w_down"]), c["k"], c["score_fn"],
                        shared=sh)
        assert r["idx"].tolist() == c["idx"], c["name"]
        assert np.allclose(r["gate"], c["gate"], atol=1e-7), c["name"]
        # ln3 is rounded to fp32 in the router weights, so gates carry ~1e-8 of rounding
        assert np.allclose(r["out"], c["out"], rtol=0, atol=1e-6), (c["name"], r["out"])


# ---- closed forms and library routines ------------------------------------------------

def _rand(seed, *shape, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def check_dense_reduction(o):
    """E = 1, k = 1: the gate is exactly 1 and the layer is h + dense SwiGLU FFN
    (the handbook's 1-expert upcycling invariant).  Reference: torch fp64 silu/matmul."""
    N, D, F = 7, 16, 24
    x, h = _rand(1, N, D), _rand(2, N, D)
    wg, wu, wd = _rand(3, 1, F, D, scale=0.3), _rand(4, 1, F, D, scale=0.3), _rand(5, 1, D, F, scale=0.3)
    r = o.moe_layer(x, h, _rand(6, 1, D), np.zeros(1, np.float32), wg, wu, wd, 1, "softmax")
    assert np.all(r["gate"] == 1.0)
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    ref = t(h) + (torch.nn.functional.silu(t(x) @ t(wg[0]).T) * (t(x) @ t(wu[0]).T)) @ t(wd[0]).T
    assert np.allclose(r["out"], ref.numpy(), rtol=1e-12, atol=1e-12)


def check_split_dense(o):
    """k = E experts that are F-slices of one dense SwiGLU, with unit gates, sum to the
    dense FFN (the handbook: the k chosen experts hold the dense layer's parameters)."""
    N, D, E, Fe = 5, 32, 8, 16
    x, h = _rand(11, N, D), _rand(12, N, D)
    Wg, Wu, Wd = _rand(13, E * Fe, D, scale=.2), _rand(14, E * Fe, D, scale=.2), _rand(15, D, E * Fe, scale=.2)
    wg = Wg.reshape(E, Fe, D)
    wu = Wu.reshape(E, Fe, D)
    wd = np.stack([Wd[:, e * Fe:(e + 1) * Fe] for e in range(E)])
    r = o.moe_layer(x, h, _rand(16, E, D), None, wg, wu, wd, E, "softmax",
                    gate_override=np.ones((N, E)))
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    ref = t(h) + (torch.nn.functional.silu(t(x) @ t(Wg).T) * (t(x) @ t(Wu).T)) @ t(Wd).T
    assert np.allclose(r["out"], ref.numpy(), rtol=1e-11, atol=1e-11)


def check_all_chosen(o):
    """k = E: softmax gates are the full softmax of the logits (scipy), sigmoid gates are
    sigma / sum sigma, whatever the bias."""
    from scipy.special import softmax, expit
    x, w = _rand(21, 9, 12), _rand(22, 6, 12)
    b = _rand(23, 6)
    r = o.route(x, w, b, 6, "softmax")
    rows = np.arange(9)[:, None]
    full = softmax(r["logits"].astype(np.float64), axis=1)
    assert np.allclose(r["gate"], full[rows, r["idx"]], atol=1e-14)
    r = o.route(x, w, b, 6, "sigmoid")
    s = expit(r["logits"].astype(np.float64))
    assert np.allclose(r["gate"], (s / s.sum(1, keepdims=True))[rows, r["idx"]], atol=1e-14)


def _round_f32(fr: Fraction) -> np.float32:
    """Correctly rounded fp32 of an exact rational (nearest, ties to even)."""
    c = np.float32(float(fr))
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        err = abs(Fraction(float(cand)) - fr)
        key = (err, int(np.frombuffer(np.float32(cand).tobytes(), np.uint32)[0]) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def check_logits_exact(o):
    """Router logits are the exact dot products rounded once to fp32 (Fraction arithmetic)."""
    x = _rand(31, 6, 7).astype(np.float32)
    w = _rand(32, 5, 7)
    got = o.router_logits(x, w)
    for n in range(6):
        for e in range(5):
            exact = sum(Fraction(float(x[n, d])) * Fraction(float(w[e, d])) for d in range(7))
            assert got[n, e] == _round_f32(exact), (n, e)


def check_library_equivalents(o):
    """Histogram = numpy.bincount, scan = cumsum, permutation = stable argsort by expert."""
    rng = np.random.default_rng(41)
    N, k, E = 300, 3, 11
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(N)]).astype(np.int32)
    counts = o.expert_counts(idx, E)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    off = o.exclusive_scan(counts)
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(counts)]))
    row_map, perm_token = o.stable_permutation(idx, off)
    order = np.argsort(idx.ravel(), kind="stable")
    assert np.array_equal(perm_token, order // k)
    inv = np.empty_like(order)
    inv[order] = np.arange(N * k)
    assert np.array_equal(row_map.ravel(), inv)


# ---- brute force ----------------------------------------------------------------------

def check_bruteforce_topk(o):
    """For E <= 10, k <= 4: the chosen set maximises the summed selection score, ties going
    to the lexicographically smallest sorted id tuple; the order is descending score.
    Integer-valued scores make ties frequent and sums exact."""
    rng = np.random.default_rng(51)
    for trial in range(200):
        E = int(rng.integers(2, 11))
        k = int(rng.integers(1, min(4, E) + 1))
        logits = rng.integers(-3, 4, size=(1, E)).astype(np.float32)
        bias = rng.integers(-2, 3, size=E).astype(np.float32)
        sel, _ = o.selection_scores(logits, bias, "softmax")
        idx, _ = o.select_topk(sel, k)
        best = None
        for sub in itertools.combinations(range(E), k):
            key = (-sum(sel[0, list(sub)]), sub)
            if best is None or key < best:
                best = key
        assert tuple(sorted(idx[0].tolist())) == best[1], (logits, bias, k, idx)
        s = sel[0, idx[0]]
        assert all(s[i] > s[i + 1] or (s[i] == s[i + 1] and idx[0][i] < idx[0][i + 1])
                   for i in range(k - 1))


# ---- invariants -----------------------------------------------------------------------

def check_invariants(o):
    """Gates >= 0 summing to 1; counts sum to N k; offsets end at N k; the permutation is a
    bijection, grouped by expert, token ids ascending inside each group; the bias moves the
    selection but never the gates of a given set; a constant bias shift changes nothing."""
    rng = np.random.default_rng(61)
    N, D, E, k = 200, 32, 12, 3
    x, w = _rand(62, N, D), _rand(63, E, D, scale=1 / math.sqrt(D))
    for fn in ("softmax", "sigmoid"):
        b = (rng.standard_normal(E) * 0.3).astype(np.float32)
        r = o.route(x, w, b, k, fn)
        assert np.all(r["gate"] >= 0) and np.allclose(r["gate"].sum(1), 1, atol=1e-12)
        # gates of the same set without bias
        _, s0 = o.selection_scores(r["logits"], None, fn)
        assert np.allclose(o.gates(r["logits"], s0, r["idx"], fn), r["gate"], atol=0, rtol=0)
        # bias shift by a constant (a power of two keeps fp32 sums exact) keeps everything
        r2 = o.route(x, w, b + np.float32(0.5), k, fn)
        assert np.array_equal(r2["idx"], r["idx"]) and np.allclose(r2["gate"], r["gate"], atol=0)
        # the bias does change the selection of some tokens
        r3 = o.route(x, w, (rng.standard_normal(E) * 3).astype(np.float32), k, fn)
        assert not np.array_equal(r3["idx"], r["idx"])
        counts = o.expert_counts(r["idx"], E)
        off = o.exclusive_scan(counts)
        assert counts.sum() == N * k and off[-1] == N * k
        row_map, perm = o.stable_permutation(r["idx"], off)
        assert np.array_equal(np.sort(row_map.ravel()), np.arange(N * k))
        for e in range(E):
            seg = perm[off[e]:off[e + 1]]
            assert np.all(np.diff(seg) > 0)
            assert np.all((r["idx"][seg] == e).any(1))
        for n in range(N):
            for j in range(k):
                assert perm[row_map[n, j]] == n
                e = r["idx"][n, j]
                assert off[e] <= row_map[n, j] < off[e + 1]


def check_bias_update_rule(o):
    """One +-gamma step: over-used experts go down by gamma, under-used up, exact target
    unchanged; fp32 arithmetic."""
    counts = np.array([5, 3, 4, 0, 4], np.int64)       # R = 16, E = 5 ... target 3.2
    b = np.array([0.0, 0.25, -0.5, 1.0, 0.0], np.float32)
    new, mm = o.bias_update(b, counts, 16, 0.125)
    assert new.dtype == np.float32
    assert new.tolist() == [-0.125, 0.375, -0.625, 1.125, -0.125]
    assert abs(mm - 5 / 3.2) < 1e-12
    new, _ = o.bias_update(b, np.array([4, 4, 4, 4, 4]), 20, 0.125)
    assert new.tolist() == b.tolist()


def check_bias_dynamics(o):
    """Repeated +-gamma steps drive a skewed router's usage toward uniform (lesson,
    'Build it' step 2 and exercise 1: balance over ~50 updates)."""
    rng = np.random.default_rng(71)
    N, D, E, k = 512, 64, 16, 2
    x = rng.standard_normal((N, D)).astype(np.float32) + 0.5
    c = np.log(np.arange(1, E + 1, dtype=np.float64) ** -1.2 / np.sum(np.arange(1, E + 1) ** -1.2))
    w = (rng.standard_normal((E, D)) / math.sqrt(D) + c[:, None] / (0.5 * D)).astype(np.float32)
    def run(gamma, steps):
        b = np.zeros(E, np.float32)
        hist = []
        for _ in range(steps):
            r = o.route(x, w, b, k, "softmax")
            counts = o.expert_counts(r["idx"], E)
            b, mm = o.bias_update(b, counts, N * k, gamma)
            hist.append(mm)
        return hist, b
    hist, _ = run(1e-3, 50)
    assert hist[-1] < hist[0]
    hist, b = run(0.05, 50)
    assert hist[-1] < 0.6 * hist[0] and hist[-1] < 1.6, hist
    # the most popular expert gets the most negative bias
    assert b[0] == b.min()


def check_capacity(o):
    """Expert capacity (lesson, load-balancing item 2): hand example, the no-op and the
    drop-everything limits, and the kept set = first `capacity` slots per expert."""
    # five tokens, k = 1, all to expert 0; capacity 2 keeps tokens 0 and 1
    idx = np.zeros((5, 1), np.int32)
    counts = o.expert_counts(idx, 2)
    off = o.exclusive_scan(np.minimum(counts, 2))
    rm, pt = o.stable_permutation(idx, off, 2)
    assert rm.ravel().tolist() == [0, 1, -1, -1, -1] and pt.tolist() == [0, 1]
    assert o.expert_capacity(1.0, 8, 2, 4) == 4 and o.expert_capacity(1.25, 10, 2, 4) == 7
    rng = np.random.default_rng(81)
    N, D, E, k, F = 40, 16, 6, 2, 8
    x, h = _rand(82, N, D), _rand(83, N, D)
    w = _rand(84, E, D)
    wg, wu, wd = _rand(85, E, F, D, scale=.3), _rand(86, E, F, D, scale=.3), _rand(87, E, D, F, scale=.3)
    full = o.moe_layer(x, h, w, None, wg, wu, wd, k)
    big = o.moe_layer(x, h, w, None, wg, wu, wd, k, capacity=N * k)
    assert np.array_equal(big["row_map"], full["row_map"]) and np.allclose(big["out"], full["out"], atol=0)
    none = o.moe_layer(x, h, w, None, wg, wu, wd, k, capacity=0)
    assert np.all(none["row_map"] == -1) and np.allclose(none["out"], h, atol=0)
    cap = 9
    r = o.moe_layer(x, h, w, None, wg, wu, wd, k, capacity=cap)
    assert np.array_equal(r["counts"], full["counts"])          # demand, before dropping
    flat_e, flat_r = r["idx"].ravel(), r["row_map"].ravel()
    for e in range(E):
        slots = np.where(flat_e == e)[0]
        assert np.all(flat_r[slots[:cap]] >= 0) and np.all(flat_r[slots[cap:]] == -1)
    # a dropped slot contributes nothing; kept slots contribute gate * expert output
    want = h.astype(np.float64).copy()
    for n in range(N):
        for j in range(k):
            if r["row_map"][n, j] >= 0:
                e = r["idx"][n, j]
                want[n] += r["gate"][n, j] * o.swiglu_expert(x[n:n + 1], wg[e], wu[e], wd[e])[0]
    assert np.allclose(r["out"], want, rtol=1e-12, atol=1e-12)


def check_token_outputs(o):
    """The layer formula evaluated for a few tokens, one expert at a time (what checks
    sampled tokens of full-size layers), equals the same formula in torch float64 from the
    same routing, and the whole layer's output on those tokens (lesson 'Concept' and
    'Shared experts': out = h + shared(xn) + sum_j gate_j * Expert_j(xn))."""
    N, D, E, F, k = 12, 16, 6, 10, 3
    x, h = _rand(91, N, D), _rand(92, N, D)
    w = _rand(93, E, D)
    wg, wu, wd = _rand(94, E, F, D, scale=.3), _rand(95, E, F, D, scale=.3), _rand(96, E, D, F, scale=.3)
    sh = (_rand(97, 1, F, D, scale=.3), _rand(98, 1, F, D, scale=.3), _rand(99, 1, D, F, scale=.3))
    for fn, shared in (("sigmoid", sh), ("softmax", None)):
        r = o.moe_layer(x, h, w, None, wg, wu, wd, k, fn, shared=shared)
        toks = np.array([0, 5, 11])
        got = o.token_outputs(toks, x[toks], h[toks], r["idx"][toks], r["gate"][toks],
                              lambda e: (wg[e], wu[e], wd[e]),
                              shared=None if shared is None else tuple(t[0] for t in shared))
        t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
        swiglu = lambda xx, a, b, c: (torch.nn.functional.silu(xx @ t(a).T) * (xx @ t(b).T)) @ t(c).T
        ref = t(h[toks]).clone()
        for i, n in enumerate(toks):
            xx = t(x[n:n + 1])
            if shared is not None:
                ref[i] += swiglu(xx, sh[0][0], sh[1][0], sh[2][0])[0]
            for j in range(k):
                e = int(r["idx"][n, j])
                ref[i] += float(r["gate"][n, j]) * swiglu(xx, wg[e], wu[e], wd[e])[0]
        assert np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12), fn
        assert np.allclose(got, r["out"][toks], rtol=1e-12, atol=1e-12), fn


ALL_CHECKS = [check_route_golden, check_layer_golden, check_dense_reduction, check_split_dense,
              check_all_chosen, check_logits_exact, check_library_equivalents,
              check_bruteforce_topk, check_invariants, check_bias_update_rule, check_bias_dynamics,
              check_capacity, check_token_outputs]
