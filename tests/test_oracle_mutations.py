"""Plant plausible mistakes in a private copy of the oracle and check that its pins catch
each one (a dropped term, a wrong sign or index, a transposed operand, a wrong tie rule)."""
import importlib.util
import os

import numpy as np
import pytest

from tests.oracle_pins import ALL_CHECKS

ORACLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "oracle", "moe_oracle.py")


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("moe_oracle_mutant", ORACLE)
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _gates_from_biased(m):
    orig = m.route
    def route(xn, w_router, bias, k, score_fn="softmax"):
        r = orig(xn, w_router, bias, k, score_fn)
        rows = np.arange(r["idx"].shape[0])[:, None]
        c = r["sel"][rows, r["idx"]]
        ex = np.exp(c - c.max(1, keepdims=True))
        r["gate"] = ex / ex.sum(1, keepdims=True)
        return r
    m.route = route


def _ties_to_higher_id(m):
    def select_topk(sel, k):
        key = np.where(np.isnan(sel), -np.inf, sel)
        E = sel.shape[1]
        order = (E - 1 - np.argsort(-key[:, ::-1], axis=1, kind="stable"))
        gap = key[np.arange(len(key)), order[:, k - 1]] - key[np.arange(len(key)), order[:, min(k, E - 1)]]
        return order[:, :k].astype(np.int32), gap
    m.select_topk = select_topk


def _silu_on_up(m):
    def swiglu_expert(x, w_gate, w_up, w_down):
        x = np.asarray(x, np.float64)
        g = x @ np.asarray(w_gate, np.float64).T
        u = x @ np.asarray(w_up, np.float64).T
        return (g * m.silu(u)) @ np.asarray(w_down, np.float64).T
    m.swiglu_expert = swiglu_expert


def _no_residual(m):
    orig = m.combine
    m.combine = lambda y, rm, g, residual=None, shared_y=None: orig(y, rm, g, None, shared_y)


def _no_shared(m):
    orig = m.combine
    m.combine = lambda y, rm, g, residual=None, shared_y=None: orig(y, rm, g, residual, None)


def _bias_sign_flipped(m):
    orig = m.bias_update
    def bias_update(b, counts, total, gamma):
        return orig(b, counts, total, -gamma)
    m.bias_update = bias_update


def _unstable_permutation(m):
    def stable_permutation(idx, offsets):
        idx = np.asarray(idx)
        N, k = idx.shape
        nxt = np.array(offsets[1:], dtype=np.int64).copy()
        row_map = np.empty((N, k), np.int64)
        perm = np.empty(N * k, np.int64)
        for n in range(N):
            for j in range(k):
                e = idx[n, j]
                nxt[e] -= 1
                row_map[n, j] = nxt[e]
                perm[nxt[e]] = n
        return row_map, perm
    m.stable_permutation = stable_permutation


def _sigmoid_unnormalised(m):
    orig = m.gates
    def gates(logits32, s, idx, fn):
        if fn == "sigmoid":
            return s[np.arange(idx.shape[0])[:, None], idx]
        return orig(logits32, s, idx, fn)
    m.gates = gates


def _softmax_no_max_subtract_all_experts(m):
    # softmax over ALL experts instead of over the chosen ones
    orig = m.gates
    def gates(logits32, s, idx, fn):
        if fn == "softmax":
            l = np.asarray(logits32, np.float64)
            p = np.exp(l) / np.exp(l).sum(1, keepdims=True)
            return p[np.arange(idx.shape[0])[:, None], idx]
        return orig(logits32, s, idx, fn)
    m.gates = gates


def _down_transposed_slice(m):
    def grouped_swiglu(x_perm, offsets, w_gate, w_up, w_down):
        x_perm = np.asarray(x_perm, np.float64)
        y = np.zeros((x_perm.shape[0], np.asarray(w_down).shape[1]))
        for e in range(len(offsets) - 1):
            a, b = int(offsets[e]), int(offsets[e + 1])
            ee = (e + 1) % (len(offsets) - 1)  # wrong expert's weights
            if b > a:
                y[a:b] = m.swiglu_expert(x_perm[a:b], w_gate[ee], w_up[ee], w_down[ee])
        return y
    m.grouped_swiglu = grouped_swiglu


def _logits_bf16(m):
    def router_logits(xn, w_router):
        import torch
        x = torch.tensor(np.asarray(xn, np.float32)).bfloat16()
        w = torch.tensor(np.asarray(w_router, np.float32)).bfloat16()
        return (x.double() @ w.double().T).float().numpy()
    m.router_logits = router_logits


def _inclusive_scan(m):
    def exclusive_scan(counts):
        c = np.cumsum(np.asarray(counts, np.int64))
        return np.concatenate([c, c[-1:]])
    m.exclusive_scan = exclusive_scan


def _token_outputs_no_shared(m):
    orig = m.token_outputs
    def token_outputs(tokens, xn_rows, h_rows, idx_rows, gate_rows, expert_weights, shared=None):
        return orig(tokens, xn_rows, h_rows, idx_rows, gate_rows, expert_weights, None)
    m.token_outputs = token_outputs


def _token_outputs_gate_of_next_slot(m):
    orig = m.token_outputs
    def token_outputs(tokens, xn_rows, h_rows, idx_rows, gate_rows, expert_weights, shared=None):
        return orig(tokens, xn_rows, h_rows, idx_rows, np.roll(gate_rows, 1, axis=1), expert_weights, shared)
    m.token_outputs = token_outputs


MUTATIONS = [_gates_from_biased, _ties_to_higher_id, _silu_on_up, _no_residual, _no_shared,
             _bias_sign_flipped, _unstable_permutation, _sigmoid_unnormalised,
             _softmax_no_max_subtract_all_experts, _down_transposed_slice, _logits_bf16,
             _inclusive_scan, _token_outputs_no_shared, _token_outputs_gate_of_next_slot]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=lambda f: f.__name__.strip("_"))
def test_pins_catch_planted_mistake(mutate):
    m = fresh_oracle()
    mutate(m)
    caught = []
    for check in ALL_CHECKS:
        try:
            check(m)
        except Exception as exc:  # noqa: BLE001 -- any failure counts as caught
            caught.append(check.__name__)
    assert caught, f"no pin caught mutation {mutate.__name__}"
