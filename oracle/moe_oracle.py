"""CPU oracle for the top-k MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy in float64.  Only the test suite, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the CUDA library and imports nothing from the
package; callers hand it plain arrays (bf16 tensors arrive as float32/float64
values, which hold every bf16 exactly).

Sources, cited by page title and section:

* [Lesson] "Mixture of Experts" lesson of the *AI Engineering from Scratch*
  course (Phase 07, Transformers Deep Dive): section "Concept" (the MoE block:
  router scores on norm(h), argmax_k, gated sum of expert outputs added to h),
  section "Load-balancing problem" (item 3: auxiliary-loss-free bias), section
  "Shared experts", and "Build it", step 1 (the router: raw dot products, bias
  added for selection only, stable sort by descending biased score, softmax over
  the chosen experts' *original* scores) and step 2 (per-expert firing counts
  drive a +-gamma bias step).
* [Handbook news] AREX Feed article on "The Ultimate MoE Training Handbook",
  paragraph on router precision (bf16 rounding can tie two close logits and
  change the winner, so the router stays fp32; GLM uses a sigmoid router) and
  the paragraph on the teaching model and upcycling (the k chosen experts hold
  as many FFN parameters as the dense layer they replace; a 1-expert MoE built
  from a dense checkpoint tracks the dense run).
* [Handbook post] the announcement's question list (softmax, sigmoid or
  sqrt(softplus) router; loss-free bias; serving with fewer experts per token).
* [Eval article] "MoE混合专家模型训练方案的评测维度与方法解析", evaluation
  dimensions table and section "1. 专家负载均衡的评测" (per-expert routed-token
  histogram).

Readings where the pages leave a step open:

* Sigmoid router: selection on sigma(logit) + bias, gates sigma_i / sum over the
  chosen sigma_j (unbiased).  No routed scaling factor, no group limit.
* sqrt(softplus) router (named in the handbook post): read the same way with
  s = sqrt(ln(1 + e^logit)).
* Order of the k outputs: descending biased score, ties to the lower expert id
  (a stable sort).  NaN scores rank as -inf.
* Bias step: b_e <- b_e + gamma * sign(R/E - count_e), sign(0) = 0, in fp32,
  applied after the forward whose counts drive it.
* Expert: SwiGLU without biases, y = W_down (SiLU(W_gate x) * (W_up x)),
  SiLU(z) = z * sigmoid(z).
* Permutation: slots (n, j) are sorted by expert, stably in slot order n*k + j.
"""
from __future__ import annotations

import numpy as np

NEAR_TIE_GAP = 1e-6


# --------------------------------------------------------------------------------------
# Router  [Lesson, "Build it" step 1; Handbook news, router-precision paragraph]
# --------------------------------------------------------------------------------------

def router_logits(xn, w_router):
    """logits[n, e] = sum_d xn[n, d] * W_r[e, d], in float64, rounded once to fp32.

    The router is one linear layer scoring each token against each expert; it is
    kept in fp32 because bf16 rounding can merge two close logits.
    """
    x = np.asarray(xn, dtype=np.float64)
    w = np.asarray(w_router, dtype=np.float64)
    return (x @ w.T).astype(np.float32)


def selection_scores(logits32, bias32, score_fn):
    """Biased score used only to choose experts, and the unbiased score the gates use.

    softmax mode: sel = logit + b, gates later from the raw logits.
    sigmoid mode: s = 1 / (1 + exp(-logit)), sel = s + b, gates later from s.
    sqrt_softplus mode: s = sqrt(ln(1 + exp(logit))), sel = s + b, gates later from s.
    All computed in float64 from the fp32 logit and the fp32 bias.
    """
    l64 = np.asarray(logits32, dtype=np.float32).astype(np.float64)
    b64 = np.zeros(l64.shape[-1]) if bias32 is None else \
        np.asarray(bias32, dtype=np.float32).astype(np.float64)
    if score_fn == "softmax":
        s = l64
    elif score_fn == "sigmoid":
        s = 1.0 / (1.0 + np.exp(-l64))
    elif score_fn == "sqrt_softplus":
        s = np.sqrt(np.logaddexp(0.0, l64))
    else:
        raise ValueError(score_fn)
    return s + b64[None, :], s


def select_topk(sel, k):
    """Indices of the k largest sel per row, in descending order; ties -> lower id.

    A stable sort by -sel over expert ids 0..E-1 gives exactly this order.  NaN
    ranks as -inf.  Also returns the gap between the k-th and (k+1)-th score.
    """
    key = np.where(np.isnan(sel), -np.inf, sel)
    order = np.argsort(-key, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int32)
    if k < sel.shape[1]:
        rows = np.arange(sel.shape[0])
        gap = key[rows, order[:, k - 1]] - key[rows, order[:, k]]
    else:
        gap = np.full(sel.shape[0], np.inf)
    return idx, gap


def gates(logits32, s_unbiased, idx, score_fn):
    """Gate weights over the chosen experts from their ORIGINAL (unbiased) scores.

    softmax mode: g_j = exp(l_j - max) / sum_i exp(l_i - max) over the chosen logits.
    sigmoid and sqrt_softplus modes: g_j = s_j / sum_i s_i over the chosen scores.
    """
    rows = np.arange(idx.shape[0])[:, None]
    if score_fn == "softmax":
        c = np.asarray(logits32, dtype=np.float32).astype(np.float64)[rows, idx]
        ex = np.exp(c - c.max(axis=1, keepdims=True))
        return ex / ex.sum(axis=1, keepdims=True)
    c = s_unbiased[rows, idx]
    return c / c.sum(axis=1, keepdims=True)


def route(xn, w_router, bias, k, score_fn="softmax"):
    """Full routing of a batch: logits, top-k ids, gates, near-tie flags and gaps."""
    logits = router_logits(xn, w_router)
    sel, s = selection_scores(logits, bias, score_fn)
    idx, gap = select_topk(sel, k)
    g = gates(logits, s, idx, score_fn)
    return dict(logits=logits, sel=sel, idx=idx, gate=g, gap=gap,
                near_tie=(gap < NEAR_TIE_GAP))


# --------------------------------------------------------------------------------------
# Histogram, scan, permutation  [Lesson, "Build it" step 2; Eval article, load histogram]
# --------------------------------------------------------------------------------------

def expert_counts(idx, E):
    """counts[e] = number of (token, slot) pairs routed to expert e."""
    flat = np.asarray(idx).reshape(-1)
    return np.array([int(np.sum(flat == e)) for e in range(E)], dtype=np.int64)


def exclusive_scan(counts):
    """offsets[0] = 0, offsets[e + 1] = offsets[e] + counts[e]."""
    off = np.zeros(len(counts) + 1, dtype=np.int64)
    for e in range(len(counts)):
        off[e + 1] = off[e] + counts[e]
    return off


def stable_permutation(idx, offsets, capacity=None):
    """Counting sort of slots by expert, stable in slot order.

    Slot s = n*k + j goes to row offsets[e] + (#earlier slots with the same e).
    Returns row_map[N, k] (slot -> row) and perm_token (row -> token).

    With a per-expert capacity [Lesson, "Load-balancing problem" item 2: each expert takes at
    most so many tokens, the overflow skips the layer], only the first `capacity` slots of an
    expert (in slot order) get a row; the others get row -1.  `offsets` must then be the
    exclusive scan of the kept counts min(count, capacity).
    """
    idx = np.asarray(idx)
    N, k = idx.shape
    nxt = np.array(offsets[:-1], dtype=np.int64).copy()
    seen = np.zeros(len(offsets) - 1, dtype=np.int64)
    row_map = np.empty((N, k), dtype=np.int64)
    perm_token = np.empty(int(offsets[-1]), dtype=np.int64)
    for n in range(N):
        for j in range(k):
            e = idx[n, j]
            if capacity is not None and seen[e] >= capacity:
                row_map[n, j] = -1
            else:
                row_map[n, j] = nxt[e]
                perm_token[nxt[e]] = n
                nxt[e] += 1
            seen[e] += 1
    return row_map, perm_token


def expert_capacity(capacity_factor, N, k, E):
    """Slots per expert for a capacity factor C: ceil(C * N * k / E)."""
    return int(np.ceil(capacity_factor * N * k / E))


# --------------------------------------------------------------------------------------
# Experts  [Lesson, "Concept" (each expert an independent SwiGLU FFN), "Shared experts"]
# --------------------------------------------------------------------------------------

def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu_expert(x, w_gate, w_up, w_down):
    """y = W_down (SiLU(W_gate x) * (W_up x)) for rows x, all in float64 (H not rounded)."""
    x = np.asarray(x, dtype=np.float64)
    g = x @ np.asarray(w_gate, dtype=np.float64).T
    u = x @ np.asarray(w_up, dtype=np.float64).T
    return (silu(g) * u) @ np.asarray(w_down, dtype=np.float64).T


def grouped_swiglu(x_perm, offsets, w_gate, w_up, w_down):
    """Apply expert e to rows offsets[e] .. offsets[e+1]-1 of the permuted activations."""
    x_perm = np.asarray(x_perm, dtype=np.float64)
    y = np.zeros((x_perm.shape[0], np.asarray(w_down).shape[1]), dtype=np.float64)
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b] = swiglu_expert(x_perm[a:b], w_gate[e], w_up[e], w_down[e])
    return y


def combine(y_perm, row_map, gate, residual=None, shared_y=None):
    """out[n] = h[n] + shared[n] + sum_j gate[n, j] * Y[row_map[n, j]]   (float64)."""
    y_perm = np.asarray(y_perm, dtype=np.float64)
    N, k = row_map.shape
    out = np.zeros((N, y_perm.shape[1]), dtype=np.float64)
    if residual is not None:
        out += np.asarray(residual, dtype=np.float64)
    if shared_y is not None:
        out += np.asarray(shared_y, dtype=np.float64)
    g = np.asarray(gate, dtype=np.float64)
    for j in range(k):
        kept = np.where(row_map[:, j] >= 0)[0]        # a dropped slot (row -1) adds nothing
        out[kept] += g[kept, j:j + 1] * y_perm[row_map[kept, j]]
    return out


# --------------------------------------------------------------------------------------
# Loss-free balancing bias  [Lesson, "Load-balancing problem" item 3 and "Build it" step 2]
# --------------------------------------------------------------------------------------

def bias_update(bias32, counts, total_assignments, gamma):
    """b_e <- b_e + gamma * sign(R/E - count_e) in fp32; returns (new bias, max/mean load).

    sign(R/E - c) is taken exactly as sign(R - E*c) on integers.
    """
    counts = np.asarray(counts, dtype=np.int64)
    E = len(counts)
    sgn = np.sign(int(total_assignments) - E * counts).astype(np.float32)
    b = np.asarray(bias32, dtype=np.float32)
    new = (b + np.float32(gamma) * sgn).astype(np.float32)
    mean = total_assignments / E
    return new, float(counts.max() / mean) if mean > 0 else 0.0


# --------------------------------------------------------------------------------------
# The layer  [Lesson, "Concept": h + sum_{e in top_k} gate(scores[e]) * Expert_e(norm(h))]
# --------------------------------------------------------------------------------------

def moe_layer(xn, h, w_router, bias, w_gate, w_up, w_down, k, score_fn="softmax",
              shared=None, gamma=None, idx_override=None, gate_override=None, capacity=None):
    """The whole forward on CPU.  Returns every intermediate the CUDA path exposes.

    ``shared`` = (w_gate[1,Fs,D], w_up[1,Fs,D], w_down[1,D,Fs]) or None.
    ``idx_override`` / ``gate_override`` replace the router's choice (routing replay).
    ``capacity`` = slots kept per expert (None: no limit); ``counts`` stays the routed
    demand, which drives the bias step.
    """
    xn = np.asarray(xn, dtype=np.float64)
    E = np.asarray(w_router).shape[0]
    r = route(xn, w_router, bias, k, score_fn)
    idx = r["idx"] if idx_override is None else np.asarray(idx_override, dtype=np.int32)
    g = r["gate"] if gate_override is None else np.asarray(gate_override, dtype=np.float64)
    counts = expert_counts(idx, E)
    kept = counts if capacity is None else np.minimum(counts, capacity)
    offsets = exclusive_scan(kept)
    row_map, perm_token = stable_permutation(idx, offsets, capacity)
    x_perm = xn[perm_token]
    y_perm = grouped_swiglu(x_perm, offsets, w_gate, w_up, w_down)
    y_sh = None
    if shared is not None:
        y_sh = swiglu_expert(xn, shared[0][0], shared[1][0], shared[2][0])
    out = combine(y_perm, row_map, g, residual=h, shared_y=y_sh)
    res = dict(r, idx=idx, gate=g, counts=counts, offsets=offsets, row_map=row_map,
               perm_token=perm_token, x_perm=x_perm, y_perm=y_perm, shared_y=y_sh, out=out)
    if gamma is not None:
        res["bias_new"], res["max_over_mean"] = bias_update(
            np.zeros(E, np.float32) if bias is None else bias, counts, idx.size, gamma)
    return res


def token_outputs(tokens, xn_rows, h_rows, idx_rows, gate_rows, expert_weights, shared=None):
    """out[n] for a few tokens only, straight from the layer formula.

    ``expert_weights(e)`` returns (w_gate[F,D], w_up[F,D], w_down[D,F]) of expert e;
    ``shared`` is the shared expert's (w_gate, w_up, w_down) or None.  Used to check
    sampled tokens of full-size layers without running every expert on the CPU.
    """
    xn_rows = np.asarray(xn_rows, dtype=np.float64)
    out = np.asarray(h_rows, dtype=np.float64).copy()
    cache = {}
    for i in range(len(tokens)):
        x = xn_rows[i:i + 1]
        if shared is not None:
            out[i] += swiglu_expert(x, *shared)[0]
        for j in range(idx_rows.shape[1]):
            e = int(idx_rows[i, j])
            if e not in cache:
                cache[e] = expert_weights(e)
            out[i] += float(gate_rows[i, j]) * swiglu_expert(x, *cache[e])[0]
    return out
