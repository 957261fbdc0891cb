"""Python binding of the C ABI in include/moe.h (ctypes; argument marshalling only).

Every function takes torch CUDA tensors, passes their device pointers and the current
torch stream to the library, and raises ``MoEError`` on a non-zero status.  Outputs
that are not supplied are allocated with ``torch.empty`` on the input's device.
There is no CPU path: without the built ``libmoe.so`` every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")
_lib = None

MOE_F32, MOE_BF16 = 0, 1
SCORE_FN = {"softmax": 0, "sigmoid": 1, "sqrt_softplus": 2}
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_CUDA",
          -4: "MOE_ERR_TIMEOUT", -5: "MOE_ERR_NAN_INPUT"}
EXPORTS = ("moe_status_string", "moe_last_device_status", "moe_version", "moe_router_topk",
           "moe_permute_workspace_bytes", "moe_permute", "moe_grouped_swiglu",
           "moe_unpermute_combine", "moe_bias_update", "moe_permute_noalloc",
           "moe_permute_noalloc_max_scratch_bytes", "moe_router_split_bytes", "moe_router_split",
           "moe_router_topk_split", "moe_router_topk_split_workspace_bytes", "moe_permute_capacity",
           "moe_grouped_swiglu_gather", "moe_grouped_swiglu_ex", "moe_expert_capacity",
           "moe_selftest_bounded_wait", "moe_permute_update_bias", "moe_grouped_swiglu_shared",
           "moe_router_topk_split_shared", "moe_grouped_swiglu_shared_h")


class MoEError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {_LIB_PATH} (run __graft_entry__.build())")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    sig = {
        "moe_status_string": ([i32], ctypes.c_char_p),
        "moe_last_device_status": ([vp], i32),
        "moe_version": ([], i32),
        "moe_router_topk": ([vp, i32, i32, i32, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp], i32),
        "moe_permute_workspace_bytes": ([i32, i32, i32], sz),
        "moe_permute": ([vp, i32, i32, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp], i32),
        "moe_grouped_swiglu": ([vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp], i32),
        "moe_grouped_swiglu_ex": ([vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp], i32),
        "moe_grouped_swiglu_gather": ([vp, i32, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp], i32),
        "moe_unpermute_combine": ([vp, vp, vp, i32, i32, i32, vp, vp, vp, i32, vp], i32),
        "moe_bias_update": ([vp, i32, i64, f32, vp, vp, vp], i32),
        "moe_permute_capacity": ([vp, i32, i32, i32, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp], i32),
        "moe_permute_noalloc": ([vp, i32, i32, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp], i32),
        "moe_permute_noalloc_max_scratch_bytes": ([], sz),
        "moe_router_split_bytes": ([i32, i32], sz),
        "moe_router_split": ([vp, i32, i32, vp, vp], i32),
        "moe_router_topk_split": ([vp, i32, i32, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp], i32),
        "moe_router_topk_split_workspace_bytes": ([i32, i32, i32], sz),
        "moe_expert_capacity": ([ctypes.c_double, i32, i32, i32], i64),
        "moe_selftest_bounded_wait": ([vp, ctypes.c_longlong, vp, vp], i32),
        "moe_permute_update_bias": ([vp, i32, i32, i32, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, f32, vp,
                                     vp, vp], i32),
        "moe_grouped_swiglu_shared": ([vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp,
                                       vp, vp], i32),
        "moe_router_topk_split_shared": ([vp, i32, i32, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp, vp, i32,
                                          vp, vp], i32),
        "moe_grouped_swiglu_shared_h": ([vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp,
                                         vp], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes, f.restype = args, res
    _lib = L
    return L


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t):
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float32:
        return MOE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _chk(name, st):
    if st != 0:
        raise MoEError(name, st)


def _need(name, t, dtype=None, shape=None, device=None):
    """Check one tensor argument before its pointer reaches the library.  The kernels trust
    the sizes passed beside the pointers, so a wrong dtype, shape or device here would make
    them read or write past a buffer; None (an optional argument left out) passes."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def last_device_status(stream=None) -> int:
    return load().moe_last_device_status(_stream(stream))


def version() -> int:
    return load().moe_version()


def selftest_bounded_wait(src, steps_out, limit_cycles=2_000_000, stream=None):
    """Launch the library's bounded-wait self-test (moe_selftest_bounded_wait): `src` is a
    device buffer of at least 4096 bytes, `steps_out` a device int32[1].  Read the timeout
    it records with last_device_status()."""
    _need("steps_out", steps_out, torch.int32, (1,))
    _cuda(src, steps_out)
    if src.numel() * src.element_size() < 4096:
        raise ValueError("src: at least 4096 bytes")
    _chk("moe_selftest_bounded_wait", load().moe_selftest_bounded_wait(
        _p(src), int(limit_cycles), _p(steps_out), _stream(stream)))


def moe_router_topk(xn, w_router, bias, k, score_fn="softmax", logits_out=None, topk_idx=None,
                    topk_gate=None, near_tie=None, want_logits=True, want_near_tie=True, stream=None):
    """Router GEMM + biased top-k + gates.  Returns (logits, idx, gate, near_tie)."""
    L = load()
    N, D = xn.shape
    E = w_router.shape[0]
    dev = xn.device
    _need("w_router", w_router, torch.float32, (E, D), dev)
    _need("bias", bias, torch.float32, (E,), dev)
    _need("logits_out", logits_out, torch.float32, (N, E), dev)
    _need("topk_idx", topk_idx, torch.int32, (N, k), dev)
    _need("topk_gate", topk_gate, torch.float32, (N, k), dev)
    _need("near_tie", near_tie, torch.uint8, (N,), dev)
    if logits_out is None and want_logits:
        logits_out = torch.empty(N, E, dtype=torch.float32, device=dev)
    if topk_idx is None:
        topk_idx = torch.empty(N, k, dtype=torch.int32, device=dev)
    if topk_gate is None:
        topk_gate = torch.empty(N, k, dtype=torch.float32, device=dev)
    if near_tie is None and want_near_tie:
        near_tie = torch.empty(N, dtype=torch.uint8, device=dev)
    _cuda(xn, w_router, bias, logits_out, topk_idx, topk_gate, near_tie)
    _chk("moe_router_topk", L.moe_router_topk(
        _p(xn), _dt(xn), N, D, _p(w_router), _p(bias), E, k, SCORE_FN[score_fn], _p(logits_out),
        _p(topk_idx), _p(topk_gate), _p(near_tie), _stream(stream)))
    return logits_out, topk_idx, topk_gate, near_tie


def moe_router_split(w_router, w_split=None, stream=None):
    """fp32 [E, D] router weight -> bf16 [3, E, D] planes with hi + mid + lo == w exactly."""
    L = load()
    E, D = w_router.shape
    _need("w_router", w_router, torch.float32)
    _need("w_split", w_split, torch.bfloat16, (3, E, D), w_router.device)
    if w_split is None:
        w_split = torch.empty(3, E, D, dtype=torch.bfloat16, device=w_router.device)
    _cuda(w_router, w_split)
    _chk("moe_router_split", L.moe_router_split(_p(w_router), E, D, _p(w_split), _stream(stream)))
    return w_split


def router_split_workspace_bytes(N, D, E) -> int:
    return int(load().moe_router_topk_split_workspace_bytes(N, D, E))


def moe_router_topk_split(xn, w_split, bias, k, score_fn="softmax", logits_out=None, topk_idx=None,
                          topk_gate=None, near_tie=None, want_near_tie=True, workspace=None,
                          stream=None):
    """The router on tensor cores (bf16 xn, split fp32 weights).  Returns (logits, idx, gate, near_tie)."""
    L = load()
    N, D = xn.shape
    E = w_split.shape[1]
    dev = xn.device
    _need("xn", xn, torch.bfloat16)
    _need("w_split", w_split, torch.bfloat16, (3, E, D), dev)
    _need("bias", bias, torch.float32, (E,), dev)
    _need("logits_out", logits_out, torch.float32, (N, E), dev)
    _need("topk_idx", topk_idx, torch.int32, (N, k), dev)
    _need("topk_gate", topk_gate, torch.float32, (N, k), dev)
    _need("near_tie", near_tie, torch.uint8, (N,), dev)
    _need("workspace", workspace, device=dev)
    if logits_out is None:
        logits_out = torch.empty(N, E, dtype=torch.float32, device=dev)
    if topk_idx is None:
        topk_idx = torch.empty(N, k, dtype=torch.int32, device=dev)
    if topk_gate is None:
        topk_gate = torch.empty(N, k, dtype=torch.float32, device=dev)
    if near_tie is None and want_near_tie:
        near_tie = torch.empty(N, dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, router_split_workspace_bytes(N, D, E)), dtype=torch.uint8,
                                device=dev)
    _cuda(xn, w_split, bias, logits_out, topk_idx, topk_gate, near_tie, workspace)
    _chk("moe_router_topk_split", L.moe_router_topk_split(
        _p(xn), N, D, _p(w_split), _p(bias), E, k, SCORE_FN[score_fn], _p(logits_out), _p(topk_idx),
        _p(topk_gate), _p(near_tie), _p(workspace), workspace.numel(), _stream(stream)))
    return logits_out, topk_idx, topk_gate, near_tie


def moe_router_topk_split_shared(xn, w_split, bias, k, shared, score_fn="softmax", logits_out=None, topk_idx=None,
                                 topk_gate=None, near_tie=None, want_near_tie=True, workspace=None, hs_out=None,
                                 stream=None):
    """moe_router_topk_split and the shared expert's first GEMM (shared = (w_gate[1,F,D],
    w_up[1,F,D], ...)) in one launch over the same token tiles.  Returns (logits, idx, gate,
    near_tie, hs) with hs [N, F] bf16 the shared expert's H."""
    L = load()
    N, D = xn.shape
    E = w_split.shape[1]
    dev = xn.device
    sg, su = shared[0], shared[1]
    F = sg.shape[1]
    _need("xn", xn, torch.bfloat16)
    _need("w_split", w_split, torch.bfloat16, (3, E, D), dev)
    _need("bias", bias, torch.float32, (E,), dev)
    _need("shared w_gate", sg, torch.bfloat16, (1, F, D), dev)
    _need("shared w_up", su, torch.bfloat16, (1, F, D), dev)
    _need("logits_out", logits_out, torch.float32, (N, E), dev)
    _need("topk_idx", topk_idx, torch.int32, (N, k), dev)
    _need("topk_gate", topk_gate, torch.float32, (N, k), dev)
    _need("near_tie", near_tie, torch.uint8, (N,), dev)
    _need("workspace", workspace, device=dev)
    _need("hs_out", hs_out, torch.bfloat16, (N, F), dev)
    e = lambda *sh, dt: torch.empty(*sh, dtype=dt, device=dev)
    logits_out = e(N, E, dt=torch.float32) if logits_out is None else logits_out
    topk_idx = e(N, k, dt=torch.int32) if topk_idx is None else topk_idx
    topk_gate = e(N, k, dt=torch.float32) if topk_gate is None else topk_gate
    if near_tie is None and want_near_tie:
        near_tie = e(N, dt=torch.uint8)
    if workspace is None:
        workspace = e(max(1, router_split_workspace_bytes(N, D, E)), dt=torch.uint8)
    hs_out = e(N, F, dt=torch.bfloat16) if hs_out is None else hs_out
    _cuda(xn, w_split, bias, sg, su, logits_out, topk_idx, topk_gate, near_tie, workspace, hs_out)
    _chk("moe_router_topk_split_shared", L.moe_router_topk_split_shared(
        _p(xn), N, D, _p(w_split), _p(bias), E, k, SCORE_FN[score_fn], _p(logits_out), _p(topk_idx),
        _p(topk_gate), _p(near_tie), _p(workspace), workspace.numel(), _p(sg), _p(su), F, _p(hs_out),
        _stream(stream)))
    return logits_out, topk_idx, topk_gate, near_tie, hs_out


def permute_workspace_bytes(N, k, E) -> int:
    return int(load().moe_permute_workspace_bytes(N, k, E))


def expert_capacity(capacity_factor, N, k, E) -> int:
    """Slots per expert for a capacity factor C (moe_expert_capacity)."""
    c = int(load().moe_expert_capacity(float(capacity_factor), int(N), int(k), int(E)))
    if c < 0:
        raise ValueError(f"moe_expert_capacity rejected C={capacity_factor}, N={N}, k={k}, E={E}")
    return c


def moe_permute(xn, topk_idx, E, counts=None, offsets=None, row_map=None, perm_token=None,
                x_perm=None, workspace=None, rows=True, copy=True, capacity=None, stream=None,
                bias_step=None):
    """Histogram + scan + stable permutation (with an optional per-expert capacity).
    bias_step = (gamma, bias, max_over_mean or None): also apply the +-gamma step to `bias`
    from this call's counts (moe_permute_update_bias).
    Returns (counts, offsets, row_map, perm_token, x_perm)."""
    L = load()
    N, k = topk_idx.shape
    dev = topk_idx.device
    D = xn.shape[1] if xn is not None else 64
    _need("topk_idx", topk_idx, torch.int32)
    if xn is not None:
        _need("xn", xn, shape=(N, D), device=dev)
    _need("counts", counts, torch.int32, (E,), dev)
    _need("offsets", offsets, torch.int32, (E + 1,), dev)
    _need("row_map", row_map, torch.int32, (N, k), dev)
    _need("perm_token", perm_token, torch.int32, (N * k,), dev)
    _need("x_perm", x_perm, None if xn is None else xn.dtype, (N * k, D), dev)
    _need("workspace", workspace, device=dev)
    if counts is None:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
    if offsets is None:
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if rows and row_map is None:
        row_map = torch.empty(N, k, dtype=torch.int32, device=dev)
    if rows and perm_token is None:
        perm_token = torch.empty(N * k, dtype=torch.int32, device=dev)
    if copy and x_perm is None:
        x_perm = torch.empty(N * k, D, dtype=xn.dtype, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, permute_workspace_bytes(N, k, E)), dtype=torch.uint8, device=dev)
    dt = _dt(xn) if xn is not None else MOE_BF16
    _cuda(xn, topk_idx, counts, offsets, row_map, perm_token, x_perm, workspace)
    if bias_step is not None:
        gamma, bias, mom = bias_step
        _need("bias", bias, torch.float32, (E,), dev)
        _need("max_over_mean", mom, torch.float32, (1,), dev)
        _cuda(bias, mom)
        _chk("moe_permute_update_bias", L.moe_permute_update_bias(
            _p(xn) if copy else None, dt, N, D, _p(topk_idx), k, E,
            int(capacity) if capacity is not None else N * k, _p(counts), _p(offsets), _p(row_map),
            _p(perm_token), _p(x_perm) if copy else None, _p(workspace),
            workspace.numel() * workspace.element_size(), float(gamma), _p(bias), _p(mom), _stream(stream)))
    elif capacity is None:
        _chk("moe_permute", L.moe_permute(
            _p(xn) if copy else None, dt, N, D, _p(topk_idx), k, E, _p(counts), _p(offsets),
            _p(row_map), _p(perm_token), _p(x_perm) if copy else None, _p(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))
    else:
        _chk("moe_permute_capacity", L.moe_permute_capacity(
            _p(xn) if copy else None, dt, N, D, _p(topk_idx), k, E, int(capacity), _p(counts),
            _p(offsets), _p(row_map), _p(perm_token), _p(x_perm) if copy else None, _p(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))
    return counts, offsets, row_map, perm_token, x_perm


def moe_permute_noalloc(xn, topk_idx, E, counts, offsets, row_map, perm_token, x_perm,
                        stream=None):
    """moe_permute for callers that cannot allocate device memory: the library keeps the
    scratch in a fixed array of its own, so only inputs and outputs are passed in (all of
    them must already exist).  Calls on one device share that array: never run two at
    once on unordered streams."""
    L = load()
    N, k = topk_idx.shape
    D = xn.shape[1]
    dev = topk_idx.device
    _need("topk_idx", topk_idx, torch.int32)
    _need("xn", xn, shape=(N, D), device=dev)
    _need("counts", counts, torch.int32, (E,), dev)
    _need("offsets", offsets, torch.int32, (E + 1,), dev)
    _need("row_map", row_map, torch.int32, (N, k), dev)
    _need("perm_token", perm_token, torch.int32, (N * k,), dev)
    _need("x_perm", x_perm, xn.dtype, (N * k, D), dev)
    _cuda(xn, topk_idx, counts, offsets, row_map, perm_token, x_perm)
    _chk("moe_permute_noalloc", L.moe_permute_noalloc(
        _p(xn), _dt(xn), N, D, _p(topk_idx), k, E, _p(counts), _p(offsets), _p(row_map),
        _p(perm_token), _p(x_perm), _stream(stream)))
    return counts, offsets, row_map, perm_token, x_perm


def moe_grouped_swiglu(x_perm, offsets, w_gate, w_up, w_down, h_workspace=None, y_perm=None,
                       stream=None, max_ctas=0):
    """Grouped SwiGLU over per-group row blocks (on at most max_ctas CTAs; 0 = every SM).
    Returns y_perm."""
    L = load()
    M, D = x_perm.shape
    G, F, _ = w_gate.shape
    dt, dev = x_perm.dtype, x_perm.device
    _need("offsets", offsets, torch.int32, (G + 1,), dev)
    _need("w_gate", w_gate, dt, (G, F, D), dev)
    _need("w_up", w_up, dt, (G, F, D), dev)
    _need("w_down", w_down, dt, (G, D, F), dev)
    _need("h_workspace", h_workspace, dt, (M, F), dev)
    _need("y_perm", y_perm, dt, (M, D), dev)
    if h_workspace is None:
        h_workspace = torch.empty(M, F, dtype=x_perm.dtype, device=x_perm.device)
    if y_perm is None:
        y_perm = torch.empty(M, D, dtype=x_perm.dtype, device=x_perm.device)
    _cuda(x_perm, offsets, w_gate, w_up, w_down, h_workspace, y_perm)
    _chk("moe_grouped_swiglu_ex", L.moe_grouped_swiglu_ex(
        _p(x_perm), _dt(x_perm), _p(offsets), G, M, D, F, _p(w_gate), _p(w_up), _p(w_down),
        _p(h_workspace), _p(y_perm), int(max_ctas), _stream(stream)))
    return y_perm


def moe_grouped_swiglu_shared(x_perm, offsets, w_gate, w_up, w_down, xn, shared, h_workspace=None, y_perm=None,
                              hs_workspace=None, shared_y=None, stream=None, perm_token=None):
    """The routed experts' SwiGLU and the always-on shared expert's (shared = (w_gate[1,F,D],
    w_up[1,F,D], w_down[1,D,F]) on xn) in the same two launches (bf16).  With perm_token the
    routed rows are gathered from xn[perm_token] and x_perm may be None.  Returns
    (y_perm, shared_y)."""
    L = load()
    G, F, D = w_gate.shape
    M = perm_token.shape[0] if perm_token is not None else x_perm.shape[0]
    N = xn.shape[0]
    dt, dev = xn.dtype, xn.device
    sg, su, sd = shared
    _need("xn", xn, torch.bfloat16, (N, D))
    if perm_token is None and x_perm is None:
        raise ValueError("x_perm or perm_token is needed")
    _need("x_perm", x_perm, dt, (M, D), dev)
    _need("perm_token", perm_token, torch.int32, (M,), dev)
    _need("offsets", offsets, torch.int32, (G + 1,), dev)
    _need("w_gate", w_gate, dt, (G, F, D), dev)
    _need("w_up", w_up, dt, (G, F, D), dev)
    _need("w_down", w_down, dt, (G, D, F), dev)
    _need("shared w_gate", sg, dt, (1, F, D), dev)
    _need("shared w_up", su, dt, (1, F, D), dev)
    _need("shared w_down", sd, dt, (1, D, F), dev)
    _need("h_workspace", h_workspace, dt, (M, F), dev)
    _need("y_perm", y_perm, dt, (M, D), dev)
    _need("hs_workspace", hs_workspace, dt, (N, F), dev)
    _need("shared_y", shared_y, dt, (N, D), dev)
    e = lambda *sh: torch.empty(*sh, dtype=dt, device=dev)
    h_workspace = e(M, F) if h_workspace is None else h_workspace
    y_perm = e(M, D) if y_perm is None else y_perm
    hs_workspace = e(N, F) if hs_workspace is None else hs_workspace
    shared_y = e(N, D) if shared_y is None else shared_y
    _cuda(x_perm, perm_token, offsets, w_gate, w_up, w_down, xn, sg, su, sd, h_workspace, y_perm, hs_workspace,
          shared_y)
    _chk("moe_grouped_swiglu_shared", L.moe_grouped_swiglu_shared(
        _p(x_perm), _p(perm_token), _p(offsets), G, M, D, F, _p(w_gate), _p(w_up), _p(w_down), _p(h_workspace),
        _p(y_perm), _p(xn), N, _p(sg), _p(su), _p(sd), _p(hs_workspace), _p(shared_y), _stream(stream)))
    return y_perm, shared_y


def moe_grouped_swiglu_shared_h(x_perm, offsets, w_gate, w_up, w_down, xn, w_down_shared, hs, y_perm=None,
                                h_workspace=None, shared_y=None, stream=None, perm_token=None):
    """moe_grouped_swiglu_shared when hs [N, F] already holds the shared expert's H (from
    moe_router_topk_split_shared): the routed experts' SwiGLU and the shared expert's second
    GEMM (w_down_shared [1, D, F]) in the routed GEMM2 launch.  Returns (y_perm, shared_y)."""
    L = load()
    G, F, D = w_gate.shape
    M = perm_token.shape[0] if perm_token is not None else x_perm.shape[0]
    N = hs.shape[0]
    dt, dev = hs.dtype, hs.device
    if perm_token is None and x_perm is None:
        raise ValueError("x_perm or perm_token is needed")
    _need("hs", hs, torch.bfloat16, (N, F))
    _need("x_perm", x_perm, dt, (M, D), dev)
    _need("perm_token", perm_token, torch.int32, (M,), dev)
    _need("xn", xn, dt, (N, D), dev)
    _need("offsets", offsets, torch.int32, (G + 1,), dev)
    _need("w_gate", w_gate, dt, (G, F, D), dev)
    _need("w_up", w_up, dt, (G, F, D), dev)
    _need("w_down", w_down, dt, (G, D, F), dev)
    _need("shared w_down", w_down_shared, dt, (1, D, F), dev)
    _need("h_workspace", h_workspace, dt, (M, F), dev)
    _need("y_perm", y_perm, dt, (M, D), dev)
    _need("shared_y", shared_y, dt, (N, D), dev)
    e = lambda *sh: torch.empty(*sh, dtype=dt, device=dev)
    h_workspace = e(M, F) if h_workspace is None else h_workspace
    y_perm = e(M, D) if y_perm is None else y_perm
    shared_y = e(N, D) if shared_y is None else shared_y
    _cuda(x_perm, perm_token, xn, offsets, w_gate, w_up, w_down, w_down_shared, hs, h_workspace, y_perm, shared_y)
    _chk("moe_grouped_swiglu_shared_h", L.moe_grouped_swiglu_shared_h(
        _p(x_perm), _p(perm_token), _p(offsets), G, M, D, F, _p(w_gate), _p(w_up), _p(w_down), _p(h_workspace),
        _p(y_perm), _p(xn), N, _p(w_down_shared), _p(hs), _p(shared_y), _stream(stream)))
    return y_perm, shared_y


def moe_grouped_swiglu_gather(xn, perm_token, offsets, w_gate, w_up, w_down, h_workspace=None,
                              y_perm=None, stream=None):
    """Grouped SwiGLU whose row i reads xn[perm_token[i]] directly (bf16).  Returns y_perm."""
    L = load()
    M = perm_token.shape[0]
    N, D = xn.shape
    G, F, _ = w_gate.shape
    dt, dev = xn.dtype, xn.device
    _need("xn", xn, torch.bfloat16)
    _need("perm_token", perm_token, torch.int32, (M,), dev)
    _need("offsets", offsets, torch.int32, (G + 1,), dev)
    _need("w_gate", w_gate, dt, (G, F, D), dev)
    _need("w_up", w_up, dt, (G, F, D), dev)
    _need("w_down", w_down, dt, (G, D, F), dev)
    _need("h_workspace", h_workspace, dt, (M, F), dev)
    _need("y_perm", y_perm, dt, (M, D), dev)
    if h_workspace is None:
        h_workspace = torch.empty(M, F, dtype=xn.dtype, device=xn.device)
    if y_perm is None:
        y_perm = torch.empty(M, D, dtype=xn.dtype, device=xn.device)
    _cuda(xn, perm_token, offsets, w_gate, w_up, w_down, h_workspace, y_perm)
    _chk("moe_grouped_swiglu_gather", L.moe_grouped_swiglu_gather(
        _p(xn), N, _p(perm_token), _p(offsets), G, M, D, F, _p(w_gate), _p(w_up), _p(w_down),
        _p(h_workspace), _p(y_perm), _stream(stream)))
    return y_perm


def moe_unpermute_combine(y_perm, row_map, topk_gate, shared_y=None, residual=None, out=None,
                          stream=None):
    """out = residual + shared_y + sum_j gate[:, j] * y_perm[row_map[:, j]]."""
    L = load()
    N, k = row_map.shape
    D = y_perm.shape[1]
    dt, dev = y_perm.dtype, y_perm.device
    _need("row_map", row_map, torch.int32, device=dev)
    _need("topk_gate", topk_gate, torch.float32, (N, k), dev)
    _need("shared_y", shared_y, dt, (N, D), dev)
    _need("residual", residual, dt, (N, D), dev)
    _need("out", out, dt, (N, D), dev)
    if out is None:
        out = torch.empty(N, D, dtype=y_perm.dtype, device=y_perm.device)
    _cuda(y_perm, row_map, topk_gate, shared_y, residual, out)
    _chk("moe_unpermute_combine", L.moe_unpermute_combine(
        _p(y_perm), _p(row_map), _p(topk_gate), N, k, D, _p(shared_y), _p(residual), _p(out),
        _dt(y_perm), _stream(stream)))
    return out


def moe_bias_update(counts, bias, total_assignments, gamma, max_over_mean=None, stream=None):
    """bias += gamma * sign(total/E - counts), in place.  Returns max_over_mean (device fp32[1])."""
    L = load()
    E = counts.shape[0]
    _need("counts", counts, torch.int32)
    _need("bias", bias, torch.float32, (E,), counts.device)
    _need("max_over_mean", max_over_mean, torch.float32, (1,), counts.device)
    if max_over_mean is None:
        max_over_mean = torch.empty(1, dtype=torch.float32, device=counts.device)
    _cuda(counts, bias, max_over_mean)
    _chk("moe_bias_update", L.moe_bias_update(
        _p(counts), E, int(total_assignments), float(gamma), _p(bias), _p(max_over_mean),
        _stream(stream)))
    return max_over_mean


def global_counts(counts, group=None):
    """Data-parallel replicas over tokens: sum the per-expert counts of every replica (one
    E-element all-reduce, the layer's only cross-replica exchange), so the +-gamma step
    that follows sees the global load and every replica keeps the same bias.  Returns the
    number of replicas.  Works on any torch.distributed backend (NCCL on GPUs, gloo on CPU)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return 1
    world = dist.get_world_size(group)
    if world > 1:
        dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    return world


# ----------------------------------------------------------------------------------------
# The whole layer: buffers allocated once, then the five calls in order.
# ----------------------------------------------------------------------------------------

@dataclass
class LayerWeights:
    w_router: torch.Tensor               # [E, D] fp32
    bias: torch.Tensor                   # [E] fp32 (updated in place by the bias step)
    w_gate: torch.Tensor                 # [E, F, D]
    w_up: torch.Tensor                   # [E, F, D]
    w_down: torch.Tensor                 # [E, D, F]
    shared: tuple | None = None          # (w_gate[1,Fs,D], w_up[1,Fs,D], w_down[1,D,Fs]) or None


class MoELayer:
    """Top-k MoE FFN layer forward on one GPU, with reusable device buffers."""

    def __init__(self, weights: LayerWeights, N: int, k: int, score_fn="softmax", gamma=1e-3,
                 dtype=torch.bfloat16, capacity_factor=None, gather=None, fuse_shared=True,
                 router_shared=False):
        """gather (bf16): the first expert GEMM reads its rows from xn through perm_token
        instead of from a permuted copy, which is then never written; False writes x_perm in
        the permute and runs the GEMM on it.  None chooses by size: gathering costs the GEMM
        roughly a tenth of its first half, the copy moves (1 + k) N D bf16 values, so it
        gathers when d_ff * k / (k + 1) <= 1024 (measured: faster on the handbook and skewed
        layers, slower on the Mixtral- and DeepSeek-V3-shaped ones).
        router_shared (bf16, shared expert with the routed d_ff): the shared expert's first
        GEMM runs in the router's launch over the same token tiles and its second in the
        routed GEMM2 launch (moe_router_topk_split_shared, moe_grouped_swiglu_shared_h); the
        same outputs, bit for bit, as the default, where both of its GEMMs ride in the routed
        launches."""
        w = weights
        self.w, self.k, self.score_fn, self.gamma = w, k, score_fn, gamma
        E = w.w_router.shape[0]
        self.capacity = None if capacity_factor is None else expert_capacity(capacity_factor, N, k, E)
        self.N = N
        self.E, self.D = w.w_router.shape
        self.F = w.w_gate.shape[1]
        dev = w.w_router.device
        R = N * k
        e = lambda *s, dt=torch.int32: torch.empty(*s, dtype=dt, device=dev)
        self.logits = e(N, self.E, dt=torch.float32)
        self.idx = e(N, k)
        self.gate = e(N, k, dt=torch.float32)
        self.near_tie = e(N, dt=torch.uint8)
        self.counts = e(self.E)
        self.offsets = e(self.E + 1)
        self.row_map = e(N, k)
        self.perm_token = e(R)
        if gather is None:
            gather = w.w_gate.shape[1] * k / (k + 1) <= 1024
        self.gather = bool(gather) and dtype == torch.bfloat16
        self.x_perm = None if self.gather else e(R, self.D, dt=dtype)
        self.h_ws = e(R, self.F, dt=dtype)
        self.y_perm = e(R, self.D, dt=dtype)
        self.out = e(N, self.D, dt=dtype)
        self.workspace = e(max(1, permute_workspace_bytes(N, k, self.E)), dt=torch.uint8)
        self.mom = e(1, dt=torch.float32)
        self.tc_router = dtype == torch.bfloat16
        self.w_split = e(3, self.E, self.D, dt=torch.bfloat16) if self.tc_router else None
        self.router_ws = e(max(1, router_split_workspace_bytes(N, self.D, self.E)), dt=torch.uint8) \
            if self.tc_router else None
        if w.shared is not None:
            Fs = w.shared[0].shape[1]
            self.sh_offsets = torch.tensor([0, N], dtype=torch.int32, device=dev)
            self.sh_h = e(N, Fs, dt=dtype)
            self.sh_y = e(N, self.D, dt=dtype)
        else:
            self.sh_y = None
        # the shared expert's tiles ride in the routed experts' launches (same d_ff, bf16)
        self.fuse_shared = bool(fuse_shared) and w.shared is not None and dtype == torch.bfloat16 \
            and w.shared[0].shape[1] == self.F
        self.router_shared = bool(router_shared) and self.fuse_shared and self.tc_router
        if router_shared and not self.router_shared:
            raise ValueError("router_shared needs bf16, a shared expert with the routed d_ff and fuse_shared")

    def forward(self, xn, h, update_bias=True, stream=None, out=None):
        """out = h + shared(xn) + sum_j gate_j Expert_j(xn), and the +-gamma bias step on
        this forward's counts (made by the permute's own launches; the bias only affects the
        next forward's routing).  Writes self.out, or `out` ([N, D], layer dtype) when given,
        and returns it."""
        self.route(xn, stream)
        self.permute(xn, stream, update_bias=update_bias)
        self.experts(xn, stream)
        self.shared_expert(xn, stream)
        return self.combine(h, stream, out)

    def capture(self, xn, h, update_bias=True, out=None):
        """Record one forward on the fixed buffers xn and h (writing self.out, or `out`) as a
        CUDA graph and return a function that replays it on the current stream (refill xn / h
        in place between replays).  Every launch of the layer goes through the C ABI on the
        capture stream; none allocates or waits on the host, so the graph holds exactly the
        kernels of an eager forward.  Replays leave out the host's launch work and most of
        the device's gaps between dependent launches: about 1.5 % of a forward at N=8192,
        D=2048, E=64, F=1024, and most of it for small batches."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        # one forward outside the capture (no bias step): the library's one-time set-up per
        # device happens here, not inside the graph
        self.forward(xn, h, update_bias=False, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.forward(xn, h, update_bias=update_bias, stream=s, out=out)
        torch.cuda.current_stream().wait_stream(s)
        return g.replay

    def permute(self, xn, stream=None, update_bias=False):
        """Histogram, scan, stable permutation (and the row copy unless gathering); with
        update_bias, the +-gamma step on these counts in the same launches.  Data-parallel
        replicas leave update_bias off and call bias_step after summing the counts."""
        moe_permute(xn, self.idx, self.E, self.counts, self.offsets, self.row_map,
                    self.perm_token, self.x_perm, self.workspace, copy=not self.gather,
                    capacity=self.capacity, stream=stream,
                    bias_step=(self.gamma, self.w.bias, self.mom) if update_bias else None)

    def experts(self, xn, stream=None):
        """Every routed expert's SwiGLU FFN over its block of permuted rows -> y_perm (and the
        shared expert's -> sh_y, in the same launches, when fused)."""
        w = self.w
        if self.router_shared:  # sh_h came from the router's launch
            moe_grouped_swiglu_shared_h(self.x_perm, self.offsets, w.w_gate, w.w_up, w.w_down, xn, w.shared[2],
                                        self.sh_h, self.y_perm, self.h_ws, self.sh_y, stream=stream,
                                        perm_token=self.perm_token if self.gather else None)
        elif self.fuse_shared:
            moe_grouped_swiglu_shared(self.x_perm, self.offsets, w.w_gate, w.w_up, w.w_down, xn, w.shared,
                                      self.h_ws, self.y_perm, self.sh_h, self.sh_y, stream=stream,
                                      perm_token=self.perm_token if self.gather else None)
        elif self.gather:
            moe_grouped_swiglu_gather(xn, self.perm_token, self.offsets, w.w_gate, w.w_up,
                                      w.w_down, self.h_ws, self.y_perm, stream=stream)
        else:
            moe_grouped_swiglu(self.x_perm, self.offsets, w.w_gate, w.w_up, w.w_down, self.h_ws,
                               self.y_perm, stream=stream)

    def shared_expert(self, xn, stream=None):
        w = self.w
        if w.shared is not None and not self.fuse_shared:
            moe_grouped_swiglu(xn, self.sh_offsets, w.shared[0], w.shared[1], w.shared[2],
                               self.sh_h, self.sh_y, stream=stream)

    def combine(self, h, stream=None, out=None):
        out = self.out if out is None else out
        return moe_unpermute_combine(self.y_perm, self.row_map, self.gate, self.sh_y, h, out,
                                     stream=stream)

    def bias_step(self, replicas=1, stream=None):
        """+-gamma step on this step's counts (summed over `replicas` data-parallel copies)."""
        moe_bias_update(self.counts, self.w.bias, self.N * self.k * replicas, self.gamma,
                        self.mom, stream=stream)

    def route(self, xn, stream=None):
        """Router + top-k.  bf16 activations: the fp32 router weight is re-split into bf16
        planes (every call, so weight updates are always seen) and run on tensor cores."""
        w = self.w
        if self.router_shared:  # and the shared expert's first GEMM, over the same token tiles
            moe_router_split(w.w_router, self.w_split, stream=stream)
            moe_router_topk_split_shared(xn, self.w_split, w.bias, self.k, w.shared, self.score_fn, self.logits,
                                         self.idx, self.gate, self.near_tie, workspace=self.router_ws,
                                         hs_out=self.sh_h, stream=stream)
        elif self.tc_router:
            moe_router_split(w.w_router, self.w_split, stream=stream)
            moe_router_topk_split(xn, self.w_split, w.bias, self.k, self.score_fn, self.logits,
                                  self.idx, self.gate, self.near_tie, workspace=self.router_ws,
                                  stream=stream)
        else:
            moe_router_topk(xn, w.w_router, w.bias, self.k, self.score_fn, self.logits, self.idx,
                            self.gate, self.near_tie, stream=stream)

    def kernels_per_forward(self, fused_bias=True):
        """Kernel launches of one forward (+ bias step, fused into the permute or not)."""
        router = 3 if self.tc_router else 1
        permute = 3 + (0 if self.gather else 1)  # histogram, scan (+ bias step), rank (+ row copy)
        bias = 0 if fused_bias else 1
        shared = 2 if (self.w.shared is not None and not self.fuse_shared) else 0
        return router + permute + 2 + shared + 1 + bias
