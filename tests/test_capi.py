"""The C-ABI library builds for sm_103a, loads without a GPU and exports every symbol the
header declares; host-side argument checks reject bad calls before any launch."""
import ctypes
import os
import re

import pytest
import torch

from mixture_experts_layer_scores_b300 import build, moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return moe.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("moe_router_topk", "moe_permute", "moe_grouped_swiglu", "moe_unpermute_combine",
               "moe_bias_update"):
        assert fn in names


def test_every_declared_symbol_exported(lib):
    raw = ctypes.CDLL(moe.lib_path())
    for name in declared_functions():
        assert hasattr(raw, name), name
    assert set(moe.EXPORTS) <= set(declared_functions())


def test_status_strings(lib):
    for code, name in moe.STATUS.items():
        assert lib.moe_status_string(code).decode() == name
    assert lib.moe_version() >= 100


def test_workspace_size(lib):
    assert lib.moe_permute_workspace_bytes(0, 8, 64) == 0
    b = lib.moe_permute_workspace_bytes(8192, 8, 64)
    assert b > 0 and b % 4 == 0 and b <= 128 * 64 * 4


def test_new_entry_points_reject_bad_arguments_before_launch(lib):
    """Only NULL pointers: each call must return its error before touching any pointer."""
    raw = ctypes.CDLL(moe.lib_path())
    f = raw.moe_permute_update_bias
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    # no bias to update
    assert f(None, 1, 16, 64, None, 2, 8, 16, None, None, None, None, None, None, 0, 1e-3, None, None, None) == -1
    g = raw.moe_grouped_swiglu_shared
    g.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int] + [ctypes.c_void_p] * 5 + [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 6
    g.restype = ctypes.c_int
    assert g(None, None, None, 0, 0, 128, 128, None, None, None, None, None, None, 0, None, None, None, None, None,
             None) == -1                                            # G < 1
    assert g(None, None, None, 4, 0, 100, 128, None, None, None, None, None, None, 0, None, None, None, None, None,
             None) == -2                                            # D not a multiple of 64
    assert g(None, None, None, 4, 64, 128, 128, None, None, None, None, None, None, 0, None, None, None, None, None,
             None) == -1                                            # routed rows but no operands
    assert g(None, None, None, 4, 0, 128, 128, None, None, None, None, None, None, 8, None, None, None, None, None,
             None) == -1                                            # shared rows but no operands
    r = raw.moe_router_topk_split_shared
    r.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5 + [ctypes.c_size_t, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    r.restype = ctypes.c_int
    assert r(None, 16, 64, None, None, 8, 2, 0, None, None, None, None, None, 0, None, None, 64, None,
             None) == -1                                            # no shared gate weights
    h = raw.moe_grouped_swiglu_shared_h
    h.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int] + [ctypes.c_void_p] * 5 + [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 4
    h.restype = ctypes.c_int
    assert h(None, None, None, 0, 0, 128, 128, None, None, None, None, None, None, 0, None, None, None,
             None) == -1                                            # G < 1
    assert h(None, None, None, 4, 0, 128, 128, None, None, None, None, None, None, 8, None, None, None,
             None) == -1                                            # shared rows, no H or weights


def test_expert_capacity_through_the_abi(lib):
    """ceil(C N k / E), capped at N k; -1 for arguments outside the domain."""
    raw = ctypes.CDLL(moe.lib_path())
    raw.moe_expert_capacity.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    raw.moe_expert_capacity.restype = ctypes.c_int64
    cap = raw.moe_expert_capacity
    assert cap(1.0, 8, 2, 4) == 4            # exactly the uniform share
    assert cap(1.25, 10, 2, 4) == 7          # 6.25 rounds up
    assert cap(0.5, 16384, 8, 64) == 1024
    assert cap(0.0, 100, 2, 8) == 0
    assert cap(100.0, 10, 2, 4) == 20        # capped at N k
    assert cap(1.0, 0, 2, 4) == 0
    assert cap(-1.0, 8, 2, 4) == -1 and cap(float("nan"), 8, 2, 4) == -1
    assert cap(1.0, -1, 2, 4) == -1 and cap(1.0, 8, 0, 4) == -1 and cap(1.0, 8, 2, 0) == -1


@pytest.mark.skipif(torch.cuda.is_available(),
                    reason="passes placeholder device addresses: a host-only check, never run beside a GPU")
def test_host_validation_rejects_before_launch(lib):
    vp = ctypes.c_void_p
    # k > E, E too large, D not a multiple of 64, null outputs: no launch happens
    assert lib.moe_router_topk(vp(16), 1, 4, 64, vp(16), None, 4, 5, 0, None, vp(16), vp(16), None, None) == -1
    assert lib.moe_router_topk(vp(16), 1, 4, 64, vp(16), None, 300, 5, 0, None, vp(16), vp(16), None, None) == -2
    assert lib.moe_router_topk(vp(16), 1, 4, 48, vp(16), None, 8, 2, 0, None, vp(16), vp(16), None, None) == -2
    assert lib.moe_router_topk(vp(16), 1, 4, 64, vp(16), None, 8, 2, 0, None, None, vp(16), None, None) == -1
    assert lib.moe_router_topk(vp(16), 1, 4, 64, vp(16), None, 8, 2, 7, None, vp(16), vp(16), None, None) == -1
    # unaligned activation pointer
    assert lib.moe_router_topk(vp(18), 1, 4, 64, vp(16), None, 8, 2, 0, None, vp(16), vp(16), None, None) == -1
    # permute: workspace too small, row_map without perm_token
    assert lib.moe_permute(vp(16), 1, 64, 64, vp(16), 2, 8, vp(16), vp(16), vp(16), vp(16), vp(16),
                           vp(16), 4, None) == -1
    assert lib.moe_permute(vp(16), 1, 64, 64, vp(16), 2, 8, vp(16), vp(16), vp(16), None, None,
                           vp(16), 1 << 20, None) == -1
    # grouped GEMM: F not a multiple of 64; M_total == 0 is a no-op
    assert lib.moe_grouped_swiglu(vp(16), 1, vp(16), 4, 100, 128, 96, vp(16), vp(16), vp(16), vp(16),
                                  vp(16), None) == -2
    assert lib.moe_grouped_swiglu(None, 1, None, 4, 0, 128, 128, None, None, None, None, None, None) == 0
    # gathered GEMM: same shape rules; null perm_token; M_total == 0 is a no-op
    assert lib.moe_grouped_swiglu_gather(vp(16), 50, vp(16), vp(16), 4, 100, 128, 96, vp(16), vp(16),
                                         vp(16), vp(16), vp(16), None) == -2
    assert lib.moe_grouped_swiglu_gather(vp(16), 50, None, vp(16), 4, 100, 128, 128, vp(16), vp(16),
                                         vp(16), vp(16), vp(16), None) == -1
    assert lib.moe_grouped_swiglu_gather(vp(24), 50, vp(16), vp(16), 4, 100, 128, 128, vp(16), vp(16),
                                         vp(16), vp(16), vp(16), None) == -1
    assert lib.moe_grouped_swiglu_gather(vp(16), 0, vp(16), vp(16), 4, 100, 128, 128, vp(16), vp(16),
                                         vp(16), vp(16), vp(16), None) == -1
    assert lib.moe_grouped_swiglu_gather(None, 0, None, None, 4, 0, 128, 128, None, None, None, None,
                                         None, None) == 0
    # capped GEMM: negative cap; the cap changes nothing about the shape rules or the no-op
    assert lib.moe_grouped_swiglu_ex(vp(16), 1, vp(16), 4, 100, 128, 128, vp(16), vp(16), vp(16), vp(16),
                                     vp(16), -1, None) == -1
    assert lib.moe_grouped_swiglu_ex(vp(16), 1, vp(16), 4, 100, 128, 96, vp(16), vp(16), vp(16), vp(16),
                                     vp(16), 8, None) == -2
    assert lib.moe_grouped_swiglu_ex(None, 1, None, 4, 0, 128, 128, None, None, None, None, None, 8,
                                     None) == 0
    # combine: k too large; bias: null counts
    assert lib.moe_unpermute_combine(vp(16), vp(16), vp(16), 4, 17, 64, None, None, vp(16), 1, None) == -2
    assert lib.moe_bias_update(None, 8, 64, ctypes.c_float(1e-3), vp(16), None, None) == -1
    # bounded-wait self-test: null source, limit outside [1000, normal limit]
    assert lib.moe_selftest_bounded_wait(None, 2_000_000, vp(16), None) == -1
    assert lib.moe_selftest_bounded_wait(vp(16), 10, vp(16), None) == -1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(moe, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        moe.load()
