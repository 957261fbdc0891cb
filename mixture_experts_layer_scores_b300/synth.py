"""Seeded synthetic inputs for the MoE layer, bit-identical on any device.

This module only draws numbers; it holds none of the layer's arithmetic.  Both
the CUDA path and the CPU oracle receive arrays made here, so the two sides see
the same bits.

Generator.  Every tensor is a named *stream*.  Element ``i`` of a stream is a
pure function of ``(seed, stream, i)``:

* ``key = splitmix64(seed * 2**20 + stream_id)`` (Python integers);
* two 64-bit words ``w_j = splitmix64_mix(key + (2i + j + 1) * GOLDEN)``,
  ``j = 0, 1`` -- Vigna's SplitMix64 output function applied to a Weyl
  counter, evaluated with wrapping int64 arithmetic;
* the eight 16-bit lanes of the two words are summed (Irwin-Hall with n = 8),
  centred and scaled to unit variance: ``z = (S - 8 * 32767.5) / sd`` with
  ``sd = sqrt(8 * (65536**2 - 1) / 12)``.  ``z`` is an approximately standard
  normal deviate bounded by +-4.9;
* ``value = fl32(float32(S - 262140) * float32(std / sd))``, then rounded to
  nearest-even bf16 when a bf16 tensor is asked for.

Every step is integer arithmetic or one IEEE fp32 multiply, so the CPU and the
GPU produce identical bits, and any slice of a tensor can be regenerated on its
own (the oracle uses that to rebuild only the experts a sampled token visits).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SRC = os.path.join(_HERE, "synth_host.c")
_HOST_LIB = os.path.join(_HERE, "libsynth_host.so")
_host = None


def build_host_lib(force: bool = False) -> str:
    """Compile the OpenMP host generator (plain C) next to this file."""
    if force or not os.path.exists(_HOST_LIB) or \
            os.path.getmtime(_HOST_LIB) < os.path.getmtime(_HOST_SRC):
        tmp = _HOST_LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-ffp-contract=off", "-fPIC",
                               "-shared", _HOST_SRC, "-o", tmp])
        os.replace(tmp, _HOST_LIB)
    return _HOST_LIB


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host_lib())
        i64, u64, f32, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p
        lib.synth_fill_f32.argtypes = [u64, i64, i64, f32, vp]
        lib.synth_gather_f32.argtypes = [u64, vp, i64, f32, vp]
        _host = lib
    return _host

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB
_IH_N = 8
_IH_MEAN2 = _IH_N * 65535  # twice the mean of the lane sum, kept integral
_IH_SD = math.sqrt(_IH_N * (65536.0 ** 2 - 1.0) / 12.0)

# Stream ids: one per named tensor.  New names must take new ids.
STREAMS = {
    "xn": 1,
    "h": 2,
    "w_router": 3,
    "w_gate": 4,
    "w_up": 5,
    "w_down": 6,
    "ws_gate": 7,
    "ws_up": 8,
    "ws_down": 9,
    "bias": 10,
    "zipf_rank": 11,
    "misc": 12,
}


def _signed(v: int) -> int:
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def splitmix64_py(x: int) -> int:
    """SplitMix64 output function on a 64-bit word (pure Python reference)."""
    z = x & MASK64
    z = ((z ^ (z >> 30)) * _C1) & MASK64
    z = ((z ^ (z >> 27)) * _C2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: str | int) -> int:
    sid = STREAMS[stream] if isinstance(stream, str) else int(stream)
    return splitmix64_py((int(seed) << 20) + sid)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    # logical right shift of int64 lanes
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _signed(_C1)
    z = (z ^ _lsr(z, 27)) * _signed(_C2)
    return z ^ _lsr(z, 31)


def words(key: int, counters: torch.Tensor) -> torch.Tensor:
    """64-bit words for int64 ``counters`` (as int64 bit patterns)."""
    z = (counters + 1) * _signed(GOLDEN) + _signed(key)
    return _mix64(z)


def _lane_sum(w: torch.Tensor) -> torch.Tensor:
    return (w & 0xFFFF) + ((w >> 16) & 0xFFFF) + ((w >> 32) & 0xFFFF) + ((w >> 48) & 0xFFFF)


def _scale(std: float) -> float:
    return float(np.float32(std / (2.0 * _IH_SD)))


def gaussian_at(seed: int, stream: str, flat_index: torch.Tensor, std: float,
                dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """Values of stream elements at int64 ``flat_index`` (same device)."""
    key = stream_key(seed, stream)
    if flat_index.device.type == "cpu":
        fi = flat_index.contiguous()
        out = torch.empty(fi.shape, dtype=torch.float32)
        _host_lib().synth_gather_f32(key, fi.data_ptr(), fi.numel(), _scale(std), out.data_ptr())
        return out if dtype == torch.float32 else out.to(dtype)
    return gaussian_torch_at(key, flat_index, std, dtype)


def gaussian_torch_at(key: int, flat_index: torch.Tensor, std: float,
                      dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """The generator in torch integer ops (any device)."""
    c = 2 * flat_index
    s2 = 2 * (_lane_sum(words(key, c)) + _lane_sum(words(key, c + 1))) - _IH_MEAN2
    # s2 = 2*(S - mean) is an even integer with |s2| < 2**21: exact in fp32.
    scale = torch.tensor(_scale(std), dtype=torch.float32, device=flat_index.device)
    v = s2.to(torch.float32) * scale
    return v if dtype == torch.float32 else v.to(dtype)


def gaussian(seed: int, stream: str, shape, std: float, dtype=torch.float32,
             device="cpu", offset: int = 0, chunk: int = 1 << 25) -> torch.Tensor:
    """A whole tensor of stream elements ``offset .. offset + numel - 1``."""
    shape = tuple(int(s) for s in shape)
    numel = int(np.prod(shape)) if shape else 1
    if torch.device(device).type == "cpu":
        buf = torch.empty(numel, dtype=torch.float32)
        _host_lib().synth_fill_f32(stream_key(seed, stream), offset, numel, _scale(std),
                                   buf.data_ptr())
        return (buf if dtype == torch.float32 else buf.to(dtype)).view(shape)
    out = torch.empty(numel, dtype=dtype, device=device)
    key = stream_key(seed, stream)
    for lo in range(0, numel, chunk):
        hi = min(numel, lo + chunk)
        idx = torch.arange(offset + lo, offset + hi, dtype=torch.int64, device=device)
        out[lo:hi] = gaussian_torch_at(key, idx, std, dtype)
    return out.view(shape)


def uniform_u64(seed: int, stream: str, n: int) -> np.ndarray:
    """``n`` raw 64-bit words of a stream (CPU, numpy uint64)."""
    key = stream_key(seed, stream)
    w = words(key, torch.arange(n, dtype=torch.int64))
    return w.numpy().view(np.uint64)


# ----------------------------------------------------------------------------------
# Workload recipes.  Shapes and value distributions of the five layer configurations.
# ----------------------------------------------------------------------------------

@dataclass(frozen=True)
class LayerConfig:
    name: str
    N: int
    D: int
    E: int
    F: int
    k: int
    score_fn: str = "softmax"      # "softmax" | "sigmoid"
    shared: int = 0                # number of always-on shared experts (0 or 1)
    F_shared: int = 0
    dtype: str = "bf16"            # activation / expert-weight dtype: "bf16" | "f32"
    x_std: float = 1.0             # std of xn and h
    gamma: float = 1e-3
    zipf_s: float = 0.0            # > 0: router skewed so expert popularity follows Zipf(s)
    zipf_mu: float = 0.5
    seed: int = 1
    k_serve: int = 0               # > 0: a second forward with this smaller k
    bias_steps: int = 1

    @property
    def R(self) -> int:
        return self.N * self.k


def _cfg_tiny():
    return LayerConfig("tiny", N=512, D=256, E=8, F=512, k=2, dtype="f32",
                       x_std=1.0 / math.sqrt(256), seed=1)


CONFIGS = {
    "tiny": _cfg_tiny(),
    "handbook": LayerConfig("handbook", N=8192, D=2048, E=64, F=1024, k=8, seed=2),
    "mixtral": LayerConfig("mixtral", N=4096, D=4096, E=8, F=14336, k=2, seed=3, bias_steps=0),
    "deepseek_v3": LayerConfig("deepseek_v3", N=4096, D=7168, E=256, F=2048, k=8,
                               score_fn="sigmoid", shared=1, F_shared=2048, seed=4),
    "skewed": LayerConfig("skewed", N=16384, D=2048, E=64, F=1024, k=8, zipf_s=1.2,
                          seed=5, k_serve=4, bias_steps=50),
}


def zipf_logit_offsets(cfg: LayerConfig) -> np.ndarray:
    """c_e = ln p_e with p_e = r_e^-s / sum_r r^-s and r_e a seeded permutation of 1..E."""
    w = uniform_u64(cfg.seed, "zipf_rank", cfg.E)
    order = np.argsort(w, kind="stable")
    rank = np.empty(cfg.E, dtype=np.int64)
    rank[order] = np.arange(1, cfg.E + 1)
    p = rank.astype(np.float64) ** (-cfg.zipf_s)
    p /= p.sum()
    return np.log(p)


def _tdt(cfg):
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def make_tokens(cfg: LayerConfig, device="cpu", seed: int | None = None, rows=None):
    """(xn, h) for all tokens, or only for the int64 token ids ``rows``."""
    seed = cfg.seed if seed is None else seed
    dt = _tdt(cfg)
    if rows is None:
        z = gaussian(seed, "xn", (cfg.N, cfg.D), cfg.x_std, torch.float32, device)
        h = gaussian(seed, "h", (cfg.N, cfg.D), cfg.x_std, dt, device)
    else:
        rows = torch.as_tensor(rows, dtype=torch.int64, device=device)
        fi = (rows[:, None] * cfg.D + torch.arange(cfg.D, device=device)[None, :])
        z = gaussian_at(seed, "xn", fi, cfg.x_std, torch.float32)
        h = gaussian_at(seed, "h", fi, cfg.x_std, dt)
    if cfg.zipf_s > 0:
        # every element of xn is shifted by mu (= mu*sqrt(D) along u = 1/sqrt(D))
        z = z + torch.tensor(cfg.zipf_mu, dtype=torch.float32, device=z.device)
    return z.to(dt), h


def make_router(cfg: LayerConfig, device="cpu"):
    """fp32 router weight [E, D] and the initial fp32 bias [E] (zero)."""
    w = gaussian(cfg.seed, "w_router", (cfg.E, cfg.D), 1.0 / math.sqrt(cfg.D),
                 torch.float32, device)
    if cfg.zipf_s > 0:
        c = zipf_logit_offsets(cfg) / (cfg.zipf_mu * cfg.D)
        w = w + torch.tensor(c, dtype=torch.float32, device=device)[:, None]
    b = torch.zeros(cfg.E, dtype=torch.float32, device=device)
    return w, b


def make_expert(cfg: LayerConfig, e: int, device="cpu", shared: bool = False):
    """(w_gate [F,D], w_up [F,D], w_down [D,F]) of routed expert ``e`` or of the shared one."""
    F = cfg.F_shared if shared else cfg.F
    D = cfg.D
    dt = _tdt(cfg)
    names = ("ws_gate", "ws_up", "ws_down") if shared else ("w_gate", "w_up", "w_down")
    off = e * F * D
    wg = gaussian(cfg.seed, names[0], (F, D), 1.0 / math.sqrt(D), dt, device, offset=off)
    wu = gaussian(cfg.seed, names[1], (F, D), 1.0 / math.sqrt(D), dt, device, offset=off)
    wd = gaussian(cfg.seed, names[2], (D, F), 1.0 / math.sqrt(F), dt, device, offset=off)
    return wg, wu, wd


def make_experts(cfg: LayerConfig, device="cpu"):
    """All routed expert weights: w_gate, w_up [E,F,D]; w_down [E,D,F]."""
    E, F, D = cfg.E, cfg.F, cfg.D
    dt = _tdt(cfg)
    wg = gaussian(cfg.seed, "w_gate", (E, F, D), 1.0 / math.sqrt(D), dt, device)
    wu = gaussian(cfg.seed, "w_up", (E, F, D), 1.0 / math.sqrt(D), dt, device)
    wd = gaussian(cfg.seed, "w_down", (E, D, F), 1.0 / math.sqrt(F), dt, device)
    return wg, wu, wd


def make_shared(cfg: LayerConfig, device="cpu"):
    if not cfg.shared:
        return None
    wg, wu, wd = make_expert(cfg, 0, device, shared=True)
    return wg[None], wu[None], wd[None]


def scaled(cfg: LayerConfig, **kw) -> LayerConfig:
    """The same recipe at other sizes (for tests that must finish on the CPU in seconds)."""
    d = dict(cfg.__dict__)
    d.update(kw)
    return LayerConfig(**d)
