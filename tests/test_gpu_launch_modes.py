"""Plain launches (MOE_PDL=0) and programmatic dependent launches (the default) run the same
kernels on the same data: every output of a layer step is bit-identical.  The mode is fixed
per process, so each runs in a child process."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

STEP = r"""
import sys, torch
sys.path.insert(0, sys.argv[2])
from mixture_experts_layer_scores_b300 import synth
from tests import parity as P
cfg = synth.scaled(synth.CONFIGS["deepseek_v3"], N=333, D=512, E=32, F=256, k=8, F_shared=512)
torch.save(P.gpu_layer(cfg, P.make_inputs(cfg, "cuda")), sys.argv[1])
"""


def test_plain_and_programmatic_launches_agree(tmp_path):
    got = {}
    for pdl in ("1", "0"):
        path = tmp_path / f"step_pdl{pdl}.pt"
        subprocess.run([sys.executable, "-c", STEP, str(path), ROOT], env=dict(os.environ, MOE_PDL=pdl),
                       check=True, timeout=600)
        got[pdl] = torch.load(path)
    assert got["1"].keys() == got["0"].keys()
    for key, a in got["1"].items():
        b = got["0"][key]
        if isinstance(a, torch.Tensor):
            assert torch.equal(a, b), key
        else:
            assert a == b, key
