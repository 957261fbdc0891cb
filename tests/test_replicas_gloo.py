"""Data-parallel replicas on CPU (gloo, world size 2): routing is per token, and the bias step
after the counts all-reduce equals the single-batch bias step bit for bit."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixture_experts_layer_scores_b300 import moe, synth
from oracle import moe_oracle


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg = synth.scaled(synth.CONFIGS["skewed"], N=256, D=128, E=16, F=64, k=4)
    x, _ = synth.make_tokens(cfg)
    w, b = synth.make_router(cfg)
    shard = x[rank * cfg.N // world:(rank + 1) * cfg.N // world]
    bias = synth.gaussian(9, "bias", (cfg.E,), 0.05).numpy()
    r = moe_oracle.route(shard.double().numpy(), w.numpy(), bias, cfg.k)
    counts = torch.tensor(moe_oracle.expert_counts(r["idx"], cfg.E), dtype=torch.int32)
    n_rep = moe.global_counts(counts)
    new_b, mom = moe_oracle.bias_update(bias, counts.numpy(), shard.shape[0] * cfg.k * n_rep, cfg.gamma)
    out[rank] = (r["idx"], new_b, mom, n_rep)
    dist.destroy_process_group()


def test_two_replicas_match_one_batch():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    cfg = synth.scaled(synth.CONFIGS["skewed"], N=256, D=128, E=16, F=64, k=4)
    x, _ = synth.make_tokens(cfg)
    w, _ = synth.make_router(cfg)
    bias = synth.gaussian(9, "bias", (cfg.E,), 0.05).numpy()
    r = moe_oracle.route(x.double().numpy(), w.numpy(), bias, cfg.k)
    full_b, full_mom = moe_oracle.bias_update(bias, moe_oracle.expert_counts(r["idx"], cfg.E),
                                              cfg.N * cfg.k, cfg.gamma)
    assert res[0][3] == world and res[1][3] == world
    assert np.array_equal(np.concatenate([res[0][0], res[1][0]]), r["idx"])
    for rank in range(world):
        assert np.array_equal(res[rank][1], full_b)      # identical biases on every replica
        assert res[rank][2] == full_mom


def test_single_process_counts_untouched():
    c = torch.arange(8, dtype=torch.int32)
    assert moe.global_counts(c) == 1 and torch.equal(c, torch.arange(8, dtype=torch.int32))
