"""Multi-rank host logic on CPU with the gloo backend (world size 2):
sharding whole groups, the global loss / KL mean combination and gradient
scale (checked against the float64 oracle on the unsharded batch), and the
benchmark's timing reduction."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from grpo_loss_gb300 import dist as D


def test_group_shard_covers_every_sequence_once_in_whole_groups():
    for B, G, W in [(32, 8, 2), (8, 4, 3), (12, 2, 4), (4, 4, 2), (30, 3, 4)]:
        seen = []
        for r in range(W):
            s0, n = D.group_shard(B, G, W, r)
            assert s0 % G == 0 and n % G == 0
            seen += list(range(s0, s0 + n))
        assert seen == list(range(B))
    with pytest.raises(ValueError):
        D.group_shard(10, 4, 2, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import grpo_oracle as O
        g = torch.Generator().manual_seed(5)
        B, T, G, d, V, beta = 8, 6, 2, 12, 40, 0.04
        N = B * T
        Hp = torch.randn(N, d, generator=g, dtype=torch.float64)
        Hr = Hp + 0.3 * torch.randn(N, d, generator=g, dtype=torch.float64)
        W = 0.4 * torch.randn(V, d, generator=g, dtype=torch.float64)
        ids = torch.randint(0, V, (N,), generator=g)
        mask = torch.ones(B, T, dtype=torch.uint8)
        mask[1, 3:] = 0
        mask[6, :] = 0
        mask = mask.reshape(-1)
        r = torch.randn(B, generator=g, dtype=torch.float64)
        A = O.advantages(r, G, 1e-4, 1)

        s0, nb = D.group_shard(B, G, world, rank)
        rows = slice(s0 * T, (s0 + nb) * T)
        A_loc = O.advantages(r[s0:s0 + nb], G, 1e-4, 1)
        f = O.forward(Hp[rows], Hr[rows], W, ids[rows], mask[rows], A_loc, nb, T, beta)
        valid = int(mask[rows].sum())
        loss, kl = D.global_loss(f["loss"], f["kl_mean"], nb, valid, B)
        gs = D.grad_scale(nb, B)
        b_loc = O.backward(Hp[rows], Hr[rows], W, ids[rows], mask[rows], A_loc, nb, T, beta,
                           grad_loss=gs)
        ms, tok = D.reduce_timing(10.0 + rank, 100.0 * (rank + 1))
        if rank == 0:
            full = O.forward(Hp, Hr, W, ids, mask, A, B, T, beta)
            b_full = O.backward(Hp, Hr, W, ids, mask, A, B, T, beta)
            results["loss"] = (loss, full["loss"])
            results["kl"] = (kl, full["kl_mean"])
            results["dH0"] = float(np.max(np.abs(b_loc["dH"] - b_full["dH"][rows])))
            results["timing"] = (ms, tok)
        else:
            results["dH1"] = float(np.max(np.abs(b_loc["dH"] - b_full_rows(Hp, Hr, W, ids, mask, A,
                                                                         B, T, beta, rows))))
    finally:
        dist.destroy_process_group()


def b_full_rows(Hp, Hr, W, ids, mask, A, B, T, beta, rows):
    from oracle import grpo_oracle as O
    return O.backward(Hp, Hr, W, ids, mask, A, B, T, beta)["dH"][rows]


def test_sharded_loss_and_gradients_equal_the_unsharded_batch():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_worker, args=(2, _free_port(), results), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(results)
    lo, lf = res["loss"]
    ko, kf = res["kl"]
    assert abs(lo - lf) <= 1e-12 * max(1.0, abs(lf))
    assert abs(ko - kf) <= 1e-12 * max(1.0, abs(kf))
    assert res["dH0"] < 1e-15 and res["dH1"] < 1e-15
    assert res["timing"] == (11.0, 300.0)
