"""Data-parallel sketching on two replicas, run as two gloo processes on the CPU.

Each replica sketches its own microbatches (the sketches are formed here by
the oracle), the sketches are summed with the package's all-reduce, and each
replica applies the update: both must end with bit-identical W, with the
summed sketch equal to the single-process sketch up to fp32 summation order.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as orc
from rank_gradient_sketching_philox_gb300 import dataparallel, synth

D_, K_, R_, T_, NMB = 48, 64, 8, 32, 5
SEED, LAYER, STEP, ALPHA_ETA = 0, 3, 1, 1e-2


def _inputs():
    """The same seeded inputs on every replica."""
    W = synth.normal_bf16((D_, K_), 0.02, 1000 + LAYER).view(torch.int16).numpy().view(np.uint16)
    P = orc.sample_rademacher(SEED, LAYER, STEP, K_, R_)
    X = [synth.normal_bf16((T_, K_), 1.0, 10 + m).view(torch.int16).numpy().view(np.uint16) for m in range(NMB)]
    D = [synth.normal_bf16((T_, D_), 1e-1, 50 + m).view(torch.int16).numpy().view(np.uint16) for m in range(NMB)]
    return W, P, X, D


def _sketch(mbs, P, X, D):
    C = np.zeros((D_, R_), np.float32)
    for m in mbs:
        C = orc.accumulate(D[m], orc.project_inputs(X[m], P), C)
    return C


def _replica(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W, P, X, D = _inputs()
        mine = dataparallel.microbatches_of(rank, world, NMB)
        flat, (C,) = dataparallel.flat_sketches([(D_, R_)], "cpu")
        C.copy_(torch.from_numpy(_sketch(mine, P, X, D)))
        dataparallel.allreduce_sketches(flat)
        W_new = orc.update_sgd(W, C.numpy(), P, ALPHA_ETA, SEED, LAYER, STEP)
        np.save(os.path.join(out_dir, "C%d.npy" % rank), C.numpy())
        np.save(os.path.join(out_dir, "W%d.npy" % rank), W_new)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_microbatch_shards_cover_each_once():
    for world in (1, 2, 3, 8):
        seen = sorted(m for r in range(world) for m in dataparallel.microbatches_of(r, world, 13))
        assert seen == list(range(13))
    with pytest.raises(ValueError):
        dataparallel.microbatches_of(2, 2, 4)


def test_flat_sketch_views_share_one_buffer():
    flat, views = dataparallel.flat_sketches([(3, 2), (5, 4)], "cpu")
    views[1][4, 3] = 7.0
    assert flat.numel() == 26 and flat[-1] == 7.0 and views[0].shape == (3, 2)


def test_two_replicas_agree_bit_for_bit(tmp_path):
    orc.lib()  # build the oracle before the replicas start
    mp.spawn(_replica, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    C0, C1 = np.load(tmp_path / "C0.npy"), np.load(tmp_path / "C1.npy")
    W0, W1 = np.load(tmp_path / "W0.npy"), np.load(tmp_path / "W1.npy")
    assert np.array_equal(C0.view(np.uint32), C1.view(np.uint32))
    assert np.array_equal(W0, W1)
    # the summed sketch is the whole batch's sketch up to fp32 summation order
    W, P, X, D = _inputs()
    C_all = _sketch(range(NMB), P, X, D)
    assert np.linalg.norm(C0 - C_all) <= 1e-6 * np.linalg.norm(C_all)
    W_all = orc.update_sgd(W, C_all, P, ALPHA_ETA, SEED, LAYER, STEP)
    assert np.mean(W0 == W_all) >= 0.999
