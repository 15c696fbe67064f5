"""Batch sharding across ranks, on CPU with the gloo backend (world size 2).

Forward and backward data are independent per image, so ranks that each hold a slice of the
batch need no exchange; the filter gradient is a sum over the batch, so ranks that each hold
a slice need exactly one all-reduce (sum) of their partial dW.  These tests check both
statements with the fp64 oracle, run as two processes that rendezvous on 127.0.0.1."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from depthwise_convolution_nhwc_gb300.inputs import Case

WORLD = 2
CASE = Case(6, 9, 11, 8, 5, 5, 1, 2, "f32", "normal", 31)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        x, w, dy = (t.double().numpy() for t in (CASE.x(), CASE.w(), CASE.dy()))
        per = CASE.N // WORLD
        sl = slice(rank * per, (rank + 1) * per)
        y = oracle.fwd(x[sl], w, CASE.stride, CASE.pad)
        dx = oracle.bwd_data(dy[sl], w, (CASE.H, CASE.W), CASE.stride, CASE.pad)
        dw = torch.from_numpy(oracle.bwd_filter(x[sl], dy[sl], (CASE.FH, CASE.FW), CASE.stride,
                                                CASE.pad))
        dist.all_reduce(dw, op=dist.ReduceOp.SUM)
        np.save(os.path.join(out_dir, f"y{rank}.npy"), y)
        np.save(os.path.join(out_dir, f"dx{rank}.npy"), dx)
        np.save(os.path.join(out_dir, f"dw{rank}.npy"), dw.numpy())
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def sharded(tmp_path_factory):
    out = tmp_path_factory.mktemp("ranks")
    mp.start_processes(_rank_main, args=(_free_port(), str(out)), nprocs=WORLD, join=True,
                       start_method="spawn")
    return {k: [np.load(out / f"{k}{r}.npy") for r in range(WORLD)] for k in ("y", "dx", "dw")}


def test_forward_and_data_gradient_shard_without_exchange(sharded):
    x, w, dy = (t.double().numpy() for t in (CASE.x(), CASE.w(), CASE.dy()))
    y = oracle.fwd(x, w, CASE.stride, CASE.pad)
    dx = oracle.bwd_data(dy, w, (CASE.H, CASE.W), CASE.stride, CASE.pad)
    assert np.array_equal(np.concatenate(sharded["y"]), y)
    assert np.array_equal(np.concatenate(sharded["dx"]), dx)


def test_filter_gradient_needs_one_all_reduce(sharded):
    x, dy = (t.double().numpy() for t in (CASE.x(), CASE.dy()))
    dw = oracle.bwd_filter(x, dy, (CASE.FH, CASE.FW), CASE.stride, CASE.pad)
    for r in range(WORLD):
        np.testing.assert_allclose(sharded["dw"][r], dw, rtol=1e-12, atol=1e-12)
    # a single shard alone is not the gradient: the exchange is required
    x0, dy0 = x[: CASE.N // WORLD], dy[: CASE.N // WORLD]
    part = oracle.bwd_filter(x0, dy0, (CASE.FH, CASE.FW), CASE.stride, CASE.pad)
    assert not np.allclose(part, dw)
