"""Multi-GPU replicas, host side, on two gloo ranks (CPU).

Each rank draws the inputs of its own replica, runs the method (here the
fp64 oracle, since this test needs no GPU) with no collective on the data
path, and the ranks agree on the slowest step time and the whole-job
throughput through the same helpers bench.py uses on GPUs (there with nccl).
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import oracle
    from linear_attention_recurrence_delta_gb300 import inputs as I, replicas
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    base = I.custom(name="rep", mode="delta", dtype="bf16", B=1, H=2, T=40, dk=8, dv=8, seed=5,
                    b_dist="l2norm", c_dist="l2norm")
    w = replicas.rank_workload(base, rank, world)
    x = I.make_inputs(w)
    o, hT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode)
    fake_ms = 1.0 + rank          # this rank's step time
    step_ms = replicas.max_over_ranks(fake_ms, dist)
    value = replicas.whole_job_tokens_per_s(w.B * w.T, world, step_ms)
    out[rank] = (w.seed, float(np.abs(o).sum()), step_ms, value, float(x["v"][0, 0, 0, 0]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    r0, r1 = out[0], out[1]
    assert r0[0] != r1[0], "each replica draws inputs of its own"
    assert r0[4] != r1[4]
    assert r0[1] != r1[1], "and so computes outputs of its own"
    assert r0[2] == r1[2] == 2.0, "both ranks see the slowest step time"
    assert r0[3] == r1[3] == pytest.approx(world * 40 / 2.0e-3), "whole-job tokens over the slowest rank's time"


def test_single_process_is_identity():
    from linear_attention_recurrence_delta_gb300 import inputs as I, replicas
    w = I.WORKLOADS["delta_bf16_8x16x4096x64"]
    assert replicas.rank_workload(w, 0, 1) is w
    assert replicas.max_over_ranks(3.5) == 3.5
    assert replicas.whole_job_tokens_per_s(1000, 1, 2.0) == pytest.approx(5e5)
