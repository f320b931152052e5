"""The multi-GPU (replica) benchmark logic with two gloo ranks on CPU: each
rank draws its own batch, the timed interval is the max over ranks, and the
whole-job rate counts every rank's work against that interval."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from exact_attention_online_gb300 import replicas
from exact_attention_online_gb300.inputs import WORKLOADS, make_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = replicas.dist_env()
        w = replicas.rank_workload(WORKLOADS["tiny"], r)
        q, _, _, _ = make_inputs(w)
        elapsed = 100.0 + 50.0 * r            # ms the rank "took"
        t_max = replicas.max_over_ranks(elapsed)
        rate = replicas.whole_job_rate(1e9, 10, ws, t_max)
        out[r] = (ws, r, local, w.seed, float(q.float().sum()), t_max, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    (ws0, r0, l0, s0, q0, t0, rate0), (ws1, r1, l1, s1, q1, t1, rate1) = res[0], res[1]
    assert (ws0, r0, l0, ws1, r1, l1) == (2, 0, 0, 2, 1, 1)
    assert s1 - s0 == replicas.RANK_SEED_STRIDE and q0 != q1   # independent batches
    assert t0 == t1 == 150.0                                    # max over ranks
    assert rate0 == rate1 == pytest.approx(1e9 * 10 * 2 / 0.150)


def test_single_process_is_identity():
    assert replicas.max_over_ranks(3.5) == 3.5
    assert replicas.whole_job_rate(2.0, 3, 1, 1000.0) == pytest.approx(6.0)
    with pytest.raises(ValueError):
        replicas.whole_job_rate(1.0, 1, 1, 0.0)
