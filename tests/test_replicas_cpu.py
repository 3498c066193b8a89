"""The benchmark's multi-process path on CPU: two gloo ranks (one per GPU on a real
run, "replicas only": no collective on the data path).  Checks the rendezvous, the
barrier and the max-over-ranks reduction of the step time, and that only rank 0
runs the CPU reference arm."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    # Each rank "measured" a different step time; every rank must report the slowest.
    t = bench.max_over_ranks(1.5 + rank, w)
    bench.barrier(w)
    out[rank] = t
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)  # no-op


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 2, 3

    assert bench.run_reference(Args()) == 0  # returns without building or timing anything


@pytest.mark.parametrize("name,kernels", [("bf16_tc_up_n1500_m4096_k1024", 2),
                                          ("q4_0_gemv_n1_m14336_k4096", 1),
                                          ("moe_q4_0_E64_m1408_k2048_t16x6", 1)])
def test_kernels_per_call(name, kernels):
    w = {x["name"]: x for x in bench.make_workloads()}[name]
    assert bench.kernels_per_call(w) == kernels
