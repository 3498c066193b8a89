"""The benchmark's multi-process path on CPU: two gloo ranks (one per GPU on a real
run, "replicas only": no collective on the data path).  Checks the rendezvous, the
barrier and the max-over-ranks reduction of the step time, and that only rank 0
runs the CPU reference arm."""
import functools
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


@functools.lru_cache(maxsize=1)
def _extras():
    return {x["name"]: x for x in bench.extra_workloads()}


def _extra(name):
    return _extras()[name]


def test_algorithmic_bytes_of_the_dual_output_band():
    """The second band adds n x dual f32 outputs and dual bias values, and no flops."""
    plain = _extra("plain_bf16_tc_q_n1500_m1024_k1024")
    dual = _extra("dual_bf16_tc_q_n1500_m1024_k1024")
    bp, fp = bench.algorithmic(plain)
    bd, fd = bench.algorithmic(dual)
    assert fd == fp == 2.0 * 1500 * 1024 * 1024
    assert bd - bp == 1500 * 1024 * 4 + 1024 * 4
    assert bench.kernels_per_call(dual) == 2


@pytest.mark.parametrize("tag,wbytes", [("bf16", 2), ("f16", 2), ("f32", 4)])
def test_algorithmic_bytes_of_the_float_gemvs(tag, wbytes):
    w = _extra(f"{tag}_gemv_n1_m4096_k4096")
    b, f = bench.algorithmic(w)
    # weights once, X, Y, bias
    assert b == 4096 * 4096 * wbytes + 4096 * 4 + 4096 * 4 + 4096 * 4
    assert f == 2.0 * 4096 * 4096
    assert bench.kernels_per_call(w) == 1


def test_traffic_record_is_dropped_when_its_source_changes(monkeypatch):
    import hashlib
    srcs = ["gemv_transformer_gb300/csrc/gemv_mma.cu", "gemv_transformer_gb300/csrc/tile_sched.cuh"]
    h = hashlib.sha256()
    for src in srcs:
        with open(os.path.join(bench.ROOT, src), "rb") as f:
            h.update(f.read())
    name = "a_workload"
    monkeypatch.setitem(bench.TRAFFIC, name, {"bytes": 123, "sources": srcs, "sha256": h.hexdigest()})
    assert bench.traffic_for(name) == 123  # recorded on the sources as they stand
    monkeypatch.setitem(bench.TRAFFIC, name, {"bytes": 123, "sources": srcs, "sha256": "0" * 64})
    assert bench.traffic_for(name) is None
    # a record on the first source alone is not one on both
    with open(os.path.join(bench.ROOT, srcs[0]), "rb") as f:
        one = hashlib.sha256(f.read()).hexdigest()
    monkeypatch.setitem(bench.TRAFFIC, name, {"bytes": 123, "sources": srcs, "sha256": one})
    assert bench.traffic_for(name) is None
    assert bench.traffic_for("no_such_workload") is None
