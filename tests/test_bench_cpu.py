"""Host-side logic of bench.py on CPU: the algorithmic FLOP / byte counts, the
clock summary, and the multi-rank (replica) timing reduction over gloo with
world size 2."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from gated_delta_rule_09_gb300 import inputs as I


def test_workload_numbers_train_shape():
    w = I.WORKLOADS["train_bf16"]
    flops, byts = bench.workload_numbers(w, [w.T] * w.B)
    # 4096 chunk-heads x 2 [3*64*128*128 + 64^2 (3*128 + 2*128)]
    assert flops == 4096 * 2 * (3 * 64 * 128 * 128 + 64 * 64 * (3 * 128 + 2 * 128))
    assert abs(flops / 1e9 - 47.245) < 1e-3
    # q,k,v read + o written (bf16) + 8 B gates per token-head + fp32 final state
    assert byts == 262144 * 512 * 2 + 262144 * 8 + 64 * 128 * 128 * 4
    assert abs(byts / 1e6 - 274.7) < 0.1


def test_workload_numbers_ragged_and_s0():
    w = I.WORKLOADS["varlen_bf16"]
    flops, byts = bench.workload_numbers(w, [65, 1])
    per = lambda n: 2 * (3 * n * 128 * 128 + n * n * (3 * 128 + 2 * 128)) * 32
    assert flops == per(64) + per(1) + per(1)
    state = 2 * 32 * 128 * 128 * 4
    assert byts == 66 * 32 * 512 * 2 + 66 * 32 * 8 + 2 * state  # S0 read + S_final written


def test_clock_summary_flags_throttle():
    rows = [dict(ts=10.0 + 0.05 * i, sm=1900.0, smax=2070.0, active="0x0", hw="Not Active",
                 hwt="Not Active", swt="Not Active", pcap="Active" if i == 3 else "Not Active")
            for i in range(10)]
    s = bench.ClockSampler.summarise(rows, 10.1, 10.3)
    assert s["sm_mhz"] == 1900.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    s2 = bench.ClockSampler.summarise(rows, 50.0, 50.001)  # outside: nearest samples
    assert s2["samples"] == 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(1.5 + rank, w)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}
