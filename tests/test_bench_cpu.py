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


def test_reference_arm_json_line(capsys):
    """`bench.py --impl reference` times the oracle on the host and prints one
    JSON line with the contract's keys (small sample: runs in about a second)."""
    import json
    bench.main(["--impl", "reference", "--workload", "small_bf16", "--steps", "2",
                "--warmup", "3", "--ref-tokens", "32"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["one_thread"]["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("small_bf16")
    # the step time matches the reported rate: B sequences x 32 tokens per step
    w = I.WORKLOADS["small_bf16"]
    assert abs(d["ms_per_step"] - 1e3 * w.B * 32 / d["value"]) < 1e-6 * d["ms_per_step"] + 1e-9


def test_kernel_source_hash_covers_every_local_include():
    """A recorded DRAM-traffic figure stays valid only while the code it was
    measured on is unchanged: the hash must cover the kernel file and every
    local header it includes (recursively)."""
    import re
    csrc = os.path.join(os.path.dirname(bench.__file__), "gated_delta_rule_09_gb300", "csrc")

    def closure(name, seen):
        if name in seen:
            return seen
        seen.add(name)
        text = open(os.path.join(csrc, name)).read()
        for inc in re.findall(r'#include "([^"]+)"', text):
            closure(inc, seen)
        return seen

    for workload, files in bench.KERNEL_SOURCES.items():
        assert closure(files[0], set()) == set(files), workload
