"""The multi-rank path of bench.py (independent replicas, slowest-rank timing) with two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [2.0, 3.5][rank]          # rank 1 is the slow one
        slow = bench.slowest_rank_ms(local_ms, world, "cpu")
        results[rank] = (slow, bench.replica_throughput(1000, world, slow))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert results[0] == results[1]
    slow, value = results[0]
    assert slow == 3.5
    assert value == pytest.approx(2 * 1000 / 3.5e-3)


def test_single_rank_needs_no_group():
    assert bench.slowest_rank_ms(1.25, 1, "cpu") == 1.25
    assert bench.replica_throughput(16384, 1, 2.0) == pytest.approx(16384 / 2e-3)


def test_traffic_records_survive_comment_edits_only():
    """A traffic record stays bound to a kernel's code: comments do not move the hash, code does."""
    code = "// header\n__global__ void k(float* a) {  // trailing note\n\n  a[0] = 1.f;\n}\n"
    assert bench.code_digest(code) == bench.code_digest("__global__ void k(float* a) {\n  a[0] = 1.f;\n}")
    assert bench.code_digest(code) != bench.code_digest(code.replace("1.f", "2.f"))



def test_kda_chunk_traffic_record_matches_its_kernels():
    """The recorded DRAM traffic of the chunk-wise KDA call is the sum of its prep and state
    kernels, captured on the benchmark's workload (None once the kernel file's code differs)."""
    rec = bench.traffic_record("kda_chunk_prefill")
    if rec is None:
        pytest.skip("no traffic record for the current kernel code")
    kern = rec["kernels"]
    assert set(kern) == {"kda_prep_kernel", "kda_state_kernel"}
    assert rec["bytes_per_launch"] == rec["read"] + rec["write"]
    assert abs(rec["read"] - sum(k["read"] for k in kern.values())) <= 2
    assert abs(rec["write"] - sum(k["write"] for k in kern.values())) <= 2
    # the records (one of 108,032 bytes per chunk and V head) dominate the traffic beyond the
    # algorithmic bytes: written by the prep kernel, read by the state kernel
    records = (4 * 4096 // 64) * 64 * 108032
    assert kern["kda_prep_kernel"]["write"] >= 0.95 * records
    assert rec["bytes_per_launch"] >= bench.kda_prefill_bytes(4096 * 4, 4, 64) + 2 * records * 0.95


def test_clock_samples_are_summarised_with_every_active_reason():
    """The bench's nvidia-smi sampler: median SM clock, maximum clock, and each throttle reason
    seen Active at least once (Not Active and unparsable lines ignored)."""
    lines = "\n".join([
        "2070, 2070, 810.2, Not Active, Not Active, Not Active, Not Active",
        "1995, 2070, 1390.0, Not Active, Not Active, Not Active, Active",
        "[N/A], 2070, 12.0, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1200.4, Active, Not Active, Not Active, Not Active",
        "garbage",
    ])
    got = bench.ClockSampler.summarize(lines)
    assert got == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown", "sw_power_cap"], "samples": 3}
    assert bench.ClockSampler.summarize("") == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
