"""The multi-GPU form of the benchmark runs independent replicas (one process per GPU, no
exchange on the data path): the timings are the maxima over the ranks and the throughput
counts every replica's tokens. Checked here with two gloo processes on the CPU."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank, 5.0]   # this replica's step, e2e and kernel times
        got = bench.max_over_ranks(mine, dist, device="cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_timings_are_maxima_over_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == [2.0, 10.0, 5.0]


def test_job_throughput_counts_every_replica():
    assert bench.job_tokens_per_s(4, 1, 0.5) == pytest.approx(8000.0)
    assert bench.job_tokens_per_s(4, 8, 0.5) == pytest.approx(64000.0)
    assert bench.max_over_ranks([1.5, 2.5], None) == [1.5, 2.5]


def test_reference_arm_prints_on_rank_zero_only():
    class A:
        config, steps, warmup = 0, 1, 0
    assert bench.run_reference(A(), rank=1, world=2) is None


def test_traffic_records_name_existing_kernel_sources():
    # a committed DRAM-traffic figure is reported only while the hash of its kernel's own
    # sources matches; the listed files must exist, and the hash must not depend on anything else
    pkg = os.path.join(ROOT, "mtp_speculative_decoding_gemma4_gb300", "csrc")
    for kernel, names in bench.KERNEL_SOURCES.items():
        for n in names:
            assert os.path.isfile(os.path.join(pkg, n)), (kernel, n)
        assert bench.kernel_source_hash(kernel) == bench.kernel_source_hash(kernel)
        assert bench.kernel_source_hash(kernel) != bench.kernel_source_hash("")
    assert bench.ncu_traffic("no_such_kernel", 1) is None


def test_sparse_head_switch_maps_to_the_abi_enum():
    from mtp_speculative_decoding_gemma4_gb300 import binding as B
    assert bench.SPARSE_HEAD == {"auto": B.HEAD_AUTO, "per-sequence": B.HEAD_PER_SEQUENCE,
                                 "cluster-major": B.HEAD_CLUSTER_MAJOR}
