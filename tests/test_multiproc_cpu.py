"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each with
its own timing, reduce to the slowest rank's time and report the whole-job
throughput; under the reference arm only rank 0 does work.  (Ranks are
independent replicas: no data-path collective exists to test.)"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, lr = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    my_ms = 2.0 + rank  # rank 1 is the slow one
    dist.barrier()
    slowest = bench.reduce_max(my_ms, dist)
    q.put((r, w, lr, slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    assert all(x[1] == 2 for x in res)
    assert all(x[3] == 3.0 for x in res)                  # both see the slowest rank
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_tokens_per_s(16384, 2, 3.0) == pytest.approx(16384 * 2 / 3e-3)


def test_reference_arm_other_ranks_do_nothing(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup = 1, 0

    w = bench.TI.WORKLOADS["tiny_f32_n512"]
    assert bench.run_reference(A(), w, 128, rank=1, world=2) == 0
    assert capsys.readouterr().out == ""


def test_algorithmic_work_counts():
    sys.path.insert(0, ROOT)
    import bench
    w = bench.TI.WORKLOADS["qwen3_1p7b_n16k_keep10"]
    K = w.Ks()[0]
    work = bench.algorithmic_work(w, K)
    M = w.M(K)
    assert M == 1868
    assert work["keybias_attn"]["flops"] == 2 * M * M * 128 * 16
    assert work["qkv_proj"]["flops"] == 2 * M * 2048 * 4096
    assert work["gate_score"]["flops"] == 2 * 16384 * 2048 * 256
    assert work["gather_rows"]["bytes"] == 2 * M * 2048 * 2 + 12 * M


def test_backward_work_counts_and_traffic_table():
    sys.path.insert(0, ROOT)
    import bench
    w = bench.TI.WORKLOADS["qwen3_1p7b_n128k_keep6p25"]
    M = w.M(w.Ks()[0])
    assert M == 8432
    bw = bench.backward_work(w, M)
    assert set(bw) == set(bench.BWD_KERNELS)
    # two products of 2 dh flops per causal (query, key) pair and q head
    assert bw["keybias_bias_grad"]["flops"] == 2 * M * M * 128 * 16
    assert bw["attn_bwd_delta"]["bytes"] == 2 * M * 16 * 128 * 2 + 16 * M * 4
    # every ncu entry names a known kernel source; a current hash gives bytes,
    # a stale one None
    for key, trf in bench.NCU_TRAFFIC.items():
        wl, kern = key.split("/")
        assert kern in bench.KERNEL_SOURCES and wl in bench.TI.WORKLOADS
        got = bench.ncu_traffic(wl, kern)
        fresh = trf["source_sha"] == bench.source_hash(bench.KERNEL_SOURCES[kern])
        assert got == (trf["bytes_per_launch"] if fresh else None)
    assert bench.ncu_traffic(w.name, "no_such_kernel") is None


def test_default_workload_traffic_is_current():
    """The bench's default workload has a DRAM-traffic entry for every kernel
    of the step, captured from the kernels' current sources (a kernel changed
    since its capture reports null traffic and fails here until re-captured)."""
    import bench
    for kern in bench.KERNELS:
        assert bench.ncu_traffic(bench.DEFAULT_WORKLOAD, kern) is not None, kern


def test_tensor_peak_follows_the_clock_record():
    """A run that held its SM clock is measured against the burst bf16 peak;
    one that was power-capped (or ran well below the maximum clock) against
    the sustained one, and the line says which."""
    import bench
    peaks = {"bf16_tflops": 1755.4, "bf16_tflops_sustained": 1377.5, "hbm_gbs": 6484.9}
    assert bench.tensor_peak(peaks, {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0,
                                     "reasons": []})[0] == 1755.4
    assert bench.tensor_peak(peaks, None)[0] == 1755.4
    p, why = bench.tensor_peak(peaks, {"sm_mhz": 1762.0, "sm_max_mhz": 2032.0,
                                       "reasons": ["sw_power_cap"]})
    assert p == 1377.5 and "sustained" in why
    assert bench.tensor_peak(peaks, {"sm_mhz": 1900.0, "sm_max_mhz": 2032.0,
                                     "reasons": []})[0] == 1377.5
