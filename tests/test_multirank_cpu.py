"""Host-side logic of the N > 1 benchmark path, run as two gloo ranks on the CPU.

Under torchrun every rank runs the same workload on its own GPU (weak scaling; the layer
shards by channel or batch with no data-path collective); the only cross-rank steps are
the barrier around the timed region and the max-over-ranks of the elapsed time, which is
what is exercised here."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench.dist_env()
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + 5.0 * rank, w, None)
    # the reference arm: only rank 0 does work; the others return 0 at once
    class A:
        steps = 1
        warmup = 0
        gpus = world
    rc = None
    if r != 0:
        rc = bench.run_reference(A, None)
    q.put((r, w, local, m, rc))
    dist.destroy_process_group()


def test_two_rank_max_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    assert all(o[3] == pytest.approx(15.0) for o in out)  # max over ranks
    assert out[1][4] == 0  # non-zero ranks of the reference arm exit without work


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_fp32_peak_from_unit_counts():
    import bench
    assert bench.derived_fp32_peak_tflops(152, 2070.0) == pytest.approx(
        152 * 128 * 2 * 2.07e9 / 1e12)


def test_cpu_baseline_brief_leg_for_forward_only_workloads():
    """The per-config oracle figures: a brief all-cores and one-thread timing, also for the
    forward-only workload (no dY)."""
    import bench
    from depthwise_receptive_field_gb300.inputs import WORKLOADS
    r = bench.cpu_baseline(WORKLOADS["c1_small_fwd"], target_s=0.02, single_s=0.02, brief=True)
    assert r["all_cores_gelem_s"] > 0 and r["one_thread_gelem_s"] > 0 and r["cores"] >= 1


def test_cpu_baseline_legs():
    """The bench's oracle baseline: an all-cores leg and a one-thread leg on bounded
    samples, the host's CPU described, and the oracle's thread count restored after."""
    import bench
    import oracle
    from depthwise_receptive_field_gb300.inputs import WORKLOADS
    before = oracle.num_threads()
    r = bench.cpu_baseline(WORKLOADS["c2_fp32_train"], target_s=0.05, single_s=0.05)
    assert r["kind"] == "oracle" and r["cores"] == before and r["value"] > 0
    assert r["single_thread"]["cores"] == 1 and r["single_thread"]["value"] > 0
    assert r["host"]["os_cpu_count"] == os.cpu_count() and r["host"]["cpu_model"]
    assert oracle.num_threads() == before
