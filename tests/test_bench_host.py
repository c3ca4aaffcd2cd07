"""bench.py host logic on CPU: work accounting and the multi-rank reduction (gloo, world size 2)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as wl


def test_kernel_work_matches_plan_stats():
    import muon_newton_schulz_09_b300 as mu
    w = wl.GPT2_124M
    work = bench.kernel_work(w)
    s = mu.plan_stats(w.shapes)
    assert work["gram_xxt"][1] + work["combine_ax_bx"][1] == pytest.approx(5 * s["flops_per_iter"])
    assert bench.step_flops(w) == pytest.approx(5 * s["flops_per_iter"])
    assert work["momentum_norm"] == ("bytes", 84934656 * 12.0)
    assert work["update"] == ("bytes", 84934656 * 6.0)


def test_kernel_work_counts_the_carried_low_part():
    w = wl.GPT2_124M
    plain, carry = bench.kernel_work(w), bench.kernel_work(w, carry=True)
    assert carry["momentum_norm"] == ("bytes", 84934656 * 14.0)
    assert carry["update"] == ("bytes", 84934656 * 8.0)
    assert carry["gram_xxt"] == plain["gram_xxt"] and carry["combine_ax_bx"] == plain["combine_ax_bx"]
    sq = bench.kernel_work(wl.SQUARE_64x1024, carry=True)
    assert sq["scale_orient"] == ("bytes", 64 * 1024 * 1024 * 6.0) and sq["copy_out"] == ("bytes", 64 * 1024 * 1024 * 8.0)


def test_matrix_fraction_sums_to_one():
    for w in wl.WORKLOADS.values():
        f = bench.matrix_fraction(w)
        assert len(f) == w.count and abs(sum(f) - 1.0) < 1e-12
    assert [wl.GPT2_124M.shapes[j] for j in bench.distinct_matrices(wl.GPT2_124M)] == [
        (768, 768), (768, 3072), (3072, 768)]


def test_whole_job_rate():
    assert bench.whole_job_rate(100, 4, 2.0) == 200.0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, rank, world)
        bench.barrier()
        m = bench.reduce_max(1.0 + rank)  # the slowest rank's time
        q.put((rank, m, bench.whole_job_rate(10, world, m)))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2.0, 10.0), (1, 2.0, 10.0)]


def test_reference_arm_rank_nonzero_does_nothing(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(workload=wl.GPT2_124M.name, steps=1, warmup=3)
    assert bench.run_reference(args) == {}


def test_reference_arm_small_workload(monkeypatch):
    w = wl.small_workload("tiny", [(32, 64), (64, 32)], kind="step", grad_std=1e-3, seed=3)
    monkeypatch.setitem(wl.WORKLOADS, "tiny", w)
    monkeypatch.delenv("RANK", raising=False)
    line = bench.run_reference(bench.argparse.Namespace(workload="tiny", steps=4, warmup=3))
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_config_matches_ours(monkeypatch):
    """Both arms print the same config object for the same workload, so their lines compare."""
    w = wl.small_workload("tiny2", [(32, 64), (64, 32)], kind="step", grad_std=1e-3, seed=4)
    monkeypatch.setitem(wl.WORKLOADS, "tiny2", w)
    monkeypatch.delenv("RANK", raising=False)
    line = bench.run_reference(bench.argparse.Namespace(workload="tiny2", steps=2, warmup=3))
    assert line["config"] == bench.config_of(w, 1, False)
    assert set(line["config"]) >= {"workload", "parallelism", "l2", "precise_carry", "alg_flops_per_step"}


def test_peak_choice_follows_the_region_length():
    """A region under a second is a kernel timed in a short burst: the burst peak applies."""
    assert not bench.uses_sustained_peak(0.022)
    assert not bench.uses_sustained_peak(0.6)
    assert bench.uses_sustained_peak(1.0) and bench.uses_sustained_peak(30.0)


def test_resident_bytes_of_the_headline_step():
    # bf16 grads (2) + fp32 momentum (4) + bf16 params (2) per element
    assert bench.resident_bytes(wl.GPT2_124M) == 84934656 * 8


def test_traffic_is_read_only_for_its_own_workload_and_sources(monkeypatch):
    """The ncu traffic of one workload's capture is never reported for another workload, another
    kernel or other kernel sources."""
    monkeypatch.setattr(bench, "source_hash", lambda: "h1")
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {"h1": {"gpt2_124m_hidden": {"newton_schulz": 3.0e9}}})
    assert bench.ncu_traffic("gpt2_124m_hidden", "newton_schulz") == 3.0e9
    assert bench.ncu_traffic("gpt2_124m_hidden_quintic", "newton_schulz") is None
    assert bench.ncu_traffic("gpt2_124m_hidden", "momentum_norm") is None
    monkeypatch.setattr(bench, "source_hash", lambda: "h2")
    assert bench.ncu_traffic("gpt2_124m_hidden", "newton_schulz") is None


def test_traffic_table_entries_name_known_workloads():
    for per_hash in bench.NCU_TRAFFIC.values():
        for name, kernels in per_hash.items():
            assert name in wl.WORKLOADS
            assert set(kernels) <= set(bench.kernel_work(wl.WORKLOADS[name]))
