"""Host-side logic of the benchmark, on CPU.

The multi-replica path: two gloo ranks on 127.0.0.1 reduce their step times to
the slowest one, and the job value counts every replica's units (weak
scaling).  The decode path does not shard across GPUs (replicas only), so this
reduction is its whole multi-rank logic.  Also the lookup of committed ncu
traffic figures and the reference arm's JSON line."""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist()
        step_ms = 1.5 if rank == 0 else 2.25  # rank 1 is the slowest replica
        ms = bench.max_over_ranks(step_ms, torch.device("cpu"))
        torch.distributed.barrier()
        results[rank] = (ws, r, local, ms, bench.job_value(ws, 131072, ms))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_replica():
    world = 2
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    for rank in range(world):
        ws, r, local, ms, value = got[rank]
        assert (ws, r, local) == (world, rank, rank)
        assert ms == 2.25
        assert value == pytest.approx(world * 131072 / 2.25e-3)


def test_single_process_keeps_its_own_time():
    assert bench.max_over_ranks(3.0, torch.device("cpu")) == 3.0
    assert bench.job_value(1, 1000, 2.0) == pytest.approx(5e5)


def test_traffic_record_is_read_only_for_the_current_sources(tmp_path, monkeypatch):
    # the bench reports ncu DRAM bytes only from a summary taken on the kernel
    # sources it runs
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text("text\ntraffic record: kernel=tq::split_ws_kernel workload=w:k3lq "
                               "source_hash=00aa11bb22cc33dd dram_bytes_per_launch=163030000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "_kernel_source_hash", lambda: "00aa11bb22cc33dd")
    assert bench._ncu_traffic("tq::split_ws_kernel", "w:k3lq") == 163030000
    assert bench._ncu_traffic("tq::split_ws_kernel", "w:k4uq") is None
    monkeypatch.setattr(bench, "_kernel_source_hash", lambda: "ffffffffffffffff")
    assert bench._ncu_traffic("tq::split_ws_kernel", "w:k3lq") is None


def test_reference_arm_prints_one_contract_line():
    # the reference arm times the oracle on the host cores and prints one JSON
    # line with the contract's keys
    import json
    import subprocess

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "KV tokens/s"
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "llama8b_gqa4_b16_8k"
