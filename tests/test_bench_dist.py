"""The multi-rank logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own replica of the layer; the timed region is closed by a
barrier and the reported time is the max over ranks. The reference arm runs
on rank 0 only; other ranks exit 0 without work.
"""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    t = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    bench.barrier(world)
    results[rank] = (t,) + bench.dist_info()
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_with_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == (15.0, 0, 2, 0)
    assert results[1] == (15.0, 1, 2, 1)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.parse_args(["--impl", "reference"])) == 0
    assert capsys.readouterr().out == ""


def test_selected_pairs_counts_the_causal_half_of_the_diagonal():
    nb = 3
    rb = np.zeros((1, nb, 1), np.uint32)
    rb[0, 0, 0] = 0b001  # diagonal only
    rb[0, 1, 0] = 0b011  # one off-diagonal + diagonal
    rb[0, 2, 0] = 0b001  # one off-diagonal, no diagonal
    assert bench.selected_pairs(rb, nb * 128) == 2 * (128 * 129 // 2) + 2 * 128 * 128
    # a short last block (n = 300: 44 tokens): its row counts 44 query rows
    assert bench.selected_pairs(rb, 300) == 2 * (128 * 129 // 2) + 128 * 128 + 44 * 128


def test_profiled_traffic_is_dropped_once_a_source_changes(tmp_path, monkeypatch):
    # The DRAM-traffic figure of a committed ncu summary is reported only
    # while the sources that decide it hash to the recorded value; a run of
    # the same recipe at another length gets the per-block figure scaled by
    # its own selected blocks; another recipe gets none.
    import hashlib
    from types import SimpleNamespace as NS
    (tmp_path / "a.cu").write_bytes(b"kernel")
    (tmp_path / "b.cu").write_bytes(b"order")
    sha = hashlib.sha256(b"kernel" + b"order").hexdigest()
    (tmp_path / "p.md").write_text(f"# summary\n\nworkload: llama8b-512k@65536\ntraffic_bytes_per_launch: 1234\n"
                                   f"selected_blocks: 100\ntraffic_bytes_per_selected_block: 12.34\n"
                                   f"source_sha256: {sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    same = NS(name="llama8b-512k@65536")
    full = NS(name="llama8b-512k")
    other = NS(name="qwen7b-128k")
    assert bench.profiled_traffic(("a.cu", "b.cu"), "p.md", same, 100)[0] == 1234
    assert bench.profiled_traffic(("a.cu", "b.cu"), "p.md", full, 1000)[0] == 12340
    assert bench.profiled_traffic(("a.cu", "b.cu"), "p.md", other, 1000)[0] is None
    (tmp_path / "b.cu").write_bytes(b"order changed")
    assert bench.profiled_traffic(("a.cu", "b.cu"), "p.md", same, 100)[0] is None
    assert bench.profiled_traffic(("a.cu", "missing.cu"), "p.md", same, 100)[0] is None


def test_committed_traffic_summary_names_the_guarded_sources():
    text = open(os.path.join(bench.ROOT, bench.TRAFFIC_PROFILE)).read()
    for key in ("source_sha256:", "traffic_bytes_per_launch:", "workload:"):
        assert key in text, key
    assert all(os.path.exists(os.path.join(bench.ROOT, f)) for f in bench.TRAFFIC_SOURCES)


def test_bench_arms_report_identical_configs():
    # Both arms put the same keys and values in `config` for a workload.
    from types import SimpleNamespace as NS
    args = bench.parse_args([])
    w = NS(name="llama8b-512k", hq=32, hkv=8, n=524288)
    assert bench.workload_config(w, args, 1) == bench.workload_config(w, bench.parse_args(["--impl", "reference"]), 1)
