"""The bench's multi-rank host logic on CPU: two gloo ranks agree on the maximum of their
timings (the whole-job time), and only rank 0 runs the reference arm."""
import os
import socket
import sys

import pytest

from tests.conftest import ROOT

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    t = bench.max_over_ranks(1.5 * (rank + 1), world)
    out.put((rank, t))
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 3.0, 1: 3.0}


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus = 1, 3, 2
    bench.run_reference(A())
    assert capsys.readouterr().out == ""


def test_profiled_traffic_follows_the_kernel_code_not_its_comments(tmp_path, monkeypatch):
    """The bench attaches the committed DRAM counters only while the profiled kernel code
    is unchanged: a comment edit keeps them, a code edit retires them."""
    sys.path.insert(0, ROOT)
    import shutil
    import bench
    srcs = []
    for rel in bench.KERNEL_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(ROOT, rel), dst)
        srcs.append(dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    prof = tmp_path / "profiles" / "kernel.md"
    prof.parent.mkdir(parents=True, exist_ok=True)
    prof.write_text(f"# capture\n\n- kernel_source_sha256_16: `{bench.kernel_source_hash()}`\n"
                    "- dram_bytes_per_launch: `123456`\n")
    monkeypatch.setattr(bench, "PROFILE", str(prof))
    assert bench.profiled_traffic() == 123456.0
    with open(srcs[0], "a") as f:
        f.write("\n// a comment added after the capture\n")
    assert bench.profiled_traffic() is not None
    with open(srcs[0], "a") as f:
        f.write("\nnamespace oattn { constexpr int kAddedAfterCapture = 1; }\n")
    assert bench.profiled_traffic() is None
