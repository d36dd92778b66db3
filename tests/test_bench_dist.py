"""bench.py's multi-rank host logic on CPU (gloo, world size 2): the barrier,
the max-over-ranks timing reduce and the sum of the column split's bytes, and the reference arm under torchrun printing
exactly one line from rank 0.  No GPU is involved."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + rank, w, torch.device("cpu"))
    total = bench.sum_over_ranks(1.0 + rank, w, torch.device("cpu"))   # the column split's job bytes
    q.put((rank, (got, total)))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: (11.0, 3.0), 1: (11.0, 3.0)}


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "0",
           "--workload", "gemv_k1024_n3072"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_kernel_source_hash_ignores_comments_only():
    """The profile records' source hash covers the code the compiler sees:
    editing a comment keeps it, editing code changes it."""
    sys.path.insert(0, ROOT)
    import bench
    base = 'int f(int x) { return x + 1; }  // add one\n/* doc */ const char *s = "a//b /* not a comment */";\n'
    same = '/* header */\nint f(int x)\n{\n    return x + 1;   // plus one\n}\nconst char *s = "a//b /* not a comment */";'
    other = 'int f(int x) { return x + 2; }\nconst char *s = "a//b /* not a comment */";'
    assert bench._code_only(base) == bench._code_only(same)
    assert bench._code_only(base) != bench._code_only(other)
    assert '"a//b /* not a comment */"' in bench._code_only(base)
    assert len(bench.kernel_source_hash()) == 16


def test_row_block_count_matches_the_header():
    """bench.py counts a call's passes over the weights with the header's
    batch rows per pass; the batch limit and the binding agree with it."""
    import re
    sys.path.insert(0, ROOT)
    import bench
    import glu_inputs as gi
    import memory_bound_glu_gb300 as mb
    hdr = open(os.path.join(ROOT, "include", "mbglu.h")).read()
    assert int(re.search(r"#define MBGLU_BLOCK_M (\d+)", hdr).group(1)) == bench.BLOCK_M == mb.BLOCK_M
    assert int(re.search(r"#define MBGLU_MAX_M (\d+)", hdr).group(1)) == mb.MAX_M
    # glu_gemv takes batches above 16 rows in one pass (the tcgen05 kernel on
    # the bench's aligned operands); add_rmsnorm_glu runs them as row blocks
    w = gi.WORKLOADS["gemv_k2560_n9728_wide"]
    assert [bench.row_blocks(w, M) for M in (1, 16, 17, 32, 33, 64)] == [1] * 6
    wn = gi.WORKLOADS["norm_gemv_k2560_n9728"]
    assert [bench.row_blocks(wn, M) for M in (1, 16, 17, 32, 33, 64)] == [1, 1, 2, 2, 3, 4]
    assert bench.row_blocks(gi.WORKLOADS["silu_mul_m4096_n9728"], 4096) == 1


def test_recorded_traffic_is_current_only_for_the_profiled_sources(monkeypatch):
    """traffic is reported only while the kernel sources hash to the profiled
    ones; otherwise it is None and the last capture is described, marked as
    taken on other sources."""
    sys.path.insert(0, ROOT)
    import bench
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["gemv_k2560_n9728/M1/hf"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["source_hash"])
    cur, last = bench.recorded_traffic("gemv_k2560_n9728", 1, "hf")
    assert cur == rec["dram_bytes_per_launch"] and last["sources_changed_since"] is False
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    cur, last = bench.recorded_traffic("gemv_k2560_n9728", 1, "hf")
    assert cur is None and last["sources_changed_since"] is True
    assert last["dram_bytes_per_launch"] == rec["dram_bytes_per_launch"]
    assert bench.recorded_traffic("gemv_k2560_n9728_wide", 32, "hf") == (None, None)


def test_clock_sampler_follows_cuda_visible_devices(monkeypatch):
    """The clocks are sampled on the GPU the rank runs on: nvidia-smi numbers
    the physical devices, CUDA those left visible."""
    import bench
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES", raising=False)
    assert bench.smi_id(0) == "0" and bench.smi_id(3) == "3"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3")
    assert bench.smi_id(0) == "3"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "4, 6,7")
    assert [bench.smi_id(i) for i in range(3)] == ["4", "6", "7"]
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-0a1b2c3d-0000-1111-2222-333344445555")
    assert bench.smi_id(0) == "GPU-0a1b2c3d-0000-1111-2222-333344445555"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "")
    assert bench.smi_id(1) == "1"
