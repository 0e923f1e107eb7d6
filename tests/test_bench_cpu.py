"""Host-side checks of bench.py that need no GPU: the reference arm (the CPU
oracle) prints the contract's JSON line, a two-rank launch through
torch.distributed.run over gloo prints it on rank 0 only, and the step-time
reduction over ranks takes the maximum."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(out: str):
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def _env(**extra):
    env = dict(os.environ)
    env.update(extra)
    return env


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "dsv3", "--steps", "1",
                        "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["higher_is_better"] is False
    assert d["config"]["workload"].startswith("dsv3")
    for key in ("global_batch", "seq_len", "parallelism"):
        assert key in d["config"], key
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_two_gloo_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--workload", "dsv3",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900,
                       env=_env(MLA_BENCH_BACKEND="gloo", OMP_NUM_THREADS="4"))
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout[-2000:]  # rank 0 alone prints
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def _ranks_worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        q.put((rank, bench.max_over_ranks(1.5 + rank, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ranks_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_default_workload_is_the_largest_single_gpu_configuration():
    """With no flags the benchmark times the multi-token causal workload end to
    end (B = 132, s_q = 2, 4096 tokens): the largest configuration of the path
    that fits one GPU; the other named workloads are reported decode-only."""
    sys.path.insert(0, ROOT)
    import bench
    from mla_paged_kv_absorbed_gb300 import inputs as gen
    assert bench.WORKLOAD == "spec"
    w = gen.WORKLOADS["spec"]
    assert (w["B"], w["s_q"], w["H"], w["seqlens"], w["q_mode"]) == (132, 2, 128, 4096, "q")
    assert set(bench.DECODE_WORKLOADS) == {"dsv3", "varlen", "long"}


def test_kernel_code_hash_ignores_comments_only():
    """The key of a recorded traffic capture survives comment and layout edits
    of the kernel source but no change of its code, string literals included."""
    sys.path.insert(0, ROOT)
    import bench
    strip = bench._strip_comments
    base = 'int f(int a) {\n  return a + 1;  // one\n}\nconst char* s = "x // y";\n'
    assert strip(base) == strip('/* doc */ int f(int a)\n{ return a + 1; }\n// tail\nconst char* s = "x // y";')
    assert strip(base) != strip(base.replace("a + 1", "a + 2"))
    assert strip(base) != strip(base.replace('"x // y"', '"x"'))
    assert strip("char c = '\\''; // q") == "char c = '\\'';"
    assert len(bench.kernel_code_sha256()) == 64
