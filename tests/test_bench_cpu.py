"""Host-side logic of bench.py that needs no GPU: the multi-rank aggregation
(max time over ranks, units summed) with two gloo ranks on CPU, and the
reference arm's JSON line on a tiny workload."""
import json
import os
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, units = bench.aggregate(1.0 + rank, 100.0 * (rank + 1), world)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    assert all(ms == 2.0 and units == 300.0 for _, ms, units in res)


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_tensor_peak_choice():
    """The prefill roofline divides by the measured burst bf16 rate for a short
    timed region and by the measured sustained rate for a long one."""
    sys.path.insert(0, ROOT)
    import bench
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        p = json.load(f)
    assert bench.measured_tensor_peak() == (p["bf16_tflops"], "measured burst")
    assert bench.measured_tensor_peak(sustained=True) == (p["bf16_tflops_sustained"], "measured sustained")


def test_source_hash_ignores_comments_only():
    import bench
    code = 'int f(int x) {\n  return x + 1;  // one\n}\n/* a note */\nconst char* s = "a // b /* c */";\n'
    same = '// header\nint f(int x) {\n\n  return x + 1;\n}\nconst char* s = "a // b /* c */";  /* x */\n'
    other = 'int f(int x) {\n  return x + 2;\n}\nconst char* s = "a // b /* c */";\n'
    assert bench.strip_comments(code) == bench.strip_comments(same)
    assert bench.strip_comments(code) != bench.strip_comments(other)
    assert '"a // b /* c */"' in bench.strip_comments(code)
    # the committed traffic figures are keyed by the current decode sources
    assert bench.recorded_traffic("llama2-7b") is not None


def test_every_decode_workload_has_traffic_on_the_current_sources():
    """Each workload the benchmark times (all but the tiny one, which fits in
    L2) has a DRAM-traffic line captured on the current decode sources, within
    a few percent above its algorithmic bytes (the excess: the newest rows
    appended in the launch and the chunk partials written)."""
    import bench
    from fp8_int8_quantized_gb300 import workloads as W
    for name in bench.DEFAULT_STEPS:
        if name == "tiny":
            continue
        t = bench.recorded_traffic(name)
        assert t is not None, name
        wl = W.WORKLOADS[name]
        alg = W.decode_bytes(wl, W.context_lens(wl))["total"]
        assert 1.0 <= t / alg < 1.03, (name, t / alg)
