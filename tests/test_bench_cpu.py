"""The benchmark's host-side contract on CPU: the reference arm (the oracle timed on the host)
prints one JSON line with the keys of the benchmark contract, and the byte counts and DRAM-traffic record
the GPU lines use behave as documented."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1",
                        "--workload", "nadam_1m"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    import oracle
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == oracle.threads() >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "nadam_1m"


def test_byte_counts_and_traffic_record():
    import bench
    # factored: 10 B per element plus fp32 row and column state (read and written)
    assert bench.factored_bytes((1024, 512)) == 10 * 1024 * 512 + 8 * (1024 + 512)
    assert bench.factored_bytes((4, 6, 3, 3)) == 10 * 216 + 8 * 24 * 6
    assert bench.factored_bytes((77,)) == 10 * 77 + 8 * 77
    # Prodigy statistics: 12 B per sampled element, 64-element blocks, every slice_p-th block
    assert bench.prodigy_bytes((640,), 11) == 12 * 64
    assert bench.prodigy_bytes((1000,), 1) == 12 * 1024
    # the committed traffic record is used only while the kernel source hashes to the captured one
    rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    for kernel, e in rec["kernels"].items():
        t = bench.traffic_per_launch(kernel, 1000)
        if e["kernel_source_sha"] == bench.kernel_hash(kernel):
            assert abs(t - 1000 * e["dram_bytes_per_param"]) < 1e-6
        else:
            assert t is None
    assert bench.traffic_per_launch("no_such_kernel", 1000) is None


def test_reference_arm_under_torchrun_two_ranks():
    """Launched as the multi-GPU bench is (torchrun, two ranks): rank 0 alone runs the oracle and
    prints one line, the other rank exits 0 without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "1", "--workload", "nadam_1m"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "nadam_1m"
