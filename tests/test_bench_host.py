"""Host-side logic of bench.py on CPU: the max-over-ranks timing and barrier
of the replica (N > 1) path with the gloo backend at world size 2, and the
reference arm launched under torchrun (rank 0 prints one JSON line, the other
rank exits without work)."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=2)
    bench.barrier(2)
    v = bench.reduce_max(1.5 + rank, 2)
    out[rank] = v
    bench.barrier(2)
    dist.destroy_process_group()


def test_replica_timing_takes_max_over_ranks():
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(port, out), nprocs=2, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_under_torchrun_world_size_2():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--steps", "1", "--warmup", "0", "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_decode_bytes_follow_the_shape():
    """Per layer of the 1.5B shape: 93,595,648 weight bytes (q/k/v with bias,
    o, gate, up, down, two gains) plus 2 * Hkv * D * 2 = 1,024 K/V bytes per
    attended slot."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    total, weights = bench.decode_bytes(synth.QWEN2_1P5B, 1024, 28)
    assert weights == 28 * 93_595_648
    assert total == 28 * (93_595_648 + 1024 * 1025)


def test_prefill_flops_follow_the_shape():
    """[1, 1024] through one 1.5B layer: 95.83 GFLOP of projections and
    4 * D * Hq * (1024 * 1025 / 2) of causal attention."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    gemm, attn = bench.prefill_flops(synth.QWEN2_1P5B, 1024)
    assert abs(sum(gemm.values()) - 95.83e9) < 0.01e9
    assert attn == 4 * 128 * 12 * (1024 * 1025 // 2)


def test_oracle_decode_sample_extrapolates_over_layers():
    sys.path.insert(0, ROOT)
    import bench
    us, secs, desc = bench.oracle_decode_sample(L=16, n_layers=3)
    assert secs > 0 and abs(us - 3 * secs * 1e6) < 1e-6 * us
    assert "extrapolated x3 layers" in desc
