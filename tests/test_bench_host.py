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


def test_prefill_kv_and_gqa4096_work_follow_the_shapes():
    """prefill_kv of 512 tokens on 3584 history slots through 28 1.5B layers:
    1,341.6 GFLOP of projections and 338.3 GFLOP of attention (1,966,336
    query-key pairs per head per layer); hidden-4096 32-layer weights:
    10,939 MB."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    gemm, attn = bench.prefill_flops(synth.QWEN2_1P5B, 512, 3584)
    assert abs(28 * sum(gemm.values()) - 1341.6e9) < 0.1e9
    assert sum(3584 + t + 1 for t in range(512)) == 1_966_336
    assert abs(28 * attn - 338.3e9) < 0.1e9
    _, wbytes = bench.decode_bytes(synth.GQA_4096, 0, 32)
    assert abs(wbytes - 10_939e6) < 1e6


def test_summary_is_last_and_compact():
    """The summary repeats the main figures and compact() keeps 4 digits."""
    sys.path.insert(0, ROOT)
    import bench
    r = {"value": 1234567.891, "ms_per_step": 0.1234567, "roofline": {"frac": 0.6791457},
         "prefill_gemm_frac_of_tensor_peak": 0.4412,
         "decode": {"1024": {"us_per_step": 1129.123, "frac_of_hbm_peak": 0.3461},
                    "e2e": {"value": 800.5}, "workload": "x"}}
    s = bench.summary(r)
    assert s["decode_us_frac"] == {"1024": [1129.123, 0.3461]}
    assert s["decode_e2e_tok_s"] == 800.5
    assert bench.compact(s)["prefill_tok_s"] == 1235000.0


def test_quantized_decode_bytes_follow_the_formats():
    """Per 1.5B layer: INT8 codes are half the fp16 matrix bytes plus one
    fp16 scale per row; int4 codes a quarter plus an fp16 scale and a zero
    byte per row and group of 128."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    s = synth.QWEN2_1P5B
    n_w = (2048 * 1536 + 1536 * 1536 + 2 * 8960 * 1536 + 1536 * 8960)
    rows = 2048 + 1536 + 2 * 8960 + 1536
    extra = 2 * 2 * 1536 + 2 * 2048           # gains, q/k/v biases
    kv = 1024 * 1025
    assert bench.quant_bytes(s, "i8", 0, 1024, 1) == n_w + 2 * rows + extra + kv
    groups = (2048 + 1536 + 2 * 8960) * (1536 // 128) + 1536 * (8960 // 128)
    assert bench.quant_bytes(s, "u4", 128, 1024, 1) == n_w // 2 + 3 * groups + extra + kv
