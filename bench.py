#!/usr/bin/env python
"""Throughput of the GB300 decoder-block library on synthetic seeded inputs.

Headline (one JSON line on rank 0): prefill tokens/s of one 1.5B-shaped layer
(hidden 1536, 12 q / 2 kv heads, head_dim 128, intermediate 8960, QKV bias)
at the static prefill shape [1, 1024], position_ids 0..1023.  A step is one
blk_prefill call (the whole block: RMSNorm, QKV + bias, RoPE + KV append,
causal GQA attention, o_proj + residual, RMSNorm, SwiGLU MLP + residual).
The L2 is flushed (a 256 MB write) before every timed step, because one
layer's weights (94 MB) fit in the 129 MB L2.

Also reported, each as an absolute number and a fraction of its roofline:
  decode         the 28-layer 1.5B stack at cache lengths 1024, 4096, 16384
                 and 32768 (one CUDA graph per step, KV appended in place),
                 us/step vs the HBM roofline (weight + KV bytes over the
                 measured copy bandwidth), plus an end-to-end figure (host
                 hidden row in, host output row out, through the public API)
  prefill_kv_28  the 28-layer 1.5B stack, 512 new tokens at positions
                 3584..4095 on 3584 history slots: tok/s, GEMM time vs the
                 tensor peak, attention time and share reported separately
  gqa4096        32 layers of hidden 4096 / 32 q heads / 2 kv heads: a
                 prefill of 100 tokens, then 256 decode steps at positions
                 100..355 (both bound by HBM bytes)
  lm_head, model_per_token, decode_batch  the model head, a whole generated
                 token, batched decode of B sequences
The weights of every leg exceed the L2 except the headline's (flushed).
The CPU oracle is timed on a bounded prefill sample (cpu_baseline) and on one
decode layer extrapolated to the stack (cpu_baseline_decode).  The last key
of the line, "summary", repeats the main figures in a few hundred bytes.

--impl reference times the CPU oracle (single-threaded f64) on the same
bounded prefill sample per step.  Under torchrun (N > 1) each rank runs an
independent replica (no collective on the data path); rank 0 prints the
whole-job numbers.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "prefill tok/s (1.5B-shaped layer, [1,1024]) + decode us/step vs ctx (28 layers)"
UNIT = "tok/s"
DECODE_CTX = (1024, 4096, 16384, 32768)
PREFILL_T = 1024
ORACLE_SAMPLE_ROWS = 32     # full-output rows of the oracle's prefill sample
PKV_HIST, PKV_T = 3584, 512        # prefill_kv leg: history slots, new tokens
G4_PREFILL, G4_DECODES = 100, 256  # hidden-4096 leg: prefill tokens, decode steps
DECODE_STEPS = 128                 # consecutive decode steps timed per context length

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of the kernel as it is built now; None when the kernel
# changed after its last capture.  The captures and their commands:
# profiles/prefill_kernels_1p5b_T1024.md (the prefill GEMMs, attention and
# split-K reduction), profiles/decode_persistent_1p5b_1layer_ctx4096.md
# (decode) and profiles/lm_head_1p5b_vocab151936.md (model head).
NCU_TRAFFIC = {
    "gemm_gateup": 58228736 + 79104,
    "gemm_down": 45917952 + 15872,
    "gemm_qkv": 10027008 + 0,
    "gemm_o": 11042560 + 0,
    "attn_prefill": 4251392 + 0,
    "splitk_reduce": 25171456 + 0,
    "lm_head": 466853632 + 206080,
    # one-layer capture scaled to the 28-layer step (traffic grows with the layers)
    ("decode_persistent", 4096): 28 * (101665280 + 4095488),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--decode-ctx", type=str, default=",".join(map(str, DECODE_CTX)))
    ap.add_argument("--decode-batch", type=str, default="8,32,64",
                    help="batch sizes of the batched decode table (ctx --decode-batch-ctx)")
    ap.add_argument("--decode-batch-ctx", type=int, default=1024)
    ap.add_argument("--only", choices=("prefill", "decode", "decode_batch", "prefill_kv",
                                       "gqa4096", "decode_layer", "decode_quant",
                                       "decode_batch_layer"), default=None,
                    help="run one part (for profiling); the headline needs the prefill.  "
                         "decode_layer runs one 1.5B-shaped layer of decode at ctx "
                         "--decode-ctx[0] (small enough for an ncu capture); "
                         "decode_batch_layer one layer of batched decode at the largest "
                         "--decode-batch, ctx --decode-batch-ctx")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        self.proc.wait()
        self.file.flush()
        rows = [r.split(",") for r in open(self.file.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ helpers

def dist_init(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available() and args.impl == "ours":
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v, ws):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def prefill_flops(s, T, L=0):
    H, Hq, Hkv, D, I = s.hidden, s.n_heads, s.n_kv_heads, s.head_dim, s.intermediate
    gemm = {
        "gemm_qkv": 2.0 * T * (Hq + 2 * Hkv) * D * H,
        "gemm_o": 2.0 * T * H * Hq * D,
        "gemm_gateup": 2.0 * T * 2 * I * H,
        "gemm_down": 2.0 * T * H * I,
    }
    pairs = sum(L + t + 1 for t in range(T))          # (query, key) pairs per head
    attn = 4.0 * D * Hq * pairs                       # QK^T and PV, 2 flops per MAC
    return gemm, attn


def decode_bytes(s, L, n_layers):
    H, Hq, Hkv, D, I = s.hidden, s.n_heads, s.n_kv_heads, s.head_dim, s.intermediate
    w = 2 * ((Hq + 2 * Hkv) * D * H + H * Hq * D + 3 * I * H + 2 * H)
    if s.has_qkv_bias:
        w += 2 * (Hq + 2 * Hkv) * D
    kv = 2 * Hkv * D * 2 * (L + 1)
    return n_layers * (w + kv), n_layers * w


# ------------------------------------------------------------- CPU oracle

_ORACLE_INPUTS = {}


def oracle_prefill_sample(n_rows: int, rotate: int = 0, t_kv: float | None = None):
    """Times the oracle on a bounded sample of the prefill workload: K/V of
    all 1024 rows plus the full block output of n_rows evenly spaced rows.
    The whole-layer figure is extrapolated from it: t_kv (the K/V of every
    row plus one output row, timed once when not given) + the sampled rows'
    cost scaled to 1024 rows.  Returns (tok/s extrapolated, seconds the
    sample took, t_kv, description)."""
    import oracle
    import synth
    s = synth.QWEN2_1P5B
    if not _ORACLE_INPUTS:
        oracle.build()
        _ORACLE_INPUTS.update(w=synth.block_weights(s, seed=0),
                              x=synth.hidden_input(s, PREFILL_T, seed=0),
                              pos=synth.positions(0, PREFILL_T))
    w, x, pos = _ORACLE_INPUTS["w"], _ORACLE_INPUTS["x"], _ORACLE_INPUTS["pos"]
    if t_kv is None:
        kc, vc = synth.kv_history(s, PREFILL_T, 0)
        t0 = time.perf_counter()
        oracle.block_forward(s, w, x, pos, 0, kc, vc, rows=[0])
        t_kv = time.perf_counter() - t0           # all K/V rows + one output row
    step = PREFILL_T // n_rows
    rows = [(i * step + rotate) % PREFILL_T for i in range(n_rows)]
    kc2, vc2 = synth.kv_history(s, PREFILL_T, 0)
    t0 = time.perf_counter()
    oracle.block_forward(s, w, x, pos, 0, kc2, vc2, rows=rows)
    spent = time.perf_counter() - t0
    t_rows = max(spent - t_kv, 1e-9)              # cost of the sampled output rows
    t_full = t_kv + t_rows * PREFILL_T / n_rows
    desc = (f"oracle on the 1.5B-shaped layer, prefill [1,1024]: K/V for all 1024 rows + full "
            f"output of {n_rows} evenly spaced rows per step; tok/s extrapolated to 1024 rows; "
            f"single-threaded")
    return PREFILL_T / t_full, spent, t_kv, desc


def synth_layers() -> int:
    import synth
    return synth.QWEN2_1P5B.n_layers


def oracle_decode_sample(L: int = 1024, n_layers: int = 28):
    """Times the oracle's decode of one token through one 1.5B-shaped layer
    at L history slots, and extrapolates to an n_layers step.  Returns
    (us per step extrapolated, seconds spent, sample description)."""
    import oracle
    import synth
    s = synth.QWEN2_1P5B
    oracle.build()
    if "w" not in _ORACLE_INPUTS:
        _ORACLE_INPUTS["w"] = synth.block_weights(s, seed=0)
    w = _ORACLE_INPUTS["w"]
    kc, vc = synth.kv_history(s, L + 1, L, seed=0)
    x = synth.hidden_input(s, 1, seed=0, stream_offset=1)
    t0 = time.perf_counter()
    oracle.block_forward(s, w, x, synth.positions(L, 1), L, kc, vc)
    spent = time.perf_counter() - t0
    desc = (f"oracle decode of one token through one 1.5B-shaped layer at ctx {L}, "
            f"extrapolated x{n_layers} layers; single-threaded")
    return spent * n_layers * 1e6, spent, desc


# ------------------------------------------------------------------ ours

def bench_ours(args, ws, rank, local):
    import torch
    import decode_qwen2_block_gb300 as blk
    from decode_qwen2_block_gb300 import build as gpu_build
    from decode_qwen2_block_gb300.stack import LayerStack
    import synth

    gpu_build.build()
    peaks = load_peaks()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    s = synth.QWEN2_1P5B
    K, W = args.steps, args.warmup
    parts = {"decode": ("decode us/step (28 layers)", bench_decode),
             "decode_batch": ("batched decode tok/s (28 layers)", bench_decode_batch),
             "prefill_kv": ("prefill_kv tok/s (28 layers, 512 on 3584)", bench_prefill_kv_stack),
             "gqa4096": ("hidden-4096 32-layer prefill + decode", bench_gqa4096),
             "decode_layer": ("decode us/launch (1 layer)", bench_decode_layer),
             "decode_batch_layer": ("batched decode us/call (1 layer)", bench_decode_batch_layer),
             "decode_quant": ("quantized decode us/step (28 layers)", bench_decode_quant)}
    if args.only in parts:
        clocks = ClockSampler(local)
        clocks.start()
        metric, fn = parts[args.only]
        res = {"metric": metric, args.only: fn(args, s, dev, stream, peaks, ws)}
        if args.only == "decode":
            res["lm_head"] = bench_lm_head(args, s, dev, stream, peaks, ws)
        res["clocks"] = clocks.stop()
        return res

    # ---------------- prefill, one layer, [1, 1024] ----------------
    T = PREFILL_T
    w_np = synth.block_weights(s, layer=0, seed=0)
    w_dev = {k: torch.from_numpy(v).to(dev) for k, v in w_np.items()}
    x_np = synth.hidden_input(s, T, seed=0)
    x = torch.from_numpy(x_np).to(dev)
    pos = torch.from_numpy(synth.positions(0, T)).to(dev)
    block = blk.Block(s, T)
    wts = blk.Block.weights(w_dev)
    kc = torch.zeros((s.n_kv_heads, T, s.head_dim), dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)
    out = torch.empty((T, s.hidden), dtype=torch.float16, device=dev)
    kn = torch.empty((T, s.n_kv_heads, s.head_dim), dtype=torch.float16, device=dev)
    vn = torch.empty_like(kn)
    wsb = torch.empty(block.workspace_bytes(T), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def prefill_step():
        block.prefill(wts, x, pos, kc, vc, out, wsb, kn, vn, stream=stream)

    for _ in range(W):
        flush.zero_()
        prefill_step()
    torch.cuda.synchronize()
    block.check()

    clocks = ClockSampler(local)
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    barrier(ws)
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        evs[i][0].record(stream)
        prefill_step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = reduce_max(sum(step_ms), ws)

    # e2e: host (pinned) inputs -> device -> block -> host outputs, every
    # step.  The step's inputs (x, then position_ids) sit back to back in one
    # pinned buffer and one device buffer, and its results (out, k_new,
    # v_new) likewise, so a step is one host->device copy, the call, and one
    # device->host copy.
    nx, npos = T * s.hidden * 2, T * 8
    nout, nkv = T * s.hidden * 2, T * s.n_kv_heads * s.head_dim * 2
    in_h = torch.empty(nx + npos, dtype=torch.uint8).pin_memory()
    in_h[:nx].copy_(torch.from_numpy(x_np).view(torch.uint8).reshape(-1))
    in_h[nx:].copy_(torch.from_numpy(synth.positions(0, T)).view(torch.uint8).reshape(-1))
    res_h = torch.empty(nout + 2 * nkv, dtype=torch.uint8).pin_memory()
    in_d = torch.empty(nx + npos, dtype=torch.uint8, device=dev)
    res_d = torch.empty(nout + 2 * nkv, dtype=torch.uint8, device=dev)
    x_e = in_d[:nx].view(torch.float16).view(T, s.hidden)
    pos_e = in_d[nx:].view(torch.int64)
    out_e = res_d[:nout].view(torch.float16).view(T, s.hidden)
    kn_e = res_d[nout:nout + nkv].view(torch.float16).view(kn.shape)
    vn_e = res_d[nout + nkv:].view(torch.float16).view(vn.shape)

    def e2e_step():
        in_d.copy_(in_h, non_blocking=True)
        block.prefill(wts, x_e, pos_e, kc, vc, out_e, wsb, kn_e, vn_e, stream=stream)
        res_h.copy_(res_d, non_blocking=True)

    for _ in range(W):
        flush.zero_()
        e2e_step()
    torch.cuda.synchronize()
    e2e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    barrier(ws)
    for i in range(K):
        flush.zero_()
        e2e_evs[i][0].record(stream)
        e2e_step()
        e2e_evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e2e_evs), ws)
    h2d = in_h.numel()
    d2h = res_h.numel()

    # per-kernel durations (events around each kernel; separate pass)
    block.timing(True)
    for i in range(K):
        flush.zero_()
        prefill_step()
        block.timing_collect(stream)
    block.timing(False)
    table = block.timing_table()
    launches_per_step = sum(n for _, n in table.values()) // K
    gemm_flops, attn_flops = prefill_flops(s, T)
    kernels = {}
    for name, (ms, n) in table.items():
        kernels[name] = {"avg_us": 1e3 * ms / n, "launches_per_step": n // K,
                         "share": ms / sum(v[0] for v in table.values())}
    dom = max(table, key=lambda k: table[k][0])
    if dom in gemm_flops or dom == "attn_prefill":
        work = gemm_flops[dom] if dom in gemm_flops else attn_flops
        per_launch = table[dom][0] / table[dom][1] * (table[dom][1] // K)   # ms per step
        achieved = work / (per_launch * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": NCU_TRAFFIC.get(dom),
                "traffic_unit": "bytes per launch (ncu, cold L2)",
                "peak_source": peaks["source"] + " bf16 dense burst (fp16 runs at the bf16 rate)"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": None, "traffic": None}
    # the split-K reduction belongs to the down projection's time
    gemm_ms = sum(table[k][0] for k in list(gemm_flops) + ["splitk_reduce"] if k in table) / K
    gemm_frac = sum(gemm_flops.values()) / (gemm_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]

    result = {
        "metric": METRIC, "value": ws * T * K / (total_ms * 1e-3), "unit": UNIT,
        "n_gpus": ws, "steps": K, "warmup": W, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations)",
        "config": {"workload": "qwen2-1.5B-shaped decoder layer, prefill [1,1024], pos 0..1023",
                   "hidden": 1536, "heads": 12, "kv_heads": 2, "head_dim": 128,
                   "intermediate": 8960, "qkv_bias": True, "layers": 1, "seq_len": T,
                   "l2": "flushed (256 MB write) before every timed step",
                   "parallelism": f"replicas x{ws}"},
        "e2e": {"value": ws * T * K / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * K,
        "roofline": roof,
        "prefill_gemm_frac_of_tensor_peak": gemm_frac,
        "kernels": kernels,
    }

    # ---------------- decode, prefill_kv, hidden 4096 ----------------
    if not args.no_decode and args.only != "prefill":
        result["decode"] = bench_decode(args, s, dev, stream, peaks, ws)
        result["lm_head"] = bench_lm_head(args, s, dev, stream, peaks, ws)
        result["decode_batch"] = bench_decode_batch(args, s, dev, stream, peaks, ws)
        result["decode_quant"] = bench_decode_quant(args, s, dev, stream, peaks, ws)
        result["prefill_kv_28"] = bench_prefill_kv_stack(args, s, dev, stream, peaks, ws)
        _STACK_W.clear()
        torch.cuda.empty_cache()
        result["gqa4096"] = bench_gqa4096(args, s, dev, stream, peaks, ws)
    result["clocks"] = clocks.stop()
    return result


def bench_model_step(args, s, dev, stream, peaks, ws, st, L):
    import torch
    import synth
    from decode_qwen2_block_gb300.model import Model
    K, W = args.steps, args.warmup
    V = synth.QWEN2_VOCAB
    hw = {k: torch.from_numpy(v).to(dev) for k, v in synth.head_weights(V, s.hidden, seed=0).items()}
    model = Model(s, None, hw, 0, stack=st)
    toks = torch.from_numpy(synth.token_ids(V, W + K + 1, seed=1)).to(dev)
    graphs = []
    for i in range(W + K):
        pos = torch.tensor([L + i], dtype=torch.int64, device=dev)
        graphs.append((model.capture_step(toks[i:i + 1], pos, L + i, toks[i + 1:i + 2],
                                          key=("model", L + i)), pos))
    for i in range(W):
        graphs[i][0].replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    barrier(ws)
    for i in range(K):
        evs[i][0].record(stream)
        graphs[W + i][0].replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    st.block.check()
    ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs), ws) / K
    nbytes, _ = decode_bytes(s, L + W + K // 2, s.n_layers)
    nbytes += V * s.hidden * 2 + s.hidden * 2   # the LM head + one embedding row
    achieved = nbytes / (ms * 1e-3) / 1e9
    del graphs
    return {"ctx": L, "us_per_token": ms * 1e3, "tok_s": ws * 1e3 / ms, "bytes_per_token": nbytes,
            "achieved_gbs": achieved, "frac_of_hbm_peak": achieved / peaks["hbm_gbs"],
            "workload": "token embedding + 28 blocks + final RMSNorm + 151936x1536 LM head + "
                        "greedy argmax; the token feeds the next step on the device"}


def bench_lm_head(args, s, dev, stream, peaks, ws):
    """Final RMSNorm + LM head + greedy argmax of one decode step (151936 x
    1536 fp16 head, 467 MB: larger than L2, so no flush is needed), and the
    embedding gather of the step's token."""
    import torch
    import synth
    import decode_qwen2_block_gb300 as blk
    K, W = max(args.steps, 10), args.warmup
    V = synth.QWEN2_VOCAB
    hw = synth.head_weights(V, s.hidden, seed=0)
    head = torch.from_numpy(hw["lm_head"]).to(dev)
    table = torch.from_numpy(hw["embed"]).to(dev)
    g = torch.from_numpy(hw["norm_g"]).to(dev)
    block = blk.Block(s, 64)
    wsb = torch.empty(block.lm_head_workspace_bytes(), dtype=torch.uint8, device=dev)
    x = torch.from_numpy(synth.hidden_input(s, 1, seed=0, stream_offset=99)).to(dev)
    tok = torch.empty(1, dtype=torch.int64, device=dev)
    xe = torch.empty((1, s.hidden), dtype=torch.float16, device=dev)
    ids = torch.from_numpy(synth.token_ids(V, 1, seed=0)).to(dev)

    def step():
        block.embed(table, ids, xe, stream=stream)
        block.lm_head(x, g, head, tok, wsb, stream=stream)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    barrier(ws)
    for i in range(K):
        evs[i][0].record(stream)
        block.lm_head(x, g, head, tok, wsb, stream=stream)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    block.check()
    ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs), ws) / K
    nbytes = V * s.hidden * 2 + s.hidden * 2 * 2 + 8
    achieved = nbytes / (ms * 1e-3) / 1e9
    block.timing(True)
    for _ in range(3):
        step()
        block.timing_collect(stream)
    block.timing(False)
    table_t = block.timing_table()
    return {"workload": f"final RMSNorm + LM head {V}x{s.hidden} fp16 + greedy argmax, 1 row "
                        "(one decode step); embedding gather of the step's token",
            "us_per_call": ms * 1e3, "achieved_gbs": achieved,
            "frac_of_hbm_peak": achieved / peaks["hbm_gbs"],
            "roofline_us": nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6,
            "traffic": NCU_TRAFFIC.get("lm_head"),
            "kernels": {k: {"avg_us": 1e3 * v[0] / v[1]} for k, v in table_t.items()}}


def bench_decode_batch(args, s, dev, stream, peaks, ws):
    """Batched decode: B sequences, one new token each, through the 28-layer
    stack (one blk_decode_batch_stack call), one CUDA graph per step.  Every
    sequence holds ctx history slots (each layer's seeded history, the same
    for every sequence of the layer); the step appends slot ctx + i.  Bytes
    per step: every layer's weights once + each sequence's K/V slots read;
    the weights (2.6 GB) exceed L2, so no flush is needed."""
    import torch
    import synth
    from decode_qwen2_block_gb300.stack import BatchStack
    K, W = args.steps, args.warmup
    Bs = [int(b) for b in args.decode_batch.split(",") if b]
    L0 = args.decode_batch_ctx
    n = s.n_layers
    C = L0 + W + K + 8
    Bmax = max(Bs)
    H = s.hidden
    wd = stack_weights(s, dev)
    caches = []
    for l in range(n):
        k, v = synth.kv_history(s, C, L0, layer=l, seed=0)
        kc = torch.from_numpy(k).to(dev).unsqueeze(0).repeat(Bmax, 1, 1, 1).contiguous()
        vc = torch.from_numpy(v).to(dev).unsqueeze(0).repeat(Bmax, 1, 1, 1).contiguous()
        caches.append((kc, vc))
    st = BatchStack(s, wd, C, Bmax, caches=caches, device=dev)
    block = st.block
    x = torch.from_numpy(synth.hidden_input(s, Bmax, seed=0, stream_offset=5)).to(dev)
    y = torch.empty((Bmax, H), dtype=torch.float16, device=dev)
    maxlen = L0 + W + K

    def step(B, lens):
        st.step(x[:B], lens, lens, maxlen, y[:B], stream=stream)

    out = {}
    for B in Bs:
        lens = [torch.full((B,), L0 + i, dtype=torch.int64, device=dev) for i in range(W + K)]
        graphs = []
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        for i in range(W + K):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    st.step(x[:B], lens[i], lens[i], maxlen, y[:B], stream=side)
            graphs.append(g)
        torch.cuda.current_stream().wait_stream(side)
        for i in range(W):
            graphs[i].replay()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        barrier(ws)
        for i in range(K):
            evs[i][0].record(stream)
            graphs[W + i].replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        block.check()
        ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs), ws) / K
        _, wbytes = decode_bytes(s, 0, n)
        kv = n * 2 * s.n_kv_heads * s.head_dim * 2 * (L0 + W + K // 2 + 1)
        nbytes = wbytes + B * kv + n * B * H * 2 * 2
        achieved = nbytes / (ms * 1e-3) / 1e9
        row = {"us_per_step": ms * 1e3, "tok_s": ws * B * 1e3 / ms, "bytes_per_step": nbytes,
               "achieved_gbs": achieved, "frac_of_hbm_peak": achieved / peaks["hbm_gbs"],
               "roofline_us": nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6}
        # per-kernel durations (eager, events per kernel), two steps
        table = kernel_table(block, lambda: step(B, lens[W]), stream)
        tot = sum(v[0] for v in table.values())
        row["kernel_share"] = {k: t / tot for k, (t, c) in table.items()}
        row["launches_per_step"] = sum(c for _, c in table.values())
        out[str(B)] = row
        del graphs
    out["ctx"] = L0
    out["workload"] = (f"qwen2-1.5B-shaped 28-layer stack, B sequences x 1 new token, "
                       f"{L0} history slots each, one CUDA graph per step")
    return out


_STACK_W = {}


def stack_weights(s, dev):
    """Device copies of every layer's seeded weights of shape s (from synth,
    the generator the tests use), made once and shared by the legs."""
    import torch
    import synth
    if s not in _STACK_W:
        _STACK_W[s] = [{k: torch.from_numpy(v).to(dev)
                        for k, v in synth.block_weights(s, layer=l, seed=0).items()}
                       for l in range(s.n_layers)]
    return _STACK_W[s]


def device_weights(s, layer: int, seed: int, dev):
    """One layer's random-init weights drawn on the device by torch's seeded
    generator: W ~ N(0, 0.02) rounded to fp16, gains 1, biases ~ N(0, 0.02).
    The same distribution as synth.block_weights (not the same bits); used
    where the host generator would take minutes (32 layers of hidden 4096)."""
    import torch
    import synth
    g = torch.Generator(device=dev)
    g.manual_seed(1000003 * seed + layer)
    w = {}
    for name, shp in synth.weight_shapes(s).items():
        if name in ("ln1_g", "ln2_g"):
            w[name] = torch.ones(shp, dtype=torch.float16, device=dev)
        else:
            w[name] = (torch.randn(shp, generator=g, device=dev) * 0.02).half()
    return w


def timed(fn, K, W, ws, stream):
    """W untimed calls of fn(i), then K calls fn(W + i) each bracketed by CUDA
    events on `stream`, with a barrier and a synchronize on both sides.
    Returns (max over ranks of the summed ms, per-call ms on this rank)."""
    import torch
    for i in range(W):
        fn(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    barrier(ws)
    torch.cuda.synchronize()
    for i in range(K):
        evs[i][0].record(stream)
        fn(W + i)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    per = [a.elapsed_time(b) for a, b in evs]
    return reduce_max(sum(per), ws), per


def kernel_table(block, run, stream, reps=2):
    """Per-kernel CUDA-event durations of `reps` eager calls of run(): {name:
    (ms per call, launches per call)}, the handle's earlier totals removed."""
    before = block.timing_table()
    block.timing(True)
    for _ in range(reps):
        run()
        block.timing_collect(stream)
    block.timing(False)
    out = {}
    for k, (t, c) in block.timing_table().items():
        t0, c0 = before.get(k, (0.0, 0))
        if c > c0:
            out[k] = ((t - t0) / reps, (c - c0) // reps)
    return out


def bench_decode(args, s, dev, stream, peaks, ws):
    """The 28-layer decode at each context length: DECODE_STEPS (or --steps,
    if more) consecutive steps timed, each appending its K/V in place."""
    import torch
    import synth
    from decode_qwen2_block_gb300.stack import LayerStack
    K, W = max(args.steps, DECODE_STEPS), args.warmup
    ctxs = [int(c) for c in args.decode_ctx.split(",") if c]
    n = s.n_layers
    C = max(ctxs) + W + K + 8
    Lmax = max(ctxs)
    wl = stack_weights(s, dev)
    caches = []
    for l in range(n):
        k, v = synth.kv_history(s, C, Lmax, layer=l, seed=0)
        caches.append((torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)))
    st = LayerStack(s, wl, C, 1, caches=caches, chain=True)
    xs_np = [synth.hidden_input(s, 1, seed=0, stream_offset=i + 1) for i in range(W + K)]
    xs = [torch.from_numpy(a).to(dev) for a in xs_np]
    out = {}
    for L in ctxs:
        poss = [torch.tensor([L + i], dtype=torch.int64, device=dev) for i in range(W + K)]
        graphs = [st.capture("decode", xs[i], poss[i], L + i, key=("decode", L, i))[0]
                  for i in range(W + K)]
        total, _ = timed(lambda i: graphs[i].replay(), K, W, ws, stream)
        st.block.check()
        ms = total / K
        nbytes, wbytes = decode_bytes(s, L + W + K // 2, n)
        achieved = nbytes / (ms * 1e-3) / 1e9
        out[str(L)] = {"us_per_step": ms * 1e3, "tok_s": ws * 1e3 / ms,
                       "bytes_per_step": nbytes, "achieved_gbs": achieved,
                       "frac_of_hbm_peak": achieved / peaks["hbm_gbs"],
                       "roofline_us": nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6,
                       "traffic": NCU_TRAFFIC.get(("decode_persistent", L))}
        del graphs
        st.graphs.clear()
    # end to end at the first context through the public API, eager: the
    # step's hidden row and position go host (pinned) -> device, the 28-layer
    # step runs (blk_decode_stack), the output row comes back to the host
    # (the hidden row and the position in one pinned buffer: one copy in)
    L = ctxs[0]
    nx = s.hidden * 2
    in_h = []
    for i in range(W + K):
        b = torch.empty(nx + 8, dtype=torch.uint8).pin_memory()
        b[:nx].copy_(torch.from_numpy(xs_np[i]).view(torch.uint8).reshape(-1))
        b[nx:].copy_(torch.tensor([L + i], dtype=torch.int64).view(torch.uint8))
        in_h.append(b)
    in_d = torch.empty(nx + 8, dtype=torch.uint8, device=dev)
    x_d = in_d[:nx].view(torch.float16).view(1, s.hidden)
    pos_d = in_d[nx:].view(torch.int64)
    out_d = torch.empty((1, s.hidden), dtype=torch.float16, device=dev)
    out_h = torch.empty((1, s.hidden), dtype=torch.float16).pin_memory()

    def e2e(i):
        in_d.copy_(in_h[i], non_blocking=True)
        st.decode_step(x_d, pos_d, L + i, out=out_d, stream=stream)
        out_h.copy_(out_d, non_blocking=True)

    total, _ = timed(e2e, K, W, ws, stream)
    st.block.check()
    ms = total / K
    out["e2e"] = {"ctx": L, "value": ws * 1e3 / ms, "unit": "tok/s", "us_per_step": ms * 1e3,
                  "h2d_bytes_per_step": in_h[0].numel(),
                  "d2h_bytes_per_step": out_h.numel() * 2,
                  "path": "blk_decode_stack through LayerStack.decode_step, eager (no graph)"}
    # the whole model per generated token at the first context: embedding +
    # the 28 blocks + final RMSNorm + LM head + greedy argmax, one graph per step
    out["model_per_token"] = bench_model_step(args, s, dev, stream, peaks, ws, st, ctxs[0])
    # per-kernel durations at the largest context (eager, events per kernel)
    L = ctxs[-1]
    pos = torch.tensor([L], dtype=torch.int64, device=dev)
    table = kernel_table(st.block, lambda: st.run("decode", xs[0], pos, L), stream)
    tot = sum(v[0] for v in table.values())
    out["kernels_at_ctx"] = L
    out["kernels"] = {k: {"avg_us": 1e3 * ms / cnt, "share": ms / tot}
                      for k, (ms, cnt) in table.items()}
    out["launches_per_step"] = sum(c for _, c in table.values())
    out["steps_per_ctx"] = K
    out["workload"] = (f"qwen2-1.5B-shaped 28-layer stack, batch-1 decode, {K} consecutive "
                       f"steps per context length (KV appended in place), one CUDA graph per step")
    return out


def quant_bytes(s, fmt: str, group: int, L: int, n_layers: int):
    """HBM bytes of one decode step with quantized projections: codes (1
    byte per weight for INT8, half a byte for int4), fp16 scales (one per
    row, or per row and group), int4 zero points (one byte per row and
    group), the fp16 gains and biases, and the K/V slots read."""
    H, Hq, Hkv, D, I = s.hidden, s.n_heads, s.n_kv_heads, s.head_dim, s.intermediate
    mats = [((Hq + 2 * Hkv) * D, H), (H, Hq * D), (2 * I, H), (H, I)]   # (rows, K)
    w = 0
    for rows, K in mats:
        if fmt == "i8":
            w += rows * K + 2 * rows
        else:
            w += rows * K // 2 + 3 * rows * (K // group)
    w += 2 * 2 * H + (2 * (Hq + 2 * Hkv) * D if s.has_qkv_bias else 0)
    kv = 2 * Hkv * D * 2 * (L + 1)
    return n_layers * (w + kv)


def device_qweights(s, fmt: str, group: int, layer: int, seed: int, dev):
    """One layer's quantized matrices drawn on the device by torch's seeded
    generator, in the layouts of include/blk.h (codes, scales near
    0.02 / spread of the codes, int4 zero points near 7.5): the same recipe
    as synth.quant_weights, not the same bits."""
    import torch
    import synth
    g = torch.Generator(device=dev)
    g.manual_seed(7919 * seed + layer)
    out = {}
    shapes = synth.weight_shapes(s)
    for name in synth.QUANT_MATRICES:
        N, K = shapes[name]
        if fmt == "i8":
            q = torch.randint(-127, 128, (N, K), generator=g, device=dev, dtype=torch.int8)
            sc = (0.02 / 42 * (1 + 0.1 * torch.randn(N, generator=g, device=dev))).half()
            out[name] = {"q": q, "scale": sc}
        else:
            q = torch.randint(0, 256, (N, K // 2), generator=g, device=dev, dtype=torch.uint8)
            sc = (0.02 / 3.5 * (1 + 0.1 * torch.randn(N, K // group, generator=g,
                                                      device=dev))).half()
            z = torch.randint(6, 10, (N, K // group), generator=g, device=dev, dtype=torch.uint8)
            out[name] = {"q": q, "scale": sc, "zero": z}
    return out


def bench_decode_quant(args, s, dev, stream, peaks, ws):
    """Batch-1 decode through the 28-layer 1.5B stack with weight-only
    quantized projections (INT8 per row; int4 in groups of 128), one CUDA
    graph per step, at the first decode context; bytes per step are the
    codes, scales, zero points, gains, biases and K/V read."""
    import torch
    import synth
    import decode_qwen2_block_gb300 as blk
    from decode_qwen2_block_gb300.stack import QuantDecodeStack
    K, W = args.steps, args.warmup
    L = int(args.decode_ctx.split(",")[0])
    n = s.n_layers
    C = L + W + K + 8
    caches = []
    for l in range(n):
        k, v = synth.kv_history(s, C, L, layer=l, seed=0)
        caches.append((torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)))
    wl = stack_weights(s, dev)
    xs = [torch.from_numpy(synth.hidden_input(s, 1, seed=0, stream_offset=i + 1)).to(dev)
          for i in range(W + K)]
    out = {}
    for fmt, group in (("i8", 0), ("u4", 128)):
        qd = [device_qweights(s, fmt, group, l, 0, dev) for l in range(n)]
        code = blk.BLK_WFMT_I8 if fmt == "i8" else blk.BLK_WFMT_U4
        qws = [blk.Block.qweights(code, group, wl[l], qd[l]) for l in range(n)]
        st = QuantDecodeStack(s, qws, C, caches=caches)
        poss = [torch.tensor([L + i], dtype=torch.int64, device=dev) for i in range(W + K)]
        graphs = [st.capture(xs[i], poss[i], L + i)[0] for i in range(W + K)]
        total, _ = timed(lambda i: graphs[i].replay(), K, W, ws, stream)
        st.block.check()
        ms = total / K
        nbytes = quant_bytes(s, fmt, group, L + W + K // 2, n)
        achieved = nbytes / (ms * 1e-3) / 1e9
        out[fmt] = {"us_per_step": ms * 1e3, "tok_s": ws * 1e3 / ms, "bytes_per_step": nbytes,
                    "achieved_gbs": achieved, "frac_of_hbm_peak": achieved / peaks["hbm_gbs"],
                    "roofline_us": nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6,
                    "group": group if fmt == "u4" else None}
        del graphs, st, qd, qws
        torch.cuda.empty_cache()
    out["ctx"] = L
    out["workload"] = ("qwen2-1.5B-shaped 28-layer stack, batch-1 decode, weight-only INT8 "
                       "(per-row scale) and int4 (groups of 128, scale + zero point), "
                       "weights drawn on the device")
    return out


def bench_decode_layer(args, s, dev, stream, peaks, ws):
    """One 1.5B-shaped layer of decode (blk_decode) at ctx --decode-ctx[0]:
    a small case for ncu captures of the decode kernel (one launch = one
    layer: 93.6 MB of weights + the K/V slots)."""
    import torch
    import synth
    from decode_qwen2_block_gb300.stack import LayerStack
    K, W = args.steps, args.warmup
    L = int(args.decode_ctx.split(",")[0])
    w = synth.block_weights(s, layer=0, seed=0)
    wl = [{k: torch.from_numpy(v).to(dev) for k, v in w.items()}]
    k, v = synth.kv_history(s, L + W + K + 8, L, layer=0, seed=0)
    st = LayerStack(s, wl, L + W + K + 8, 1, caches=[(torch.from_numpy(k).to(dev),
                                                      torch.from_numpy(v).to(dev))])
    x = torch.from_numpy(synth.hidden_input(s, 1, seed=0, stream_offset=1)).to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    poss = [torch.tensor([L + i], dtype=torch.int64, device=dev) for i in range(W + K)]

    def step(i):
        flush.zero_()
        st.decode_step(x, poss[i], L + i, stream=stream)

    total, per = timed(step, K, W, ws, stream)
    st.block.check()
    nbytes, _ = decode_bytes(s, L + W + K // 2, 1)
    return {"ctx": L, "us_per_launch_incl_flush": total / K * 1e3, "bytes_per_launch": nbytes,
            "workload": f"one 1.5B-shaped layer, decode at ctx {L}, L2 flushed before each call"}


def bench_decode_batch_layer(args, s, dev, stream, peaks, ws):
    """One 1.5B-shaped layer of batched decode (blk_decode_batch) for B =
    the largest --decode-batch sequences at ctx --decode-batch-ctx: a small
    case for ncu captures of the batched kernels (94 MB of weights, B x the
    K/V slots)."""
    import torch
    import synth
    K, W = args.steps, args.warmup
    B = max(int(b) for b in args.decode_batch.split(",") if b)
    L = args.decode_batch_ctx
    C = L + W + K + 8
    w = synth.block_weights(s, layer=0, seed=0)
    wd = {k: torch.from_numpy(v).to(dev) for k, v in w.items()}
    from decode_qwen2_block_gb300 import Block
    block = Block(s, C)
    wts = Block.weights(wd)
    k, v = synth.kv_history(s, C, L, layer=0, seed=0)
    kc = torch.from_numpy(k).to(dev).unsqueeze(0).repeat(B, 1, 1, 1).contiguous()
    vc = torch.from_numpy(v).to(dev).unsqueeze(0).repeat(B, 1, 1, 1).contiguous()
    x = torch.from_numpy(synth.hidden_input(s, B, seed=0, stream_offset=5)).to(dev)
    out = torch.empty_like(x)
    wsb = torch.empty(block.decode_batch_workspace_bytes(B), dtype=torch.uint8, device=dev)
    lens = [torch.full((B,), L + i, dtype=torch.int64, device=dev) for i in range(W + K)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(i):
        flush.zero_()
        block.decode_batch(wts, x, lens[i], lens[i], L + W + K, kc, vc, out, wsb, stream=stream)

    total, _ = timed(step, K, W, ws, stream)
    block.check()
    return {"B": B, "ctx": L, "us_per_call_incl_flush": total / K * 1e3,
            "workload": f"one 1.5B-shaped layer, batched decode of {B} sequences at ctx {L}, "
                        f"L2 flushed before each call"}


def bench_prefill_kv_stack(args, s, dev, stream, peaks, ws):
    """prefill_kv through the 28-layer 1.5B stack: 512 new tokens at
    positions 3584..4095 on 3584 seeded history slots per layer (the
    TopOp paper's Listing 2 block with history K/V, per layer).  One call =
    one blk_prefill_stack (each layer's last kernel also normalises the next
    layer's input).  GEMM flops are 1,341.6 GFLOP per
    call and attention 338.3 GFLOP; their kernel times (events around each
    kernel, separate pass) are reported apart."""
    import torch
    import synth
    from decode_qwen2_block_gb300.stack import LayerStack
    K, W = args.steps, args.warmup
    n, L0, T = s.n_layers, PKV_HIST, PKV_T
    C = L0 + T
    wl = stack_weights(s, dev)
    caches = []
    for l in range(n):
        k, v = synth.kv_history(s, C, L0, layer=l, seed=0)
        caches.append((torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)))
    st = LayerStack(s, wl, C, T, caches=caches, chain=True)
    x = torch.from_numpy(synth.hidden_input(s, T, seed=0, stream_offset=7)).to(dev)
    pos = torch.from_numpy(synth.positions(L0, T)).to(dev)

    def step(i=0):
        st.run("prefill_kv", x, pos, L0, stream=stream)

    total, _ = timed(step, K, W, ws, stream)
    st.block.check()
    ms = total / K
    gemm, attn = prefill_flops(s, T, L0)
    gemm_flops, attn_flops = n * sum(gemm.values()), n * attn
    table = kernel_table(st.block, step, stream)
    tot = sum(v[0] for v in table.values())
    gemm_ms = sum(table[k][0] for k in list(gemm) + ["splitk_reduce"] if k in table)
    attn_ms = sum(table[k][0] for k in ("attn_prefill", "attn_merge") if k in table)
    peak = peaks["bf16_tflops"]
    del st, caches
    return {"workload": "qwen2-1.5B-shaped 28-layer stack, prefill_kv of 512 tokens at positions "
                        "3584..4095 on 3584 history slots per layer",
            "ms_per_call": ms, "tok_s": ws * T / (ms * 1e-3),
            "gemm_gflop": gemm_flops / 1e9, "attn_gflop": attn_flops / 1e9,
            "gemm_us": gemm_ms * 1e3, "gemm_tflops": gemm_flops / (gemm_ms * 1e-3) / 1e12,
            "gemm_frac_of_tensor_peak": gemm_flops / (gemm_ms * 1e-3) / 1e12 / peak,
            "gemm_target_us": gemm_flops / (0.6 * peak * 1e12) * 1e6,
            "attn_us": attn_ms * 1e3, "attn_tflops": attn_flops / (attn_ms * 1e-3) / 1e12,
            "attn_frac_of_tensor_peak": attn_flops / (attn_ms * 1e-3) / 1e12 / peak,
            "attn_share_of_kernel_time": attn_ms / tot,
            "whole_call_frac_of_tensor_peak": (gemm_flops + attn_flops) / (ms * 1e-3) / 1e12 / peak,
            "kernels": {k: {"us_per_call": 1e3 * t, "launches": c, "share": t / tot}
                        for k, (t, c) in table.items()}}


def bench_gqa4096(args, s15, dev, stream, peaks, ws):
    """The TopOp paper's Figure 2 example shape (32 layers, hidden 4096, 32 q
    heads, 2 kv heads, head_dim 128, intermediate 11008, no bias): one
    32-layer prefill of 100 tokens (positions 0..99), then 256 decode steps
    at positions 100..355 appending to the same caches.  Both are bound by
    the weight bytes (10.94 GB per pass).  Weights are drawn on the device
    (device_weights); inputs from synth."""
    import torch
    import synth
    from decode_qwen2_block_gb300.stack import LayerStack
    s = synth.GQA_4096
    K, W = args.steps, args.warmup
    n, T, ND = s.n_layers, G4_PREFILL, G4_DECODES
    C = T + ND + 8
    wl = [device_weights(s, l, 0, dev) for l in range(n)]
    st = LayerStack(s, wl, C, T, chain=True)
    x = torch.from_numpy(synth.hidden_input(s, T, seed=0)).to(dev)
    pos = torch.from_numpy(synth.positions(0, T)).to(dev)

    def prefill(i=0):
        st.run("prefill", x, pos, 0, stream=stream)

    total, _ = timed(prefill, K, W, ws, stream)
    st.block.check()
    pre_ms = total / K
    _, wbytes = decode_bytes(s, 0, n)
    pre_bytes = wbytes + n * 2 * s.n_kv_heads * s.head_dim * 2 * T
    pre_gbs = pre_bytes / (pre_ms * 1e-3) / 1e9
    table = kernel_table(st.block, prefill, stream)
    tot = sum(v[0] for v in table.values())
    # the decode steps continue from the prefill's caches (slots 0..99)
    xd = torch.from_numpy(synth.hidden_input(s, ND, seed=0, stream_offset=3)).to(dev)
    poss = torch.arange(T, T + ND, dtype=torch.int64, device=dev)
    outs = torch.empty((2, s.hidden), dtype=torch.float16, device=dev)

    def dec(i):
        st.decode_step(xd[i:i + 1], poss[i:i + 1], T + i, out=outs[i % 2:i % 2 + 1], stream=stream)

    # warm-up: the first decode steps, then every one of the 256 steps timed
    total, per = timed(lambda i: dec(i - W if i >= W else i), ND, W, ws, stream)
    st.block.check()
    dec_ms = total / ND
    kv_avg = n * 2 * s.n_kv_heads * s.head_dim * 2 * (T + ND / 2 + 0.5)
    dec_bytes = wbytes + kv_avg
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    del st, wl
    torch.cuda.empty_cache()
    hbm = peaks["hbm_gbs"]
    return {"workload": "hidden 4096, 32 q / 2 kv heads, head_dim 128, intermediate 11008, 32 "
                        "layers: prefill of 100 tokens, then 256 decode steps (positions 100..355)",
            "prefill_us": pre_ms * 1e3, "prefill_tok_s": ws * T / (pre_ms * 1e-3),
            "prefill_bytes": pre_bytes, "prefill_gbs": pre_gbs,
            "prefill_frac_of_hbm_peak": pre_gbs / hbm,
            "prefill_roofline_us": pre_bytes / (hbm * 1e9) * 1e6,
            "prefill_kernels": {k: {"us_per_call": 1e3 * t, "share": t / tot}
                                for k, (t, c) in table.items()},
            "decode_us_per_step": dec_ms * 1e3, "decode_tok_s": ws * 1e3 / dec_ms,
            "decode_us_first_last": [per[0] * 1e3, per[-1] * 1e3],
            "decode_bytes_per_step": dec_bytes, "decode_gbs": dec_gbs,
            "decode_frac_of_hbm_peak": dec_gbs / hbm,
            "decode_roofline_us": dec_bytes / (hbm * 1e9) * 1e6,
            "weights": "drawn on the device by a seeded generator (same distribution as the "
                       "host generator); inputs from the host generator"}


# ------------------------------------------------------------------ main

def compact(v, digits=4):
    """Rounds every float to `digits` significant digits (keeps the line short)."""
    if isinstance(v, float):
        return float(f"{v:.{digits}g}")
    if isinstance(v, dict):
        return {k: compact(x, digits) for k, x in v.items()}
    if isinstance(v, (list, tuple)):
        return [compact(x, digits) for x in v]
    return v


def summary(r):
    """The main figures in a few hundred bytes, placed last in the line."""
    out = {"prefill_tok_s": r.get("value"), "prefill_ms": r.get("ms_per_step"),
           "prefill_gemm_frac": r.get("prefill_gemm_frac_of_tensor_peak"),
           "roofline_frac": (r.get("roofline") or {}).get("frac")}
    dec = r.get("decode")
    if dec:
        out["decode_us_frac"] = {c: [dec[c]["us_per_step"], dec[c]["frac_of_hbm_peak"]]
                                 for c in dec if c.isdigit()}
        if "e2e" in dec:
            out["decode_e2e_tok_s"] = dec["e2e"]["value"]
        if "model_per_token" in dec:
            out["model_us_per_token"] = dec["model_per_token"]["us_per_token"]
    pkv = r.get("prefill_kv_28")
    if pkv:
        out["cfg4_prefill_kv"] = {"ms": pkv["ms_per_call"], "tok_s": pkv["tok_s"],
                                  "gemm_us": pkv["gemm_us"],
                                  "gemm_frac": pkv["gemm_frac_of_tensor_peak"],
                                  "attn_us": pkv["attn_us"],
                                  "attn_frac": pkv["attn_frac_of_tensor_peak"],
                                  "attn_share": pkv["attn_share_of_kernel_time"]}
    g4 = r.get("gqa4096")
    if g4:
        out["cfg5_gqa4096"] = {"prefill_us": g4["prefill_us"],
                               "prefill_frac": g4["prefill_frac_of_hbm_peak"],
                               "decode_us": g4["decode_us_per_step"],
                               "decode_frac": g4["decode_frac_of_hbm_peak"]}
    dq = r.get("decode_quant")
    if dq:
        out["decode_quant_us_frac"] = {f: [dq[f]["us_per_step"], dq[f]["frac_of_hbm_peak"]]
                                       for f in ("i8", "u4") if f in dq}
    db = r.get("decode_batch")
    if db:
        out["decode_batch_us_frac"] = {b: [db[b]["us_per_step"], db[b]["frac_of_hbm_peak"]]
                                       for b in db if b.isdigit()}
    if "cpu_baseline" in r:
        out["cpu_oracle_tok_s"] = r["cpu_baseline"]["value"]
    return out


def reference_arm(args, ws, rank):
    """The oracle, as it stands, on the host cores: each step is the bounded
    prefill sample that cpu_baseline also times; value is its tok/s
    extrapolated to the whole [1,1024] layer, ms_per_step the sample's own
    wall time."""
    if rank != 0:
        return
    per_step, times = [], []
    t_kv = None
    for i in range(args.warmup + args.steps):
        tok_s, secs, t_kv, desc = oracle_prefill_sample(ORACLE_SAMPLE_ROWS, rotate=i, t_kv=t_kv)
        if i >= args.warmup:
            per_step.append(tok_s)
            times.append(secs)
    v = statistics.mean(per_step)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": "qwen2-1.5B-shaped decoder layer, prefill [1,1024], pos 0..1023",
                       "sample": f"{ORACLE_SAMPLE_ROWS} of 1024 output rows per step, "
                                 "value extrapolated to 1024 rows"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": desc, "extrapolated": True,
                             "host_cores": os.cpu_count()},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(compact(line)))


def main():
    args = parse()
    ws, rank, local = dist_init(args)
    if args.impl == "reference":
        reference_arm(args, ws, rank)
        return
    result = bench_ours(args, ws, rank, local)
    if rank == 0 and not args.no_cpu and args.only is None:
        tok_s, secs, _, desc = oracle_prefill_sample(ORACLE_SAMPLE_ROWS)
        result["cpu_baseline"] = {"value": tok_s, "unit": UNIT, "cores": 1, "kind": "oracle",
                                  "sample": desc, "extrapolated": True,
                                  "host_cores": os.cpu_count(), "seconds": secs}
        if "decode" in result:
            us, secs_d, desc_d = oracle_decode_sample(1024, synth_layers())
            result["cpu_baseline_decode"] = {"value": us, "unit": "us/step", "cores": 1,
                                             "kind": "oracle", "sample": desc_d,
                                             "extrapolated": True, "seconds": secs_d}
    if rank == 0:
        if args.only is None:
            result["summary"] = summary(result)
        print(json.dumps(compact(result), separators=(",", ":")))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
