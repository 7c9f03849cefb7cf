"""Sliding-window attention (blk_set_window) on the GPU against the oracle
with the same window, in every phase and entry point: the query in slot p
attends slots [max(0, p - W + 1), p] (the reading of the "swa" layer
forward that the ds4.c study notes name without a window).  Slots before a
query's window hold NaN in the cache where the case allows it, so a read of
one would reach the output.  Tolerance: relative L2 <= 1e-2 and max abs
<= 5e-2 per tensor, the bound of every parity test."""
import numpy as np
import pytest
import torch

import decode_qwen2_block_gb300 as blk
import oracle
import synth
from gpu_harness import DevBlock, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _nan_before(kc, vc, lo):
    """Caches with slots [0, lo) replaced by NaN (host copies for the GPU)."""
    k, v = kc.copy(), vc.copy()
    if lo > 0:
        k[:, :lo] = np.float16(np.nan)
        v[:, :lo] = np.float16(np.nan)
    return k, v


def _check(db, s, phase, x, L, kc_np, vc_np, W, rows=None, nan_lo=0):
    """One call with window W on the GPU (caches with NaN below nan_lo) and
    the oracle on the clean caches."""
    T = x.shape[0]
    pos = synth.positions(L, T)
    kg, vg = _nan_before(kc_np, vc_np, nan_lo)
    kc, vc = to_dev(kg), to_dev(vg)
    out, kn, vn = db.run(phase, to_dev(x), to_dev(pos), L, kc, vc)
    torch.cuda.synchronize()
    db.block.check()
    o_ref, k_ref, v_ref = oracle.block_forward(s, db_w(db), x, pos, L, kc_np.copy(), vc_np.copy(),
                                               rows=rows, window=W)
    got = out.cpu().numpy()
    assert_close(got if rows is None else got[rows], o_ref, f"{phase} L={L} W={W} out")
    assert_close(kn.cpu().numpy(), k_ref, f"{phase} k_new")
    assert_close(vn.cpu().numpy(), v_ref, f"{phase} v_new")


_W_NP = {}


def db_w(db):
    return _W_NP[id(db)]


def _devblock(s, seed, C, max_T, W):
    w = synth.block_weights(s, seed=seed)
    db = DevBlock(s, w, C, max_T)
    db.block.set_window(W)
    _W_NP[id(db)] = w
    return db


@pytest.mark.parametrize("W", [1, 5, 13])
def test_tiny_window_all_phases(W):
    s, C = synth.TINY, 64
    db = _devblock(s, 11, C, 16, W)
    x = synth.hidden_input(s, 30, seed=11)
    kc, vc = synth.kv_history(s, C, 0)
    # prefill 16, then prefill_kv 4 on it, then decodes; the oracle's caches
    # follow the oracle's own K/V (bit-exact identities are not assumed)
    for phase, L, T in (("prefill", 0, 16), ("prefill_kv", 16, 4), ("decode", 20, 1),
                        ("decode", 21, 1)):
        _check(db, s, phase, x[L:L + T], L, kc, vc, W, nan_lo=max(0, L - W))
        oracle.block_forward(s, db_w(db), x[L:L + T], synth.positions(L, T), L, kc, vc, window=W)


def test_1p5b_prefill_window_across_row_blocks():
    """T = 1024 with W = 300: every 128-row block starts its tiles at its
    own window and masks the rows' lower edges; rows sampled across blocks."""
    s, T, W = synth.QWEN2_1P5B, 1024, 300
    db = _devblock(s, 12, T, T, W)
    x = synth.hidden_input(s, T, seed=12)
    kc, vc = synth.kv_history(s, T, 0)
    _check(db, s, "prefill", x, 0, kc, vc, W, rows=[0, 127, 128, 299, 300, 555, 1023])


def test_1p5b_prefill_kv_window_on_history():
    """512 new rows on 3584 history slots with W = 1000: the first row's
    window starts at slot 2585, so slots [0, 2585) are NaN."""
    s, L, T, W = synth.QWEN2_1P5B, 3584, 512, 1000
    db = _devblock(s, 13, L + T, T, W)
    x = synth.hidden_input(s, T, seed=13)
    kc, vc = synth.kv_history(s, L + T, L, seed=13)
    _check(db, s, "prefill_kv", x, L, kc, vc, W, rows=[0, 100, 511], nan_lo=L + 1 - W)


@pytest.mark.parametrize("W", [64, 700, 5000])
def test_1p5b_decode_window(W):
    s, L = synth.QWEN2_1P5B, 4000
    db = _devblock(s, 14, L + 8, 1, W)
    x = synth.hidden_input(s, 1, seed=14)
    kc, vc = synth.kv_history(s, L + 8, L, seed=14)
    _check(db, s, "decode", x, L, kc, vc, W, nan_lo=max(0, L + 1 - W))


def test_batched_decode_window_mixed_lengths():
    s, W = synth.QWEN2_1P5B, 300
    lens = [0, 100, 2000]
    C = max(lens) + 8
    w = synth.block_weights(s, seed=15)
    db = DevBlock(s, w, C, 1)
    db.block.set_window(W)
    hist = [synth.kv_history(s, C, L, layer=b, seed=15) for b, L in enumerate(lens)]
    kg = np.stack([_nan_before(k, v, max(0, L + 1 - W))[0] for (k, v), L in zip(hist, lens)])
    vg = np.stack([_nan_before(k, v, max(0, L + 1 - W))[1] for (k, v), L in zip(hist, lens)])
    x = synth.hidden_input(s, len(lens), seed=15)
    lens_d = to_dev(np.array(lens, dtype=np.int64))
    out = torch.empty((len(lens), s.hidden), dtype=torch.float16, device="cuda")
    ws = torch.empty(db.block.decode_batch_workspace_bytes(len(lens)), dtype=torch.uint8,
                     device="cuda")
    db.block.decode_batch(db.w, to_dev(x), lens_d, lens_d, max(lens), to_dev(kg), to_dev(vg),
                          out, ws)
    torch.cuda.synchronize()
    db.block.check()
    for b, L in enumerate(lens):
        k, v = hist[b][0].copy(), hist[b][1].copy()
        o_ref, _, _ = oracle.block_forward(s, w, x[b:b + 1], [L], L, k, v, window=W)
        assert_close(out[b:b + 1].cpu().numpy(), o_ref, f"batched seq {b} (L={L})")


def test_quantized_decode_window():
    """The quantized decode path shares the persistent kernel's attention."""
    s, L, W, group = synth.QWEN2_1P5B, 2000, 500, 128
    w = synth.block_weights(s, seed=16)
    q = synth.quant_weights(s, "u4", seed=16, group=group)
    m64 = {n: oracle.dequant_u4(m["q"], m["scale"], m["zero"], group) for n, m in q.items()}
    b = blk.Block(s, L + 8)
    b.set_window(W)
    wd = {k: to_dev(v) for k, v in w.items()}
    qd = {n: {k: to_dev(v) for k, v in m.items()} for n, m in q.items()}
    qw = blk.Block.qweights(blk.BLK_WFMT_U4, group, wd, qd)
    ws = torch.empty(b.qworkspace_bytes(1), dtype=torch.uint8, device="cuda")
    kc_np, vc_np = synth.kv_history(s, L + 8, L, seed=16)
    kg, vg = _nan_before(kc_np, vc_np, L + 1 - W)
    kc, vc = to_dev(kg), to_dev(vg)
    x = synth.hidden_input(s, 1, seed=16)
    out = torch.empty((1, s.hidden), dtype=torch.float16, device="cuda")
    b.run_q("decode", qw, to_dev(x), to_dev(synth.positions(L, 1)), L, kc, vc, out, ws)
    torch.cuda.synchronize()
    b.check()
    o_ref, _, _ = oracle.block_forward(s, w, x, synth.positions(L, 1), L, kc_np, vc_np,
                                       mats64=m64, window=W)
    assert_close(out.cpu().numpy(), o_ref, "quantized decode with a window")


def test_negative_window_is_refused():
    b = blk.Block(synth.TINY, 16)
    assert blk.blk_set_window(b.handle, -1) == blk.BLK_ERR_SHAPE
    assert blk.blk_set_window(b.handle, 0) == blk.BLK_OK
