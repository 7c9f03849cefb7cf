"""YaRN RoPE (blk_set_rope_yarn) on the GPU against the oracle with the same
parameters, in every phase and in batched decode.  The ds4.c study notes
(Part 4, "Trace 1: YaRN frequency scaling") give the ramp and the correction
dimension; the blend and the magnitude are the readings in include/blk.h,
which the oracle follows too.  Positions run past the original context, the
case YaRN exists for.  Tolerance: relative L2 <= 1e-2 and max abs <= 5e-2
per tensor, the bound of every parity test."""
import numpy as np
import pytest
import torch

import decode_qwen2_block_gb300 as blk
import oracle
import synth
from gpu_harness import DevBlock, assert_close, to_dev

pytestmark = pytest.mark.gpu

# 8x interpolation with the ramp, as on the notes' scaled layers
YARN = {"freq_scale": 0.125, "ext_factor": 1.0, "attn_factor": 1.0, "beta_fast": 32.0,
        "beta_slow": 1.0, "n_ctx_orig": 4096}


def _check(db, w, s, phase, x, L, kc_np, vc_np, yarn, rows=None, pos=None):
    T = x.shape[0]
    pos = synth.positions(L, T) if pos is None else pos
    kc, vc = to_dev(kc_np), to_dev(vc_np)
    out, kn, vn = db.run(phase, to_dev(x), to_dev(pos), L, kc, vc)
    torch.cuda.synchronize()
    db.block.check()
    o_ref, k_ref, v_ref = oracle.block_forward(s, w, x, pos, L, kc_np.copy(), vc_np.copy(),
                                               rows=rows, yarn=yarn)
    got = out.cpu().numpy()
    assert_close(got if rows is None else got[rows], o_ref, f"{phase} L={L} out")
    assert_close(kn.cpu().numpy(), k_ref, f"{phase} k_new")
    assert_close(vn.cpu().numpy(), v_ref, f"{phase} v_new")
    return out


def test_tiny_all_phases_with_yarn():
    """Original context 64 on the tiny shape (head_dim 64): the ramp runs
    from below pair 0 to pair 8, so pairs sit on, below and above it."""
    s, C = synth.TINY, 160
    y = dict(YARN, n_ctx_orig=64, freq_scale=0.25, attn_factor=1.1)
    w = synth.block_weights(s, seed=21)
    db = DevBlock(s, w, C, 64)
    db.block.set_rope_yarn(y)
    x = synth.hidden_input(s, 120, seed=21)
    kc, vc = synth.kv_history(s, C, 0)
    # the oracle's caches follow the oracle's own K/V
    for phase, L, T in (("prefill", 0, 64), ("prefill_kv", 64, 40), ("decode", 104, 1),
                        ("decode", 105, 1)):
        _check(db, w, s, phase, x[L:L + T], L, kc, vc, y)
        oracle.block_forward(s, w, x[L:L + T], synth.positions(L, T), L, kc, vc, yarn=y)


def test_1p5b_prefill_with_yarn_past_the_original_context():
    """T = 1024 new rows at positions 30000.. (beyond n_ctx_orig = 4096)."""
    s, T = synth.QWEN2_1P5B, 1024
    w = synth.block_weights(s, seed=22)
    db = DevBlock(s, w, 32768, T)
    db.block.set_rope_yarn(YARN)
    x = synth.hidden_input(s, T, seed=22)
    kc, vc = synth.kv_history(s, 32768, 0)
    pos = synth.positions(30000, T)
    _check(db, w, s, "prefill", x, 0, kc, vc, YARN, rows=[0, 511, 1023], pos=pos)


def test_1p5b_decode_with_yarn_on_a_long_history():
    s, L = synth.QWEN2_1P5B, 20000
    w = synth.block_weights(s, seed=23)
    db = DevBlock(s, w, L + 8, 1)
    y = dict(YARN, attn_factor=0.9)
    db.block.set_rope_yarn(y)
    x = synth.hidden_input(s, 1, seed=23)
    kc, vc = synth.kv_history(s, L + 8, L, seed=23)
    _check(db, w, s, "decode", x, L, kc, vc, y)


def test_batched_decode_with_yarn():
    s = synth.QWEN2_1P5B
    lens = [5, 3000, 9000]
    C = max(lens) + 8
    w = synth.block_weights(s, seed=24)
    db = DevBlock(s, w, C, 1)
    db.block.set_rope_yarn(YARN)
    hist = [synth.kv_history(s, C, L, layer=b, seed=24) for b, L in enumerate(lens)]
    x = synth.hidden_input(s, len(lens), seed=24)
    lens_d = to_dev(np.array(lens, dtype=np.int64))
    out = torch.empty((len(lens), s.hidden), dtype=torch.float16, device="cuda")
    ws = torch.empty(db.block.decode_batch_workspace_bytes(len(lens)), dtype=torch.uint8,
                     device="cuda")
    db.block.decode_batch(db.w, to_dev(x), lens_d, lens_d, max(lens),
                          to_dev(np.stack([k for k, _ in hist])),
                          to_dev(np.stack([v for _, v in hist])), out, ws)
    torch.cuda.synchronize()
    db.block.check()
    for b, L in enumerate(lens):
        k, v = hist[b][0].copy(), hist[b][1].copy()
        o_ref, _, _ = oracle.block_forward(s, w, x[b:b + 1], [L], L, k, v, yarn=YARN)
        assert_close(out[b:b + 1].cpu().numpy(), o_ref, f"batched seq {b} (L={L})")


def test_plain_rope_comes_back_bit_for_bit():
    """set_rope_yarn(None) rebuilds the plain table: the output then equals a
    fresh handle's, bit for bit."""
    s, L = synth.QWEN2_1P5B, 700
    w = synth.block_weights(s, seed=25)
    x = synth.hidden_input(s, 1, seed=25)
    kc, vc = synth.kv_history(s, L + 8, L, seed=25)
    fresh = DevBlock(s, w, L + 8, 1)
    a = fresh.run("decode", to_dev(x), to_dev(synth.positions(L, 1)), L, to_dev(kc), to_dev(vc))[0]
    db = DevBlock(s, w, L + 8, 1)
    db.block.set_rope_yarn(YARN)
    y = db.run("decode", to_dev(x), to_dev(synth.positions(L, 1)), L, to_dev(kc), to_dev(vc))[0]
    db.block.set_rope_yarn(None)
    b = db.run("decode", to_dev(x), to_dev(synth.positions(L, 1)), L, to_dev(kc), to_dev(vc))[0]
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("field,value", [("freq_scale", 0.0), ("freq_scale", 1.5),
                                         ("ext_factor", -0.1), ("ext_factor", 2.0),
                                         ("attn_factor", 0.0), ("beta_fast", 0.0),
                                         ("beta_slow", -1.0), ("n_ctx_orig", 0)])
def test_out_of_range_yarn_fields_are_refused(field, value):
    b = blk.Block(synth.TINY, 16)
    y = blk.BlkYarn(*(dict(YARN, **{field: value})[k] for k in blk.YARN_FIELDS))
    assert blk.blk_set_rope_yarn(b.handle, y) == blk.BLK_ERR_SHAPE
    assert blk.blk_set_rope_yarn(None, None) == blk.BLK_ERR_NULL
    assert blk.blk_set_rope_yarn(b.handle, None) == blk.BLK_OK
