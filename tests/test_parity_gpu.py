"""GPU parity: the library's three phases against the CPU oracle, through the
C ABI, on every block shape; cache placement checked bit for bit.

Tolerances (per tensor): relative L2 <= 1e-2 and max |err| <= 5e-2 on
unit-scale activations; K/V cache slots must equal the returned k_new/v_new
bit for bit, and every slot outside [cache_len, cache_len + T) must keep its
previous bits.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import DevBlock, assert_close, to_dev

pytestmark = pytest.mark.gpu
SENTINEL = np.float16(-3.5)


def _check_cache(kc_dev, vc_dev, kc_before, vc_before, kn, vn, L, T):
    kc = kc_dev.cpu().numpy().view(np.uint16)
    vc = vc_dev.cpu().numpy().view(np.uint16)
    kb, vb = kc_before.view(np.uint16), vc_before.view(np.uint16)
    assert np.array_equal(kc[:, L:L + T], kn.cpu().numpy().view(np.uint16).transpose(1, 0, 2))
    assert np.array_equal(vc[:, L:L + T], vn.cpu().numpy().view(np.uint16).transpose(1, 0, 2))
    for got, before in ((kc, kb), (vc, vb)):
        assert np.array_equal(got[:, :L], before[:, :L]), "history slots changed"
        assert np.array_equal(got[:, L + T:], before[:, L + T:]), "slots past the new rows changed"


def _step(db, shape, w, phase, x, L, kc_o, vc_o, kc, vc, rows=None, check_cache=True):
    T = x.shape[0]
    pos = synth.positions(L, T)
    kb, vb = (kc.cpu().numpy(), vc.cpu().numpy()) if check_cache else (None, None)
    out, kn, vn = db.run(phase, to_dev(x), to_dev(pos), L, kc, vc)
    torch.cuda.synchronize()
    db.block.check()
    o_ref, k_ref, v_ref = oracle.block_forward(shape, w, x, pos, L, kc_o, vc_o, rows=rows)
    got = out.cpu().numpy() if rows is None else out.cpu().numpy()[rows]
    res = {"out": assert_close(got, o_ref, f"{phase} L={L} T={T} out"),
           "k": assert_close(kn.cpu().numpy(), k_ref, f"{phase} L={L} k_new"),
           "v": assert_close(vn.cpu().numpy(), v_ref, f"{phase} L={L} v_new")}
    if check_cache:
        _check_cache(kc, vc, kb, vb, kn, vn, L, T)
    return res, out


def test_tiny_block_all_phases():
    """Tiny block: prefill 16 (pos 0..15), prefill_kv 4, then 8 decode steps."""
    s, C = synth.TINY, 40
    w = synth.block_weights(s, seed=0)
    x = synth.hidden_input(s, 28, seed=0)
    kc_o, vc_o = synth.kv_history(s, C, 0, sentinel=SENTINEL)
    kc, vc = to_dev(kc_o), to_dev(vc_o)
    db = DevBlock(s, w, C, 16)
    _step(db, s, w, "prefill", x[:16], 0, kc_o, vc_o, kc, vc)
    _step(db, s, w, "prefill_kv", x[16:20], 16, kc_o, vc_o, kc, vc)
    for t in range(20, 28):
        _step(db, s, w, "decode", x[t:t + 1], t, kc_o, vc_o, kc, vc)


@pytest.mark.parametrize("phase,L,T", [
    ("prefill", 0, 1), ("prefill", 0, 13), ("prefill", 0, 130),       # ragged tails
    ("prefill_kv", 0, 5), ("prefill_kv", 77, 61), ("prefill_kv", 199, 1),
    ("decode", 0, 1),                                                # first token: self only
    ("decode", 255, 1),                                              # last cache slot
])
def test_tiny_shape_edges(phase, L, T):
    s, C = synth.TINY, 256
    w = synth.block_weights(s, seed=1)
    x = synth.hidden_input(s, T, seed=1, stream_offset=L + 1)
    kc_o, vc_o = synth.kv_history(s, C, L, seed=1, sentinel=SENTINEL)
    kc, vc = to_dev(kc_o), to_dev(vc_o)
    db = DevBlock(s, w, C, max(T, 1))
    _step(db, s, w, phase, x, L, kc_o, vc_o, kc, vc)


def test_tiny_prefill_kv_long_history_split_over_ctas():
    """head_dim 64: 8 new rows on 1000 history slots; the block's 8 K/V tiles
    are split over several CTAs and merged (the D = 64 merge path)."""
    s, C, L, T = synth.TINY, 1024, 1000, 8
    w = synth.block_weights(s, seed=4)
    x = synth.hidden_input(s, T, seed=4, stream_offset=L + 1)
    kc_o, vc_o = synth.kv_history(s, C, L, seed=4, sentinel=SENTINEL)
    kc, vc = to_dev(kc_o), to_dev(vc_o)
    db = DevBlock(s, w, C, T)
    _step(db, s, w, "prefill_kv", x, L, kc_o, vc_o, kc, vc)


def test_decode_first_token_returns_v_through_wo():
    """At cache_len 0 the decode attention sees only its own key, so the
    attention output is v itself (self-only first token)."""
    s, C = synth.TINY, 8
    w = synth.block_weights(s, seed=2)
    w["w_down"] = np.zeros_like(w["w_down"])
    Wo = np.zeros((256, 256), np.float16)
    Wo[np.arange(256), np.arange(256)] = 1.0     # s.hidden == n_heads * head_dim
    w["wo"] = Wo
    x = synth.hidden_input(s, 1, seed=2)
    kc_o, vc_o = synth.kv_history(s, C, 0)
    db = DevBlock(s, w, C, 1)
    out, kn, vn = db.run("decode", to_dev(x), to_dev(synth.positions(0, 1)), 0, to_dev(kc_o),
                         to_dev(vc_o))
    G = s.n_heads // s.n_kv_heads
    v_heads = np.repeat(vn.cpu().numpy()[0].astype(np.float64), G, axis=0).reshape(-1)
    want = x[0].astype(np.float64) + v_heads
    assert np.max(np.abs(out.cpu().numpy()[0].astype(np.float64) - want)) <= 2 ** -7


def test_prefill_1p5b_layer_t1024():
    """1.5B-shaped layer (QKV bias), static prefill [1, 1024]: every K/V row
    and a sample of output rows against the oracle."""
    s, T = synth.QWEN2_1P5B, 1024
    w = synth.block_weights(s, seed=0)
    x = synth.hidden_input(s, T, seed=0)
    kc_o, vc_o = synth.kv_history(s, T, 0)
    kc, vc = to_dev(kc_o), to_dev(vc_o)
    db = DevBlock(s, w, T, T)
    rows = [0, 1, 63, 64, 127, 128, 500, 777, 1022, 1023]
    _step(db, s, w, "prefill", x, 0, kc_o, vc_o, kc, vc, rows=rows)


@pytest.mark.parametrize("L", [1024, 4096, 16384, 32768])
def test_decode_1p5b_layer_long_context(L):
    """1.5B-shaped layer, decode over a history of ~N(0,1) K/V."""
    s, C = synth.QWEN2_1P5B, 32768 + 128
    w = synth.block_weights(s, seed=0)
    kc_o, vc_o = synth.kv_history(s, C, L, seed=0, sentinel=SENTINEL)
    kc, vc = to_dev(kc_o), to_dev(vc_o)
    db = DevBlock(s, w, C, 1)
    for step in range(2):
        x = synth.hidden_input(s, 1, seed=0, stream_offset=step + 1)
        _step(db, s, w, "decode", x, L + step, kc_o, vc_o, kc, vc, check_cache=(step == 0))


def test_prefill_kv_1p5b_layer():
    """1.5B-shaped layer, 512 new tokens (pos 3584..4095) on 3584 history slots."""
    s, L, T = synth.QWEN2_1P5B, 3584, 512
    w = synth.block_weights(s, seed=0)
    x = synth.hidden_input(s, T, seed=0)
    kc_o, vc_o = synth.kv_history(s, L + T, L, seed=0)
    kc, vc = to_dev(kc_o), to_dev(vc_o)
    db = DevBlock(s, w, L + T, T)
    rows = [0, 1, 200, 255, 256, 511]
    _step(db, s, w, "prefill_kv", x, L, kc_o, vc_o, kc, vc, rows=rows)


def test_gqa4096_layer_prefill_then_decode():
    """hidden 4096, 32 q / 2 kv heads (group 16), no bias: prefill of 100
    tokens then decode steps."""
    s, C = synth.GQA_4096, 356
    w = synth.block_weights(s, seed=0)
    x = synth.hidden_input(s, 104, seed=0)
    kc_o, vc_o = synth.kv_history(s, C, 0)
    kc, vc = to_dev(kc_o), to_dev(vc_o)
    db = DevBlock(s, w, C, 100)
    _step(db, s, w, "prefill", x[:100], 0, kc_o, vc_o, kc, vc, rows=[0, 37, 99])
    for t in range(100, 103):
        _step(db, s, w, "decode", x[t:t + 1], t, kc_o, vc_o, kc, vc)


def test_prefill_kv_long_history_split_over_ctas_repeatable():
    """1.5B-shaped layer, 128 new rows on 8064 history slots: the 64 K/V tiles
    of the row block are split over 11 CTAs whose partials are merged; a
    second identical call returns the same bits (the merge counters are left
    at zero)."""
    s, L, T = synth.QWEN2_1P5B, 8064, 128
    w = synth.block_weights(s, seed=3)
    x = synth.hidden_input(s, T, seed=3)
    kc_o, vc_o = synth.kv_history(s, L + T, L, seed=3)
    kc, vc = to_dev(kc_o), to_dev(vc_o)
    db = DevBlock(s, w, L + T, T)
    rows = [0, 1, 64, 126, 127]
    _, out1 = _step(db, s, w, "prefill_kv", x, L, kc_o, vc_o, kc, vc, rows=rows)
    _, out2 = _step(db, s, w, "prefill_kv", x, L, kc_o, vc_o, kc, vc, rows=rows)
    assert torch.equal(out1, out2)
