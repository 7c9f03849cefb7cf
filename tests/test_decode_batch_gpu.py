"""GPU parity of batched decode: B sequences with their own caches and cache
lengths in one call, each checked against the oracle's decode of that
sequence alone (relative L2 <= 1e-2, max abs <= 5e-2), the new K/V slot
bit-exact and every
other cache slot untouched."""
import numpy as np
import pytest
import torch

import decode_qwen2_block_gb300 as blk
import oracle
import synth
from gpu_harness import assert_close, to_dev

pytestmark = pytest.mark.gpu
SENTINEL = np.float16(-3.5)


def _run_batch(s, w, lens, C, seed, max_len=None, sentinel=SENTINEL):
    B = len(lens)
    hist = [synth.kv_history(s, C, L, layer=b, seed=seed, sentinel=sentinel)
            for b, L in enumerate(lens)]
    kc_np = np.stack([k for k, _ in hist])
    vc_np = np.stack([v for _, v in hist])
    x = synth.hidden_input(s, B, seed=seed, stream_offset=5)
    pos = np.array(lens, dtype=np.int64)          # position = cache length
    block = blk.Block(s, C)
    wd = {k: to_dev(v) for k, v in w.items()}
    wts = blk.Block.weights(wd)
    kc, vc = to_dev(kc_np), to_dev(vc_np)
    out = torch.empty((B, s.hidden), dtype=torch.float16, device="cuda")
    kn = torch.empty((B, s.n_kv_heads, s.head_dim), dtype=torch.float16, device="cuda")
    vn = torch.empty_like(kn)
    ws = torch.empty(block.decode_batch_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    block.decode_batch(wts, to_dev(x), to_dev(pos), to_dev(pos), max(lens) if max_len is None else max_len,
                       kc, vc, out, ws, k_new=kn, v_new=vn)
    torch.cuda.synchronize()
    block.check()
    return x, kc_np, vc_np, out.cpu().numpy(), kn.cpu().numpy(), vn.cpu().numpy(), \
        kc.cpu().numpy(), vc.cpu().numpy()


def _check(s, w, lens, C, seed, sample=None, **kw):
    """Every sequence's cache placement; the oracle's decode for the
    sequences in `sample` (all when None)."""
    x, kc0, vc0, out, kn, vn, kc1, vc1 = _run_batch(s, w, lens, C, seed, **kw)
    for b, L in enumerate(lens):
        if sample is None or b in sample:
            kc_o, vc_o = kc0[b].copy(), vc0[b].copy()
            o_ref, k_ref, v_ref = oracle.block_forward(s, w, x[b:b + 1], [L], L, kc_o, vc_o)
            assert_close(out[b:b + 1], o_ref, f"seq {b} L={L} out")
            assert_close(kn[b:b + 1], k_ref, f"seq {b} k_new")
            assert_close(vn[b:b + 1], v_ref, f"seq {b} v_new")
        # slot L holds the returned K/V bit for bit; every other slot is unchanged
        assert np.array_equal(kc1[b][:, L].view(np.uint16), kn[b].view(np.uint16))
        assert np.array_equal(vc1[b][:, L].view(np.uint16), vn[b].view(np.uint16))
        for got, before in ((kc1[b], kc0[b]), (vc1[b], vc0[b])):
            mask = np.ones(got.shape[1], bool)
            mask[L] = False
            assert np.array_equal(got[:, mask].view(np.uint16), before[:, mask].view(np.uint16))


def test_tiny_batch_of_three_lengths():
    s = synth.TINY
    w = synth.block_weights(s, seed=7)
    _check(s, w, [0, 37, 100], 128, seed=7)


def test_1p5b_batch_mixed_lengths():
    s = synth.QWEN2_1P5B
    w = synth.block_weights(s, seed=8)
    _check(s, w, [1000, 4095, 17, 2048], 4096 + 64, seed=8)


def test_tiny_batch_past_one_row_tile():
    """130 sequences: the activation operand is a full 128-row tile plus a
    2-row tile (the second SM pair's A box is partly out of range)."""
    s = synth.TINY
    w = synth.block_weights(s, seed=12)
    rng = np.random.default_rng(12)
    lens = [int(v) for v in rng.integers(0, 62, size=130)]
    _check(s, w, lens, 64, seed=12)


@pytest.mark.parametrize("B", [3, 80])
def test_nan_in_unused_slots_is_never_read(B):
    """Every slot past a sequence's length holds NaN: slots past the end of a
    split share a tile with real ones, and none of them may reach the output
    (3 sequences: one CTA per SM; 80 x 2 kv heads: two CTAs per SM, and
    the few-row projections with their 128-row activation box)."""
    s = synth.TINY
    w = synth.block_weights(s, seed=14)
    rng = np.random.default_rng(14)
    lens = [int(v) for v in rng.integers(0, 190, size=B)]
    _check(s, w, lens, 192, seed=14, sentinel=np.float16(np.nan))


def test_1p5b_bench_launch_configuration():
    """The batched bench's configuration: 64 sequences near ctx 1024 (two
    attention splits; the few-row projections split QKV 4 ways, o_proj 8 and
    down 12); the oracle checks three sequences, the cache placement all 64."""
    s = synth.QWEN2_1P5B
    w = synth.block_weights(s, seed=13)
    lens = [1024 - (b % 7) for b in range(64)]
    _check(s, w, lens, 1024 + 8, seed=13, sample=(0, 37, 63))


def test_gqa4096_batch_and_a_generous_length_bound():
    """16 query heads per kv head (a full MMA tile of rows); max_cache_len far
    above the actual lengths only changes the split count."""
    s = synth.GQA_4096
    w = synth.block_weights(s, seed=9)
    _check(s, w, [300, 5], 512, seed=9, max_len=511)


def test_batch_equals_single_sequence_decode():
    """The same sequence through blk_decode and through a batch of 5."""
    s = synth.QWEN2_1P5B
    w = synth.block_weights(s, seed=10)
    C, L = 1024, 700
    k0, v0 = synth.kv_history(s, C, L, seed=10)
    x = synth.hidden_input(s, 5, seed=10)
    block = blk.Block(s, C)
    wd = {k: to_dev(v) for k, v in w.items()}   # kept alive: the handle holds raw pointers
    wts = blk.Block.weights(wd)
    out1 = torch.empty((1, s.hidden), dtype=torch.float16, device="cuda")
    ws1 = torch.empty(block.workspace_bytes(1), dtype=torch.uint8, device="cuda")
    kc1, vc1 = to_dev(k0), to_dev(v0)
    block.decode(wts, to_dev(x[2:3]), to_dev(np.array([L])), L, kc1, vc1, out1, ws1)
    kcb = to_dev(np.stack([k0] * 5))
    vcb = to_dev(np.stack([v0] * 5))
    lens = to_dev(np.array([L] * 5, dtype=np.int64))
    outb = torch.empty((5, s.hidden), dtype=torch.float16, device="cuda")
    wsb = torch.empty(block.decode_batch_workspace_bytes(5), dtype=torch.uint8, device="cuda")
    block.decode_batch(wts, to_dev(x), lens, lens, L, kcb, vcb, outb, wsb)
    torch.cuda.synchronize()
    block.check()
    assert_close(outb[2:3].cpu().numpy(), out1.cpu().numpy().astype(np.float64), "batch vs single")


@pytest.mark.parametrize("shape_name", ["TINY", "QWEN2_1P5B"])
def test_batch_argument_errors_and_bad_length(shape_name):
    """A length past max_ctx is refused on the host when max_cache_len says
    so, else reported on the device with nothing written for that sequence
    (1.5B: the QKV projection splits K and the attention kernel finishes it)."""
    s = getattr(synth, shape_name)
    w = synth.block_weights(s, seed=11)
    C, B = 64, 2
    block = blk.Block(s, C)
    wd = {k: to_dev(v) for k, v in w.items()}   # kept alive: the handle holds raw pointers
    wts = blk.Block.weights(wd)
    kc = torch.zeros((B, s.n_kv_heads, C, s.head_dim), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    x = torch.zeros((B, s.hidden), dtype=torch.float16, device="cuda")
    out = torch.empty_like(x)
    ws = torch.empty(block.decode_batch_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    lens = torch.tensor([3, 70], dtype=torch.int64, device="cuda")   # 70 >= max_ctx
    with pytest.raises(blk.BlkError) as e:
        block.decode_batch(wts, x, lens, lens, C, kc, vc, out, ws)
    assert e.value.status == blk.BLK_ERR_CACHE_OVERFLOW
    block.decode_batch(wts, x, lens, lens, C - 1, kc, vc, out, ws)
    torch.cuda.synchronize()
    with pytest.raises(blk.BlkError) as e:
        block.check()
    assert e.value.status == blk.BLK_ERR_POSITION
    assert not kc[1].any() and not vc[1].any()           # nothing written for the bad sequence


def _stack_inputs(s, n_layers, B, C, seed):
    wl = [synth.block_weights(s, layer=l, seed=seed) for l in range(n_layers)]
    lens = [3 + 11 * b for b in range(B)]
    caches = []
    for l in range(n_layers):
        hist = [synth.kv_history(s, C, L, layer=100 * l + b, seed=seed, sentinel=SENTINEL)
                for b, L in enumerate(lens)]
        caches.append((np.stack([k for k, _ in hist]), np.stack([v for _, v in hist])))
    x = synth.hidden_input(s, B, seed=seed, stream_offset=9)
    return wl, lens, caches, x


@pytest.mark.parametrize("shape_name,n,B,C,fused", [
    # up to 128 sequences the few-row projections always split the down K:
    # its reduction is fused with the next layer's RMSNorm 1
    ("TINY", 3, 5, 64, True),
    ("QWEN2_1P5B", 2, 3, 64, True),
    ("QWEN2_1P5B", 3, 64, 704, True),   # the bench's batch size
    # 130 sequences take the 2-SM GEMMs, whose tiny down K is too short to
    # split: the next layer's RMSNorm 1 runs as its own kernel
    ("TINY", 2, 130, 1440, False),
])
def test_batch_stack_equals_one_call_per_layer(shape_name, n, B, C, fused):
    """blk_decode_batch_stack = blk_decode_batch per layer, bit for bit
    (outputs and every cache).  The stack writes layer l + 1's RMSNorm 1 from
    layer l's tail (fused with the down split-K reduction when the down
    projection splits K), so its launches differ from the per-layer calls'
    while the bits must not."""
    from decode_qwen2_block_gb300.stack import BatchStack
    s = getattr(synth, shape_name)
    wl, lens, caches, x = _stack_inputs(s, n, B, C, seed=15)
    wd = [{k: to_dev(v) for k, v in w.items()} for w in wl]
    lens_d = to_dev(np.array(lens, dtype=np.int64))
    st = BatchStack(s, wd, C, B, caches=[(to_dev(k), to_dev(v)) for k, v in caches])
    out = torch.empty((B, s.hidden), dtype=torch.float16, device="cuda")
    st.block.timing(True)
    st.step(to_dev(x), lens_d, lens_d, max(lens), out)
    st.block.timing_collect()
    st.block.timing(False)
    torch.cuda.synchronize()
    st.block.check()
    launched = {k: c for k, (_, c) in st.block.timing_table().items()}
    if fused:
        assert launched.get("splitk_reduce_norm") == n - 1
        assert launched.get("splitk_reduce") == 1           # the last layer's
    else:
        assert "splitk_reduce_norm" not in launched
    block = blk.Block(s, C)
    ws = torch.empty(block.decode_batch_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    cur = to_dev(x)
    ref_caches = [(to_dev(k), to_dev(v)) for k, v in caches]
    for l in range(n):
        nxt = torch.empty_like(cur)
        block.decode_batch(blk.Block.weights(wd[l]), cur, lens_d, lens_d, max(lens),
                           ref_caches[l][0], ref_caches[l][1], nxt, ws)
        cur = nxt
    torch.cuda.synchronize()
    block.check()
    assert torch.equal(out.view(torch.int16), cur.view(torch.int16))
    for (k1, v1), (k2, v2) in zip(st.caches, ref_caches):
        assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
        assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))


def test_batch_stack_checks_every_layer_before_enqueueing():
    from decode_qwen2_block_gb300.stack import BatchStack
    s, n, B, C = synth.TINY, 3, 2, 64
    wl, lens, caches, x = _stack_inputs(s, n, B, C, seed=16)
    wd = [{k: to_dev(v) for k, v in w.items()} for w in wl]
    st = BatchStack(s, wd, C, B, caches=[(to_dev(k), to_dev(v)) for k, v in caches])
    st._w_arr[2].wq = None                       # the last layer is bad
    lens_d = to_dev(np.array(lens, dtype=np.int64))
    out = torch.empty((B, s.hidden), dtype=torch.float16, device="cuda")
    with pytest.raises(blk.BlkError) as e:
        st.step(to_dev(x), lens_d, lens_d, max(lens), out)
    assert e.value.status == blk.BLK_ERR_NULL
    torch.cuda.synchronize()
    for (kc, vc), (k0, v0) in zip(st.caches, caches):   # nothing ran: caches unchanged
        assert np.array_equal(kc.cpu().numpy().view(np.uint16), k0.view(np.uint16))
        assert np.array_equal(vc.cpu().numpy().view(np.uint16), v0.view(np.uint16))
