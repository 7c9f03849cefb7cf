"""Error behaviour of the C ABI with a live handle: every bad argument gives
its status code and enqueues nothing; an out-of-range position id is
clamped on the device and reported by blk_check."""
import ctypes

import numpy as np
import pytest
import torch

import decode_qwen2_block_gb300 as blk
import synth
from gpu_harness import DevBlock, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    s, C = synth.TINY, 32
    w = synth.block_weights(s, seed=0)
    db = DevBlock(s, w, C, 8)
    x = to_dev(synth.hidden_input(s, 8, seed=0))
    pos = to_dev(synth.positions(0, 8))
    kc = torch.zeros((2, C, 64), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    out = torch.empty((8, 256), dtype=torch.float16, device="cuda")
    return s, db, x, pos, kc, vc, out


def _prefill(db, x, pos, T, kc, vc, out, ws=None, ws_bytes=None, w=None):
    ws = db.ws if ws is None else ws
    nb = ws.numel() if ws_bytes is None else ws_bytes
    return blk.blk_prefill(db.block.handle, db.w if w is None else w, x, pos, T, kc, vc, out,
                           None, None, ws.data_ptr() if hasattr(ws, "data_ptr") else ws, nb,
                           torch.cuda.current_stream().cuda_stream)


def test_argument_errors(setup):
    s, db, x, pos, kc, vc, out = setup
    P = lambda t: t.data_ptr()
    assert _prefill(db, P(x), P(pos), 8, P(kc), P(vc), P(out)) == blk.BLK_OK
    assert _prefill(db, None, P(pos), 8, P(kc), P(vc), P(out)) == blk.BLK_ERR_NULL
    assert _prefill(db, P(x) + 2, P(pos), 7, P(kc), P(vc), P(out)) == blk.BLK_ERR_ALIGN
    assert _prefill(db, P(x), P(pos) + 4, 8, P(kc), P(vc), P(out)) == blk.BLK_ERR_ALIGN
    assert _prefill(db, P(x), P(pos), 0, P(kc), P(vc), P(out)) == blk.BLK_ERR_SHAPE
    assert _prefill(db, P(x), P(pos), 8, P(kc), P(vc), P(out), ws_bytes=1024) == blk.BLK_ERR_WORKSPACE
    w = blk.Block.weights(db.w_dev)
    w.wq = None
    assert _prefill(db, P(x), P(pos), 8, P(kc), P(vc), P(out), w=w) == blk.BLK_ERR_NULL
    # gains (and biases) are read as 16-byte vectors: a 2-byte-aligned gain is refused
    for name in ("ln1_g", "ln2_g"):
        w = blk.Block.weights(db.w_dev)
        setattr(w, name, db.w_dev[name].data_ptr() + 2)
        assert _prefill(db, P(x), P(pos), 8, P(kc), P(vc), P(out), w=w) == blk.BLK_ERR_ALIGN
    h = db.block.handle
    stream = torch.cuda.current_stream().cuda_stream
    ws, nb = db.ws.data_ptr(), db.ws.numel()
    assert blk.blk_prefill_kv(h, db.w, P(x), P(pos), 8, 30, P(kc), P(vc), P(out), None, None,
                              ws, nb, stream) == blk.BLK_ERR_CACHE_OVERFLOW
    assert blk.blk_prefill_kv(h, db.w, P(x), P(pos), 8, -1, P(kc), P(vc), P(out), None, None,
                              ws, nb, stream) == blk.BLK_ERR_CACHE_OVERFLOW
    assert blk.blk_decode(h, db.w, P(x), P(pos), 32, P(kc), P(vc), P(out), None, None,
                          ws, nb, stream) == blk.BLK_ERR_CACHE_OVERFLOW
    torch.cuda.synchronize()
    assert blk.blk_check(h, stream) == blk.BLK_OK


def test_out_of_range_position_is_clamped_and_reported(setup):
    s, db, x, _, kc, vc, out = setup
    bad = torch.tensor([5, 10 ** 9], dtype=torch.int64, device="cuda")
    o, _, _ = db.run("prefill", x[:2], bad, 0, kc, vc)
    stream = torch.cuda.current_stream().cuda_stream
    assert blk.blk_check(db.block.handle, stream) == blk.BLK_ERR_POSITION
    assert torch.isfinite(o.float()).all()
    # the status word is cleared by the check
    assert blk.blk_check(db.block.handle, stream) == blk.BLK_OK


def test_workspace_size_is_monotone(setup):
    s, db, *_ = setup
    sizes = [db.block.workspace_bytes(t) for t in (1, 2, 8, 100)]
    assert all(a <= b for a, b in zip(sizes, sizes[1:]))
    assert db.block.workspace_bytes(0) == 0


def test_workspace_queries_cover_every_smaller_call():
    """blk_workspace_bytes(max_T) and blk_decode_batch_workspace_bytes(max_B)
    never shrink as the bound grows: a workspace sized for a bound serves
    every smaller call (the attention's partial buffers alone do shrink at
    some sizes)."""
    for s in (synth.TINY, synth.QWEN2_1P5B):
        b = blk.Block(s, 4096)
        t_sizes = [b.workspace_bytes(T) for T in range(1, 3000, 5)]
        assert all(x <= y for x, y in zip(t_sizes, t_sizes[1:]))
        b_sizes = [b.decode_batch_workspace_bytes(B) for B in range(1, 400)]
        assert all(x <= y for x, y in zip(b_sizes, b_sizes[1:]))


def test_bounded_wait_times_out_and_the_context_stays_usable(setup):
    """A device wait on a flag that nothing sets gives up after its limit,
    blk_check reports the timeout, and the same context then runs the block."""
    import time
    s, db, x, pos, kc, vc, out = setup
    P = lambda t: t.data_ptr()
    h = db.block.handle
    stream = torch.cuda.current_stream().cuda_stream
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    assert blk.blk_wait_probe(h, P(flag), 50_000_000, stream) == blk.BLK_OK
    assert blk.blk_check(h, stream) == blk.BLK_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 10
    flag.fill_(1)
    assert blk.blk_wait_probe(h, P(flag), 50_000_000, stream) == blk.BLK_OK
    assert blk.blk_check(h, stream) == blk.BLK_OK
    assert _prefill(db, P(x), P(pos), 8, P(kc), P(vc), P(out)) == blk.BLK_OK
    assert blk.blk_check(h, stream) == blk.BLK_OK
    assert blk.blk_wait_probe(h, P(flag), 10, stream) == blk.BLK_ERR_SHAPE
    assert blk.blk_wait_probe(h, P(flag) + 2, 50_000_000, stream) == blk.BLK_ERR_ALIGN
