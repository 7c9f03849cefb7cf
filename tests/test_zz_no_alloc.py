"""blk_decode_static: the decode entry point for callers that cannot allocate
device memory (e.g. a plugin inside a framework that owns all device memory,
or a serving loop that must not call cudaMalloc because it can synchronize the
device).  It uses a fixed 1 MiB array compiled into the library instead of a
caller-provided workspace.

Checked through the C ABI against the workspace-taking blk_decode, on two
decode calls in a row (the second call reuses the array left over by the
first): both run the same deterministic kernel on the same inputs, so the
outputs and cache slots must be identical bit for bit.  Around the second
call (the array's address is already known) the device's free memory, read
with cudaMemGetInfo, must not change.  This file sorts last so that a run
stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import decode_qwen2_block_gb300 as blk
import oracle
import synth
from gpu_harness import DevBlock, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _empty_outputs(s):
    out = torch.empty((1, s.hidden), dtype=torch.float16, device="cuda")
    kn = torch.empty((1, s.n_kv_heads, s.head_dim), dtype=torch.float16, device="cuda")
    return out, kn, torch.empty_like(kn)


def _host_caches(kc, vc, L):
    """Host copies of the caches with slot L (the call's own) cleared: the
    oracle writes it itself."""
    k, v = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
    k[:, L:] = 0
    v[:, L:] = 0
    return k, v


def _decode_static(db, x, pos, L, kc, vc, outs):
    out, kn, vn = outs
    rc = blk.blk_decode_static(db.block.handle, db.w, x.data_ptr(), pos.data_ptr(), L,
                               kc.data_ptr(), vc.data_ptr(), out.data_ptr(), kn.data_ptr(),
                               vn.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == blk.BLK_OK, blk.blk_status_str(rc)
    return out, kn, vn


@pytest.mark.parametrize("shape_name,L", [("TINY", 30), ("QWEN2_1P5B", 4096), ("GQA_4096", 300)])
def test_static_scratch_decode_matches_workspace_decode(shape_name, L):
    s = getattr(synth, shape_name)
    C = L + 16
    w = synth.block_weights(s, seed=0)
    kc_np, vc_np = synth.kv_history(s, C, L, seed=0)
    db = DevBlock(s, w, C, 1)
    kc_ws, vc_ws = to_dev(kc_np), to_dev(vc_np)      # cache for the workspace path
    kc_st, vc_st = to_dev(kc_np), to_dev(vc_np)      # cache for the static path
    for step in range(2):                             # two calls in a row
        x = to_dev(synth.hidden_input(s, 1, seed=0, stream_offset=step + 1))
        pos = to_dev(synth.positions(L + step, 1))
        ref = db.run("decode", x, pos, L + step, kc_ws, vc_ws)
        outs = _empty_outputs(s)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        got = _decode_static(db, x, pos, L + step, kc_st, vc_st, outs)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert blk.blk_check(db.block.handle, torch.cuda.current_stream().cuda_stream) == blk.BLK_OK
        if step == 1:   # the array's address was looked up by the first call
            assert free_after == free_before, "blk_decode_static changed free device memory"
        for name, g, r in zip(("out", "k_new", "v_new"), got, ref):
            assert torch.equal(g.view(torch.int16), r.view(torch.int16)), f"step {step} {name}"
        assert torch.equal(kc_st.view(torch.int16), kc_ws.view(torch.int16))
        assert torch.equal(vc_st.view(torch.int16), vc_ws.view(torch.int16))
    # and both equal the oracle's decode within the tolerance of every parity test
    o_ref, k_ref, v_ref = oracle.block_forward(s, w, synth.hidden_input(s, 1, seed=0, stream_offset=2),
                                               synth.positions(L + 1, 1), L + 1, *_host_caches(kc_st, vc_st, L + 1))
    assert_close(got[0].cpu().numpy(), o_ref, "out vs oracle")
    assert_close(got[1].cpu().numpy(), k_ref, "k_new vs oracle")


def test_static_scratch_rejects_shapes_over_its_limit():
    # hidden 12288, 96 query heads over 6 kv heads: about 1.1 MiB of scratch.
    # The call must be refused before anything is enqueued, so the weights are
    # never read: one zero buffer large enough for every matrix stands in.
    s = synth.BlockShape(12288, 96, 6, 128, 12288, False)
    C = 64
    blkh = blk.Block(s, C)
    big = torch.zeros(s.hidden * s.hidden, dtype=torch.float16, device="cuda")
    gains = torch.ones(s.hidden, dtype=torch.float16, device="cuda")
    w_dev = {k: (gains if k.startswith("ln") else big) for k in synth.weight_shapes(s)}
    w = blk.Block.weights(w_dev)
    x = torch.zeros((1, s.hidden), dtype=torch.float16, device="cuda")
    pos = to_dev(synth.positions(10, 1))
    kc = torch.zeros((s.n_kv_heads, C, s.head_dim), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    out = torch.full((1, s.hidden), 7.0, dtype=torch.float16, device="cuda")
    before = kc.clone()
    rc = blk.blk_decode_static(blkh.handle, w, x.data_ptr(), pos.data_ptr(), 10,
                               kc.data_ptr(), vc.data_ptr(), out.data_ptr(), None, None,
                               torch.cuda.current_stream().cuda_stream)
    assert rc == blk.BLK_ERR_SCRATCH_LIMIT
    # a missing pointer is reported before the size limit
    rc = blk.blk_decode_static(blkh.handle, w, None, pos.data_ptr(), 10,
                               kc.data_ptr(), vc.data_ptr(), out.data_ptr(), None, None,
                               torch.cuda.current_stream().cuda_stream)
    assert rc == blk.BLK_ERR_NULL
    torch.cuda.synchronize()
    assert torch.equal(kc, before)           # nothing was enqueued
    assert torch.all(out == 7.0)
