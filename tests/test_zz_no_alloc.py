"""blk_decode_static: the decode entry point for callers that cannot allocate
device memory (e.g. a plugin inside a framework that owns all device memory,
or a serving loop that must not call cudaMalloc because it can synchronize the
device).  It uses a fixed 1 MiB array compiled into the library instead of a
caller-provided workspace.

Checked through the C ABI against the workspace-taking blk_decode, on two
decode calls in a row (the second call reuses the array left over by the
first).  This file sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import decode_qwen2_block_gb300 as blk
import synth
from gpu_harness import DevBlock, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _decode_static(db, x, pos, L, kc, vc):
    s = db.shape
    out = torch.empty((1, s.hidden), dtype=torch.float16, device="cuda")
    kn = torch.empty((1, s.n_kv_heads, s.head_dim), dtype=torch.float16, device="cuda")
    vn = torch.empty_like(kn)
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
        got = _decode_static(db, x, pos, L + step, kc_st, vc_st)
        torch.cuda.synchronize()
        assert blk.blk_check(db.block.handle, torch.cuda.current_stream().cuda_stream) == blk.BLK_OK
        for name, g, r in zip(("out", "k_new", "v_new"), got, ref):
            assert_close(g.cpu().numpy(), r.cpu().numpy(), f"step {step} {name}")
        assert torch.equal(kc_st[:, L + step], kc_ws[:, L + step])
        assert torch.equal(vc_st[:, L + step], vc_ws[:, L + step])


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
    torch.cuda.synchronize()
    assert torch.equal(kc, before)           # nothing was enqueued
    assert torch.all(out == 7.0)
