"""GPU parity of the model head around the block stack: token embedding (bit for
bit), final RMSNorm + LM head logits (relative L2 <= 1e-2, max abs <= 5e-2)
and the greedy token. Where several tokens are correct (logits closer than the
tolerance) the test checks that the returned one is valid: its oracle logit is
within the tolerance of the largest; when the oracle's two best logits are
further apart than twice the tolerance the token must equal the oracle's.
Equal weight rows give equal fp32 logits on the GPU, so the lowest-index rule
is checked exactly."""
import numpy as np
import pytest
import torch

import decode_qwen2_block_gb300 as blk
import oracle
import synth
from gpu_harness import MAX_ABS_TOL, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _block(shape):
    return blk.Block(shape, 64)


def _check_tokens(tok, ref_logits, what):
    for t, v in enumerate(tok):
        row = ref_logits[t]
        best = row.max()
        assert row[v] >= best - MAX_ABS_TOL, f"{what} t={t}: token {v} is not a valid argmax"
        top2 = np.sort(row)[-2:]
        if top2[1] - top2[0] > 2 * MAX_ABS_TOL:
            assert v == int(np.argmax(row)), f"{what} t={t}"


def _run_head(b, x_np, hw, want_logits=True):
    x = to_dev(x_np)
    W = to_dev(hw["lm_head"])
    g = to_dev(hw["norm_g"])
    T, V = x_np.shape[0], hw["lm_head"].shape[0]
    tokens = torch.full((T,), -5, dtype=torch.int64, device="cuda")
    logits = torch.full((T, V), float("nan"), dtype=torch.float32, device="cuda") if want_logits else None
    ws = torch.empty(b.lm_head_workspace_bytes(), dtype=torch.uint8, device="cuda")
    b.lm_head(x, g, W, tokens, ws, logits=logits)
    torch.cuda.synchronize()
    b.check()
    return (None if logits is None else logits.cpu().numpy()), tokens.cpu().numpy()


@pytest.mark.parametrize("T", [1, 3, 8])
def test_tiny_lm_head_logits_and_tokens(T):
    s = synth.TINY
    hw = synth.head_weights(1000, s.hidden, seed=5, gain_std=0.1)
    x = synth.hidden_input(s, T, seed=5, stream_offset=7)
    b = _block(s)
    got, tok = _run_head(b, x, hw)
    ref, ref_tok = oracle.lm_head(x, hw["norm_g"], hw["lm_head"], eps=s.rms_eps)
    for t in range(T):
        assert_close(got[t], ref[t], f"logits t={t}")
    _check_tokens(tok, ref, "tiny")


def test_lm_head_1p5b_full_vocabulary():
    """151936 x 1536 LM head, one row (a decode step) and two rows."""
    s = synth.QWEN2_1P5B
    hw = synth.head_weights(synth.QWEN2_VOCAB, s.hidden, seed=0)
    b = _block(s)
    for T in (1, 2):
        x = synth.hidden_input(s, T, seed=0, stream_offset=11 + T)
        got, tok = _run_head(b, x, hw)
        ref, _ = oracle.lm_head(x, hw["norm_g"], hw["lm_head"], eps=s.rms_eps)
        for t in range(T):
            assert_close(got[t], ref[t], f"1.5B logits T={T} t={t}")
        _check_tokens(tok, ref, f"1.5B T={T}")
        _, tok2 = _run_head(b, x, hw, want_logits=False)   # tokens only: same decision
        assert np.array_equal(tok, tok2)


def test_lm_head_ties_give_the_lowest_index():
    s = synth.TINY
    V, H = 777, s.hidden
    x = synth.hidden_input(s, 2, seed=9)
    hw = {"norm_g": np.ones(H, np.float16),
          "lm_head": (synth.normal_f16(9, 1, (V, H), std=0.02))}
    # the same best row at 700, 41 and 512 (and twice as large as any other)
    best = np.sign(x[0].astype(np.float64)).astype(np.float16) * np.float16(0.5)
    W = hw["lm_head"].copy()
    for v in (700, 41, 512):
        W[v] = best
    hw["lm_head"] = W
    b = _block(s)
    got, tok = _run_head(b, x, hw)
    assert tok[0] == 41
    assert got[0][41] == got[0][512] == got[0][700]


def test_embed_rows_bit_exact_and_bad_id_reported():
    s = synth.QWEN2_1P5B
    hw = synth.head_weights(synth.QWEN2_VOCAB, s.hidden, seed=1)
    ids = synth.token_ids(synth.QWEN2_VOCAB, 37, seed=3)
    ids[0], ids[1] = 0, synth.QWEN2_VOCAB - 1
    b = _block(s)
    table = to_dev(hw["embed"])
    x = torch.empty((ids.size, s.hidden), dtype=torch.float16, device="cuda")
    b.embed(table, to_dev(ids), x)
    torch.cuda.synchronize()
    b.check()
    want = oracle.embed(hw["embed"], ids)
    assert np.array_equal(x.cpu().numpy().view(np.uint16), want.view(np.uint16))
    bad = torch.tensor([5, synth.QWEN2_VOCAB, -1], dtype=torch.int64, device="cuda")
    xb = torch.full((3, s.hidden), 1.0, dtype=torch.float16, device="cuda")
    b.embed(table, bad, xb)
    torch.cuda.synchronize()
    with pytest.raises(blk.BlkError) as e:
        b.check()
    assert e.value.status == blk.BLK_ERR_TOKEN
    out = xb.cpu().numpy()
    assert np.array_equal(out[0].view(np.uint16), hw["embed"][5].view(np.uint16))
    assert not out[1:].any()


def test_lm_head_argument_errors():
    s = synth.TINY
    b = _block(s)
    hw = synth.head_weights(100, s.hidden, seed=2)
    W, g = to_dev(hw["lm_head"]), to_dev(hw["norm_g"])
    tokens = torch.empty(9, dtype=torch.int64, device="cuda")
    ws = torch.empty(b.lm_head_workspace_bytes(), dtype=torch.uint8, device="cuda")
    for T in (0, 9):
        x = torch.zeros((max(T, 1), s.hidden), dtype=torch.float16, device="cuda")
        rc = blk.blk_lm_head(b.handle, x.data_ptr(), T, g.data_ptr(), W.data_ptr(), 100, None,
                             tokens.data_ptr(), ws.data_ptr(), ws.numel(), 0)
        assert rc == blk.BLK_ERR_SHAPE
    x = torch.zeros((1, s.hidden), dtype=torch.float16, device="cuda")
    rc = blk.blk_lm_head(b.handle, x.data_ptr(), 1, g.data_ptr(), W.data_ptr(), 100, None,
                         tokens.data_ptr(), ws.data_ptr(), 16, 0)
    assert rc == blk.BLK_ERR_WORKSPACE
    rc = blk.blk_lm_head(b.handle, x.data_ptr(), 1, g.data_ptr(), W.data_ptr() + 2, 100, None,
                         tokens.data_ptr(), ws.data_ptr(), ws.numel(), 0)
    assert rc == blk.BLK_ERR_ALIGN
    gp = torch.zeros(s.hidden + 8, dtype=torch.float16, device="cuda")
    rc = blk.blk_lm_head(b.handle, x.data_ptr(), 1, gp.data_ptr() + 2, W.data_ptr(), 100, None,
                         tokens.data_ptr(), ws.data_ptr(), ws.numel(), 0)
    assert rc == blk.BLK_ERR_ALIGN


def test_lm_head_hidden_4096_three_stage_ring():
    """hidden 4096 (the larger GQA shape) takes the three-stage ring; each
    16-row group arrives in three column chunks (24, 24, 16 blocks)."""
    s = synth.GQA_4096
    hw = synth.head_weights(5003, s.hidden, seed=21, gain_std=0.1)
    b = _block(s)
    x = synth.hidden_input(s, 4, seed=21, stream_offset=3)
    got, tok = _run_head(b, x, hw)
    ref, _ = oracle.lm_head(x, hw["norm_g"], hw["lm_head"], eps=s.rms_eps)
    for t in range(4):
        assert_close(got[t], ref[t], f"H=4096 logits t={t}")
    _check_tokens(tok, ref, "H=4096")
