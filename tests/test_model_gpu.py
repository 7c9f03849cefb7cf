"""End to end on the GPU: token embedding -> a stack of decoder blocks ->
final RMSNorm + LM head -> greedy token, the next step reading the token from
device memory (the pages' decode loop).  Each step is checked against the
oracle run on the same token (teacher forcing): logits within the tolerance
(relative L2 <= 1e-2, max abs <= 5e-2) and a valid greedy token (exact when the oracle's two best logits
are more than twice the tolerance apart)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from decode_qwen2_block_gb300.model import Model
from gpu_harness import MAX_ABS_TOL, assert_close, to_dev

pytestmark = pytest.mark.gpu


def test_tiny_model_greedy_decode_matches_oracle_step_by_step():
    s, n_layers, V, C, L = synth.TINY, 2, 500, 64, 24
    wl = [synth.block_weights(s, layer=l, seed=6) for l in range(n_layers)]
    hw = synth.head_weights(V, s.hidden, seed=6, gain_std=0.1)
    caches = [synth.kv_history(s, C, L, layer=l, seed=6) for l in range(n_layers)]
    model = Model(s, [{k: to_dev(v) for k, v in w.items()} for w in wl],
                  {k: to_dev(v) for k, v in hw.items()}, C,
                  caches=[(to_dev(k), to_dev(v)) for k, v in caches])
    n, first = 5, 123
    logits = []
    toks = model.generate(first, L, n, logits_out=logits)
    torch.cuda.synchronize()
    model.block.check()
    toks = toks.cpu().numpy()
    kc = [k.copy() for k, _ in caches]
    vc = [v.copy() for _, v in caches]
    cur = first
    for i in range(n):
        x = oracle.embed(hw["embed"], [cur])
        for l in range(n_layers):
            x, _, _ = oracle.block_forward(s, wl[l], x, [L + i], L + i, kc[l], vc[l])
        ref, _ = oracle.lm_head(x, hw["norm_g"], hw["lm_head"], eps=s.rms_eps)
        got = logits[i].cpu().numpy()[0]
        assert_close(got, ref[0], f"step {i} logits")
        t = int(toks[i])
        assert ref[0][t] >= ref[0].max() - MAX_ABS_TOL, f"step {i}: token {t} not a valid argmax"
        top2 = np.sort(ref[0])[-2:]
        if top2[1] - top2[0] > 2 * MAX_ABS_TOL:
            assert t == int(np.argmax(ref[0])), f"step {i}"
        cur = t   # the oracle follows the GPU's choice


def test_model_step_graph_replays_match_eager_steps():
    """A captured step replays to the same token as the eager step."""
    s, V, C, L = synth.TINY, 300, 48, 10
    wl = [synth.block_weights(s, layer=0, seed=8)]
    hw = synth.head_weights(V, s.hidden, seed=8)
    k0, v0 = synth.kv_history(s, C, L, seed=8)
    dev = lambda a: to_dev(a)
    m1 = Model(s, [{k: dev(v) for k, v in wl[0].items()}], {k: dev(v) for k, v in hw.items()}, C,
               caches=[(dev(k0), dev(v0))])
    m2 = Model(s, [{k: dev(v) for k, v in wl[0].items()}], {k: dev(v) for k, v in hw.items()}, C,
               caches=[(dev(k0), dev(v0))])
    tin = torch.tensor([42], dtype=torch.int64, device="cuda")
    pos = torch.tensor([L], dtype=torch.int64, device="cuda")
    t1 = torch.empty(1, dtype=torch.int64, device="cuda")
    t2 = torch.empty(1, dtype=torch.int64, device="cuda")
    m1.step(tin, pos, L, t1)
    g = m2.capture_step(tin, pos, L, t2)
    g.replay()
    torch.cuda.synchronize()
    m1.block.check()
    m2.block.check()
    assert int(t1.item()) == int(t2.item())
    assert torch.equal(m1.stack.caches[0][0], m2.stack.caches[0][0])
