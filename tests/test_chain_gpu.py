"""GPU checks across calls: the phase-chain identities of the three-phase
split, bitwise agreement of the overlapped (BLK_FLAG_CHAIN) and CUDA-graph
launch configurations with plain launches, determinism, and layer-local
parity of full-size layer stacks in the launch configuration the benchmark
times."""
import numpy as np
import pytest
import torch

import decode_qwen2_block_gb300 as blk
import oracle
import synth
from decode_qwen2_block_gb300.stack import LayerStack
from gpu_harness import DevBlock, assert_close, to_dev, weights_to_dev

pytestmark = pytest.mark.gpu


def _run_chain(db, s, x, splits, C):
    kc = torch.zeros((s.n_kv_heads, C, s.head_dim), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    outs, L = [], 0
    for phase, T in splits:
        pos = to_dev(synth.positions(L, T))
        o, _, _ = db.run(phase, to_dev(x[L:L + T]), pos, L, kc, vc)
        outs.append(o)
        L += T
    torch.cuda.synchronize()
    return torch.cat(outs).cpu().numpy(), kc.cpu().numpy(), vc.cpu().numpy()


def test_phase_chain_identities_gpu():
    """prefill(T) ~ prefill(T-k) -> prefill_kv(k) ~ prefill(T-1) -> decode."""
    s, C, T = synth.TINY, 32, 16
    w = synth.block_weights(s, seed=4)
    x = synth.hidden_input(s, T, seed=4)
    db = DevBlock(s, w, C, T)
    full, kf, vf = _run_chain(db, s, x, [("prefill", T)], C)
    for splits in ([("prefill", 12), ("prefill_kv", 4)],
                   [("prefill", 15), ("decode", 1)],
                   [("prefill", 8)] + [("decode", 1)] * 8):
        o, k, v = _run_chain(db, s, x, splits, C)
        assert_close(o, full, f"chain {splits[:2]} out")
        assert_close(k[:, :T], kf[:, :T], "chain K cache")
        assert_close(v[:, :T], vf[:, :T], "chain V cache")


def test_repeat_calls_are_bitwise_deterministic():
    s, C = synth.QWEN2_1P5B, 2048
    w = synth.block_weights(s, seed=0)
    db = DevBlock(s, w, C, 64)
    kc_o, vc_o = synth.kv_history(s, C, 1000)
    x = synth.hidden_input(s, 64, seed=0)
    res = []
    for _ in range(2):
        kc, vc = to_dev(kc_o), to_dev(vc_o)
        o1, k1, _ = db.run("decode", to_dev(x[:1]), to_dev(synth.positions(1000, 1)), 1000, kc, vc)
        o2, k2, _ = db.run("prefill_kv", to_dev(x), to_dev(synth.positions(1001, 64)), 1001, kc, vc)
        torch.cuda.synchronize()
        res.append([t.cpu().numpy().view(np.uint16) for t in (o1, k1, o2, k2)])
    for a, b in zip(*res):
        assert np.array_equal(a, b)


def _stack(s, n_layers, C, L, seed=0):
    wl = [weights_to_dev(synth.block_weights(s, layer=l, seed=seed)) for l in range(n_layers)]
    host_caches = [synth.kv_history(s, C, L, layer=l, seed=seed) for l in range(n_layers)]
    return wl, host_caches


def test_chain_flag_and_graph_match_plain_launches_bitwise():
    s, n, C, L = synth.QWEN2_1P5B, 4, 1024 + 8, 1000
    wl, hc = _stack(s, n, C, L)
    x = to_dev(synth.hidden_input(s, 1, seed=0))
    pos = to_dev(synth.positions(L, 1))
    results = []
    for mode in ("plain", "chain", "graph"):
        caches = [(to_dev(k), to_dev(v)) for k, v in hc]
        st = LayerStack(s, wl, C, 1, caches=caches, chain=(mode != "plain"))
        if mode == "graph":
            g, out = st.capture("decode", x, pos, L)
            g.replay()
        else:
            out = st.run("decode", x, pos, L)
        torch.cuda.synchronize()
        st.block.check()
        results.append((out.cpu().numpy().view(np.uint16).copy(),
                        caches[-1][0][:, L].cpu().numpy().view(np.uint16)))
    for r in results[1:]:
        assert np.array_equal(r[0], results[0][0])
        assert np.array_equal(r[1], results[0][1])


def test_decode_stack_one_launch_equals_per_layer_calls():
    """blk_decode_stack (all layers in one launch) gives the same bits as one
    blk_decode call per layer; 40 tiny layers also cover the split into
    launches of at most 32 layers."""
    for s, n, C, L in ((synth.QWEN2_1P5B, 3, 600, 513), (synth.TINY, 40, 64, 37)):
        wl, hc = _stack(s, n, C, L)
        x = to_dev(synth.hidden_input(s, 1, seed=3))
        pos = to_dev(synth.positions(L, 1))
        c1 = [(to_dev(k), to_dev(v)) for k, v in hc]
        c2 = [(to_dev(k), to_dev(v)) for k, v in hc]
        st1 = LayerStack(s, wl, C, 1, caches=c1)
        st2 = LayerStack(s, wl, C, 1, caches=c2)
        one = st1.decode_step(x, pos, L).clone()
        ins = []
        per = st2.run("decode", x, pos, L, layer_outputs=ins).clone()
        torch.cuda.synchronize()
        st1.block.check()
        assert torch.equal(one, per)
        for (k1, v1), (k2, v2) in zip(c1, c2):
            assert torch.equal(k1[:, L], k2[:, L]) and torch.equal(v1[:, L], v2[:, L])


def _layer_local(s, wl_np_fn, caches_before, layer_inputs, pos, L, rows, outs_next, layers):
    for l in layers:
        w = wl_np_fn(l)
        kc_o, vc_o = caches_before[l]
        x_l = layer_inputs[l].cpu().numpy()
        o_ref, _, _ = oracle.block_forward(s, w, x_l, pos, L, kc_o, vc_o, rows=rows)
        got = outs_next[l].cpu().numpy()
        if rows is not None:
            got = got[rows]
        assert_close(got, o_ref, f"layer {l}")


@pytest.mark.parametrize("L", [4096, 32768])
def test_decode_28_layer_stack_graph_layer_local(L):
    """28 layers of the 1.5B shape, decode at cache length 4096 and at the
    longest context the benchmark times (32768), captured in a CUDA graph
    with the overlapped launch (the benchmark's configuration).  Each checked
    layer is compared with the oracle run on the GPU's own input to that
    layer."""
    s = synth.QWEN2_1P5B
    C = L + 128
    n = s.n_layers
    wl, hc = _stack(s, n, C, L)
    caches = [(to_dev(k), to_dev(v)) for k, v in hc]
    st = LayerStack(s, wl, C, 1, caches=caches, chain=True)
    x = to_dev(synth.hidden_input(s, 1, seed=0))
    pos = to_dev(synth.positions(L, 1))
    # layer inputs from an eager pass (bitwise equal to the graph, checked above)
    ins = []
    st2_caches = [(to_dev(k), to_dev(v)) for k, v in hc]
    st2 = LayerStack(s, wl, C, 1, caches=st2_caches, chain=True)
    final_eager = st2.run("decode", x, pos, L, layer_outputs=ins).clone()
    g, out = st.capture("decode", x, pos, L)
    g.replay()
    torch.cuda.synchronize()
    st.block.check()
    assert torch.equal(out, final_eager)
    outs_next = ins[1:] + [final_eager]
    _layer_local(s, lambda l: synth.block_weights(s, layer=l, seed=0), hc, ins,
                 synth.positions(L, 1), L, None, outs_next, layers=[0, 13, 27])


def test_prefill_kv_28_layer_stack_layer_local():
    """28 layers of the 1.5B shape: 512 new tokens on a 3584-slot history."""
    s, L, T = synth.QWEN2_1P5B, 3584, 512
    C = L + T
    n = s.n_layers
    wl, hc = _stack(s, n, C, L)
    caches = [(to_dev(k), to_dev(v)) for k, v in hc]
    st = LayerStack(s, wl, C, T, caches=caches, chain=True)
    x = to_dev(synth.hidden_input(s, T, seed=0))
    pos = to_dev(synth.positions(L, T))
    ins = []
    final = st.run("prefill_kv", x, pos, L, layer_outputs=ins).clone()
    torch.cuda.synchronize()
    st.block.check()
    # the benchmark's path, one blk_prefill_stack call, gives the same bits
    caches2 = [(to_dev(k), to_dev(v)) for k, v in hc]
    st2 = LayerStack(s, wl, C, T, caches=caches2, chain=True)
    one = st2.run("prefill_kv", x, pos, L).clone()
    torch.cuda.synchronize()
    st2.block.check()
    assert torch.equal(one.view(torch.int16), final.view(torch.int16))
    for (k1, v1), (k2, v2) in zip(caches, caches2):
        assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
        assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    outs_next = ins[1:] + [final]
    _layer_local(s, lambda l: synth.block_weights(s, layer=l, seed=0), hc, ins,
                 synth.positions(L, T), L, [0, 255, 511], outs_next, layers=[0, 27])


@pytest.mark.parametrize("shape_name,n,T", [("TINY", 3, 40), ("QWEN2_1P5B", 3, 1024),
                                            ("QWEN2_1P5B", 2, 2048)])
def test_prefill_stack_equals_one_call_per_layer(shape_name, n, T):
    """blk_prefill_stack = blk_prefill per layer, bit for bit (output and
    caches), with the down projection's K split fused with the next layer's
    RMSNorm 1 (1.5B at T = 1024: 3 splits) or not split at all (T = 2048;
    the tiny shape's K is too short to split)."""
    s = getattr(synth, shape_name)
    wl = [weights_to_dev(synth.block_weights(s, layer=l, seed=4)) for l in range(n)]
    x = to_dev(synth.hidden_input(s, T, seed=4))
    pos = to_dev(synth.positions(0, T))
    outs = []
    for mode in ("per_layer", "stack"):
        st = LayerStack(s, wl, T, T, chain=True)
        o = st.run("prefill", x, pos, 0, layer_outputs=[] if mode == "per_layer" else None)
        torch.cuda.synchronize()
        st.block.check()
        outs.append((o.clone(), [(k.clone(), v.clone()) for k, v in st.caches]))
    (o1, c1), (o2, c2) = outs
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    for (k1, v1), (k2, v2) in zip(c1, c2):
        assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
        assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))


def test_gqa4096_prefill_then_64_decodes_layer_local():
    """The hidden-4096 shape (32 q / 2 kv heads, head_dim 128, intermediate
    11008, the TopOp paper's Figure 2 example) through a 4-layer stack: a
    prefill of 100 tokens, then 64 decode steps at positions 100..163, each
    step appending to the caches the earlier steps wrote.  Layer- and
    step-local against the oracle: every step's K/V slot of every layer
    (the oracle given that layer's input and the GPU's cache before the
    step), and the full output of every layer at the prefill (sampled rows)
    and at four of the decode steps, within the parity tolerance (relative L2
    <= 1e-2, max abs <= 5e-2 per tensor)."""
    s, n, T, ND = synth.GQA_4096, 4, 100, 64
    C = T + ND + 8
    w_np = [synth.block_weights(s, layer=l, seed=2) for l in range(n)]
    wl = [weights_to_dev(w) for w in w_np]
    st = LayerStack(s, wl, C, T, chain=True)
    x = synth.hidden_input(s, T, seed=2)
    ins_p = []
    final_p = st.run("prefill", to_dev(x), to_dev(synth.positions(0, T)), 0,
                     layer_outputs=ins_p).clone()
    torch.cuda.synchronize()
    st.block.check()
    after_prefill = [(k.cpu().numpy().copy(), v.cpu().numpy().copy()) for k, v in st.caches]
    rows = [0, 57, 99]
    for l in range(n):
        k0 = np.zeros_like(after_prefill[l][0])
        v0 = np.zeros_like(after_prefill[l][1])
        o_ref, k_ref, v_ref = oracle.block_forward(s, w_np[l], ins_p[l].cpu().numpy(),
                                                   synth.positions(0, T), 0, k0, v0, rows=rows)
        got = (ins_p[l + 1] if l + 1 < n else final_p).cpu().numpy()[rows]
        assert_close(got, o_ref, f"prefill layer {l}")
        assert_close(after_prefill[l][0][:, :T].transpose(1, 0, 2), k_ref, f"prefill K layer {l}")
        assert_close(after_prefill[l][1][:, :T].transpose(1, 0, 2), v_ref, f"prefill V layer {l}")
    xd = synth.hidden_input(s, ND, seed=2, stream_offset=1)
    step_ins, step_outs = [], []
    for i in range(ND):
        ins = []
        o = st.run("decode", to_dev(xd[i:i + 1]), to_dev(synth.positions(T + i, 1)), T + i,
                   layer_outputs=ins).clone()
        step_ins.append([a.cpu().numpy() for a in ins])
        step_outs.append(o.cpu().numpy())
    torch.cuda.synchronize()
    st.block.check()
    final = [(k.cpu().numpy(), v.cpu().numpy()) for k, v in st.caches]
    full_steps = (0, 21, 42, 63)
    for i in range(ND):
        L = T + i
        for l in range(n):
            kc_o = final[l][0].copy()
            vc_o = final[l][1].copy()
            kc_o[:, L:] = 0
            vc_o[:, L:] = 0
            o_ref, k_ref, v_ref = oracle.block_forward(
                s, w_np[l], step_ins[i][l], synth.positions(L, 1), L, kc_o, vc_o,
                rows=None if i in full_steps else [])
            assert_close(final[l][0][:, L], k_ref[0], f"step {i} K layer {l}")
            assert_close(final[l][1][:, L], v_ref[0], f"step {i} V layer {l}")
            if i in full_steps:
                got = step_ins[i][l + 1] if l + 1 < n else step_outs[i]
                assert_close(got, o_ref, f"step {i} out layer {l}")


def test_prefill_stack_checks_every_layer_before_enqueueing():
    """A bad argument of the last layer is reported before any layer runs:
    every cache stays as it was; a workspace too small is refused, and the
    stack's workspace size covers the one-layer calls' plus two activation
    buffers."""
    s, n, T, C = synth.TINY, 3, 8, 32
    wl = [weights_to_dev(synth.block_weights(s, layer=l, seed=6)) for l in range(n)]
    st = LayerStack(s, wl, C, T, chain=True)
    for kc, vc in st.caches:
        kc.fill_(1.5)
        vc.fill_(-2.0)
    st._w_arr[2].w_down = None                   # the last layer is bad
    x = to_dev(synth.hidden_input(s, T, seed=6))
    pos = to_dev(synth.positions(0, T))
    with pytest.raises(blk.BlkError) as e:
        st.prefill_step(x, pos, 0)
    assert e.value.status == blk.BLK_ERR_NULL
    torch.cuda.synchronize()
    for kc, vc in st.caches:                     # nothing ran
        assert bool((kc == 1.5).all()) and bool((vc == -2.0).all())
    st._w_arr[2].w_down = st._w_arr[1].w_down
    one = blk.blk_prefill_stack_workspace_bytes(st.block.handle, T)
    assert one > blk.blk_workspace_bytes(st.block.handle, T)
    out = torch.empty((T, s.hidden), dtype=torch.float16, device="cuda")
    rc = blk.blk_prefill_stack(st.block.handle, st._w_arr, n, st._kc_arr, st._vc_arr,
                               x.data_ptr(), pos.data_ptr(), T, 0, out.data_ptr(),
                               st.ws.data_ptr(), 1024, None)
    assert rc == blk.BLK_ERR_WORKSPACE
