"""Weight-only quantized projections (INT8 with a scale per output row, int4
with a scale and a zero point per group of inputs) in all three phases,
through the C ABI, against the oracle run on the same quantized weights
(dequantized exactly in f64: oracle.dequant_i8 / dequant_u4).

The TpuOp dialect of the MLIR-compilation paper (§2.2) carries INT8 and
W4A16 weights with scales and zero points.  Each step is checked layer- and
call-local: the oracle gets the GPU's cache as it was before the call, so
the comparison does not accumulate drift.  Tolerance: relative L2 <= 1e-2
and max abs <= 5e-2 per tensor (out, k_new, v_new), the bound of every parity test;
the kernels round each weight once to fp16 (scale * (code - zero)), which
that bound covers."""
import numpy as np
import pytest
import torch

import decode_qwen2_block_gb300 as blk
import oracle
import synth
from gpu_harness import assert_close, to_dev, weights_to_dev

pytestmark = pytest.mark.gpu

# a small shape whose every K is a multiple of 32 and of 64 (int4 rules)
SMALL = synth.BlockShape(256, 4, 2, 64, 768, False)
FMT = {"i8": blk.BLK_WFMT_I8, "u4": blk.BLK_WFMT_U4}


def _mats64(q, fmt, group):
    if fmt == "i8":
        return {n: oracle.dequant_i8(m["q"], m["scale"]) for n, m in q.items()}
    return {n: oracle.dequant_u4(m["q"], m["scale"], m["zero"], group) for n, m in q.items()}


def _qdev(q):
    return {n: {k: to_dev(v) for k, v in m.items()} for n, m in q.items()}


class QBlock:
    def __init__(self, s, fmt, group, C, max_T, seed=3, layer=0):
        self.s, self.fmt, self.group = s, fmt, group
        self.w = synth.block_weights(s, layer=layer, seed=seed)     # gains and biases
        self.q = synth.quant_weights(s, fmt, layer=layer, seed=seed, group=group)
        self.m64 = _mats64(self.q, fmt, group)
        self.wd, self.qd = weights_to_dev(self.w), _qdev(self.q)
        self.block = blk.Block(s, C)
        self.qw = blk.Block.qweights(FMT[fmt], group, self.wd, self.qd)
        self.ws = torch.empty(self.block.qworkspace_bytes(max_T), dtype=torch.uint8, device="cuda")

    def run(self, phase, x, pos, L, kc, vc):
        s = self.s
        T = x.shape[0]
        out = torch.empty((T, s.hidden), dtype=torch.float16, device="cuda")
        kn = torch.empty((T, s.n_kv_heads, s.head_dim), dtype=torch.float16, device="cuda")
        vn = torch.empty_like(kn)
        self.block.run_q(phase, self.qw, to_dev(x), to_dev(pos), L, kc, vc, out, self.ws, kn, vn)
        return out, kn, vn


def _check_phase(qb, phase, x, L, kc, vc, rows=None):
    """Runs one call on the GPU and checks it against the oracle fed the
    GPU's cache as it was before the call."""
    s = qb.s
    T = x.shape[0]
    pos = synth.positions(L, T)
    kc_o, vc_o = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
    kc_o[:, L:] = 0
    vc_o[:, L:] = 0
    out, kn, vn = qb.run(phase, x, pos, L, kc, vc)
    torch.cuda.synchronize()
    qb.block.check()
    o_ref, k_ref, v_ref = oracle.block_forward(s, qb.w, x, pos, L, kc_o, vc_o, rows=rows,
                                               mats64=qb.m64)
    got = out.cpu().numpy()
    assert_close(got if rows is None else got[rows], o_ref, f"{phase} L={L} out")
    assert_close(kn.cpu().numpy(), k_ref, f"{phase} L={L} k_new")
    assert_close(vn.cpu().numpy(), v_ref, f"{phase} L={L} v_new")
    # the cache slots written in place are the returned K/V, bit for bit
    kslots = kc[:, L:L + T, :].permute(1, 0, 2).contiguous()
    assert torch.equal(kslots.view(torch.int16), kn.view(torch.int16))


@pytest.mark.parametrize("shape_name,fmt,group,T0,T1,steps", [
    ("TINY", "i8", 0, 16, 4, 8),
    ("SMALL", "u4", 64, 16, 4, 8),
    ("SMALL", "i8", 0, 40, 24, 4),
    ("QWEN2_1P5B", "i8", 0, 64, 32, 3),
    ("QWEN2_1P5B", "u4", 128, 64, 32, 3),
])
def test_quantized_phases_match_oracle(shape_name, fmt, group, T0, T1, steps):
    s = SMALL if shape_name == "SMALL" else getattr(synth, shape_name)
    C = T0 + T1 + steps + 8
    qb = QBlock(s, fmt, group, C, max(T0, T1))
    kc = torch.zeros((s.n_kv_heads, C, s.head_dim), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    x = synth.hidden_input(s, T0 + T1 + steps, seed=3)
    rows = None if s.hidden <= 256 else [0, T0 // 2, T0 - 1]
    _check_phase(qb, "prefill", x[:T0], 0, kc, vc, rows=rows)
    rows = None if s.hidden <= 256 else [0, T1 - 1]
    _check_phase(qb, "prefill_kv", x[T0:T0 + T1], T0, kc, vc, rows=rows)
    for i in range(steps):
        L = T0 + T1 + i
        _check_phase(qb, "decode", x[L:L + 1], L, kc, vc)


@pytest.mark.parametrize("fmt,group", [("i8", 0), ("u4", 128)])
def test_quantized_decode_on_long_history(fmt, group):
    """1.5B shape, decode after 4000 seeded history slots (the attention
    splits its range over many CTAs) with both formats."""
    s, L = synth.QWEN2_1P5B, 4000
    C = L + 8
    qb = QBlock(s, fmt, group, C, 1, seed=5)
    k_o, v_o = synth.kv_history(s, C, L, seed=5)
    kc, vc = to_dev(k_o), to_dev(v_o)
    x = synth.hidden_input(s, 2, seed=5)
    for i in range(2):
        _check_phase(qb, "decode", x[i:i + 1], L + i, kc, vc)


def test_quantized_decode_stack_equals_per_layer_calls():
    """blk_decode_stack_q over 3 layers gives the same bits as one
    blk_decode_q call per layer."""
    from decode_qwen2_block_gb300.stack import QuantDecodeStack
    s, n, L = synth.QWEN2_1P5B, 3, 300
    C = L + 8
    layers = [QBlock(s, "u4", 128, C, 1, seed=7, layer=l) for l in range(n)]
    hist = [synth.kv_history(s, C, L, layer=l, seed=7) for l in range(n)]
    c1 = [(to_dev(k), to_dev(v)) for k, v in hist]
    c2 = [(to_dev(k), to_dev(v)) for k, v in hist]
    st = QuantDecodeStack(s, [qb.qw for qb in layers], C, caches=c1)
    x = to_dev(synth.hidden_input(s, 1, seed=7))
    pos = to_dev(synth.positions(L, 1))
    one = st.decode_step(x, pos, L).clone()
    cur = x
    for qb, (kc, vc) in zip(layers, c2):
        out = torch.empty_like(cur)
        qb.block.run_q("decode", qb.qw, cur, pos, L, kc, vc, out, qb.ws)
        cur = out
    torch.cuda.synchronize()
    st.block.check()
    assert torch.equal(one, cur)
    for (k1, v1), (k2, v2) in zip(c1, c2):
        assert torch.equal(k1[:, L], k2[:, L]) and torch.equal(v1[:, L], v2[:, L])


def test_quantized_shape_rules_are_enforced():
    """int4 needs every K to be a multiple of 32 (packed rows 16-byte
    aligned) and of the group: the tiny shape (intermediate 688) is refused
    before anything runs; an unknown format too."""
    s = synth.TINY
    qb = QBlock(s, "i8", 0, 32, 4)
    q4 = {n: {"q": torch.zeros(1, dtype=torch.uint8, device="cuda"),
              "scale": torch.zeros(1, dtype=torch.float16, device="cuda"),
              "zero": torch.zeros(1, dtype=torch.uint8, device="cuda")} for n in blk.QMATRIX_FIELDS}
    qw = blk.Block.qweights(blk.BLK_WFMT_U4, 16, qb.wd, q4)
    kc = torch.zeros((s.n_kv_heads, 32, s.head_dim), dtype=torch.float16, device="cuda")
    x = torch.zeros((1, s.hidden), dtype=torch.float16, device="cuda")
    pos = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(blk.BlkError) as e:
        qb.block.run_q("decode", qw, x, pos, 0, kc, kc.clone(), x.clone(), qb.ws)
    assert e.value.status == blk.BLK_ERR_SHAPE
    qw.format = 7
    with pytest.raises(blk.BlkError) as e:
        qb.block.run_q("prefill", qw, x, pos, 0, kc, kc.clone(), x.clone(), qb.ws)
    assert e.value.status == blk.BLK_ERR_SHAPE
