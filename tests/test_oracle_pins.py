"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test names the property it checks.  None of them re-types an oracle
formula and compares it with itself: they use closed forms, invariants,
special cases, the page's printed constants, an independent fp16 conversion
(numpy) and a brute-force matrix restatement on small cases.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
from brute_block import block as brute_block

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fp16 codec

def test_half_decode_every_pattern_matches_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    ours = np.array([oracle.half_to_double(b) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[np.isinf(ref)], ref[np.isinf(ref)])


def test_half_encode_matches_numpy_rne():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000), rng.standard_normal(5000) * 1e-5, rng.standard_normal(5000) * 2e4,
        (np.arange(1, 2049) + 0.5) * 2.0 ** -10, (np.arange(1, 1024) + 0.5) * 2.0 ** -24,
        [0.0, -0.0, 65504.0, 65519.999, 65520.0, 7e4, 2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -14 * (1 - 2.0 ** -12)],
    ])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    ours = np.array([oracle.double_to_half(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(ours, ref)


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    c, n, eps = 3.0, 64, 1e-6
    y = oracle.rmsnorm(np.full(n, c), eps=eps)
    assert np.allclose(y, c / math.sqrt(c * c + eps), rtol=0, atol=1e-15)


def test_rmsnorm_scale_invariance_and_unit_rms():
    x = synth.normal_f64(0, 100, 0, 1536)
    y1 = oracle.rmsnorm(x, eps=1e-6)
    y2 = oracle.rmsnorm(1000.0 * x, eps=1e-6)
    assert np.allclose(y1, y2, rtol=1e-6, atol=0)
    ms = np.mean(x * x)
    assert math.isclose(math.sqrt(np.mean(y1 * y1)), math.sqrt(ms / (ms + 1e-6)), rel_tol=1e-12)


def test_rmsnorm_gain_is_elementwise():
    x = synth.normal_f64(0, 101, 0, 32)
    g = np.arange(1, 33, dtype=np.float64)
    assert np.allclose(oracle.rmsnorm(x, g), oracle.rmsnorm(x) * g, rtol=1e-15, atol=0)


# -------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    # ds4.c study notes, part 4 'RoPE rotation': pos = 0 gives angle 0, no rotation
    v = synth.normal_f64(0, 102, 0, 128)
    assert np.array_equal(oracle.rope(v, 0.0), v)


def test_rope_one_hot_pins_pairing_sign_and_frequency():
    D, theta, p = 8, 10000.0, 3.0
    for i in range(D // 2):
        w = theta ** (-2.0 * i / D)
        e = np.zeros(D)
        e[i] = 1.0
        out = oracle.rope(e, p, theta)
        want = np.zeros(D)
        want[i] = math.cos(p * w)            # first half keeps cos
        want[i + D // 2] = math.sin(p * w)   # partner at i + D/2 gets +sin
        assert np.allclose(out, want, atol=1e-15), i
        e = np.zeros(D)
        e[i + D // 2] = 1.0
        out = oracle.rope(e, p, theta)
        want = np.zeros(D)
        want[i] = -math.sin(p * w)
        want[i + D // 2] = math.cos(p * w)
        assert np.allclose(out, want, atol=1e-15), i


def test_rope_preserves_pair_norms_and_composes():
    D = 128
    v = synth.normal_f64(0, 103, 0, D)
    a, b = 123.0, 4567.0
    r = oracle.rope(v, a)
    n0 = v[: D // 2] ** 2 + v[D // 2:] ** 2
    n1 = r[: D // 2] ** 2 + r[D // 2:] ** 2
    assert np.allclose(n0, n1, rtol=1e-12)
    assert np.allclose(oracle.rope(r, b), oracle.rope(v, a + b), atol=1e-9)


def test_rope_scores_depend_on_relative_position_only():
    D = 64
    q = synth.normal_f64(0, 104, 0, D)
    k = synth.normal_f64(0, 105, 0, D)
    s1 = oracle.rope(q, 50.0) @ oracle.rope(k, 20.0)
    s2 = oracle.rope(q, 1030.0) @ oracle.rope(k, 1000.0)
    assert math.isclose(s1, s2, rel_tol=1e-9, abs_tol=1e-9)


# ------------------------------------------------------------ linear / silu

def test_linear_one_hot_selects_a_column_and_bias_adds():
    W = synth.normal_f16(0, 106, (24, 40))
    for j in (0, 7, 39):
        e = np.zeros(40)
        e[j] = 1.0
        assert np.array_equal(oracle.linear(W, e), W[:, j].astype(np.float64))
    b = synth.normal_f16(0, 107, (24,))
    y = oracle.linear(np.zeros((24, 40), np.float16), np.ones(40), b)
    assert np.array_equal(y, b.astype(np.float64))


def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert math.isclose(oracle.silu(40.0), 40.0, rel_tol=1e-15)
    assert abs(oracle.silu(-40.0)) < 1e-15
    for z in (0.3, 1.7, 5.0):
        # silu(z) - silu(-z) = z for every z
        assert math.isclose(oracle.silu(z) - oracle.silu(-z), z, rel_tol=1e-14)
        assert math.isclose(oracle.silu(z), z * (0.5 + 0.5 * math.tanh(z / 2)), rel_tol=1e-14)


# --------------------------------------------------------------- attention

def test_attend_single_key_returns_v():
    # ds4.c study notes, part 4 'first token': attention over itself only
    D = 64
    q = synth.normal_f64(0, 108, 0, D)
    K = synth.normal_f16(0, 109, (1, D))
    V = synth.normal_f16(0, 110, (1, D))
    assert np.array_equal(oracle.attend(q, K, V, 1 / 8), V[0].astype(np.float64))


def test_attend_identical_keys_gives_mean_of_v():
    D, n = 128, 37
    q = synth.normal_f64(0, 111, 0, D)
    K = np.tile(synth.normal_f16(0, 112, (1, D)), (n, 1))
    V = synth.normal_f16(0, 113, (n, D))
    o = oracle.attend(q, K, V, 1 / math.sqrt(D))
    assert np.allclose(o, V.astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-15)


def test_attend_two_key_closed_form_pins_scale():
    D, c = 64, 5.0
    q = np.zeros(D)
    q[0] = c
    K = np.zeros((2, D), np.float16)
    K[0, 0] = 1.0
    V = np.zeros((2, D), np.float16)
    V[0, :] = 2.0
    V[1, :] = -1.0
    o = oracle.attend(q, K, V, 1 / math.sqrt(D))
    e = math.exp(c / math.sqrt(D))
    assert np.allclose(o, (2.0 * e - 1.0) / (e + 1.0), rtol=1e-14)


def test_attend_split_merge_equals_one_pass():
    # log-sum-exp merge of two halves equals attention over the whole range
    D, n, a = 64, 50, 19
    q = synth.normal_f64(0, 114, 0, D)
    K = synth.normal_f16(0, 115, (n, D))
    V = synth.normal_f16(0, 116, (n, D))
    s = 1 / 8

    def stats(Kp):
        sc = (Kp.astype(np.float64) @ q) * s
        m = sc.max()
        return m, np.exp(sc - m).sum()

    o1, o2 = oracle.attend(q, K[:a], V[:a], s), oracle.attend(q, K[a:], V[a:], s)
    (m1, l1), (m2, l2) = stats(K[:a]), stats(K[a:])
    m = max(m1, m2)
    w1, w2 = l1 * math.exp(m1 - m), l2 * math.exp(m2 - m)
    merged = (w1 * o1 + w2 * o2) / (w1 + w2)
    assert np.allclose(merged, oracle.attend(q, K, V, s), rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ whole block

def _tiny_case(T, L, max_ctx=64, seed=0, sentinel=-7.0):
    s = synth.TINY
    w = synth.block_weights(s, seed=seed)
    x = synth.hidden_input(s, T, seed=seed)
    kc, vc = synth.kv_history(s, max_ctx, L, seed=seed, sentinel=sentinel)
    return s, w, x, synth.positions(L, T), kc, vc


@pytest.mark.parametrize("T,L", [(16, 0), (4, 16), (1, 20), (7, 9)])
def test_block_matches_bruteforce_restatement(T, L):
    s, w, x, pos, kc, vc = _tiny_case(T, L)
    bo, bk, bv = brute_block(s, w, x, pos, L, kc.copy(), vc.copy())
    out, kn, vn = oracle.block_forward(s, w, x, pos, L, kc, vc)
    # K/V are rounded from f64 in both; allow a one-ulp difference where the
    # two summation orders straddle a rounding boundary
    assert np.max(np.abs(kn.astype(np.float64) - bk.astype(np.float64))) <= 2.0 ** -10
    assert np.max(np.abs(vn.astype(np.float64) - bv.astype(np.float64))) <= 2.0 ** -10
    d = np.abs(out.astype(np.float64) - bo.astype(np.float64))
    assert d.max() <= 2.0 ** -8          # at most one fp16 ulp at |out| < 8
    assert np.mean(out.view(np.uint16) == bo.view(np.uint16)) > 0.99


def test_block_cache_placement_and_untouched_slots():
    T, L, C = 5, 11, 40
    s, w, x, pos, kc, vc = _tiny_case(T, L, max_ctx=C)
    k0, v0 = kc.copy(), vc.copy()
    out, kn, vn = oracle.block_forward(s, w, x, pos, L, kc, vc)
    assert np.array_equal(kc[:, L:L + T, :].view(np.uint16), kn.transpose(1, 0, 2).view(np.uint16))
    assert np.array_equal(vc[:, L:L + T, :].view(np.uint16), vn.transpose(1, 0, 2).view(np.uint16))
    for arr, ref in ((kc, k0), (vc, v0)):
        assert np.array_equal(arr[:, :L].view(np.uint16), ref[:, :L].view(np.uint16))
        assert np.array_equal(arr[:, L + T:].view(np.uint16), ref[:, L + T:].view(np.uint16))


def test_block_residual_passthrough_with_zero_output_weights():
    s, w, x, pos, kc, vc = _tiny_case(6, 3)
    w = dict(w, wo=np.zeros_like(w["wo"]), w_down=np.zeros_like(w["w_down"]))
    out, _, _ = oracle.block_forward(s, w, x, pos, 3, kc, vc)
    assert np.array_equal(out.view(np.uint16), x.view(np.uint16))


def test_block_kv_from_bias_only():
    # zero K/V weights: k = RoPE(bk) at each position, v = bv
    s = synth.BlockShape(64, 2, 1, 32, 48, True)
    w = synth.block_weights(s, seed=3)
    w["wk"] = np.zeros_like(w["wk"])
    w["wv"] = np.zeros_like(w["wv"])
    T = 3
    x = synth.hidden_input(s, T, seed=3)
    kc, vc = synth.kv_history(s, 8, 0)
    pos = np.array([0, 5, 9], np.int64)
    _, kn, vn = oracle.block_forward(s, w, x, pos, 0, kc, vc)
    bk = w["bk"].astype(np.float64)
    D = 32
    for t, p in enumerate(pos):
        c = np.cos(p * 10000.0 ** (-np.arange(0, D, 2) / D))
        sn = np.sin(p * 10000.0 ** (-np.arange(0, D, 2) / D))
        want = np.concatenate([bk[:16] * c - bk[16:] * sn, bk[16:] * c + bk[:16] * sn])
        assert np.array_equal(kn[t, 0].view(np.uint16), want.astype(np.float16).view(np.uint16)) or \
            np.max(np.abs(kn[t, 0].astype(np.float64) - want)) <= 2.0 ** -11
        assert np.array_equal(vn[t, 0].view(np.uint16), w["bv"].view(np.uint16))


def test_block_gqa_mapping_and_output_orientation():
    # V of kv head g is the constant g + 1, so every query head's attention
    # output is the constant of its kv head; Wo is a permutation matrix, Wd = 0.
    s = synth.BlockShape(256, 4, 2, 64, 32, False)
    w = synth.block_weights(s, seed=5)
    w["wv"] = np.zeros_like(w["wv"])
    T, L, C = 2, 6, 16
    x = synth.hidden_input(s, T, seed=5)
    kc, vc = synth.kv_history(s, C, L, seed=5)
    vc[0, :L] = 1.0
    vc[1, :L] = 2.0
    w["w_down"] = np.zeros_like(w["w_down"])
    perm = (np.arange(256) * 5 + 3) % 256          # not an involution
    Wo = np.zeros((256, 256), np.float16)
    Wo[np.arange(256), perm] = 1.0                 # out[o] = attn[perm[o]]
    w["wo"] = Wo
    # new rows contribute v = 0, so restrict to keys where that is harmless:
    # expected attn = (sum over history of const * p) = const * (mass on history)
    out, _, _ = oracle.block_forward(s, w, x, synth.positions(L, T), L, kc, vc)
    # recompute history mass with the component functions is circular; instead
    # check the structure: within each kv group the output of Wo is constant per
    # group and group 1 is exactly twice group 0 (same softmax mass per head is
    # not implied, so compare ratios per query head)
    attn_est = out.astype(np.float64) - x.astype(np.float64)   # [T, 256] = attn[perm]
    attn = np.empty_like(attn_est)
    attn[:, perm] = attn_est
    heads = attn.reshape(T, 4, 64)
    # inside one head all 64 dims equal (V is constant across d)
    assert np.allclose(heads, heads[..., :1], atol=2.0 ** -9)
    # heads 0,1 (kv 0) see constant 1, heads 2,3 (kv 1) see 2; the new rows
    # add a little mass on v = 0, so values are in (0, c]
    assert np.all(heads[:, 0:2] <= 1.0 + 2 ** -9) and np.all(heads[:, 0:2] > 0.5)
    assert np.all(heads[:, 2:4] <= 2.0 + 2 ** -8) and np.all(heads[:, 2:4] > 1.0)


def test_block_causality():
    T, L = 8, 4
    s, w, x, pos, kc, vc = _tiny_case(T, L)
    out1, _, _ = oracle.block_forward(s, w, x, pos, L, kc.copy(), vc.copy())
    x2 = x.copy()
    x2[5:] = synth.hidden_input(s, 3, seed=9)
    out2, _, _ = oracle.block_forward(s, w, x2, pos, L, kc.copy(), vc.copy())
    assert np.array_equal(out1[:5].view(np.uint16), out2[:5].view(np.uint16))
    assert not np.array_equal(out1[5:].view(np.uint16), out2[5:].view(np.uint16))


def test_block_position_shift_invariance():
    T = 12
    s, w, x, pos, kc, vc = _tiny_case(T, 0)
    out1, k1, _ = oracle.block_forward(s, w, x, pos, 0, kc.copy(), vc.copy())
    out2, k2, _ = oracle.block_forward(s, w, x, pos + 1000, 0, kc.copy(), vc.copy())
    assert not np.array_equal(k1.view(np.uint16), k2.view(np.uint16))
    # only relative positions reach the scores; K is rounded after rotation,
    # so allow the resulting tiny difference
    assert np.max(np.abs(out1.astype(np.float64) - out2.astype(np.float64))) <= 2.0 ** -7


def test_block_rows_subset_equals_full():
    s, w, x, pos, kc, vc = _tiny_case(9, 5)
    full, kf, vf = oracle.block_forward(s, w, x, pos, 5, kc.copy(), vc.copy())
    rows = [8, 0, 4]
    sub, ks, vs = oracle.block_forward(s, w, x, pos, 5, kc.copy(), vc.copy(), rows=rows)
    assert np.array_equal(sub.view(np.uint16), full[rows].view(np.uint16))
    assert np.array_equal(ks.view(np.uint16), kf.view(np.uint16))


def test_phase_chain_identities_bit_exact():
    """prefill(T) == prefill(T-k) -> prefill_kv(k) == prefill(T-1) -> decode
    (the three-phase split of the TopOp/TpuOp paper, section 4.1)."""
    T, C = 16, 32
    s, w, x, pos, _, _ = _tiny_case(T, 0, max_ctx=C)
    kc0, vc0 = synth.kv_history(s, C, 0)
    full, kf, vf = oracle.block_forward(s, w, x, pos, 0, kc0, vc0)

    for k in (1, 4, 7):
        kc, vc = synth.kv_history(s, C, 0)
        o1, _, _ = oracle.block_forward(s, w, x[:T - k], pos[:T - k], 0, kc, vc)
        o2, _, _ = oracle.block_forward(s, w, x[T - k:], pos[T - k:], T - k, kc, vc)
        assert np.array_equal(np.concatenate([o1, o2]).view(np.uint16), full.view(np.uint16))
        assert np.array_equal(kc.view(np.uint16), kc0.view(np.uint16))
        assert np.array_equal(vc.view(np.uint16), vc0.view(np.uint16))

    kc, vc = synth.kv_history(s, C, 0)
    outs = [oracle.block_forward(s, w, x[:T - 4], pos[:T - 4], 0, kc, vc)[0]]
    for t in range(T - 4, T):    # four decode steps
        outs.append(oracle.block_forward(s, w, x[t:t + 1], pos[t:t + 1], t, kc, vc)[0])
    assert np.array_equal(np.concatenate(outs).view(np.uint16), full.view(np.uint16))


def test_oracle_rejects_bad_arguments():
    s, w, x, pos, kc, vc = _tiny_case(4, 0, max_ctx=8)
    with pytest.raises(ValueError):
        oracle.block_forward(s, w, x, pos, 6, kc, vc)          # 6 + 4 > max_ctx
    with pytest.raises(ValueError):
        oracle.block_forward(s, w, x, pos, 0, kc, vc, rows=[4])


# ------------------------------------------------------ page constants

def test_page_param_count_pins_the_1p5b_shape():
    """The packed-parameter count printed by the buddy-mlir runtime equals the
    element count of 28 blocks of the 1.5B shape (with q/k/v bias), the
    embedding, final norm, an untied LM head and a head_dim/2 RoPE buffer."""
    c = json.load(open(os.path.join(GOLDEN, "page_constants.json")))
    s = synth.QWEN2_1P5B
    assert s.head_dim == c["head_dim_named_HiddenSize"]
    assert s.n_kv_heads == c["kv_heads_named_HeadNum"]
    per_layer = sum(int(np.prod(v)) for v in synth.weight_shapes(s).values())
    total = s.n_layers * per_layer + 2 * c["MaxVocabSize"] * s.hidden + s.hidden + s.head_dim // 2
    assert total == c["ParamsSize"]
    # K and V per layer make the 56 cache fields of the prefill return struct
    assert 2 * s.n_layers == c["kv_fields_in_prefill_returns"]
    assert c["kv_cache_shape"][1:] == [s.n_kv_heads, c["MaxTokenLength"], s.head_dim]


def test_page_gqa_example_shape():
    c = json.load(open(os.path.join(GOLDEN, "gqa_example_shape.json")))
    s = synth.GQA_4096
    assert (s.n_layers, s.hidden, s.n_kv_heads, s.head_dim) == (
        c["num_layers"], c["hidden_size"], c["kv_head"], c["head_dim"])


# ------------------------------------------------ embedding, LM head, argmax

def test_embed_matches_array_indexing_and_rejects_bad_ids():
    rng = np.random.default_rng(11)
    E = rng.standard_normal((97, 24)).astype(np.float16)
    ids = np.array([0, 96, 5, 5, 40], dtype=np.int64)
    x = oracle.embed(E, ids)
    assert np.array_equal(x.view(np.uint16), E[ids].view(np.uint16))
    for bad in ([-1], [97], [3, 1 << 40]):
        with pytest.raises(ValueError):
            oracle.embed(E, bad)


def test_lm_head_closed_form_for_rank_one_weights_and_constant_input():
    # x = a (constant row): RMSNorm gives a / sqrt(a^2 + eps) * g; rows of W
    # that are c_v * u give logits c_v * (a / sqrt(a^2 + eps)) * sum(u * g).
    H, V, a, eps = 64, 33, 0.75, 1e-6
    rng = np.random.default_rng(12)
    u = rng.integers(-3, 4, size=H).astype(np.float16)
    g = (1 + rng.integers(-2, 3, size=H) / 8).astype(np.float16)
    c = rng.integers(-5, 6, size=V).astype(np.float64)
    W = (c[:, None] * u[None, :].astype(np.float64)).astype(np.float16)
    x = np.full((1, H), a, dtype=np.float16)
    logits, token = oracle.lm_head(x, g, W, eps=eps)
    dot = float(np.sum(u.astype(np.float64) * g.astype(np.float64)))
    want = c * (a / math.sqrt(a * a + eps)) * dot
    assert np.allclose(logits[0], want, rtol=1e-12, atol=1e-12)
    assert token[0] == int(np.flatnonzero(want == want.max())[0])


def test_lm_head_row_permutation_permutes_logits():
    rng = np.random.default_rng(13)
    H, V = 48, 71
    W = (rng.standard_normal((V, H)) * 0.1).astype(np.float16)
    g = np.ones(H, np.float16)
    x = rng.standard_normal((3, H)).astype(np.float16)
    perm = rng.permutation(V)
    l1, t1 = oracle.lm_head(x, g, W)
    l2, t2 = oracle.lm_head(x, g, W[perm])
    assert np.array_equal(l2, l1[:, perm])
    assert np.array_equal(perm[t2], t1)


def test_lm_head_rmsnorm_scale_invariance_with_zero_eps():
    rng = np.random.default_rng(14)
    H, V = 40, 29
    W = (rng.standard_normal((V, H)) * 0.1).astype(np.float16)
    g = (1 + rng.standard_normal(H) * 0.1).astype(np.float16)
    x = rng.standard_normal((2, H)).astype(np.float16)
    l1, _ = oracle.lm_head(x, g, W, eps=0.0)
    l2, _ = oracle.lm_head((x.astype(np.float64) * 4).astype(np.float16), g, W, eps=0.0)
    assert np.allclose(l1, l2, rtol=1e-13, atol=1e-13)


def test_lm_head_ties_go_to_the_lowest_index():
    rng = np.random.default_rng(15)
    H, V = 32, 50
    x = rng.standard_normal((1, H)).astype(np.float16)
    g = np.ones(H, np.float16)
    W = np.zeros((V, H), np.float16)
    best = np.sign(x[0]).astype(np.float16)          # the row with the largest dot product
    for v in (17, 3, 41):                            # three equal maxima
        W[v] = best
    W[8] = (best.astype(np.float64) * 0.5).astype(np.float16)
    _, token = oracle.lm_head(x, g, W)
    assert token[0] == 3


# ------------------------------------------- weight-only quantized projections

def test_dequant_i8_hand_computed_rows():
    """w = s[o] * q: signs, the clip values and a different scale per row."""
    q = np.array([[1, -2, 127], [0, 5, -127]], dtype=np.int8)
    s = np.array([0.5, 0.25], dtype=np.float16)
    want = np.array([[0.5, -1.0, 63.5], [0.0, 1.25, -31.75]])
    assert np.array_equal(oracle.dequant_i8(q, s), want)


def test_dequant_u4_nibble_order_groups_and_zero_points():
    """Two codes per byte, the even input in the low nibble; each group of
    inputs has its own scale and zero point."""
    packed = np.array([[0x21, 0xF0, 0x3C],
                       [0x00, 0xFF, 0x87]], dtype=np.uint8)
    # group = 2: groups are inputs (0,1), (2,3), (4,5)
    scale = np.array([[1.0, 0.5, 2.0],
                      [0.25, 1.0, -1.0]], dtype=np.float16)
    zero = np.array([[1, 8, 3],
                     [0, 15, 7]], dtype=np.uint8)
    # row 0 codes: 1, 2 | 0, 15 | 12, 3 ; row 1 codes: 0, 0 | 15, 15 | 7, 8
    want = np.array([[0.0, 1.0, -4.0, 3.5, 18.0, 0.0],
                     [0.0, 0.0, 0.0, 0.0, -0.0, -1.0]])
    got = oracle.dequant_u4(packed, scale, zero, group=2)
    assert np.array_equal(got, want)
    with pytest.raises(ValueError):     # K = 6 is not a multiple of 4
        oracle.dequant_u4(packed, scale[:, :1], zero[:, :1], group=4)


def _exact_quant_case(s, fmt, seed):
    """Quantized matrices whose weights fp16 holds exactly (power-of-two
    scales, codes within +-15), with the fp16 copy of those weights."""
    rng = np.random.default_rng(seed)
    mats, f16 = {}, {}
    for name in oracle.MATRIX_FIELDS:
        N, K = synth.weight_shapes(s)[name]
        if fmt == "i8":
            q = rng.integers(-15, 16, size=(N, K)).astype(np.int8)
            sc = np.full(N, 2.0 ** -8, dtype=np.float16)
            w = oracle.dequant_i8(q, sc)
        else:
            group = 16
            codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
            packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
            sc = np.full((N, K // group), 2.0 ** -7, dtype=np.float16)
            z = rng.integers(0, 16, size=(N, K // group)).astype(np.uint8)
            w = oracle.dequant_u4(packed, sc, z, group)
        assert np.array_equal(w.astype(np.float16).astype(np.float64), w)   # exact in fp16
        mats[name] = w
        f16[name] = w.astype(np.float16)
    return mats, f16


@pytest.mark.parametrize("fmt", ["i8", "u4"])
def test_block_with_f64_weights_equals_the_fp16_block_when_exact(fmt):
    """Dequantized weights that fp16 holds exactly give, through the f64-weight
    entry, the same bits as the pinned fp16 block: prefill and a decode on
    history (out, k_new, v_new and every cache slot)."""
    s = synth.TINY
    base = synth.block_weights(s, seed=3)
    mats, f16 = _exact_quant_case(s, fmt, seed=3)
    w16 = dict(base, **f16)
    for T, L in ((6, 0), (1, 9)):
        x = synth.hidden_input(s, T, seed=3, stream_offset=T)
        pos = synth.positions(L, T)
        ka, va = synth.kv_history(s, 32, L, seed=3)
        kb, vb = ka.copy(), va.copy()
        ra = oracle.block_forward(s, w16, x, pos, L, ka, va)
        rb = oracle.block_forward(s, base, x, pos, L, kb, vb, mats64=mats)
        for a, b in zip(ra, rb):
            assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
        assert np.array_equal(ka.view(np.uint16), kb.view(np.uint16))
        assert np.array_equal(va.view(np.uint16), vb.view(np.uint16))


@pytest.mark.parametrize("fmt", ["i8", "u4"])
def test_block_with_dequantized_weights_matches_bruteforce(fmt):
    """Seeded quantized weights (not exact in fp16) through the f64-weight
    entry against the independent numpy restatement fed the same f64 matrices,
    at the one-ulp tolerance of the fp16 block's brute-force pin."""
    s = synth.TINY
    T, L = 4, 16
    base = synth.block_weights(s, seed=5)
    qw = synth.quant_weights(s, fmt, seed=5, group=16)
    mats = {}
    for name, d in qw.items():
        mats[name] = (oracle.dequant_i8(d["q"], d["scale"]) if fmt == "i8"
                      else oracle.dequant_u4(d["q"], d["scale"], d["zero"], 16))
    x = synth.hidden_input(s, T, seed=5)
    pos = synth.positions(L, T)
    kc, vc = synth.kv_history(s, 64, L, seed=5, sentinel=-7.0)
    bo, bk, bv = brute_block(s, dict(base, **mats), x, pos, L, kc.copy(), vc.copy())
    out, kn, vn = oracle.block_forward(s, base, x, pos, L, kc, vc, mats64=mats)
    assert np.max(np.abs(kn.astype(np.float64) - bk.astype(np.float64))) <= 2.0 ** -10
    assert np.max(np.abs(vn.astype(np.float64) - bv.astype(np.float64))) <= 2.0 ** -10
    assert np.abs(out.astype(np.float64) - bo.astype(np.float64)).max() <= 2.0 ** -8
    assert np.mean(out.view(np.uint16) == bo.view(np.uint16)) > 0.99


# ------------------------------------------------------------ sliding window
# The ds4.c study notes name a sliding-window ("swa") layer forward without
# stating its window; the reading pinned here: the query in slot p attends
# the last W slots, [max(0, p - W + 1), p].

@pytest.mark.parametrize("T,L", [(16, 0), (4, 16), (1, 30)])
def test_window_covering_the_context_equals_full_attention(T, L):
    s, w, x, pos, kc, vc = _tiny_case(T, L)
    full = oracle.block_forward(s, w, x, pos, L, kc.copy(), vc.copy())
    for W in (L + T, L + T + 5, 64):
        win = oracle.block_forward(s, w, x, pos, L, kc.copy(), vc.copy(), window=W)
        for a, b in zip(full, win):
            assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_window_of_one_gives_each_row_the_output_of_a_lone_token():
    """With W = 1 a row attends only its own slot: softmax over one key is
    1, so the attention output is the row's own V whatever q, the history or
    the position; the block output equals a one-token prefill of that row."""
    T, L = 6, 20
    s, w, x, pos, kc, vc = _tiny_case(T, L)
    out, kn, vn = oracle.block_forward(s, w, x, pos, L, kc, vc, window=1)
    for t in range(T):
        k1, v1 = synth.kv_history(s, 8, 0)
        o1, _, _ = oracle.block_forward(s, w, x[t:t + 1], synth.positions(0, 1), 0, k1, v1)
        assert np.array_equal(out[t:t + 1].view(np.uint16), o1.view(np.uint16))


def test_slots_outside_the_window_are_never_read():
    T, L, W = 5, 30, 12
    s, w, x, pos, kc, vc = _tiny_case(T, L)
    ref = oracle.block_forward(s, w, x, pos, L, kc.copy(), vc.copy(), window=W)
    junk_k, junk_v = kc.copy(), vc.copy()
    lo = L + 1 - W                      # the first row's first visible slot
    rng = np.random.default_rng(5)
    junk_k[:, :lo] = rng.normal(0, 50, junk_k[:, :lo].shape).astype(np.float16)
    junk_v[:, :lo] = np.float16(np.nan)
    got = oracle.block_forward(s, w, x, pos, L, junk_k, junk_v, window=W)
    for a, b in zip(ref, got):
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    # and one slot more does change it: the window edge is where it says
    junk_v[:, lo] = np.float16(3.0)
    moved = oracle.block_forward(s, w, x, pos, L, kc.copy(), junk_v, window=W)
    assert not np.array_equal(moved[0][0].view(np.uint16), ref[0][0].view(np.uint16))


@pytest.mark.parametrize("T,L,W", [(16, 0, 5), (7, 9, 4), (4, 16, 10), (1, 25, 3)])
def test_window_matches_band_masked_bruteforce(T, L, W):
    s, w, x, pos, kc, vc = _tiny_case(T, L)
    bo, bk, bv = brute_block(s, w, x, pos, L, kc.copy(), vc.copy(), window=W)
    out, kn, vn = oracle.block_forward(s, w, x, pos, L, kc, vc, window=W)
    d = np.abs(out.astype(np.float64) - bo.astype(np.float64))
    assert d.max() <= 2.0 ** -8
    assert np.mean(out.view(np.uint16) == bo.view(np.uint16)) > 0.99
    full = oracle.block_forward(s, w, x, pos, L, kc.copy(), vc.copy())[0]
    assert not np.array_equal(full.view(np.uint16), out.view(np.uint16))


# ------------------------------------------------------------ YaRN RoPE
# The ds4.c study notes (Part 4, "Trace 1: YaRN frequency scaling") give the
# ramp and the correction dimension; the blend of the original and scaled
# frequencies and the magnitude factor are readings (oracle/blk_oracle.h).

YARN = {"freq_scale": 0.125, "ext_factor": 1.0, "attn_factor": 1.3, "beta_fast": 32.0,
        "beta_slow": 1.0, "n_ctx_orig": 4096}


def test_yarn_ramp_closed_forms():
    low, high = 7.0, 19.0
    assert oracle.yarn_ramp(low, high, 2 * 7) == 1.0        # start of the ramp: original
    assert oracle.yarn_ramp(low, high, 2 * 19) == 0.0       # its end: scaled
    assert oracle.yarn_ramp(low, high, 2 * 13) == 0.5       # half way
    assert oracle.yarn_ramp(low, high, 0) == 1.0 and oracle.yarn_ramp(low, high, 126) == 0.0
    # the pair index is i0 / 2 (i0 counts elements): i0 = 2 * 10 sits at 1 - 3/12
    assert oracle.yarn_ramp(low, high, 20) == 0.75
    # high == low: a step at low (the 0.001 floor on the width)
    assert oracle.yarn_ramp(5.0, 5.0, 10) == 1.0 and oracle.yarn_ramp(5.0, 5.0, 12) == 0.0


@pytest.mark.parametrize("n_dims,ctx,n_rot,base", [(128, 4096, 32.0, 10000.0),
                                                   (128, 4096, 1.0, 10000.0),
                                                   (64, 32768, 4.0, 1e6)])
def test_yarn_corr_dim_is_where_a_pair_turns_n_rot_times(n_dims, ctx, n_rot, base):
    """Defining property: pair d's wavelength 2 pi base^(2d / n_dims) fits
    n_rot times into the original context."""
    d = oracle.yarn_corr_dim(n_dims, ctx, n_rot, base)
    wavelength = 2.0 * math.pi * base ** (2.0 * d / n_dims)
    assert math.isclose(ctx / wavelength, n_rot, rel_tol=1e-12)
    # more turns = a higher frequency = a lower pair index
    assert oracle.yarn_corr_dim(n_dims, ctx, 2 * n_rot, base) < d


def test_yarn_off_equals_plain_rope():
    v = synth.normal_f64(0, 120, 0, 128)
    off = dict(YARN, freq_scale=1.0, ext_factor=0.0, attn_factor=1.0)
    for p in (0.0, 1.0, 777.0, 40000.0):
        assert np.array_equal(oracle.rope_yarn(v, p, off), oracle.rope(v, p))


def test_yarn_without_the_ramp_is_position_interpolation():
    """ext_factor = 0: every pair runs at freq_scale times its frequency, i.e.
    plain RoPE at position pos * freq_scale (exact for a power-of-two scale)."""
    v = synth.normal_f64(0, 121, 0, 128)
    pi_only = dict(YARN, ext_factor=0.0, attn_factor=1.0)
    for p in (3.0, 1000.0, 50000.0):
        assert np.array_equal(oracle.rope_yarn(v, p, pi_only), oracle.rope(v, p * 0.125))


def test_yarn_pairs_below_and_above_the_ramp():
    """Pairs below corr_dim(beta_fast) keep the original angle, pairs above
    corr_dim(beta_slow) take the interpolated one; all are scaled by the
    magnitude m = attn_factor * (1 + 0.1 ln(1 / freq_scale))."""
    D, p = 128, 9000.0
    low = oracle.yarn_corr_dim(D, 4096, 32.0, 10000.0)
    high = oracle.yarn_corr_dim(D, 4096, 1.0, 10000.0)
    assert 10 < low < high < 60
    m = 1.3 * (1.0 + 0.1 * math.log(8.0))
    v = synth.normal_f64(0, 122, 0, D)
    got = oracle.rope_yarn(v, p, YARN)
    orig, interp = oracle.rope(v, p), oracle.rope(v, p * 0.125)
    h = D // 2
    for i in range(h):
        idx = [i, i + h]
        if i <= math.floor(low):
            assert np.allclose(got[idx], m * orig[idx], rtol=1e-12, atol=1e-12), i
        elif i >= math.ceil(high):
            assert np.allclose(got[idx], m * interp[idx], rtol=1e-12, atol=1e-12), i


def test_yarn_pair_on_the_ramp_turns_by_the_blended_angle():
    D, p = 128, 5.0                    # small angles: read back with atan2
    low = oracle.yarn_corr_dim(D, 4096, 32.0, 10000.0)
    high = oracle.yarn_corr_dim(D, 4096, 1.0, 10000.0)
    m = 1.3 * (1.0 + 0.1 * math.log(8.0))
    for i in range(math.ceil(low), math.floor(high) + 1):
        r = oracle.yarn_ramp(low, high, 2 * i)
        assert 0.0 < r < 1.0
        e = np.zeros(D)
        e[i] = 1.0
        out = oracle.rope_yarn(e, p, YARN)
        a = p * 10000.0 ** (-2.0 * i / D)
        want = 0.125 * a * (1.0 - r) + a * r
        assert math.isclose(math.atan2(out[i + D // 2], out[i]), want, rel_tol=1e-12), i
        assert math.isclose(math.hypot(out[i], out[i + D // 2]), m, rel_tol=1e-12), i


def test_block_with_yarn_off_or_interpolating_equals_plain_block():
    """The block threads YaRN through RoPE of q and k only: switched off it
    is the plain block bit for bit, and pure interpolation by 1/2 at even
    positions is the plain block at half those positions."""
    T, L = 5, 9
    s, w, x, pos, kc, vc = _tiny_case(T, L)
    off = dict(YARN, freq_scale=1.0, ext_factor=0.0, attn_factor=1.0)
    plain = oracle.block_forward(s, w, x, pos, L, kc.copy(), vc.copy())
    got = oracle.block_forward(s, w, x, pos, L, kc.copy(), vc.copy(), yarn=off)
    for a, b in zip(plain, got):
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    half = dict(off, freq_scale=0.5)
    got = oracle.block_forward(s, w, x, 2 * pos, L, kc.copy(), vc.copy(), yarn=half)
    for a, b in zip(plain, got):
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    # and the full YaRN rotation does change the block
    on = oracle.block_forward(s, w, x, pos + 5000, L, kc.copy(), vc.copy(), yarn=YARN)
    ref = oracle.block_forward(s, w, x, pos + 5000, L, kc.copy(), vc.copy())
    assert not np.array_equal(on[0].view(np.uint16), ref[0].view(np.uint16))
