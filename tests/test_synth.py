"""The seeded generator: determinism, counter independence, distribution, and
its fp16 rounding checked against numpy's independent conversion."""
import numpy as np
import pytest

import synth


def test_deterministic_and_counter_based():
    a = synth.normal_f16(0, 7, (5000,))
    b = synth.normal_f16(0, 7, (5000,))
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    # element i depends only on (seed, stream, i): a slice drawn from an offset
    # equals the same slice of the full draw
    tail = synth.normal_f64(0, 7, 1234, 100)
    full = synth.normal_f64(0, 7, 0, 1334)
    assert np.array_equal(tail, full[1234:])


def test_streams_and_seeds_differ():
    a = synth.normal_f64(0, 1, 0, 1000)
    b = synth.normal_f64(0, 2, 0, 1000)
    c = synth.normal_f64(1, 1, 0, 1000)
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.1
    assert abs(np.corrcoef(a, c)[0, 1]) < 0.1


def test_threaded_fill_matches_single_thread():
    n = (1 << 21) * 3 + 17
    a = synth.normal_f16(3, 9, (n,), std=0.02, threads=4)
    b = synth.normal_f16(3, 9, (n,), std=0.02, threads=1)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_standard_normal_moments():
    z = synth.normal_f64(0, 11, 0, 400_000)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1.0) < 0.01
    # fourth moment of N(0,1) is 3
    assert abs((z ** 4).mean() - 3.0) < 0.05


def test_fp16_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(100_000),
        rng.standard_normal(20_000) * 1e-5,          # subnormal range
        rng.standard_normal(20_000) * 3e4,           # near overflow
        # exact ties between neighbouring fp16 values, both parities
        (np.arange(1, 2049, dtype=np.float64) + 0.5) * 2.0 ** -10,
        (np.arange(1, 1024, dtype=np.float64) + 0.5) * 2.0 ** -24,
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -25, 2.0 ** -26, np.inf, -np.inf],
    ])
    ours = synth.round_f16(vals).view(np.uint16)
    ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_quant_weights_are_seeded_and_in_range():
    a = synth.quant_weights(synth.TINY, "i8", seed=1)
    b = synth.quant_weights(synth.TINY, "i8", seed=1)
    c = synth.quant_weights(synth.TINY, "i8", seed=2)
    shapes = synth.weight_shapes(synth.TINY)
    for n in synth.QUANT_MATRICES:
        N, K = shapes[n]
        assert a[n]["q"].shape == (N, K) and a[n]["q"].dtype == np.int8
        assert np.array_equal(a[n]["q"], b[n]["q"]) and not np.array_equal(a[n]["q"], c[n]["q"])
        assert a[n]["q"].min() >= -127 and a[n]["scale"].shape == (N,)
        assert a[n]["scale"].dtype == np.float16 and (a[n]["scale"] > 0).all()
    u = synth.quant_weights(synth.TINY, "u4", group=16)
    for n in synth.QUANT_MATRICES:
        N, K = shapes[n]
        assert u[n]["q"].shape == (N, K // 2) and u[n]["q"].dtype == np.uint8
        assert u[n]["scale"].shape == (N, K // 16) and u[n]["zero"].shape == (N, K // 16)
        assert u[n]["zero"].max() <= 15
    # distinct matrices draw from distinct streams
    assert not np.array_equal(u["wk"]["q"], u["wv"]["q"])
    with pytest.raises(ValueError):            # intermediate 688 is not a multiple of 128
        synth.quant_weights(synth.TINY, "u4", group=128)
