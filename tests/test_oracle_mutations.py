"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/blk_oracle.cpp (a flipped
sign, a wrong index, a dropped term, swapped operands), builds it on the CPU,
points the oracle wrapper at the mutant and checks that at least one pin of
tests/test_oracle_pins.py fails.  The real oracle is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "blk_oracle.cpp")

# (name, text in blk_oracle.cpp, replacement)
MUTATIONS = [
    ("rope sign", "v[i] = a * c - b * s;", "v[i] = a * c + b * s;"),
    ("rope partner index", "const double a = v[i], b = v[i + half];",
     "const double a = v[i], b = v[(i + 1) % D];"),
    ("rope frequency", "std::pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(D))",
     "std::pow(theta, -1.0 * static_cast<double>(i) / static_cast<double>(D))"),
    ("gqa mapping", "const int64_t g = hq / group;", "const int64_t g = hq % Hkv;"),
    ("attention scale", "const double scale = 1.0 / std::sqrt(static_cast<double>(D));",
     "const double scale = 1.0 / static_cast<double>(D);"),
    ("causal mask edge", "L + t + 1 - lo, D, D, scale", "L + t - lo, D, D, scale"),
    ("window one slot too wide", "? L + t + 1 - cfg->window : 0;", "? L + t - cfg->window : 0;"),
    ("window ignored", "(cfg->window > 0 && L + t + 1 > cfg->window)", "(false)"),
    ("dropped k bias", "linear(wk, bias ? w->bk : nullptr", "linear(wk, nullptr"),
    ("dropped rmsnorm eps", "std::sqrt(sum_sq / static_cast<double>(n) + eps)",
     "std::sqrt(sum_sq / static_cast<double>(n))"),
    ("dropped attention residual", "for (int64_t i = 0; i < H; ++i) h[i] += h2d(x[t * H + i]);",
     "for (int64_t i = 0; i < H; ++i) h[i] += 0.0;"),
    ("swapped swiglu operands", "act[j] = orc_silu(gate[j]) * up[j];",
     "act[j] = orc_silu(up[j]) * gate[j];"),
    ("transposed linear", "acc += M::val(row, i) * x[i];",
     "acc += M::val(W.p, i * n_out + o) * x[i];"),
    ("softmax max not subtracted consistently", "s[j] = std::exp(s[j] - m);", "s[j] = std::exp(s[j] - 0.5 * m);"),
    ("v stored rotated", "const uint16_t vh = encode_half(v[g * D + d]);",
     "const uint16_t vh = encode_half(k[g * D + d]);"),
    ("argmax ties to the higher index", "if (z[v] > z[best]) best = v;",
     "if (z[v] >= z[best]) best = v;"),
    ("dropped final norm gain", "orc_rmsnorm(row.data(), gain.data(), H, eps, y.data());",
     "orc_rmsnorm(row.data(), nullptr, H, eps, y.data());"),
    ("embedding row from the position", "x[t * H + i] = E[ids[t] * H + i];",
     "x[t * H + i] = E[t * H + i];"),
    ("i8: the first row's scale everywhere", "const double s = h2d(scale[o]);",
     "const double s = h2d(scale[0]);"),
    ("u4: nibble order swapped", "const int code = (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
     "const int code = (i % 2 == 0) ? (byte >> 4) : (byte & 0x0F);"),
    ("u4: zero point dropped", "(static_cast<double>(code) - static_cast<double>(zero[g]))",
     "(static_cast<double>(code) - 0.0)"),
    ("u4: the next group's scale and zero", "const int64_t g = o * ng + i / group;",
     "const int64_t g = o * ng + (i / group + 1) % ng;"),
    ("f64 weights: v projected with wk", "MatF64{m->wv}", "MatF64{m->wk}"),
    ("yarn ramp inverted", "return 1.0 - std::min(1.0, std::max(0.0, y));",
     "return std::min(1.0, std::max(0.0, y));"),
    ("yarn ramp on the element index", "static_cast<double>(i0 / 2) - low",
     "static_cast<double>(i0) - low"),
    ("yarn corr dim without the factor 2", "(2.0 * std::log(base))", "(std::log(base))"),
    ("yarn betas swapped", "orc_yarn_corr_dim(D, y->n_ctx_orig, y->beta_fast, theta);",
     "orc_yarn_corr_dim(D, y->n_ctx_orig, y->beta_slow, theta);"),
    ("yarn blend weights swapped", "const double angle = a_int * (1.0 - r) + a_orig * r;",
     "const double angle = a_orig * (1.0 - r) + a_int * r;"),
    ("yarn magnitude dropped", "? y->attn_factor * (1.0 + 0.1 * std::log(1.0 / y->freq_scale))",
     "? y->attn_factor"),
    ("yarn ignored by the block", "if (cfg->use_yarn)", "if (false)"),
]

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _run_pins():
    """Returns the names of pin tests that fail under the current oracle lib."""
    failed = []
    for fn in PIN_TESTS:
        params = getattr(fn, "pytestmark", [])
        cases = [()]
        for mark in params:
            if mark.name == "parametrize":
                cases = [c if isinstance(c, tuple) else (c,) for c in mark.args[1]]
        for case in cases:
            try:
                fn(*case)
            except Exception:  # noqa: BLE001 - any failure counts as caught
                failed.append(fn.__name__)
                break
    return failed


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert old in src, f"mutation anchor for '{name}' not found"
    mutant_src = tmp_path / "blk_oracle.cpp"
    mutant_src.write_text(src.replace(old, new, 1))
    (tmp_path / "blk_oracle.h").write_text(open(SRC.replace(".cpp", ".h")).read())
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                           str(mutant_src), "-o", str(lib)])
    saved = oracle._lib
    oracle._lib = None
    real_build = oracle.build
    try:
        oracle.build = lambda force=False: str(lib)
        failed = _run_pins()
    finally:
        oracle.build = real_build
        oracle._lib = saved
    assert failed, f"no pin caught the planted mistake '{name}'"


def test_unmutated_oracle_passes_every_pin():
    assert _run_pins() == []
