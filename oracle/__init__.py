"""Python access to the CPU oracle — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``blk_oracle.cpp`` (plain,
single-threaded f64 C++; contract and readings in ``blk_oracle.h``) through
ctypes, and shares no code with the GPU library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "blk_oracle.cpp"), os.path.join(_HERE, "blk_oracle.h")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

WEIGHT_FIELDS = ("ln1_g", "wq", "wk", "wv", "bq", "bk", "bv", "wo", "ln2_g",
                 "w_gate", "w_up", "w_down")


class OrcYarn(ctypes.Structure):
    _fields_ = [("freq_scale", ctypes.c_double), ("ext_factor", ctypes.c_double),
                ("attn_factor", ctypes.c_double), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double), ("n_ctx_orig", ctypes.c_int64)]


YARN_FIELDS = ("freq_scale", "ext_factor", "attn_factor", "beta_fast", "beta_slow", "n_ctx_orig")


class OrcConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int64), ("n_heads", ctypes.c_int64),
                ("n_kv_heads", ctypes.c_int64), ("head_dim", ctypes.c_int64),
                ("intermediate", ctypes.c_int64), ("rms_eps", ctypes.c_double),
                ("rope_theta", ctypes.c_double), ("max_ctx", ctypes.c_int64),
                ("has_qkv_bias", ctypes.c_int64), ("window", ctypes.c_int64),
                ("use_yarn", ctypes.c_int64), ("yarn", OrcYarn)]


class OrcWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


MATRIX_FIELDS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


class OrcWeightsF64(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in MATRIX_FIELDS]


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++: -O2, no FP contraction, no fast-math."""
    newest = max(os.path.getmtime(s) for s in _SRC)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", _SRC[0], "-o", tmp])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i64, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
            lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_half_to_double.restype = dbl
            lib.orc_double_to_half.argtypes = [dbl]
            lib.orc_double_to_half.restype = ctypes.c_uint16
            lib.orc_rmsnorm.argtypes = [vp, vp, i64, dbl, vp]
            lib.orc_rmsnorm.restype = None
            lib.orc_rope.argtypes = [vp, i64, dbl, dbl]
            lib.orc_rope.restype = None
            lib.orc_yarn_ramp.argtypes = [dbl, dbl, i64]
            lib.orc_yarn_ramp.restype = dbl
            lib.orc_yarn_corr_dim.argtypes = [i64, i64, dbl, dbl]
            lib.orc_yarn_corr_dim.restype = dbl
            lib.orc_rope_yarn.argtypes = [vp, i64, dbl, dbl, ctypes.POINTER(OrcYarn)]
            lib.orc_rope_yarn.restype = None
            lib.orc_linear.argtypes = [vp, vp, vp, i64, i64, vp]
            lib.orc_linear.restype = None
            lib.orc_silu.argtypes = [dbl]
            lib.orc_silu.restype = dbl
            lib.orc_attend.argtypes = [vp, vp, vp, i64, i64, i64, dbl, vp]
            lib.orc_attend.restype = None
            lib.orc_block_forward.argtypes = [ctypes.POINTER(OrcConfig), ctypes.POINTER(OrcWeights),
                                              vp, vp, i64, i64, vp, vp, vp, vp, vp, i64, vp]
            lib.orc_block_forward.restype = ctypes.c_int
            lib.orc_block_forward_f64w.argtypes = [ctypes.POINTER(OrcConfig),
                                                   ctypes.POINTER(OrcWeights),
                                                   ctypes.POINTER(OrcWeightsF64), vp, vp, i64,
                                                   i64, vp, vp, vp, vp, vp, i64, vp]
            lib.orc_block_forward_f64w.restype = ctypes.c_int
            lib.orc_dequant_i8.argtypes = [vp, vp, i64, i64, vp]
            lib.orc_dequant_i8.restype = None
            lib.orc_dequant_u4.argtypes = [vp, vp, vp, i64, i64, i64, vp]
            lib.orc_dequant_u4.restype = ctypes.c_int
            lib.orc_embed.argtypes = [vp, i64, i64, vp, i64, vp]
            lib.orc_embed.restype = ctypes.c_int
            lib.orc_lm_head.argtypes = [vp, i64, i64, vp, dbl, vp, i64, vp, vp]
            lib.orc_lm_head.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected fp16 bits, got {a.dtype}")
    return a


# ---- component functions (for the pin tests) ------------------------------

def half_to_double(bits: int) -> float:
    return _load().orc_half_to_double(int(bits))


def double_to_half(v: float) -> int:
    return int(_load().orc_double_to_half(float(v)))


def rmsnorm(x, g=None, eps: float = 1e-6) -> np.ndarray:
    x = _f64(x)
    g = None if g is None else _f64(g)
    y = np.empty_like(x)
    _load().orc_rmsnorm(x.ctypes.data, None if g is None else g.ctypes.data, x.size, eps, y.ctypes.data)
    return y


def rope(v, pos: float, theta: float = 10000.0) -> np.ndarray:
    v = _f64(v).copy()
    _load().orc_rope(v.ctypes.data, v.size, float(pos), float(theta))
    return v


def _yarn(y) -> "OrcYarn":
    """OrcYarn from a dict with the YARN_FIELDS keys."""
    return OrcYarn(*(float(y[k]) if k != "n_ctx_orig" else int(y[k]) for k in YARN_FIELDS))


def yarn_ramp(low: float, high: float, i0: int) -> float:
    return _load().orc_yarn_ramp(float(low), float(high), int(i0))


def yarn_corr_dim(n_dims: int, n_ctx_orig: int, n_rot: float, base: float) -> float:
    return _load().orc_yarn_corr_dim(int(n_dims), int(n_ctx_orig), float(n_rot), float(base))


def rope_yarn(v, pos: float, yarn: dict, theta: float = 10000.0) -> np.ndarray:
    """rotate_half RoPE with YaRN frequencies and magnitude; ``yarn`` holds
    the YARN_FIELDS keys."""
    v = _f64(v).copy()
    y = _yarn(yarn)
    _load().orc_rope_yarn(v.ctypes.data, v.size, float(pos), float(theta), ctypes.byref(y))
    return v


def linear(W, x, b=None) -> np.ndarray:
    W = _u16(W)
    x = _f64(x)
    n_out, n_in = W.shape
    bb = None if b is None else _u16(b)
    y = np.empty(n_out, dtype=np.float64)
    _load().orc_linear(W.ctypes.data, None if bb is None else bb.ctypes.data, x.ctypes.data,
                       n_out, n_in, y.ctypes.data)
    return y


def silu(z: float) -> float:
    return _load().orc_silu(float(z))


def attend(q, K, V, scale: float) -> np.ndarray:
    """One query head against rows of K/V (fp16 [n_keys, D])."""
    q = _f64(q)
    K, V = _u16(K), _u16(V)
    n, D = K.shape
    o = np.empty(D, dtype=np.float64)
    _load().orc_attend(q.ctypes.data, K.ctypes.data, V.ctypes.data, n, D, D, float(scale), o.ctypes.data)
    return o


# ---- the whole block --------------------------------------------------------

def block_forward(shape, weights: dict, x, pos, L: int, k_cache, v_cache, max_ctx: int | None = None,
                  rows=None, mats64: dict | None = None, window: int = 0,
                  yarn: dict | None = None):
    """Run the block for T = len(x) new tokens on top of L history slots.

    ``shape`` is a ``synth.BlockShape``.  ``k_cache``/``v_cache`` (fp16
    [Hkv, max_ctx, D]) are updated in place.  Returns (out, k_new, v_new);
    ``out`` covers ``rows`` (all rows when None).  ``mats64``, if given, holds
    the seven matrices as f64 values (e.g. dequantized weights, see
    ``dequant_i8`` / ``dequant_u4``); ``weights`` then supplies only the gains
    and biases.  ``window`` > 0: sliding-window attention over the last
    ``window`` slots (the query's own slot included); 0 = full attention.
    ``yarn``: YaRN RoPE parameters (the YARN_FIELDS keys), None = plain RoPE."""
    lib = _load()
    x = _u16(x)
    T = x.shape[0]
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    kc, vc = k_cache.view(np.uint16), v_cache.view(np.uint16)
    if not (kc.flags.c_contiguous and vc.flags.c_contiguous):
        raise ValueError("caches must be C-contiguous")
    C = kc.shape[1] if max_ctx is None else max_ctx
    cfg = OrcConfig(shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.intermediate,
                    shape.rms_eps, shape.rope_theta, C, 1 if shape.has_qkv_bias else 0, int(window),
                    0 if yarn is None else 1, OrcYarn() if yarn is None else _yarn(yarn))
    keep = {}
    wts = OrcWeights()
    for name in WEIGHT_FIELDS:
        arr = weights.get(name)
        if mats64 is not None and name in MATRIX_FIELDS:
            arr = None
        if arr is None:
            setattr(wts, name, None)
            continue
        arr = _u16(arr)
        keep[name] = arr
        setattr(wts, name, arr.ctypes.data)
    Hkv, D, H = shape.n_kv_heads, shape.head_dim, shape.hidden
    k_new = np.empty((T, Hkv, D), dtype=np.uint16)
    v_new = np.empty((T, Hkv, D), dtype=np.uint16)
    if rows is None:
        rows_arr, n_rows = None, T
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows_arr.size
    out = np.empty((n_rows, H), dtype=np.uint16)
    args = (x.ctypes.data, pos.ctypes.data, T, L, kc.ctypes.data, vc.ctypes.data,
            k_new.ctypes.data, v_new.ctypes.data,
            None if rows_arr is None else rows_arr.ctypes.data, n_rows, out.ctypes.data)
    if mats64 is None:
        rc = lib.orc_block_forward(ctypes.byref(cfg), ctypes.byref(wts), *args)
    else:
        m64 = OrcWeightsF64()
        for name in MATRIX_FIELDS:
            arr = _f64(mats64[name])
            keep["m64_" + name] = arr
            setattr(m64, name, arr.ctypes.data)
        rc = lib.orc_block_forward_f64w(ctypes.byref(cfg), ctypes.byref(wts), ctypes.byref(m64),
                                        *args)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return out.view(np.float16), k_new.view(np.float16), v_new.view(np.float16)


# ---- weight-only quantized projections -----------------------------------------

def dequant_i8(q, scale) -> np.ndarray:
    """f64 w[o][i] = scale[o] * q[o][i] (q int8 [N, K], scale fp16 [N])."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = _u16(scale)
    N, K = q.shape
    if s.shape != (N,):
        raise ValueError("one scale per output row")
    w = np.empty((N, K), dtype=np.float64)
    _load().orc_dequant_i8(q.ctypes.data, s.ctypes.data, N, K, w.ctypes.data)
    return w


def dequant_u4(packed, scale, zero, group: int) -> np.ndarray:
    """f64 w[o][i] = scale[o][i//group] * (code(o, i) - zero[o][i//group]);
    packed uint8 [N, K/2] holds two 4-bit codes per byte, the even i in the
    low nibble; scale fp16 and zero uint8 are [N, K/group]."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    s = _u16(scale)
    z = np.ascontiguousarray(zero, dtype=np.uint8)
    N, K2 = packed.shape
    K = 2 * K2
    if K % group or s.shape != (N, K // group) or z.shape != (N, K // group):
        raise ValueError("scale / zero must be [N, K/group] with K a multiple of group")
    w = np.empty((N, K), dtype=np.float64)
    if _load().orc_dequant_u4(packed.ctypes.data, s.ctypes.data, z.ctypes.data, N, K, group,
                              w.ctypes.data) != 0:
        raise ValueError("oracle rejected the arguments")
    return w


# ---- around the block stack ---------------------------------------------------

def embed(E, ids) -> np.ndarray:
    """x[t] = E[ids[t]] (fp16 rows)."""
    E = _u16(E)
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    V, H = E.shape
    x = np.empty((ids.size, H), dtype=np.uint16)
    if _load().orc_embed(E.ctypes.data, V, H, ids.ctypes.data, ids.size, x.ctypes.data) != 0:
        raise ValueError("token id outside the vocabulary")
    return x.view(np.float16)


def lm_head(x, g, W, eps: float = 1e-6, want_logits: bool = True):
    """Final RMSNorm, LM head and greedy token of each row of x (fp16 [T, H]).
    Returns (logits f64 [T, vocab] or None, token int64 [T])."""
    x, g, W = _u16(x), _u16(g), _u16(W)
    T, H = x.shape
    V = W.shape[0]
    logits = np.empty((T, V), dtype=np.float64) if want_logits else None
    token = np.empty(T, dtype=np.int64)
    rc = _load().orc_lm_head(x.ctypes.data, T, H, g.ctypes.data, float(eps), W.ctypes.data, V,
                             None if logits is None else logits.ctypes.data, token.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return logits, token
