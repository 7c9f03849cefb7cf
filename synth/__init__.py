"""Seeded synthetic inputs shared by the CPU oracle and the GPU harness.

Nothing here computes any part of the decoder block: the module draws numbers
(see ``synth.c`` for the generator's definition), names the streams each
tensor is drawn from, and lays out the shapes a block call needs.

Input recipe (every config):
  * weights ~ N(0, 0.02) fp16, one stream per (layer, tensor);
  * RMSNorm gains = 1 (stated for the tiny block and used for every shape);
  * q/k/v biases ~ N(0, 0.02) where the shape has them, no other biases;
  * hidden-state input ~ N(0, 1) fp16;
  * pre-filled KV-cache history ~ N(0, 1) fp16;
  * position_ids = cache_len + t (int64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# Stream numbering: stream = layer * 64 + tensor id; inputs use layer 4095.
TENSOR_IDS = {
    "wq": 1, "wk": 2, "wv": 3, "bq": 4, "bk": 5, "bv": 6, "wo": 7,
    "w_gate": 8, "w_up": 9, "w_down": 10,
    "x": 20, "k_hist": 21, "v_hist": 22,
    "embed": 30, "lm_head": 31, "norm_g": 32,
}
INPUT_LAYER = 4095
# Weight-only quantized matrices: codes come from the matrix's own stream,
# scales and zero points from two more streams per matrix.
QUANT_MATRICES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
for _i, _n in enumerate(QUANT_MATRICES):
    TENSOR_IDS[_n + "_scale"] = 33 + _i
    TENSOR_IDS[_n + "_zero"] = 40 + _i


def build(force: bool = False) -> str:
    """Compile libsynth.so with gcc (plain C, strict IEEE: no contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, dbl = ctypes.c_uint64, ctypes.c_double
            lib.synth_normal_f16.argtypes = [u64, u64, u64, u64, dbl, dbl, ctypes.c_void_p]
            lib.synth_normal_f16.restype = None
            lib.synth_normal_f64.argtypes = [u64, u64, u64, u64, ctypes.c_void_p]
            lib.synth_normal_f64.restype = None
            lib.synth_round_f16.argtypes = [ctypes.c_void_p, u64, ctypes.c_void_p]
            lib.synth_round_f16.restype = None
            _lib = lib
    return _lib


def stream_id(layer: int, name: str) -> int:
    return layer * 64 + TENSOR_IDS[name]


_CHUNK = 1 << 21


def normal_f16(seed: int, stream: int, shape, std: float = 1.0, mean: float = 0.0,
               threads: int | None = None) -> np.ndarray:
    """fp16 array of the given shape filled from one stream (element order = C order)."""
    lib = _load()
    n = int(np.prod(shape)) if len(tuple(shape)) else 1
    out = np.empty(n, dtype=np.uint16)
    ptr = out.ctypes.data

    def work(start):
        cnt = min(_CHUNK, n - start)
        lib.synth_normal_f16(seed, stream, start, cnt, mean, std, ptr + 2 * start)

    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        nt = threads or min(len(starts), os.cpu_count() or 1)
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(work, starts))
    return out.view(np.float16).reshape(shape)


def normal_f64(seed: int, stream: int, first: int, count: int) -> np.ndarray:
    lib = _load()
    out = np.empty(count, dtype=np.float64)
    lib.synth_normal_f64(seed, stream, first, count, out.ctypes.data)
    return out


def round_f16(values: np.ndarray) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.size, dtype=np.uint16)
    lib.synth_round_f16(v.ctypes.data, v.size, out.ctypes.data)
    return out.view(np.float16).reshape(v.shape)


@dataclass(frozen=True)
class BlockShape:
    """Shape of one decoder block (all tensors fp16, weights [out, in])."""
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    has_qkv_bias: bool
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0
    n_layers: int = 1


TINY = BlockShape(256, 4, 2, 64, 688, False)
QWEN2_1P5B = BlockShape(1536, 12, 2, 128, 8960, True, n_layers=28)
GQA_4096 = BlockShape(4096, 32, 2, 128, 11008, False, n_layers=32)


def weight_shapes(s: BlockShape) -> dict:
    H, D = s.hidden, s.head_dim
    shapes = {
        "ln1_g": (H,), "wq": (s.n_heads * D, H), "wk": (s.n_kv_heads * D, H),
        "wv": (s.n_kv_heads * D, H), "wo": (H, s.n_heads * D), "ln2_g": (H,),
        "w_gate": (s.intermediate, H), "w_up": (s.intermediate, H),
        "w_down": (H, s.intermediate),
    }
    if s.has_qkv_bias:
        shapes.update({"bq": (s.n_heads * D,), "bk": (s.n_kv_heads * D,), "bv": (s.n_kv_heads * D,)})
    return shapes


def block_weights(s: BlockShape, layer: int = 0, seed: int = 0, std: float = 0.02) -> dict:
    """Random-init weights of one layer: W ~ N(0, std), gains 1, biases ~ N(0, std)."""
    w = {}
    for name, shp in weight_shapes(s).items():
        if name in ("ln1_g", "ln2_g"):
            w[name] = np.ones(shp, dtype=np.float16)
        else:
            w[name] = normal_f16(seed, stream_id(layer, name), shp, std=std)
    return w


def quant_weights(s: BlockShape, fmt: str, layer: int = 0, seed: int = 0,
                  group: int = 128) -> dict:
    """Seeded weight-only quantized matrices of one layer: {name: {"q", "scale"
    [, "zero"]}} for the seven matrices.  Codes, scales and zero points are
    drawn directly (nothing is quantized here), sized so that the weights
    they stand for have a spread near N(0, 0.02):
      "i8": q int8 [N, K] = rint(42 z) clipped to [-127, 127]; scale fp16 [N]
            = fp16(0.02/42 * (1 + 0.1 z'))
      "u4": codes rint(7.5 + 3.5 z) clipped to [0, 15], packed two per byte
            along K (even k in the low nibble), uint8 [N, K/2]; scale fp16
            [N, K/group] = fp16(0.02/3.5 * (1 + 0.1 z')); zero uint8
            [N, K/group] = rint(7.5 + 0.5 z'') clipped to [0, 15]
    with z, z', z'' standard normal draws."""
    out = {}
    shapes = weight_shapes(s)
    for name in QUANT_MATRICES:
        N, K = shapes[name]
        z = normal_f64(seed, stream_id(layer, name), 0, N * K).reshape(N, K)
        if fmt == "i8":
            q = np.clip(np.rint(42.0 * z), -127, 127).astype(np.int8)
            zs = normal_f64(seed, stream_id(layer, name + "_scale"), 0, N)
            out[name] = {"q": q, "scale": round_f16(0.02 / 42.0 * (1.0 + 0.1 * zs))}
        elif fmt == "u4":
            if K % group or group % 2:
                raise ValueError(f"{name}: K={K} is not a multiple of the group {group}")
            codes = np.clip(np.rint(7.5 + 3.5 * z), 0, 15).astype(np.uint8)
            packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
            ng = K // group
            zs = normal_f64(seed, stream_id(layer, name + "_scale"), 0, N * ng).reshape(N, ng)
            zz = normal_f64(seed, stream_id(layer, name + "_zero"), 0, N * ng).reshape(N, ng)
            out[name] = {"q": packed,
                         "scale": round_f16(0.02 / 3.5 * (1.0 + 0.1 * zs)),
                         "zero": np.clip(np.rint(7.5 + 0.5 * zz), 0, 15).astype(np.uint8)}
        else:
            raise ValueError(f"unknown format {fmt!r}")
    return out


def hidden_input(s: BlockShape, T: int, seed: int = 0, stream_offset: int = 0) -> np.ndarray:
    """x ~ N(0, 1), shape [T, hidden]; stream_offset picks an independent draw."""
    return normal_f16(seed, stream_id(INPUT_LAYER, "x") + 64 * 4096 * stream_offset, (T, s.hidden))


def kv_history(s: BlockShape, max_ctx: int, L: int, layer: int = 0, seed: int = 0,
               sentinel: np.float16 | None = None):
    """K/V caches [Hkv, max_ctx, D] with slots [0, L) ~ N(0, 1); other slots
    hold `sentinel` (default 0)."""
    shp = (s.n_kv_heads, max_ctx, s.head_dim)
    fill = np.float16(0) if sentinel is None else np.float16(sentinel)
    k = np.full(shp, fill, dtype=np.float16)
    v = np.full(shp, fill, dtype=np.float16)
    if L > 0:
        hist_shape = (s.n_kv_heads, L, s.head_dim)
        k[:, :L, :] = normal_f16(seed, stream_id(layer, "k_hist"), hist_shape)
        v[:, :L, :] = normal_f16(seed, stream_id(layer, "v_hist"), hist_shape)
    return k, v


def positions(L: int, T: int) -> np.ndarray:
    return np.arange(L, L + T, dtype=np.int64)


QWEN2_VOCAB = 151936   # vocabulary of the 1.5B model (buddy-mlir page, prefill/decode table)


def head_weights(vocab: int, hidden: int, seed: int = 0, std: float = 0.02,
                 gain_std: float = 0.0) -> dict:
    """Embedding table and LM head ~ N(0, std) [vocab, hidden]; final RMSNorm
    gain 1 (or ~ N(1, gain_std) when gain_std > 0)."""
    w = {"embed": normal_f16(seed, stream_id(INPUT_LAYER - 1, "embed"), (vocab, hidden), std=std),
         "lm_head": normal_f16(seed, stream_id(INPUT_LAYER - 1, "lm_head"), (vocab, hidden), std=std)}
    if gain_std > 0:
        w["norm_g"] = normal_f16(seed, stream_id(INPUT_LAYER - 1, "norm_g"), (hidden,), std=gain_std,
                                 mean=1.0)
    else:
        w["norm_g"] = np.ones(hidden, dtype=np.float16)
    return w


def token_ids(vocab: int, T: int, seed: int = 0) -> np.ndarray:
    """T token ids uniform in [0, vocab) (numpy's seeded generator)."""
    return np.random.default_rng(seed).integers(0, vocab, size=T, dtype=np.int64)
