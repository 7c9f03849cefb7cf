"""GB300 decoder-block library: Python binding of libblk.so.

The binding only marshals arguments: every step of the block runs in the
library's CUDA kernels (see include/blk.h for the contract).  It loads the
in-tree ``libblk.so`` and raises if it has not been built; there is no CPU or
PyTorch fallback.

Low-level functions carry the C names (``blk_create``, ``blk_prefill``,
``blk_prefill_kv``, ``blk_decode``, ...) and take plain integers for device
pointers.  ``Block`` is a convenience wrapper taking torch CUDA tensors.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libblk.so")

BLK_OK = 0
BLK_ERR_NULL = -1
BLK_ERR_ALIGN = -2
BLK_ERR_SHAPE = -3
BLK_ERR_CACHE_OVERFLOW = -4
BLK_ERR_WORKSPACE = -5
BLK_ERR_CUDA = -6
BLK_ERR_DEVICE_TIMEOUT = -7
BLK_ERR_POSITION = -8
BLK_ERR_DEVICE = -9
BLK_ERR_SCRATCH_LIMIT = -10
BLK_ERR_TOKEN = -11
BLK_STATIC_SCRATCH_BYTES = 1 << 20
BLK_FLAG_CHAIN = 1
BLK_WFMT_F16, BLK_WFMT_I8, BLK_WFMT_U4 = 0, 1, 2

EXPORTED = ("blk_create", "blk_destroy", "blk_set_flags", "blk_workspace_bytes", "blk_prefill",
            "blk_prefill_kv", "blk_decode", "blk_check", "blk_status_str", "blk_timing",
            "blk_timing_collect", "blk_timing_read", "blk_decode_static", "blk_decode_stack",
            "blk_set_trace", "blk_embed", "blk_lm_head_workspace_bytes", "blk_lm_head",
            "blk_decode_batch_workspace_bytes", "blk_decode_batch",
            "blk_decode_batch_stack_workspace_bytes", "blk_decode_batch_stack",
            "blk_wait_probe", "blk_qworkspace_bytes", "blk_prefill_q", "blk_prefill_kv_q",
            "blk_decode_q", "blk_decode_stack_q", "blk_set_window", "blk_set_rope_yarn",
            "blk_prefill_stack_workspace_bytes", "blk_prefill_stack")
BLK_N_KERNELS = 16

WEIGHT_FIELDS = ("ln1_g", "wq", "wk", "wv", "bq", "bk", "bv", "wo", "ln2_g", "w_gate", "w_up",
                 "w_down")


class BlkConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("max_ctx", ctypes.c_int64),
                ("has_qkv_bias", ctypes.c_int32)]


class BlkWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class BlkQMatrix(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("zero", ctypes.c_void_p)]


QMATRIX_FIELDS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


class BlkQWeights(ctypes.Structure):
    _fields_ = ([("format", ctypes.c_int32), ("group", ctypes.c_int32)] +
                [(n, ctypes.c_void_p) for n in ("ln1_g", "bq", "bk", "bv", "ln2_g")] +
                [(n, BlkQMatrix) for n in QMATRIX_FIELDS])


YARN_FIELDS = ("freq_scale", "ext_factor", "attn_factor", "beta_fast", "beta_slow", "n_ctx_orig")


class BlkYarn(ctypes.Structure):
    _fields_ = [("freq_scale", ctypes.c_double), ("ext_factor", ctypes.c_double),
                ("attn_factor", ctypes.c_double), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double), ("n_ctx_orig", ctypes.c_int64)]


class BlkError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {blk_status_str(status)} ({status})" if what else
                         f"{blk_status_str(status)} ({status})")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libblk.so (once).  Raises if it is missing: build it first with
    ``python -c 'import __graft_entry__ as g; g.build()'``."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libblk.so not found at {path}; the CUDA library must be built "
                           "(decode_qwen2_block_gb300/build.py) — there is no fallback")
    lib = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.blk_create.argtypes = [ctypes.POINTER(BlkConfig), ctypes.POINTER(vp)]
    lib.blk_create.restype = i32
    lib.blk_destroy.argtypes = [vp]
    lib.blk_destroy.restype = None
    lib.blk_set_flags.argtypes = [vp, ctypes.c_uint32]
    lib.blk_set_flags.restype = i32
    lib.blk_set_window.argtypes = [vp, i64]
    lib.blk_set_window.restype = i32
    lib.blk_set_rope_yarn.argtypes = [vp, ctypes.POINTER(BlkYarn)]
    lib.blk_set_rope_yarn.restype = i32
    lib.blk_workspace_bytes.argtypes = [vp, i64]
    lib.blk_workspace_bytes.restype = ctypes.c_size_t
    lib.blk_prefill.argtypes = [vp, ctypes.POINTER(BlkWeights), vp, vp, i64, vp, vp, vp, vp, vp,
                                vp, ctypes.c_size_t, vp]
    lib.blk_prefill.restype = i32
    lib.blk_prefill_kv.argtypes = [vp, ctypes.POINTER(BlkWeights), vp, vp, i64, i64, vp, vp, vp,
                                   vp, vp, vp, ctypes.c_size_t, vp]
    lib.blk_prefill_kv.restype = i32
    lib.blk_decode.argtypes = [vp, ctypes.POINTER(BlkWeights), vp, vp, i64, vp, vp, vp, vp, vp,
                               vp, ctypes.c_size_t, vp]
    lib.blk_decode.restype = i32
    lib.blk_set_trace.argtypes = [vp, vp, ctypes.c_size_t]
    lib.blk_set_trace.restype = i32
    lib.blk_decode_stack.argtypes = [vp, ctypes.POINTER(BlkWeights), i32, ctypes.POINTER(vp),
                                     ctypes.POINTER(vp), vp, vp, i64, vp, ctypes.POINTER(vp),
                                     ctypes.POINTER(vp), vp, ctypes.c_size_t, vp]
    lib.blk_decode_stack.restype = i32
    lib.blk_decode_static.argtypes = [vp, ctypes.POINTER(BlkWeights), vp, vp, i64, vp, vp, vp, vp,
                                      vp, vp]
    lib.blk_decode_static.restype = i32
    lib.blk_wait_probe.argtypes = [vp, vp, ctypes.c_uint64, vp]
    lib.blk_wait_probe.restype = i32
    lib.blk_check.argtypes = [vp, vp]
    lib.blk_check.restype = i32
    lib.blk_status_str.argtypes = [i32]
    lib.blk_status_str.restype = ctypes.c_char_p
    lib.blk_timing.argtypes = [vp, i32]
    lib.blk_timing.restype = i32
    lib.blk_timing_collect.argtypes = [vp, vp]
    lib.blk_timing_collect.restype = i32
    lib.blk_timing_read.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_char_p)]
    lib.blk_timing_read.restype = i32
    lib.blk_decode_batch_workspace_bytes.argtypes = [vp, i64]
    lib.blk_decode_batch_workspace_bytes.restype = ctypes.c_size_t
    lib.blk_decode_batch.argtypes = [vp, ctypes.POINTER(BlkWeights), vp, vp, vp, i64, i64, vp, vp,
                                     vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.blk_decode_batch.restype = i32
    lib.blk_prefill_stack_workspace_bytes.argtypes = [vp, i64]
    lib.blk_prefill_stack_workspace_bytes.restype = ctypes.c_size_t
    lib.blk_prefill_stack.argtypes = [vp, ctypes.POINTER(BlkWeights), i32, ctypes.POINTER(vp),
                                      ctypes.POINTER(vp), vp, vp, i64, i64, vp, vp, ctypes.c_size_t,
                                      vp]
    lib.blk_prefill_stack.restype = i32
    lib.blk_decode_batch_stack_workspace_bytes.argtypes = [vp, i64]
    lib.blk_decode_batch_stack_workspace_bytes.restype = ctypes.c_size_t
    lib.blk_decode_batch_stack.argtypes = [vp, ctypes.POINTER(BlkWeights), i32, ctypes.POINTER(vp),
                                           ctypes.POINTER(vp), vp, vp, vp, i64, i64, vp, vp,
                                           ctypes.c_size_t, vp]
    lib.blk_decode_batch_stack.restype = i32
    lib.blk_embed.argtypes = [vp, vp, i64, vp, i64, vp, vp]
    lib.blk_embed.restype = i32
    lib.blk_lm_head_workspace_bytes.argtypes = [vp]
    lib.blk_lm_head_workspace_bytes.restype = ctypes.c_size_t
    lib.blk_lm_head.argtypes = [vp, vp, i64, vp, vp, i64, vp, vp, vp, ctypes.c_size_t, vp]
    lib.blk_lm_head.restype = i32
    qw = ctypes.POINTER(BlkQWeights)
    lib.blk_qworkspace_bytes.argtypes = [vp, i64]
    lib.blk_qworkspace_bytes.restype = ctypes.c_size_t
    lib.blk_prefill_q.argtypes = [vp, qw, vp, vp, i64, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.blk_prefill_q.restype = i32
    lib.blk_prefill_kv_q.argtypes = [vp, qw, vp, vp, i64, i64, vp, vp, vp, vp, vp, vp,
                                     ctypes.c_size_t, vp]
    lib.blk_prefill_kv_q.restype = i32
    lib.blk_decode_q.argtypes = [vp, qw, vp, vp, i64, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.blk_decode_q.restype = i32
    lib.blk_decode_stack_q.argtypes = [vp, qw, i32, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, vp,
                                       i64, vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp,
                                       ctypes.c_size_t, vp]
    lib.blk_decode_stack_q.restype = i32
    _lib = lib
    return lib


# ---- C-named entry points (plain integer pointers) ---------------------------

def blk_status_str(status: int) -> str:
    return load().blk_status_str(int(status)).decode()


def blk_create(cfg: BlkConfig) -> int:
    h = ctypes.c_void_p()
    rc = load().blk_create(ctypes.byref(cfg), ctypes.byref(h))
    if rc != BLK_OK:
        raise BlkError(rc, "blk_create")
    return h.value


def blk_destroy(handle: int) -> None:
    load().blk_destroy(handle)


def blk_set_flags(handle: int, flags: int) -> int:
    return load().blk_set_flags(handle, flags)


def blk_set_window(handle: int, window: int) -> int:
    return load().blk_set_window(handle, window)


def blk_set_rope_yarn(handle: int, yarn) -> int:
    """yarn: a BlkYarn, or None for plain RoPE."""
    return load().blk_set_rope_yarn(handle, None if yarn is None else ctypes.byref(yarn))


def blk_workspace_bytes(handle: int, max_T: int) -> int:
    return load().blk_workspace_bytes(handle, max_T)


def blk_prefill(handle, w: BlkWeights, x, pos, T, k_cache, v_cache, out, k_new, v_new, ws,
                ws_bytes, stream) -> int:
    return load().blk_prefill(handle, ctypes.byref(w), x, pos, T, k_cache, v_cache, out, k_new,
                              v_new, ws, ws_bytes, stream)


def blk_prefill_kv(handle, w: BlkWeights, x, pos, T, cache_len, k_cache, v_cache, out, k_new,
                   v_new, ws, ws_bytes, stream) -> int:
    return load().blk_prefill_kv(handle, ctypes.byref(w), x, pos, T, cache_len, k_cache, v_cache,
                                 out, k_new, v_new, ws, ws_bytes, stream)


def blk_decode(handle, w: BlkWeights, x, pos, cache_len, k_cache, v_cache, out, k_new, v_new, ws,
               ws_bytes, stream) -> int:
    return load().blk_decode(handle, ctypes.byref(w), x, pos, cache_len, k_cache, v_cache, out,
                             k_new, v_new, ws, ws_bytes, stream)


def blk_set_trace(handle, buf_ptr, nbytes) -> int:
    return load().blk_set_trace(handle, buf_ptr, nbytes)


def blk_decode_stack(handle, w_array, n_layers, k_caches, v_caches, x, pos, cache_len, out,
                     k_new, v_new, ws, ws_bytes, stream) -> int:
    """w_array: (BlkWeights * n); k_caches/v_caches/k_new/v_new: (c_void_p * n) or None."""
    return load().blk_decode_stack(handle, w_array, n_layers, k_caches, v_caches, x, pos,
                                   cache_len, out, k_new, v_new, ws, ws_bytes, stream)


def blk_decode_static(handle, w: BlkWeights, x, pos, cache_len, k_cache, v_cache, out, k_new,
                      v_new, stream) -> int:
    """Decode with the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/blk.h)."""
    return load().blk_decode_static(handle, ctypes.byref(w), x, pos, cache_len, k_cache, v_cache,
                                    out, k_new, v_new, stream)


def blk_qworkspace_bytes(handle, max_T: int) -> int:
    return load().blk_qworkspace_bytes(handle, max_T)


def blk_prefill_q(handle, w: BlkQWeights, x, pos, T, k_cache, v_cache, out, k_new, v_new, ws,
                  ws_bytes, stream) -> int:
    return load().blk_prefill_q(handle, ctypes.byref(w), x, pos, T, k_cache, v_cache, out, k_new,
                                v_new, ws, ws_bytes, stream)


def blk_prefill_kv_q(handle, w: BlkQWeights, x, pos, T, cache_len, k_cache, v_cache, out, k_new,
                     v_new, ws, ws_bytes, stream) -> int:
    return load().blk_prefill_kv_q(handle, ctypes.byref(w), x, pos, T, cache_len, k_cache, v_cache,
                                   out, k_new, v_new, ws, ws_bytes, stream)


def blk_decode_q(handle, w: BlkQWeights, x, pos, cache_len, k_cache, v_cache, out, k_new, v_new,
                 ws, ws_bytes, stream) -> int:
    return load().blk_decode_q(handle, ctypes.byref(w), x, pos, cache_len, k_cache, v_cache, out,
                               k_new, v_new, ws, ws_bytes, stream)


def blk_decode_stack_q(handle, w_array, n_layers, k_caches, v_caches, x, pos, cache_len, out,
                       k_new, v_new, ws, ws_bytes, stream) -> int:
    return load().blk_decode_stack_q(handle, w_array, n_layers, k_caches, v_caches, x, pos,
                                     cache_len, out, k_new, v_new, ws, ws_bytes, stream)


def blk_decode_batch_workspace_bytes(handle, max_B: int) -> int:
    return load().blk_decode_batch_workspace_bytes(handle, max_B)


def blk_decode_batch(handle, w: BlkWeights, x, pos, cache_lens, B, max_cache_len, k_cache,
                     v_cache, out, k_new, v_new, ws, ws_bytes, stream) -> int:
    return load().blk_decode_batch(handle, ctypes.byref(w), x, pos, cache_lens, B, max_cache_len,
                                   k_cache, v_cache, out, k_new, v_new, ws, ws_bytes, stream)


def blk_wait_probe(handle, flag_ptr, limit_ns: int, stream) -> int:
    """One kernel waiting (bounded) for the device int at flag_ptr; see include/blk.h."""
    return load().blk_wait_probe(handle, flag_ptr, limit_ns, stream)


def blk_prefill_stack_workspace_bytes(handle, max_T: int) -> int:
    return load().blk_prefill_stack_workspace_bytes(handle, max_T)


def blk_prefill_stack(handle, w_array, n_layers, k_caches, v_caches, x, pos, T, cache_len, out,
                      ws, ws_bytes, stream) -> int:
    """w_array: (BlkWeights * n); k_caches/v_caches: (c_void_p * n)."""
    return load().blk_prefill_stack(handle, w_array, n_layers, k_caches, v_caches, x, pos, T,
                                    cache_len, out, ws, ws_bytes, stream)


def blk_decode_batch_stack_workspace_bytes(handle, max_B: int) -> int:
    return load().blk_decode_batch_stack_workspace_bytes(handle, max_B)


def blk_decode_batch_stack(handle, w_array, n_layers, k_caches, v_caches, x, pos, cache_lens, B,
                           max_cache_len, out, ws, ws_bytes, stream) -> int:
    """w_array: (BlkWeights * n); k_caches/v_caches: (c_void_p * n)."""
    return load().blk_decode_batch_stack(handle, w_array, n_layers, k_caches, v_caches, x, pos,
                                         cache_lens, B, max_cache_len, out, ws, ws_bytes, stream)


def blk_embed(handle, table, vocab, ids, T, x, stream) -> int:
    return load().blk_embed(handle, table, vocab, ids, T, x, stream)


def blk_lm_head_workspace_bytes(handle) -> int:
    return load().blk_lm_head_workspace_bytes(handle)


def blk_lm_head(handle, x, T, norm_g, w_lm, vocab, logits, tokens, ws, ws_bytes, stream) -> int:
    return load().blk_lm_head(handle, x, T, norm_g, w_lm, vocab, logits, tokens, ws, ws_bytes,
                              stream)


def blk_check(handle, stream) -> int:
    return load().blk_check(handle, stream)


def blk_timing(handle, on: bool) -> int:
    return load().blk_timing(handle, 1 if on else 0)


def blk_timing_collect(handle, stream) -> int:
    return load().blk_timing_collect(handle, stream)


def blk_timing_read(handle, kernel: int):
    """Returns (name, total_ms, launches) or None for an unknown id."""
    ms, n, name = ctypes.c_double(), ctypes.c_int64(), ctypes.c_char_p()
    rc = load().blk_timing_read(handle, kernel, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(name))
    if rc != BLK_OK:
        return None
    return name.value.decode(), ms.value, n.value


# ---- torch convenience wrapper ------------------------------------------------

def _ptr(t):
    return None if t is None else t.data_ptr()


class Block:
    """One block shape on the current CUDA device.

    ``shape`` needs the attributes hidden, n_heads, n_kv_heads, head_dim,
    intermediate, has_qkv_bias, rms_eps, rope_theta."""

    def __init__(self, shape, max_ctx: int, chain: bool = False):
        self.shape = shape
        self.max_ctx = int(max_ctx)
        self.cfg = BlkConfig(shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                             shape.intermediate, shape.rms_eps, shape.rope_theta, self.max_ctx,
                             1 if shape.has_qkv_bias else 0)
        self.handle = blk_create(self.cfg)
        if chain:
            blk_set_flags(self.handle, BLK_FLAG_CHAIN)

    def close(self):
        if getattr(self, "handle", None):
            blk_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_chain(self, on: bool):
        blk_set_flags(self.handle, BLK_FLAG_CHAIN if on else 0)

    def set_window(self, window: int):
        """Sliding-window attention over the last `window` slots (0 = full)."""
        rc = blk_set_window(self.handle, window)
        if rc != BLK_OK:
            raise BlkError(rc, "blk_set_window")

    def set_rope_yarn(self, yarn: dict | None):
        """YaRN RoPE with the YARN_FIELDS parameters (None: plain RoPE)."""
        y = None if yarn is None else BlkYarn(*(yarn[k] for k in YARN_FIELDS))
        rc = blk_set_rope_yarn(self.handle, y)
        if rc != BLK_OK:
            raise BlkError(rc, "blk_set_rope_yarn")

    def workspace_bytes(self, max_T: int) -> int:
        return blk_workspace_bytes(self.handle, max_T)

    @staticmethod
    def weights(wdict) -> BlkWeights:
        w = BlkWeights()
        for n in WEIGHT_FIELDS:
            setattr(w, n, _ptr(wdict.get(n)))
        return w

    @staticmethod
    def qweights(fmt: int, group: int, wdict, qdict) -> BlkQWeights:
        """Quantized weights: gains and biases from ``wdict`` (fp16 tensors),
        the seven matrices from ``qdict[name] = {"q", "scale"[, "zero"]}``
        (device tensors in the layouts of include/blk.h)."""
        w = BlkQWeights()
        w.format, w.group = fmt, group
        for n in ("ln1_g", "bq", "bk", "bv", "ln2_g"):
            setattr(w, n, _ptr(wdict.get(n)))
        for n in QMATRIX_FIELDS:
            m = getattr(w, n)
            m.q, m.scale, m.zero = (_ptr(qdict[n]["q"]), _ptr(qdict[n]["scale"]),
                                    _ptr(qdict[n].get("zero")))
        return w

    def qworkspace_bytes(self, max_T: int) -> int:
        return blk_qworkspace_bytes(self.handle, max_T)

    def run_q(self, phase: str, w: BlkQWeights, x, pos, cache_len: int, k_cache, v_cache, out,
              ws, k_new=None, v_new=None, stream=None):
        """One call of the quantized prefill / prefill_kv / decode."""
        nb = ws.numel() * ws.element_size()
        st = self._stream(stream)
        if phase == "prefill":
            rc = blk_prefill_q(self.handle, w, _ptr(x), _ptr(pos), x.shape[0], _ptr(k_cache),
                               _ptr(v_cache), _ptr(out), _ptr(k_new), _ptr(v_new), _ptr(ws), nb, st)
        elif phase == "prefill_kv":
            rc = blk_prefill_kv_q(self.handle, w, _ptr(x), _ptr(pos), x.shape[0], cache_len,
                                  _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(k_new),
                                  _ptr(v_new), _ptr(ws), nb, st)
        elif phase == "decode":
            rc = blk_decode_q(self.handle, w, _ptr(x), _ptr(pos), cache_len, _ptr(k_cache),
                              _ptr(v_cache), _ptr(out), _ptr(k_new), _ptr(v_new), _ptr(ws), nb, st)
        else:
            raise ValueError(phase)
        if rc != BLK_OK:
            raise BlkError(rc, f"blk_{phase}_q")

    @staticmethod
    def _stream(stream):
        import torch
        s = torch.cuda.current_stream() if stream is None else stream
        return s.cuda_stream

    def prefill(self, w: BlkWeights, x, pos, k_cache, v_cache, out, ws, k_new=None, v_new=None,
                stream=None):
        rc = blk_prefill(self.handle, w, _ptr(x), _ptr(pos), x.shape[0], _ptr(k_cache),
                         _ptr(v_cache), _ptr(out), _ptr(k_new), _ptr(v_new), _ptr(ws),
                         ws.numel() * ws.element_size(), self._stream(stream))
        if rc != BLK_OK:
            raise BlkError(rc, "blk_prefill")

    def prefill_kv(self, w: BlkWeights, x, pos, cache_len: int, k_cache, v_cache, out, ws,
                   k_new=None, v_new=None, stream=None):
        rc = blk_prefill_kv(self.handle, w, _ptr(x), _ptr(pos), x.shape[0], cache_len,
                            _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(k_new), _ptr(v_new),
                            _ptr(ws), ws.numel() * ws.element_size(), self._stream(stream))
        if rc != BLK_OK:
            raise BlkError(rc, "blk_prefill_kv")

    def decode(self, w: BlkWeights, x, pos, cache_len: int, k_cache, v_cache, out, ws,
               k_new=None, v_new=None, stream=None):
        rc = blk_decode(self.handle, w, _ptr(x), _ptr(pos), cache_len, _ptr(k_cache),
                        _ptr(v_cache), _ptr(out), _ptr(k_new), _ptr(v_new), _ptr(ws),
                        ws.numel() * ws.element_size(), self._stream(stream))
        if rc != BLK_OK:
            raise BlkError(rc, "blk_decode")

    def decode_batch_workspace_bytes(self, max_B: int) -> int:
        return blk_decode_batch_workspace_bytes(self.handle, max_B)

    def decode_batch(self, w: BlkWeights, x, pos, cache_lens, max_cache_len: int, k_cache,
                     v_cache, out, ws, k_new=None, v_new=None, stream=None):
        """One decode step of B = x.shape[0] sequences (caches [B, Hkv, max_ctx, D])."""
        rc = blk_decode_batch(self.handle, w, _ptr(x), _ptr(pos), _ptr(cache_lens), x.shape[0],
                              max_cache_len, _ptr(k_cache), _ptr(v_cache), _ptr(out),
                              _ptr(k_new), _ptr(v_new), _ptr(ws), ws.numel() * ws.element_size(),
                              self._stream(stream))
        if rc != BLK_OK:
            raise BlkError(rc, "blk_decode_batch")

    def embed(self, table, ids, x, stream=None):
        """x[t] = table[ids[t]] (fp16 [vocab, hidden] table, int64 ids)."""
        rc = blk_embed(self.handle, _ptr(table), table.shape[0], _ptr(ids), ids.numel(), _ptr(x),
                       self._stream(stream))
        if rc != BLK_OK:
            raise BlkError(rc, "blk_embed")

    def lm_head_workspace_bytes(self) -> int:
        return blk_lm_head_workspace_bytes(self.handle)

    def lm_head(self, x, norm_g, w_lm, tokens, ws, logits=None, stream=None):
        """Final RMSNorm + LM head + greedy argmax of the rows of x (fp16 [T, hidden])."""
        rc = blk_lm_head(self.handle, _ptr(x), x.shape[0], _ptr(norm_g), _ptr(w_lm),
                         w_lm.shape[0], _ptr(logits), _ptr(tokens), _ptr(ws),
                         ws.numel() * ws.element_size(), self._stream(stream))
        if rc != BLK_OK:
            raise BlkError(rc, "blk_lm_head")

    def timing(self, on: bool):
        rc = blk_timing(self.handle, on)
        if rc != BLK_OK:
            raise BlkError(rc, "blk_timing")

    def timing_collect(self, stream=None):
        return blk_timing_collect(self.handle, self._stream(stream))

    def timing_table(self) -> dict:
        """{kernel name: (total_ms, launches)} for kernels launched at least once."""
        out = {}
        for k in range(BLK_N_KERNELS):
            r = blk_timing_read(self.handle, k)
            if r and r[0] and r[2] > 0:
                out[r[0]] = (r[1], r[2])
        return out

    def check(self, stream=None):
        rc = blk_check(self.handle, self._stream(stream))
        if rc != BLK_OK:
            raise BlkError(rc, "device status")
