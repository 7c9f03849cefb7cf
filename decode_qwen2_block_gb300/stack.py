"""A stack of decoder blocks driven through the C ABI.

Runs one phase over every layer in order (layer l's output is layer l+1's
input), with the BLK_FLAG_CHAIN promise set so that each layer's first
kernel overlaps the previous layer's last kernel, and can capture a decode
step into a CUDA graph (one graph per cache length, since cache_len is a
by-value argument).  All work is the library's kernels; torch only supplies
device memory, streams and graphs.
"""
from __future__ import annotations

import ctypes

import torch

from . import (BLK_ERR_SHAPE, BLK_OK, BlkError, Block, BlkQWeights, BlkWeights,
               blk_decode_batch_stack, blk_decode_batch_stack_workspace_bytes, blk_decode_stack,
               blk_decode_stack_q, blk_prefill_stack, blk_prefill_stack_workspace_bytes)


class LayerStack:
    def __init__(self, shape, layer_weights, max_ctx: int, max_T: int, caches=None,
                 chain: bool = True, device="cuda"):
        """layer_weights: list of dicts of fp16 CUDA tensors (one per layer).
        caches: optional list of (k_cache, v_cache) per layer; allocated
        (zero-filled) when None."""
        self.shape = shape
        self.n_layers = len(layer_weights)
        self.block = Block(shape, max_ctx, chain=chain)
        self.wdev = layer_weights
        self.w = [Block.weights(wd) for wd in layer_weights]
        H, Hkv, D = shape.hidden, shape.n_kv_heads, shape.head_dim
        if caches is None:
            caches = [(torch.zeros((Hkv, max_ctx, D), dtype=torch.float16, device=device),
                       torch.zeros((Hkv, max_ctx, D), dtype=torch.float16, device=device))
                      for _ in range(self.n_layers)]
        self.caches = caches
        # one workspace for every call: the one-layer calls, decode, and the
        # prefill stack (which also keeps its activation buffers in it)
        nbytes = max(self.block.workspace_bytes(max_T),
                     blk_prefill_stack_workspace_bytes(self.block.handle, max_T))
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.max_T = max_T
        # ping-pong activations between layers
        self.bufs = [torch.empty((max_T, H), dtype=torch.float16, device=device) for _ in range(2)]
        self.graphs = {}
        n = self.n_layers
        self._w_arr = (BlkWeights * n)(*self.w)
        self._kc_arr = (ctypes.c_void_p * n)(*[kc.data_ptr() for kc, _ in caches])
        self._vc_arr = (ctypes.c_void_p * n)(*[vc.data_ptr() for _, vc in caches])

    def decode_step(self, x, pos, cache_len: int, out=None, stream=None):
        """One token through every layer in one library call (blk_decode_stack).
        Returns the last layer's output."""
        out = self.bufs[0][:1] if out is None else out
        s = torch.cuda.current_stream() if stream is None else stream
        rc = blk_decode_stack(self.block.handle, self._w_arr, self.n_layers, self._kc_arr,
                              self._vc_arr, x.data_ptr(), pos.data_ptr(), cache_len,
                              out.data_ptr(), None, None, self.ws.data_ptr(),
                              self.ws.numel(), s.cuda_stream)
        if rc != BLK_OK:
            raise BlkError(rc, "blk_decode_stack")
        return out

    def prefill_step(self, x, pos, cache_len: int, out=None, stream=None):
        """T new tokens through every layer in one library call
        (blk_prefill_stack; prefill when cache_len is 0, else prefill_kv).
        Returns the last layer's output."""
        T = x.shape[0]
        out = self.bufs[0][:T] if out is None else out
        s = torch.cuda.current_stream() if stream is None else stream
        rc = blk_prefill_stack(self.block.handle, self._w_arr, self.n_layers, self._kc_arr,
                               self._vc_arr, x.data_ptr(), pos.data_ptr(), T, cache_len,
                               out.data_ptr(), self.ws.data_ptr(), self.ws.numel(), s.cuda_stream)
        if rc != BLK_OK:
            raise BlkError(rc, "blk_prefill_stack")
        return out

    def run(self, phase: str, x, pos, cache_len: int, layer_outputs=None, stream=None):
        """Runs `phase` over all layers; returns the last layer's output (a
        view of an internal buffer).  layer_outputs, if given, is a list that
        receives a copy of each layer's input (for layer-local checks); the
        layers then run as one call each."""
        T = x.shape[0]
        if phase == "decode" and layer_outputs is None:
            return self.decode_step(x, pos, cache_len, stream=stream)
        if layer_outputs is None:
            return self.prefill_step(x, pos, 0 if phase == "prefill" else cache_len,
                                     stream=stream)
        cur = x
        for l in range(self.n_layers):
            out = self.bufs[l % 2][:T]
            if layer_outputs is not None:
                layer_outputs.append(cur.clone())
            kc, vc = self.caches[l]
            if phase == "decode":
                self.block.decode(self.w[l], cur, pos, cache_len, kc, vc, out, self.ws,
                                  stream=stream)
            elif phase == "prefill":
                self.block.prefill(self.w[l], cur, pos, kc, vc, out, self.ws, stream=stream)
            else:
                self.block.prefill_kv(self.w[l], cur, pos, cache_len, kc, vc, out, self.ws,
                                      stream=stream)
            cur = out
        return cur

    def capture(self, phase: str, x, pos, cache_len: int, key=None):
        """Captures one pass over all layers into a CUDA graph.  x and pos must
        stay alive and at the same address for every replay."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                out = self.run(phase, x, pos, cache_len, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        self.graphs[key if key is not None else (phase, cache_len)] = (g, out)
        return g, out


class BatchStack:
    """B sequences, one new token each, through a stack of decoder blocks in
    one library call per step (blk_decode_batch_stack)."""

    def __init__(self, shape, layer_weights, max_ctx: int, max_B: int, caches=None,
                 device="cuda"):
        """layer_weights: list of dicts of fp16 CUDA tensors (one per layer).
        caches: optional list of (k_cache, v_cache) per layer, each
        [max_B, Hkv, max_ctx, D]; allocated (zero-filled) when None.  A step
        with B <= max_B sequences uses the first B of every cache."""
        self.shape = shape
        self.n_layers = len(layer_weights)
        self.block = Block(shape, max_ctx, chain=True)
        self.wdev = layer_weights
        self.w = [Block.weights(wd) for wd in layer_weights]
        Hkv, D = shape.n_kv_heads, shape.head_dim
        if caches is None:
            caches = [(torch.zeros((max_B, Hkv, max_ctx, D), dtype=torch.float16, device=device),
                       torch.zeros((max_B, Hkv, max_ctx, D), dtype=torch.float16, device=device))
                      for _ in range(self.n_layers)]
        self.caches = caches
        self.max_B = max_B
        nbytes = blk_decode_batch_stack_workspace_bytes(self.block.handle, max_B)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        n = self.n_layers
        self._w_arr = (BlkWeights * n)(*self.w)
        self._kc_arr = (ctypes.c_void_p * n)(*[kc.data_ptr() for kc, _ in caches])
        self._vc_arr = (ctypes.c_void_p * n)(*[vc.data_ptr() for _, vc in caches])

    def step(self, x, pos, cache_lens, max_cache_len: int, out, stream=None):
        """x, out: fp16 [B, hidden]; pos, cache_lens: int64 [B] on the device;
        max_cache_len bounds the cache lengths.  Returns out."""
        B = x.shape[0]
        if B > self.max_B:
            raise BlkError(BLK_ERR_SHAPE, "BatchStack.step: B > max_B")
        s = torch.cuda.current_stream() if stream is None else stream
        rc = blk_decode_batch_stack(self.block.handle, self._w_arr, self.n_layers, self._kc_arr,
                                    self._vc_arr, x.data_ptr(), pos.data_ptr(),
                                    cache_lens.data_ptr(), B, max_cache_len, out.data_ptr(),
                                    self.ws.data_ptr(), self.ws.numel(), s.cuda_stream)
        if rc != BLK_OK:
            raise BlkError(rc, "blk_decode_batch_stack")
        return out


class QuantDecodeStack:
    """Decode through a stack of blocks with weight-only quantized projections
    (blk_decode_stack_q), one library call per step."""

    def __init__(self, shape, qweights, max_ctx: int, caches=None, chain: bool = True,
                 device="cuda"):
        """qweights: list of BlkQWeights (one per layer; the tensors they
        point to must stay alive).  caches: optional list of (k_cache,
        v_cache) per layer, [Hkv, max_ctx, D]; zero-filled when None."""
        self.shape = shape
        self.n_layers = len(qweights)
        self.block = Block(shape, max_ctx, chain=chain)
        Hkv, D = shape.n_kv_heads, shape.head_dim
        if caches is None:
            caches = [(torch.zeros((Hkv, max_ctx, D), dtype=torch.float16, device=device),
                       torch.zeros((Hkv, max_ctx, D), dtype=torch.float16, device=device))
                      for _ in range(self.n_layers)]
        self.caches = caches
        self.ws = torch.empty(self.block.qworkspace_bytes(1), dtype=torch.uint8, device=device)
        self.out = torch.empty((1, shape.hidden), dtype=torch.float16, device=device)
        n = self.n_layers
        self._w_arr = (BlkQWeights * n)(*qweights)
        self._kc_arr = (ctypes.c_void_p * n)(*[kc.data_ptr() for kc, _ in caches])
        self._vc_arr = (ctypes.c_void_p * n)(*[vc.data_ptr() for _, vc in caches])

    def decode_step(self, x, pos, cache_len: int, out=None, stream=None):
        out = self.out if out is None else out
        s = torch.cuda.current_stream() if stream is None else stream
        rc = blk_decode_stack_q(self.block.handle, self._w_arr, self.n_layers, self._kc_arr,
                                self._vc_arr, x.data_ptr(), pos.data_ptr(), cache_len,
                                out.data_ptr(), None, None, self.ws.data_ptr(), self.ws.numel(),
                                s.cuda_stream)
        if rc != BLK_OK:
            raise BlkError(rc, "blk_decode_stack_q")
        return out

    def capture(self, x, pos, cache_len: int):
        """One decode step captured into a CUDA graph (x, pos stay alive)."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                out = self.decode_step(x, pos, cache_len, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        return g, out
