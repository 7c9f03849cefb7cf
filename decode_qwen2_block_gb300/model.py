"""A whole decoder-only model driven through the C ABI: token embedding, the
stack of decoder blocks, final RMSNorm + LM head, greedy next token.

This is the inference loop of the pages (the MLIR-compilation page's §2.3:
tokens -> embedding -> blocks -> LM head -> logits -> sampling; the buddy-mlir
DeepSeek-R1 page's §6.4.6 decode loop: greedy argmax, the token becomes the
next step's input, cache position + 1).  The next token stays on the device:
a step reads the previous step's token from device memory, so steps can be
captured into CUDA graphs and replayed back to back without a host round
trip.  All work is the library's kernels; torch supplies memory, streams and
graphs.
"""
from __future__ import annotations

import torch

from .stack import LayerStack


class Model:
    def __init__(self, shape, layer_weights, head_weights, max_ctx: int, caches=None,
                 device="cuda", stack=None):
        """layer_weights: list of per-layer dicts of fp16 CUDA tensors (or an
        existing LayerStack as `stack`); head_weights: dict with "embed"
        [vocab, hidden], "norm_g" [hidden] and "lm_head" [vocab, hidden] fp16
        CUDA tensors."""
        self.shape = shape
        self.stack = stack if stack is not None else LayerStack(
            shape, layer_weights, max_ctx, 1, caches=caches, device=device)
        self.block = self.stack.block
        self.embed_w = head_weights["embed"]
        self.norm_g = head_weights["norm_g"]
        self.head_w = head_weights["lm_head"]
        self.vocab = self.head_w.shape[0]
        H = shape.hidden
        self.x = torch.empty((1, H), dtype=torch.float16, device=device)
        self.head_ws = torch.empty(self.block.lm_head_workspace_bytes(), dtype=torch.uint8,
                                   device=device)
        self.graphs = {}

    def step(self, token_in, pos, cache_len: int, token_out, logits=None, stream=None):
        """token_in (int64 [1], device) at position pos (int64 [1]) with
        cache_len history slots -> token_out (int64 [1]); the block stack
        appends this token's K/V at slot cache_len of every layer."""
        self.block.embed(self.embed_w, token_in, self.x, stream=stream)
        h = self.stack.decode_step(self.x, pos, cache_len, stream=stream)
        self.block.lm_head(h, self.norm_g, self.head_w, token_out, self.head_ws, logits=logits,
                           stream=stream)
        return token_out

    def capture_step(self, token_in, pos, cache_len: int, token_out, key=None):
        """CUDA graph of one step; the tensors must stay alive at the same
        addresses for every replay."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.step(token_in, pos, cache_len, token_out, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        self.graphs[key if key is not None else cache_len] = g
        return g

    def generate(self, first_token: int, start: int, n_tokens: int, logits_out=None):
        """Greedy decode of n_tokens after first_token placed at position
        `start` (cache_len = start history slots).  Returns the int64 device
        tensor of the n_tokens generated ids.  logits_out, if given, is a list
        that receives each step's fp32 logits [1, vocab]."""
        dev = self.x.device
        toks = torch.empty(n_tokens + 1, dtype=torch.int64, device=dev)
        toks[0] = first_token
        for i in range(n_tokens):
            pos = torch.tensor([start + i], dtype=torch.int64, device=dev)
            lg = None
            if logits_out is not None:
                lg = torch.empty((1, self.vocab), dtype=torch.float32, device=dev)
            self.step(toks[i:i + 1], pos, start + i, toks[i + 1:i + 2], logits=lg)
            if lg is not None:
                logits_out.append(lg)
        return toks[1:]
