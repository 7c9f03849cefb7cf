"""Shared helpers for the GPU tests: move synthetic inputs to the device, run
the library's phases through the C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import decode_qwen2_block_gb300 as blk

REL_L2_TOL = 1e-2      # per tensor, relative L2 error
MAX_ABS_TOL = 5e-2     # per tensor, max absolute error (unit-scale activations)


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def weights_to_dev(w: dict, device="cuda") -> dict:
    return {k: to_dev(v, device) for k, v in w.items()}


def errors(got, want):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(want, dtype=np.float64)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    return float(rel), float(np.max(np.abs(g - r))) if g.size else 0.0


def assert_close(got, want, what=""):
    rel, mx = errors(got, want)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite output"
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, f"{what}: rel_l2={rel:.3e} max_abs={mx:.3e}"
    return rel, mx


class DevBlock:
    """A Block plus device copies of weights and a workspace."""

    def __init__(self, shape, w_np: dict, max_ctx: int, max_T: int, chain=False):
        self.shape = shape
        self.block = blk.Block(shape, max_ctx, chain=chain)
        self.w_dev = weights_to_dev(w_np)
        self.w = blk.Block.weights(self.w_dev)
        nbytes = self.block.workspace_bytes(max_T)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.max_ctx = max_ctx

    def run(self, phase: str, x: torch.Tensor, pos: torch.Tensor, L: int, kc, vc,
            want_new=True, stream=None):
        T = x.shape[0]
        s = self.shape
        out = torch.empty((T, s.hidden), dtype=torch.float16, device="cuda")
        kn = torch.empty((T, s.n_kv_heads, s.head_dim), dtype=torch.float16, device="cuda") if want_new else None
        vn = torch.empty_like(kn) if want_new else None
        if phase == "prefill":
            assert L == 0
            self.block.prefill(self.w, x, pos, kc, vc, out, self.ws, kn, vn, stream=stream)
        elif phase == "prefill_kv":
            self.block.prefill_kv(self.w, x, pos, L, kc, vc, out, self.ws, kn, vn, stream=stream)
        elif phase == "decode":
            assert T == 1
            self.block.decode(self.w, x, pos, L, kc, vc, out, self.ws, kn, vn, stream=stream)
        else:
            raise ValueError(phase)
        return out, kn, vn
