"""A second, independent restatement of the decoder block, for small cases.

Written in matrix form with numpy f64: a dense [T, L+T] score matrix with an
explicit -inf causal mask, GQA by repeating each kv head over its group of
query heads (repeat_interleave order), RoPE by rotate_half on whole tensors.
It shares no code with ``oracle/`` and is only meant to catch a plumbing
mistake there (a swapped weight, a transposed operand, a wrong mask edge).
"""
import numpy as np


def _rms(x, g, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def _rotate_half(x):
    half = x.shape[-1] // 2
    return np.concatenate([-x[..., half:], x[..., :half]], axis=-1)


def _rope(x, pos, theta):
    # x: [T, heads, D]; pos: [T]
    D = x.shape[-1]
    inv = theta ** (-np.arange(0, D, 2, dtype=np.float64) / D)       # [D/2]
    ang = pos.astype(np.float64)[:, None] * inv[None, :]               # [T, D/2]
    cos = np.concatenate([np.cos(ang), np.cos(ang)], axis=-1)[:, None, :]
    sin = np.concatenate([np.sin(ang), np.sin(ang)], axis=-1)[:, None, :]
    return x * cos + _rotate_half(x) * sin


def block(shape, w, x16, pos, L, kc16, vc16, window=0):
    """Returns (out fp16 [T,H], k_new fp16, v_new fp16); caches are not modified.
    window > 0: row t sees only slots [L + t - window + 1, L + t] (a band of
    the score matrix)."""
    H, Hq, Hkv, D = shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim
    f = lambda a: np.asarray(a, dtype=np.float64)
    x = f(x16)
    T = x.shape[0]
    xn = _rms(x, f(w["ln1_g"]), shape.rms_eps)
    q = xn @ f(w["wq"]).T
    k = xn @ f(w["wk"]).T
    v = xn @ f(w["wv"]).T
    if shape.has_qkv_bias:
        q, k, v = q + f(w["bq"]), k + f(w["bk"]), v + f(w["bv"])
    q = _rope(q.reshape(T, Hq, D), pos, shape.rope_theta)
    k = _rope(k.reshape(T, Hkv, D), pos, shape.rope_theta)
    v = v.reshape(T, Hkv, D)
    k16, v16 = k.astype(np.float16), v.astype(np.float16)
    # keys/values visible to the new rows: history then the new (fp16) rows
    K = np.concatenate([f(kc16[:, :L, :]), f(k16).transpose(1, 0, 2)], axis=1)  # [Hkv, L+T, D]
    V = np.concatenate([f(vc16[:, :L, :]), f(v16).transpose(1, 0, 2)], axis=1)
    G = Hq // Hkv
    K = np.repeat(K, G, axis=0)                                        # [Hq, L+T, D]
    V = np.repeat(V, G, axis=0)
    S = np.einsum("thd,hjd->htj", q, K) / np.sqrt(D)                   # [Hq, T, L+T]
    mask = np.full((T, L + T), -np.inf)
    for t in range(T):
        lo = max(0, L + t + 1 - window) if window > 0 else 0
        mask[t, lo: L + t + 1] = 0.0
    S = S + mask[None]
    P = np.exp(S - S.max(axis=-1, keepdims=True))
    P = P / P.sum(axis=-1, keepdims=True)
    attn = np.einsum("htj,hjd->thd", P, V).reshape(T, Hq * D)
    h = x + attn @ f(w["wo"]).T
    hn = _rms(h, f(w["ln2_g"]), shape.rms_eps)
    g = hn @ f(w["w_gate"]).T
    u = hn @ f(w["w_up"]).T
    a = g / (1.0 + np.exp(-g)) * u
    out = h + a @ f(w["w_down"]).T
    return out.astype(np.float16), k16, v16
