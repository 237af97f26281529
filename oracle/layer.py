"""Oracle Llama layer pieces around the tree attention: RMSNorm, the projection
GEMMs with their epilogues (residual add, SwiGLU), and the layer.

The basal-rs Architecture page ("01 / Request path: GPU forward pass") runs the
Llama model in f16 over the batch as one compact token list.  The page names
the model and its precision, not the layer's arithmetic; the layer here is the
standard Llama decoder layer (pre-norm RMSNorm, grouped-query attention with
rotary positions, SwiGLU MLP, residual adds), with f16 storage of every
activation between steps.  Each step is computed in float64 from the f16
values it reads and rounded to f16 where the product stores a tensor:

* rmsnorm:  n = x / sqrt(mean(x^2) + eps), rounded to f16, times the f16
            weight, rounded to f16 (the Llama order: normalise in high
            precision, cast, then scale);
* gemm:     A B^T in float64, the epilogue (+ R; or silu(g) * u with
            silu(g) = g / (1 + e^-g)) in float64, one rounding to f16;
* layer:    the sequence in tree_layer.h, with tree RoPE and tree attention
            taken from ``oracle.rope`` and ``oracle.attention``;
* last_layer: the final layer computed for every token, then the rows of the
            readout slots (the last token of each leaf) taken, normalised by the
            model's final RMSNorm and multiplied by the answer letters' LM-head
            rows: the page's pruning only skips work whose results are never
            read, so the full layer restricted to those rows is its definition.

Test infrastructure only (see the package docstring).
"""
from __future__ import annotations

import numpy as np

from . import attention as oatt
from . import rope as orope


def f16(x) -> np.ndarray:
    return np.asarray(x, np.float64).astype(np.float16)


def rmsnorm(x16, w16, eps: float) -> np.ndarray:
    """Rows of x (f16) normalised by their root mean square, scaled by w (f16)."""
    x = np.asarray(x16, np.float16).astype(np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    n = f16(x / np.sqrt(ms + eps))
    return f16(n.astype(np.float64) * np.asarray(w16, np.float16).astype(np.float64))


def silu(g):
    g = np.asarray(g, np.float64)
    return g / (1.0 + np.exp(-g))


def gemm(a16, b16, epi: str = "store", r16=None) -> np.ndarray:
    """A [m, k] times B^T (B [n, k], or [2n, k] = [gate; up] for 'swiglu'), epilogue, f16 out."""
    a = np.asarray(a16, np.float16).astype(np.float64)
    b = np.asarray(b16, np.float16).astype(np.float64)
    if epi == "swiglu":
        n = b.shape[0] // 2
        return f16(silu(a @ b[:n].T) * (a @ b[n:].T))
    c = a @ b.T
    if epi == "residual":
        c = c + np.asarray(r16, np.float16).astype(np.float64)
    return f16(c)


def layer(plan, x16, res_k16, res_v16, weights: dict, hq: int, hkv: int, d: int, theta: float,
          eps: float = 1e-5):
    """One Llama layer over the forward tokens of a batch.

    x16: f16 [n_fwd, hidden] (the forward tokens in packed order);
    res_k16, res_v16: f16 [n_res, hkv * d] post-RoPE K and V of the resident
    tokens (may have 0 rows); weights: f16 arrays w_in [hidden], wq [hq d,
    hidden], wk, wv [hkv d, hidden], wo [hidden, hq d], w_post [hidden],
    wgu [2 f, hidden] (gate rows, then up rows), wd [hidden, f].
    Returns (y, q, k, v, o, h) with q, k post-RoPE (f16) and k, v over all
    n_tot = n_res + n_fwd tokens.
    """
    n_res = plan.n_res
    xn = rmsnorm(x16, weights["w_in"], eps)
    q = gemm(xn, weights["wq"])
    k_f = gemm(xn, weights["wk"])
    v_f = gemm(xn, weights["wv"])
    n_fwd = q.shape[0]
    pos = np.asarray(plan.pos[n_res:n_res + n_fwd])
    q = orope.rope_f16(q.reshape(n_fwd, hq, d), pos, theta)
    k_f = orope.rope_f16(k_f.reshape(n_fwd, hkv, d), pos, theta)
    k = np.concatenate([np.asarray(res_k16, np.float16).reshape(n_res, hkv, d), k_f], axis=0)
    v = np.concatenate([np.asarray(res_v16, np.float16).reshape(n_res, hkv, d),
                        v_f.reshape(n_fwd, hkv, d)], axis=0)
    o16 = f16(oatt.attend_paths(plan, q, k, v)).reshape(n_fwd, hq * d)
    h = gemm(o16, weights["wo"], "residual", x16)
    hn = rmsnorm(h, weights["w_post"], eps)
    g = gemm(hn, weights["wgu"], "swiglu")
    y = gemm(g, weights["wd"], "residual", h)
    return y, q, k, v, o16, h


def letter_logits(plan, y16, w_final16, w_letters16, eps: float = 1e-5) -> np.ndarray:
    """float64 [n_slots, stride] logits of the readout slots from the final layer's output rows."""
    rows = np.asarray(plan.slot_tok) - plan.n_res
    f = rmsnorm(np.asarray(y16, np.float16)[rows], w_final16, eps).astype(np.float64)
    return f @ np.asarray(w_letters16, np.float16).astype(np.float64).T


def last_layer(plan, x16, res_k16, res_v16, weights: dict, hq: int, hkv: int, d: int, theta: float, w_final16,
               w_letters16, eps: float = 1e-5):
    y = layer(plan, x16, res_k16, res_v16, weights, hq, hkv, d, theta, eps)[0]
    return letter_logits(plan, y, w_final16, w_letters16, eps)
