"""Oracle rotary embedding with tree positions, float64.

Position: the basal-rs Architecture page ("03 / Packing: Attention over tree
blocks") gives a token's rotary position as its position in its own prompt.
The planner's ``pos`` table holds exactly that (the number of prompt tokens
before it on its root-to-leaf path).

Rotation: the page names RoPE without a formula.  The plain reading taken
here is the Llama form over pairs (i, i + d/2) ("rotate half"):

    a_i = pos * theta ** (-2 i / d),    i = 0 .. d/2 - 1
    y_i       = x_i cos a_i - x_{i+d/2} sin a_i
    y_{i+d/2} = x_{i+d/2} cos a_i + x_i sin a_i

computed in float64 and rounded once to float16 (round to nearest even), the
storage type of Q and K.  The AstrAI inference page ("Rotary Embedding
Backend") keeps the cos/sin pairs as a [max_len, dim/2, 2] float32 table; the
oracle evaluates them in float64 directly.

Test infrastructure only: see the package docstring.
"""
from __future__ import annotations

import numpy as np


def angles(pos: np.ndarray, d: int, theta: float) -> np.ndarray:
    """[len(pos), d/2] rotation angles in float64."""
    i = np.arange(d // 2, dtype=np.float64)
    inv = np.power(np.float64(theta), -2.0 * i / d)
    return np.asarray(pos, np.float64)[:, None] * inv[None, :]


def rotate(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate x[..., tokens, heads, d] (any float) at per-token positions; float64 out."""
    x = np.asarray(x, np.float64)
    n, h, d = x.shape
    a = angles(pos, d, theta)[:, None, :]          # [n, 1, d/2]
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_f16(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """The stored result: float64 rotation rounded to float16."""
    return rotate(x, pos, theta).astype(np.float16)


def apply_plan(plan, q_pre: np.ndarray, k_in: np.ndarray, theta: float):
    """Rotate every forward token's Q and K; resident K rows are left as given.

    q_pre : [n_fwd, hq, d] f16, rows = packed tokens n_res .. n_tot-1
    k_in  : [n_tot, hkv, d] f16, rows of resident tokens already rotated
    returns (q_rot, k_rot) as float16 arrays
    """
    pos_f = plan.pos[plan.n_res:]
    q_rot = rope_f16(q_pre, pos_f, theta)
    k_rot = np.array(k_in, np.float16, copy=True)
    k_rot[plan.n_res:] = rope_f16(k_in[plan.n_res:], pos_f, theta)
    return q_rot, k_rot
