"""Oracle attention over tree blocks, float64.

Definition used (basal-rs Architecture page, "03 / Packing: Attention over tree
blocks"): a token sees the earlier tokens of its own block and every token of
its ancestor blocks; sibling branches are masked, so the result equals running
each full prompt on its own.  The oracle therefore does exactly that: it
materialises every root-to-leaf prompt as its own sequence, runs plain dense
causal attention on it,

    o_i = sum_j softmax_j(q_i . k_j / sqrt(d)) v_j        (j <= i on the prompt)

(the 1/sqrt(d_k) scale as written on the AstrAI inference page, "KV Cache"),
and writes each forward token's output back to its packed row.  Grouped
heads: q head h reads kv head h // (hq / hkv).

Inputs are the float16 values the kernel reads (post-RoPE Q and K, V), taken to
float64; the output is float64.

``attend_rows`` computes single rows from the same definition (the row's own
prompt prefix), for sampled checks at sizes where whole prompts are too slow;
``brute_force`` runs masked softmax attention over the whole packed row with the
mask built by walking parent links, for tiny inputs.

Test infrastructure only: see the package docstring.
"""
from __future__ import annotations

import numpy as np

from .plan import Plan, brute_mask, path_tokens


def _dense_causal(qp, kp, vp, q_first: int, scale: float, groups: int):
    """Causal attention of prompt positions q_first.. over the prompt's keys.

    qp [nq, hq, d] are the queries at prompt positions q_first .. q_first+nq-1;
    kp/vp [L, hkv, d] are all prompt keys/values (L = q_first + nq).
    """
    nq, hq, d = qp.shape
    L = kp.shape[0]
    out = np.empty((nq, hq, d), np.float64)
    qpos = q_first + np.arange(nq)
    causal = np.arange(L)[None, :] <= qpos[:, None]           # [nq, L]
    for h in range(hq):
        g = h // groups
        s = (qp[:, h, :] @ kp[:, g, :].T) * scale              # [nq, L]
        s = np.where(causal, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vp[:, g, :]
    return out


def attend_paths(plan: Plan, q_rot, k_rot, v, *, check_shared: bool = False,
                 block_rows: int = 1024) -> np.ndarray:
    """[n_fwd, hq, d] float64 outputs, one prompt at a time.

    Each forward token is computed on the first prompt (in leaf order) that
    contains it.  With ``check_shared`` every prompt is computed in full and a
    token shared by several prompts must get the same value from each.
    """
    q = np.asarray(q_rot, np.float64)
    k = np.asarray(k_rot, np.float64)
    vv = np.asarray(v, np.float64)
    n_fwd, hq, d = q.shape
    hkv = k.shape[1]
    groups = hq // hkv
    scale = 1.0 / np.sqrt(d)
    out = np.full((n_fwd, hq, d), np.nan)
    done = np.zeros(n_fwd, bool)
    has_child = np.zeros(plan.n_blocks, bool)
    has_child[plan.blk_parent[plan.blk_parent >= 0]] = True
    for leaf in np.nonzero(~has_child)[0]:
        toks = path_tokens(plan, int(leaf))                    # packed tokens of the prompt
        fwd = toks >= plan.n_res
        first = int(np.argmax(fwd)) if fwd.any() else len(toks)
        if check_shared:
            start = first
        else:
            pending = [a for a in range(first, len(toks)) if not done[toks[a] - plan.n_res]]
            if not pending:
                continue
            start = pending[0]
        kp, vp = k[toks], vv[toks]
        for a0 in range(start, len(toks), block_rows):
            a1 = min(a0 + block_rows, len(toks))
            rows = toks[a0:a1] - plan.n_res
            o = _dense_causal(q[rows], kp[:a1], vp[:a1], a0, scale, groups)
            if check_shared:
                prev = done[rows]
                if prev.any():
                    np.testing.assert_allclose(out[rows[prev]], o[prev], rtol=0, atol=1e-12)
            out[rows] = o
            done[rows] = True
    assert done.all(), "a forward token lies on no prompt"
    return out


def attend_rows(plan: Plan, q_rot, k_rot, v, rows) -> np.ndarray:
    """Outputs [len(rows), hq, d] for selected forward rows only.

    Each row's keys are its own prompt up to itself: the tokens of its ancestor
    blocks (walking parent links) and its block's tokens up to the row.
    """
    q = np.asarray(q_rot)
    n_fwd, hq, d = q.shape
    hkv = k_rot.shape[1]
    groups = hq // hkv
    scale = 1.0 / np.sqrt(d)
    blk_of = np.searchsorted(plan.blk_start, np.arange(plan.n_tot), side="right") - 1
    out = np.empty((len(rows), hq, d), np.float64)
    for n, r in enumerate(rows):
        t = int(r) + plan.n_res
        b = int(blk_of[t])
        keys = [np.arange(plan.blk_start[b], t + 1)]
        x = plan.blk_parent[b]
        while x >= 0:
            keys.append(np.arange(plan.blk_start[x], plan.blk_start[x] + plan.blk_len[x]))
            x = plan.blk_parent[x]
        keys = np.concatenate(keys[::-1])
        kk = np.asarray(k_rot[keys], np.float64)
        vk = np.asarray(v[keys], np.float64)
        qq = np.asarray(q[int(r)], np.float64)
        for h in range(hq):
            g = h // groups
            s = (kk[:, g, :] @ qq[h]) * scale
            s -= s.max()
            p = np.exp(s)
            p /= p.sum()
            out[n, h] = p @ vk[:, g, :]
    return out


def lse_rows(plan: Plan, q_rot, k_rot, rows) -> np.ndarray:
    """[len(rows), hq] natural log of sum_j exp(q.k_j / sqrt(d)) over each row's own keys."""
    q = np.asarray(q_rot)
    n_fwd, hq, d = q.shape
    groups = hq // k_rot.shape[1]
    out = np.empty((len(rows), hq), np.float64)
    for n, r in enumerate(rows):
        t = int(r) + plan.n_res
        b = int(np.searchsorted(plan.blk_start, t, side="right") - 1)
        keys = [np.arange(plan.blk_start[b], t + 1)]
        x = plan.blk_parent[b]
        while x >= 0:
            keys.append(np.arange(plan.blk_start[x], plan.blk_start[x] + plan.blk_len[x]))
            x = plan.blk_parent[x]
        kk = np.asarray(k_rot[np.concatenate(keys)], np.float64)
        for h in range(hq):
            s = (kk[:, h // groups, :] @ np.asarray(q[int(r), h], np.float64)) / np.sqrt(d)
            m = s.max()
            out[n, h] = m + np.log(np.exp(s - m).sum())
    return out


def brute_force(plan: Plan, q_rot, k_rot, v) -> np.ndarray:
    """Masked softmax attention over the whole packed row (tiny inputs only)."""
    m = brute_mask(plan)[plan.n_res:]                          # forward queries x all keys
    q = np.asarray(q_rot, np.float64)
    k = np.asarray(k_rot, np.float64)
    vv = np.asarray(v, np.float64)
    n_fwd, hq, d = q.shape
    groups = hq // k.shape[1]
    out = np.empty((n_fwd, hq, d))
    for h in range(hq):
        g = h // groups
        s = q[:, h, :] @ k[:, g, :].T / np.sqrt(d)
        s = np.where(m, s, -np.inf)
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vv[:, g, :]
    return out


def visible_pairs(plan: Plan) -> int:
    """Count of visible (query, key) pairs by brute force (tiny inputs only)."""
    return int(brute_mask(plan)[plan.n_res:].sum())
