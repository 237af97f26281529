"""Oracle planner: prompts of a batch -> prefix trees -> one packed token row.

Follows the basal-rs Architecture page:

* "01 / Request path: Batch and prefix tree" -- the prompts of a batch are
  arranged into rows; each row is a tree whose shared prefixes are computed
  once; a row holds at most 32,768 tokens, a forward pass processes at most
  8192, a tree is at most 8 blocks deep, and identical prompts share a single
  readout.
* "03 / Packing: Attention over tree blocks" -- before computation the tree is
  turned into one row of tokens; a token sees the earlier tokens of its own
  block and all tokens of its ancestor blocks; its rotary position is its
  position in its own prompt.
* "03 / Packing: Shared state computed once" -- the template is computed once
  at startup (here: its K/V are resident before the forward).
* "04 / Scheduling" -- a long row runs as several forwards of at most 8192
  tokens, each resuming with the tensors of the earlier ones.

Where the page leaves a step open this module takes the plain reading:
blocks are packed in depth-first pre-order with children in input order;
sibling blocks with equal non-zero content key and equal length are one block
(at any depth, their children are pooled); resident tokens must lead the
packed order; forward chunk c covers the packed tokens
[n_res + c*max_fwd, n_res + (c+1)*max_fwd); a readout slot is the last token of
every leaf block, slots numbered in packed order.

Test infrastructure only: see the package docstring.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

OK = 0
ERR_INVALID_ARG = 1
ERR_BAD_TREE = 2
ERR_DEPTH = 3
ERR_ROW_TOO_LONG = 4
ERR_UNSUPPORTED = 5


class PlanError(ValueError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


@dataclass
class Plan:
    # canonical blocks in packed order
    n_blocks: int
    blk_start: np.ndarray      # first packed token of the block
    blk_len: np.ndarray
    blk_parent: np.ndarray     # packed index of the parent block, -1 for a root
    blk_depth: np.ndarray      # 1 for a root
    blk_pos0: np.ndarray       # tokens on the path before the block
    blk_send: np.ndarray       # end (exclusive) of the block's subtree in packed tokens
    blk_resident: np.ndarray
    block_map: np.ndarray      # input block -> packed block
    # tokens
    n_tot: int
    n_res: int
    pos: np.ndarray            # [n_tot] position in own prompt
    send: np.ndarray           # [ceil(n_tot/bn)*bn] subtree end of each key's block, 0 past n_tot
    # forward chunks and tiles
    max_fwd: int
    bm: int
    bn: int
    chunk_q0: np.ndarray
    chunk_q1: np.ndarray
    chunk_t0: np.ndarray       # first Q tile of the chunk
    chunk_t1: np.ndarray
    qt_row0: np.ndarray        # packed token range of each Q tile
    qt_row1: np.ndarray
    qt_ent0: np.ndarray        # entry range of each Q tile (CSR)
    qt_ent1: np.ndarray
    ent: np.ndarray            # (kv_tile << 1) | partial
    qt_order: np.ndarray       # per chunk, its Q tiles longest-first
    # readout
    n_slots: int
    slot_tok: np.ndarray       # packed token of each readout slot
    blk_slot: np.ndarray       # slot of each packed block, -1 if not a leaf
    # work
    pairs: int                 # visible (query, key) pairs over the forward tokens

    @property
    def n_fwd(self) -> int:
        return self.n_tot - self.n_res

    @property
    def n_chunks(self) -> int:
        return int(self.chunk_q0.shape[0])


def _validate(parent, length, nb, max_depth):
    for b in range(nb):
        p = int(parent[b])
        if p < -1 or p >= nb or p == b:
            raise PlanError(ERR_BAD_TREE, f"block {b}: parent {p} out of range")
        if int(length[b]) <= 0:
            raise PlanError(ERR_BAD_TREE, f"block {b}: length {int(length[b])} <= 0")
    # every parent chain must reach a root within nb steps (no cycles)
    depth = np.zeros(nb, np.int64)
    for b in range(nb):
        d, x = 0, b
        while x != -1:
            d += 1
            if d > nb:
                raise PlanError(ERR_BAD_TREE, f"block {b}: parent chain has a cycle")
            x = int(parent[x])
        depth[b] = d
        if d > max_depth:
            raise PlanError(ERR_DEPTH, f"block {b}: depth {d} > {max_depth}")
    return depth


def make_plan(parent, length, key, resident, *, max_fwd=8192, bm=128, bn=128,
              max_depth=8, max_row=32768, leaf1=None, leaf2=None) -> tuple[Plan, dict]:
    """Plan one batch.  Returns the plan and the question -> slot maps."""
    parent = np.asarray(parent, np.int64)
    length = np.asarray(length, np.int64)
    key = np.asarray(key, np.uint64)
    resident = np.asarray(resident, np.int64)
    nb = parent.shape[0]
    if nb == 0:
        raise PlanError(ERR_INVALID_ARG, "empty forest")
    if max_fwd <= 0 or max_fwd % bm != 0 or bm != 128 or bn != 128:
        raise PlanError(ERR_UNSUPPORTED, "tile sizes must be 128 and max_fwd a multiple of 128")
    _validate(parent, length, nb, max_depth)

    children = [[] for _ in range(nb)]
    roots = []
    for b in range(nb):
        (roots if parent[b] < 0 else children[int(parent[b])]).append(b)

    # merge identical siblings (trie semantics), top-down
    canon = -np.ones(nb, np.int64)
    canon_children = {}          # canonical block -> canonical children in order

    def merge(members):          # members: input blocks under one canonical parent, index order
        order, seen = [], {}
        pooled = {}
        for b in members:
            ident = (int(length[b]), int(key[b])) if int(key[b]) != 0 else None
            if ident is not None and ident in seen:
                c = seen[ident]
                canon[b] = c
                if int(resident[b]) != int(resident[c]):
                    raise PlanError(ERR_INVALID_ARG, f"blocks {c} and {b} merge but disagree on residency")
            else:
                canon[b] = b
                order.append(b)
                if ident is not None:
                    seen[ident] = b
            pooled.setdefault(int(canon[b]), []).extend(children[b])
        return order, pooled

    top, pooled = merge(roots)
    stack = list(pooled.items())
    while stack:
        c, kids = stack.pop()
        order, sub = merge(sorted(kids))
        canon_children[c] = order
        stack.extend(sub.items())

    # depth-first pre-order over canonical blocks
    packed = []
    def visit(c):
        packed.append(c)
        for ch in canon_children.get(c, []):
            visit(ch)
    for r in top:
        visit(r)
    nbc = len(packed)
    pidx = {c: i for i, c in enumerate(packed)}

    blk_len = np.array([length[c] for c in packed], np.int64)
    blk_start = np.zeros(nbc, np.int64)
    blk_start[1:] = np.cumsum(blk_len)[:-1]
    n_tot = int(blk_len.sum())
    blk_parent = np.array([pidx[int(canon[parent[c]])] if parent[c] >= 0 else -1 for c in packed], np.int64)
    blk_depth = np.zeros(nbc, np.int64)
    blk_pos0 = np.zeros(nbc, np.int64)
    for i in range(nbc):               # parents precede children in pre-order
        p = blk_parent[i]
        blk_depth[i] = 1 if p < 0 else blk_depth[p] + 1
        blk_pos0[i] = 0 if p < 0 else blk_pos0[p] + blk_len[p]
    # subtree end: walk blocks in reverse pre-order accumulating subtree sizes
    sub = blk_len.copy()
    for i in range(nbc - 1, -1, -1):
        if blk_parent[i] >= 0:
            sub[blk_parent[i]] += sub[i]
    blk_send = blk_start + sub
    blk_res = np.array([resident[c] for c in packed], np.int64)

    # a row is one tree: its token count is the root's subtree size
    for i in range(nbc):
        if blk_parent[i] < 0 and sub[i] > max_row:
            raise PlanError(ERR_ROW_TOO_LONG, f"row of {int(sub[i])} tokens > {max_row}")

    # resident tokens must form the leading part of the packed row
    n_res = 0
    seen_fwd = False
    for i in range(nbc):
        if blk_res[i]:
            if seen_fwd:
                raise PlanError(ERR_INVALID_ARG, "resident blocks must precede all forward blocks in packed order")
            n_res += int(blk_len[i])
        else:
            seen_fwd = True
    if n_res == n_tot:
        raise PlanError(ERR_INVALID_ARG, "no forward tokens")

    # per-token tables
    pos = np.zeros(n_tot, np.int64)
    send_tok = np.zeros(n_tot, np.int64)
    for i in range(nbc):
        s, L = blk_start[i], blk_len[i]
        pos[s:s + L] = blk_pos0[i] + np.arange(L)
        send_tok[s:s + L] = blk_send[i]
    n_kvt = -(-n_tot // bn)
    send = np.zeros(n_kvt * bn, np.int64)
    send[:n_tot] = send_tok

    # forward chunks and Q tiles
    n_fwd = n_tot - n_res
    n_chunks = -(-n_fwd // max_fwd)
    chunk_q0 = n_res + max_fwd * np.arange(n_chunks)
    chunk_q1 = np.minimum(chunk_q0 + max_fwd, n_tot)
    qt_row0, qt_row1, chunk_t0, chunk_t1 = [], [], [], []
    for c in range(n_chunks):
        chunk_t0.append(len(qt_row0))
        r = int(chunk_q0[c])
        while r < chunk_q1[c]:
            qt_row0.append(r)
            qt_row1.append(min(r + bm, int(chunk_q1[c])))
            r += bm
        chunk_t1.append(len(qt_row0))

    # tile classes from the definition: key j is visible to query i iff
    # j <= i and i < send[j] (pre-order makes every subtree one interval)
    ent, qt_ent0, qt_ent1 = [], [], []
    for t in range(len(qt_row0)):
        i0, i1 = qt_row0[t], qt_row1[t]
        qt_ent0.append(len(ent))
        n_kt = (i1 - 1) // bn + 1
        j = np.arange(n_kt * bn)
        sj = send[:n_kt * bn]
        real = j < n_tot
        # some query of the tile sees key j
        vis = real & (np.maximum(j, i0) < np.minimum(sj, i1))
        # every query of the tile sees key j
        full = real & (j <= i0) & (i1 - 1 < sj)
        vis = vis.reshape(n_kt, bn).any(axis=1)
        full = full.reshape(n_kt, bn).all(axis=1)
        for kt in range(n_kt):
            if vis[kt]:
                ent.append((kt << 1) | (0 if full[kt] else 1))
        qt_ent1.append(len(ent))

    # longest-first Q tile order inside each chunk (ties: lower tile first)
    qt_order = []
    for c in range(n_chunks):
        ts = list(range(chunk_t0[c], chunk_t1[c]))
        ts.sort(key=lambda t: (-(qt_ent1[t] - qt_ent0[t]), t))
        qt_order.extend(ts)

    # readout slots: last token of every leaf block, packed order
    has_child = np.zeros(nbc, bool)
    for i in range(nbc):
        if blk_parent[i] >= 0:
            has_child[blk_parent[i]] = True
    blk_slot = -np.ones(nbc, np.int64)
    slot_tok = []
    for i in range(nbc):
        if not has_child[i]:
            blk_slot[i] = len(slot_tok)
            slot_tok.append(int(blk_start[i] + blk_len[i] - 1))

    # visible pairs over forward tokens: the keys of query i are exactly the
    # tokens of its prompt up to and including itself
    pairs = int((pos[n_res:] + 1).sum())

    block_map = np.array([pidx[int(canon[b])] for b in range(nb)], np.int64)
    plan = Plan(
        n_blocks=nbc, blk_start=blk_start, blk_len=blk_len, blk_parent=blk_parent,
        blk_depth=blk_depth, blk_pos0=blk_pos0, blk_send=blk_send, blk_resident=blk_res,
        block_map=block_map, n_tot=n_tot, n_res=n_res, pos=pos, send=send,
        max_fwd=max_fwd, bm=bm, bn=bn,
        chunk_q0=np.asarray(chunk_q0, np.int64), chunk_q1=np.asarray(chunk_q1, np.int64),
        chunk_t0=np.asarray(chunk_t0, np.int64), chunk_t1=np.asarray(chunk_t1, np.int64),
        qt_row0=np.asarray(qt_row0, np.int64), qt_row1=np.asarray(qt_row1, np.int64),
        qt_ent0=np.asarray(qt_ent0, np.int64), qt_ent1=np.asarray(qt_ent1, np.int64),
        ent=np.asarray(ent, np.int64), qt_order=np.asarray(qt_order, np.int64),
        n_slots=len(slot_tok), slot_tok=np.asarray(slot_tok, np.int64), blk_slot=blk_slot,
        pairs=pairs,
    )
    q = {}
    if leaf1 is not None:
        r1, r2 = [], []
        for a, b in zip(np.asarray(leaf1), np.asarray(leaf2)):
            for lf, out in ((int(a), r1), (int(b), r2)):
                if lf < 0 or lf >= nb:
                    raise PlanError(ERR_INVALID_ARG, f"question leaf {lf} out of range")
                s = int(blk_slot[block_map[lf]])
                if s < 0:
                    raise PlanError(ERR_INVALID_ARG, f"question block {lf} is not a leaf")
                out.append(s)
        q = dict(r1=np.asarray(r1, np.int64), r2=np.asarray(r2, np.int64))
    return plan, q


def plan_forest(forest, **kw):
    """Convenience wrapper over a ``synth.Forest``."""
    return make_plan(forest.parent, forest.length, forest.key, forest.resident, **kw)


def token_block(plan: Plan) -> np.ndarray:
    """Packed block index of every packed token."""
    out = np.zeros(plan.n_tot, np.int64)
    for i in range(plan.n_blocks):
        out[plan.blk_start[i]:plan.blk_start[i] + plan.blk_len[i]] = i
    return out


def brute_mask(plan: Plan) -> np.ndarray:
    """Dense visibility matrix [n_tot, n_tot] straight from the page's rule.

    Query i sees key j iff j's block is a proper ancestor of i's block (walking
    parent links), or both sit in the same block and j <= i.  Uses only the
    block parent links and block ranges, not the subtree ends.
    """
    blk = token_block(plan)
    n = plan.n_tot
    m = np.zeros((n, n), bool)
    anc = []
    for b in range(plan.n_blocks):
        s, x = set(), plan.blk_parent[b]
        while x >= 0:
            s.add(int(x))
            x = plan.blk_parent[x]
        anc.append(s)
    for i in range(n):
        bi = blk[i]
        for j in range(n):
            bj = blk[j]
            m[i, j] = (bj in anc[bi]) or (bj == bi and j <= i)
    return m


def mask_from_tables(plan: Plan) -> np.ndarray:
    """Visibility rebuilt from the packed tables (interval rule j<=i<send[j])."""
    n = plan.n_tot
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return (j <= i) & (i < plan.send[:n][None, :])


def path_tokens(plan: Plan, b: int) -> np.ndarray:
    """Packed tokens of the prompt ending with block b (root first)."""
    chain = []
    x = b
    while x >= 0:
        chain.append(x)
        x = plan.blk_parent[x]
    chain.reverse()
    return np.concatenate([np.arange(plan.blk_start[c], plan.blk_start[c] + plan.blk_len[c]) for c in chain])
