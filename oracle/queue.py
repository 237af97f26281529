"""Oracle request planner: request cost, HRRN / FIFO order, batch formation.

Follows the basal-rs Architecture page, "01 / Request path" (Validation and
planning; HRRN queue; Batch and prefix tree) and "04 / Scheduling":

* a request's cost is the number of tokens to compute when shared prefixes are
  counted once: here, the total length of the distinct prompt prefixes that
  end in a block, each prefix taken as the tuple of (key, length) pairs from
  the root; a block with key 0 is unique, resident roots (the template) are
  free;
* the queue serves the request with the highest
  (waiting time + estimated runtime) / estimated runtime, the estimate being
  cost x ms_per_token; fifo serves by arrival;
* requests costing more than long_tokens (0: no long lane) wait in a separate
  long lane; short batches go first, a long request runs alone;
* a short batch is the first request in schedule order and each later one
  whose prompts fit: the batch's cost, shared prefixes once across requests,
  stays within max_batch_tokens.

Readings where the page is silent, stated in the design notes: ties in
priority go to the earlier arrival, then to the earlier push; a request that
would make a row (tree) longer than max_row, add a second resident root, or
turn a readout prompt of the batch into a strict prefix of another prompt does
not fit; "fits" is checked for every later request, not only the next one.

Plain Python sets of tuples, no trie: a different construction from the
library's.  Test infrastructure only (see the package docstring).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from itertools import count


@dataclass
class Request:
    id: int
    arrival: float
    prompts: list            # [[(key, length), ...], ...] root first
    questions: list = field(default_factory=list)  # [(prompt1, prompt2), ...]
    seq: int = 0


def _paths(prompts, uniq):
    """Distinct prefixes of the prompts; key-0 blocks get a fresh identity per occurrence."""
    out = []
    for p in prompts:
        ident = []
        for key, length in p:
            ident.append((key, length) if key != 0 else ("u", next(uniq), length))
            out.append(tuple(ident))
    return out


def prompt_ids(prompts, uniq):
    """The full prefix (identity tuple) of each prompt, with the same key-0 rule."""
    res = []
    for p in prompts:
        ident = []
        for key, length in p:
            ident.append((key, length) if key != 0 else ("u", next(uniq), length))
        res.append(tuple(ident))
    return res


def cost_of(prefixes, resident_keys) -> int:
    """Tokens of the distinct prefixes, resident roots excluded."""
    tot = 0
    for pre in set(prefixes):
        last = pre[-1]
        if len(pre) == 1 and last[0] in resident_keys and last[0] != 0 and last[0] != "u":
            continue
        tot += last[-1]
    return tot


def request_cost(prompts, resident_keys=()) -> int:
    return cost_of(_paths(prompts, count()), set(resident_keys))


def priority(cost: int, arrival: float, now: float, ms_per_token: float) -> float:
    est = max(cost, 1) * ms_per_token
    return (max(0.0, now - arrival) + est) / est


def schedule(reqs, costs, now, ms_per_token, fifo=False):
    """Requests in the order the queue serves them."""
    if fifo:
        return sorted(reqs, key=lambda r: (r.arrival, r.seq))
    return sorted(reqs, key=lambda r: (-priority(costs[r.id], r.arrival, now, ms_per_token), r.arrival, r.seq))


class Queue:
    def __init__(self, max_batch_tokens=8192, long_tokens=4096, fifo=False, ms_per_token=0.01,
                 max_depth=8, max_row=32768, resident_keys=()):
        self.max_batch_tokens, self.long_tokens, self.fifo = max_batch_tokens, long_tokens, fifo
        self.ms_per_token, self.max_depth, self.max_row = ms_per_token, max_depth, max_row
        self.resident = set(resident_keys)
        self.reqs: list[Request] = []
        self.costs: dict[int, int] = {}
        self._seq = count()

    def push(self, rid, arrival, prompts, questions=()) -> int:
        c = request_cost(prompts, self.resident)
        self.reqs.append(Request(rid, arrival, [list(p) for p in prompts], list(questions), next(self._seq)))
        self.costs[rid] = c
        return c

    def cancel(self, rid):
        self.reqs = [r for r in self.reqs if r.id != rid]

    def _long(self, r):
        return self.long_tokens > 0 and self.costs[r.id] > self.long_tokens

    def _fits(self, members):
        """Batch cost, rows, resident roots and readout leaves of a set of requests."""
        uniq = count()
        prefixes, readout = [], set()
        for r in members:
            ids = prompt_ids(r.prompts, uniq)
            for pid in ids:
                for k in range(1, len(pid) + 1):
                    prefixes.append(pid[:k])
            for a, b in r.questions:
                readout.add(ids[a])
                readout.add(ids[b])
        pset = set(prefixes)
        for ro in readout:
            if any(len(p) > len(ro) and p[:len(ro)] == ro for p in pset):
                return None
        rows = {}
        for p in pset:
            rows[p[0]] = rows.get(p[0], 0) + p[-1][-1]
        if any(v > self.max_row for v in rows.values()):
            return None
        res_roots = {p for p in pset if len(p) == 1 and p[0][0] in self.resident and p[0][0] not in (0, "u")}
        if len(res_roots) > 1:
            return None
        return cost_of(prefixes, self.resident)

    def pop(self, now):
        """(lane, [ids], cost) of the next batch, or None."""
        short = [r for r in self.reqs if not self._long(r)]
        lng = [r for r in self.reqs if self._long(r)]
        lane, pool = (0, short) if short else (1, lng)
        if not pool:
            return None
        order = schedule(pool, self.costs, now, self.ms_per_token, self.fifo)
        members = [order[0]]
        cost = self._fits(members)
        if lane == 0:
            for r in order[1:]:
                c = self._fits(members + [r])
                if c is not None and c <= self.max_batch_tokens:
                    members.append(r)
                    cost = c
        taken = {r.id for r in members}
        self.reqs = [r for r in self.reqs if r.id not in taken]
        return lane, [r.id for r in members], cost
