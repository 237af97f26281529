"""tree_runtime_step: one call per batch must give exactly what the separate calls give.

The runtime chains the plan transfer, tree_rope, tree_attn_fwd and readout_decide on one
stream with programmatic dependent launches and two alternating plan buffers; every
output is compared bit for bit with the same calls made one by one, and the whole chain
once more against the oracle.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import plan as oplan
from oracle import readout as ordo
from oracle import rope as orope

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import prefix_tree_packed_gb300 as lib
    return lib


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


class Batch:
    """Inputs of one batch on the device, and the separate-call chain as the reference."""

    def __init__(self, lib, forest, hq, hkv, d, seed, max_fwd=8192, leaf1=None, leaf2=None, theta=500000.0,
                 stride=8):
        kw = dict(leaf1=leaf1, leaf2=leaf2) if leaf1 is not None else {}
        self.lib, self.hq, self.hkv, self.d, self.theta, self.stride = lib, hq, hkv, d, theta, stride
        self.spec = lib.Spec.from_forest(forest, max_fwd=max_fwd, **kw)
        self.plan = lib.Plan.from_forest(forest, max_fwd=max_fwd, **kw)
        i = self.plan.info
        self.info = i
        self.q, self.k, self.v = synth.draw_qkv(i.n_fwd, i.n_tot, hq, hkv, d, seed)
        self.tab = _dev(lib.rope_table(i.max_pos, d, theta))
        rng = np.random.default_rng(seed + 5)
        self.nq = i.n_questions
        self.logits = (rng.standard_normal((max(i.n_slots, 1), stride)) * 2).astype(np.float32)
        self.n = rng.integers(2, stride + 1, max(self.nq, 1)).astype(np.int32)
        self.T = rng.choice([0.7, 1.0, 1.3], max(self.nq, 1)).astype(np.float32)

    def buffers(self):
        b = dict(q=_dev(self.q), k=_dev(self.k), v=_dev(self.v),
                 o=torch.zeros((self.info.n_fwd, self.hq, self.d), dtype=torch.float16, device="cuda"),
                 logits=_dev(self.logits), n=_dev(self.n), T=_dev(self.T),
                 pc=torch.full((max(self.nq, 1), self.stride), -1.0, device="cuda"),
                 ch=torch.full((max(self.nq, 1),), -9, dtype=torch.int32, device="cuda"),
                 st=torch.zeros(1, dtype=torch.int32, device="cuda"))
        return b

    def step(self, rt, b, stream=None):
        return rt.step(self.spec, b["q"], b["k"], b["v"], b["o"], self.tab, self.info.max_pos, self.hq, self.hkv,
                       self.d, logits=b["logits"], stride=self.stride, n_letters=b["n"], temperature=b["T"],
                       p_cal=b["pc"], choice=b["ch"], status=b["st"], stream=stream)

    def reference(self):
        """The same batch through the separate calls."""
        lib, i = self.lib, self.info
        b = self.buffers()
        dev = torch.empty(i.dev_bytes, dtype=torch.uint8, device="cuda")
        s = torch.cuda.current_stream()
        self.plan.upload(dev, i.dev_bytes, s)
        work = torch.zeros(2, dtype=torch.int32, device="cuda")
        for c in range(i.n_chunks):
            ci = self.plan.chunk(c)
            rows = slice(ci.q0 - i.n_res, ci.q1 - i.n_res)
            lib.tree_rope(self.plan, dev, c, b["q"][rows], b["k"], self.hq, self.hkv, self.d, self.tab, i.max_pos, s)
            lib.tree_attn_fwd(self.plan, dev, c, b["q"][rows], b["k"], b["v"], b["o"][rows], None, self.hq, self.hkv,
                              self.d, status=b["st"], stream=s, work=work)
        if self.nq:
            base = dev.data_ptr()
            lib.readout_decide(b["logits"], self.stride, base + i.off_r1, base + i.off_r2, b["n"], b["T"], self.nq,
                               b["pc"], None, b["ch"], b["st"], s)
        torch.cuda.synchronize()
        return b


def _same(got, want, nq):
    assert int(got["st"].item()) == 0
    for key in ("q", "k", "o"):
        assert torch.equal(got[key], want[key]), key
    if nq:
        assert torch.equal(got["pc"], want["pc"])
        assert torch.equal(got["ch"], want["ch"])


def _rt(lib, max_plan_bytes=1 << 20, max_chunks=8):
    return lib.Runtime(max_plan_bytes, max_chunks)


def test_runtime_step_matches_separate_calls_and_oracle(lib):
    w = synth.workload(2)
    bt = Batch(lib, w.forest, w.hq, w.hkv, w.d, w.seed, leaf1=w.leaf1, leaf2=w.leaf2, theta=w.theta)
    rt = _rt(lib)
    got = bt.buffers()
    info = bt.step(rt, got)
    torch.cuda.synchronize()
    assert info.n_fwd == bt.info.n_fwd and info.n_questions == bt.nq
    _same(got, bt.reference(), bt.nq)
    # and the chain against the oracle
    p, qm = oplan.plan_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
    qr, kr = orope.apply_plan(p, bt.q, bt.k, w.theta)
    ref = oatt.attend_paths(p, qr, kr, bt.v)
    assert np.abs(got["o"].float().cpu().numpy() - ref).max() <= 2e-3
    ref_pc, _, _ = ordo.decide(bt.logits, qm["r1"], qm["r2"], bt.n, bt.T, bt.stride)
    assert np.abs(got["pc"].cpu().numpy() - ref_pc).max() <= 1e-5
    rt.close()


def test_runtime_consecutive_steps_of_different_batches(lib):
    """Steps queued back to back without synchronising alternate the plan buffers."""
    rng = np.random.default_rng(77)
    batches = []
    w1, w3 = synth.workload(1), synth.workload(3)
    batches.append(Batch(lib, w1.forest, w1.hq, w1.hkv, w1.d, 1, leaf1=w1.leaf1, leaf2=w1.leaf2))
    batches.append(Batch(lib, w3.forest, w3.hq, w3.hkv, w3.d, 3))
    for seed in range(4):
        while True:
            f = synth.random_forest(rng, n_roots=int(rng.integers(1, 4)), max_blocks=int(rng.integers(3, 25)),
                                    max_len=int(rng.integers(1, 150)), resident_root=bool(seed % 2))
            try:
                oplan.plan_forest(f, max_fwd=128)
                break
            except oplan.PlanError:
                continue
        hq, hkv, d = [(4, 4, 64), (8, 2, 128), (6, 2, 64), (4, 2, 128)][seed]
        batches.append(Batch(lib, f, hq, hkv, d, 10 + seed, max_fwd=128))   # several chunks
    rt = _rt(lib, max_chunks=64)
    outs = []
    for bt in batches + batches[:2]:
        b = bt.buffers()
        bt.step(rt, b)
        outs.append((bt, b))
    torch.cuda.synchronize()
    for bt, b in outs:
        _same(b, bt.reference(), bt.nq)
    rt.close()


def test_runtime_capacity_checked(lib):
    w = synth.workload(2)
    bt = Batch(lib, w.forest, w.hq, w.hkv, w.d, w.seed, leaf1=w.leaf1, leaf2=w.leaf2)
    rt = _rt(lib, max_plan_bytes=1024)
    with pytest.raises(lib.TreeError) as e:
        bt.step(rt, bt.buffers())
    assert e.value.code == lib.TREE_ERR_UNSUPPORTED
    rt.close()
    w4 = synth.workload(4)
    spec = lib.Spec.from_forest(w4.forest, max_fwd=w4.max_fwd)
    rt = _rt(lib, max_chunks=2)
    x = torch.zeros(16, dtype=torch.float16, device="cuda")
    with pytest.raises(lib.TreeError) as e:
        rt.step(spec, x, x, x, x, torch.zeros(16, device="cuda"), 1 << 20, 32, 8, 128)
    assert e.value.code == lib.TREE_ERR_UNSUPPORTED
    rt.close()


def test_queue_batches_run_through_the_runtime(lib):
    """Requests -> queue -> batches (merged prefix trees) -> one runtime step each; every step equals
    the separate calls on the same batch, and the attention equals the oracle on the batch's forest."""
    q = lib.Queue(resident_keys=[1])
    rng = np.random.default_rng(31)
    for rid in range(12):
        doc = int(rng.integers(0, 3))
        prompts, qs = [], []
        for qi in range(int(rng.integers(1, 3))):
            qkey = int(rng.integers(1, 1 << 40))
            for o in range(2):
                prompts.append([(1, 53), (100 + doc, 1500 + 1000 * doc), (qkey, int(rng.integers(10, 60))),
                                (int(rng.integers(1, 1 << 40)), int(rng.integers(5, 20)))])
            qs.append((len(prompts) - 2, len(prompts) - 1))
        q.push(rid, float(rid), prompts, qs)
    rt = _rt(lib, max_chunks=8)
    steps = 0
    now = 20.0
    while True:
        b = q.pop(now)
        if b is None:
            break
        forest = synth.Forest(b.parent, b.length, b.key, b.resident)
        bt = Batch(lib, forest, 8, 2, 64, 40 + steps, leaf1=b.leaf1, leaf2=b.leaf2)
        assert bt.info.n_fwd == b.cost
        got = bt.buffers()
        bt.step(rt, got)
        torch.cuda.synchronize()
        _same(got, bt.reference(), bt.nq)
        p, _ = oplan.plan_forest(forest, leaf1=b.leaf1, leaf2=b.leaf2)
        qr, kr = orope.apply_plan(p, bt.q, bt.k, 500000.0)
        assert np.abs(got["o"].float().cpu().numpy() - oatt.attend_paths(p, qr, kr, bt.v)).max() <= 2e-3
        steps += 1
        now += 5.0
    assert steps >= 2 and q.info() == (0, 0)
    rt.close()


def _pinned(x):
    return torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


def test_runtime_host_buffer_steps(lib):
    """tree_runtime_step_host: inputs and outputs in page-locked host memory, batches issued back to
    back (the runtime's two device sets in turn, uploads on its copy stream); every batch's output
    and decisions equal the separate calls on the same batch bit for bit, p_avg the oracle's."""
    w = synth.workload(2)
    stride = 8
    batches = [Batch(lib, w.forest, w.hq, w.hkv, w.d, w.seed + s, leaf1=w.leaf1, leaf2=w.leaf2, theta=w.theta,
                     stride=stride) for s in range(3)]
    rng = np.random.default_rng(12)
    while True:  # a batch without questions, several chunks
        f = synth.random_forest(rng, n_roots=3, max_blocks=20, max_len=150, resident_root=True)
        try:
            oplan.plan_forest(f, max_fwd=8192)
            break
        except oplan.PlanError:
            continue
    batches.insert(1, Batch(lib, f, w.hq, w.hkv, w.d, 99, theta=w.theta, stride=stride))
    rt = _rt(lib)
    with pytest.raises(lib.TreeError) as e:   # no device sets yet
        bt = batches[0]
        rt.step_host(bt.spec, _pinned(bt.q), _pinned(bt.k), _pinned(bt.v), bt.tab, bt.info.max_pos)
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    rt.attach_io(max_fwd=max(b.info.n_fwd for b in batches), max_tot=max(b.info.n_tot for b in batches), hq=w.hq,
                 hkv=w.hkv, d=w.d, stride=stride, max_slots=max(b.info.n_slots for b in batches),
                 max_questions=max(b.nq for b in batches))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for bt in batches + batches[:2]:
        i, nq = bt.info, bt.nq
        h = dict(q=_pinned(bt.q), k=_pinned(bt.k), v=_pinned(bt.v), logits=_pinned(bt.logits), n=_pinned(bt.n),
                 T=_pinned(bt.T), o=torch.full((i.n_fwd, bt.hq, bt.d), 7.0, dtype=torch.float16).pin_memory(),
                 pc=torch.full((max(nq, 1), stride), -1.0).pin_memory(),
                 pa=torch.full((max(nq, 1), stride), -1.0).pin_memory(),
                 ch=torch.full((max(nq, 1),), -9, dtype=torch.int32).pin_memory())
        info = rt.step_host(bt.spec, h["q"], h["k"], h["v"], bt.tab, i.max_pos, o=h["o"], logits=h["logits"],
                            n_letters=h["n"], temperature=h["T"], p_cal=h["pc"], p_avg=h["pa"], choice=h["ch"],
                            status=st)
        assert info.n_fwd == i.n_fwd and info.n_questions == nq
        outs.append((bt, h))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for bt, h in outs:
        ref = bt.reference()
        assert torch.equal(h["o"], ref["o"].cpu())
        if bt.nq:
            assert torch.equal(h["pc"], ref["pc"].cpu())
            assert torch.equal(h["ch"], ref["ch"].cpu())
            _, qm = oplan.plan_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
            _, ref_pa, _ = ordo.decide(bt.logits, qm["r1"], qm["r2"], bt.n, bt.T, stride)
            assert np.abs(h["pa"].numpy() - ref_pa).max() <= 1e-5
        else:
            assert float(h["pc"][0, 0]) == -1.0 and int(h["ch"][0]) == -9   # nothing to decide: untouched
    rt.close()


def test_runtime_host_capacity_checked(lib):
    w = synth.workload(2)
    bt = Batch(lib, w.forest, w.hq, w.hkv, w.d, w.seed, leaf1=w.leaf1, leaf2=w.leaf2)
    rt = _rt(lib)
    rt.attach_io(max_fwd=bt.info.n_fwd - 128, max_tot=bt.info.n_tot, hq=w.hq, hkv=w.hkv, d=w.d, stride=8,
                 max_slots=bt.info.n_slots, max_questions=bt.nq)
    h = [_pinned(x) for x in (bt.q, bt.k, bt.v, bt.logits, bt.n, bt.T)]
    with pytest.raises(lib.TreeError) as e:
        rt.step_host(bt.spec, h[0], h[1], h[2], bt.tab, bt.info.max_pos, logits=h[3], n_letters=h[4],
                     temperature=h[5])
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    with pytest.raises(lib.TreeError) as e:
        rt.attach_io(max_fwd=128, max_tot=128, hq=6, hkv=4, d=64)   # hq not a multiple of hkv
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    rt.close()
