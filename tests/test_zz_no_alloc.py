"""tree_attn_fwd_noalloc on the GPU, checked against tree_attn_fwd.

Some callers of this library cannot give it device scratch memory: a plain C
host program that links only this library and has no device allocator of its
own, or an application whose device memory is owned by another runtime's pool,
where a private cudaMalloc would slip past that pool's accounting and stall the
whole device while it runs.  For them the library keeps the attention kernel's
work counters in a small device array of its own; this file checks that the
results are the ones the caller-counter entry point gives, call after call.

It sits in a file of its own, collected last, so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest

import synth
from oracle import plan as oplan
from oracle import rope as orope

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import prefix_tree_packed_gb300 as lib
    return lib


def _setup(lib, forest, hq, hkv, d, seed, max_fwd):
    plan = lib.Plan.from_forest(forest, max_fwd=max_fwd)
    i = plan.info
    dev = torch.empty(i.dev_bytes, dtype=torch.uint8, device="cuda")
    plan.upload(dev, i.dev_bytes, torch.cuda.current_stream())
    p, _ = oplan.plan_forest(forest, max_fwd=max_fwd)
    q, k, v = synth.draw_qkv(p.n_fwd, p.n_tot, hq, hkv, d, seed)
    qr, kr = orope.apply_plan(p, q, k, 500000.0)
    to = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return plan, dev, to(qr), to(kr), to(v)


def _compare(lib, forest, hq, hkv, d, seed, max_fwd=8192):
    """Every chunk twice through the entry point without allocation, all calls on one stream with
    a single synchronize at the end, against tree_attn_fwd with a caller counter.  Only the home
    of the work counter differs and every work item is computed the same way whichever CTA takes
    it, so the outputs must be the same bits."""
    plan, dev, q, k, v = _setup(lib, forest, hq, hkv, d, seed, max_fwd)
    i = plan.info
    s = torch.cuda.current_stream()
    work = torch.zeros(2, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    refs, outs = [], []
    for c in range(i.n_chunks):
        ci = plan.chunk(c)
        a, b = ci.q0 - i.n_res, ci.q1 - i.n_res
        ref = torch.empty((b - a, hq, d), dtype=torch.float16, device="cuda")
        lib.tree_attn_fwd(plan, dev, c, q[a:b], k, v, ref, None, hq, hkv, d, status=status, stream=s, work=work)
        refs.append(ref)
    for _ in range(2):  # two calls in a row reuse the built-in counter of each chunk
        for c in range(i.n_chunks):
            ci = plan.chunk(c)
            a, b = ci.q0 - i.n_res, ci.q1 - i.n_res
            o = torch.full((b - a, hq, d), float("nan"), dtype=torch.float16, device="cuda")
            lib.tree_attn_fwd_noalloc(plan, dev, c, q[a:b], k, v, o, None, hq, hkv, d, status=status, stream=s)
            outs.append((c, o))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for c, o in outs:
        assert torch.equal(o, refs[c]), f"chunk {c}: max-abs {(o.float() - refs[c].float()).abs().max().item()}"
    assert torch.isfinite(torch.cat([r.float().reshape(-1) for r in refs])).all()


def test_noalloc_matches_tree_attn_fwd_one_chunk(lib):
    w = synth.workload(2)
    _compare(lib, w.forest, w.hq, w.hkv, w.d, w.seed)


def test_noalloc_matches_tree_attn_fwd_several_chunks(lib):
    rng = np.random.default_rng(77)
    f = synth.random_forest(rng, n_roots=2, max_blocks=18, max_len=140, resident_root=True)
    _compare(lib, f, 8, 2, 128, 5, max_fwd=128)


def test_noalloc_rejects_a_caller_counter_and_too_many_chunks(lib):
    w = synth.workload(1)
    plan, dev, q, k, v = _setup(lib, w.forest, w.hq, w.hkv, w.d, w.seed, 8192)
    o = torch.empty_like(q)
    work = torch.zeros(2, dtype=torch.int32, device="cuda")
    p = lib.AttnParams(w.hq, w.hkv, w.d, 0.0, work.data_ptr())
    import ctypes as C
    rc = lib._lib.tree_attn_fwd_noalloc(plan.handle, dev.data_ptr(), 0, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        o.data_ptr(), None, C.byref(p), None, None)
    assert rc == lib.TREE_ERR_INVALID_ARG
    # two 16,500-token rows in 128-token chunks: 258 chunks, more than the built-in counters
    big = lib.Plan([-1, -1], [16500, 16500], max_fwd=128)
    assert big.info.n_chunks > 256
    with pytest.raises(lib.TreeError) as e:
        lib.tree_attn_fwd_noalloc(big, dev, 0, q, k, v, o, None, w.hq, w.hkv, w.d)
    assert e.value.code == lib.TREE_ERR_UNSUPPORTED
