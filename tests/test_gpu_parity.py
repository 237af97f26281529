"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Tolerances:
  plan tables, readout slots, choices      bit-exact
  RoPE outputs (f16)                       within 1 f16 ulp, almost all equal
  attention outputs (f16)                  max-abs 2e-3 against the float64 oracle
  LSE (f32)                                max-abs 1e-3 (natural log units)
  decision probabilities (f32)             max-abs 1e-5
"""
import numpy as np
import pytest

import synth
from oracle import attention as oatt
from oracle import plan as oplan
from oracle import readout as ordo
from oracle import rope as orope

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL_O = 2e-3
ATOL_P = 1e-5


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import prefix_tree_packed_gb300 as lib
    return lib


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


class Run:
    """A plan on the device plus helpers to call the library."""

    def __init__(self, lib, forest, max_fwd=8192, leaf1=None, leaf2=None, tiling=0, pack_heads=0):
        self.lib = lib
        kw = dict(leaf1=leaf1, leaf2=leaf2) if leaf1 is not None else {}
        self.plan = lib.Plan.from_forest(forest, max_fwd=max_fwd, tiling=tiling, pack_heads=pack_heads, **kw)
        self.oplan, self.oq = oplan.plan_forest(forest, max_fwd=max_fwd, **kw)
        i = self.plan.info
        self.dev = torch.empty(i.dev_bytes, dtype=torch.uint8, device="cuda")
        self.plan.upload(self.dev, i.dev_bytes, torch.cuda.current_stream())

    def rope(self, q, k, hq, hkv, d, theta, chunk):
        i = self.plan.info
        tab = _dev(self.lib.rope_table(i.max_pos, d, theta))
        self.lib.tree_rope(self.plan, self.dev, chunk, q, k, hq, hkv, d, tab, i.max_pos,
                           torch.cuda.current_stream())

    def attn(self, q, k, v, hq, hkv, d, chunk, lse=None, status=None, work=None):
        ci = self.plan.chunk(chunk)
        o = torch.empty((ci.q1 - ci.q0, hq, d), dtype=torch.float16, device="cuda")
        self.lib.tree_attn_fwd(self.plan, self.dev, chunk, q, k, v, o, lse, hq, hkv, d,
                               status=status, stream=torch.cuda.current_stream(), work=work)
        return o


def test_staged_upload_matches_plan_image(lib):
    w = synth.workload(2)
    plan = lib.Plan.from_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
    i = plan.info
    want = plan.tables()["image"]
    assert len(want) == i.dev_bytes
    dev = [torch.full((i.dev_bytes,), 0xAB, dtype=torch.uint8, device="cuda") for _ in range(2)]
    pin = torch.empty(i.dev_bytes, dtype=torch.uint8).pin_memory()
    cs = torch.cuda.Stream()
    plan.upload_staged(dev[0], i.dev_bytes, pin, i.dev_bytes, cs)
    cs.synchronize()
    plan.upload(dev[1], i.dev_bytes, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert np.array_equal(dev[0].cpu().numpy(), want)
    assert np.array_equal(dev[1].cpu().numpy(), want)


def _f16_ulp(x):
    x = np.abs(x.astype(np.float32))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -14)))
    return 2.0 ** (e - 10)


# ---------------------------------------------------------------- readout

def _check_readout(lib, logits, r1, r2, n, T, stride):
    nq = len(r1)
    pc = torch.full((nq, stride), -7.0, device="cuda")
    pa = torch.full((nq, stride), -7.0, device="cuda")
    ch = torch.full((nq,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.readout_decide(_dev(logits), stride, _dev(np.int32(r1)), _dev(np.int32(r2)), _dev(np.int32(n)),
                       _dev(np.float32(T)), nq, pc, pa, ch, st, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_pc, ref_pa, _ = ordo.decide(logits, r1, r2, n, T, stride)
    assert np.abs(pc.cpu().numpy() - ref_pc).max() <= ATOL_P
    assert np.abs(pa.cpu().numpy() - ref_pa).max() <= ATOL_P
    got = ch.cpu().numpy()
    want = ordo.choice_f32(logits, r1, r2, n)
    diff = np.nonzero(got != want)[0]
    # an f32 near-tie may legitimately resolve either way; both must be maxima of p
    for q in diff:
        top = np.sort(ref_pa[q])[::-1]
        assert top[0] - top[1] < 1e-6 and abs(ref_pa[q, got[q]] - top[0]) < 1e-6
    assert len(diff) <= max(1, nq // 10000)


def test_readout_worked_example(lib):
    logits = np.array([[3.2, 0.9, -0.4], [0.4, 1.1, 2.6]], np.float32)
    _check_readout(lib, logits, [0], [1], [3], [1.0], 3)


def test_readout_workload_one_and_two(lib):
    for n in (1, 2):
        w = synth.workload(n)
        p, q = oplan.plan_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
        logits = synth.draw_logits(p.n_slots, w.letter_stride, w.logit_sigma, w.seed)
        _check_readout(lib, logits, q["r1"], q["r2"], w.n_letters, w.temperature, w.letter_stride)


def test_readout_65536_questions(lib):
    b = synth.draw_readout_batch()
    _check_readout(lib, b["logits"], b["r1"], b["r2"], b["n_letters"], b["temperature"], b["stride"])


@pytest.mark.parametrize("with_avg", [False, True])
def test_readout_262144_questions_sampled(lib, with_avg):
    """A batch of 262,144 questions (8,192 tiles, more than one wave of resident warps): sampled
    questions against the oracle, every question of the first and last tiles and a stretch across
    the middle included; with and without p_avg."""
    b = synth.draw_readout_batch(262144, seed=9)
    nq, stride = len(b["r1"]), b["stride"]
    pc = torch.full((nq, stride), -7.0, device="cuda")
    pa = torch.full((nq, stride), -7.0, device="cuda") if with_avg else None
    ch = torch.full((nq,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.readout_decide(_dev(b["logits"]), stride, _dev(b["r1"]), _dev(b["r2"]), _dev(b["n_letters"]),
                       _dev(b["temperature"]), nq, pc, pa, ch, st, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rng = np.random.default_rng(3)
    qs = np.unique(np.concatenate([np.arange(64), np.arange(nq - 64, nq), np.arange(131000, 131400),
                                   rng.choice(nq, 4000, replace=False)]))
    ref_pc, ref_pa, _ = ordo.decide(b["logits"], b["r1"][qs], b["r2"][qs], b["n_letters"][qs],
                                    b["temperature"][qs], stride)
    assert np.abs(pc.cpu().numpy()[qs] - ref_pc).max() <= ATOL_P
    if with_avg:
        assert np.abs(pa.cpu().numpy()[qs] - ref_pa).max() <= ATOL_P
    got = ch.cpu().numpy()[qs]
    want = ordo.choice_f32(b["logits"], b["r1"][qs], b["r2"][qs], b["n_letters"][qs])
    for k in np.nonzero(got != want)[0]:
        top = np.sort(ref_pa[k])[::-1]
        assert top[0] - top[1] < 1e-6 and abs(ref_pa[k, got[k]] - top[0]) < 1e-6


@pytest.mark.parametrize("stride,nmax", [(1, 1), (3, 2), (10, 10), (16, 16), (17, 17), (31, 20), (32, 32), (33, 33),
                                         (40, 33), (255, 255), (300, 255)])
def test_readout_sizes(lib, stride, nmax):
    rng = np.random.default_rng(stride)
    nq = 333
    logits = (rng.standard_normal((2 * nq, stride)) * 3).astype(np.float32)
    n = rng.integers(1, nmax + 1, nq)
    n[0] = nmax
    T = rng.choice([0.5, 1.0, 2.0], nq)
    _check_readout(lib, logits, 2 * np.arange(nq), 2 * np.arange(nq) + 1, n, T, stride)


def test_readout_every_exact_stride_scattered_rows(lib):
    """Strides 1..16 each have their own kernel instance: every one, with the two orders' rows
    scattered over the logits buffer (a random permutation) and a ragged last tile."""
    for stride in range(1, 17):
        rng = np.random.default_rng(100 + stride)
        nq = 32 * 9 + 7
        logits = (rng.standard_normal((2 * nq + 5, stride)) * 3).astype(np.float32)
        rows = rng.permutation(2 * nq + 5)[:2 * nq]
        n = rng.integers(1, stride + 1, nq)
        n[0] = stride
        T = rng.choice([0.5, 1.0, 2.0], nq)
        _check_readout(lib, logits, rows[:nq], rows[nq:], n, T, stride)


@pytest.mark.parametrize("stride", [10, 7, 20])
def test_readout_unaligned_buffers(lib, stride):
    """Logits, p_cal and p_avg at 4-byte (not 8- or 16-byte) aligned addresses: the kernels fall
    back from letter-pair loads and 16-byte stores to single floats, with the same results."""
    rng = np.random.default_rng(7 + stride)
    nq = 32 * 5 + 19
    logits = (rng.standard_normal((2 * nq, stride)) * 3).astype(np.float32)
    n = rng.integers(1, min(stride, 10) + 1, nq)
    T = rng.choice([0.5, 1.0, 2.0], nq)
    lg = torch.zeros(2 * nq * stride + 1, device="cuda")
    lg[1:] = _dev(logits).reshape(-1)
    pcb = torch.full((nq * stride + 1,), -7.0, device="cuda")
    pab = torch.full((nq * stride + 1,), -7.0, device="cuda")
    ch = torch.full((nq,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r1, r2 = np.arange(nq) * 2, np.arange(nq) * 2 + 1
    lib.readout_decide(lg[1:], stride, _dev(np.int32(r1)), _dev(np.int32(r2)), _dev(np.int32(n)),
                       _dev(np.float32(T)), nq, pcb[1:], pab[1:], ch, st, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_pc, ref_pa, _ = ordo.decide(logits, r1, r2, n, T, stride)
    assert float(pcb[0]) == -7.0 and float(pab[0]) == -7.0
    assert np.abs(pcb[1:].cpu().numpy().reshape(nq, stride) - ref_pc).max() <= ATOL_P
    assert np.abs(pab[1:].cpu().numpy().reshape(nq, stride) - ref_pa).max() <= ATOL_P


def test_readout_bad_arguments_flagged(lib):
    logits = np.zeros((4, 6), np.float32)
    pc = torch.full((2, 6), -7.0, device="cuda")
    ch = torch.full((2,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.readout_decide(_dev(logits), 6, _dev(np.int32([0, 2])), _dev(np.int32([1, 3])), _dev(np.int32([3, 7])),
                       _dev(np.float32([1.0, 1.0])), 2, pc, None, ch, st, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert int(st.item()) == lib.TREE_ERR_INVALID_ARG
    assert ch.cpu().tolist() == [0, -1]           # equal logits: lowest index; bad question: -1
    assert np.all(pc.cpu().numpy()[1] == 0)
    st.zero_()
    lib.readout_decide(_dev(logits), 6, _dev(np.int32([0])), _dev(np.int32([1])), _dev(np.int32([3])),
                       _dev(np.float32([0.0])), 1, pc, None, ch, st, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert int(st.item()) == lib.TREE_ERR_INVALID_ARG
    lib.readout_decide(0, 6, 0, 0, 0, 0, 0, 0)    # no questions: no-op
    with pytest.raises(lib.TreeError):
        lib.readout_decide(_dev(logits), 0, 0, 0, 0, 0, 1, pc)


# ---------------------------------------------------------------- RoPE

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_rope_workloads(lib, n):
    w = synth.workload(n)
    r = Run(lib, w.forest, w.max_fwd)
    p = r.oplan
    q, k, v = synth.draw_qkv(p.n_fwd, p.n_tot, w.hq, w.hkv, w.d, w.seed)
    qr_ref, kr_ref = orope.apply_plan(p, q, k, w.theta)
    kd = _dev(k)
    qr = np.empty_like(q)
    for c in range(p.n_chunks):
        ci = r.plan.chunk(c)
        qd = _dev(q[ci.q0 - p.n_res: ci.q1 - p.n_res])
        r.rope(qd, kd, w.hq, w.hkv, w.d, w.theta, c)
        torch.cuda.synchronize()
        qr[ci.q0 - p.n_res: ci.q1 - p.n_res] = qd.cpu().numpy()
    kr = kd.cpu().numpy()
    for got, ref, x in ((qr, qr_ref, q), (kr, kr_ref, k)):
        d = np.abs(got.astype(np.float64) - ref.astype(np.float64))
        # the kernel evaluates x1*cos - x2*sin in f32 from an f32 table: before the
        # final f16 rounding it is within a few f32 ulps of (|x1| + |x2|) of the
        # exact value, so after rounding it may differ by one f16 ulp plus that
        xa = np.abs(x.astype(np.float64))
        h = x.shape[-1] // 2
        partner = np.concatenate([xa[..., h:], xa[..., :h]], axis=-1)
        bound = _f16_ulp(ref) + 2.0 ** -20 * (xa + partner)
        assert np.all(d <= bound), f"worst excess {(d - bound).max()}"
        assert (d > 0).mean() < 1e-3
    assert np.array_equal(kr[: p.n_res], k[: p.n_res])     # resident rows untouched


def test_rope_keys_only(lib):
    """q=None rotates the keys exactly as the call on queries and keys does, and nothing else."""
    w = synth.workload(3)
    r = Run(lib, w.forest, w.max_fwd)
    p, i = r.oplan, r.plan.info
    q, k, _ = synth.draw_qkv(p.n_fwd, p.n_tot, w.hq, w.hkv, w.d, w.seed)
    tab = _dev(lib.rope_table(i.max_pos, w.d, w.theta))
    s = torch.cuda.current_stream()
    ka, kb, qd = _dev(k), _dev(k), _dev(q)
    lib.tree_rope(r.plan, r.dev, 0, qd, ka, w.hq, w.hkv, w.d, tab, i.max_pos, s)
    lib.tree_rope(r.plan, r.dev, 0, None, kb, w.hq, w.hkv, w.d, tab, i.max_pos, s)
    torch.cuda.synchronize()
    assert torch.equal(ka, kb)
    assert not torch.equal(kb, _dev(k))


# ---------------------------------------------------------------- attention

def _boundary_rows(p):
    """Forward rows on either side of every chunk seam and of every block start and end:
    the rows where the visible key set changes."""
    rows = set()
    for c in range(p.n_chunks):
        a, b = int(p.chunk_q0[c]) - p.n_res, int(p.chunk_q1[c]) - p.n_res
        rows.update((a, a + 1, b - 2, b - 1))
    for b in range(p.n_blocks):
        s, e = int(p.blk_start[b]), int(p.blk_start[b] + p.blk_len[b])
        rows.update(t - p.n_res for t in (s, s + 1, e - 2, e - 1))
    return sorted(r for r in rows if 0 <= r < p.n_fwd)


def _attn_check(lib, forest, hq, hkv, d, seed, max_fwd=8192, full=True, rows_per_chunk=48, lse=True,
                dynamic=True, tiling=0, extra_rows=(), pack_heads=0):
    r = Run(lib, forest, max_fwd, tiling=tiling, pack_heads=pack_heads)
    work = torch.zeros(2, dtype=torch.int32, device="cuda") if dynamic else None
    p = r.oplan
    q, k, v = synth.draw_qkv(p.n_fwd, p.n_tot, hq, hkv, d, seed)
    qr, kr = orope.apply_plan(p, q, k, 500000.0)     # oracle RoPE output is the attention input
    kd, vd = _dev(kr), _dev(v)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs, lses = [], []
    for c in range(p.n_chunks):
        ci = r.plan.chunk(c)
        qd = _dev(qr[ci.q0 - p.n_res: ci.q1 - p.n_res])
        ld = torch.full((ci.q1 - ci.q0, hq), np.nan, device="cuda") if lse else None
        o = r.attn(qd, kd, vd, hq, hkv, d, c, lse=ld, status=st, work=work)
        torch.cuda.synchronize()
        if work is not None:
            assert work.cpu().tolist() == [0, 0]      # the last CTA hands the counter back zeroed
        outs.append(o.float().cpu().numpy())
        if lse:
            lses.append(ld.cpu().numpy())
    assert int(st.item()) == 0
    got = np.concatenate(outs)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(seed + 7)
    if full:
        ref = oatt.attend_paths(p, qr, kr, v)
        err = np.abs(got - ref)
        assert err.max() <= ATOL_O, f"max err {err.max()} at {np.unravel_index(err.argmax(), err.shape)}"
        rows = rng.choice(p.n_fwd, min(p.n_fwd, 64), replace=False)
    else:
        rows = []
        for c in range(p.n_chunks):
            a, b = int(p.chunk_q0[c]) - p.n_res, int(p.chunk_q1[c]) - p.n_res
            rows += [a, b - 1] + list(rng.integers(a, b, rows_per_chunk - 2))
        rows = np.unique(np.array(rows + list(extra_rows), dtype=np.int64))
        ref = oatt.attend_rows(p, qr, kr, v, rows)
        err = np.abs(got[rows] - ref)
        assert err.max() <= ATOL_O, f"max err {err.max()}"
    if lse:
        lg = np.concatenate(lses)[rows]
        lr = oatt.lse_rows(p, qr, kr, rows)
        assert np.abs(lg - lr).max() <= 1e-3
    return got


@pytest.mark.parametrize("tiling", [0, 1])
@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_attention_workloads_full(lib, n, tiling):
    w = synth.workload(n)
    _attn_check(lib, w.forest, w.hq, w.hkv, w.d, w.seed, w.max_fwd, full=True, tiling=tiling)


@pytest.mark.parametrize("tiling", [0, 1])
def test_attention_long_row_four_chunks_sampled(lib, tiling):
    """The 32,768-token row in four chunks, on random rows of each chunk plus every row beside a
    chunk seam or a block boundary (the question and option blocks of the last chunk)."""
    w = synth.workload(4)
    p, _ = oplan.plan_forest(w.forest, max_fwd=w.max_fwd)
    seams = _boundary_rows(p)
    assert len(seams) == 76   # 4 per chunk seam and per block edge, shared ones counted once
    _attn_check(lib, w.forest, w.hq, w.hkv, w.d, w.seed, w.max_fwd, full=False, rows_per_chunk=40, tiling=tiling,
                extra_rows=seams)


@pytest.mark.parametrize("tiling", [0, 1])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (6, 2), (32, 32)])
def test_attention_odd_head_ratio_d128(lib, hq, hkv, tiling):
    """At head dim 128 an odd number of q heads per kv head runs the kernel instance that takes one
    q head per work item (one softmax warpgroup, its epilogue deferred behind the next item's first
    tile, P over S in tensor memory): the mixed rows of the Llama-8B-shaped workload, in full."""
    w = synth.workload(3)
    _attn_check(lib, w.forest, hq, hkv, 128, w.seed + hq, w.max_fwd, full=True, tiling=tiling)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 2), (8, 4), (12, 2), (6, 6)])
def test_attention_d64_head_ratios(lib, hq, hkv):
    """Head dim 64 takes a kernel instance by the q/kv head ratio: an even ratio runs two q heads per
    work item (32/8, 16/2, 8/4, 12/2, with one or more pairs per kv head), an odd one a head per item
    (6/6).  The Llama-1B-shaped rows in full, and random forests in chunks."""
    w = synth.workload(2)
    _attn_check(lib, w.forest, hq, hkv, 64, 40 + hq, w.max_fwd, full=True)
    rng = np.random.default_rng(hq * 10 + hkv)
    f = synth.random_forest(rng, n_roots=3, max_blocks=25, max_len=150, dup_prob=0.2, resident_root=True)
    _attn_check(lib, f, hq, hkv, 64, 3, max_fwd=256, full=True, dynamic=False)


@pytest.mark.parametrize("seed", range(6))
def test_attention_random_forests_odd_ratio_d128(lib, seed):
    rng = np.random.default_rng(900 + seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 4)), max_blocks=int(rng.integers(3, 30)),
                            max_len=int(rng.integers(1, 300)), dup_prob=0.2, resident_root=bool(seed % 2))
    try:
        oplan.plan_forest(f, max_fwd=256)
    except oplan.PlanError:
        pytest.skip("forest has no forward tokens")
    hq, hkv = [(3, 3), (6, 2), (5, 1)][seed % 3]
    _attn_check(lib, f, hq, hkv, 128, seed, max_fwd=int(rng.choice([128, 256, 8192])), dynamic=bool(seed % 2),
                tiling=seed % 2)


@pytest.mark.parametrize("seed", range(8))
def test_attention_random_forests(lib, seed):
    rng = np.random.default_rng(500 + seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 4)), max_blocks=int(rng.integers(3, 30)),
                            max_len=int(rng.integers(1, 200)), dup_prob=0.2, resident_root=bool(seed % 2))
    try:
        oplan.plan_forest(f, max_fwd=256)
    except oplan.PlanError:
        pytest.skip("forest has no forward tokens")
    hq, hkv, d = [(4, 4, 64), (8, 2, 128), (4, 1, 64), (6, 3, 128)][seed % 4]
    _attn_check(lib, f, hq, hkv, d, seed, max_fwd=int(rng.choice([128, 256, 8192])), dynamic=bool(seed % 2),
                tiling=seed // 4)


# ---------------------------------------------------------------- gathered key tiles, packed heads

@pytest.mark.parametrize("pack", [0, 4])
@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_attention_gathered_workloads_full(lib, n, pack):
    """Gathered key tiles (tiling 2), alone and with the four q heads of a kv head packed into each
    MMA tile (32 tokens x 4 heads, two such tiles per item sharing its K/V tiles): every workload in
    full.  The tiny tree has one q head per kv head, so it is never packed."""
    w = synth.workload(n)
    if pack and w.hq // w.hkv != pack:
        pytest.skip("the workload's q/kv head ratio is not the packing")
    _attn_check(lib, w.forest, w.hq, w.hkv, w.d, w.seed, w.max_fwd, full=True, tiling=2, pack_heads=pack)


@pytest.mark.parametrize("n", [2, 3, 5])
def test_attention_position_tiled_packed_heads_full(lib, n):
    """Tiling by position with the four q heads of a kv head packed into each MMA tile."""
    w = synth.workload(n)
    _attn_check(lib, w.forest, w.hq, w.hkv, w.d, w.seed, w.max_fwd, full=True, tiling=1, pack_heads=w.hq // w.hkv)


@pytest.mark.parametrize("seed", range(4))
def test_attention_position_tiled_packed_heads_random_forests(lib, seed):
    rng = np.random.default_rng(2100 + seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 4)), max_blocks=int(rng.integers(3, 40)),
                            max_len=int(rng.choice([4, 30, 150])), dup_prob=0.2, resident_root=bool(seed % 2))
    try:
        oplan.plan_forest(f, max_fwd=256)
    except oplan.PlanError:
        pytest.skip("forest has no forward tokens")
    hq, hkv, d = [(8, 2, 64), (8, 4, 128), (16, 2, 64), (32, 8, 128)][seed]
    _attn_check(lib, f, hq, hkv, d, seed, max_fwd=int(rng.choice([128, 256, 8192])), dynamic=bool(seed % 2),
                tiling=1, pack_heads=hq // hkv)


def test_attention_gathered_long_row_sampled(lib):
    w = synth.workload(4)
    p, _ = oplan.plan_forest(w.forest, max_fwd=w.max_fwd)
    _attn_check(lib, w.forest, w.hq, w.hkv, w.d, w.seed, w.max_fwd, full=False, rows_per_chunk=40, tiling=2,
                pack_heads=4, extra_rows=_boundary_rows(p))


@pytest.mark.parametrize("seed", range(10))
def test_attention_gathered_random_forests(lib, seed):
    """Random forests in chunks; packings of 2, 4 and 8 heads (MMA tiles of 64, 32 and 16 tokens per
    head) at head dims 64 and 128, and unpacked gathered tiles with one or two heads per item."""
    rng = np.random.default_rng(1700 + seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 5)), max_blocks=int(rng.integers(3, 60)),
                            max_len=int(rng.choice([4, 20, 150])), dup_prob=0.2, resident_root=bool(seed % 2))
    try:
        oplan.plan_forest(f, max_fwd=256)
    except oplan.PlanError:
        pytest.skip("forest has no forward tokens")
    hq, hkv, d, pack = [(8, 2, 64, 4), (8, 4, 128, 2), (16, 2, 64, 8), (4, 4, 64, 0), (3, 3, 128, 0),
                        (32, 8, 128, 4), (16, 8, 64, 2), (16, 2, 128, 8), (6, 2, 64, 0), (8, 1, 128, 8)][seed]
    _attn_check(lib, f, hq, hkv, d, seed, max_fwd=int(rng.choice([128, 256, 8192])), dynamic=bool(seed % 3),
                tiling=2, pack_heads=pack)


def test_attention_packing_must_match_head_ratio(lib):
    w = synth.workload(5)
    r = Run(lib, w.forest, w.max_fwd, tiling=2, pack_heads=2)
    p = r.oplan
    q = torch.zeros((p.n_fwd, 32, 128), dtype=torch.float16, device="cuda")
    kv = torch.zeros((p.n_tot, 8, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(lib.TreeError):
        r.attn(q, kv, kv, 32, 8, 128, 0)


@pytest.mark.parametrize("n", [2, 5])
def test_attention_round_robin_schedule(lib, n):
    """Without a work counter every CTA takes a fixed share of the items."""
    w = synth.workload(n)
    _attn_check(lib, w.forest, w.hq, w.hkv, w.d, w.seed, w.max_fwd, full=True, dynamic=False)


def test_attention_work_counter_reused_across_calls(lib):
    w = synth.workload(2)
    r = Run(lib, w.forest)
    p = r.oplan
    q, k, v = synth.draw_qkv(p.n_fwd, p.n_tot, w.hq, w.hkv, w.d, w.seed)
    qr, kr = orope.apply_plan(p, q, k, w.theta)
    qd, kd, vd = _dev(qr), _dev(kr), _dev(v)
    work = torch.zeros(2, dtype=torch.int32, device="cuda")
    outs = [r.attn(qd, kd, vd, w.hq, w.hkv, w.d, 0, work=work) for _ in range(3)]
    torch.cuda.synchronize()
    assert work.cpu().tolist() == [0, 0]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    stat = r.attn(qd, kd, vd, w.hq, w.hkv, w.d, 0)
    torch.cuda.synchronize()
    assert torch.equal(stat, outs[0])     # same arithmetic whatever the schedule


def test_attention_chunked_equals_unchunked(lib):
    rng = np.random.default_rng(42)
    f = synth.random_forest(rng, n_roots=2, max_blocks=20, max_len=150, resident_root=True)
    a = _attn_check(lib, f, 8, 2, 64, 3, max_fwd=128, lse=False)
    b = _attn_check(lib, f, 8, 2, 64, 3, max_fwd=8192, lse=False)
    assert np.abs(a - b).max() <= 2 * ATOL_O


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 64), (8, 2, 128), (3, 3, 64)])
def test_attention_timeout_self_test_reports_and_recovers(lib, hq, hkv, d):
    """A wait that runs out (on a barrier nothing arrives on) is reported in the
    status word, writes no output, and leaves the context usable."""
    w = synth.workload(2)
    r = Run(lib, w.forest)
    p = r.oplan
    q, k, v = synth.draw_qkv(p.n_fwd, p.n_tot, hq, hkv, d, 31)
    qr, kr = orope.apply_plan(p, q, k, w.theta)
    qd, kd, vd = _dev(qr), _dev(kr), _dev(v)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    work = torch.zeros(2, dtype=torch.int32, device="cuda")
    o = torch.full((p.n_fwd, hq, d), 7.0, dtype=torch.float16, device="cuda")
    lib.tree_attn_fwd(r.plan, r.dev, 0, qd, kd, vd, o, None, hq, hkv, d, status=st,
                      stream=torch.cuda.current_stream(), work=work, self_test=True)
    torch.cuda.synchronize()
    assert int(st.item()) == lib.TREE_ERR_TIMEOUT
    assert bool((o == 7.0).all())                     # nothing written
    assert work.cpu().tolist() == [0, 0]              # the counter is handed back all the same
    st.zero_()
    got = r.attn(qd, kd, vd, hq, hkv, d, 0, status=st, work=work)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rng = np.random.default_rng(5)
    rows = rng.choice(p.n_fwd, 48, replace=False)
    ref = oatt.attend_rows(p, qr, kr, v, rows)
    assert np.abs(got.float().cpu().numpy()[rows] - ref).max() <= ATOL_O


def test_attention_rejects_bad_shapes(lib):
    w = synth.workload(1)
    r = Run(lib, w.forest)
    x = torch.zeros((96, 4, 64), dtype=torch.float16, device="cuda")
    for hq, hkv, d in ((4, 3, 64), (4, 4, 96), (4, 4, 256)):
        with pytest.raises(lib.TreeError) as e:
            lib.tree_attn_fwd(r.plan, r.dev, 0, x, x, x, x, None, hq, hkv, d)
        assert e.value.code == lib.TREE_ERR_UNSUPPORTED
    with pytest.raises(lib.TreeError) as e:
        lib.tree_attn_fwd(r.plan, r.dev, 1, x, x, x, x, None, 4, 4, 64)
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    with pytest.raises(lib.TreeError) as e:
        lib.tree_attn_fwd(r.plan, r.dev, 0, x.data_ptr() + 2, x, x, x, None, 4, 4, 64)
    assert e.value.code == lib.TREE_ERR_UNSUPPORTED


# ---------------------------------------------------------------- whole path

def test_pipeline_workload_two(lib):
    """Plan -> RoPE -> attention -> readout on the GPU against the oracle chain."""
    w = synth.workload(2)
    r = Run(lib, w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
    p = r.oplan
    q, k, v = synth.draw_qkv(p.n_fwd, p.n_tot, w.hq, w.hkv, w.d, w.seed)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    r.rope(qd, kd, w.hq, w.hkv, w.d, w.theta, 0)
    o = r.attn(qd, kd, vd, w.hq, w.hkv, w.d, 0)
    logits = synth.draw_logits(p.n_slots, w.letter_stride, w.logit_sigma, w.seed)
    i = r.plan.info
    nq = i.n_questions
    pc = torch.empty((nq, w.letter_stride), device="cuda")
    ch = torch.empty(nq, dtype=torch.int32, device="cuda")
    base = r.dev.data_ptr()
    lib.readout_decide(_dev(logits), w.letter_stride, base + i.off_r1, base + i.off_r2, _dev(w.n_letters),
                       _dev(w.temperature), nq, pc, None, ch, None, torch.cuda.current_stream())
    torch.cuda.synchronize()
    qr, kr = orope.apply_plan(p, q, k, w.theta)
    ref = oatt.attend_paths(p, qr, kr, v)
    assert np.abs(o.float().cpu().numpy() - ref).max() <= ATOL_O
    ref_pc, _, _ = ordo.decide(logits, r.oq["r1"], r.oq["r2"], w.n_letters, w.temperature, w.letter_stride)
    assert np.abs(pc.cpu().numpy() - ref_pc).max() <= ATOL_P
    assert np.array_equal(ch.cpu().numpy(), ordo.choice_f32(logits, r.oq["r1"], r.oq["r2"], w.n_letters))
