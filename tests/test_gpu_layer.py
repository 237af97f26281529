"""tree_gemm and tree_rmsnorm (include/tree_layer.h) against the float64 oracle."""
import numpy as np
import pytest

import prefix_tree_packed_gb300 as lib
from oracle import layer as ol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _ulp16(x):
    return np.spacing(np.abs(np.asarray(x, np.float16))).astype(np.float64)


def _close16(got, ref, extra=0.0, ulps=1):
    """At most `ulps` f16 ulps of the reference apart (plus `extra` absolute)."""
    g = np.asarray(got, np.float16).astype(np.float64)
    r = np.asarray(ref, np.float16).astype(np.float64)
    bad = np.abs(g - r) > ulps * _ulp16(r) + extra
    assert not bad.any(), f"{int(bad.sum())} elements off; worst {np.abs(g - r).max():.3g}"


def _inputs(m, n_b, k, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((m, k)).astype(np.float16)
    b = (rng.standard_normal((n_b, k)) / np.sqrt(k)).astype(np.float16)
    r = rng.standard_normal((m, n_b)).astype(np.float16)
    return a, b, r


SHAPES = [(128, 256, 64), (300, 264, 136), (1000, 768, 520), (2048, 3072, 2048), (77, 8, 8), (129, 520, 4096)]


@pytest.mark.parametrize("tile_n", [0, 64, 256])
@pytest.mark.parametrize("m,n,k", SHAPES)
@pytest.mark.parametrize("epi", ["store", "residual", "swiglu"])
def test_gemm_matches_oracle(m, n, k, epi, tile_n):
    dev = torch.device("cuda")
    n_b = 2 * n if epi == "swiglu" else n
    a, b, r = _inputs(m, n_b, k, seed=m + n + k)
    r = r[:, :n].copy()
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    tr = torch.from_numpy(r).to(dev)
    tc = torch.full((m, n), float("nan"), dtype=torch.float16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    code = {"store": lib.GEMM_STORE, "residual": lib.GEMM_RESIDUAL, "swiglu": lib.GEMM_SWIGLU}[epi]
    lib.gemm(ta, tb, tc, m, n, k, code, r=tr if epi == "residual" else None, status=st, tile_n=tile_n)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = ol.gemm(a, b, epi, r)
    # f32 accumulation against float64: one f16 rounding apart, plus the f32 sum's error
    _close16(tc.cpu().numpy(), ref, extra=1e-4)


@pytest.mark.parametrize("m,n,k", [(300, 264, 136), (1000, 768, 520), (77, 8, 8), (129, 520, 4096)])
@pytest.mark.parametrize("epi", ["store", "residual", "swiglu"])
def test_gemm_tile_width_changes_nothing(m, n, k, epi):
    """Narrow and wide tiles give bit-identical outputs (each is the same f32 sum over k)."""
    dev = torch.device("cuda")
    n_b = 2 * n if epi == "swiglu" else n
    a, b, r = _inputs(m, n_b, k, seed=3 * m + n)
    r = r[:, :n].copy()
    ta, tb, tr = (torch.from_numpy(x).to(dev) for x in (a, b, r))
    code = {"store": lib.GEMM_STORE, "residual": lib.GEMM_RESIDUAL, "swiglu": lib.GEMM_SWIGLU}[epi]
    outs = []
    for tile_n in (64, 256):
        tc = torch.empty((m, n), dtype=torch.float16, device=dev)
        lib.gemm(ta, tb, tc, m, n, k, code, r=tr if epi == "residual" else None, tile_n=tile_n)
        outs.append(tc)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


def test_gemm_residual_in_place_and_empty():
    dev = torch.device("cuda")
    a, b, r = _inputs(200, 256, 128, seed=9)
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    tc = torch.from_numpy(r).to(dev)
    lib.gemm(ta, tb, tc, 200, 256, 128, lib.GEMM_RESIDUAL, r=tc)   # C = A B^T + C
    torch.cuda.synchronize()
    _close16(tc.cpu().numpy(), ol.gemm(a, b, "residual", r), extra=1e-4)
    lib.gemm(ta, tb, tc, 0, 256, 128)  # m = 0: nothing to do


def test_gemm_argument_checks():
    dev = torch.device("cuda")
    x = torch.zeros(64, 64, dtype=torch.float16, device=dev)
    with pytest.raises(lib.TreeError) as e:
        lib.gemm(x, x, x, 64, 60, 64)
    assert e.value.code == lib.TREE_ERR_UNSUPPORTED
    with pytest.raises(lib.TreeError) as e:
        lib.gemm(x, x, x, 64, 64, 64, 7)
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    with pytest.raises(lib.TreeError) as e:
        lib.gemm(x, x, x, 64, 64, 64, lib.GEMM_RESIDUAL)
    assert e.value.code == lib.TREE_ERR_INVALID_ARG


@pytest.mark.parametrize("rows,cols", [(1000, 2048), (3, 8), (257, 4096), (64, 16384)])
def test_rmsnorm_matches_oracle(rows, cols):
    dev = torch.device("cuda")
    rng = np.random.default_rng(rows + cols)
    x = (rng.standard_normal((rows, cols)) * 3).astype(np.float16)
    w = rng.standard_normal(cols).astype(np.float16)
    tx, tw = torch.from_numpy(x).to(dev), torch.from_numpy(w).to(dev)
    ty = torch.empty_like(tx)
    lib.rmsnorm(tx, tw, ty, rows, cols, 1e-5)
    torch.cuda.synchronize()
    ref = ol.rmsnorm(x, w, 1e-5)
    # f32 statistics against float64: the normalised value may round to the other
    # f16 neighbour (one ulp of n), which the weight scales
    n_ulp = _ulp16(ol.f16(ref.astype(np.float64) / np.where(w == 0, 1, w).astype(np.float64)))
    g = ty.cpu().numpy().astype(np.float64)
    r = ref.astype(np.float64)
    assert (np.abs(g - r) <= _ulp16(r) + n_ulp * np.abs(w.astype(np.float64)) + 1e-7).all()
    lib.rmsnorm(tx, tw, tx, rows, cols, 1e-5)   # in place
    torch.cuda.synchronize()
    assert torch.equal(tx, ty)


# ---------------------------------------------------------------- the whole layer

LAYERS = {
    # workload: (hidden, ffn) around its attention shapes
    1: (256, 512),
    2: (2048, 8192),   # Llama-1B-shaped
}


def _ws_offsets(n_fwd, hidden, qd, ffn):
    up = lambda b: (b + 255) & ~255
    xn = 0
    q = xn + up(n_fwd * hidden * 2)
    o = q + up(n_fwd * qd * 2)
    h = o + up(n_fwd * qd * 2)
    g = h + up(n_fwd * hidden * 2)
    return dict(xn=xn, q=q, o=o, h=h, g=g, total=g + up(n_fwd * ffn * 2))


@pytest.mark.parametrize("wn", [1, 2])
def test_layer_matches_oracle(wn):
    import synth
    from oracle import plan as oplan
    dev = torch.device("cuda")
    w = synth.workload(wn)
    hidden, ffn = LAYERS[wn]
    plan = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd)
    i = plan.info
    n_fwd, n_res = i.n_tot - i.n_res, i.n_res
    wts, x, rk, rv = synth.draw_layer(n_fwd, n_res, hidden, w.hq, w.hkv, w.d, ffn, w.seed)
    td = {k: torch.from_numpy(v).to(dev) for k, v in wts.items()}
    lw = lib.layer_weights(hidden, w.hq, w.hkv, w.d, ffn, td)
    nbytes = lib.layer_workspace_bytes(plan, lw)
    qd, kvd = w.hq * w.d, w.hkv * w.d
    off = _ws_offsets(n_fwd, hidden, qd, ffn)
    assert nbytes == off["total"]
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    pdev = torch.empty(i.dev_bytes, dtype=torch.uint8, device=dev)
    plan.upload(pdev, i.dev_bytes)
    tab = torch.from_numpy(lib.rope_table(i.max_pos, w.d, w.theta)).to(dev)
    tx = torch.from_numpy(x).to(dev)
    kc = torch.zeros(i.n_tot, kvd, dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)
    kc[:n_res] = torch.from_numpy(rk).to(dev)
    vc[:n_res] = torch.from_numpy(rv).to(dev)
    y = torch.empty_like(tx)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    work = torch.zeros(2 * i.n_chunks, dtype=torch.int32, device=dev)
    lib.layer_fwd(plan, pdev, lw, tx, kc, vc, y, tab, i.max_pos, ws, nbytes, work=work, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    def buf(name, cols):
        return ws[off[name]: off[name] + n_fwd * cols * 2].view(torch.float16).view(n_fwd, cols).cpu().numpy()

    q_g, o_g, h_g, hn_g, g_g = buf("q", qd), buf("o", qd), buf("h", hidden), buf("xn", hidden), buf("g", ffn)
    k_g, v_g, y_g = kc.cpu().numpy(), vc.cpu().numpy(), y.cpu().numpy()
    # each step against the oracle applied to the library's own input of that step
    # (the normalised value may round to its other neighbour before the weight scales it)
    _close16(hn_g, ol.rmsnorm(h_g, wts["w_post"], 1e-5), extra=1e-7, ulps=2)
    _close16(g_g, ol.gemm(hn_g, wts["wgu"], "swiglu"), extra=1e-4)
    _close16(y_g, ol.gemm(g_g, wts["wd"], "residual", h_g), extra=1e-4)
    _close16(h_g, ol.gemm(o_g, wts["wo"], "residual", x), extra=1e-4)
    op, _ = oplan.plan_forest(w.forest, max_fwd=w.max_fwd)
    from oracle import attention as oatt
    o_ref = oatt.attend_paths(op, q_g.reshape(n_fwd, w.hq, w.d), k_g.reshape(-1, w.hkv, w.d),
                              v_g.reshape(-1, w.hkv, w.d)).reshape(n_fwd, qd)
    assert np.abs(o_g.astype(np.float64) - o_ref).max() <= 2e-3
    # the whole layer from its input: every f16 rounding of the chain may land on the
    # other neighbour; a flip of one ulp at one step moves y by about an ulp of that
    # step's values (the random weights keep rows at unit scale), so y stays within a
    # few ulps of its scale
    y_ref, q_ref, k_ref, v_ref, o16_ref, h_ref = ol.layer(op, x, rk, rv, wts, w.hq, w.hkv, w.d, w.theta)
    np.testing.assert_array_equal(k_g[:n_res], rk)
    assert np.abs(v_g[n_res:].astype(np.float64) - v_ref[n_res:].reshape(n_fwd, kvd).astype(np.float64)).max() <= 2 ** -9
    err = np.abs(y_g.astype(np.float64) - y_ref.astype(np.float64)).max()
    scale = np.abs(y_ref.astype(np.float64)).max()
    assert err <= 2e-2 * max(1.0, scale), (err, scale)


def _last_ws_offsets(n_fwd, n_slots, hidden, qd, ffn):
    up = lambda b: (b + 255) & ~255
    o = {}
    o["xn"] = 0
    o["q"] = o["xn"] + up(n_fwd * hidden * 2)
    o["o"] = o["q"] + up(n_fwd * qd * 2)
    o["xs"] = o["o"] + up(n_fwd * qd * 2)
    o["os"] = o["xs"] + up(n_slots * hidden * 2)
    o["hs"] = o["os"] + up(n_slots * qd * 2)
    o["hns"] = o["hs"] + up(n_slots * hidden * 2)
    o["gs"] = o["hns"] + up(n_slots * hidden * 2)
    o["ys"] = o["gs"] + up(n_slots * ffn * 2)
    o["fs"] = o["ys"] + up(n_slots * hidden * 2)
    o["total"] = o["fs"] + up(n_slots * hidden * 2)
    return o


@pytest.mark.parametrize("wn", [1, 2])
def test_last_layer_logits_and_readout(wn):
    """The final layer pruned to the readout rows, its letter logits, and the decision from them."""
    import synth
    from oracle import plan as oplan
    from oracle import readout as ordo
    dev = torch.device("cuda")
    w = synth.workload(wn)
    hidden, ffn = LAYERS[wn]
    stride = 8
    plan = lib.Plan.from_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
    i = plan.info
    n_fwd, n_res, S = i.n_tot - i.n_res, i.n_res, i.n_slots
    wts, x, rk, rv = synth.draw_layer(n_fwd, n_res, hidden, w.hq, w.hkv, w.d, ffn, w.seed)
    wf, wl = synth.draw_head(hidden, stride, w.seed)
    td = {k: torch.from_numpy(v).to(dev) for k, v in wts.items()}
    lw = lib.layer_weights(hidden, w.hq, w.hkv, w.d, ffn, td)
    nbytes = lib.last_layer_workspace_bytes(plan, lw)
    qd, kvd = w.hq * w.d, w.hkv * w.d
    off = _last_ws_offsets(n_fwd, S, hidden, qd, ffn)
    assert nbytes == off["total"]
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    pdev = torch.empty(i.dev_bytes, dtype=torch.uint8, device=dev)
    plan.upload(pdev, i.dev_bytes)
    tab = torch.from_numpy(lib.rope_table(i.max_pos, w.d, w.theta)).to(dev)
    tx = torch.from_numpy(x).to(dev)
    kc = torch.zeros(i.n_tot, kvd, dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)
    kc[:n_res] = torch.from_numpy(rk).to(dev)
    vc[:n_res] = torch.from_numpy(rv).to(dev)
    twf, twl = torch.from_numpy(wf).to(dev), torch.from_numpy(wl).to(dev)
    logits = torch.full((S, stride), float("nan"), device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.last_layer_fwd(plan, pdev, lw, tx, kc, vc, tab, i.max_pos, twf, twl, stride, logits, ws, nbytes, status=st)
    # the decision from the logits, on the device (the plan's question -> slot maps)
    p_cal = torch.empty((i.n_questions, stride), device=dev)
    choice = torch.empty(i.n_questions, dtype=torch.int32, device=dev)
    base = pdev.data_ptr()
    lib.readout_decide(logits, stride, base + i.off_r1, base + i.off_r2, torch.from_numpy(w.n_letters).to(dev),
                       torch.from_numpy(w.temperature).to(dev), i.n_questions, p_cal, None, choice, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lg = logits.cpu().numpy().astype(np.float64)

    op, qmap = oplan.plan_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
    # step: the letter logits from the library's own final-layer rows (one f16 rounding of the
    # normalised row, then an f32 dot product)
    ys = ws[off["ys"]: off["ys"] + S * hidden * 2].view(torch.float16).view(S, hidden).cpu().numpy()
    fs_ref = ol.rmsnorm(ys, wf, 1e-5).astype(np.float64)
    step_ref = fs_ref @ wl.astype(np.float64).T
    row_scale = np.abs(fs_ref) @ np.abs(wl.astype(np.float64)).T
    assert (np.abs(lg - step_ref) <= 2 * 2 ** -10 * row_scale + 1e-4).all()
    # end to end against the oracle's full final layer restricted to the readout rows
    ref = ol.last_layer(op, x, rk, rv, wts, w.hq, w.hkv, w.d, w.theta, wf, wl)
    err = np.abs(lg - ref).max()
    assert err <= 2e-2 * max(1.0, np.abs(ref).max()), err
    _check_decisions(lg, ref, qmap, w.n_letters, w.temperature, stride, p_cal.cpu().numpy(), choice.cpu().numpy())


def _check_decisions(lg, ref, qmap, n_letters, temperature, stride, p_cal, choice, min_checked=0.75):
    """Decisions of a decision forward.  (1) The readout of the library's own logits: the
    oracle's readout applied to them gives the device's p_cal within 1e-5 and its choices exactly
    (an f32 near-tie, top-two gap under 1e-6, may go either way).  (2) End to end: wherever the
    logit error of a question cannot swap the oracle's top two options, the choice is the
    oracle's.  With every logit of the question within eps of the oracle's, each softmax
    probability moves by at most a factor exp(+-2 eps), so the average p by at most
    (exp(2 eps) - 1) * p; a top-two gap above twice that keeps the argmax.  Most questions must
    be decided that way (a vacuous check fails)."""
    from oracle import readout as ordo
    own_pc, own_p, own_choice = ordo.decide(lg, qmap["r1"], qmap["r2"], n_letters, temperature, stride)
    assert np.abs(p_cal - own_pc).max() <= 1e-5
    ref_pc, ref_p, ref_choice = ordo.decide(ref, qmap["r1"], qmap["r2"], n_letters, temperature, stride)
    assert np.abs(p_cal - ref_pc).max() <= 5e-2
    checked = 0
    for qi in range(len(n_letters)):
        n = int(n_letters[qi])
        own = np.sort(own_p[qi][:n])
        if n < 2 or own[-1] - own[-2] > 1e-6:
            assert choice[qi] == own_choice[qi], qi
        rows = [int(qmap["r1"][qi]), int(qmap["r2"][qi])]
        eps = float(np.abs(lg[rows, :n] - ref[rows, :n]).max())
        srt = np.sort(ref_p[qi][:n])
        if n < 2 or srt[-1] - srt[-2] > 2 * (np.exp(2 * eps) - 1) * srt[-1]:
            assert choice[qi] == ref_choice[qi], qi
            checked += 1
    assert checked >= int(min_checked * len(n_letters)), (checked, len(n_letters))


def test_model_fwd_equals_layer_calls_and_oracle():
    """Three layers on the tiny tree: bit-identical to calling the layers one by one, and near the oracle."""
    import synth
    from oracle import plan as oplan
    dev = torch.device("cuda")
    w = synth.workload(1)
    hidden, ffn = LAYERS[1]
    stride, L = 8, 3
    plan = lib.Plan.from_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
    i = plan.info
    n_fwd, n_res, S = i.n_tot - i.n_res, i.n_res, i.n_slots
    qd, kvd = w.hq * w.d, w.hkv * w.d
    layers, tds, x = [], [], None
    for l in range(L):
        wts, x_l, _, _ = synth.draw_layer(n_fwd, n_res, hidden, w.hq, w.hkv, w.d, ffn, w.seed + 17 * l)
        x = x_l if x is None else x
        td = {k: torch.from_numpy(v).to(dev) for k, v in wts.items()}
        tds.append((wts, td))
        layers.append(lib.layer_weights(hidden, w.hq, w.hkv, w.d, ffn, td))
    wf, wl = synth.draw_head(hidden, stride, w.seed)
    twf, twl = torch.from_numpy(wf).to(dev), torch.from_numpy(wl).to(dev)
    pdev = torch.empty(i.dev_bytes, dtype=torch.uint8, device=dev)
    plan.upload(pdev, i.dev_bytes)
    tab = torch.from_numpy(lib.rope_table(i.max_pos, w.d, w.theta)).to(dev)
    tx = torch.from_numpy(x).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def caches():
        return ([torch.zeros(i.n_tot, kvd, dtype=torch.float16, device=dev) for _ in range(L)],
                [torch.zeros(i.n_tot, kvd, dtype=torch.float16, device=dev) for _ in range(L)])

    kc, vc = caches()
    nb = lib.model_workspace_bytes(plan, layers[0])
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    logits = torch.empty((S, stride), device=dev)
    lib.model_fwd(plan, pdev, layers, tx, kc, vc, tab, i.max_pos, twf, twl, stride, logits, ws, nb, status=st)
    # the same layers called one by one
    kc2, vc2 = caches()
    nl = lib.layer_workspace_bytes(plan, layers[0])
    ws2 = torch.empty(max(nl, lib.last_layer_workspace_bytes(plan, layers[0])), dtype=torch.uint8, device=dev)
    cur = tx
    for l in range(L - 1):
        nxt = torch.empty_like(tx)
        lib.layer_fwd(plan, pdev, layers[l], cur, kc2[l], vc2[l], nxt, tab, i.max_pos, ws2, ws2.numel(), status=st)
        cur = nxt
    logits2 = torch.empty((S, stride), device=dev)
    lib.last_layer_fwd(plan, pdev, layers[-1], cur, kc2[-1], vc2[-1], tab, i.max_pos, twf, twl, stride, logits2, ws2,
                       ws2.numel(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(logits, logits2)
    for l in range(L):
        assert torch.equal(kc[l], kc2[l]) and torch.equal(vc[l], vc2[l])
    # the oracle model: layer after layer in float64 with f16 storage
    op, _ = oplan.plan_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
    empty = np.zeros((0, kvd), np.float16)
    h = x
    for l in range(L - 1):
        h = ol.layer(op, h, empty, empty, tds[l][0], w.hq, w.hkv, w.d, w.theta)[0]
    ref = ol.last_layer(op, h, empty, empty, tds[-1][0], w.hq, w.hkv, w.d, w.theta, wf, wl)
    lgm = logits.cpu().numpy().astype(np.float64)
    err = np.abs(lgm - ref).max()
    # each layer contributes the single-layer bound
    assert err <= L * 2e-2 * max(1.0, np.abs(ref).max()), err
    # the decisions of the whole forward (readout on the device from the model's logits)
    _, qmap = oplan.plan_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
    p_cal = torch.empty((i.n_questions, stride), device=dev)
    choice = torch.empty(i.n_questions, dtype=torch.int32, device=dev)
    base = pdev.data_ptr()
    lib.readout_decide(logits, stride, base + i.off_r1, base + i.off_r2, torch.from_numpy(w.n_letters).to(dev),
                       torch.from_numpy(w.temperature).to(dev), i.n_questions, p_cal, None, choice, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check_decisions(lgm, ref, qmap, w.n_letters, w.temperature, stride, p_cal.cpu().numpy(), choice.cpu().numpy())


def test_long_session_slices_equal_model_fwd():
    """A long request run one layer per slice, with a short batch run between slices, gives the
    same logits bit for bit as the whole forward in one call; so does the short batch."""
    import synth
    dev = torch.device("cuda")
    hidden, ffn, stride, L = 256, 512, 8, 4

    def setup(wn, seed):
        w = synth.workload(wn)
        plan = lib.Plan.from_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2, max_fwd=w.max_fwd)
        i = plan.info
        n_fwd, n_res = i.n_tot - i.n_res, i.n_res
        kvd = w.hkv * w.d
        layers, keep = [], []
        x = None
        for l in range(L):
            wts, x_l, rk, rv = synth.draw_layer(n_fwd, n_res, hidden, w.hq, w.hkv, w.d, ffn, seed + 31 * l)
            x = x_l if x is None else x
            td = {k: torch.from_numpy(v).to(dev) for k, v in wts.items()}
            keep.append(td)
            layers.append(lib.layer_weights(hidden, w.hq, w.hkv, w.d, ffn, td))
        wf, wl = synth.draw_head(hidden, stride, seed)
        pdev = torch.empty(i.dev_bytes, dtype=torch.uint8, device=dev)
        plan.upload(pdev, i.dev_bytes)
        tab = torch.from_numpy(lib.rope_table(i.max_pos, w.d, w.theta)).to(dev)
        env = dict(w=w, plan=plan, i=i, layers=layers, keep=keep, x=torch.from_numpy(x).to(dev), pdev=pdev, tab=tab,
                   wf=torch.from_numpy(wf).to(dev), wl=torch.from_numpy(wl).to(dev), kvd=kvd, rk=rk, rv=rv)
        return env

    def buffers(env):
        i, kvd = env["i"], env["kvd"]
        kc = [torch.zeros(i.n_tot, kvd, dtype=torch.float16, device=dev) for _ in range(L)]
        vc = [torch.zeros(i.n_tot, kvd, dtype=torch.float16, device=dev) for _ in range(L)]
        for t in kc:
            t[:i.n_res] = torch.from_numpy(env["rk"]).to(dev)
        for t in vc:
            t[:i.n_res] = torch.from_numpy(env["rv"]).to(dev)
        nb = lib.model_workspace_bytes(env["plan"], env["layers"][0])
        return kc, vc, torch.empty(nb, dtype=torch.uint8, device=dev), nb, torch.empty((i.n_slots, stride), device=dev)

    def whole(env):
        kc, vc, ws, nb, lg = buffers(env)
        lib.model_fwd(env["plan"], env["pdev"], env["layers"], env["x"], kc, vc, env["tab"], env["i"].max_pos,
                      env["wf"], env["wl"], stride, lg, ws, nb)
        return lg

    long_env = setup(4, 400)    # the 32,768-token row in 4 chunks: the long lane
    short_env = setup(1, 100)   # the tiny tree: a short batch
    ref_long, ref_short = whole(long_env), whole(short_env)
    kc, vc, ws, nb, lg = buffers(long_env)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    sess = lib.Session(long_env["plan"], long_env["pdev"], long_env["layers"], long_env["x"], kc, vc, long_env["tab"],
                       long_env["i"].max_pos, long_env["wf"], long_env["wl"], stride, lg, ws, nb, status=st)
    slices, done, shorts = 0, False, []
    while not done:
        ran, done = sess.run(0.0)   # a zero slice: yield after every layer
        assert ran == 1
        slices += 1
        shorts.append(whole(short_env))   # a short batch takes the GPU between slices
    sess.close()
    torch.cuda.synchronize()
    assert slices == L and int(st.item()) == 0
    assert torch.equal(lg, ref_long)
    for s_ in shorts:
        assert torch.equal(s_, ref_short)
    # a long slice runs every layer at once
    kc, vc, ws, nb, lg2 = buffers(long_env)
    sess = lib.Session(long_env["plan"], long_env["pdev"], long_env["layers"], long_env["x"], kc, vc, long_env["tab"],
                       long_env["i"].max_pos, long_env["wf"], long_env["wl"], stride, lg2, ws, nb)
    assert sess.run(1e9) == (L, True)
    sess.close()
    assert torch.equal(lg2, ref_long)


@pytest.mark.parametrize("m", [300, 2048, 5000])
def test_gemm_qkv_split_equals_separate_gemms(m):
    """One GEMM over [Wq; Wk; Wv] writes the three outputs bit-identical to three GEMMs."""
    dev = torch.device("cuda")
    nq, nkv, k = 512, 128, 256
    a, b, _ = _inputs(m, nq + 2 * nkv, k, seed=m)
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    q = torch.empty((m, nq), dtype=torch.float16, device=dev)
    kk = torch.empty((m, nkv), dtype=torch.float16, device=dev)
    v = torch.empty((m, nkv), dtype=torch.float16, device=dev)
    lib.gemm_qkv(ta, tb, q, kk, v, m, nq, nkv, k)
    ref = [torch.empty((m, n), dtype=torch.float16, device=dev) for n in (nq, nkv, nkv)]
    lib.gemm(ta, tb[:nq].contiguous(), ref[0], m, nq, k)
    lib.gemm(ta, tb[nq:nq + nkv].contiguous(), ref[1], m, nkv, k)
    lib.gemm(ta, tb[nq + nkv:].contiguous(), ref[2], m, nkv, k)
    torch.cuda.synchronize()
    assert torch.equal(q, ref[0]) and torch.equal(kk, ref[1]) and torch.equal(v, ref[2])
    _close16(q.cpu().numpy(), ol.gemm(a, b[:nq]), extra=1e-4)
