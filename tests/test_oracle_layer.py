"""Oracle layer pieces pinned to closed forms and to library routines on special cases."""
import numpy as np

from oracle import layer as ol


def test_rmsnorm_closed_forms():
    # [3, 4]: mean square 12.5, so n = [3, 4] / sqrt(12.5 + eps)
    x = np.array([[3.0, 4.0]], np.float16)
    w = np.array([1.0, 2.0], np.float16)
    y = ol.rmsnorm(x, w, 0.0)
    n = np.array([3.0, 4.0]) / np.sqrt(12.5)
    assert y.dtype == np.float16
    np.testing.assert_array_equal(y[0], (n.astype(np.float16).astype(np.float64) * [1.0, 2.0]).astype(np.float16))
    # a constant row normalises to its sign; eps shrinks it by sqrt(c^2 / (c^2 + eps))
    x = np.full((2, 8), [[-0.5], [2.0]], np.float16)
    w = np.ones(8, np.float16)
    np.testing.assert_array_equal(ol.rmsnorm(x, w, 0.0), np.sign(x.astype(np.float64)).astype(np.float16))
    y = ol.rmsnorm(x[1:], w, 1.0).astype(np.float64)
    np.testing.assert_allclose(y, 2.0 / np.sqrt(4.0 + 1.0), rtol=2 ** -10)
    # scale invariance (eps = 0): rmsnorm(a x) = rmsnorm(x) for a power of two
    x = np.random.default_rng(0).standard_normal((4, 64)).astype(np.float16)
    w = np.random.default_rng(1).standard_normal(64).astype(np.float16)
    np.testing.assert_array_equal(ol.rmsnorm(x, w, 0.0), ol.rmsnorm((x.astype(np.float64) * 4).astype(np.float16), w, 0.0))


def test_gemm_against_integer_matmul():
    # small integers: every product and sum is exact in f64 and the result exact in f16
    rng = np.random.default_rng(2)
    a = rng.integers(-4, 5, (37, 24)).astype(np.float16)
    b = rng.integers(-4, 5, (19, 24)).astype(np.float16)
    exact = a.astype(np.int64) @ b.astype(np.int64).T
    np.testing.assert_array_equal(ol.gemm(a, b).astype(np.int64), exact)
    r = rng.integers(-8, 9, (37, 19)).astype(np.float16)
    np.testing.assert_array_equal(ol.gemm(a, b, "residual", r).astype(np.int64), exact + r.astype(np.int64))


def test_swiglu_closed_forms():
    assert ol.silu(0.0) == 0.0
    np.testing.assert_allclose(ol.silu(40.0), 40.0, rtol=1e-15)
    x = np.linspace(-6, 6, 13)
    np.testing.assert_allclose(ol.silu(-x), ol.silu(x) - x, atol=1e-14)   # silu(-x) = silu(x) - x
    np.testing.assert_allclose(ol.silu(x), x * 0.5 * (1 + np.tanh(x / 2)), atol=1e-14)
    # swiglu with the up half equal to ones is silu of the gate
    rng = np.random.default_rng(3)
    a = rng.integers(-3, 4, (5, 16)).astype(np.float16)
    g = rng.integers(-2, 3, (4, 16)).astype(np.float16)
    u_one = np.zeros((4, 16), np.float16)
    u_one[:, 0] = 1
    a1 = a.copy()
    a1[:, 0] = 1
    got = ol.gemm(a1, np.concatenate([g, u_one]), "swiglu")
    np.testing.assert_array_equal(got, ol.silu(a1.astype(np.float64) @ g.astype(np.float64).T).astype(np.float16))


def test_letter_logits_special_case():
    # rows of +-1 normalise to +-1 (eps 0) times the final weight; logits are then a plain matmul
    from types import SimpleNamespace
    rng = np.random.default_rng(4)
    y = np.where(rng.random((6, 16)) < 0.5, -1.0, 1.0).astype(np.float16)
    wf = rng.integers(-2, 3, 16).astype(np.float16)
    wl = rng.integers(-3, 4, (8, 16)).astype(np.float16)
    plan = SimpleNamespace(slot_tok=np.array([7, 3, 5]), n_res=2)
    got = ol.letter_logits(plan, y, wf, wl, eps=0.0)
    rows = y[[5, 1, 3]].astype(np.int64) * wf.astype(np.int64)
    np.testing.assert_array_equal(got, rows @ wl.astype(np.int64).T)


def _chain_layer_inputs(n: int, hidden: int, hq: int, hkv: int, d: int, ffn: int):
    import synth
    from oracle import plan as oplan
    forest = synth.Forest(np.array([-1], np.int32), np.array([n], np.int32), np.zeros(1, np.uint64),
                          np.zeros(1, np.uint8))
    plan, _ = oplan.plan_forest(forest)
    w, x, rk, rv = synth.draw_layer(n, 0, hidden, hq, hkv, d, ffn, seed=11)
    return plan, w, x, rk, rv


def test_layer_residual_adds_pass_their_input_through_zero_projections():
    # wo = 0: the attention block's residual add returns the layer input; wd = 0: the MLP's residual
    # add returns the attention block's output h (which differs from the input when wo != 0)
    hidden, hq, hkv, d, ffn = 32, 4, 2, 16, 48
    plan, w, x, rk, rv = _chain_layer_inputs(20, hidden, hq, hkv, d, ffn)
    _, _, _, _, _, h = ol.layer(plan, x, rk, rv, dict(w, wo=np.zeros_like(w["wo"])), hq, hkv, d, 500000.0)
    np.testing.assert_array_equal(h, x)
    y, _, _, _, _, h = ol.layer(plan, x, rk, rv, dict(w, wd=np.zeros_like(w["wd"])), hq, hkv, d, 500000.0)
    assert not np.array_equal(h, x)
    np.testing.assert_array_equal(y, h)


def test_layer_with_zero_queries_averages_the_values():
    # wq = 0: every score is 0, so on a chain token i's attention output is the plain mean of the
    # value rows 0..i of its kv head (the values are the normalised input times wv, rounded to f16)
    hidden, hq, hkv, d, ffn = 32, 4, 2, 16, 48
    n = 24
    plan, w, x, rk, rv = _chain_layer_inputs(n, hidden, hq, hkv, d, ffn)
    w = dict(w, wq=np.zeros_like(w["wq"]))
    _, q, _, v, o16, _ = ol.layer(plan, x, rk, rv, w, hq, hkv, d, 500000.0)
    assert not np.any(q)
    xn = ol.rmsnorm(x, w["w_in"], 1e-5).astype(np.float64)
    vv = (xn @ w["wv"].astype(np.float64).T).astype(np.float16).astype(np.float64).reshape(n, hkv, d)
    np.testing.assert_array_equal(v.astype(np.float64), vv)
    mean = np.cumsum(vv, axis=0) / np.arange(1, n + 1)[:, None, None]
    want = np.repeat(mean, hq // hkv, axis=1).reshape(n, hq * d)   # q head h reads kv head h // 2
    np.testing.assert_allclose(o16.astype(np.float64), want, rtol=2 ** -10, atol=2 ** -24)
