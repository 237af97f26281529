"""Pins for the oracle's rotary embedding with tree positions (CPU only)."""
import numpy as np

import synth
from oracle import plan as oplan
from oracle import rope


def test_position_zero_is_identity():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 64)).astype(np.float16)
    y = rope.rope_f16(x, np.zeros(5, np.int64), 500000.0)
    assert np.array_equal(x, y)


def test_two_dims_is_a_plane_rotation():
    # d = 2: one pair, frequency theta^0 = 1, angle = pos
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 1, 2))
    pos = np.arange(7) * 3
    y = rope.rotate(x, pos, 10000.0)
    for t in range(7):
        c, s = np.cos(pos[t]), np.sin(pos[t])
        R = np.array([[c, -s], [s, c]])
        np.testing.assert_allclose(y[t, 0], R @ x[t, 0], rtol=1e-14, atol=1e-14)


def test_matches_complex_multiplication():
    # pair (i, i + d/2) as the complex number x_i + 1j x_{i+d/2}, times exp(1j a_i)
    rng = np.random.default_rng(2)
    d, theta = 128, 500000.0
    x = rng.standard_normal((9, 2, d))
    pos = rng.integers(0, 32768, 9)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    freq = theta ** (-np.arange(0, d, 2) / d)
    w = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    ref = np.concatenate([w.real, w.imag], axis=-1)
    np.testing.assert_allclose(rope.rotate(x, pos, theta), ref, rtol=1e-11, atol=1e-11)


def test_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(3)
    d = 64
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    ref = None
    for m in (5, 100, 3000, 20000):
        n = m - 4
        s = float(np.sum(rope.rotate(q, [m], 500000.0) * rope.rotate(k, [n], 500000.0)))
        ref = s if ref is None else ref
        assert abs(s - ref) < 1e-9


def test_positions_are_depth_in_own_prompt():
    w = synth.workload(2)
    p, _ = oplan.plan_forest(w.forest)
    # packed: template 0..127, row 0: document 128..639, question 640..687, leaves 688..727, 728..767
    assert p.pos[0] == 0 and p.pos[127] == 127
    assert p.pos[128] == 128 and p.pos[639] == 639
    assert p.pos[640] == 640 and p.pos[687] == 687
    assert p.pos[688] == 688 and p.pos[727] == 727
    # the second option leaf restarts at the same position as its sibling
    assert p.pos[728] == 688 and p.pos[767] == 727
    # the second question of the row starts right after the document
    assert p.pos[768] == 640
    # row 1 starts again after the template
    assert p.pos[128 + 1024] == 128


def test_resident_rows_untouched_forward_rows_rotated():
    w = synth.workload(2)
    p, _ = oplan.plan_forest(w.forest)
    rng = np.random.default_rng(4)
    q = rng.standard_normal((p.n_fwd, 2, 8)).astype(np.float16)
    k = rng.standard_normal((p.n_tot, 1, 8)).astype(np.float16)
    qr, kr = rope.apply_plan(p, q, k, 500000.0)
    assert np.array_equal(kr[: p.n_res], k[: p.n_res])
    np.testing.assert_array_equal(kr[p.n_res:], rope.rope_f16(k[p.n_res:], p.pos[p.n_res:], 500000.0))
    np.testing.assert_array_equal(qr, rope.rope_f16(q, p.pos[p.n_res:], 500000.0))
