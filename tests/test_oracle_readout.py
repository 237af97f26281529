"""Pins for the oracle's two-order readout and calibration (CPU only).

The formulas are those of the basal-rs Architecture page, "02 / Basal protocol:
Two option orders and calibration"; the worked example's printed values sit in
tests/golden/worked_example.json.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from oracle import readout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


@pytest.fixture(scope="module")
def ex():
    with open(GOLDEN) as f:
        return json.load(f)


def test_worked_example_per_order(ex):
    # each order's softmax, rounded as printed
    s1 = sp_softmax(np.array(ex["order1_logits"], np.float64))
    s2 = sp_softmax(np.array(ex["order2_logits"], np.float64))
    assert np.allclose(np.round(s1, 2), ex["order1_probs_printed"])
    assert np.allclose(np.round(s2, 2), ex["order2_probs_printed"])


def test_worked_example_average_and_calibration(ex):
    p, p_cal = readout.decide_one(ex["order1_logits"], ex["order2_logits"], ex["temperature"])
    assert np.allclose(np.round(p, 2), ex["average_printed"]), p
    assert np.allclose(np.round(p_cal, 2), ex["calibrated_printed"]), p_cal
    # "Returns" is chosen
    logits = np.array([ex["order1_logits"], ex["order2_logits"]], np.float32)
    _, _, ch = readout.decide(logits, [0], [1], [3], [1.0])
    assert ch[0] == 0


def test_worked_example_needs_the_reversal(ex):
    # without putting order 2 back into the original order the printed average is not reached
    s1 = sp_softmax(np.array(ex["order1_logits"]))
    s2 = sp_softmax(np.array(ex["order2_logits"]))
    wrong = (s1 + s2) / 2
    assert not np.allclose(np.round(wrong, 2), ex["average_printed"])


def _random_q(rng, n):
    return rng.normal(0, 3, n), rng.normal(0, 3, n)


def test_matches_library_softmax_composition():
    rng = np.random.default_rng(0)
    for _ in range(200):
        n = int(rng.integers(1, 40))
        l1, l2 = _random_q(rng, n)
        T = float(rng.choice([0.5, 0.7, 1.0, 1.3, 2.0]))
        p, pc = readout.decide_one(l1, l2, T)
        ref_p = (sp_softmax(l1) + sp_softmax(l2)[::-1]) / 2
        ref_pc = sp_softmax(np.log(np.maximum(ref_p, 1e-12)) / T)
        np.testing.assert_allclose(p, ref_p, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(pc, ref_pc, rtol=1e-12, atol=1e-15)


def test_t1_is_identity():
    rng = np.random.default_rng(1)
    for _ in range(100):
        n = int(rng.integers(2, 12))
        l1, l2 = _random_q(rng, n)
        p, pc = readout.decide_one(l1, l2, 1.0)
        np.testing.assert_allclose(pc, p, rtol=1e-12, atol=1e-15)


def test_temperature_keeps_the_choice_and_moves_confidence():
    rng = np.random.default_rng(2)
    for _ in range(200):
        n = int(rng.integers(2, 12))
        l1, l2 = _random_q(rng, n)
        p, _ = readout.decide_one(l1, l2, 1.0)
        top = int(np.argmax(p))
        for T in (0.5, 0.7, 1.3, 2.0):
            _, pc = readout.decide_one(l1, l2, T)
            assert int(np.argmax(pc)) == top
            if p[top] < 1 - 1e-9:
                if T < 1:
                    assert pc[top] > p[top]      # sharpens
                else:
                    assert pc[top] < p[top]      # flattens


def test_symmetric_orders_reduce_to_one_softmax():
    rng = np.random.default_rng(3)
    for _ in range(50):
        l1 = rng.normal(0, 2, int(rng.integers(2, 10)))
        p, _ = readout.decide_one(l1, l1[::-1], 1.0)
        np.testing.assert_allclose(p, sp_softmax(l1), rtol=1e-13)


def test_single_letter_and_clamp():
    p, pc = readout.decide_one([5.0], [-3.0], 0.7)
    assert p[0] == 1.0 and pc[0] == 1.0
    # a probability far below 1e-12 is clamped before the log
    p, pc = readout.decide_one([0.0, -200.0], [-200.0, 0.0], 0.5)
    assert p[1] < 1e-80
    expect = sp_softmax(np.log([p[0], 1e-12]) / 0.5)
    np.testing.assert_allclose(pc, expect, rtol=1e-12)


def test_batch_layout_and_padding():
    rng = np.random.default_rng(4)
    logits = rng.normal(0, 2, (8, 6)).astype(np.float32)
    p_cal, p_avg, ch = readout.decide(logits, [0, 2, 4], [1, 3, 5], [3, 6, 1], [1.0, 0.7, 1.3])
    assert p_cal.shape == (3, 6)
    assert np.all(p_cal[0, 3:] == 0) and np.all(p_cal[2, 1:] == 0)
    np.testing.assert_allclose(p_cal.sum(axis=1), 1.0, rtol=1e-12)
    _, pc1 = readout.decide_one(logits[2, :6], logits[3, :6], 0.7)
    np.testing.assert_allclose(p_cal[1], pc1)
    assert np.array_equal(readout.choice_f32(logits, [0, 2, 4], [1, 3, 5], [3, 6, 1]), ch)
