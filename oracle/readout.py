"""Oracle letter readout: two option orders, average, temperature calibration.

Follows the basal-rs Architecture page, "02 / Basal protocol: Two option orders
and calibration".  Each question is asked twice, with its n options in the
original order and in reverse order.  Letter logits become probabilities per
order; the order-2 distribution is put back into the original option order and
the two are averaged; the average is calibrated with the question type's
temperature T:

    p     = (softmax(l_order1) + reverse(softmax(l_order2))) / 2
    p_cal = softmax(log(max(p, 1e-12)) / T)

Readings where the page is silent: "reverse" maps order-2 letter k to original
option n-1-k (the page's example lists the same options in reverse order);
the logarithm is natural; T > 0.  The chosen option is the argmax of p_cal,
lowest index on ties; since the clamp and log/T/softmax are monotone and the p
sum to 1, that is the argmax of p, which is the form used for the decision.
The page adds that T changes confidence, not the selected option.

Probabilities are computed in float64.  The decision itself is also taken in
float32 (``choice_f32``), the precision the kernel decides in, so that both
sides take an argmax in the same precision.

Test infrastructure only: see the package docstring.
"""
from __future__ import annotations

import numpy as np

CLAMP = 1e-12


def _softmax(x):
    x = x - x.max()
    e = np.exp(x)
    return e / e.sum()


def decide_one(l1, l2, T: float):
    """(p, p_cal) for one question from its order-1 and order-2 letter logits."""
    l1 = np.asarray(l1, np.float64)
    l2 = np.asarray(l2, np.float64)
    s1 = _softmax(l1)
    s2 = _softmax(l2)
    p = (s1 + s2[::-1]) / 2.0
    p_cal = _softmax(np.log(np.maximum(p, CLAMP)) / np.float64(T))
    return p, p_cal


def decide(logits, r1, r2, n_letters, temperature, stride=None):
    """Batch readout.  Returns p_cal [nq, stride] (zero past n), p [nq, stride], choice [nq]."""
    logits = np.asarray(logits)
    stride = logits.shape[1] if stride is None else stride
    nq = len(r1)
    p_cal = np.zeros((nq, stride), np.float64)
    p_avg = np.zeros((nq, stride), np.float64)
    choice = np.zeros(nq, np.int64)
    for q in range(nq):
        n = int(n_letters[q])
        p, pc = decide_one(logits[r1[q], :n], logits[r2[q], :n], float(temperature[q]))
        p_avg[q, :n] = p
        p_cal[q, :n] = pc
        choice[q] = int(np.argmax(p))
    return p_cal, p_avg, choice


def choice_f32(logits, r1, r2, n_letters):
    """The decision taken in float32 arithmetic (argmax of the f32 average)."""
    logits = np.asarray(logits, np.float32)
    out = np.zeros(len(r1), np.int64)
    for q in range(len(r1)):
        n = int(n_letters[q])
        a = logits[r1[q], :n].astype(np.float32)
        b = logits[r2[q], :n].astype(np.float32)
        ea = np.exp(a - a.max())
        eb = np.exp(b - b.max())
        s1 = ea / ea.sum(dtype=np.float32)
        s2 = eb / eb.sum(dtype=np.float32)
        p = (s1 + s2[::-1]) * np.float32(0.5)
        out[q] = int(np.argmax(p))
    return out
