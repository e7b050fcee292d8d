"""Pins for the LM-head statistics oracle (CPU only).

* Closed form: identity hidden states give logits = weight^T exactly.
* The logits against an explicit triple loop, and the statistics against
  scipy.special.logsumexp (log S + m / T = logsumexp(l / T)), a first-occurrence argmax loop and
  direct indexing for the gathers.
* Temperature: the argmax does not depend on T; S tends to V as T grows; T = 1 and T = 0.5 differ.
* Ties: equal maxima give the lowest index.
"""
import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import lmhead as OL


def _loop_logits(h, w):
    M, H = h.shape
    V = w.shape[0]
    out = np.zeros((M, V))
    for m in range(M):
        for v in range(V):
            acc = 0.0
            for k in range(H):
                acc += float(h[m, k]) * float(w[v, k])
            out[m, v] = acc
    return out


def test_identity_hidden_gives_the_weight():
    rng = np.random.default_rng(0)
    H, V = 6, 11
    w = rng.standard_normal((V, H))
    assert np.array_equal(OL.logits(np.eye(H), w), w.T)


@pytest.mark.parametrize("T", [1.0, 0.5, 2.0])
def test_statistics_against_loops_and_scipy(T):
    rng = np.random.default_rng(1)
    M, H, V = 5, 7, 13
    h = rng.standard_normal((M, H))
    w = rng.standard_normal((V, H))
    lg = _loop_logits(h, w)
    assert np.allclose(OL.logits(h, w), lg, atol=1e-12)
    gi = rng.integers(-1, V, size=(M, 4))
    st = OL.lm_head_stats(h, w, T, gi)
    for m in range(M):
        best = 0
        for v in range(1, V):
            if lg[m, v] > lg[m, best]:
                best = v
        assert st["argmax"][m] == best
        assert st["max"][m] == pytest.approx(lg[m].max(), abs=1e-12)
        assert np.log(st["sumexp"][m]) + st["max"][m] / T == pytest.approx(
            logsumexp(lg[m] / T), abs=1e-12)
        for g in range(4):
            if gi[m, g] < 0:
                assert np.isnan(st["gather"][m, g])
            else:
                assert st["gather"][m, g] == pytest.approx(lg[m, gi[m, g]], abs=1e-12)


def test_temperature_behaviour():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((4, 50))
    a = OL.row_stats(lg, 1.0)
    b = OL.row_stats(lg, 0.5)
    c = OL.row_stats(lg, 1e6)
    assert np.array_equal(a["argmax"], b["argmax"])
    assert not np.allclose(a["sumexp"], b["sumexp"])
    assert np.allclose(c["sumexp"], 50, rtol=1e-5)


def test_ties_take_the_lowest_index():
    lg = np.array([[0.0, 3.0, 1.0, 3.0], [5.0, 5.0, 5.0, 5.0]])
    st = OL.row_stats(lg, 1.0)
    assert list(st["argmax"]) == [1, 0]
    assert list(st["top_gap"]) == [0.0, 0.0]
