"""Pins of the draft top-k oracle: brute force over small rows (every token's rank by
counting), forced ties to the lower index, the confidences summing to one over the
whole vocabulary (k = V), the closed form of a two-level row, and non-finite rows."""
import math

import numpy as np

from oracle.draft import draft_topk


def test_rank_by_counting_and_ties():
    rng = np.random.default_rng(1)
    for _ in range(40):
        V = int(rng.integers(2, 40))
        row = (rng.integers(-4, 5, size=V) * 0.5).astype(np.float32)  # many ties
        k = int(rng.integers(1, V + 1))
        tok, _, st = draft_topk(row[None], k, 1.0)
        assert st[0] == 0
        for r, t in enumerate(tok[0]):
            above = sum(1 for j in range(V) if (row[j] > row[t]) or (row[j] == row[t] and j < t))
            assert above == r


def test_full_row_confidences_sum_to_one():
    rng = np.random.default_rng(2)
    row = (rng.standard_normal(64) * 3).astype(np.float32)
    for T in (0.3, 1.0, 2.5):
        _, p, _ = draft_topk(row[None], 64, T)
        assert abs(p.sum() - 1.0) < 1e-12
        assert (np.diff(p[0]) <= 0).all()   # listed by rank: non-increasing


def test_closed_form_two_levels():
    # a row with one logit at a and V - 1 at b: p(top) = 1 / (1 + (V - 1) e^{(b - a)/T})
    V, a, b, T = 100, 2.0, -1.0, 0.8
    row = np.full(V, b, dtype=np.float32)
    row[37] = a
    tok, p, _ = draft_topk(row[None], 3, T)
    assert tok[0].tolist() == [37, 0, 1]
    top = 1.0 / (1.0 + (V - 1) * math.exp((b - a) / T))
    assert abs(p[0, 0] - top) < 1e-15
    assert abs(p[0, 1] - (1 - top) / (V - 1)) < 1e-15


def test_bf16_bits_and_nonfinite_rows():
    x = np.array([1.0, 3.0, -2.0, 3.0], dtype=np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    tok, _, _ = draft_topk(bits[None], 2, 1.0)
    assert tok[0].tolist() == [1, 3]
    bad = np.array([[0.0, np.nan, 1.0], [np.inf, 0.0, 0.0], [-np.inf] * 3], dtype=np.float32)
    tok, p, st = draft_topk(bad, 2, 1.0)
    assert st.tolist() == [1, 1, 1]
    assert (tok == -1).all() and (p == 0).all()
