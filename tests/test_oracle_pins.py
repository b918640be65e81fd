"""Pins for the CPU oracle: Philox known answers, the pages' worked examples and
brute-force / library checks of the sampling transforms.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --- Philox4x32-10 -----------------------------------------------------------

def _kat_rows():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            w = [int(x, 16) for x in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


@pytest.mark.parametrize("ctr,key,expect", _kat_rows())
def test_philox_known_answers(ctr, key, expect):
    assert list(oracle.philox4x32_10(ctr, key)) == expect


def test_uniform_construction_is_open_closed_unit_interval():
    # U = ((x >> 8) + 1) * 2^-24: smallest 2^-24, largest exactly 1, 2^24 equal steps.
    assert oracle.uniform_from_word(0) == 2.0 ** -24
    assert oracle.uniform_from_word(0xFFFFFFFF) == 1.0
    assert oracle.uniform_from_word(0x000000FF) == 2.0 ** -24
    assert oracle.uniform_from_word(0x00000100) == 2.0 * 2.0 ** -24


def test_uniform_keying_and_moments():
    # distinct (batch, node, word) give distinct draws; mean/variance of U(0,1]
    us = np.array([oracle.uniform(1234, 5, b, n, w) for b in range(40) for n in range(25)
                   for w in (0, 1)])
    assert len(np.unique(us)) == len(us)
    assert abs(us.mean() - 0.5) < 4 * math.sqrt(1 / 12 / len(us))
    assert abs(us.var() - 1 / 12) < 0.01
    # the key (seed) and the offset both change the stream
    assert oracle.uniform(1, 0, 0, 0, 0) != oracle.uniform(2, 0, 0, 0, 0)
    assert oracle.uniform(1, 0, 0, 0, 0) != oracle.uniform(1, 1, 0, 0, 0)
    assert oracle.uniform(1, 0, 0, 0, 0) != oracle.uniform(1, 1 << 32, 0, 0, 0)


# --- worked examples printed on the pages --------------------------------------

def _example(name):
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        return json.load(f)[name]


@pytest.mark.parametrize("name", ["tutorial_section_2_4", "eagle3_section_6"])
def test_worked_examples(name):
    ex = _example(name)
    p = np.log(np.array(ex["p_rows"], dtype=np.float64)).astype(np.float32)
    q = np.log(np.array(ex["q_rows"], dtype=np.float64)).astype(np.float32)
    N, V = p.shape
    parents = np.array([ex["parent_idx"]], dtype=np.int32)
    tokens = np.array([ex["draft_tokens"]], dtype=np.int32)
    ua = np.full((1, N), 0.5)
    for node, spec in ex["u_accept"].items():
        ua[0, int(node)] = spec["value"]
    uf = np.full((1, N), 0.5)
    depth = N - 1
    out = oracle.verify_tree(p[None], q[None], tokens, parents, depth, 1.0, 0, 1.0, seed=0,
                             u_accept=ua, u_final=uf)
    exp = ex["expect"]
    assert out["accept_len"][0] == exp["accept_len"]
    n_tok = exp["accept_len"] + 1
    assert list(out["tokens"][0, :n_tok]) == exp["tokens"]
    assert all(t == -1 for t in out["tokens"][0, n_tok:])
    assert list(out["path"][0, :n_tok]) == exp["path"]
    for node, a in exp["alpha"].items():
        # fp32-rounded ln(prob) logits carry ~1e-7 relative error into the ratio
        assert out["alpha"][0, int(node)] == pytest.approx(a, rel=1e-6, abs=1e-7)
    # the page's printed values themselves
    pv = ex["page_values"]
    for pd, qd, node in zip(pv["p_draft_token"], pv["q_draft_token"], range(1, N)):
        assert out["alpha"][0, node] == pytest.approx(min(1.0, pd / qd), rel=1e-6)
    if "alpha_node2" in pv:
        assert out["alpha"][0, 2] == pytest.approx(pv["alpha_node2"], rel=1e-6)
        assert pv["r_node2"] > pv["alpha_node2"]
    if "alpha_rounded" in pv:
        assert np.round(out["alpha"][0, 1:N], 2).tolist() == pv["alpha_rounded"]
    # untested nodes carry NaN
    tested = {int(k) for k in exp["alpha"]}
    for n in range(1, N):
        if n not in tested:
            assert math.isnan(out["alpha"][0, n])


# --- sampling transforms ---------------------------------------------------------

def _brute_force_filter(z, T, top_k, top_p):
    """Kept set by exhaustive search: top-k = the k largest (ties to lower index);
    top-p = the smallest subset of the top-k set with normalised mass >= top_p,
    which must consist of its largest members (ties to lower index)."""
    V = len(z)
    key = sorted(range(V), key=lambda i: (-z[i], i))
    K = top_k if 0 < top_k < V else V
    topk = key[:K]
    w = {i: math.exp((z[i] - max(z)) / T) for i in topk}
    s_k = sum(w.values())
    if top_p >= 1.0:
        return set(topk)
    for size in range(1, K + 1):
        best = None
        for sub in itertools.combinations(topk, size):
            mass = sum(w[i] for i in sub) / s_k
            if mass >= top_p:
                best = sub
                break
        if best is not None:
            # among subsets of this size, the one kept is the rank-order prefix
            prefix = topk[:size]
            assert sum(w[i] for i in prefix) / s_k >= top_p
            return set(prefix)
    return set(topk)


@pytest.mark.parametrize("seed", range(12))
def test_filter_matches_brute_force_on_small_rows(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(3, 9))
    # coarse values force ties
    z = (rng.integers(-4, 5, size=V) * 0.5).astype(np.float32)
    T = float(np.float32(rng.choice([0.3, 0.7, 1.0, 2.5])))
    top_k = int(rng.choice([0, 1, 2, 3, V - 1, V, V + 3]))
    top_p = float(np.float32(rng.choice([1.0, 0.95, 0.9, 0.5, 0.2])))
    probs, info = oracle.filter_row(z, T, top_k, top_p)
    kept = _brute_force_filter(z.astype(np.float64).tolist(), T, top_k, top_p)
    if info.near:
        pytest.skip("top-p decision within 1e-6 of its threshold")
    assert set(np.nonzero(probs)[0].tolist()) <= kept
    assert info.kept == len(kept)
    assert probs.sum() == pytest.approx(1.0, abs=1e-12)
    # kept probabilities are the renormalised softmax weights
    zs = z.astype(np.float64)
    w = np.exp((zs - zs.max()) / T)
    ref = np.zeros(V)
    idx = sorted(kept)
    ref[idx] = w[idx] / w[idx].sum()
    np.testing.assert_allclose(probs, ref, rtol=1e-12, atol=1e-15)
    # the cut is the last kept token in rank order
    order = sorted(range(V), key=lambda i: (-zs[i], i))
    assert info.cut_idx == order[len(kept) - 1]


def test_filter_without_truncation_is_softmax():
    rng = np.random.default_rng(3)
    for T in (0.25, 0.7, 1.0, 3.0):
        z = rng.normal(0, 3, size=1000).astype(np.float32)
        probs, info = oracle.filter_row(z, T, 0, 1.0)
        np.testing.assert_allclose(probs, softmax(z.astype(np.float64) / T), rtol=1e-12)
        assert info.kept == 1000
        assert info.argmax == int(np.argmax(z))


def test_greedy_and_top1_filters_are_one_hot_at_lowest_index_max():
    z = np.array([1.0, 3.0, -2.0, 3.0, 0.5], dtype=np.float32)
    for T, k in ((0.0, 0), (1.0, 1), (0.4, 1)):
        probs, info = oracle.filter_row(z, T, k, 1.0)
        assert info.argmax == 1
        np.testing.assert_array_equal(probs, np.eye(5)[1])


def test_top_p_is_rank_prefix_with_index_ties():
    # four tied maxima: top-p 0.5 of an exactly uniform top set keeps exactly half,
    # the lower indices first
    z = np.array([0.0, 2.0, 2.0, -1.0, 2.0, 2.0], dtype=np.float32)
    probs, info = oracle.filter_row(z, 1.0, 4, 0.5)
    np.testing.assert_allclose(probs, [0, 0.5, 0.5, 0, 0, 0], atol=1e-15)
    assert info.cut_idx == 2
    assert info.near  # cumulative mass hits 0.5 exactly


def test_bf16_rows_use_exact_widening():
    vals = np.array([1.0, -0.5, 2.5, 2.5, -3.0], dtype=np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    p32, i32 = oracle.filter_row(vals, 0.8, 0, 0.9)
    p16, i16 = oracle.filter_row(bits, 0.8, 0, 0.9)
    np.testing.assert_array_equal(p32, p16)
    assert i32.cut_idx == i16.cut_idx


def test_negative_zero_ties_with_positive_zero():
    z = np.array([-0.0, 0.0, -1.0], dtype=np.float32)
    probs, info = oracle.filter_row(z, 1.0, 1, 1.0)
    assert info.argmax == 0 and probs[0] == 1.0


@pytest.mark.parametrize("row,bad", [
    ([0.0, float("nan"), 1.0], True),
    ([0.0, float("inf"), 1.0], True),
    ([float("-inf")] * 3, True),
    ([float("-inf"), 0.0, float("-inf")], False),
])
def test_non_finite_rows(row, bad):
    _, info = oracle.filter_row(np.array(row, dtype=np.float32), 1.0, 0, 0.9)
    assert info.status == (1 if bad else 0)
    if not bad:
        assert info.argmax == 1 and info.kept == 1
