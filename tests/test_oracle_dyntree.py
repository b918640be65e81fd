"""Pins of the EAGLE-2 dynamic-tree oracle (EAGLE / EAGLE-2 paper translation, sections
2.3.1-2.3.2; LLM speculative decoding: EAGLE, section 4.2.1) against facts the pages
and the mathematics fix: a hand-worked instance, exact dyadic values, the rounding
bound of a product, brute-force selection over all subsets, the tie rule, the
connectedness the pages promise, breadth-first order and the ancestor mask as a
transitive closure."""
import itertools
import json
import pathlib

import numpy as np
import pytest

from oracle import dyntree
from speculative_decoding_tree_spec_gb300.workloads import make_draft_candidates

GOLDEN = pathlib.Path(__file__).parent / "golden" / "eagle2_rerank_small.json"


def _golden():
    return json.loads(GOLDEN.read_text())


def test_golden_values_and_draft():
    g = _golden()
    val, dep = dyntree.values_and_depths(np.array(g["cand_parent"]), np.array(g["cand_prob"], np.float32))
    assert val.tolist() == g["values"]
    assert dep.tolist() == g["depths"]
    out = dyntree.build_tree(g["cand_parent"], g["cand_token"], np.array(g["cand_prob"], np.float32),
                             g["root_token"], g["m"])
    for k, v in g["expected"].items():
        assert np.asarray(out[k]).tolist() == v, k


def test_golden_expand():
    g = _golden()
    val, _ = dyntree.values_and_depths(np.array(g["cand_parent"]), np.array(g["cand_prob"], np.float32))
    e = g["expand"]
    got = dyntree.expand_topk(val[e["layer_begin"]:e["layer_end"]], e["k"])
    assert [e["layer_begin"] + i for i in got] == e["expected"]


def test_dyadic_values_exact():
    # a chain of confidences 1/2 has value 2^-depth exactly
    n = 20
    par = np.array([-1] + list(range(n - 1)))
    val, dep = dyntree.values_and_depths(par, np.full(n, 0.5, np.float32))
    assert dep.tolist() == list(range(1, n + 1))
    assert val.tolist() == [2.0 ** -(i + 1) for i in range(n)]


def test_value_within_rounding_bound_of_exact_product():
    d = make_draft_candidates(1, layers=6, seed=3)
    val, dep = dyntree.values_and_depths(d.parent[0], d.prob[0])
    for i in range(len(val)):
        exact, x = 1.0, i
        while x >= 0:
            exact *= float(d.prob[0, x])
            x = int(d.parent[0, x])
        bound = dep[i] * 2.0 ** -24 * exact * 1.0001
        assert abs(float(val[i]) - exact) <= bound, i


def test_child_value_never_exceeds_parent():
    d = make_draft_candidates(2, seed=4)
    for b in range(2):
        val, _ = dyntree.values_and_depths(d.parent[b], d.prob[b])
        for i, p in enumerate(d.parent[b]):
            if p >= 0:
                assert val[i] <= val[p]


def _beats(val, dep, i, j):
    """The selection order of the pages: larger value, then shallower, then lower number."""
    return (val[i], -dep[i], -i) > (val[j], -dep[j], -j)


def _random_small(rng, n, levels=0):
    par = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], dtype=np.int32)
    prob = rng.random(n).astype(np.float32)
    if levels:
        prob = (np.floor(prob * levels) / levels).astype(np.float32)
    return par, prob


@pytest.mark.parametrize("levels", [0, 4])
def test_selection_matches_brute_force(levels):
    rng = np.random.default_rng(11 + levels)
    for _ in range(60):
        n = int(rng.integers(1, 9))
        m = int(rng.integers(1, n + 1))
        par, prob = _random_small(rng, n, levels)
        val, dep = dyntree.values_and_depths(par, prob)
        out = dyntree.build_tree(par, np.arange(n), prob, -1, m)
        chosen = set(int(s) for s in out["src"][1:])
        # every m-subset: the chosen one has the largest value sum
        best = max(sum(float(val[i]) for i in s) for s in itertools.combinations(range(n), m))
        assert sum(float(val[i]) for i in chosen) == best
        # and it is exactly the candidates beaten by fewer than m others
        pairwise = {i for i in range(n) if sum(_beats(val, dep, j, i) for j in range(n)) < m}
        assert chosen == pairwise
        # connected: the parent of a kept candidate is kept (or is the root)
        for c in chosen:
            assert par[c] < 0 or int(par[c]) in chosen


def test_tie_prefers_shallower_then_lower_number():
    # candidates 1 (depth 1) and 2 (depth 2) tie at 1/4; the shallower one is kept
    out = dyntree.build_tree([-1, -1, 0], [5, 6, 7], np.array([0.5, 0.25, 0.5], np.float32), 0, 2)
    assert out["src"].tolist() == [-1, 0, 1]
    # equal value and depth: the lower number
    out = dyntree.build_tree([-1, -1, -1], [5, 6, 7], np.array([0.25, 0.5, 0.25], np.float32), 0, 2)
    assert out["src"].tolist() == [-1, 0, 1]
    assert out["tokens"].tolist() == [0, 5, 6]


def test_flatten_breadth_first_and_mask_closure():
    d = make_draft_candidates(3, seed=5, levels=8)
    for b in range(3):
        m = 59
        out = dyntree.build_tree(d.parent[b], d.token[b], d.prob[b], d.root[b], m)
        src, par, pos = out["src"], out["parent_idx"], out["position_ids"]
        _, dep = dyntree.values_and_depths(d.parent[b], d.prob[b])
        keys = [(int(dep[s]), int(s)) for s in src[1:]]
        assert keys == sorted(keys)
        assert par[0] == -1 and pos[0] == 0 and out["tokens"][0] == d.root[b]
        for j in range(1, m + 1):
            assert 0 <= par[j] < j
            assert out["tokens"][j] == d.token[b, src[j]]
            assert pos[j] == pos[par[j]] + 1
            cp = int(d.parent[b, src[j]])
            assert (par[j] == 0) if cp < 0 else (src[par[j]] == cp)
        # ancestor-or-self mask = reflexive transitive closure of the parent relation
        M = m + 1
        A = np.zeros((M, M), dtype=np.int64)
        for j in range(1, M):
            A[j, par[j]] = 1
        R = np.eye(M, dtype=np.int64)
        step = np.eye(M, dtype=np.int64) + A
        for _ in range(int(pos.max()) + 1):
            R = np.minimum(R @ step, 1)
        assert np.array_equal(out["mask"], R.astype(np.uint8))


def test_expand_topk_brute_force():
    rng = np.random.default_rng(12)
    for _ in range(50):
        n = int(rng.integers(1, 30))
        vals = (np.floor(rng.random(n) * 6) / 6).astype(np.float32)
        k = int(rng.integers(1, n + 3))
        got = dyntree.expand_topk(vals, k)
        assert len(got) == min(k, n)
        for r, i in enumerate(got):
            ahead = [j for j in range(n) if (vals[j], -j) > (vals[i], -i)]
            assert len(ahead) == r


def test_flatten_is_breadth_first_on_any_numbering():
    """Candidate numbers need not grow with depth (a list may interleave layers): the
    flattened order is by depth first, then number."""
    rng = np.random.default_rng(21)
    for _ in range(40):
        n = int(rng.integers(2, 12))
        par, prob = _random_small(rng, n)
        m = int(rng.integers(1, n + 1))
        out = dyntree.build_tree(par, np.arange(n), prob, -1, m)
        _, dep = dyntree.values_and_depths(par, prob)
        keys = [(int(dep[s]), int(s)) for s in out["src"][1:]]
        assert keys == sorted(keys)
        assert out["position_ids"][1:].tolist() == [k[0] for k in keys]
