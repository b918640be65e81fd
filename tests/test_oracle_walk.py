"""Pins for the oracle's tree walk against what the pages and the mathematics fix:
the greedy argmax chain, categorical sampling at N=1, the chain acceptance rate
sum_x min(p, q), exact distribution preservation (averaged over drafts drawn
from q), and a chi-squared test of the emitted tokens.  CPU only."""
import itertools
import math

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import oracle
from speculative_decoding_tree_spec_gb300 import workloads as wl


def _greedy_chain(p, tokens, parents):
    """The target's greedy continuation along the tree: at node u emit argmax p_u;
    continue into the first child whose draft token equals it."""
    N = len(parents)
    u, acc, path = 0, [], [0]
    while True:
        t = int(np.argmax(p[u]))
        nxt = [c for c in range(1, N) if parents[c] == u and tokens[c] == t]
        if not nxt:
            return acc + [t], path
        acc.append(t)
        path.append(nxt[0])
        u = nxt[0]


@pytest.mark.parametrize("seed", range(6))
def test_greedy_output_is_target_argmax_chain(seed):
    rng = np.random.default_rng(seed)
    B, N, V, D = 16, 12, 6, 4
    parents = np.stack([wl.random_tree(N, D, 3, rng) for _ in range(B)])
    p = rng.integers(-3, 4, size=(B, N, V)).astype(np.float32)  # many argmax ties
    q = rng.normal(size=(B, N, V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
    # bias drafts toward the target argmax so that long acceptances occur
    for b in range(B):
        for c in range(1, N):
            if rng.random() < 0.6:
                tokens[b, c] = int(np.argmax(p[b, parents[b, c]]))
    out = oracle.verify_tree(p, q, tokens, parents, D, 0.0, 0, 1.0, seed=seed)
    for b in range(B):
        toks, path = _greedy_chain(p[b], tokens[b], parents[b])
        n = len(toks)
        assert out["accept_len"][b] == n - 1
        assert out["tokens"][b, :n].tolist() == toks
        assert out["path"][b, :n].tolist() == path
        assert (out["tokens"][b, n:] == -1).all()


@pytest.mark.parametrize("seed", range(4))
def test_top1_sampling_equals_greedy(seed):
    rng = np.random.default_rng(100 + seed)
    B, N, V, D = 32, 9, 7, 3
    parents = np.stack([wl.random_tree(N, D, 3, rng) for _ in range(B)])
    p = rng.normal(0, 2, size=(B, N, V)).astype(np.float32)
    q = rng.normal(0, 2, size=(B, N, V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for b in range(B):
        for c in range(1, N):
            if rng.random() < 0.5:
                tokens[b, c] = int(np.argmax(p[b, parents[b, c]]))
    g = oracle.verify_tree(p, q, tokens, parents, D, 0.0, 0, 1.0, seed=seed)
    for T in (0.5, 1.0):
        s = oracle.verify_tree(p, q, tokens, parents, D, T, 1, 1.0, seed=seed)
        np.testing.assert_array_equal(s["accept_len"], g["accept_len"])
        np.testing.assert_array_equal(s["tokens"], g["tokens"])
        np.testing.assert_array_equal(s["path"], g["path"])


def test_root_only_tree_is_categorical_inverse_cdf():
    rng = np.random.default_rng(7)
    B, V, T = 400, 50, 0.9
    p = rng.normal(0, 2, size=(B, 1, V)).astype(np.float32)
    out = oracle.verify_tree(p, p, np.zeros((B, 1), np.int32), np.full((B, 1), -1, np.int32), 0,
                             T, 0, 1.0, seed=99, offset=3)
    for b in range(B):
        probs = softmax(p[b, 0].astype(np.float64) / T)
        r = oracle.uniform(99, 3, b, 0, 1)
        expect = int(np.searchsorted(np.cumsum(probs), r * probs.sum(), side="left"))
        if out["near"][b]:
            continue
        assert out["tokens"][b, 0] == expect
        assert out["accept_len"][b] == 0 and out["path"][b, 0] == 0


def test_chain_acceptance_rate_is_sum_of_min_p_q():
    """Chain drafts (branching 1) are the standard algorithm: at every position the
    acceptance probability is sum_x min(p(x), q(x)) when x ~ q."""
    rng = np.random.default_rng(11)
    gamma, V, B, T = 3, 32, 20000, 1.0
    p = rng.normal(0, 3, size=(gamma + 1, V)).astype(np.float32)
    q = (p + rng.normal(0, 1, size=p.shape)).astype(np.float32)
    parents = np.tile(wl.chain_tree(gamma + 1), (B, 1))
    P = softmax(p.astype(np.float64) / T, axis=-1)
    Q = softmax(q.astype(np.float64) / T, axis=-1)
    tokens = np.zeros((B, gamma + 1), np.int32)
    for i in range(gamma):
        tokens[:, i + 1] = rng.choice(V, size=B, p=Q[i])
    out = oracle.verify_tree(p, q, tokens, parents, gamma, T, 0, 1.0, seed=5,
                             batch_broadcast=True)
    acc = out["accept_len"]
    for i in range(gamma):
        reached = (acc >= i).sum()
        accepted = (acc >= i + 1).sum()
        beta = np.minimum(P[i], Q[i]).sum()
        sd = math.sqrt(beta * (1 - beta) / reached)
        assert abs(accepted / reached - beta) < 4 * sd, (i, accepted / reached, beta)


def _first_token_law(p, q, parents, T, top_k, top_p, V):
    """Exact law of the first emitted token, averaged over sibling drafts drawn
    i.i.d. from the filtered draft row at the root.  For each draft combination
    the walk is run with every root child forced to reject (u = 1); the alphas it
    reports along that path and its final distribution give the branch
    probabilities by the law of total probability."""
    Q, _ = oracle.filter_row(q[0], T, top_k, top_p)
    kids = [c for c in range(1, len(parents)) if parents[c] == 0]
    support = np.nonzero(Q)[0]
    law = np.zeros(V)
    combos = list(itertools.product(support, repeat=len(kids)))
    B = len(combos)
    tokens = np.zeros((B, len(parents)), np.int32)
    for bi, combo in enumerate(combos):
        for c, x in zip(kids, combo):
            tokens[bi, c] = x
    ua = np.ones((B, len(parents)))
    out = oracle.verify_tree(p, q, tokens, np.tile(parents, (B, 1)), 8, T, top_k, top_p,
                             seed=1, u_accept=ua, want_final_dist=True, batch_broadcast=True)
    for bi, combo in enumerate(combos):
        weight = np.prod([Q[x] for x in combo])
        stay = 1.0
        for c, x in zip(kids, combo):
            a = out["alpha"][bi, c]
            law[x] += weight * stay * a
            stay *= (1 - a)
            if a == 1.0:
                break
        else:
            law += weight * stay * out["final_dist"][bi]
    return law


@pytest.mark.parametrize("case", range(8))
def test_exact_distribution_preservation_at_root(case):
    rng = np.random.default_rng(1000 + case)
    V = int(rng.integers(3, 6))
    k_root = int(rng.integers(1, 4))
    parents = np.array([-1] + [0] * k_root + [1], dtype=np.int32)
    N = len(parents)
    T = float(np.float32(rng.choice([0.6, 1.0, 1.7])))
    top_k = int(rng.choice([0, V - 1]))
    top_p = float(np.float32(rng.choice([1.0, 0.9])))
    p = rng.normal(0, 1.5, size=(N, V)).astype(np.float32)
    q = (p + rng.normal(0, 1.2, size=(N, V))).astype(np.float32)
    law = _first_token_law(p, q, parents, T, top_k, top_p, V)
    P, _ = oracle.filter_row(p[0], T, top_k, top_p)
    np.testing.assert_allclose(law, P, atol=1e-12)


def test_chi_squared_first_and_second_tokens():
    """Philox-driven walks: the first token follows filt(p_root); after the walk
    accepts the root's child c, the next token follows filt(p_c)."""
    rng = np.random.default_rng(21)
    V, T, top_k, top_p = 6, 1.0, 0, 1.0
    parents = np.array([-1, 0, 0, 1, 1, 2], dtype=np.int32)   # root -> {1,2}; 1 -> {3,4}; 2 -> {5}
    N = len(parents)
    p = rng.normal(0, 1.2, size=(N, V)).astype(np.float32)
    q = (p + rng.normal(0, 1.0, size=(N, V))).astype(np.float32)
    B = 200000
    Qs = [oracle.filter_row(q[u], T, top_k, top_p)[0] for u in range(N)]
    tokens = np.zeros((B, N), np.int32)
    for c in range(1, N):
        tokens[:, c] = rng.choice(V, size=B, p=Qs[parents[c]])
    out = oracle.verify_tree(p, q, tokens, np.tile(parents, (B, 1)), 3, T, top_k, top_p,
                             seed=77, batch_broadcast=True, nthreads=4)
    P0 = oracle.filter_row(p[0], T, top_k, top_p)[0]
    first = out["tokens"][:, 0]
    obs = np.bincount(first, minlength=V)
    assert stats.chisquare(obs, P0 * B).pvalue > 1e-3
    for c in (1, 2):
        sel = out["path"][:, 1] == c
        second = out["tokens"][sel, 1]
        Pc = oracle.filter_row(p[c], T, top_k, top_p)[0]
        obs = np.bincount(second, minlength=V)
        assert stats.chisquare(obs, Pc * sel.sum()).pvalue > 1e-3


@pytest.mark.parametrize("bad", ["root", "order", "token", "depth"])
def test_invalid_trees_are_reported(bad):
    V, N, D = 5, 4, 3
    parents = np.array([[-1, 0, 1, 2]], np.int32)
    tokens = np.array([[0, 1, 2, 3]], np.int32)
    if bad == "root":
        parents[0, 0] = 0
    elif bad == "order":
        parents[0, 2] = 3
    elif bad == "token":
        tokens[0, 3] = V
    elif bad == "depth":
        D = 2
    p = np.zeros((1, N, V), np.float32)
    out = oracle.verify_tree(p, p, tokens, parents, D, 1.0, 0, 1.0, seed=0)
    assert out["status"][0] == 2
    assert out["accept_len"][0] == -1
    assert (out["tokens"][0] == -1).all() and (out["path"][0] == -1).all()


def test_non_finite_row_on_the_walk_is_reported():
    V, N = 4, 3
    parents = np.array([[-1, 0, 1]], np.int32)
    tokens = np.array([[0, 2, 1]], np.int32)
    p = np.zeros((1, N, V), np.float32)
    q = np.zeros((1, N, V), np.float32)
    q[0, 0, 1] = np.nan
    out = oracle.verify_tree(p, q, tokens, parents, 2, 1.0, 0, 1.0, seed=0)
    assert out["status"][0] == 1 and out["accept_len"][0] == -1
    # greedy never reads q
    out = oracle.verify_tree(p, q, tokens, parents, 2, 0.0, 0, 1.0, seed=0)
    assert out["status"][0] == 0


def test_near_bits_name_the_decision_at_its_boundary():
    """The near flag says which decision sat within 1e-6 of its threshold: an accept
    test with r equal to alpha, a final draw with r on a CDF step, a top-p cut whose
    cumulative mass lands on top_p."""
    V, T = 4, 1.0
    # root with one child; p uniform, q concentrated so alpha of token 0 is 1/4 / 1/2
    p = np.zeros((1, 2, V), np.float32)
    q = np.zeros((1, 2, V), np.float32)
    q[0, 0] = np.log(np.array([2.0, 1.0, 0.5, 0.5], np.float32))
    tok = np.array([[0, 0]], np.int32)
    par = np.array([[-1, 0]], np.int32)
    Q = np.array([2.0, 1.0, 0.5, 0.5]) / 4.0
    alpha = 0.25 / Q[0]
    ua = np.array([[0.0, alpha]], np.float64)
    uf = np.full((1, 2), 0.37, np.float64)
    out = oracle.verify_tree(p, q, tok, par, 1, T, 0, 1.0, seed=1, u_accept=ua, u_final=uf)
    assert oracle.near_reasons(out["near"][0]) == ["accept"]
    # rejected (r above alpha), then the draw from norm(max(0, p - q)) lands on a step
    resid = np.maximum(0.0, 0.25 - Q)
    cdf = np.cumsum(resid) / resid.sum()
    ua = np.array([[0.0, 0.9]], np.float64)
    uf = np.array([[cdf[2], 0.0]], np.float64)
    out = oracle.verify_tree(p, q, tok, par, 1, T, 0, 1.0, seed=1, u_accept=ua, u_final=uf)
    assert oracle.near_reasons(out["near"][0]) == ["draw"]
    assert out["tokens"][0, 0] == 2
    # a leaf root whose top-p threshold equals a cumulative mass: p-row cut only
    p1 = np.log(np.array([[[4.0, 2.0, 1.0, 1.0]]], np.float32))
    out = oracle.verify_tree(p1, p1, np.zeros((1, 1), np.int32), np.full((1, 1), -1, np.int32),
                             0, T, 0, 0.75, seed=1, u_final=np.array([[0.3]]))
    assert oracle.near_reasons(out["near"][0]) == ["p_cut"]
    # a node with children whose q row has that cut too: both cut bits
    out = oracle.verify_tree(np.concatenate([p1, p1], 1), np.concatenate([p1, p1], 1),
                             tok, par, 1, T, 0, 0.75, seed=1, u_accept=np.array([[0.0, 0.5]]),
                             u_final=np.full((1, 2), 0.3))
    assert {"p_cut", "q_cut"} <= set(oracle.near_reasons(out["near"][0]))
