"""spec_tree_expand_topk and spec_tree_build against the oracle of the EAGLE-2 dynamic
tree on the same candidate lists: bit-exact on every output (values are fp32 products
taken root-first on both sides, so every comparison and tie is decided identically)."""
import numpy as np
import pytest
import torch

from oracle import dyntree
from speculative_decoding_tree_spec_gb300 import binding
from speculative_decoding_tree_spec_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _dev(d):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    return t(d.parent), t(d.token), t(d.prob), t(d.root)


def _check_build(d, m):
    par, tok, prob, root = _dev(d)
    out = binding.tree_build(par, tok, prob, root, m)
    torch.cuda.synchronize()
    B = d.parent.shape[0]
    assert out["status"].cpu().tolist() == [0] * B
    for b in range(B):
        ref = dyntree.build_tree(d.parent[b], d.token[b], d.prob[b], int(d.root[b]), m)
        for k in ("tokens", "parent_idx", "position_ids", "src", "mask"):
            got = out[k][b].cpu().numpy()
            assert np.array_equal(got, ref[k]), (b, k)
    return out


@pytest.mark.parametrize("levels", [0, 8], ids=["continuous", "tied"])
@pytest.mark.parametrize("B,m", [(16, 59), (3, 509), (5, 1)])
def test_build_matches_oracle(B, m, levels):
    d = wl.make_draft_candidates(B, seed=100 + m + levels, levels=levels)
    _check_build(d, m)


def test_build_keeps_all_candidates():
    d = wl.make_draft_candidates(4, layers=3, expand_k=2, children=4, seed=7)
    _check_build(d, d.parent.shape[1])


def test_build_single_candidate():
    d = wl.DraftCandidates(np.array([[-1]], np.int32), np.array([[42]], np.int32),
                           np.array([[0.3]], np.float32), np.array([9], np.int32))
    out = _check_build(d, 1)
    assert out["tokens"][0].tolist() == [9, 42]


def _random_forest(B, n, seed, levels=0):
    rng = np.random.default_rng(seed)
    par = np.empty((B, n), np.int32)
    for b in range(B):
        par[b] = [-1] + [int(rng.integers(-1, i)) for i in range(1, n)]
    prob = rng.random((B, n)).astype(np.float32)
    if levels:
        prob = (np.floor(prob * levels) / levels).astype(np.float32)
    tok = rng.integers(0, 1 << 20, size=(B, n)).astype(np.int32)
    root = rng.integers(0, 1 << 20, size=B).astype(np.int32)
    return wl.DraftCandidates(par, tok, prob, root)


@pytest.mark.parametrize("n,m", [(4096, 4095), (4096, 60), (777, 300), (777, 700), (2000, 1024),
                                 (2000, 1025), (300, 300)])
def test_build_max_sizes(n, m):
    _check_build(_random_forest(2, n, seed=n + m, levels=16), m)


def test_build_flags_malformed_trees():
    d = _random_forest(6, 40, seed=9)
    d.parent[1, 5] = 5                      # parent not before its child
    d.prob[2, 7] = np.float32("nan")
    d.prob[3, 0] = np.float32(1.5)
    d.parent[4] = [-1] + list(range(39))    # a chain of depth 40: fine
    chain = wl.DraftCandidates(np.array([[-1] + list(range(69))], np.int32),
                               np.zeros((1, 70), np.int32), np.full((1, 70), 0.9, np.float32),
                               np.zeros(1, np.int32))
    par, tok, prob, root = _dev(d)
    m = 12
    out = binding.tree_build(par, tok, prob, root, m)
    st = out["status"].cpu().tolist()
    assert st == [0, 2, 2, 2, 0, 0]
    for b in (1, 2, 3):
        for k in ("tokens", "parent_idx", "position_ids", "src"):
            assert out[k][b].cpu().tolist() == [-1] * (m + 1)
        assert int(out["mask"][b].sum()) == 0
    for b in (0, 4, 5):
        ref = dyntree.build_tree(d.parent[b], d.token[b], d.prob[b], int(d.root[b]), m)
        for k in ("tokens", "parent_idx", "position_ids", "src", "mask"):
            assert np.array_equal(out[k][b].cpu().numpy(), ref[k]), (b, k)
    # a chain deeper than 64 candidates is rejected
    par, tok, prob, root = _dev(chain)
    assert binding.tree_build(par, tok, prob, root, 5)["status"].cpu().tolist() == [2]


@pytest.mark.parametrize("levels", [0, 8], ids=["continuous", "tied"])
def test_expand_matches_oracle(levels):
    B, layers, ek, ch = 8, 6, 10, 10
    d = wl.make_draft_candidates(B, layers=layers, expand_k=ek, children=ch, seed=31, levels=levels)
    par, _, prob, _ = _dev(d)
    bounds = [(0, ch)] + [(ch + i * ek * ch, ch + (i + 1) * ek * ch) for i in range(layers - 1)]
    for lo, hi in bounds:
        for k in (1, ek, hi - lo + 3):
            got = binding.tree_expand_topk(par, prob, lo, hi, k).cpu().numpy()
            for b in range(B):
                val, _ = dyntree.values_and_depths(d.parent[b], d.prob[b])
                ref = [lo + i for i in dyntree.expand_topk(val[lo:hi], k)]
                ref += [-1] * (k - len(ref))
                assert got[b].tolist() == ref, (lo, hi, k, b)


def test_expand_empty_range():
    d = wl.make_draft_candidates(2, seed=3)
    par, _, prob, _ = _dev(d)
    assert binding.tree_expand_topk(par, prob, 5, 5, 3).cpu().tolist() == [[-1] * 3] * 2


def test_built_draft_feeds_verify():
    """The flattened draft is a valid spec_verify_tree input: greedy verify of a target
    whose argmax follows one root-to-leaf path of the draft accepts that whole path."""
    d = wl.make_draft_candidates(4, seed=17)
    par, tok, prob, root = _dev(d)
    m = 59
    out = binding.tree_build(par, tok, prob, root, m)
    N, V = m + 1, 128256
    toks = out["tokens"]
    parent = out["parent_idx"]
    logits = torch.zeros((4, N, V), dtype=torch.float32, device=DEV)
    pidx = parent.cpu().numpy()
    t = toks.cpu().numpy()
    want = []
    for b in range(4):
        # the seeded draft has no two siblings with one token, so the walk is unique
        for u in range(N):
            kids = [int(t[b, c]) for c in range(1, N) if pidx[b, c] == u]
            assert len(kids) == len(set(kids))
        leaf = N - 1                        # the last position is a deepest node
        chain = [leaf]
        while pidx[b, chain[-1]] > 0:
            chain.append(int(pidx[b, chain[-1]]))
        chain = chain[::-1]
        want.append(len(chain))
        node = 0
        for c in chain:
            logits[b, node, int(t[b, c])] = 10.0 + b
            node = c
        logits[b, node, 0] = 10.0           # bonus token after the leaf
    res = binding.verify_tree(logits, None, toks.contiguous(), parent.contiguous(),
                              int(out["position_ids"].max()), 0.0)
    torch.cuda.synchronize()
    assert res["status"].cpu().tolist() == [0] * 4
    got = res["accept_len"].cpu().tolist()
    assert got == want


@pytest.mark.parametrize("levels", [0, 16], ids=["continuous", "tied"])
def test_expand_long_ranges(levels):
    """Ranges past one, two and four members per thread, and past the counting limit."""
    d = _random_forest(3, 4096, seed=77 + levels, levels=levels)
    par, _, prob, _ = _dev(d)
    vals = [dyntree.values_and_depths(d.parent[b], d.prob[b])[0] for b in range(3)]
    for lo, hi in [(0, 256), (100, 400), (1000, 1600), (2000, 3024), (3000, 4096), (0, 4096)]:
        for k in (7, 300):
            got = binding.tree_expand_topk(par, prob, lo, hi, k).cpu().numpy()
            for b in range(3):
                ref = [lo + i for i in dyntree.expand_topk(vals[b][lo:hi], k)]
                ref += [-1] * (k - len(ref))
                assert got[b].tolist() == ref, (lo, hi, k, b)
