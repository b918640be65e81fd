"""Pins of the per-request oracle: a batch with every tree under the same parameters is
the batched oracle itself (the per-tree Philox keying by batch index), a greedy tree
is the target's argmax chain, and invalid values are reported per tree."""
import numpy as np

import oracle
from speculative_decoding_tree_spec_gb300 import workloads as wl


def _inputs(B=6, N=12, V=48, seed=3):
    w = wl.WORKLOADS["tree60_b64_v128256"].with_(B=B, N=N, V=V, depth=4, dtype="f32")
    inp = wl.build_inputs(w, seed=seed)
    return w, wl.host_logits(inp["p"]), wl.host_logits(inp["q"]), inp


def test_uniform_parameters_equal_the_batched_oracle():
    w, p, q, inp = _inputs()
    B = w.B
    ref = oracle.verify_tree(p, q, inp["tokens"], inp["parents"], inp["max_depth"], 0.8, 10, 0.9,
                             seed=11)
    per = oracle.verify_tree_per_request(p, q, inp["tokens"], inp["parents"], inp["max_depth"],
                                         [0.8] * B, [10] * B, [0.9] * B, seed=11)
    for b in range(B):
        for k in ("accept_len", "tokens", "path", "alpha", "status"):
            np.testing.assert_array_equal(per[b][k][0], ref[k][b], err_msg=f"{k} tree {b}")


def test_greedy_tree_is_the_argmax_chain():
    w, p, q, inp = _inputs(seed=5)
    B = w.B
    T = [0.0 if b % 2 == 0 else 1.0 for b in range(B)]
    per = oracle.verify_tree_per_request(p, q, inp["tokens"], inp["parents"], inp["max_depth"],
                                         T, [0] * B, [1.0] * B, seed=2)
    for b in range(0, B, 2):
        node, n = 0, 0
        par, tok = inp["parents"][b], inp["tokens"][b]
        while True:
            am = int(np.argmax(p[b, node]))
            kids = [c for c in range(len(par)) if par[c] == node and tok[c] == am]
            if not kids:
                assert per[b]["tokens"][0][n] == am
                break
            node = kids[0]
            n += 1
        assert per[b]["accept_len"][0] == n


def test_invalid_parameters_are_per_tree():
    w, p, q, inp = _inputs()
    T = [0.7, -1.0, float("nan"), 0.7, float("inf"), 0.7]
    k = [0, 0, 0, -3, 0, 0]
    pp = [1.0, 1.0, 1.0, 1.0, 1.0, 0.0]
    per = oracle.verify_tree_per_request(p, q, inp["tokens"], inp["parents"], inp["max_depth"],
                                         T, k, pp, seed=1)
    assert per[0] is not None
    assert all(per[b] is None for b in range(1, 6))
