"""spec_verify_tree_noalloc (the verify call that uses the library's own static
scratch instead of a caller workspace) against spec_verify_tree on the same inputs.

The GPU tests make two calls in a row of the no-allocation entry point, with
different inputs and random offsets, and compare each with the workspace entry
point: accepted lengths, tokens, paths and statuses exactly, acceptance
probabilities within the parity tolerance of the logit dtype.  The file name sorts
last so that the first call on the device may come after every other test."""
import os

import numpy as np
import pytest
import torch

import __graft_entry__
from parity_helpers import ALPHA_RTOL
from speculative_decoding_tree_spec_gb300 import binding
from speculative_decoding_tree_spec_gb300 import workloads as wl

DEV = "cuda:0"
BASE = wl.WORKLOADS["tree60_b64_v128256"].with_(B=16, V=20000)
CASES = {
    "sampling-topp-bf16": BASE,
    "greedy-bf16": BASE.with_(temperature=0.0, top_p=1.0),
    "topk-f32": wl.WORKLOADS["tree26_b256_v152064"].with_(B=12, V=9001, dtype="f32"),
    "visited-only-bf16": BASE.with_(extra={"flags": binding.SPEC_FLAG_VISITED_ONLY}),
}


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(binding.LIB_PATH):
        __graft_entry__.build()
    return binding.lib()


def _inputs(w, seed):
    inp = wl.build_inputs(w, seed=seed, device=torch.device(DEV))
    inp["tokens_d"] = torch.as_tensor(inp["tokens"], device=DEV)
    inp["parents_d"] = torch.as_tensor(inp["parents"], device=DEV)
    return inp


def _outputs(B, N, W):
    return {
        "accept_len": torch.full((B,), -7, dtype=torch.int32, device=DEV),
        "tokens": torch.full((B, W), -7, dtype=torch.int32, device=DEV),
        "path": torch.full((B, W), -7, dtype=torch.int32, device=DEV),
        "status": torch.full((B,), -7, dtype=torch.int32, device=DEV),
        "alpha": torch.full((B, N), -7.0, dtype=torch.float32, device=DEV),
    }


def _noalloc(w, inp, seed, offset, out, counters=None):
    binding.verify_tree_noalloc(inp["p"], inp["q"], inp["tokens_d"], inp["parents_d"],
                                inp["max_depth"], w.temperature, w.top_k, w.top_p,
                                seed=seed, offset=offset, flags=w.extra.get("flags", 0),
                                out=out, counters=counters)


def _with_workspace(w, inp, seed, offset):
    return binding.verify_tree(inp["p"], inp["q"], inp["tokens_d"], inp["parents_d"],
                               inp["max_depth"], w.temperature, w.top_k, w.top_p,
                               seed=seed, offset=offset, flags=w.extra.get("flags", 0),
                               want_counters=True)


def _same(w, a, b, tag):
    for k in ("accept_len", "tokens", "path", "status"):
        np.testing.assert_array_equal(a[k].cpu().numpy(), b[k].cpu().numpy(),
                                      err_msg=f"{tag}: {k}")
    ga = a["alpha"].cpu().numpy().astype(np.float64)
    gb = b["alpha"].cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(np.isnan(ga), np.isnan(gb), err_msg=f"{tag}: alpha NaN")
    m = ~np.isnan(gb)
    np.testing.assert_allclose(ga[m], gb[m], rtol=ALPHA_RTOL[w.dtype], atol=0,
                               err_msg=f"{tag}: alpha")


@pytest.mark.gpu
@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_workspace_entry_point_twice_in_a_row(L, case):
    w = CASES[case]
    runs = [(_inputs(w, seed=101), 5, 0), (_inputs(w, seed=202), 5, 1)]
    outs = []
    counters = []
    for inp, seed, offset in runs:
        out = _outputs(w.B, w.N, inp["max_depth"] + 1)
        cnt = torch.zeros(8, dtype=torch.int64, device=DEV)
        _noalloc(w, inp, seed, offset, out, cnt)
        outs.append(out)
        counters.append(cnt)
    torch.cuda.synchronize()
    for i, (inp, seed, offset) in enumerate(runs):
        ref = _with_workspace(w, inp, seed, offset)
        torch.cuda.synchronize()
        _same(w, outs[i], ref, f"{case} call {i}")
        # fallback_rows is left out: whether a row overflows its candidate window
        # depends on how the block's warps interleave (each filters against the
        # running maximum it last saw), and the exact fallback gives the same cut
        got = counters[i].cpu().numpy().view("uint64")[:5]
        want = [ref["counters"][k] for k in ("dense_rows", "dense_bytes", "walk_bytes",
                                            "residual_passes", "final_draws")]
        assert [int(x) for x in got] == want, (case, i)


@pytest.mark.gpu
def test_noalloc_leaves_device_memory_unchanged(L):
    w = CASES["sampling-topp-bf16"]
    inp = _inputs(w, seed=303)
    out = _outputs(w.B, w.N, inp["max_depth"] + 1)
    _noalloc(w, inp, 9, 0, out)  # set-up and module loading happen here
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for offset in (1, 2):
        _noalloc(w, inp, 9, offset, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    ref = _with_workspace(w, inp, 9, 2)
    torch.cuda.synchronize()
    _same(w, out, ref, "after repeated calls")
