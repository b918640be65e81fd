"""Per-request sampling parameters: spec_verify_tree_per_request against the oracle,
tree by tree under each tree's own temperature / top-k / top-p (bit-exact on accepted
lengths, tokens and paths, alphas within the dtype's tolerance), and against the
batched entry point when every tree shares one setting (identical outputs)."""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import ALPHA_RTOL, gpu_inputs, log_exclusions
from speculative_decoding_tree_spec_gb300 import binding
from speculative_decoding_tree_spec_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (temperature, top_k, top_p) cycled over the trees: greedy, plain, top-p, top-k,
# both, top-k >= V (off), a cold and a hot temperature
MIX = [(0.0, 0, 1.0), (1.0, 0, 1.0), (0.7, 0, 0.9), (1.0, 50, 1.0), (0.6, 20, 0.8),
       (1.0, 1 << 30, 1.0), (0.3, 0, 0.95), (1.7, 0, 1.0)]


def _arrays(B, mix=MIX):
    T = torch.tensor([mix[b % len(mix)][0] for b in range(B)], dtype=torch.float32, device=DEV)
    k = torch.tensor([mix[b % len(mix)][1] for b in range(B)], dtype=torch.int32, device=DEV)
    p = torch.tensor([mix[b % len(mix)][2] for b in range(B)], dtype=torch.float32, device=DEV)
    return T, k, p


def _run(inp, T, k, p, flags=0, seed=9):
    out = binding.verify_tree_per_request(inp["p"], inp["q"], inp["tokens_d"], inp["parents_d"],
                                          inp["max_depth"], T, k, p, seed=seed, flags=flags)
    torch.cuda.synchronize()
    return {a: v.cpu().numpy() for a, v in out.items()}


def _check_vs_oracle(w, inp, gpu, T, k, p, seed=9):
    ph, qh = wl.host_logits(inp["p"]), wl.host_logits(inp["q"])
    ref = oracle.verify_tree_per_request(ph, qh, inp["tokens"], inp["parents"], inp["max_depth"],
                                         T.cpu().numpy(), k.cpu().numpy(), p.cpu().numpy(),
                                         seed=seed)
    compared = 0
    skipped = []
    for b, o in enumerate(ref):
        if o is None:
            assert gpu["status"][b] == 2 and gpu["accept_len"][b] == -1, b
            continue
        if o["near"][0]:
            skipped.append((b, oracle.near_reasons(o["near"][0])))
            continue
        compared += 1
        assert gpu["status"][b] == o["status"][0], b
        assert gpu["accept_len"][b] == o["accept_len"][0], (b, gpu["accept_len"][b], o["accept_len"][0])
        np.testing.assert_array_equal(gpu["tokens"][b], o["tokens"][0], err_msg=f"tree {b}")
        np.testing.assert_array_equal(gpu["path"][b], o["path"][0], err_msg=f"tree {b}")
        ga, oa = gpu["alpha"][b].astype(np.float64), o["alpha"][0]
        np.testing.assert_array_equal(np.isnan(ga), np.isnan(oa), err_msg=f"tree {b}")
        m = ~np.isnan(oa)
        err = np.abs(ga[m] - oa[m]) / np.maximum(np.abs(oa[m]), 1e-30)
        err = np.where(oa[m] == 0, np.abs(ga[m]), err)
        assert (err <= ALPHA_RTOL[w.dtype]).all(), (b, err.max() if err.size else 0)
    log_exclusions(w, skipped)
    return compared


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("flags", [0, binding.SPEC_FLAG_VISITED_ONLY], ids=["dense", "visited"])
def test_mixed_parameters_match_oracle(dtype, flags):
    w = wl.WORKLOADS["tree60_b64_v128256"].with_(B=16, N=26, V=8192 + 40, depth=5, dtype=dtype)
    inp = gpu_inputs(w, seed=41)
    T, k, p = _arrays(w.B)
    gpu = _run(inp, T, k, p, flags)
    assert _check_vs_oracle(w, inp, gpu, T, k, p) >= w.B // 2


@pytest.mark.parametrize("setting", [(0.7, 0, 0.9), (1.0, 50, 0.95), (0.0, 0, 1.0)],
                         ids=["top-p", "top-k+p", "greedy"])
@pytest.mark.parametrize("flags", [0, binding.SPEC_FLAG_VISITED_ONLY], ids=["dense", "visited"])
def test_uniform_arrays_equal_the_batched_call(setting, flags):
    w = wl.WORKLOADS["tree60_b64_v128256"].with_(B=24, N=30, V=32000, depth=5)
    inp = gpu_inputs(w, seed=42)
    T, k, p = _arrays(w.B, [setting])
    per = _run(inp, T, k, p, flags, seed=5)
    ref = binding.verify_tree(inp["p"], inp["q"], inp["tokens_d"], inp["parents_d"],
                              inp["max_depth"], *setting, seed=5, flags=flags)
    torch.cuda.synchronize()
    for a in ("accept_len", "tokens", "path", "status"):
        np.testing.assert_array_equal(per[a], ref[a].cpu().numpy(), err_msg=a)
    np.testing.assert_array_equal(per["alpha"], ref["alpha"].cpu().numpy())


def test_invalid_parameters_flag_only_their_trees():
    w = wl.WORKLOADS["tree60_b64_v128256"].with_(B=8, N=20, V=4096, depth=4, dtype="f32")
    inp = gpu_inputs(w, seed=43)
    T = torch.tensor([0.7, -1.0, float("nan"), 0.7, float("inf"), 0.7, 0.0, 1.0],
                     dtype=torch.float32, device=DEV)
    k = torch.tensor([0, 0, 0, -3, 0, 0, 0, 5], dtype=torch.int32, device=DEV)
    p = torch.tensor([1.0, 1.0, 1.0, 1.0, 1.0, 0.0, 1.0, float("nan")], dtype=torch.float32,
                     device=DEV)
    gpu = _run(inp, T, k, p)
    assert gpu["status"].tolist() == [0, 2, 2, 2, 2, 2, 0, 2]
    _check_vs_oracle(w, inp, gpu, T, k, p)


def test_optional_arrays_default_off():
    w = wl.WORKLOADS["tree60_b64_v128256"].with_(B=8, N=20, V=4096, depth=4)
    inp = gpu_inputs(w, seed=44)
    T = torch.full((w.B,), 0.9, dtype=torch.float32, device=DEV)
    a = _run(inp, T, None, None)
    b = _run(inp, T, torch.zeros(w.B, dtype=torch.int32, device=DEV),
             torch.ones(w.B, dtype=torch.float32, device=DEV))
    for key in ("accept_len", "tokens", "path", "alpha", "status"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
