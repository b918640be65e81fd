"""Shared helpers of the GPU parity tests: run one workload through the CUDA library
and through the oracle on the same seeded inputs and compare them."""
import concurrent.futures as cf
import json
import os

import numpy as np
import torch

import oracle
from speculative_decoding_tree_spec_gb300 import binding
from speculative_decoding_tree_spec_gb300 import workloads as wl

# Probability tolerance of the verify outputs (relative), by logit dtype.
ALPHA_RTOL = {"f32": 1e-5, "bf16": 2e-3}


def gpu_inputs(w, seed):
    dev = torch.device("cuda:0")
    inp = wl.build_inputs(w, seed=seed, device=dev)
    inp["tokens_d"] = torch.as_tensor(inp["tokens"], device=dev)
    inp["parents_d"] = torch.as_tensor(inp["parents"], device=dev)
    return inp


def run_gpu(w, inp, seed=7, offset=0, flags=0, top_k=None, top_p=None, temperature=None):
    T = w.temperature if temperature is None else temperature
    k = w.top_k if top_k is None else top_k
    p = w.top_p if top_p is None else top_p
    out = binding.verify_tree(inp["p"], inp["q"], inp["tokens_d"], inp["parents_d"],
                              inp["max_depth"], T, k, p, seed=seed, offset=offset, flags=flags,
                              want_counters=True)
    torch.cuda.synchronize()
    return {k2: (v.cpu().numpy() if torch.is_tensor(v) else v) for k2, v in out.items()}


def run_oracle(w, inp, trees=None, seed=7, offset=0, top_k=None, top_p=None, temperature=None,
               threads=1):
    T = w.temperature if temperature is None else temperature
    k = w.top_k if top_k is None else top_k
    p = w.top_p if top_p is None else top_p
    sel = np.arange(w.B) if trees is None else np.asarray(trees)
    idx = torch.as_tensor(sel, device=inp["p"].device)
    ph = wl.host_logits(inp["p"].index_select(0, idx))
    qh = wl.host_logits(inp["q"].index_select(0, idx))
    # the oracle keys its uniforms on the tree index: run each sampled tree at its own b
    # (one tree per task; the oracle's C walk releases the interpreter lock)
    def one(j):
        b = sel[j]
        return oracle.verify_tree(ph[j:j + 1], qh[j:j + 1], inp["tokens"][b:b + 1],
                                  inp["parents"][b:b + 1], inp["max_depth"], T, k, p,
                                  seed=seed, offset=offset, nthreads=1, **_batch_index(b))

    if threads > 1:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            outs = list(ex.map(one, range(len(sel))))
    else:
        outs = [one(j) for j in range(len(sel))]
    return sel, outs


def _batch_index(b):
    return {"batch_index": int(b)}


def log_exclusions(w, excluded):
    """Every tree left out of a comparison, with the decisions that put it within 1e-6
    of a boundary: printed, and appended as one JSON line to the file named by
    PARITY_EXCLUSION_LOG when that is set."""
    if not excluded:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    rec = {"test": test, "workload": w.name, "B": w.B, "N": w.N, "V": w.V,
           "excluded": [{"tree": int(b), "near": why} for b, why in excluded]}
    print("parity exclusions:", json.dumps(rec))
    path = os.environ.get("PARITY_EXCLUSION_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def compare(w, gpu, sel, outs, check_alpha=True):
    """Exact comparison of accepted length, tokens and path on every tree that the
    oracle does not flag as within 1e-6 of a decision boundary; alphas within the
    dtype's tolerance.  Every excluded tree is logged with the decisions that
    excluded it.  Returns (number compared, number excluded, max alpha error)."""
    compared = excluded = 0
    max_err = 0.0
    rtol = ALPHA_RTOL[w.dtype]
    skipped = []
    for j, b in enumerate(sel):
        o = outs[j]
        if o["near"][0]:
            excluded += 1
            skipped.append((b, oracle.near_reasons(o["near"][0])))
            continue
        compared += 1
        assert gpu["status"][b] == o["status"][0], (b, gpu["status"][b], o["status"][0])
        assert gpu["accept_len"][b] == o["accept_len"][0], (b, gpu["accept_len"][b], o["accept_len"][0])
        np.testing.assert_array_equal(gpu["tokens"][b], o["tokens"][0], err_msg=f"tree {b}")
        np.testing.assert_array_equal(gpu["path"][b], o["path"][0], err_msg=f"tree {b}")
        if check_alpha:
            ga = gpu["alpha"][b].astype(np.float64)
            oa = o["alpha"][0]
            np.testing.assert_array_equal(np.isnan(ga), np.isnan(oa), err_msg=f"tree {b}")
            m = ~np.isnan(oa)
            if m.any():
                err = np.abs(ga[m] - oa[m]) / np.maximum(np.abs(oa[m]), 1e-30)
                err = np.where(oa[m] == 0, np.abs(ga[m]), err)
                max_err = max(max_err, float(err.max()))
                assert err.max() <= rtol, (b, err.max())
    log_exclusions(w, skipped)
    return compared, excluded, max_err
