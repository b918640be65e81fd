"""Edge cases run through the checked build of the library (compiled with
-DSPEC_CHECK: the dense pass's and the walk's buffer indices are checked on the
device, and an index out of range sets a bit of an error word instead of being
used).  Run as a script in a child process (the library path is chosen before the
library loads): argv[1] is the checked library's path.  Every case is compared with
the oracle as the parity tests compare it; the script prints, as JSON, the trees
compared per case and the two error words read after all cases."""
import json
import sys

import numpy as np
import torch

from speculative_decoding_tree_spec_gb300 import binding

binding.LIB_PATH = sys.argv[1]

import oracle  # noqa: E402
from parity_helpers import compare, gpu_inputs, run_gpu, run_oracle  # noqa: E402
from speculative_decoding_tree_spec_gb300 import workloads as wl  # noqa: E402

W = wl.WORKLOADS
C3 = W["tree60_b64_v128256"]
C4 = W["tree26_b256_v152064"]

CASES = {
    # one warp per tree (no cut, small vocabularies)
    "small-v1": C3.with_(B=40, N=5, V=1, dtype="f32", depth=3, temperature=0.9, top_p=1.0),
    "small-v7": C3.with_(B=200, N=12, V=7, dtype="bf16", depth=4, temperature=0.9, top_p=1.0),
    "small-v33": C3.with_(B=200, N=64, V=33, dtype="f32", depth=6, temperature=1.1, top_p=1.0),
    # cluster walk on small and ragged vocabularies with cuts
    "cut-v33-f32": C3.with_(B=20, N=12, V=33, dtype="f32", depth=4, top_p=0.8),
    "cut-v7-bf16": C3.with_(B=20, N=12, V=7, dtype="bf16", depth=4, top_p=0.8),
    "topk-ragged": C3.with_(B=8, N=40, V=5003, temperature=1.3, top_k=7, top_p=0.8),
    "window-c8": C3.with_(B=6, V=40000),
    "topk-c8": C4.with_(B=8, V=40000),
    "tree60-b64-v32000": C3.with_(V=32000),
    "fp32-plain": C3.with_(B=8, N=33, V=999, dtype="f32", temperature=0.9, top_p=1.0),
}


def run(name, w, flags=0):
    inp = gpu_inputs(w, 61)
    gpu = run_gpu(w, inp, seed=62, flags=flags)
    sel, outs = run_oracle(w, inp, seed=62)
    n, ex, err = compare(w, gpu, sel, outs)
    return n


def main():
    assert binding.lib().spec_check_build() == 1, "not the checked build"
    out = {}
    for name, w in CASES.items():
        out[name] = run(name, w)
    out["visited-only"] = run("visited-only", C3.with_(B=6, V=40000),
                              flags=binding.SPEC_FLAG_VISITED_ONLY)
    out["exact-select"] = run("exact-select", C4.with_(B=6, V=20000),
                              flags=binding.SPEC_FLAG_EXACT_SELECT)
    # every logit equal: the top-k lists cannot make room and the rows take the exact
    # selection
    rng = np.random.default_rng(3)
    B, N, V = 6, 7, 20000
    par = np.stack([wl.random_tree(N, 3, 3, rng) for _ in range(B)])
    p = torch.zeros((B, N, V), dtype=torch.bfloat16)
    q = torch.as_tensor(np.round(rng.normal(0, 2, size=(B, N, V)) * 2) / 2).to(torch.bfloat16)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    dev = "cuda:0"
    pd = wl.empty_rows((B, N, V), torch.bfloat16, dev)
    qd = wl.empty_rows((B, N, V), torch.bfloat16, dev)
    pd.copy_(p)
    qd.copy_(q)
    res = binding.verify_tree(pd, qd, torch.as_tensor(tok, device=dev),
                              torch.as_tensor(par, device=dev), 3, 1.0, 100, 0.905, seed=3)
    torch.cuda.synchronize()
    ref = oracle.verify_tree(wl.host_logits(p), wl.host_logits(q), tok, par, 3, 1.0, 100, 0.905,
                             seed=3)
    keep = ref["near"] == 0
    assert (res["status"].cpu().numpy() == ref["status"]).all()
    assert (res["tokens"].cpu().numpy()[keep] == ref["tokens"][keep]).all()
    out["all-ties"] = int(keep.sum())
    out["words"] = binding.check_errors()
    print(json.dumps(out))


if __name__ == "__main__":
    main()
