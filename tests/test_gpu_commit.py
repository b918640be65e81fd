"""spec_commit_accepted_path against the oracle on the same caches and paths: bit-exact."""
import numpy as np
import pytest
import torch

from oracle.commit import commit_accepted_path as oracle_commit
from speculative_decoding_tree_spec_gb300 import binding
from speculative_decoding_tree_spec_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _paths(B, N, W, seed):
    """Accepted paths of random trees: a random root-to-node walk per tree."""
    rng = np.random.default_rng(seed)
    w = wl.WORKLOADS["tree60_b64_v128256"].with_(B=B, N=N, depth=W - 1)
    parents = wl.make_parents(w, seed)
    path = np.full((B, W), -1, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        node, k = 0, 0
        path[b, 0] = 0
        while True:
            kids = [c for c in range(N) if parents[b][c] == node]
            if not kids or rng.random() < 0.25:
                break
            node = int(rng.choice(kids))
            k += 1
            path[b, k] = node
        acc[b] = k
    acc[0] = -1  # a failed tree
    return path, acc


@pytest.mark.parametrize("P,B,N,n_pos,row_bytes", [(4, 8, 30, 200, 2048), (1, 16, 60, 128, 48),
                                                    (64, 4, 26, 96, 4096 + 16)],
                         ids=["kv", "narrow-rows", "many-planes"])
def test_commit_matches_oracle(P, B, N, n_pos, row_bytes):
    W = 7
    path, acc = _paths(B, N, W, seed=P + B)
    prefix = np.random.default_rng(1).integers(0, n_pos - N, size=B).astype(np.int32)
    g = torch.Generator(device="cpu").manual_seed(3)
    cache = torch.randint(0, 256, (P, B, n_pos, row_bytes), dtype=torch.uint8, generator=g)
    want = oracle_commit(cache.numpy(), prefix, path, acc)
    d = cache.to(DEV)
    binding.commit_accepted_path(d, torch.as_tensor(prefix, device=DEV),
                                 torch.as_tensor(path, device=DEV), torch.as_tensor(acc, device=DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(d.cpu().numpy(), want)


def test_commit_after_verify_on_bf16_cache():
    """The verify outputs drive the commit of a bf16 [layers*2, B, positions, heads*dim] cache."""
    w = wl.WORKLOADS["tree60_b64_v128256"].with_(B=6, V=5000)
    inp = wl.build_inputs(w, seed=4, device=torch.device(DEV))
    out = binding.verify_tree(inp["p"], inp["q"], torch.as_tensor(inp["tokens"], device=DEV),
                              torch.as_tensor(inp["parents"], device=DEV), inp["max_depth"],
                              w.temperature, w.top_k, w.top_p, seed=2)
    n_pos = 96
    prefix = torch.tensor([3, 7, 11, 0, 20, 30], dtype=torch.int32, device=DEV)
    cache = torch.randn((8, w.B, n_pos, 256), generator=torch.Generator(device=DEV).manual_seed(1),
                        device=DEV).to(torch.bfloat16)
    want = oracle_commit(cache.view(torch.uint8).cpu().numpy(), prefix.cpu().numpy(),
                         out["path"].cpu().numpy(), out["accept_len"].cpu().numpy())
    binding.commit_accepted_path(cache, prefix, out["path"], out["accept_len"])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cache.view(torch.uint8).cpu().numpy(), want)
