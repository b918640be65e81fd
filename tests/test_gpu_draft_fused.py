"""spec_draft_topk_fused_lmhead: the draft logits F W^T formed on the tensor cores and
ranked in the same call.  The children must equal the oracle's top-k of the bf16
logits the GEMM forms (handed out on request) exactly, the confidences within 1e-5
relative; the same as spec_draft_topk on those logits; and the same whether the
logits go to the caller's buffer or stay in the workspace."""
import numpy as np
import pytest
import torch

from oracle.draft import draft_topk as oracle_draft
from speculative_decoding_tree_spec_gb300 import binding

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(R, V, d, seed, w_std=0.02):
    g = torch.Generator(device=DEV).manual_seed(seed)
    f = torch.randn((R, d), generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn((V, d), generator=g, device=DEV) * w_std).to(torch.bfloat16)
    return f, w


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check(R, V, d, k, T, seed, rows=None):
    f, w = _inputs(R, V, d, seed)
    a = binding.draft_topk_fused_lmhead(f, w, k, T, want_logits=True)
    b = binding.draft_topk_fused_lmhead(f, w, k, T, want_logits=False)
    torch.cuda.synchronize()
    assert a["status"].cpu().tolist() == [0] * R
    for key in ("tokens", "probs", "status"):
        assert torch.equal(a[key], b[key]), key
    # the row-by-row kernel on the written logits ranks identically
    c = binding.draft_topk(a["logits"], k, T)
    torch.cuda.synchronize()
    assert torch.equal(a["tokens"], c["tokens"])
    rel = ((a["probs"].double() - c["probs"].double()).abs() / c["probs"].double()).max().item()
    assert rel <= 2e-5, rel
    host = _bits(a["logits"])
    for r in (range(R) if rows is None else rows):
        tok, prob, st = oracle_draft(host[r:r + 1], k, T)
        assert st[0] == 0
        assert a["tokens"][r].cpu().tolist() == tok[0].tolist(), r
        gp = a["probs"][r].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(gp - prob[0]) / prob[0]) <= 1e-5, r


@pytest.mark.parametrize("R,V,d", [(50, 1000, 128), (130, 4096 + 40, 200), (1, 300, 64)],
                         ids=["ragged", "two-row-tiles-ragged-k", "one-row"])
@pytest.mark.parametrize("k", [1, 10, 32])
def test_fused_draft_small(R, V, d, k):
    _check(R, V, d, min(k, V), 1.0, seed=R + V + k)


def test_fused_draft_temperature():
    _check(64, 5000, 256, 10, 0.6, seed=3)


def test_fused_draft_full_size_sampled():
    """The bench configuration: 640 rows, V = 128256, d = 4096, k = 10."""
    _check(640, 128256, 4096, 10, 1.0, seed=11, rows=range(0, 640, 71))
