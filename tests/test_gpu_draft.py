"""spec_draft_topk against the oracle on the same rows: children bit-exact (ties to the
lower index), confidences within 1e-5 relative."""
import numpy as np
import pytest
import torch

from oracle.draft import draft_topk as oracle_draft
from speculative_decoding_tree_spec_gb300 import binding
from speculative_decoding_tree_spec_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _rows(kind, R, V, dtype, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    if kind == "gauss":
        x = torch.randn((R, V), generator=g) * 3
    elif kind == "ties":
        x = torch.randint(-5, 6, (R, V), generator=g).float() * 0.5
    elif kind == "masked":
        x = torch.randn((R, V), generator=g) * 2
        x[torch.rand((R, V), generator=g) < 0.995] = float("-inf")
        x[:, 3] = 0.0
    else:
        raise ValueError(kind)
    return x.to(dtype)


def _check(x, k, T):
    d = wl.empty_rows(tuple(x.shape), x.dtype, DEV)
    d.copy_(x)
    out = binding.draft_topk(d, k, T)
    torch.cuda.synchronize()
    host = x.view(torch.int16).numpy().view(np.uint16) if x.dtype == torch.bfloat16 else x.numpy()
    tok, prob, st = oracle_draft(host, k, T)
    np.testing.assert_array_equal(out["status"].cpu().numpy(), st)
    np.testing.assert_array_equal(out["tokens"].cpu().numpy(), tok)
    gp = out["probs"].cpu().numpy().astype(np.float64)
    big = prob > 1e-30
    rel = np.abs(gp[big] - prob[big]) / prob[big]
    assert rel.max(initial=0.0) <= 1e-5, rel.max()
    assert np.all(np.abs(gp[~big]) <= 1e-30)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("kind", ["gauss", "ties", "masked"])
@pytest.mark.parametrize("k", [1, 10, 16, 32])
def test_draft_topk_matches_oracle(dtype, kind, k):
    _check(_rows(kind, 24, 32000 + 7, dtype, seed=k + len(kind)), k, 1.0)


@pytest.mark.parametrize("T", [0.25, 0.7, 2.0])
def test_draft_topk_temperatures(T):
    _check(_rows("gauss", 16, 128256, torch.bfloat16, seed=5), 10, T)


def test_draft_topk_small_and_ragged_rows():
    for V in (1, 5, 8, 9, 33, 257):
        k = min(V, 10)
        _check(_rows("gauss", 7, V, torch.float32, seed=V), k, 1.0)


def test_draft_topk_nonfinite_rows():
    x = _rows("gauss", 6, 5000, torch.float32, seed=2)
    x[1, 17] = float("nan")
    x[2, 4000] = float("inf")
    x[3, :] = float("-inf")
    _check(x, 10, 1.0)


def test_draft_topk_full_size_sampled():
    """The bench configuration (640 rows of V = 128256 bf16, k = 10): a sample of rows."""
    R, V = 640, 128256
    x = _rows("gauss", R, V, torch.bfloat16, seed=9)
    d = wl.empty_rows((R, V), torch.bfloat16, DEV)
    d.copy_(x)
    out = binding.draft_topk(d, 10, 1.0)
    torch.cuda.synchronize()
    host = x.view(torch.int16).numpy().view(np.uint16)
    for r in range(0, R, 53):
        tok, prob, st = oracle_draft(host[r:r + 1], 10, 1.0)
        assert out["tokens"][r].cpu().tolist() == tok[0].tolist(), r
        gp = out["probs"][r].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(gp - prob[0]) / prob[0]) <= 1e-5, r


def _adversarial(R_kind, V, dtype):
    """Rows whose largest logits arrive late, all at once, or tied in the thousands."""
    g = torch.Generator(device="cpu").manual_seed(11)
    if R_kind == "ascending":      # every later block beats all earlier ones
        x = torch.linspace(-8.0, 8.0, V).repeat(2, 1)
    elif R_kind == "descending":
        x = torch.linspace(8.0, -8.0, V).repeat(2, 1)
    elif R_kind == "constant":     # one value: the lowest indices win
        x = torch.full((2, V), 1.25)
    elif R_kind == "two_level":    # a few hundred tied maxima scattered over the row
        x = torch.zeros((2, V))
        x[torch.rand((2, V), generator=g) < 0.003] = 1.0
    elif R_kind == "late":         # the largest logits all in the row's last stretch
        x = torch.randn((2, V), generator=g)
        x[:, V - 3000:] += 6.0
    else:
        raise ValueError(R_kind)
    return x.to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("kind", ["ascending", "descending", "constant", "two_level", "late"])
def test_draft_topk_adversarial_orders(dtype, kind):
    """Full-vocabulary rows where a block of a round offers more candidates than the
    kernel's per-round buffer, or where every round raises the list: children still
    bit-exact with ties to the lower index."""
    x = _adversarial(kind, 128256, dtype)
    for k in (1, 10, 32):
        _check(x, k, 1.0)
