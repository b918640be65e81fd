"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on the
same seeded inputs.  Token ids, accepted lengths, paths, argmax and cut indices
must match exactly; probabilities within 1e-5 relative for fp32 logits and 2e-3
for bf16 logits.  Trees / rows the oracle flags as within 1e-6 of a decision
boundary are excluded from the exact comparison and counted."""
import os

import numpy as np
import pytest
import torch

import oracle
from parity_helpers import compare, gpu_inputs, run_gpu, run_oracle
from speculative_decoding_tree_spec_gb300 import binding
from speculative_decoding_tree_spec_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
W = wl.WORKLOADS


# --- Philox ----------------------------------------------------------------------

def test_philox_words_match_oracle():
    rng = np.random.default_rng(0)
    n = 4096
    b = rng.integers(0, 2**31 - 1, size=n).astype(np.int32)
    node = rng.integers(0, 5000, size=n).astype(np.int32)
    for seed, offset in ((0, 0), (0xDEADBEEFCAFEF00D, 0), (12345, (7 << 32) | 99)):
        g = binding.philox_words(seed, offset, torch.as_tensor(b, device=DEV),
                                 torch.as_tensor(node, device=DEV)).cpu().numpy()
        for i in range(0, n, 97):
            ctr = [node[i], b[i], offset & 0xFFFFFFFF, offset >> 32]
            key = [seed & 0xFFFFFFFF, seed >> 32]
            assert list(g[i]) == list(oracle.philox4x32_10(ctr, key)), i


# --- the dense row pass ----------------------------------------------------------

def _rows(kind, R, V, dtype, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    if kind == "gauss":
        x = torch.randn((R, V), generator=g) * 3
    elif kind == "ties":
        x = torch.randint(-6, 7, (R, V), generator=g).float() * 0.5
    elif kind == "flat":
        x = torch.randn((R, V), generator=g) * 0.05
    elif kind == "zipf":
        rank = torch.stack([torch.randperm(V, generator=g) for _ in range(R)]).float() + 1
        x = -1.1 * torch.log(rank) + torch.randn((R, V), generator=g) * 2
    elif kind == "masked":
        x = torch.randn((R, V), generator=g) * 3
        x[torch.rand((R, V), generator=g) < 0.7] = float("-inf")
        x[:, 0] = 0.0
    else:
        raise ValueError(kind)
    return x.to(dtype)


def _dev_rows(x):
    """Device copy of [R, V] rows with a 16-byte aligned row pitch."""
    d = wl.empty_rows(tuple(x.shape), x.dtype, DEV)
    d.copy_(x)
    return d


def _check_rows(x, T, k, p, flags=0):
    st = binding.filter_rows(_dev_rows(x), T, k, p, flags)
    torch.cuda.synchronize()
    st = {a: b.cpu().numpy() for a, b in st.items()}
    host = x.view(torch.int16).numpy().view(np.uint16) if x.dtype == torch.bfloat16 else x.numpy()
    _, infos = oracle.filter_rows(host, T, k, p)
    rtol = 2e-3 if x.dtype == torch.bfloat16 else 1e-5
    worst = 0.0
    near = 0
    for r, info in enumerate(infos):
        assert st["status"][r] == info.status, r
        if info.status:
            continue
        assert st["argmax"][r] == info.argmax, r
        assert st["m"][r] == np.float32(info.m), r
        if info.near:
            near += 1
            continue
        V = x.shape[1]
        if T > 0 and not (0 < k < V) and p >= 1:
            # nothing truncated: the row reports the "every token passes" cut
            assert (st["cut_key"][r], st["cut_idx"][r], st["kept"][r]) == (0, V - 1, V)
            assert info.kept == V
        else:
            assert st["cut_idx"][r] == info.cut_idx, (r, st["cut_idx"][r], info.cut_idx)
        assert st["kept"][r] == info.kept, (r, st["kept"][r], info.kept)
        rel = abs(st["s_f"][r] - info.s_f) / info.s_f
        worst = max(worst, rel)
        assert rel <= rtol, (r, st["s_f"][r], info.s_f)
    return st, worst, near


PARAMS = [(0.0, 0, 1.0), (1.0, 0, 1.0), (0.7, 0, 0.9), (1.0, 50, 0.95), (0.5, 5, 1.0),
          (2.0, 0, 0.5), (1.0, 1, 1.0), (0.8, 0, 0.999), (1.3, 300, 0.8)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("kind", ["gauss", "ties", "flat", "zipf", "masked"])
@pytest.mark.parametrize("V", [1, 7, 33, 1000, 32000])
def test_filter_rows_match_oracle(dtype, kind, V):
    x = _rows(kind, 6, V, dtype, seed=V * 31 + len(kind))
    for T, k, p in PARAMS:
        st, worst, near = _check_rows(x, T, k, p)
        if T > 0 and (p < 1 or 0 < k < V):
            st2 = binding.filter_rows(_dev_rows(x), T, k, p, binding.SPEC_FLAG_EXACT_SELECT)
            torch.cuda.synchronize()
            for key in ("cut_idx", "kept", "s_f", "cut_key", "argmax", "m"):
                np.testing.assert_array_equal(st[key], st2[key].cpu().numpy(), err_msg=key)


@pytest.mark.parametrize("V", [128256, 152064])
def test_filter_rows_large_vocab(V):
    for kind, (T, k, p) in (("gauss", (0.7, 0, 0.9)), ("zipf", (1.0, 50, 0.95)),
                            ("flat", (1.0, 0, 0.9)), ("ties", (1.0, 0, 0.95))):
        x = _rows(kind, 4, V, torch.bfloat16, seed=V + k)
        st, worst, near = _check_rows(x, T, k, p)
        st2 = binding.filter_rows(_dev_rows(x), T, k, p, binding.SPEC_FLAG_EXACT_SELECT)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(st["cut_idx"], st2["cut_idx"].cpu().numpy())
        np.testing.assert_array_equal(st["s_f"], st2["s_f"].cpu().numpy())


def test_filter_rows_non_finite():
    x = torch.randn((5, 100)) * 2
    x[0, 3] = float("nan")
    x[1, 50] = float("inf")
    x[2, :] = float("-inf")
    x[3, :90] = float("-inf")
    for T, k, p in ((0.0, 0, 1.0), (1.0, 0, 1.0), (1.0, 0, 0.9), (1.0, 20, 1.0)):
        st = binding.filter_rows(_dev_rows(x), T, k, p)
        torch.cuda.synchronize()
        s = st["status"].cpu().numpy()
        assert list(s) == [1, 1, 1, 0, 0], (T, k, p, s)


def test_bounded_wait_self_test_reports_timeout():
    """The stall self-test withholds one copy's completion: the row pass's bounded
    wait gives up, the rows report SPEC_ROW_TIMEOUT, and the next call is normal."""
    x = _rows("gauss", 8, 40000, torch.bfloat16, seed=1)
    for T, k, p in ((0.7, 0, 0.9), (1.0, 0, 1.0), (0.0, 0, 1.0)):
        st = binding.filter_rows(_dev_rows(x), T, k, p, binding.SPEC_FLAG_TEST_STALL)
        torch.cuda.synchronize()
        assert (st["status"].cpu().numpy() == binding.SPEC_ROW_TIMEOUT).all()
        st = binding.filter_rows(_dev_rows(x), T, k, p)
        torch.cuda.synchronize()
        assert (st["status"].cpu().numpy() == 0).all()
    w = W["tree60_b64_v128256"].with_(B=4, V=40000)
    inp = gpu_inputs(w, 2)
    out = run_gpu(w, inp, flags=binding.SPEC_FLAG_TEST_STALL)
    assert (out["status"] == binding.SPEC_ROW_TIMEOUT).all()
    assert (out["accept_len"] == -1).all()
    out = run_gpu(w, inp)
    assert (out["status"] == 0).all()


def test_filter_rows_negative_zero_ties():
    x = torch.tensor([[-0.0, 0.0, -1.0, -0.0, -3.0]])
    st = binding.filter_rows(_dev_rows(x), 1.0, 2, 1.0)
    torch.cuda.synchronize()
    assert st["argmax"].item() == 0 and st["cut_idx"].item() == 1


# --- the full verify step ----------------------------------------------------------

def _parity(w, seed, trees=None, **kw):
    inp = gpu_inputs(w, seed)
    gpu = run_gpu(w, inp, seed=seed + 1, **kw)
    sel, outs = run_oracle(w, inp, trees=trees, seed=seed + 1, **{k: v for k, v in kw.items()
                                                                if k != "flags"})
    n, ex, err = compare(w, gpu, sel, outs)
    assert n >= max(1, len(sel) // 2), f"too many excluded trees: {ex} of {len(sel)}"
    return gpu, n, ex, err


def test_chain_v32_full():
    w = W["chain_g3_v32"]
    gpu, n, ex, err = _parity(w, seed=3)
    assert n > 9900


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_eagle10_v32000(T):
    w = W["eagle10_v32000"].with_(B=24, temperature=T)
    _parity(w, seed=11)


@pytest.mark.parametrize("w", [
    W["tree60_b64_v128256"].with_(B=6),
    W["tree26_b256_v152064"].with_(B=6),
    W["tree60_b64_v128256"].with_(B=6, dtype="f32", V=32000),
    W["tree26_b256_v152064"].with_(B=6, temperature=0.0),
    W["tree60_b64_v128256"].with_(B=8, N=40, V=5003, temperature=1.3, top_k=7, top_p=0.8),
    W["tree60_b64_v128256"].with_(B=8, N=33, V=999, dtype="f32", temperature=0.9, top_k=0,
                                  top_p=1.0),
], ids=["c3-reduced", "c4-reduced", "c3-f32", "c4-greedy", "ragged-topk-topp", "f32-plain"])
def test_random_trees(w):
    _parity(w, seed=21)


# --- the benchmarked workloads at their own sizes: the launch geometry the bench times
# (the walk's cluster size follows B: 4 CTAs per tree at B = 64, one at B = 256) -------

HOST_THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.mark.parametrize("name,seed,min_compared", [
    ("tree60_b64_v128256", 20261202, 32), ("tree60_b64_v128256", 5, 32),
    ("tree26_b256_v152064", 20261202, 128), ("tree26_b256_v152064", 77, 128)])
def test_benchmarked_workload_every_tree(name, seed, min_compared):
    w = W[name]
    inp = gpu_inputs(w, seed)
    gpu = run_gpu(w, inp, seed=seed + 1)
    sel, outs = run_oracle(w, inp, seed=seed + 1, threads=HOST_THREADS)
    n, ex, err = compare(w, gpu, sel, outs)
    print(f"{name} seed {seed}: {n} trees compared, {ex} excluded, max alpha error {err:.2e}, "
          f"cut rows through the full-row selection {gpu['counters']['fallback_rows']}")
    assert len(sel) == w.B and n >= min_compared, (n, ex)


# --- the dense pass of a tree launch reads exactly the rows the walk may need -------

@pytest.mark.parametrize("per_request", [False, True])
def test_tree_row_pass_reads_exactly_the_needed_rows(per_request):
    """Every target row's statistics, and those of the draft rows of nodes with a
    child (of sampled trees), equal spec_filter_rows' on the same rows; no other draft
    row is written.  (The statistics sit at the start of the workspace: B*N target
    records, then, 256-byte aligned, B*N draft records.)"""
    w = W["tree60_b64_v128256"].with_(V=32000)
    B, N, V = w.B, w.N, w.V
    inp = gpu_inputs(w, 3)
    ws = torch.full((binding.workspace_size(B, N, V),), 0xAB, dtype=torch.uint8, device=DEV)
    phases = binding.SPEC_PHASE_PREPARE | binding.SPEC_PHASE_ROWS
    temps = np.array([0.0 if (per_request and b % 3 == 0) else 0.7 for b in range(B)],
                     np.float32)
    if per_request:
        binding.verify_tree_per_request(inp["p"], inp["q"], inp["tokens_d"], inp["parents_d"],
                                        inp["max_depth"], torch.as_tensor(temps, device=DEV),
                                        workspace=ws, phases=phases)
    else:
        binding.verify_tree(inp["p"], inp["q"], inp["tokens_d"], inp["parents_d"],
                            inp["max_depth"], 0.7, workspace=ws, phases=phases)
    torch.cuda.synchronize()
    BN = B * N
    off_q = (BN * 32 + 255) // 256 * 256
    got_p = ws[:BN * 32].view(BN, 32).cpu().numpy()
    got_q = ws[off_q:off_q + BN * 32].view(BN, 32).cpu().numpy()
    rows = {k: inp[k].as_strided((BN, V), (inp[k].stride(1), 1)) for k in ("p", "q")}
    ref = {}
    for k in ("p", "q"):
        st = torch.empty((BN, 32), dtype=torch.uint8, device=DEV)
        assert binding.lib().spec_filter_rows(rows[k].data_ptr(), binding._dtype_code(rows[k]),
                                              BN, V, rows[k].stride(0),
                                              binding.params(0.7, 0, 1.0, 0), st.data_ptr(),
                                              0) == 0
        torch.cuda.synchronize()
        ref[k] = st.cpu().numpy()
    par = inp["parents"]
    has_child = np.zeros((B, N), bool)
    for b in range(B):
        for ch in range(1, N):
            if 0 <= par[b, ch] < ch:
                has_child[b, par[b, ch]] = True
    sampled = np.repeat(temps > 0, N)
    need_q = has_child.reshape(-1) & sampled
    # target rows: every record (greedy trees: the maximum and its index)
    np.testing.assert_array_equal(got_p[sampled], ref["p"][sampled])
    g = got_p[~sampled].view(np.int32)
    r = ref["p"][~sampled].view(np.int32)
    np.testing.assert_array_equal(g[:, [0, 6]], r[:, [0, 6]])
    np.testing.assert_array_equal(got_q[need_q], ref["q"][need_q])
    assert (got_q[~need_q] == 0xAB).all()


# --- small vocabularies without a cut: one warp per tree, no dense pass --------------

@pytest.mark.parametrize("dtype,V,N", [("f32", 256, 64), ("bf16", 200, 40), ("f32", 33, 12),
                                       ("bf16", 1, 5), ("f32", 32, 4)])
def test_small_vocabulary_walk(dtype, V, N):
    w = W["tree60_b64_v128256"].with_(B=300, N=N, V=V, dtype=dtype, depth=min(6, N - 1),
                                      temperature=0.9, top_k=0, top_p=1.0)
    gpu, n, ex, err = _parity(w, seed=51)
    # the rows it visits are read by the walk itself
    assert gpu["counters"]["dense_rows"] == 0 and gpu["counters"]["walk_bytes"] > 0


# --- the top-k route of bf16 rows (per-CTA lists under a rising threshold) ----------

@pytest.mark.parametrize("w", [
    W["tree26_b256_v152064"].with_(B=32, top_k=128),
    W["tree26_b256_v152064"].with_(B=32, top_k=129),
    W["tree26_b256_v152064"].with_(B=300, N=6, V=3001, depth=3, top_k=5, top_p=1.0),
    W["tree60_b64_v128256"].with_(B=16, top_k=20),
    W["tree60_b64_v128256"].with_(B=16, V=9000, top_k=1, top_p=0.5),
], ids=["k128-largest-listed", "k129-window-route", "k5-ragged-one-cta", "gauss-k20-topp",
        "k1"])
def test_topk_route(w):
    _parity(w, seed=41)


def test_topk_route_equals_exact_selection():
    w = W["tree26_b256_v152064"].with_(B=16, V=40000)
    inp = gpu_inputs(w, 12)
    a = run_gpu(w, inp, seed=13)
    b = run_gpu(w, inp, seed=13, flags=binding.SPEC_FLAG_EXACT_SELECT)
    for key in ("accept_len", "tokens", "path", "status"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    np.testing.assert_array_equal(a["alpha"], b["alpha"])
    # every cut row took the list route; the flag sent every one to the exact selection
    assert a["counters"]["fallback_rows"] == 0 and b["counters"]["fallback_rows"] > 0


@pytest.mark.parametrize("levels,k", [(6, 100), (200, 50), (2, 3), (0, 100)])
def test_topk_route_ties(levels, k):
    """Logits on a coarse grid tie in large groups at the k-th key: the cut is the
    k-th token in (logit desc, index asc) order whether the lists hold the tied group
    or leave the row to the exact selection (levels 0: every p logit ties, more than
    a list holds)."""
    rng = np.random.default_rng(levels)
    B, N, V = 12, 7, 20000
    par = np.stack([wl.random_tree(N, 3, 3, rng) for _ in range(B)])

    def grid(x):
        return np.zeros_like(x) if levels == 0 else np.round(x * levels / 6) * 6 / levels

    p = grid(rng.normal(0, 2, size=(B, N, V))).astype(np.float32)
    q = np.round(rng.normal(0, 2, size=(B, N, V)) * 2).astype(np.float32) / 2
    ph = torch.as_tensor(p).to(torch.bfloat16)
    qh = torch.as_tensor(q).to(torch.bfloat16)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    out = binding.verify_tree(_dev_rows(ph), _dev_rows(qh), torch.as_tensor(tok, device=DEV),
                              torch.as_tensor(par, device=DEV), 3, 1.0, k, 0.905, seed=3)
    torch.cuda.synchronize()
    gpu = {a: b.cpu().numpy() for a, b in out.items()}
    ref = oracle.verify_tree(wl.host_logits(ph), wl.host_logits(qh), tok, par, 3, 1.0, k, 0.905,
                             seed=3)
    _assert_same(gpu, ref)
    assert (ref["near"] == 0).sum() >= B // 2


def test_topk_route_far_kth_token():
    """An outlier maximum puts the k-th largest logit far below the window's floor
    (m - 9 T): the lists are collected again with no floor and the rows still
    take the list route."""
    rng = np.random.default_rng(17)
    B, N, V, k = 10, 6, 30000, 40
    par = np.stack([wl.random_tree(N, 3, 2, rng) for _ in range(B)])
    p = rng.normal(0, 1, size=(B, N, V)).astype(np.float32)
    q = rng.normal(0, 1, size=(B, N, V)).astype(np.float32)
    p[:, :, 7] = 25.0
    q[:, :, 11] = 20.0
    ph = torch.as_tensor(p).to(torch.bfloat16)
    qh = torch.as_tensor(q).to(torch.bfloat16)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    tok[:, 1::2] = 7
    out = binding.verify_tree(_dev_rows(ph), _dev_rows(qh), torch.as_tensor(tok, device=DEV),
                              torch.as_tensor(par, device=DEV), 3, 1.0, k, 1.0, seed=5,
                              want_counters=True)
    torch.cuda.synchronize()
    gpu = {a: (b.cpu().numpy() if torch.is_tensor(b) else b) for a, b in out.items()}
    ref = oracle.verify_tree(wl.host_logits(ph), wl.host_logits(qh), tok, par, 3, 1.0, k, 1.0,
                             seed=5)
    _assert_same(gpu, ref)
    assert gpu["counters"]["fallback_rows"] == 0


def test_exact_select_flag_gives_identical_outputs():
    w = W["tree60_b64_v128256"].with_(B=6, V=40000)
    inp = gpu_inputs(w, 5)
    a = run_gpu(w, inp, seed=9)
    b = run_gpu(w, inp, seed=9, flags=binding.SPEC_FLAG_EXACT_SELECT)
    for key in ("accept_len", "tokens", "path", "status"):
        np.testing.assert_array_equal(a[key], b[key])
    np.testing.assert_array_equal(a["alpha"], b["alpha"])
    # the walk cuts the rows it visits: the p row of every node on the accepted path
    # and the q row of those with children; the flag sends each through the exact
    # full-row selection
    cut_rows = 0
    for t in range(w.B):
        path = b["path"][t][: b["accept_len"][t] + 1]
        has_child = set(inp["parents"][t][1:].tolist())
        cut_rows += len(path) + sum(int(n) in has_child for n in path)
    assert b["counters"]["fallback_rows"] == cut_rows


def test_top1_sampling_equals_greedy_on_gpu():
    w = W["tree26_b256_v152064"].with_(B=8, V=20000)
    inp = gpu_inputs(w, 8)
    g = run_gpu(w, inp, temperature=0.0, top_k=0, top_p=1.0)
    s = run_gpu(w, inp, temperature=0.9, top_k=1, top_p=1.0)
    np.testing.assert_array_equal(g["accept_len"], s["accept_len"])
    np.testing.assert_array_equal(g["tokens"], s["tokens"])


def test_repeat_calls_are_bit_identical():
    w = W["tree60_b64_v128256"].with_(B=8, V=50000)
    inp = gpu_inputs(w, 4)
    a = run_gpu(w, inp, seed=3, offset=10)
    b = run_gpu(w, inp, seed=3, offset=10)
    c = run_gpu(w, inp, seed=3, offset=11)
    for key in ("accept_len", "tokens", "path", "alpha"):
        np.testing.assert_array_equal(a[key], b[key])
    assert not np.array_equal(a["tokens"], c["tokens"]) or not np.array_equal(a["alpha"], c["alpha"])


# --- edge cases --------------------------------------------------------------------

def _manual(p, q, tokens, parents, D, T, k=0, top_p=1.0, seed=1, broadcast=False):
    pd = _dev_rows(torch.as_tensor(p))
    qd = _dev_rows(torch.as_tensor(q))
    out = binding.verify_tree(pd, qd, torch.as_tensor(tokens, device=DEV),
                              torch.as_tensor(parents, device=DEV), D, T, k, top_p, seed=seed,
                              batch_broadcast=broadcast)
    torch.cuda.synchronize()
    gpu = {a: b.cpu().numpy() for a, b in out.items()}
    ref = oracle.verify_tree(np.asarray(p), np.asarray(q), tokens, parents, D, T, k, top_p,
                             seed=seed, batch_broadcast=broadcast)
    return gpu, ref


def _assert_same(gpu, ref):
    keep = ref["near"] == 0
    np.testing.assert_array_equal(gpu["status"], ref["status"])
    np.testing.assert_array_equal(gpu["accept_len"][keep], ref["accept_len"][keep])
    np.testing.assert_array_equal(gpu["tokens"][keep], ref["tokens"][keep])
    np.testing.assert_array_equal(gpu["path"][keep], ref["path"][keep])


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_root_only_and_single_token_vocab(T):
    rng = np.random.default_rng(1)
    p = rng.normal(size=(50, 1, 77)).astype(np.float32)
    gpu, ref = _manual(p, p, np.zeros((50, 1), np.int32), np.full((50, 1), -1, np.int32), 0, T)
    _assert_same(gpu, ref)
    p1 = rng.normal(size=(5, 3, 1)).astype(np.float32)
    par = np.tile(np.array([-1, 0, 1], np.int32), (5, 1))
    gpu, ref = _manual(p1, p1, np.zeros((5, 3), np.int32), par, 2, T)
    _assert_same(gpu, ref)
    assert (gpu["accept_len"] == 2).all()


def test_invalid_trees_and_nonfinite_rows():
    rng = np.random.default_rng(2)
    B, N, V = 6, 5, 40
    p = rng.normal(size=(B, N, V)).astype(np.float32)
    q = rng.normal(size=(B, N, V)).astype(np.float32)
    par = np.tile(np.array([-1, 0, 0, 1, 3], np.int32), (B, 1))
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    par[1, 0] = 0          # root must be -1
    par[2, 3] = 4          # parent after child
    tok[3, 2] = V          # token out of range
    p[4, 0, 5] = np.nan    # non-finite root row
    gpu, ref = _manual(p, q, tok, par, 3, 1.0)
    assert list(gpu["status"][:5]) == [0, 2, 2, 2, 1]
    _assert_same(gpu, ref)
    gpu, ref = _manual(p, q, tok, par, 2, 1.0)   # depth 3 > max_depth 2: all invalid
    assert (gpu["status"] == 2).all() and (gpu["accept_len"] == -1).all()


def test_broadcast_rows_and_deep_chain():
    rng = np.random.default_rng(3)
    N, V, B = 300, 64, 40
    p = rng.normal(0, 0.3, size=(N, V)).astype(np.float32)
    q = (p + rng.normal(0, 0.05, size=(N, V))).astype(np.float32)
    par = np.tile(wl.chain_tree(N), (B, 1))
    tok = np.zeros((B, N), np.int32)
    tok[:, 1:] = rng.integers(0, V, size=(B, N - 1))
    gpu, ref = _manual(p, q, tok, par, N - 1, 1.0, broadcast=True)
    _assert_same(gpu, ref)


def test_max_nodes_tree():
    rng = np.random.default_rng(4)
    N, V, B = binding.SPEC_MAX_NODES, 16, 2
    par = np.stack([wl.random_tree(N, 12, 4, rng) for _ in range(B)])
    p = rng.normal(size=(B, N, V)).astype(np.float32)
    q = rng.normal(size=(B, N, V)).astype(np.float32)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for T in (0.0, 1.0):
        gpu, ref = _manual(p, q, tok, par, 12, T)
        _assert_same(gpu, ref)


def test_chi_squared_first_token_on_gpu():
    """1e6 trees sharing one set of rows: the first emitted token follows filt(p_root)
    when the siblings are drawn i.i.d. from filt(q_root)."""
    from scipy import stats
    rng = np.random.default_rng(5)
    V, T, k, tp = 8, 0.9, 6, 0.95
    parents = np.array([-1, 0, 0, 0, 1, 1, 2], np.int32)
    N = len(parents)
    p = rng.normal(0, 1.0, size=(N, V)).astype(np.float32)
    q = (p + rng.normal(0, 0.8, size=(N, V))).astype(np.float32)
    B = 1_000_000
    Qs = [oracle.filter_row(q[u], T, k, tp)[0] for u in range(N)]
    tok = np.zeros((B, N), np.int32)
    for c in range(1, N):
        tok[:, c] = rng.choice(V, size=B, p=Qs[parents[c]])
    out = binding.verify_tree(_dev_rows(torch.as_tensor(p)), _dev_rows(torch.as_tensor(q)),
                              torch.as_tensor(tok, device=DEV),
                              torch.as_tensor(np.tile(parents, (B, 1)), device=DEV), 2, T, k, tp,
                              seed=2024, batch_broadcast=True, want_alpha=False)
    first = out["tokens"][:, 0].cpu().numpy()
    P0 = oracle.filter_row(p[0], T, k, tp)[0]
    obs = np.bincount(first, minlength=V)
    m = P0 > 0
    assert obs[~m].sum() == 0
    assert stats.chisquare(obs[m], P0[m] * B).pvalue > 1e-3


# --- visited-rows-only schedule (no dense pass) -----------------------------------

@pytest.mark.parametrize("w", [
    W["tree60_b64_v128256"].with_(B=6),
    W["tree26_b256_v152064"].with_(B=6),
    W["tree60_b64_v128256"].with_(B=6, dtype="f32", V=32000),
    W["tree26_b256_v152064"].with_(B=6, temperature=0.0),
    W["tree60_b64_v128256"].with_(B=8, N=40, V=5003, temperature=1.3, top_k=7, top_p=0.8),
    W["tree60_b64_v128256"].with_(B=8, N=33, V=999, dtype="f32", temperature=0.9, top_k=0,
                                  top_p=1.0),
    W["chain_g3_v32"].with_(B=500),
    W["eagle10_v32000"].with_(B=8, temperature=0.0),
], ids=["c3-reduced", "c4-reduced", "c3-f32", "c4-greedy", "ragged-topk-topp", "f32-plain",
        "chain", "eagle10-greedy"])
def test_visited_only_matches_oracle(w):
    _parity(w, seed=31, flags=binding.SPEC_FLAG_VISITED_ONLY)


def test_visited_only_equals_dense_schedule():
    w = W["tree60_b64_v128256"].with_(B=8, V=40000)
    inp = gpu_inputs(w, 5)
    a = run_gpu(w, inp, seed=9)
    b = run_gpu(w, inp, seed=9, flags=binding.SPEC_FLAG_VISITED_ONLY)
    for key in ("accept_len", "tokens", "path", "status"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    np.testing.assert_array_equal(np.isnan(a["alpha"]), np.isnan(b["alpha"]))
    m = ~np.isnan(a["alpha"])
    np.testing.assert_allclose(a["alpha"][m], b["alpha"][m], rtol=1e-5, atol=1e-7)
    # no dense pass: no dense rows read
    assert b["counters"]["dense_rows"] == 0 and a["counters"]["dense_rows"] > 0
