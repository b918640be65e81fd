"""Host-side argument checks of the C ABI, called with addresses that are never
dereferenced.  Every call here must return during host validation, before anything
is launched; this module is therefore only ever run in a child process that sees no
GPU (CUDA_VISIBLE_DEVICES=""), so that a validation regression fails the test with a
CUDA error instead of launching a kernel on a bogus address.  Run as a script it
prints the return code of every case as JSON."""
import json
import sys

from speculative_decoding_tree_spec_gb300 import binding

FAKE = 1 << 20  # a 16- and 256-byte aligned address that the host never dereferences

VERIFY_CASES = [
    (dict(B=0), 0),
    (dict(dtype=7), -2),
    (dict(N=0), -1),
    (dict(V=0), -1),
    (dict(B=-1), -1),
    (dict(max_depth=-1), -1),
    (dict(N=5000), -6),
    (dict(V=(1 << 21) + 8, row_pitch=(1 << 21) + 8), -6),
    (dict(params=("p", -1.0)), -1),
    (dict(params=("p", float("nan"))), -1),
    (dict(params=("p", float("inf"))), -1),
    (dict(params=("p", 0.7, 0, 0.0)), -1),
    (dict(params=("p", 0.7, 0, float("nan"))), -1),
    (dict(params=("p", 0.7, 0, 0.9, 8)), -1),
    (dict(logits_p=None), -1),
    (dict(logits_q=None), -1),
    (dict(draft_tokens=None), -1),
    (dict(parent_idx=None), -1),
    (dict(out_accept_len=None), -1),
    (dict(out_tokens=None), -1),
    (dict(out_path=None), -1),
    (dict(workspace=None), -1),
    (dict(row_pitch=999), -1),
    (dict(batch_stride=-8), -1),
    (dict(logits_p=FAKE + 2), -3),
    (dict(logits_q=FAKE + 8), -3),
    (dict(row_pitch=1001, batch_stride=8008), -3),
    (dict(batch_stride=8004), -3),
    (dict(ws_bytes=1024), -4),
    (dict(workspace=FAKE + 128), -4),
    (dict(B=0, logits_q=None, params=("p", 0.0)), 0),   # greedy may omit q
]


def _params(spec):
    if spec is None:
        return binding.params(0.7, 0, 0.9)
    _, *a = spec
    if len(a) == 4:
        return binding.params(a[0], a[1], a[2], flags=a[3])
    return binding.params(*a)


def _verify(L, **kw):
    a = dict(logits_p=FAKE, logits_q=FAKE, dtype=1, B=4, N=8, V=1000, row_pitch=1000,
             batch_stride=8000, draft_tokens=FAKE, parent_idx=FAKE, max_depth=3, params=None,
             seed=1, offset=0, out_accept_len=FAKE, out_tokens=FAKE, out_path=FAKE,
             out_alpha=None, out_status=None, out_counters=None, workspace=FAKE,
             ws_bytes=1 << 40, stream=None)
    a.update(kw)
    return L.spec_verify_tree(a["logits_p"], a["logits_q"], a["dtype"], a["B"], a["N"], a["V"],
                              a["row_pitch"], a["batch_stride"], a["draft_tokens"],
                              a["parent_idx"], a["max_depth"], _params(a["params"]), a["seed"],
                              a["offset"], a["out_accept_len"], a["out_tokens"], a["out_path"],
                              a["out_alpha"], a["out_status"], a["out_counters"], a["workspace"],
                              a["ws_bytes"], a["stream"])


def run_all():
    L = binding.lib()
    out = {}
    out["verify"] = [_verify(L, **kw) for kw, _ in VERIFY_CASES]

    f = L.spec_filter_rows
    p = binding.params(1.0, 50, 0.9)
    out["filter_rows"] = [
        f(FAKE, 1, 0, 100, 104, p, FAKE, None), f(FAKE, 1, -1, 100, 104, p, FAKE, None),
        f(FAKE, 3, 4, 100, 104, p, FAKE, None), f(None, 1, 4, 100, 104, p, FAKE, None),
        f(FAKE, 1, 4, 100, 104, p, None, None), f(FAKE, 1, 4, 100, 99, p, FAKE, None),
        f(FAKE, 1, 4, 100, 100, p, FAKE, None),
        f(FAKE, 1, 4, 100, 104, binding.params(0.5, 0, -0.1), FAKE, None)]

    g = L.spec_philox_words
    out["philox"] = [g(1, 0, FAKE, FAKE, 0, FAKE, None), g(1, 0, FAKE, FAKE, -1, FAKE, None),
                     g(1, 0, None, FAKE, 4, FAKE, None), g(1, 0, FAKE, FAKE, 4, FAKE + 4, None)]

    t = L.spec_tree_build
    args, outs = [FAKE] * 4, [FAKE] * 7
    out["tree_build"] = [
        t(*args, 0, 10, 5, *outs, None), t(*args, -1, 10, 5, *outs, None),
        t(*args, 1, 0, 1, *outs, None), t(*args, 1, 4097, 5, *outs, None),
        t(*args, 1, 10, 0, *outs, None), t(*args, 1, 10, 11, *outs, None),
        t(*args, 1, 4096, 4096, *outs, None), t(None, FAKE, FAKE, FAKE, 1, 10, 5, *outs, None),
        t(*args, 1, 10, 5, FAKE, FAKE, FAKE, FAKE, None, FAKE, None)]

    e = L.spec_tree_expand_topk
    out["tree_expand"] = [
        e(FAKE, FAKE, 0, 10, 0, 10, 3, FAKE, None), e(FAKE, FAKE, 1, 10, 5, 4, 3, FAKE, None),
        e(FAKE, FAKE, 1, 10, 0, 11, 3, FAKE, None), e(FAKE, FAKE, 1, 10, -1, 5, 3, FAKE, None),
        e(FAKE, FAKE, 1, 10, 0, 10, 0, FAKE, None), e(FAKE, None, 1, 10, 0, 10, 3, FAKE, None),
        e(FAKE, FAKE, 1, 10, 0, 10, 3, None, None)]

    r = L.spec_verify_tree_per_request
    pr = lambda T=FAKE, q=FAKE, B=2: (7, FAKE, q, 1, B, 4, 1000, 1000, 4000, FAKE, FAKE, 3, T,
                                      None, None, 0, 0, 0, FAKE, FAKE, FAKE, None, None, None,
                                      FAKE, 1 << 40, None)
    out["per_request"] = [r(*pr(B=0)), r(*pr(T=None)), r(*pr(q=None))]

    d = L.spec_draft_topk
    out["draft_topk"] = [
        d(FAKE, 1, 0, 100, 104, 10, 1.0, FAKE, FAKE, None, None),
        d(FAKE, 1, 4, 100, 104, 0, 1.0, FAKE, FAKE, None, None),
        d(FAKE, 1, 4, 100, 104, 33, 1.0, FAKE, FAKE, None, None),
        d(FAKE, 1, 4, 8, 8, 9, 1.0, FAKE, FAKE, None, None),
        d(FAKE, 1, 4, 100, 104, 10, 0.0, FAKE, FAKE, None, None),
        d(FAKE, 1, 4, 100, 104, 10, float("nan"), FAKE, FAKE, None, None),
        d(FAKE, 1, 4, 100, 99, 10, 1.0, FAKE, FAKE, None, None),
        d(FAKE, 1, 4, 100, 100, 10, 1.0, FAKE, FAKE, None, None),
        d(FAKE, 3, 4, 100, 104, 10, 1.0, FAKE, FAKE, None, None),
        d(None, 1, 4, 100, 104, 10, 1.0, FAKE, FAKE, None, None)]

    fz = L.spec_draft_topk_fused_lmhead
    ws = L.spec_draft_fused_workspace_size(4, 1000, 10)
    ok = lambda **kw: dict(dict(feat=FAKE, w=FAKE, d=64, R=4, V=1000, k=10, T=1.0, lg=None,
                                pitch=0, tok=FAKE, pr=FAKE, st=None, ws=FAKE, wsb=ws), **kw)
    call = lambda a: fz(a["feat"], a["w"], a["d"], a["R"], a["V"], a["k"], a["T"], a["lg"],
                        a["pitch"], a["tok"], a["pr"], a["st"], a["ws"], a["wsb"], None)
    out["draft_fused"] = [
        call(ok(R=0)), call(ok(k=0)), call(ok(k=33)), call(ok(T=0.0)), call(ok(d=60)),
        call(ok(feat=FAKE + 8)), call(ok(lg=FAKE, pitch=999)), call(ok(lg=FAKE, pitch=1001)),
        call(ok(wsb=ws - 1)), call(ok(ws=FAKE + 128)), call(ok(w=None))]

    # the no-allocation entry point refuses trees above its static scratch before it
    # touches the device
    out["noalloc_too_large"] = L.spec_verify_tree_noalloc(
        FAKE, FAKE, binding.SPEC_BF16, 5000, 60, 1000, 1000, 60000, FAKE, FAKE, 3,
        binding.params(0.7, 0, 0.9), 1, 0, FAKE, FAKE, FAKE, None, None, None, None)
    return out


if __name__ == "__main__":
    json.dump(run_all(), sys.stdout)
