"""The C-ABI library loads, exports every function include/*.h declares, and
rejects bad arguments on the host before launching anything.  CPU only: no call
here reaches the GPU (every case returns during host-side validation)."""
import ctypes
import glob
import os
import re

import pytest

import __graft_entry__
from speculative_decoding_tree_spec_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return binding.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for must in ("spec_verify_tree", "spec_verify_workspace_size", "spec_filter_rows",
                 "spec_philox_words", "spec_error_string"):
        assert must in names


@pytest.mark.parametrize("name", _declared_functions())
def test_library_exports_declared_symbol(L, name):
    assert hasattr(L, name), f"{name} declared in include/ but not exported"


def test_struct_sizes_match_header():
    assert ctypes.sizeof(binding.SamplingParams) == 16
    assert ctypes.sizeof(binding.RowStats) == 32
    assert ctypes.sizeof(binding.Counters) == 64


def test_error_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6, 17):
        s = L.spec_error_string(code)
        assert s and len(s) > 3


def test_workspace_size(L):
    ws = L.spec_verify_workspace_size(64, 60, 128256, 1)
    assert ws >= 64 * 60 * 32 * 2
    assert ws % 256 == 0
    assert L.spec_verify_workspace_size(64, 60, 128256, 0) == ws
    assert L.spec_verify_workspace_size(-1, 60, 100, 1) == 0
    assert L.spec_verify_workspace_size(4, 0, 100, 1) == 0
    assert L.spec_verify_workspace_size(4, 5000, 100, 1) == 0
    assert L.spec_verify_workspace_size(4, 5, 1 << 22, 1) == 0
    assert L.spec_verify_workspace_size(4, 5, 100, 9) == 0


FAKE = 1 << 20  # a 16- and 256-byte aligned address that the host never dereferences


def _call(L, **kw):
    a = dict(logits_p=FAKE, logits_q=FAKE, dtype=1, B=4, N=8, V=1000, row_pitch=1000,
             batch_stride=8000, draft_tokens=FAKE, parent_idx=FAKE, max_depth=3,
             params=binding.params(0.7, 0, 0.9), seed=1, offset=0, out_accept_len=FAKE,
             out_tokens=FAKE, out_path=FAKE, out_alpha=None, out_status=None,
             out_counters=None, workspace=FAKE, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return L.spec_verify_tree(a["logits_p"], a["logits_q"], a["dtype"], a["B"], a["N"], a["V"],
                              a["row_pitch"], a["batch_stride"], a["draft_tokens"],
                              a["parent_idx"], a["max_depth"], a["params"], a["seed"],
                              a["offset"], a["out_accept_len"], a["out_tokens"], a["out_path"],
                              a["out_alpha"], a["out_status"], a["out_counters"], a["workspace"],
                              a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 0),
    (dict(dtype=7), -2),
    (dict(N=0), -1),
    (dict(V=0), -1),
    (dict(B=-1), -1),
    (dict(max_depth=-1), -1),
    (dict(N=5000), -6),
    (dict(V=(1 << 21) + 8, row_pitch=(1 << 21) + 8), -6),
    (dict(params=binding.params(-1.0)), -1),
    (dict(params=binding.params(float("nan"))), -1),
    (dict(params=binding.params(float("inf"))), -1),
    (dict(params=binding.params(0.7, 0, 0.0)), -1),
    (dict(params=binding.params(0.7, 0, float("nan"))), -1),
    (dict(params=binding.params(0.7, 0, 0.9, flags=8)), -1),
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
])
def test_host_validation(L, kw, code):
    assert _call(L, **kw) == code


def test_greedy_may_omit_draft_logits(L):
    # q is never read at temperature 0: a NULL q passes validation (B=0: nothing launched)
    assert _call(L, B=0, logits_q=None, params=binding.params(0.0)) == 0


def test_filter_rows_validation(L):
    f = L.spec_filter_rows
    p = binding.params(1.0, 50, 0.9)
    assert f(FAKE, 1, 0, 100, 104, p, FAKE, None) == 0
    assert f(FAKE, 1, -1, 100, 104, p, FAKE, None) == -1
    assert f(FAKE, 3, 4, 100, 104, p, FAKE, None) == -2
    assert f(None, 1, 4, 100, 104, p, FAKE, None) == -1
    assert f(FAKE, 1, 4, 100, 104, p, None, None) == -1
    assert f(FAKE, 1, 4, 100, 99, p, FAKE, None) == -1
    assert f(FAKE, 1, 4, 100, 100, p, FAKE, None) == -3   # 200-byte pitch
    assert f(FAKE, 1, 4, 100, 104, binding.params(0.5, 0, -0.1), FAKE, None) == -1


def test_philox_validation(L):
    assert L.spec_philox_words(1, 0, FAKE, FAKE, 0, FAKE, None) == 0
    assert L.spec_philox_words(1, 0, FAKE, FAKE, -1, FAKE, None) == -1
    assert L.spec_philox_words(1, 0, None, FAKE, 4, FAKE, None) == -1
    assert L.spec_philox_words(1, 0, FAKE, FAKE, 4, FAKE + 4, None) == -3


def test_tree_build_validation(L):
    f = L.spec_tree_build
    args = [FAKE] * 4
    outs = [FAKE] * 7
    assert f(*args, 0, 10, 5, *outs, None) == 0            # no trees: nothing launched
    assert f(*args, -1, 10, 5, *outs, None) == -1
    assert f(*args, 1, 0, 1, *outs, None) == -1            # no candidates
    assert f(*args, 1, 4097, 5, *outs, None) == -1         # above the candidate limit
    assert f(*args, 1, 10, 0, *outs, None) == -1           # keeps nothing
    assert f(*args, 1, 10, 11, *outs, None) == -1          # m > n
    assert f(*args, 1, 4096, 4096, *outs, None) == -1      # m + 1 nodes above the limit
    assert f(None, FAKE, FAKE, FAKE, 1, 10, 5, *outs, None) == -1
    assert f(*args, 1, 10, 5, FAKE, FAKE, FAKE, FAKE, None, FAKE, None) == -1


def test_tree_expand_validation(L):
    f = L.spec_tree_expand_topk
    assert f(FAKE, FAKE, 0, 10, 0, 10, 3, FAKE, None) == 0
    assert f(FAKE, FAKE, 1, 10, 5, 4, 3, FAKE, None) == -1    # empty-backwards range
    assert f(FAKE, FAKE, 1, 10, 0, 11, 3, FAKE, None) == -1   # range past n
    assert f(FAKE, FAKE, 1, 10, -1, 5, 3, FAKE, None) == -1
    assert f(FAKE, FAKE, 1, 10, 0, 10, 0, FAKE, None) == -1   # k = 0
    assert f(FAKE, None, 1, 10, 0, 10, 3, FAKE, None) == -1
    assert f(FAKE, FAKE, 1, 10, 0, 10, 3, None, None) == -1


def test_per_request_validation(L):
    f = L.spec_verify_tree_per_request
    args = lambda T=FAKE, q=FAKE, B=2: (7, FAKE, q, 1, B, 4, 1000, 1000, 4000, FAKE, FAKE, 3, T,
                                        None, None, 0, 0, 0, FAKE, FAKE, FAKE, None, None, None,
                                        FAKE, 1 << 20, None)
    assert f(*args(B=0)) == 0                     # no trees: nothing launched
    assert f(*args(T=None)) == -1                 # the temperatures are required
    assert f(*args(q=None)) == -1                 # the draft logits are required


def test_draft_topk_validation(L):
    f = L.spec_draft_topk
    assert f(FAKE, 1, 0, 100, 104, 10, 1.0, FAKE, FAKE, None, None) == 0   # no rows
    assert f(FAKE, 1, 4, 100, 104, 0, 1.0, FAKE, FAKE, None, None) == -1   # k = 0
    assert f(FAKE, 1, 4, 100, 104, 33, 1.0, FAKE, FAKE, None, None) == -1  # k above 32
    assert f(FAKE, 1, 4, 8, 8, 9, 1.0, FAKE, FAKE, None, None) == -1       # k above V
    assert f(FAKE, 1, 4, 100, 104, 10, 0.0, FAKE, FAKE, None, None) == -1  # T = 0
    assert f(FAKE, 1, 4, 100, 104, 10, float("nan"), FAKE, FAKE, None, None) == -1
    assert f(FAKE, 1, 4, 100, 99, 10, 1.0, FAKE, FAKE, None, None) == -1   # pitch < V
    assert f(FAKE, 1, 4, 100, 100, 10, 1.0, FAKE, FAKE, None, None) == -3  # 200-byte pitch
    assert f(FAKE, 3, 4, 100, 104, 10, 1.0, FAKE, FAKE, None, None) == -2  # dtype
    assert f(None, 1, 4, 100, 104, 10, 1.0, FAKE, FAKE, None, None) == -1


def test_draft_fused_validation(L):
    f = L.spec_draft_topk_fused_lmhead
    ws = L.spec_draft_fused_workspace_size(4, 1000, 10)
    assert ws > 0 and L.spec_draft_fused_workspace_size(4, 1000, 33) == 0
    ok = lambda **kw: dict(dict(feat=FAKE, w=FAKE, d=64, R=4, V=1000, k=10, T=1.0, lg=None, pitch=0,
                                tok=FAKE, pr=FAKE, st=None, ws=FAKE, wsb=ws), **kw)
    call = lambda a: f(a["feat"], a["w"], a["d"], a["R"], a["V"], a["k"], a["T"], a["lg"],
                       a["pitch"], a["tok"], a["pr"], a["st"], a["ws"], a["wsb"], None)
    assert call(ok(R=0)) == 0
    assert call(ok(k=0)) == -1
    assert call(ok(k=33)) == -1
    assert call(ok(T=0.0)) == -1
    assert call(ok(d=60)) == -3          # rows of the tensor maps must be 16-byte multiples
    assert call(ok(feat=FAKE + 8)) == -3
    assert call(ok(lg=FAKE, pitch=999)) == -1
    assert call(ok(lg=FAKE, pitch=1001)) == -3
    assert call(ok(wsb=ws - 1)) == -4
    assert call(ok(ws=FAKE + 128)) == -4
    assert call(ok(w=None)) == -1
