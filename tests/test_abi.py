"""The C-ABI library loads, exports every function include/*.h declares, and
rejects bad arguments on the host before launching anything.  CPU only.  The calls
that pass never-dereferenced addresses run in a child process that sees no GPU
(tests/host_validation_cases.py), so a regression in the host checks shows up as a
wrong return code there and can never launch a kernel on such an address."""
import ctypes
import glob
import json
import os
import re
import subprocess
import sys

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



import host_validation_cases as hv  # noqa: E402  (the table only; it is run in a child)


@pytest.fixture(scope="module")
def codes(L):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    here = os.path.dirname(os.path.abspath(__file__))
    env["PYTHONPATH"] = os.pathsep.join([ROOT, here, env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, os.path.join(here, "host_validation_cases.py")],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr
    return json.loads(r.stdout)


@pytest.mark.parametrize("i", range(len(hv.VERIFY_CASES)),
                         ids=[",".join(sorted(kw)) for kw, _ in hv.VERIFY_CASES])
def test_host_validation(codes, i):
    assert codes["verify"][i] == hv.VERIFY_CASES[i][1], hv.VERIFY_CASES[i]


def test_filter_rows_validation(codes):
    assert codes["filter_rows"] == [0, -1, -2, -1, -1, -1, -3, -1]


def test_philox_validation(codes):
    assert codes["philox"] == [0, -1, -1, -3]


def test_tree_build_validation(codes):
    # no trees (nothing launched), B < 0, no candidates, above the candidate limit, keeps
    # nothing, m > n, m + 1 nodes above the limit, null inputs, null mask
    assert codes["tree_build"] == [0, -1, -1, -1, -1, -1, -1, -1, -1]


def test_tree_expand_validation(codes):
    # no trees, empty-backwards range, range past n, negative start, k = 0, null probs,
    # null output
    assert codes["tree_expand"] == [0, -1, -1, -1, -1, -1, -1]


def test_per_request_validation(codes):
    # no trees (nothing launched); the temperatures are required; so are the draft logits
    assert codes["per_request"] == [0, -1, -1]


def test_draft_topk_validation(codes):
    # no rows, k = 0, k above 32, k above V, T = 0, T NaN, pitch < V, 200-byte pitch,
    # dtype, null logits
    assert codes["draft_topk"] == [0, -1, -1, -1, -1, -1, -1, -3, -2, -1]


def test_draft_fused_validation(L, codes):
    ws = L.spec_draft_fused_workspace_size(4, 1000, 10)
    assert ws > 0 and L.spec_draft_fused_workspace_size(4, 1000, 33) == 0
    # no rows, k = 0, k = 33, T = 0, d not a multiple of 8, misaligned features, pitch < V,
    # odd pitch, workspace too small, misaligned workspace, null weight
    assert codes["draft_fused"] == [0, -1, -1, -1, -3, -3, -1, -3, -4, -4, -1]


def test_noalloc_rejects_trees_above_the_static_limit(L, codes):
    assert codes["noalloc_too_large"] == -6
    assert int(L.spec_verify_workspace_size(5000, 60, 1000, binding.SPEC_BF16)) > \
        binding.SPEC_STATIC_WORKSPACE_BYTES
