"""The checked build (device-side index checks, compiled with -DSPEC_CHECK) runs the
edge cases of tests/checked_cases.py -- small and ragged vocabularies, one warp per
tree, the window and top-k routes at eight CTAs per tree, the visited-rows-only
schedule, the exact selection, every logit tied -- with results equal to the
oracle's and no index caught out of range."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_edge_cases():
    from speculative_decoding_tree_spec_gb300 import build

    path = build.build(check=True)
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests"),
                                         env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_cases.py"), path],
                       capture_output=True, text=True, env=env, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["words"] == [0, 0], out
    compared = {k: v for k, v in out.items() if k != "words"}
    assert all(v > 0 for v in compared.values()), compared
