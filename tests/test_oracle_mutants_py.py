"""The pins of the numpy oracles (dynamic tree, draft top-k, accepted-path commit,
per-request verify) must catch plausible mistakes.  Each case plants one mistake in a
copy of the oracle's source on the CPU, loads the copy as a module, and runs the pin
tests of that oracle against it: at least one pin has to fail."""
import importlib
import inspect
import os
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    # dynamic tree (oracle/dyntree.py; pins in tests/test_oracle_dyntree.py)
    "dyntree:value_sum": ("dyntree", "val[i] = np.float32(pv * np.float32(cand_prob[i]))",
                          "val[i] = np.float32(pv + np.float32(cand_prob[i]))"),
    "dyntree:depth_off_by_one": ("dyntree", "dep[i] = 1 if p < 0 else dep[p] + 1",
                                 "dep[i] = 0 if p < 0 else dep[p] + 1"),
    "dyntree:tie_to_deeper": ("dyntree", "key=lambda i: (-float(val[i]), int(dep[i]), i))",
                              "key=lambda i: (-float(val[i]), -int(dep[i]), i))"),
    "dyntree:flatten_by_number": ("dyntree", "flat = sorted(keep, key=lambda i: (int(dep[i]), i))",
                                  "flat = sorted(keep)"),
    "dyntree:parent_position": ("dyntree", "parent[j] = 0 if p < 0 else pos[p]",
                                "parent[j] = 0 if p < 0 else pos[p] - 1"),
    "dyntree:mask_transposed": ("dyntree", "mask[j, a] = 1", "mask[a, j] = 1"),
    "dyntree:expand_ties_higher": ("dyntree",
                                   "key=lambda i: (-float(values[i]), i))",
                                   "key=lambda i: (-float(values[i]), -i))"),
    # draft top-k (oracle/draft.py; pins in tests/test_oracle_draft.py)
    "draft:ties_higher": ("draft", "key=lambda i: (-z[i], i))[:k]", "key=lambda i: (-z[i], -i))[:k]"),
    "draft:temperature_dropped": ("draft", "w = np.exp((z - m) / temperature)", "w = np.exp(z - m)"),
    "draft:normaliser_over_kept": ("draft", "probs[r, :len(order)] = w[order] / s",
                                   "probs[r, :len(order)] = w[order] / w[order].sum()"),
    "draft:nan_kept": ("draft", "if np.isnan(z).any() or m == np.inf or m == -np.inf:",
                       "if m == np.inf or m == -np.inf:"),
    # accepted-path commit (oracle/commit.py; pins in tests/test_oracle_commit.py)
    "commit:reverse_order": ("commit", "for k in range(1, a + 1):", "for k in range(a, 0, -1):"),
    "commit:destination_off_by_one": ("commit", "dst = base + k", "dst = base + k - 1"),
    "commit:failed_tree_moved": ("commit", "a = int(accept_len[b])", "a = abs(int(accept_len[b]))"),
    # per-request verify (oracle/__init__.py; pins in tests/test_oracle_per_request.py)
    "per_request:batch_index_zero": ("__init__", "offset, batch_index=b))", "offset, batch_index=0))"),
    "per_request:invalid_accepted": ("__init__",
                                     "if not (np.isfinite(T) and T >= 0.0) or not (p > 0.0) or k < 0:",
                                     "if False:"),
}

PINS = {
    "dyntree": "test_oracle_dyntree",
    "draft": "test_oracle_draft",
    "commit": "test_oracle_commit",
    "__init__": "test_oracle_per_request",
}


def _mutant(module: str, find: str, repl: str) -> types.ModuleType:
    name = "oracle" if module == "__init__" else f"oracle.{module}"
    path = os.path.join(ROOT, "oracle", f"{module}.py")
    src = open(path).read()
    assert src.count(find) == 1, f"mutation anchor not found once in {path}: {find!r}"
    mod = types.ModuleType(name + "_mutant")
    mod.__file__ = path  # the C oracle loader locates its library relative to this
    exec(compile(src.replace(find, repl), path, "exec"), mod.__dict__)
    return mod


def _run_pins(pin_module, attr: str, mutant) -> list:
    """Run every test function of the pin module with its oracle reference swapped;
    returns the names of those that failed."""
    failed = []
    saved = getattr(pin_module, attr)
    setattr(pin_module, attr, mutant)
    try:
        for name, fn in inspect.getmembers(pin_module, inspect.isfunction):
            if not name.startswith("test_"):
                continue
            params = inspect.signature(fn).parameters
            marks = getattr(fn, "pytestmark", [])
            cases = [()]
            for m in marks:
                if m.name == "parametrize":
                    argnames = [a.strip() for a in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
                    cases = [tuple(v) if len(argnames) > 1 else (v,) for v in m.args[1]]
            for case in cases:
                kwargs = dict(zip(list(params), case)) if case else {}
                try:
                    fn(**kwargs)
                except Exception:  # a failing pin (assertion, or the mutant breaking outright)
                    failed.append(name)
                    break
    finally:
        setattr(pin_module, attr, saved)
    return failed


@pytest.mark.parametrize("case", sorted(MUTANTS))
def test_pins_catch_planted_mistake(case):
    module, find, repl = MUTANTS[case]
    mutant = _mutant(module, find, repl)
    pins = importlib.import_module(PINS[module])
    if module == "__init__":
        attr = "oracle"
    elif module == "draft":
        # the draft pins import the function itself
        mutant_fn = mutant.draft_topk
        failed = []
        saved = pins.draft_topk
        pins.draft_topk = mutant_fn
        try:
            for name, fn in inspect.getmembers(pins, inspect.isfunction):
                if name.startswith("test_"):
                    try:
                        fn()
                    except Exception:
                        failed.append(name)
        finally:
            pins.draft_topk = saved
        assert failed, f"mutant {case} passed every pin"
        return
    elif module == "commit":
        mutant_fn = mutant.commit_accepted_path
        failed = []
        saved = pins.commit_accepted_path
        pins.commit_accepted_path = mutant_fn
        try:
            for name, fn in inspect.getmembers(pins, inspect.isfunction):
                if name.startswith("test_"):
                    try:
                        fn()
                    except Exception:
                        failed.append(name)
        finally:
            pins.commit_accepted_path = saved
        assert failed, f"mutant {case} passed every pin"
        return
    else:
        attr = module
    failed = _run_pins(pins, attr, mutant)
    assert failed, f"mutant {case} passed every pin"
