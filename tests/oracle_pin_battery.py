"""Runs every oracle pin (the test functions of tests/test_oracle_*.py, each
parametrisation expanded) against the oracle package found first on
sys.path, and prints a JSON summary: {"ran": n, "failed": [names],
"skipped": n, "oracle": path}.

Used by tests/test_oracle_mutations.py, which points it at copies of the
oracle with one planted mistake each:

    python tests/oracle_pin_battery.py <directory holding the oracle copy>
"""
import importlib
import itertools
import json
import os
import sys


def _param_sets(fn):
    """All keyword-argument sets of a test function's parametrize marks."""
    axes = []
    for mark in getattr(fn, "pytestmark", []):
        if mark.name != "parametrize":
            continue
        names, values = mark.args[0], mark.args[1]
        if isinstance(names, str):
            names = [n.strip() for n in names.split(",") if n.strip()]
        rows = []
        for v in values:
            v = getattr(v, "values", v)  # pytest.param(...)
            if len(names) == 1 and not (isinstance(v, tuple) and len(v) == 1):
                v = (v,)
            rows.append(dict(zip(names, v)))
        axes.append(rows)
    if not axes:
        return [{}]
    return [dict(kv for d in combo for kv in d.items()) for combo in itertools.product(*axes)]


def run(oracle_dir):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path[:0] = [oracle_dir, root]
    import oracle  # the copy under oracle_dir
    import pytest
    assert os.path.dirname(os.path.dirname(oracle.__file__)) == os.path.abspath(oracle_dir)
    ran, failed, skipped = 0, [], 0
    for modname in ("test_oracle_formats", "test_oracle_cache_write", "test_oracle_attention",
                    "test_oracle_mla"):
        mod = importlib.import_module(f"tests.{modname}")
        for name, fn in sorted(vars(mod).items()):
            if not name.startswith("test_") or not callable(fn):
                continue
            for kw in _param_sets(fn):
                ran += 1
                try:
                    fn(**kw)
                except pytest.skip.Exception:
                    skipped += 1
                except Exception:  # an assertion, an oracle error, a wrong shape ...
                    failed.append(f"{modname}.{name}{kw if kw else ''}")
    return {"ran": ran, "failed": failed, "skipped": skipped, "oracle": oracle.__file__}


if __name__ == "__main__":
    print(json.dumps(run(sys.argv[1])))
