"""The oracles against tests/golden/oracle_tiny.json, their own outputs on tiny
seeded inputs written by tests/golden/make_golden.py (which calls only
oracle/ and the shared input generator). The inputs must come back
bit-identical (the generator is deterministic); the outputs within 1e-12
relative (the fp64 oracle's summation order is fixed, so only the compiler's
contraction of multiply-adds can move a last bit). A change of an oracle's
arithmetic fails here until the fixture is regenerated on purpose.
"""
import importlib.util
import json
import os

import numpy as np
import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def golden():
    import __graft_entry__  # noqa: F401  (puts the repo root on sys.path)

    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(HERE, "oracle_tiny.json")) as f:
        return json.load(f), mod.cases()


def _walk(stored, fresh, path=""):
    assert set(stored) == set(fresh), path
    for k in stored:
        a, b = stored[k], fresh[k]
        p = f"{path}/{k}"
        if isinstance(a, dict):
            _walk(a, b, p)
        elif a is None or isinstance(a, (int, float)):
            assert a == b, p
        else:
            a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
            assert a.shape == b.shape, p
            if "/inputs/" in p + "/" or k in ("z", "ln_w", "ln_b", "r_k"):
                assert np.array_equal(a, b), f"{p}: input changed"
            else:
                np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-15, err_msg=p)


@pytest.mark.parametrize("case", ["wkv7", "wkv7_logit", "epilogue", "rwkv8"])
def test_oracle_matches_its_fixture(golden, case):
    stored, fresh = golden
    _walk(stored[case], fresh[case], case)
