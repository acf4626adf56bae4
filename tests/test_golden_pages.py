"""Host arithmetic pinned to the worked numbers the pages print
(tests/golden/pages_worked_numbers.json, each case with its citation)."""
import json
import math
import os

import pytest

from memory_bound_decode_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_worked_numbers.json")
CASES = json.load(open(GOLDEN))["cases"]


def _close(got, want, rel):
    if isinstance(want, dict):
        return all(_close(got[k], v, rel) for k, v in want.items())
    if isinstance(want, list):
        return len(got) == len(want) and all(_close(g, w, rel) for g, w in zip(got, want))
    if rel == 0.0:
        return got == want
    return math.isclose(got, want, rel_tol=rel)


@pytest.mark.parametrize("case", CASES, ids=[c["id"] for c in CASES])
def test_page_number(case):
    assert case["cite"]
    got = getattr(roofline, case["fn"])(**case["args"])
    assert _close(got, case["expected"], case["rel"]), (case["id"], got, case["expected"])


def test_bytes_formula_configs():
    # N*K*2 + B*K*2 + B*N*4 for the decode projections of the workloads
    assert roofline.algorithmic_bytes(1024, 4096) == 8_400_896
    assert roofline.algorithmic_bytes(4096, 14336) == 117_485_568
    assert roofline.algorithmic_bytes(6144, 4096) == 50_364_416
    assert roofline.algorithmic_bytes(28672, 4096) == 235_003_904
    layer = (roofline.algorithmic_bytes(6144, 4096) + roofline.algorithmic_bytes(4096, 4096)
             + roofline.algorithmic_bytes(28672, 4096) + roofline.algorithmic_bytes(4096, 14336))
    assert layer == 436_432_896
    assert 32 * layer + roofline.algorithmic_bytes(128256, 4096) == 15_017_047_040
