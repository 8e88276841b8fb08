"""The fp64 oracle against brute force, closed forms and invariants (CPU)."""
import json
import math
import os

import pytest

import oracle
from tests import oracle_pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "result_table.json")


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_bad_arguments_are_rejected(orc):
    from gqa_flash_attention_causal_gb300.inputs import normal_bf16
    q = normal_bf16((4, 32, 128), 1)
    k = normal_bf16((4, 8, 128), 2)
    with pytest.raises(ValueError):
        orc.prefill_rows(q, k, k, [4])          # row out of range
    with pytest.raises(ValueError):
        orc.prefill(q, normal_bf16((4, 5, 128), 3), normal_bf16((4, 5, 128), 3))


def test_result_table_fixture_is_consistent():
    """The transcribed table agrees with the page's own speedup column
    (FA2 ms / ours ms, printed to 2 decimals) and its min/max/average claim."""
    t = json.load(open(GOLDEN))
    ratios = []
    for wl, n, fa2, ours, _start, final in t["rows"]:
        assert wl in ("prefill", "decode") and n & (n - 1) == 0
        r = fa2 / ours
        # decode times carry 3 decimals, so the quotient is only good to ~5%
        tol = 0.006 if wl == "prefill" else 0.05 * final
        assert abs(r - final) <= tol, (wl, n, r, final)
        ratios.append(final)
    s = t["summary"]
    assert min(ratios) == s["speedup_min"] and max(ratios) == s["speedup_max"]
    # the page's "average 1.17x" is not the arithmetic mean of its own column
    # (1.185); it matches the geometric mean (1.176) to within rounding
    geo = math.exp(sum(math.log(r) for r in ratios) / len(ratios))
    assert abs(geo - s["speedup_mean"]) < 0.01
