"""Each planted mistake in the oracle is caught by at least one pin (CPU only).

The oracle's C source carries a handful of deliberate mistakes behind ``ORACLE_MUTATION``
(a dropped scale, an off-by-one causal mask, a dropped max in the LSE, the wrong operand in P.V,
a dropped normalisation, a shifted value index, an ignored value descale, a wrong e4m3 exponent
bias, a base-2 LSE, two block-descale indexing slips,
four backward slips).  The default build has none.
"""
import os

import pytest

from oracle import oracle as orc_mod
from tests.oracle_pins import PINS

MUTATIONS = {
    1: "scale dropped",
    2: "causal diagonal excluded",
    3: "max dropped from LSE",
    4: "K used in place of V",
    5: "normalisation dropped",
    6: "value row index shifted",
    7: "value descale ignored",
    8: "e4m3 exponent bias 8",
    9: "LSE in base 2",
    10: "query block descale read from the first head",
    11: "key block descale applied to the values",
    12: "backward: scale dropped from dK",
    13: "backward: D dropped",
    14: "backward: P factor of dS dropped",
    15: "backward: dS used in place of P for dV",
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS), ids=lambda m: MUTATIONS[m])
def test_pins_catch_planted_mistake(tmp_path, mutation):
    path = orc_mod.build(os.path.join(str(tmp_path), f"liboracle_m{mutation}.so"), mutation)
    orc = orc_mod.Oracle(path)
    assert orc.mutation == mutation
    caught = []
    for p in PINS:
        try:
            p(orc)
        except (AssertionError, RuntimeError, FloatingPointError):
            caught.append(p.__name__)
    assert caught, f"no pin caught mutation {mutation} ({MUTATIONS[mutation]})"
