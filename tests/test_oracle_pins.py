"""The fp64 oracle against its pins (CPU only)."""
import os

import numpy as np
import pytest

from oracle import oracle as orc_mod
from tests.oracle_pins import PINS


@pytest.fixture(scope="module")
def orc():
    return orc_mod.get()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


def test_unmutated_build(orc):
    assert orc.mutation == 0


def test_bad_arguments_are_rejected(orc):
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(RuntimeError):
        orc.attention_fwd(q, q, q, 1.0, rows=[4])
    with pytest.raises(ValueError):
        orc.attention_fwd(q, q[:, :, :3], q, 1.0)
    with pytest.raises(TypeError):
        orc.attention_fwd(q.astype(np.float32), q, q, 1.0)


def test_bf16_inputs_match_f64_on_decoded_values(orc):
    """The bf16 path decodes first, then runs the same evaluation as f64 inputs."""
    from workloads import random_inputs
    inp = random_inputs(1, 2, 50, 16, "bf16", seed=3)
    o, lse = orc_mod.attention_fwd_inputs(inp, 0.25, True)
    q, k, v = (getattr(inp, n).to(dtype=__import__("torch").float64).numpy() for n in "qkv")
    o2, l2 = orc.attention_fwd(q, k, v, 0.25, True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, l2)


def test_threads_do_not_change_results(orc):
    rng = np.random.default_rng(5)
    q, k, v = rng.standard_normal((3, 2, 3, 130, 8))
    a = orc.attention_fwd(q, k, v, 0.3, True, threads=1)
    b = orc.attention_fwd(q, k, v, 0.3, True, threads=max(2, os.cpu_count() or 2))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_backward_bf16_inputs_match_f64_on_decoded_values(orc):
    from workloads import random_bwd_inputs

    inp = random_bwd_inputs(1, 2, 40, 16, seed=5)
    g16 = orc.attention_bwd(*(inp.raw(n) for n in ("q", "k", "v", "do")), 0.25, True, "bf16")
    g64 = orc.attention_bwd(*(getattr(inp, n).double().numpy() for n in ("q", "k", "v", "do")),
                            0.25, True)
    for key in ("dq", "dk", "dv", "o", "lse", "delta"):
        np.testing.assert_array_equal(g16[key], g64[key])


def test_backward_rejects_bad_arguments(orc):
    x = np.zeros((1, 1, 4, 2), dtype=np.uint8)
    with pytest.raises(ValueError):
        orc.attention_bwd(x, x, x, x, 1.0, False, "e4m3")
