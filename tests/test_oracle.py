"""The CPU oracle against its pins (CPU only).

``oracle_pins`` holds checks that tie the oracle to the pages and to the
mathematics.  The faithful build must pass every pin; each build with a planted
mistake (a dropped fade, a read before the write, a wrong sign, a wrong index,
a dropped beta, a missing floor, the fade in the wrong place, a missing key
normalisation, the wrong probe vector, a wrong widening of bf16 or fp32
inputs, reversed convolution taps or window, a missing Swish, a convolution
across a sequence boundary, an unbounded or mis-scaled decay mapping) must
fail at least one of them.  A marshalling mistake on the Python
side (bf16 passed through float16) is planted the same way.
"""
import os

import pytest

import oracle
from oracle import build as oracle_build
from tests import oracle_pins

MUTATIONS = {
    1: "no fade",
    2: "read before write",
    3: "erase with the wrong sign",
    4: "wrong state row in the read",
    5: "beta dropped from the write",
    6: "no floor on log alpha",
    7: "fade after the write",
    8: "key not normalised",
    9: "state probed with the query",
    10: "bf16 input widened with the wrong shift",
    11: "fp32 input cut to bf16",
    12: "convolution taps applied newest first",
    13: "no Swish on v",
    14: "decay logit through the old unbounded softplus",
    15: "decay scale outside the sigmoid",
    16: "convolution window read newest first",
    17: "convolution reads across a packed-sequence boundary",
    18: "convolution output truncated to bf16 instead of rounded",
}


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    assert orc.mutation == 0
    pin(orc)


@pytest.mark.parametrize("m", sorted(MUTATIONS), ids=lambda m: MUTATIONS[m].replace(" ", "_"))
def test_pins_catch_planted_mistake(tmp_path, m):
    path = oracle_build.build(out_path=os.path.join(tmp_path, f"m{m}.so"), mutation=m)
    bad = oracle.Oracle(path)
    assert bad.mutation == m
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(bad)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught planted mistake {m} ({MUTATIONS[m]})"


def test_pins_catch_bf16_marshalled_as_float16(orc, monkeypatch):
    """bf16 tensors handed over as float16 values (a plausible marshalling slip
    in the front-end) lose range and precision; the widening pin sees it."""
    import numpy as np
    import torch

    from oracle import oracle as front

    good = front._as_buffer

    def wrong(x):
        if isinstance(x, torch.Tensor) and x.dtype == torch.bfloat16:
            return x.to(torch.float16).to(torch.float32).numpy(), front._F32
        return good(x)

    monkeypatch.setattr(front, "_as_buffer", wrong)
    with pytest.raises(AssertionError):
        oracle_pins.pin_input_widening(orc)
    monkeypatch.setattr(front, "_as_buffer", good)
    oracle_pins.pin_input_widening(orc)
    assert np.isfinite(good(torch.zeros(2, dtype=torch.bfloat16))[0]).all()


def test_state_sizes_golden():
    """The state layout [N, H, d_k, d_v] fp32 holds the pages' counts."""
    import numpy as np
    g = oracle_pins.golden("state_sizes.json")
    per_layer = int(np.prod((1, g["heads"], g["d_k"], g["d_v"])))
    assert per_layer == g["numbers_per_layer"]
    assert per_layer * g["kda_layers"] == g["numbers_per_sequence"]
    assert round(g["numbers_per_sequence"] * 4 / 2 ** 20) == g["mib_fp32"]


def test_oracle_rejects_bad_arguments(orc):
    import numpy as np
    q = np.zeros((4, 1, 4))
    with pytest.raises(ValueError):
        orc.prefill(q, q, q, q, np.zeros((4, 1)), None, np.array([0, 3, 2], dtype=np.int32))
    with pytest.raises(ValueError):
        orc.prefill(q, q, q, q, np.zeros((4, 1)), None, None, heads=(0, 2))
