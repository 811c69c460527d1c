"""The CPU oracle against its pins (see ``oracle_pins.py`` for what each
pin rests on)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_toy_fixture_is_reproduced(orc):
    """Regression: the stored toy outputs (written by tests/golden/make_golden.py
    from the oracle) are reproduced bit for bit."""
    import json
    import os

    import numpy as np

    import synth
    from tests.golden.make_golden import toy_fixture

    path = os.path.join(os.path.dirname(__file__), "golden", "toy_seed0_oracle.json")
    stored = json.load(open(path))
    fresh = toy_fixture()
    for key in ("ids", "counts", "offsets", "perm", "inv_perm", "out_hex"):
        assert stored[key] == fresh[key], key
    assert np.all(np.isfinite(np.array([[float.fromhex(v) for v in r] for r in stored["out_hex"]])))
    assert synth.TOY.Ms == (4,)
