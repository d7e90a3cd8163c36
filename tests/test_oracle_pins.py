"""The oracle against what the definitions fix (CPU only)."""
import numpy as np
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("pin", pins.FAST_PINS, ids=lambda p: p.__name__)
def test_fast_pin(o, pin):
    pin(o)


def test_f16_decode_exhaustive(o):
    pins.pin_f16_decode_exhaustive(o)


def test_bf16_decode_exhaustive(o):
    pins.pin_bf16_decode_exhaustive(o)


def test_f16_encode_exhaustive_nonnegative(o):
    pins.pin_f16_encode_exhaustive(o)


def test_check_rules():
    """The tolerance checker accepts an error inside both rules and rejects
    one outside either."""
    rng = np.random.default_rng(3)
    y_ref = rng.normal(0, 1, 1000)
    absum = np.abs(y_ref) * 10 + 1
    assert oracle.check(y_ref + 1e-4 * absum * rng.uniform(-1, 1, 1000) * 0, y_ref, absum)["ok"]
    small = y_ref * (1 + 1e-3)
    assert oracle.check(small, y_ref, absum)["ok"]
    big_one = y_ref.copy(); big_one[5] += 0.011 * absum[5]
    assert not oracle.check(big_one, y_ref, absum)["ok"]
    l2 = y_ref * (1 + 3e-3)
    assert not oracle.check(l2, y_ref, absum)["ok"]
    nan = y_ref.copy(); nan[0] = np.nan
    assert not oracle.check(nan, y_ref, absum)["ok"]


def test_quantize_rejects_bad_k(o):
    with pytest.raises(ValueError):
        o.quantize(np.zeros((2, 33), np.float32))
