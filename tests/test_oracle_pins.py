"""The fp64 oracle against its pins (CPU only; see tests/oracle_pins.py)."""

import pytest

import oracle
from oracle_pins import PINS


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin, lib):
    if pin.__name__ == "pin_bruteforce_highprecision":
        pytest.importorskip("mpmath")
    if pin.__name__ == "pin_library_sdpa":
        pytest.importorskip("scipy")
    pin(lib)


def test_oracle_rejects_bad_arguments(lib):
    import numpy as np
    q = np.zeros((1, 3, 4, 8), dtype=np.uint16)
    k = np.zeros((1, 2, 4, 8), dtype=np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.attn_fwd(q, k, k, True, 1.0, lib=lib)  # Hq % Hkv != 0
    pool = np.zeros((2, 1, 16, 8), dtype=np.uint16)
    table = np.array([[0, 5]], dtype=np.int32)  # block 5 is outside a 2-block pool
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(np.zeros((1, 1, 8), np.uint16), pool, pool, table,
                            np.array([20], np.int32), 1.0, lib=lib)


def test_oracle_empty_shapes(lib):
    import numpy as np
    q = np.zeros((0, 2, 5, 8), dtype=np.uint16)
    o, lse = oracle.attn_fwd(q, q[:, :1], q[:, :1], True, 1.0, lib=lib)
    assert o.shape == (0, 2, 5, 8) and lse.shape == (0, 2, 5)
    q = np.zeros((1, 2, 0, 8), dtype=np.uint16)
    o, lse = oracle.attn_fwd(q, q, q, False, 1.0, lib=lib)
    assert o.size == 0 and lse.size == 0
