"""The code-parity rule itself (host logic, no GPU): a code may differ from
the oracle's only at a near tie, (d2 - d1) < 1e-6 d2 on the oracle's
distances; any other difference fails."""
import numpy as np
import pytest

from oracle import parity


def _oracle_out(codes, d1, d2):
    return {"codes": np.asarray(codes), "d1": np.asarray(d1, float),
            "d2": np.asarray(d2, float)}


def test_identical_codes_pass():
    o = _oracle_out([[1, 2, 3]], [[1.0, 2.0, 3.0]], [[2.0, 3.0, 4.0]])
    assert parity.check_codes(np.array([[1, 2, 3]]), o) == {
        "subvectors": 3, "mismatch": 0, "near_tie": 0}


def test_near_tie_mismatch_is_counted():
    # second code: gap 5e-7 relative -> near tie
    o = _oracle_out([[1, 2]], [[1.0, 2.0]], [[1.5, 2.0 * (1 + 5e-7)]])
    res = parity.check_codes(np.array([[1, 7]]), o)
    assert res == {"subvectors": 2, "mismatch": 1, "near_tie": 1}


@pytest.mark.parametrize("rel", [1e-6, 2e-6, 1e-3])
def test_mismatch_beyond_near_tie_fails(rel):
    o = _oracle_out([[4]], [[1.0]], [[1.0 / (1.0 - rel)]])
    with pytest.raises(AssertionError):
        parity.check_codes(np.array([[5]]), o)


def test_allclose_report_tolerance():
    ok, err, _ = parity.allclose_report([1.0 + 0.0119], [1.0])
    assert ok and abs(err - 0.0119) < 1e-12
    ok, _, excess = parity.allclose_report([1.0 + 0.0121], [1.0])
    assert not ok and excess > 0
