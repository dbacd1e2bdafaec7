"""The parity report the GPU tests gate on (tests/gpu_util.parity_stats),
checked on hand-made BF16 bit patterns: infinities match only the same
infinity, NaN only NaN, and finite values pass within 1e-2 + 1e-2*|ref|."""
import numpy as np

from tests import gpu_util as gu

INF, NINF, NAN, ONE, TWO = 0x7F80, 0xFF80, 0x7FC0, 0x3F80, 0x4000


def _bits(*v):
    return np.array(v, dtype=np.uint16)


def test_matching_infinities_pass():
    st = gu.parity_stats(_bits(INF, NINF, ONE), _bits(INF, NINF, ONE))
    assert st["fail"] == 0 and st["inf_matched"] == 2 and st["max_abs"] == 0.0


def test_infinity_against_other_values_fails():
    assert gu.parity_stats(_bits(INF), _bits(NINF))["fail"] == 1
    assert gu.parity_stats(_bits(INF), _bits(ONE))["fail"] == 1
    assert gu.parity_stats(_bits(ONE), _bits(NINF))["fail"] == 1


def test_nan_only_matches_nan():
    assert gu.parity_stats(_bits(NAN), _bits(NAN))["fail"] == 0
    assert gu.parity_stats(_bits(NAN), _bits(ONE))["fail"] == 1
    assert gu.parity_stats(_bits(ONE), _bits(NAN))["fail"] == 1


def test_finite_gate():
    # 1.0 against 1.0078125 (one BF16 spacing): |d| = 0.0078 <= 0.01 + 0.01
    assert gu.parity_stats(_bits(0x3F81), _bits(ONE))["fail"] == 0
    # 2.0 against 1.0 fails
    assert gu.parity_stats(_bits(TWO), _bits(ONE))["fail"] == 1
