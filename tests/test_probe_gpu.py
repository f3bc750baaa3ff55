"""The exponential-unit probe behind the bench's exponential ceiling
(fa_ex2_throughput): a plausible rate, stable across calls, and the context
usable afterwards."""
import pytest

import exact_attention_79_gb300 as pkg

pytestmark = pytest.mark.gpu


def test_ex2_throughput_is_plausible_and_stable(fa):
    a = pkg.ex2_throughput()
    b = pkg.ex2_throughput()
    fa.check_device_status()
    # an SM has 128 lanes, so at most 128 results per cycle; a rate below one
    # result per 64 lane-cycles (2 per SM cycle) would mean the probe measured
    # something else
    assert 2.0 <= a <= 128.0, a
    assert abs(a - b) <= 0.1 * a, (a, b)
