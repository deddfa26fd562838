"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda p: p.__name__)
def test_oracle_pin(ora, pin):
    pin(ora)


def test_openmp_threads_do_not_change_results(ora):
    import numpy as np
    import workloads as W

    s = W.decode_step(2, 8, 2, 64, 300, "bf16", [299, 130], seed=1)
    args = (W.raw_bits(s.q), W.raw_bits(s.k_cache), W.raw_bits(s.v_cache), s.position_ids.numpy(),
            8, 2, "bf16")
    one = ora.decode_attn(*args, threads=1)
    many = ora.decode_attn(*args, threads=max(2, ora.max_threads()))
    assert np.array_equal(one, many)
