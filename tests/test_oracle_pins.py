"""The float64 oracle against facts that do not come from it (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_row_mask_samples_rows(orc):
    c = oracle_pins.dense_case(2, 4, 2, 8, 4, 2, [5, 9], seed=3)
    full = oracle_pins.run(orc, c, 0.3, True)
    import numpy as np

    mask = np.zeros(2 * 4 * 2, dtype=np.uint8)
    mask[[1, 6, 13]] = 1
    part = oracle_pins.run(orc, c, 0.3, True, row_mask=mask)
    flat_full = full.reshape(-1, 8)
    flat_part = part.reshape(-1, 8)
    for i in range(16):
        if mask[i]:
            assert np.array_equal(flat_full[i], flat_part[i])
        else:
            assert not flat_part[i].any()


def test_threads_do_not_change_result(orc):
    import numpy as np

    c = oracle_pins.dense_case(3, 8, 2, 16, 4, 2, [30, 7, 19], seed=5)
    one = oracle_pins.run(orc, c, 0.25, True, threads=1)
    many = oracle_pins.run(orc, c, 0.25, True, threads=4)
    assert np.array_equal(one, many)


def test_bad_block_is_an_error(orc):
    c = oracle_pins.dense_case(1, 2, 1, 8, 4, 1, [6], seed=1)
    c["block_table"][0, 1] = c["k_cache"].shape[0] + 5
    with pytest.raises(ValueError):
        oracle_pins.run(orc, c, 0.3, False)
