"""The oracle against its pins (CPU only)."""
import pytest

import _pins


@pytest.mark.parametrize("pin", _pins.PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_openmp_matches_single_thread(orc):
    """Spreading the (row, head) problems over threads changes no bit."""
    import numpy as np
    rng = np.random.default_rng(3)
    c = _pins.make_tiny(rng, [5, 33, 70, 2], [1, 4, 9, 2], hq=4, hkv=2, d=16, bs=8)
    a = orc.paged_attention(c["dtype"], c["q"], c["k_pool"], c["v_pool"], c["block_tables"],
                            c["context_lens"], c["scale"], query_start_loc=c["query_start_loc"],
                            num_threads=1)
    b = orc.paged_attention(c["dtype"], c["q"], c["k_pool"], c["v_pool"], c["block_tables"],
                            c["context_lens"], c["scale"], query_start_loc=c["query_start_loc"],
                            num_threads=4)
    assert np.array_equal(a, b)


def test_rejects_block_outside_pool(orc):
    import numpy as np
    rng = np.random.default_rng(5)
    c = _pins.make_tiny(rng, [9], [1], hq=2, hkv=1, d=8, bs=4)
    c["block_tables"][0, 1] = c["k_pool"].shape[0]
    with pytest.raises(ValueError):
        _pins.run_case(orc, c)


def test_zero_length_gives_zero(orc):
    import numpy as np
    rng = np.random.default_rng(6)
    c = _pins.make_tiny(rng, [0, 3], [1, 1], hq=2, hkv=1, d=8, bs=4)
    # A decode row over an empty context: no key, output 0 by definition.
    c["qlens"] = [1, 1]
    out = _pins.run_case(orc, c, decode=True)
    assert np.all(out[0] == 0.0)
