"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
import synth
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.get())


def test_synth_generator_definition():
    """SplitMix64 against values computed from its published definition, and the Box-Muller
    deviates are N(0,1) in bulk and reproducible element by element."""
    # splitmix64 of the state after one increment from seed 0 (first output of the generator)
    assert synth.splitmix64(0) == 0xE220A8397B1DCDAF
    x = synth.normal_bf16(7, synth.TAG_Q, (1 << 16,))
    f = synth.bf16_bits_to_f32(x).astype(np.float64)
    assert abs(f.mean()) < 0.02 and abs(f.std() - 1.0) < 0.02
    for i in (0, 1, 12345, 65535):
        assert synth.normal_bf16_at(7, synth.TAG_Q, i) == int(x[i])
    k2 = synth.normal_bf16(7, synth.TAG_K, (64,), mult=2.0)
    k1 = synth.normal_bf16(7, synth.TAG_K, (64,))
    assert np.array_equal(synth.bf16_bits_to_f32(k2), 2 * synth.bf16_bits_to_f32(k1))


def test_sampled_rows_cover_boundaries():
    rows = synth.sample_rows(131072, 16, 256, seed=1)
    assert rows.size == 256 and len(set(rows.tolist())) == 256
    m = 131072 // 32
    for c in range(32):
        assert c * m in rows and c * m + m - 1 in rows
    assert 0 in rows and 131071 in rows
