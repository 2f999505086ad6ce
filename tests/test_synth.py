"""The seeded input generator (host side): addressable, deterministic, right moments."""
import numpy as np

import synth


def test_keys_distinct_and_stable():
    ks = {synth.stream_key(0, a, b) for a in range(8) for b in range(8)}
    assert len(ks) == 64
    assert synth.stream_key(0, 1, 2) == synth.stream_key(0, 1, 2)
    assert synth.stream_key(0, 1, 2) != synth.stream_key(1, 1, 2)


def test_positions_are_addressable():
    key = synth.stream_key(0, 3)
    full = synth.normal_f32(key, 5000, 0.02, idx0=100)
    idx = np.random.default_rng(0).permutation(5000)[:777]
    part = synth.normal_f32_at(key, idx + 100, 0.02)
    assert part.tobytes() == full[idx].tobytes()
    bf = synth.normal_bf16(key, 5000, 0.02, idx0=100)
    assert synth.normal_bf16_at(key, idx + 100, 0.02).tobytes() == bf[idx].tobytes()


def test_moments_and_tails():
    x = synth.normal_f32(synth.stream_key(7), 1 << 20, 1e-3).astype(np.float64)
    assert abs(x.mean()) < 5e-6
    assert abs(x.std() / 1e-3 - 1) < 5e-3
    assert np.abs(x).max() <= 6e-3
    a = synth.normal_f32(synth.stream_key(8), 1 << 16, 1e-4, absval=True)
    assert np.all(a >= 0)


def test_padding_is_zero():
    x = synth.normal_f32(synth.stream_key(9), 64, 1.0, idx0=10, n_valid=50)
    assert np.all(x[40:] == 0) and np.all(x[:40] != 0)
