"""The seeded input generator: published known answers and basic statistics. CPU only."""
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        assert synth.philox4x32_10(v[0:4], v[4:6]) == tuple(v[6:10])


def test_normal_moments_and_determinism():
    z = synth.normal_f32(0, 7, 2_000_000)
    assert abs(z.mean()) < 3e-3 and abs(z.std() - 1) < 3e-3
    np.testing.assert_array_equal(z[1000:1010], synth.normal_f32(0, 7, 10, offset=1000))
    assert not np.array_equal(z[:100], synth.normal_f32(1, 7, 100))


def test_bf16_is_round_to_nearest_of_the_f32_draw():
    f = synth.normal_f32(3, 2, 100000, 0.0, 0.02)
    b = synth.bf16_to_f32(synth.normal_bf16(3, 2, 100000, 0.0, 0.02))
    rel = np.abs(b - f) / np.abs(f)
    assert rel.max() <= 2.0 ** -8
    # round to nearest: no value is more than half a bf16 ulp away
    ulp = np.abs(f) * 2.0 ** -7
    assert (np.abs(b - f) <= 0.5 * ulp * 1.0001 + 1e-30).all()


def test_uniform_int_range():
    v = synth.uniform_int(1, 3, 100000, 0, 2048)
    assert v.min() == 0 and v.max() == 2047
    assert abs(v.mean() - 1023.5) < 10


def test_full_shape_weight_bytes():
    # temporal 13.153 GB + text head 0.262 GB + depformer 2.668 GB of streamed weights,
    # plus embedding tables and gains
    assert abs(synth.weight_nbytes(synth.FULL) / 1e9 - 16.743) < 0.01
