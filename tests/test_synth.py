"""The seeded input generators: published SplitMix64 vectors and the
workload recipes (sizes, value ranges, tie forcing)."""
import numpy as np

import synth


def test_splitmix64_published_vectors():
    # First outputs of SplitMix64 seeded with 1234567 and with 0, as published
    # with the reference implementation (splitmix64.c).
    assert [synth.splitmix64_at(1234567, i) for i in range(5)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]
    assert synth.splitmix64_at(0, 0) == 0xE220A8397B1DCDAF


def test_i32_uniform_is_top_half_of_stream():
    a = synth.i32_uniform(1000, 9, nthreads=3)
    exp = [np.uint32(synth.splitmix64_at(9, i) >> 32).view(np.int32) for i in range(1000)]
    assert a.tolist() == [int(v) for v in exp]
    b = synth.i32_uniform(1000, 9, nthreads=1)
    assert np.array_equal(a, b)


def test_i32_mod_and_ascending():
    a = synth.i32_mod(5000, 4, 1000)
    assert a.min() >= 0 and a.max() <= 999
    assert a.tolist()[:3] == [synth.splitmix64_at(4, i) % 1000 for i in range(3)]
    assert synth.i32_ascending(10).tolist() == list(range(10))


def test_normal_moments():
    z = synth.f32_normal(1 << 20, 5)
    assert abs(float(z.mean())) < 0.01
    assert abs(float(z.std()) - 1.0) < 0.01


def test_tie_forcing_recipe():
    rows, cols = 16, 4096
    base = synth.f32_rows_normal(rows, cols, 5)
    tied = synth.f32_rows_tied(rows, cols, 5, frac=0.01)
    m = int(0.01 * cols)
    for r in range(rows):
        mx = base[r].max()
        changed = np.count_nonzero(tied[r] != base[r])
        assert changed <= m and changed >= m - 1
        assert np.count_nonzero(tied[r] == mx) in (m, m + 1)
        assert tied[r].max() == mx
