"""The seeded input generator (shared by the oracle tests and the GPU tests)."""
import numpy as np
import pytest

from fp32_sgemm_gb300 import inputs


def _splitmix64_sequential(seed, count):
    # Stateful form of the published generator: state advances by the golden
    # gamma before every output.
    mask = (1 << 64) - 1
    state = seed & mask
    out = []
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & mask
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_published_vector():
    # First five outputs of SplitMix64 seeded with 1234567, the vector that
    # reference implementations of the generator print.
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(v) for v in inputs.splitmix64(1234567, 0, 5)] == want


@pytest.mark.parametrize("seed", [0, 1, 4, 2**63 + 12345])
def test_counter_form_equals_sequential(seed):
    seq = _splitmix64_sequential(seed, 300)
    got = [int(v) for v in inputs.splitmix64(seed, 0, 300)]
    assert got == seq
    # Any window of the stream is the same numbers.
    assert [int(v) for v in inputs.splitmix64(seed, 137, 50)] == seq[137:187]


def test_uniform_values_exact_and_in_range():
    x = inputs.draw(7, 0, 200_000, "uniform")
    assert x.dtype == np.float32
    assert x.min() >= -1.0 and x.max() < 1.0
    # Every value is a multiple of 2^-23: exactly representable in fp32.
    scaled = x.astype(np.float64) * 2.0 ** 23
    assert np.all(scaled == np.round(scaled))
    assert abs(float(x.mean())) < 0.01
    assert abs(float(x.astype(np.float64).var()) - 1.0 / 3.0) < 0.01


def test_integer_values():
    x = inputs.draw(11, 0, 90_000, "integer")
    assert set(np.unique(x).tolist()) == set(range(-4, 5))
    counts = np.bincount((x + 4).astype(np.int64), minlength=9)
    assert counts.min() > 9000 and counts.max() < 11000


def test_problem_stream_layout():
    p = inputs.make_problem(5, 7, 3, 9, alpha=0.5, beta=0.25, lda=4, ldb=9, ldc=8)
    flat = inputs.draw(9, 0, 5 * 3 + 3 * 7 + 5 * 7, "uniform")
    np.testing.assert_array_equal(p.A[:, :3].ravel(), flat[:15])
    np.testing.assert_array_equal(p.B[:, :7].ravel(), flat[15:36])
    np.testing.assert_array_equal(p.C0[:, :7].ravel(), flat[36:])
    assert np.isnan(p.A[:, 3:]).all() and np.isnan(p.B[:, 7:]).all()
    assert np.isnan(p.C0[:, 7:]).all()
    assert (p.lda, p.ldb, p.ldc) == (4, 9, 8)


def test_workload_recipes():
    w = inputs.WORKLOADS
    assert (w["sgemm_4096"].M, w["sgemm_4096"].seed) == (4096, 2)
    odd = w["sgemm_4095x4097x1023"]
    assert (odd.M, odd.N, odd.K, odd.alpha, odd.beta, odd.seed) == (4095, 4097, 1023, 0.5, 0.25, 3)
    assert w["sgemm_8192"].samples == 65536


def test_sample_entries_in_range_and_seeded():
    r, c = inputs.sample_entries(8192, 8192, 65536, 4)
    assert r.min() >= 0 and r.max() < 8192 and c.min() >= 0 and c.max() < 8192
    r2, c2 = inputs.sample_entries(8192, 8192, 65536, 4)
    assert np.array_equal(r, r2) and np.array_equal(c, c2)
    assert len(set(zip(r[:1000].tolist(), c[:1000].tolist()))) > 990


def test_pattern_is_integer_valued_and_library_independent():
    torch = pytest.importorskip("torch")
    r = np.arange(40)[:, None]
    c = np.arange(33)[None, :]
    a = inputs.pattern(r, c, 3)
    b = inputs.pattern(torch.from_numpy(r), torch.from_numpy(c), 3).numpy()
    assert a.dtype == np.float32 and b.dtype == np.float32
    np.testing.assert_array_equal(a, b)
    assert set(np.unique(a)) <= set(range(-4, 5))
    assert a[2, 5] == ((2 * 7 + 5 * 13 + 3 * 5) % 9) - 4
