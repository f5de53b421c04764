"""The seeded operand generator: stream definition, layouts and recipes."""

import numpy as np

import synth

MASK = (1 << 64) - 1


def splitmix64_scalar(seed, count):
    """The sequential splitmix64 generator, one draw at a time."""
    state, out = seed & MASK, []
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & MASK
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
        out.append(z ^ (z >> 31))
    return out


def test_counter_form_matches_sequential_generator():
    for seed in (0, 1, 1003, 2 ** 63 + 12345):
        ref = splitmix64_scalar(seed, 50)
        got = [int(v) for v in synth.splitmix64(seed, 0, 50)]
        assert got == ref
        assert [int(v) for v in synth.splitmix64(seed, 20, 30)] == ref[20:]


def test_published_seed_zero_values():
    # the widely quoted first outputs of splitmix64 seeded with 0
    got = [int(v) for v in synth.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_recipes_and_layout():
    a, b = synth.operands(7, 5, 9, seed=42, kind="uniform")
    assert a.shape == (7, 9) and b.shape == (5, 9)
    assert a.dtype == np.float16 and b.dtype == np.float16
    u = synth.uniform01(42, 0, 7 * 9 + 5 * 9)
    assert np.array_equal(a.reshape(-1), (2 * u[:63] - 1).astype(np.float16))
    assert np.array_equal(b.reshape(-1), (2 * u[63:] - 1).astype(np.float16))
    assert np.all(np.abs(a.astype(np.float64)) <= 1.0)

    ai, bi = synth.operands(64, 32, 256, seed=9, kind="int")
    vals = set(np.unique(ai).tolist()) | set(np.unique(bi).tolist())
    assert vals <= {-2.0, -1.0, 0.0, 1.0, 2.0} and len(vals) == 5

    an, bn = synth.operands(128, 64, 1024, seed=5, kind="normal")
    assert abs(float(an.astype(np.float64).std()) - 1.0) < 0.02
    assert abs(float(bn.astype(np.float64).std()) * 32.0 - 1.0) < 0.03  # 1/sqrt(1024)

    # both operands scaled: the same draws, A divided by sqrt(K) as well
    a2, b2 = synth.operands(128, 64, 1024, seed=5, kind="normal_both")
    assert np.array_equal(b2, bn)
    u = synth.uniform01(5, 0, 2 * 128 * 1024)
    z = np.sqrt(-2 * np.log1p(-u[0::2])) * np.cos(2 * np.pi * u[1::2]) / 32.0
    assert np.array_equal(a2.reshape(-1), z.astype(np.float16))


def test_chunking_is_invisible():
    n = synth._CHUNK + 1000
    a, _ = synth.operands(1, 1, n, seed=77, kind="normal")
    u = synth.uniform01(77, 0, 2 * n)
    z = np.sqrt(-2 * np.log1p(-u[0::2])) * np.cos(2 * np.pi * u[1::2])
    assert np.array_equal(a.reshape(-1), z.astype(np.float16))
