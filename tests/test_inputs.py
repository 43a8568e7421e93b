"""The seeded input generator: the published splitmix64 definition, the value
semantics of the RWKV-7 time-mix inputs, and exact bf16 rounding."""
import numpy as np
import pytest

GAMMA = np.uint64(0x9E3779B97F4A7C15)


def _splitmix64_np(seed: int, m: np.ndarray) -> np.ndarray:
    """Vectorised splitmix64 (Steele, Lea, Flood 2014): output m of a
    generator seeded with `seed` is mix(seed + (m + 1) * gamma)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (m.astype(np.uint64) + np.uint64(1)) * GAMMA
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def test_splitmix64_matches_independent_vectorised_definition(gen_mod):
    lib = gen_mod._load()
    m = np.array([0, 1, 2, 3, 1000, 123456789, 2**40 + 7], dtype=np.uint64)
    for seed in (0, 1, 0xDEADBEEF, 2**63 + 5):
        ref = _splitmix64_np(seed, m)
        got = np.array([lib.wkv7_gen_splitmix64_at(seed, int(x)) for x in m], dtype=np.uint64)
        np.testing.assert_array_equal(got, ref)


def test_splitmix64_sequential_state_agrees(gen_mod):
    """The counter form equals the usual stateful form (state += gamma, then mix)."""
    lib = gen_mod._load()
    state = 42
    for m in range(20):
        state = (state + 0x9E3779B97F4A7C15) % 2**64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) % 2**64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) % 2**64
        z = z ^ (z >> 31)
        assert lib.wkv7_gen_splitmix64_at(42, m) == z


def test_uniform_and_normal_distribution(gen_mod):
    lib = gen_mod._load()
    u = np.array([lib.wkv7_gen_uniform_at(3, m) for m in range(20000)])
    assert u.min() > 0.0 and u.max() <= 1.0
    assert abs(u.mean() - 0.5) < 0.01
    ref = ((_splitmix64_np(3, np.arange(20000)) >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0**-53
    np.testing.assert_array_equal(u, ref)
    z = np.array([lib.wkv7_gen_normal_at(3, q) for q in range(20000)])
    u1, u2 = ref[0::2], ref[1::2]
    np.testing.assert_allclose(z[:10000], np.sqrt(-2 * np.log(u1)) * np.cos(2 * np.pi * u2), rtol=1e-12, atol=1e-12)
    assert abs(z.mean()) < 0.03 and abs(z.std() - 1.0) < 0.03


def _bf16_from_f32_bits(x32: np.ndarray) -> np.ndarray:
    b = x32.view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_bf16_round_to_nearest_even(gen_mod):
    lib = gen_mod._load()
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(5000) * 10.0 ** rng.integers(-6, 6, 5000)).astype(np.float32)
    got = np.array([lib.wkv7_gen_bf16_rne(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(got, _bf16_from_f32_bits(x))
    # ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1.0);
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6 -> even (1 + 2^-6)
    assert lib.wkv7_gen_bf16_rne(1.0 + 2**-8) == 0x3F80
    assert lib.wkv7_gen_bf16_rne(1.0 + 3 * 2**-8) == 0x3F82
    # just above the tie rounds up (a float32 detour would lose this)
    assert lib.wkv7_gen_bf16_rne(1.0 + 2**-8 + 2**-40) == 0x3F81
    assert lib.wkv7_gen_bf16_rne(-2.0) == 0xC000
    assert lib.wkv7_gen_bf16_rne(float("inf")) == 0x7F80


def test_value_semantics(gen_mod):
    B, T, H, N = 2, 16, 3, 16
    d = gen_mod.generate(B, T, H, N, "f64", 0.1)
    lo = np.exp(-0.606531)
    assert d["w"].min() > lo and d["w"].max() < 1.0
    kk = -d["a"]
    np.testing.assert_allclose(np.linalg.norm(kk, axis=-1), 1.0, rtol=1e-11)
    ratio = d["b"] / kk
    assert ratio.min() > 0.0 and ratio.max() < 1.0  # sigmoid(u)
    for n in ("r", "k", "v"):
        assert abs(d[n].std() * np.sqrt(N) - 1.0) < 0.15
    assert abs(d["dy"].std() - 1.0) < 0.15
    assert abs(d["s_init"].std() - 0.1) < 0.02
    # streams are distinct
    assert not np.allclose(d["r"], d["k"])


def test_storage_kinds_round_the_same_values(gen_mod):
    shape = (1, 8, 2, 16)
    d64 = gen_mod.generate(*shape, "f64")
    d32 = gen_mod.generate(*shape, "f32")
    dbf = gen_mod.generate(*shape, "bf16")
    lib = gen_mod._load()
    for n in gen_mod.NAMES:
        np.testing.assert_array_equal(d32[n], d64[n].astype(np.float32))
        ref = np.array([lib.wkv7_gen_bf16_rne(float(v)) for v in d64[n].ravel()], dtype=np.uint16)
        np.testing.assert_array_equal(dbf[n].ravel(), ref)
        np.testing.assert_allclose(gen_mod.as_f64(dbf[n], "bf16"), d64[n], rtol=2**-8)


def test_thread_count_does_not_change_values(gen_mod):
    a = gen_mod.generate(2, 33, 3, 16, "f32", 0.1, nthreads=1)
    b = gen_mod.generate(2, 33, 3, 16, "f32", 0.1, nthreads=5)
    for n in list(gen_mod.NAMES) + ["s_init"]:
        np.testing.assert_array_equal(a[n], b[n])


def test_invalid_arguments(gen_mod):
    with pytest.raises(RuntimeError):
        gen_mod.generate(0, 4, 1, 16)
