"""The bf16 parity bar of parity_bars.check_bf16 on planted mistakes (CPU):
rounding-level noise passes, and a single wrong element, one wrong step of a
chunk, a sign flip, a wrong value in a near-empty chunk and a nonzero value
where the reference is exactly zero each fail, although several of them pass
the whole-tensor relative L2 bar alone."""
import numpy as np
import pytest

from parity_bars import REL_L2, check_bf16, stats


def _ref(seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((2, 130, 3, 64)), rng


def test_rounding_noise_passes():
    ref, rng = _ref()
    check_bf16("y", ref * (1 + 4.5e-3 * rng.standard_normal(ref.shape)), ref)


@pytest.mark.parametrize("mistake", ["one_element", "one_step", "sign_flip", "near_empty_chunk"])
def test_planted_mistakes_fail(mistake):
    ref, rng = _ref(1)
    got = ref * (1 + 1e-3 * rng.standard_normal(ref.shape))
    if mistake == "one_element":
        got[1, 17, 2, 5] += ref.std()
    elif mistake == "one_step":
        got[0, 32, 1, :] += 0.5 * ref[0, 32, 1, :]
    elif mistake == "sign_flip":
        got[1, 100, 0, 7] *= -1
        ref[1, 100, 0, 7] = ref.std()
        got[1, 100, 0, 7] = -ref[1, 100, 0, 7]
    else:  # the last (ragged) chunk is a thousand times smaller than the rest
        ref[0, 128:] *= 1e-3
        got = ref.copy()
        got[0, 129, 0, 3] += 0.2 * ref.std()
    whole = stats(got, ref)[0]
    if mistake != "one_step":
        assert whole <= REL_L2  # the whole-tensor bar alone would pass it
    with pytest.raises(AssertionError):
        check_bf16("dr", got, ref)


def test_zero_reference_needs_zero():
    z = np.zeros((1, 1, 2, 64))
    check_bf16("dw", z, z)
    g = z.copy()
    g[0, 0, 1, 3] = 1e-12
    with pytest.raises(AssertionError):
        check_bf16("dw", g, z)


def test_states_are_checked_per_head():
    rng = np.random.default_rng(2)
    ref = rng.standard_normal((4, 8, 16, 16))
    ref[3, 7] *= 1e-2  # one head with a small state
    got = ref.copy()
    got[3, 7] += 1e-2 * ref[3, 7].std() * 40 * rng.standard_normal((16, 16))
    assert stats(got, ref, "state")[0] <= REL_L2
    with pytest.raises(AssertionError):
        check_bf16("s_final", got, ref, "state")
