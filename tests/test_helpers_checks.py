"""The x_last check of the chain tests on planted cases (CPU): it accepts the run-to-run
differences the fp32 split-K sums can cause and rejects a missing residual, a stale residual and
a shifted row."""
import numpy as np
import pytest

from oracle import moe_oracle as orc

from helpers import check_x_last, residual_step


def _bf16_bits(v):
    return np.array([orc.double_to_bf16(t) for t in np.asarray(v, dtype=np.float64).ravel()], dtype=np.uint16)


def _case(seed=3, n=2048):
    rng = np.random.default_rng(seed)
    r = _bf16_bits(rng.standard_normal(n))
    out = _bf16_bits(0.7 * rng.standard_normal(n))
    return r, out, residual_step(r, out)


def _one_step(bits, idx, steps=1):
    """bits with the elements at idx moved `steps` bf16 steps away from zero."""
    b = bits.copy()
    b[idx] = b[idx] + steps  # larger magnitudes of the same sign (finite, non-extreme values)
    return b


def test_exact_cases():
    r, out, want = _case()
    check_x_last(want, r, out, exact=True)
    with pytest.raises(AssertionError):
        check_x_last(_one_step(want, [5]), r, out, exact=True)


def test_accepts_chain_divergence():
    """The chain's own x_{n-1} a step away in 65 elements: x_last follows it."""
    r, out, _ = _case()
    idx = np.arange(0, 2048, 31)[:65]
    r_chain = _one_step(r, idx)
    check_x_last(residual_step(r_chain, out), r, out, exact=False)


@pytest.mark.parametrize("mistake", ["no residual", "stale residual", "shifted row", "many steps"])
def test_rejects_mistakes(mistake):
    r, out, want = _case()
    if mistake == "no residual":
        got = out
    elif mistake == "stale residual":  # another token's x
        r2, _, _ = _case(seed=4)
        got = residual_step(r2, out)
    elif mistake == "shifted row":
        got = np.roll(want, 1)
    else:  # three steps off in a fifth of the elements
        got = _one_step(want, np.arange(0, 2048, 5), steps=3)
    with pytest.raises(AssertionError):
        check_x_last(got, r, out, exact=False)
