"""The argument behind the kernels' division-free e4m3 quantiser, checked in numpy fp32 (CPU).

The kernels take the code of the IEEE fp32 quotient x / s (s = amax / 448) without dividing: with
r = RN(1/s), the products x * RN(r (1 - 2^-20)) and x * RN(r (1 + 2^-20)) bracket the correctly rounded
quotient, and when both convert to the same e4m3 code that is the quotient's code; otherwise they divide.
This test replays that rule with numpy's IEEE fp32 arithmetic and torch's nearest-even e4m3 cast on random
bf16 blocks across many scale magnitudes and on quotients placed exactly on, and next to, every e4m3
rounding boundary, and checks that the rule never takes a code other than the quotient's.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

F32 = np.float32
LO = F32(1 - 2.0 ** -20)
HI = F32(1 + 2.0 ** -20)


def e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest-even e4m3 codes, saturated to +-448 (the kernels' cvt.rn.satfinite)."""
    t = torch.from_numpy(np.clip(v, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def rule(x: np.ndarray, amax: np.ndarray):
    """(codes by the bracketing rule, codes of the quotient, fraction taken without division)."""
    s = np.where(amax > 0, amax / F32(448), F32(1)).astype(F32)
    with np.errstate(over="ignore", divide="ignore"):
        r = (F32(1) / s).astype(F32)
    lo, hi = (r * LO).astype(F32), (r * HI).astype(F32)
    with np.errstate(over="ignore", invalid="ignore"):
        cl, ch = e4m3((x * lo).astype(F32)), e4m3((x * hi).astype(F32))
        quotient = e4m3((x / s).astype(F32))
    fast = (s >= F32(2.0 ** -125)) & (s <= F32(2.0 ** 125)) & (cl == ch)
    return np.where(fast, cl, quotient), quotient, fast.mean()


def bf16(v: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(v, dtype=F32).view(np.uint32) & 0xFFFF0000).view(F32)


@pytest.mark.parametrize("exp", [-60, -30, -10, -3, 0, 3, 10, 30, 60])
def test_random_blocks_take_the_quotients_codes(exp):
    rng = np.random.default_rng(100 + exp)
    x = bf16(rng.standard_normal((4096, 128)).astype(F32) * F32(2.0 ** exp))
    amax = np.abs(x).max(axis=1, keepdims=True) * np.ones_like(x)
    got, want, frac = rule(x, amax)
    assert np.array_equal(got, want)
    assert frac > 0.99, "the division is the exception"


def boundary_quotients() -> np.ndarray:
    """Every e4m3 rounding boundary (midpoints of the normal range, subnormal midpoints, 2^-10), and 448."""
    b = [(1 + (2 * m + 1) / 16) * 2.0 ** e for e in range(-6, 9) for m in range(8)]
    b += [(j + 0.5) * 2.0 ** -9 for j in range(7)] + [2.0 ** -10, 448.0]
    return np.array([v for v in b if v <= 448.0], dtype=F32)


@pytest.mark.parametrize("exp", [-100, -20, -7, 0, 7, 20, 100])
def test_quotients_on_and_beside_every_boundary(exp):
    q = boundary_quotients()
    x = q * F32(2.0 ** exp)                      # scale 2^exp exactly: x / s = q
    near = np.concatenate([x, np.nextafter(x, F32(0)), np.nextafter(x, F32(np.inf)), -x])
    amax = np.full(near.shape, F32(448.0 * 2.0 ** exp))
    got, want, frac = rule(near, amax)
    assert np.array_equal(got, want)
    assert frac < 0.5, "ties and their neighbours go to the division"


def test_scales_outside_the_fast_range_divide():
    x = np.array([1e-38, -3e-39, 2e-39, 0.0], dtype=F32)
    amax = np.full(x.shape, F32(1e-38))          # s = amax / 448 is subnormal: 1/s would overflow
    got, want, frac = rule(x, amax)
    assert np.array_equal(got, want) and frac == 0.0


def test_a_wider_window_would_be_needed_with_a_coarser_reciprocal():
    """Plant a mistake: a reciprocal rounded to bf16 (error 2^-9) breaks the bracket, and the rule then takes
    codes other than the quotient's. The exact r = RN(1/s) is what the bracket relies on."""
    rng = np.random.default_rng(5)
    x = bf16(rng.standard_normal((2048, 128)).astype(F32))
    amax = np.abs(x).max(axis=1, keepdims=True) * np.ones_like(x)
    s = (amax / F32(448)).astype(F32)
    r = bf16(F32(1) / s)
    cl, ch = e4m3((x * (r * LO).astype(F32)).astype(F32)), e4m3((x * (r * HI).astype(F32)).astype(F32))
    want = e4m3((x / s).astype(F32))
    assert np.any((cl == ch) & (cl != want))
