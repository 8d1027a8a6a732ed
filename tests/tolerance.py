"""Parity tolerances, written once and used by every GPU test.

The bound is a maximum relative error of 2e-3 against the fp64 oracle, with
the relative error of element i taken as |x_i - r_i| / max(|r_i|, tau) and
tau = 1e-2 * RMS(r), so that elements near zero are judged against the
tensor's scale rather than their own.

bf16 outputs: the unit roundoff of bf16 (2^-8 ~ 3.9e-3) is larger than 2e-3,
so the final rounding alone can exceed the bound.  For a bf16 tensor the test
is |x - r| <= 2e-3 * max(|r|, tau) + ulp_bf16(max(|r|, |x|)) / 2: the fp32
result must meet the bound, and rounding it to bf16 may add half a unit in
the last place.
"""
import numpy as np

REL_BOUND = 2e-3


def _tau(r: np.ndarray) -> float:
    return 1e-2 * float(np.sqrt(np.mean(r * r))) + 1e-30


def max_rel_err(x: np.ndarray, r: np.ndarray) -> float:
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if r.size == 0:
        return 0.0
    return float(np.max(np.abs(x - r) / np.maximum(np.abs(r), _tau(r))))


def ulp_bf16(a: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(np.asarray(a, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def assert_f32_close(x, r, what: str, bound: float = REL_BOUND) -> float:
    e = max_rel_err(x, r)
    assert e <= bound, f"{what}: max relative error {e:.3e} > {bound:.1e}"
    return e


def assert_bf16_close(x, r, what: str, bound: float = REL_BOUND) -> float:
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    allowed = bound * np.maximum(np.abs(r), _tau(r)) + 0.5 * ulp_bf16(np.maximum(np.abs(r), np.abs(x)))
    bad = np.abs(x - r) > allowed
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {x.size} elements outside tolerance; "
                           f"worst |x-r|={np.max(np.abs(x - r)):.3e}")
    return max_rel_err(x, r)


def assert_act_close(x, r, act: str, what: str) -> float:
    return assert_bf16_close(x, r, what) if act == "bf16" else assert_f32_close(x, r, what)
