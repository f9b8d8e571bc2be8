"""The decode kernel's start-up arithmetic, checked on the CPU.

The kernel splits its granules over CTAs with floor(U c / N) and locates each
CTA's first unit by a quotient and remainder.  Below 2^22 it divides with a
float reciprocal instead of the integer-division sequence (udiv_fast in
decode.cu): the exact operand times a reciprocal of d within one ulp, rounded
toward zero, is within one of the quotient, and one remainder step corrects
it.  This test replays that step with every reciprocal the bound allows (the
float32 values within one ulp of 1/d) and checks the exact quotient comes out.
"""
import numpy as np
import pytest


def _recips_within_one_ulp(d):
    exact = 1.0 / np.float64(d)
    f = np.float32(exact)
    cands = {f, np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(np.inf))}
    out = []
    for c in cands:
        ulp = np.float64(np.spacing(np.float32(abs(c))))
        if abs(np.float64(c) - exact) <= ulp:
            out.append(np.float32(c))
    assert out
    return out


def _mul_rz(a, r):
    exact = a.astype(np.float64) * np.float64(r)  # a < 2^22, r 24 bits: exact in fp64
    f = exact.astype(np.float32)
    over = np.abs(f.astype(np.float64)) > np.abs(exact)
    f[over] = np.nextafter(f[over], np.float32(0))
    return f


def udiv_fast_model(a, d, r):
    """The kernel's steps for a < 2^22, d < 2^22, with the reciprocal r."""
    q = np.trunc(_mul_rz(a, r)).astype(np.int64)
    rem = a.astype(np.int64) - q * d
    q = np.where(rem < 0, q - 1, np.where(rem >= d, q + 1, q))
    return q


@pytest.mark.parametrize("d", list(range(1, 300)) + [607, 1023, 1024, 1025, 4095, 65535, 65536, 1 << 21,
                                                     (1 << 22) - 1])
def test_udiv_fast_exact_for_every_allowed_reciprocal(d):
    rng = np.random.default_rng(d)
    lim = 1 << 22
    a = np.concatenate([np.arange(0, 3000), rng.integers(0, lim, 20000), lim - 1 - np.arange(64),
                        (np.arange(1, 200) * d).clip(0, lim - 1), (np.arange(1, 200) * d - 1).clip(0, lim - 1)])
    a = a[a < lim].astype(np.int64)
    for r in _recips_within_one_ulp(d):
        q = udiv_fast_model(a, d, r)
        assert np.array_equal(q, a // d), f"d={d} r={r!r}"


def split_point_model(U, c, N):
    """The kernel's 32-bit form of floor(U c / N) for U < 2^31."""
    q, r = U // N, U % N
    return q * c + (r * c) // N


def test_split_points_cover_the_granules_once():
    rng = np.random.default_rng(0)
    for _ in range(3000):
        N = int(rng.integers(1, 400))
        U = int(rng.integers(1, 1 << 31)) if rng.random() < 0.5 else int(rng.integers(1, 5000))
        Nw = min(U, N)
        cuts = [split_point_model(U, c, Nw) for c in range(Nw + 1)]
        assert cuts == [U * c // Nw for c in range(Nw + 1)]
        assert cuts[0] == 0 and cuts[-1] == U and all(b > a for a, b in zip(cuts, cuts[1:]))
