"""Pins of the oracle's counter-based generator, stochastic rounding and
random Hadamard transform (CPU only)."""
import numpy as np
import pytest
import scipy.linalg
import scipy.stats

import oracle as o


# Known-answer vectors of Philox-4x32-10 published with the reference
# implementation of Salmon et al., "Parallel random numbers: as easy as 1, 2,
# 3" (SC'11): (counter, key) -> output.
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", PHILOX_KAT)
def test_philox_known_answers(ctr, key, want):
    assert tuple(int(v) for v in o.philox(ctr, key)) == want


def test_philox_uniformity_chi2():
    words = np.array([o.sr_word(1234, j, 0) for j in range(40000)], np.uint64)
    counts = np.bincount((words >> np.uint64(24)).astype(np.int64), minlength=256)
    _, p = scipy.stats.chisquare(counts)
    assert p > 1e-4


def test_sr_word_counter_mapping():
    seed = 0x0123456789ABCDEF
    for j in (0, 1, 2, 3, 4, 7, 1 << 33, (1 << 33) + 5):
        g = j >> 2
        out = o.philox((g & 0xFFFFFFFF, g >> 32, 1, 0), (seed & 0xFFFFFFFF, seed >> 32))
        assert o.sr_word(seed, j, 1) == out[j & 3]


# ------------------------------------------------------------------ RHT
def test_rht_unit_vectors_give_scaled_sylvester_columns():
    H = scipy.linalg.hadamard(16).astype(np.float64)  # Sylvester construction
    for signs in (0, 0xFFFF, 0xA5C3, o.rht_sign_mask(7)):
        s = np.array([-1.0 if (signs >> j) & 1 else 1.0 for j in range(16)])
        M = np.stack([o.rht16(np.eye(16, dtype=np.float32)[k], signs) for k in range(16)], axis=1)
        assert np.array_equal(M, 0.25 * H * s[None, :])
        assert np.array_equal(M @ M.T, np.eye(16))  # H H^T = 16 I


def test_rht_parseval_and_linearity():
    rng = np.random.default_rng(3)
    signs = o.rht_sign_mask(11)
    for _ in range(200):
        x = rng.standard_normal(16).astype(np.float32)
        v = o.rht16(x, signs).astype(np.float64)
        assert abs(np.sum(v * v) - np.sum(x.astype(np.float64) ** 2)) <= 1e-5 * np.sum(x.astype(np.float64) ** 2)


def test_rht_preserves_wgrad_with_shared_signs():
    """dW = dY^T X over M: the same random-sign transform applied to every
    16-run along M of both operands leaves it unchanged (orthonormal).  Small
    integer inputs keep every fp32 butterfly step exact."""
    rng = np.random.default_rng(5)
    Mtok, N, K = 64, 8, 6
    X = rng.integers(-8, 9, (Mtok, K)).astype(np.float32)
    dY = rng.integers(-8, 9, (Mtok, N)).astype(np.float32)
    signs = o.rht_sign_mask(99)

    def rht_cols(A):
        out = np.empty_like(A)
        for c in range(A.shape[1]):
            for m0 in range(0, A.shape[0], 16):
                out[m0:m0 + 16, c] = o.rht16(A[m0:m0 + 16, c], signs)
        return out

    ref = dY.astype(np.float64).T @ X.astype(np.float64)
    got = rht_cols(dY).astype(np.float64).T @ rht_cols(X).astype(np.float64)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ SR
def test_sr_exact_values_never_move():
    for mag in (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0):
        for r in (0, 1, 0xFFFFFFFF, 0x80000000):
            assert o.decode(o.E2M1, [o.sr_encode_e2m1(mag, r)])[0] == mag
            assert o.decode(o.E2M1, [o.sr_encode_e2m1(-mag, r)])[0] == -mag


def test_sr_threshold_extremes():
    # r >> 8 == 0 always rounds up when frac > 0
    assert o.sr_encode_e2m1(1.0000001, 0) == 3
    assert o.sr_encode_e2m1(4.5, 0xFF) == 7
    # r >> 8 == 2^24 - 1 rounds up only when frac > 1 - 2^-24
    top = 0xFFFFFFFF
    assert o.sr_encode_e2m1(np.nextafter(np.float32(1.5), np.float32(0)), top) == 2
    # fp32 below 6 has frac = 1 - 2^-22: r24 = 2^24 - 1 is not below 2^24 - 4
    assert o.sr_encode_e2m1(5.9999995, top) == 6
    # just below 0.5: frac = 1 - 2^-24, so frac * 2^24 = 2^24 - 1: only r24 <= 2^24 - 2 rounds up
    below_half = np.nextafter(np.float32(0.5), np.float32(0))
    assert o.sr_encode_e2m1(below_half, top) == 0
    assert o.sr_encode_e2m1(below_half, 0xFFFFFEFF) == 1
    assert o.sr_encode_e2m1(1.25, 0x7FFFFFFF) == 3  # frac 0.5, r24 = 2^23 - 1 < 2^23
    assert o.sr_encode_e2m1(1.25, 0x80000000) == 2  # r24 = 2^23, not < 2^23
    # beyond the range saturates; sign is kept
    assert o.sr_encode_e2m1(7.0, 0) == 7 and o.sr_encode_e2m1(-7.0, 0) == 15
    assert o.sr_encode_e2m1(np.nan, 0) == 7


@pytest.mark.parametrize("y", [0.3, 1.1, 2.7, -3.3, 5.2, 0.01])
def test_sr_is_unbiased(y):
    n = 200000
    rng = np.random.default_rng(17)
    rs = rng.integers(0, 2 ** 32, n, dtype=np.uint64)
    vals = o.decode(o.E2M1, np.array([o.sr_encode_e2m1(y, int(r)) for r in rs], np.uint8))
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    a = abs(np.float32(y))
    lo = mags[mags <= a].max()
    hi = mags[mags > a].min()
    sigma = (hi - lo) * 0.5 / np.sqrt(n)
    assert abs(vals.mean() - np.float32(y)) < 5 * sigma
    assert set(np.abs(vals)) <= {lo, hi}
