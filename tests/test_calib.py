"""The library's own calibration of the rotated-INT2 cache (host parts, no GPU): its
eigensolver, the up-projection-aware basis and the clip thresholds against the
oracle's fit (numpy's eigh with the same ascending order and sign rule) and against
properties the definitions fix (orthogonality, a diagonal ascending R^T Sigma R, the
clip rate)."""
import numpy as np
import pytest

import workloads
from oracle import int2 as oint2


@pytest.fixture(scope="module")
def mla():
    from mla_latent_kv_08_gb300 import build
    build.build()
    import mla_latent_kv_08_gb300 as m
    m.load_library()
    return m


def test_eigh_small_against_numpy(mla):
    rng = np.random.default_rng(0)
    for d in (1, 2, 3, 7, 64):
        A = rng.standard_normal((d, d))
        A = A @ A.T + 0.1 * np.eye(d)
        w, R64, R32 = mla.calib_eigh(A)
        ref = np.linalg.eigh(A)[0]
        assert np.all(np.diff(w) >= 0)
        np.testing.assert_allclose(w, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        assert np.abs(R64.T @ R64 - np.eye(d)).max() < 1e-12
        assert np.abs(R64.T @ A @ R64 - np.diag(w)).max() < 1e-10 * np.abs(w).max()
        # sign rule: the largest-magnitude entry of each column is positive
        assert np.all(R64[np.argmax(np.abs(R64), axis=0), np.arange(d)] > 0)
        np.testing.assert_array_equal(R32, R64.astype(np.float32))


def test_eigh_of_the_int2_calibration_matches_the_oracle_fit(mla):
    """Sigma of the INT2 workload's calibration law (512 dims): the same eigenvalues as
    the oracle to 1e-10 relative and the same R up to rounding (distinct eigenvalues)."""
    w0 = workloads.int2_rotated(4, B=1, H=8, len_range=(10, 20), n_calib=8192)
    S = oint2.latent_covariance(w0.calib)
    Rref, wref = oint2.fit_rotation(w0.calib)
    w, R64, _ = mla.calib_eigh(S)
    assert np.abs(w - wref).max() <= 1e-10 * np.abs(wref).max()
    assert np.abs(R64 - Rref).max() < 1e-8
    # a rotation with a repeated eigenvalue still diagonalises (any basis is correct)
    D = np.diag(np.array([1.0, 1.0, 2.0, 3.0]))
    w2, R2, _ = mla.calib_eigh(D)
    np.testing.assert_allclose(w2, [1, 1, 2, 3], atol=1e-15)
    assert np.abs(R2.T @ D @ R2 - np.diag(w2)).max() < 1e-15


def test_weighted_basis_matches_the_oracle(mla):
    rng = np.random.default_rng(1)
    r, H = 64, 4
    X = rng.standard_normal((4096, r)) * np.exp(rng.uniform(-1, 1, r))
    W_UK = rng.standard_normal((H, 16, r)) / 8
    W_UV = rng.standard_normal((H, r, 16)) / 8
    S = oint2.latent_covariance(X)
    M = oint2.projection_energy(W_UK, W_UV)
    Rref, wref = oint2.fit_rotation_weighted(X, W_UK, W_UV)
    w, R64, _ = mla.calib_eigh_weighted(S, M)
    assert np.abs(w - wref).max() <= 1e-10 * np.abs(wref).max()
    assert np.abs(R64 - Rref).max() < 1e-8
    # M = I: the weighted basis is the plain one
    w1, R1, _ = mla.calib_eigh_weighted(S, np.eye(r))
    _, Rp, _ = mla.calib_eigh(S)
    assert np.abs(R1 - Rp).max() < 1e-8


def test_thresholds_match_the_oracle_percentiles(mla):
    w0 = workloads.int2_rotated(4, B=1, H=8, len_range=(10, 20), n_calib=8192)
    R, _ = oint2.fit_rotation(w0.calib)
    ref = oint2.clip_thresholds(w0.calib, R).astype(np.float32)
    absY = np.abs(np.asarray(w0.calib, np.float64) @ R)
    clip = mla.calib_thresholds(absY.copy(), 32, 99.0)
    np.testing.assert_array_equal(clip, ref)
    # about 1 % of the calibration values lie above their group's threshold
    frac = np.mean(absY > np.repeat(clip.astype(np.float64), 32)[None, :])
    assert abs(frac - 0.01) < 0.001
    # pct = 0 / 100 give the minimum / maximum of each group
    lo = mla.calib_thresholds(absY.copy(), 32, 0.0)
    hi = mla.calib_thresholds(absY.copy(), 32, 100.0)
    np.testing.assert_array_equal(lo, absY.reshape(-1, 16, 32).transpose(1, 0, 2).reshape(16, -1).min(1).astype(np.float32))
    np.testing.assert_array_equal(hi, absY.reshape(-1, 16, 32).transpose(1, 0, 2).reshape(16, -1).max(1).astype(np.float32))
