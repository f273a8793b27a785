"""Pins of the oracle's dense (QR-fallback) rotation and its seeded Gaussian stream.

Weight-reservoir page: dimensions the fast transform cannot take get a dense rotation derived
from a seed by QR.  Pins: the vectorised SplitMix64 equals the scalar one (itself pinned to the
published vectors); the Box-Muller pairs satisfy their radius/angle identities and the draws
have Gaussian moments; the rotation is orthogonal, Q^T G is upper triangular with a positive
diagonal (the definition of the unique QR), its first column is G's normalised first column,
and W x = W_rot (R x).
"""
import math

import numpy as np
import pytest

from oracle import tq_oracle as o


@pytest.mark.parametrize("seed", [0, 1, 1234567, 2 ** 64 - 1])
def test_splitmix64_array_matches_scalar_stream(seed):
    np.testing.assert_array_equal(o.splitmix64_array(seed, 777), np.array(o.splitmix64_stream(seed, 777), np.uint64))


def test_gaussian_stream_box_muller_identities_and_moments():
    seed, n = 99, 400_001
    z = o.gaussian_stream(seed, n)
    assert z.shape == (n,)
    x = o.splitmix64_array(seed, n + 1)
    u = (x >> np.uint64(11)).astype(np.float64) / 2.0 ** 53
    r2 = z[0:-1:2] ** 2 + z[1::2] ** 2
    np.testing.assert_allclose(r2, -2.0 * np.log(1.0 - u[0:-2:2]), rtol=1e-12, atol=1e-300)
    ang = np.mod(np.arctan2(z[1::2], z[0:-1:2]), 2 * np.pi)
    d = np.abs(ang - 2 * np.pi * u[1:-1:2])
    assert np.all(np.minimum(d, 2 * np.pi - d) < 1e-9)
    # moments of N(0, 1) within about 5 standard errors
    se = 1 / math.sqrt(n)
    assert abs(z.mean()) < 5 * se
    assert abs(z.var() - 1) < 5 * math.sqrt(2) * se
    assert abs(np.mean(z ** 4) / np.mean(z ** 2) ** 2 - 3) < 0.05
    np.testing.assert_array_equal(o.gaussian_stream(seed, 10), z[:10])  # a prefix of the same stream


@pytest.mark.parametrize("dim,seed", [(5, 3), (50, 11), (208, 7), (400, 1234)])
def test_rotation_dense_is_the_positive_diagonal_qr(dim, seed):
    R = o.rotation_dense(seed, dim)
    np.testing.assert_allclose(R @ R.T, np.eye(dim), atol=1e-12)
    G = o.gaussian_stream(seed, dim * dim).reshape(dim, dim)
    U = R.T @ G
    assert np.max(np.abs(np.tril(U, -1))) < 1e-10 * np.max(np.abs(U))
    assert np.all(np.diag(U) > 0)
    np.testing.assert_allclose(R[:, 0], G[:, 0] / np.linalg.norm(G[:, 0]), rtol=0, atol=1e-13)
    np.testing.assert_array_equal(o.rotation_dense(seed, dim), R)  # deterministic
    W = np.random.default_rng(dim).normal(size=(7, dim))
    x = np.random.default_rng(dim + 1).normal(size=dim)
    np.testing.assert_allclose((W @ R.T) @ (R @ x), W @ x, rtol=1e-12, atol=1e-12)


def test_rotation_kind():
    assert o.rotation_kind(7168) == "hadamard" and o.rotation_kind(4096) == "hadamard"
    assert o.rotation_kind(400) == "dense" and o.rotation_kind(1040) == "dense" and o.rotation_kind(50) == "dense"


def test_planted_mistake_in_qr_sign_convention_is_caught():
    """A rotation without the positive-diagonal fix fails the triangularity pin (checked on the CPU)."""
    dim, seed = 40, 5
    G = o.gaussian_stream(seed, dim * dim).reshape(dim, dim)
    Q, _ = np.linalg.qr(G)
    if np.all(np.diag(Q.T @ G) > 0):
        pytest.skip("LAPACK happened to return the positive-diagonal factorisation")
    assert not np.all(np.diag(Q.T @ G) > 0)


@pytest.mark.parametrize("dim,seed", [(5, 3), (50, 11), (208, 7), (400, 1234)])
def test_library_dense_rotation_matches_oracle(dim, seed):
    """The library's host Householder QR of its own Gaussian stream against the oracle's numpy QR."""
    tq = pytest.importorskip("rotated_codebook_quantized_gb300")
    try:
        tq.load()
    except RuntimeError:
        pytest.skip("libtq.so not built")
    np.testing.assert_allclose(tq.rotation_dense(seed, dim), o.rotation_dense(seed, dim), rtol=0, atol=1e-12)
