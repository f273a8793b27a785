"""Pins of the fp64 oracle against things other than itself.

Each test ties an oracle function to a published table, a closed form, an
invariant or a brute-force evaluation, chosen so that a plausible slip (a
dropped term, a wrong sign or index, a transposed operand) fails at least one
of them.  No GPU is involved.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy import integrate

from oracle import tq_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- codebook

@pytest.mark.parametrize("L", [2, 3, 4, 8, 16])
def test_codebook_matches_published_table(L):
    """Max (1960) Table I: optimum N(0,1) quantizer outputs, thresholds and MSE."""
    g = json.load(open(os.path.join(GOLDEN, "lloyd_max_gaussian.json")))
    book = g["books"][str(L)]
    tol = g["tolerance_abs"]
    c, t = o.lloyd_max_gaussian(L)
    pos_c = c[c >= 0] if L % 2 else c[L // 2:]
    pos_t = t[t >= 0]
    np.testing.assert_allclose(pos_c, book["outputs"], atol=tol)
    np.testing.assert_allclose(pos_t, book["thresholds"], atol=tol)
    assert abs(o.codebook_distortion(c, t) - book["mse"]) < 2e-5 + 1e-3 * book["mse"]


@pytest.mark.parametrize("L", [2, 3, 4, 8, 16, 256])
def test_codebook_is_stationary_by_quadrature(L):
    """Centroid condition checked by numerical integration (not the closed form used inside)."""
    c, t = o.lloyd_max_gaussian(L)
    edges = np.concatenate(([-np.inf], t, [np.inf]))
    pdf = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    for i in range(L):
        a, b = max(edges[i], -40.0), min(edges[i + 1], 40.0)
        m0 = integrate.quad(pdf, a, b, epsabs=0, epsrel=1e-13, limit=200)[0]
        m1 = integrate.quad(lambda x: x * pdf(x), a, b, epsabs=1e-15, epsrel=1e-13, limit=200)[0]
        assert abs(m1 / m0 - c[i]) < 1e-9 * max(1.0, abs(c[i])), (L, i, m1 / m0, c[i])
    np.testing.assert_array_equal(t, 0.5 * (c[:-1] + c[1:]))


@pytest.mark.parametrize("L", [2, 3, 4, 8, 16, 256])
def test_codebook_symmetric_and_ordered(L):
    c, t = o.lloyd_max_gaussian(L)
    assert np.all(np.diff(c) > 0) and np.all(np.diff(t) > 0)
    np.testing.assert_array_equal(c, -c[::-1])
    if L % 2 == 0:
        assert t[L // 2 - 1] == 0.0
    else:
        assert c[L // 2] == 0.0


@pytest.mark.parametrize("L", [3, 8, 16])
def test_distortion_formula_by_quadrature(L):
    c, t = o.lloyd_max_gaussian(L)
    edges = np.concatenate(([-40.0], t, [40.0]))
    pdf = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    mse = sum(integrate.quad(lambda x, ci=ci: (x - ci) ** 2 * pdf(x), edges[i], edges[i + 1], epsrel=1e-12)[0]
              for i, ci in enumerate(c))
    assert abs(mse - o.codebook_distortion(c, t)) < 1e-12


def test_ternary_book_is_affine():
    """The three-level book is {-c, 0, +c} ("The ternary tier")."""
    c, _ = o.lloyd_max_gaussian(3)
    assert c[1] == 0.0 and c[2] == -c[0] and c[2] - c[1] == c[1] - c[0]


# ---------------------------------------------------------------- signs

def test_splitmix64_published_vectors():
    # Seed 0: outputs widely reproduced from the reference splitmix64.c.
    assert o.splitmix64_stream(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # Seed 1234567: the Rosetta Code "Pseudo-random numbers/Splitmix64" task vector.
    assert o.splitmix64_stream(1234567, 5) == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                                               4593380528125082431, 16408922859458223821]


def test_signs_are_top_bits():
    s = o.rotation_signs(1234567, 5)
    # top bits of the vector above: 6457.. < 2^63, 3203.. < 2^63, 9817.. >= 2^63, 4593.. < 2^63, 16408.. >= 2^63
    np.testing.assert_array_equal(s, [1, 1, -1, 1, -1])
    big = o.rotation_signs(7, 1 << 14)
    assert abs(int(big.astype(np.int64).sum())) < 5 * math.sqrt(1 << 14)


# ---------------------------------------------------------------- Hadamard / rotation

@pytest.mark.parametrize("n", [1, 2, 4, 8, 64, 256])
def test_hadamard_closed_form(n):
    """Sylvester order: H[i, j] = (-1)^popcount(i & j)."""
    H = o.hadamard(n)
    ref = np.array([[(-1) ** bin(i & j).count("1") for j in range(n)] for i in range(n)], dtype=np.float64)
    np.testing.assert_array_equal(H, ref)
    np.testing.assert_array_equal(H @ H.T, n * np.eye(n))


def test_rotation_block_reading():
    assert o.rotation_block(7168) == 1024
    assert o.rotation_block(1536) == 512
    assert o.rotation_block(4096) == 4096
    assert o.rotation_block(2048) == 2048
    assert o.rotation_block(128) == 128


@pytest.mark.parametrize("dim,block", [(512, 512), (7168 // 4, 256), (1536, 512)])
def test_rotation_orthonormal_and_equivariant(dim, block):
    signs = o.rotation_signs(11, dim)
    R = o.rotation_matrix(signs, block)
    assert np.max(np.abs(R @ R.T - np.eye(dim))) <= 1e-15
    g = np.random.default_rng(0)
    W = g.normal(size=(7, dim))
    x = g.normal(size=(3, dim))
    W_rot = W @ R.T
    lhs = x @ W.T
    rhs = o.rotate(x, signs, block) @ W_rot.T
    assert np.linalg.norm(lhs - rhs) / np.linalg.norm(lhs) <= 1e-13


def test_rotation_sign_side():
    """Signs act on the input before H: column j of R is sign_j times column j of H/sqrt(b)."""
    signs = np.array([1, -1, -1, 1], dtype=np.int8)
    R = o.rotation_matrix(signs, 4)
    e1 = np.array([0.0, 1.0, 0.0, 0.0])
    np.testing.assert_array_equal(R @ e1, -np.array([1.0, -1.0, 1.0, -1.0]) / 2)


def test_kurtosis_drops_after_rotation():
    """Outlier-laden rows become near-Gaussian after rotation (sanity, cf. 27.7 -> 3.2)."""
    g = np.random.default_rng(3)
    W = g.normal(0, 0.02, size=(256, 1024))
    W[g.random(W.shape) < 0.01] *= 30.0
    kurt = lambda a: float(np.mean((a - a.mean()) ** 4) / np.var(a) ** 2)
    before = kurt(W)
    after = kurt(W @ o.rotation_matrix(o.rotation_signs(1, 1024), 1024).T)
    assert before > 20 and abs(after - 3.0) < 0.3


# ---------------------------------------------------------------- packing

def test_pack_known_words():
    # 4-bit: code j at bits [4j, 4j+4)
    w = o.pack(np.array([[1, 2, 3, 4, 5, 6, 7, 8, 9]]), 16)
    assert w.tolist() == [[0x87654321, 0x9]]
    # 3-bit: 10 codes per word, top two bits zero
    w = o.pack(np.array([[7] * 10 + [1]]), 8)
    assert w.tolist() == [[0x3FFFFFFF, 1]]
    # 2-bit: 16 codes per word
    assert o.pack(np.array([[3] * 16]), 4).tolist() == [[0xFFFFFFFF]]
    # 8-bit: 4 codes per word
    assert o.pack(np.array([[0x11, 0x22, 0x33, 0x44, 0xFF]]), 256).tolist() == [[0x44332211, 0xFF]]
    # ternary: trit j has weight 3^j; the all-twos word is 3^20 - 1 < 2^32
    assert o.pack(np.array([[1, 2]]), 3).tolist() == [[7]]
    allmax = o.pack(np.full((1, 20), 2), 3)
    assert int(allmax[0, 0]) == 3 ** 20 - 1 == 3486784400 < 2 ** 32
    # padding: stride larger than needed leaves zero words
    assert o.pack(np.array([[1]]), 16, stride_words=4).tolist() == [[1, 0, 0, 0]]


@pytest.mark.parametrize("L", [2, 3, 4, 8, 16, 256])
@pytest.mark.parametrize("K", [1, 19, 20, 21, 64, 333])
def test_pack_unpack_roundtrip(L, K):
    g = np.random.default_rng(L * 1000 + K)
    codes = g.integers(0, L, size=(5, K))
    words = o.pack(codes, L)
    assert words.shape == (5, o.row_words(L, K))
    np.testing.assert_array_equal(o.unpack(words, L, K), codes)


def test_codes_per_word():
    assert [o.codes_per_word(L) for L in (2, 3, 4, 8, 16, 256)] == [32, 20, 16, 10, 8, 4]


# ---------------------------------------------------------------- snap / encode

@pytest.mark.parametrize("L", [3, 4, 8, 16, 256])
def test_snap_is_nearest_centroid(L):
    c, t = o.lloyd_max_gaussian(L)
    c32 = c.astype(np.float32).astype(np.float64)
    g = np.random.default_rng(L)
    u = np.concatenate([g.normal(size=4000) * 1.5, t.astype(np.float32), [0.0, -0.0, 50.0, -50.0]])
    idx = o.snap(u, t)
    u32 = u.astype(np.float32).astype(np.float64)
    t32 = t.astype(np.float32).astype(np.float64)
    for k, uk in enumerate(u32):
        # brute force: the lowest index whose cell holds uk, cells (t_{i-1}, t_i]
        i = 0
        while i < L - 1 and not (uk <= t32[i]):
            i += 1
        assert idx[k] == i
        # and it is a nearest centroid (up to the fp32 rounding of the thresholds)
        d = np.abs(uk - c32)
        assert d[idx[k]] <= d.min() + 1e-6


def test_snap_tie_goes_low():
    c, t = o.lloyd_max_gaussian(8)
    assert o.snap(np.array([t[3]]), t)[0] == 3  # exactly on threshold 3 -> cell 3 (lower)
    assert o.snap(np.array([np.nextafter(np.float32(t[3]), np.float32(9))]), t)[0] == 4


def test_encode_brute_force_tiny():
    """Encode of a few rotated rows, redone with plain Python loops."""
    L, G = 8, 8
    c, t = o.lloyd_max_gaussian(L)
    g = np.random.default_rng(5)
    v = g.normal(size=(3, 32))
    v[1, 8:16] = 0.0  # an all-zero group
    codes, s16 = o.encode_rotated(v, G, t)
    for r in range(3):
        for gi in range(32 // G):
            vals = [float(x) for x in v[r, gi * G:(gi + 1) * G]]
            s = math.sqrt(sum(x * x for x in vals) / G)
            assert s16[r, gi] == np.float16(s)
            for j, x in enumerate(vals):
                u = x / s if s > 0 else 0.0
                u32 = float(np.float32(u))
                best = min(range(L), key=lambda i: (abs(u32 - float(np.float32(c[i]))), i))
                assert codes[r, gi * G + j] == best
    assert np.all(o.dequantize(codes, s16, c, G)[1, 8:16] == 0.0)


@pytest.mark.parametrize("L", [3, 8, 16])
def test_encode_mse_near_codebook_distortion(L):
    """On Gaussian data the normalised snap error approaches the book's distortion."""
    c, t = o.lloyd_max_gaussian(L)
    g = np.random.default_rng(9)
    v = g.normal(size=(64, 4096))
    codes, _ = o.encode_rotated(v, 4096, t)
    s = np.sqrt(np.mean(v * v, axis=1, keepdims=True))
    err = np.mean((v / s - c[codes]) ** 2)
    assert abs(err - o.codebook_distortion(c, t)) < 0.03 * o.codebook_distortion(c, t)


def test_quantize_equals_rotate_then_encode():
    W, x = (np.random.default_rng(1).normal(size=(4, 256)), None)
    signs = o.rotation_signs(3, 256)
    c, t = o.lloyd_max_gaussian(16)
    a = o.quantize(W, signs, 256, 64, t)
    b = o.encode_rotated(W @ o.rotation_matrix(signs, 256).T, 64, t)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------- qmv family

def _tiny_layer(L=16, N=24, K=128, G=32, seed=0):
    g = np.random.default_rng(seed)
    W = g.normal(0, 0.02, size=(N, K))
    signs = o.rotation_signs(seed + 1, K)
    c, t = o.lloyd_max_gaussian(L)
    codes, s16 = o.quantize(W, signs, K, G, t)
    return W, signs, c, t, codes, s16


def test_qmv_is_dequantize_then_matmul():
    """y = W_rot_hat (R x) equals (W_rot_hat R) x: the reference dequantize-and-multiply."""
    W, signs, c, t, codes, s16 = _tiny_layer()
    x = np.random.default_rng(2).normal(size=(3, 128))
    What = o.dequantize(codes, s16, c, 32)
    y = o.qmv(What, o.rotate(x, signs, 128))
    R = o.rotation_matrix(signs, 128)
    W_back = What @ R  # un-rotated dequantized weights
    y2 = np.array([[sum(W_back[n, k] * x[tt, k] for k in range(128)) for n in range(24)] for tt in range(3)])
    assert np.max(np.abs(y - y2)) <= 1e-12 * np.max(np.abs(y2))
    # and it approximates the unquantized layer within the 4-bit book's error
    rel = np.linalg.norm(y - x @ W.T) / np.linalg.norm(x @ W.T)
    assert rel < 0.2


def test_gather_and_multi_gather_by_loops():
    banks = [_tiny_layer(L=3, N=8, K=64, G=16, seed=s) for s in range(4)]
    signs = banks[0][1]
    Wh = [o.dequantize(b[4], b[5], b[2], 16) for b in banks]
    bank = lambda e: Wh[e]
    x = np.random.default_rng(7).normal(size=(2, 64))
    xr = o.rotate(x, signs, 64)
    ids = np.array([[3, 1], [0, 3]])
    y = o.gather_qmv(bank, ids, xr)
    for tt in range(2):
        for j in range(2):
            ref = [sum(Wh[ids[tt, j]][n, k] * xr[tt, k] for k in range(64)) for n in range(8)]
            np.testing.assert_allclose(y[tt, j], ref, rtol=1e-12, atol=1e-14)
    pe = np.array([2, 2, 0])
    xp = np.random.default_rng(8).normal(size=(3, 64))
    ym = o.multi_gather_qmv(bank, pe, xp)
    for p in range(3):
        np.testing.assert_allclose(ym[p], [float(np.dot(Wh[pe[p]][n], xp[p])) for n in range(8)], rtol=1e-12)


# ---------------------------------------------------------------- MoE glue

def test_route_brute_force_with_ties():
    logits = np.array([[0.5, 2.0, 2.0, -1.0, 2.0, 0.1],
                       [1.0, 1.0, 1.0, 1.0, 1.0, 1.0]], dtype=np.float32)
    ids, p = o.route(logits, 3)
    assert ids.tolist() == [[1, 2, 4], [0, 1, 2]]
    np.testing.assert_allclose(p, np.full((2, 3), 1 / 3), rtol=1e-15)
    g = np.random.default_rng(0)
    lg = g.normal(size=(5, 16)).astype(np.float32)
    ids, p = o.route(lg, 4)
    for tt in range(5):
        best = sorted(itertools.combinations(range(16), 4), key=lambda s: -sum(float(lg[tt, e]) for e in s))[0]
        assert set(ids[tt]) == set(best)
        z = np.exp(lg[tt, ids[tt]].astype(np.float64))
        np.testing.assert_allclose(p[tt], z / z.sum(), rtol=1e-13)
        assert all(lg[tt, ids[tt][i]] >= lg[tt, ids[tt][i + 1]] for i in range(3))


def test_sort_pairs_stable():
    ids = np.array([[2, 0], [0, 2], [1, 2]])
    perm, off = o.sort_pairs(ids, 4)
    assert perm.tolist() == [1, 2, 4, 0, 3, 5]
    assert off.tolist() == [0, 2, 3, 6, 6]


def test_swiglu_and_combine_closed_form():
    gu = np.array([[0.0, 1.0, 3.0, 4.0]])  # gate = [0, 1], up = [3, 4]
    h = o.swiglu(gu, 2)
    np.testing.assert_allclose(h, [[0.0, 4.0 / (1.0 + math.exp(-1.0))]], rtol=1e-15)
    y = np.arange(12, dtype=np.float64).reshape(1, 3, 4)
    p = np.array([[0.5, 0.25, 0.25]])
    np.testing.assert_allclose(o.combine(y, p), [[0.5 * y[0, 0] + 0.25 * y[0, 1] + 0.25 * y[0, 2]][0]])


def test_gather_qmm_by_loops():
    banks = [_tiny_layer(L=8, N=6, K=32, G=16, seed=s) for s in range(3)]
    Wh = [o.dequantize(b[4], b[5], b[2], 16) for b in banks]
    ids = np.array([[2, 0], [0, 1], [2, 1]])
    perm, off = o.sort_pairs(ids, 3)
    x = np.random.default_rng(4).normal(size=(3, 32))
    Y = o.gather_qmm(lambda e: Wh[e], x, perm, off, 2)
    for i, f in enumerate(perm):
        e = ids.reshape(-1)[f]
        np.testing.assert_allclose(Y[i], Wh[e] @ x[f // 2], rtol=1e-13)
    D = o.dequant_experts(lambda e: Wh[e], [1, 2])
    np.testing.assert_array_equal(D[1], Wh[2])


# ---------------------------------------------------------------- KV cache

def test_kv_attend_without_quantization_is_textbook_attention():
    g = np.random.default_rng(1)
    Hq, Hkv, T, D = 8, 2, 37, 16
    q = g.normal(size=(Hq, D))
    k = g.normal(size=(T, Hkv, D))
    v = g.normal(size=(T, Hkv, D))
    signs = o.rotation_signs(5, D)
    R = o.rotation_matrix(signs, D)
    k_rot = (k.reshape(-1, D) @ R.T).reshape(T, Hkv, D).transpose(1, 0, 2)
    v_rot = (v.reshape(-1, D) @ R.T).reshape(T, Hkv, D).transpose(1, 0, 2)
    out = o.kv_attend(q, k_rot, v_rot, signs)
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        s = np.array([float(np.dot(q[h], k[tt, kv])) for tt in range(T)]) / math.sqrt(D)
        p = np.exp(s - s.max())
        p /= p.sum()
        ref = sum(p[tt] * v[tt, kv] for tt in range(T))
        np.testing.assert_allclose(out[h], ref, rtol=1e-12, atol=1e-13)


def test_kv_quantize_layout():
    g = np.random.default_rng(2)
    X = g.normal(size=(5, 3, 32))
    signs = o.rotation_signs(1, 32)
    c, t = o.lloyd_max_gaussian(8)
    codes, s16 = o.kv_quantize(X, signs, 8, t)
    assert codes.shape == (3, 5, 32) and s16.shape == (3, 5, 4)
    v = X[4, 2] @ o.rotation_matrix(signs, 32).T
    c2, s2 = o.encode_rotated(v[None], 8, t)
    np.testing.assert_array_equal(codes[2, 4], c2[0])
    np.testing.assert_array_equal(s16[2, 4], s2[0])


# ---------------------------------------------------------------- planted mistakes

def test_planted_hadamard_transpose_or_sign_is_caught(monkeypatch):
    """A Hadamard with one flipped entry fails the closed-form pin."""
    good = o.hadamard

    def bad(n):
        H = good(n).copy()
        if n >= 4:
            H[1, 2] = -H[1, 2]
        return H

    monkeypatch.setattr(o, "hadamard", bad)
    with pytest.raises(AssertionError):
        test_hadamard_closed_form(8)


def test_planted_snap_tie_rule_is_caught(monkeypatch):
    """Sending threshold ties to the upper cell fails the brute-force snap pin."""
    def bad_snap(u, thresholds):
        u32 = np.asarray(u, np.float64).astype(np.float32)
        return np.searchsorted(np.asarray(thresholds).astype(np.float32), u32, side="right").astype(np.int64)

    monkeypatch.setattr(o, "snap", bad_snap)
    with pytest.raises(AssertionError):
        test_snap_tie_goes_low()


def test_planted_codebook_drift_is_caught(monkeypatch):
    """A book solved to the wrong fixed point (one centroid shifted) fails quadrature."""
    good = o.lloyd_max_gaussian

    def bad(L, **kw):
        c, t = good(L, **kw)
        c = c.copy()
        c[-1] += 1e-4
        return c, 0.5 * (c[:-1] + c[1:])

    monkeypatch.setattr(o, "lloyd_max_gaussian", bad)
    with pytest.raises(AssertionError):
        test_codebook_is_stationary_by_quadrature(8)
