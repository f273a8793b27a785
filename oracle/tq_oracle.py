"""Plain fp64 CPU oracle for rotated-codebook (TurboQuant-style) quantization.

TEST INFRASTRUCTURE ONLY.  This module is the independent, slow, obviously
correct statement of what the CUDA library computes.  Only the test suite, the
smoke check in ``__graft_entry__`` and the ``cpu_baseline`` / ``--impl
reference`` legs of ``bench.py`` may import it.  The product path never calls
it, and it shares no code, tables or constants with the CUDA sources.

Every function cites the passage of the method it restates.  Page names used in
the citations:

* "How it works" -- manjunathshiva.github.io/turboquant-mlx/how-it-works,
  sections "Quantizing a weight, with no data", "The ternary tier (1.58 bits)",
  "Running a quantized layer", "The KV cache", "Configuration that converter
  and loader share".
* "Running a 1T-Parameter Model on a Laptop" -- your-ssd-is-a-gpu.vercel.app,
  sections on the MoE router, the Hadamard construction (create_hadamard_matrix)
  and the TurboQuant KV cache (update_and_fetch).

Readings taken where the pages are silent are listed in the docstrings and
collected in the design notes.  Floating-point work is fp64 throughout, except
where a float decides an integer: the nearest-centroid decision is taken in
fp32 (the precision the GPU kernels compute in), so both sides decide in the
same precision.

The dense QR-fallback rotation (``rotation_dense``) draws its Gaussian matrix
from SplitMix64 through the Box-Muller transform; the CUDA library implements
the same generator from its published definition on its own side.

Parity pins: every public function here is pinned by a ``-m "not gpu"`` test
against something other than itself (published tables, closed forms,
invariants, brute force).  No function is unpinned.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import ndtr  # standard normal CDF, a library primitive

# ---------------------------------------------------------------------------
# Codebook: Gaussian Lloyd-Max quantizer
# ---------------------------------------------------------------------------


def _phi(x):
    """Standard normal density; +-inf map to 0."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    fin = np.isfinite(x)
    out[fin] = np.exp(-0.5 * x[fin] ** 2) / math.sqrt(2.0 * math.pi)
    return out


def _cell_means(t_full):
    """E[X | t_{i-1} < X < t_i] for X ~ N(0,1), cells given by the edges t_full.

    Closed form of the truncated-normal mean: (phi(a) - phi(b)) / (Phi(b) - Phi(a)).
    """
    a, b = t_full[:-1], t_full[1:]
    # Cell mass without cancellation in the upper tail: Phi(b) - Phi(a) equals
    # Q(a) - Q(b) with Q(x) = Phi(-x), which keeps its digits for a > 0.
    mass = np.where(a > 0, ndtr(-a) - ndtr(-b), ndtr(b) - ndtr(a))
    return (_phi(a) - _phi(b)) / mass, mass


def lloyd_max_gaussian(levels: int, tol: float = 1e-15, max_newton: int = 100):
    """Gaussian Lloyd-Max codebook with ``levels`` reconstruction points.

    "How it works", section "Quantizing a weight, with no data", step "Snap to
    a codebook": the quantizer that minimises error for a Gaussian, one fixed
    codebook per bit width; section "The ternary tier" gives the three-level
    book {-c, 0, +c}.

    The Lloyd-Max quantizer is defined by its two stationarity conditions:
    every threshold is the midpoint of its two neighbouring centroids, and every
    centroid is the conditional mean of N(0,1) over its cell.  This solver runs
    Lloyd's alternation of those two conditions from equiprobable cells, then
    finishes with Newton steps on the same fixed-point equation (the Lloyd map
    converges slowly for many levels; Newton reaches the same unique fixed point,
    the Gaussian being log-concave).

    Returns (centroids[levels], thresholds[levels-1]) ascending, fp64.
    """
    L = int(levels)
    if L < 2:
        raise ValueError("levels must be >= 2")
    # Equiprobable cells, centroid = cell mean.
    q = np.array([_ndtri_bisect(i / L) for i in range(1, L)])
    c, _ = _cell_means(np.concatenate(([-np.inf], q, [np.inf])))

    def lloyd_map(cv):
        t = 0.5 * (cv[:-1] + cv[1:])
        m, _ = _cell_means(np.concatenate(([-np.inf], t, [np.inf])))
        return m

    for _ in range(200):
        c = lloyd_map(c)
    c = 0.5 * (c - c[::-1])
    for _ in range(max_newton):
        t = 0.5 * (c[:-1] + c[1:])
        t_full = np.concatenate(([-np.inf], t, [np.inf]))
        m, mass = _cell_means(t_full)
        resid = m - c
        if np.max(np.abs(resid)) <= tol:
            break
        # Jacobian of the Lloyd map: d m_i / d t_i = phi(t_i)(t_i - m_i)/P_i,
        # d m_i / d t_{i-1} = phi(t_{i-1})(m_i - t_{i-1})/P_i, d t_i/d c_i =
        # d t_i / d c_{i+1} = 1/2.
        J = np.zeros((L, L))
        for i in range(L):
            if i < L - 1:  # upper edge t_i = (c_i + c_{i+1})/2
                d = _phi(t_full[i + 1]) * (t_full[i + 1] - m[i]) / mass[i]
                J[i, i] += 0.5 * d
                J[i, i + 1] += 0.5 * d
            if i > 0:  # lower edge t_{i-1} = (c_{i-1} + c_i)/2
                d = _phi(t_full[i]) * (m[i] - t_full[i]) / mass[i]
                J[i, i - 1] += 0.5 * d
                J[i, i] += 0.5 * d
        step = np.linalg.solve(J - np.eye(L), -resid)
        c = c + step
        # N(0,1) is symmetric, so its (unique) Lloyd-Max quantizer is too:
        # c_i = -c_{L-1-i}.  Enforcing it exactly makes the middle threshold of
        # an even book exactly 0.
        c = 0.5 * (c - c[::-1])
    t = 0.5 * (c[:-1] + c[1:])
    return c, t


def _ndtri_bisect(p: float) -> float:
    """Inverse normal CDF by bisection (only used to seed the solver)."""
    lo, hi = -40.0, 40.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if ndtr(mid) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def codebook_distortion(centroids, thresholds) -> float:
    """Mean squared error E[(X - Q(X))^2] of a codebook for X ~ N(0,1).

    For a stationary (centroid-condition) quantizer this equals
    1 - sum_i P_i c_i^2.
    """
    t_full = np.concatenate(([-np.inf], np.asarray(thresholds, np.float64), [np.inf]))
    mass = ndtr(t_full[1:]) - ndtr(t_full[:-1])
    return float(1.0 - np.sum(mass * np.asarray(centroids, np.float64) ** 2))


# ---------------------------------------------------------------------------
# Rotation: seeded +-1 signs and Sylvester Hadamard blocks
# ---------------------------------------------------------------------------

_MASK64 = (1 << 64) - 1


def splitmix64_stream(seed: int, n: int):
    """First ``n`` outputs of SplitMix64 (Steele, Lea & Flood, OOPSLA 2014).

    The pages record only that the rotation is a d-length sign vector derived
    from a seed kept in the config ("How it works", section "Configuration that
    converter and loader share"); they name no generator.  SplitMix64 is the
    reading taken: the state advances by the golden-gamma constant once per
    output and each output is the published mix of the state.
    """
    s = seed & _MASK64
    out = []
    for _ in range(n):
        s = (s + 0x9E3779B97F4A7C15) & _MASK64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        z = z ^ (z >> 31)
        out.append(z)
    return out


def rotation_signs(seed: int, dim: int) -> np.ndarray:
    """Sign vector s[i] = -1 if the top bit of the i-th SplitMix64 output is set, else +1."""
    return np.array([-1 if (z >> 63) else 1 for z in splitmix64_stream(seed, dim)], dtype=np.int8)


def hadamard(n: int) -> np.ndarray:
    """Unnormalised Sylvester Hadamard matrix of order n (a power of two).

    "Running a 1T-Parameter Model on a Laptop", create_hadamard_matrix: start
    from [[1]] and double with [[H, H], [H, -H]].
    """
    if n < 1 or (n & (n - 1)) != 0:
        raise ValueError("order must be a power of two")
    H = np.ones((1, 1), dtype=np.float64)
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def rotation_block(dim: int) -> int:
    """Hadamard block size for an input dimension (a reading of the pages).

    The pages apply a Hadamard rotation along the input dimension and fall back
    to something else for dimensions a fast transform cannot take.  Reading: the
    rotation is block-diagonal with equal power-of-two Sylvester blocks, the
    block being the largest power of two that divides ``dim`` (7168 -> 1024,
    1536 -> 512, 4096 -> 4096).  This is exactly orthonormal for every dim.
    """
    return dim & (-dim)


def rotation_kind(dim: int) -> str:
    """Which rotation a layer of input dimension ``dim`` takes (a reading of the pages).

    The weight-reservoir page falls back from the fast Hadamard transform to a
    QR-derived dense rotation for dimensions the transform cannot take.  With
    the block-diagonal reading above every dim has a Hadamard rotation, but a
    block below 64 mixes too few values to make a group Gaussian; such dims
    (e.g. 400 = 16 x 25, odd dims) take the dense rotation.
    """
    return "hadamard" if rotation_block(dim) >= 64 else "dense"


def splitmix64_array(seed: int, n: int) -> np.ndarray:
    """The first ``n`` SplitMix64 outputs as a uint64 array (the stream of
    ``splitmix64_stream``, computed for all indices at once: state_i = seed + (i+1) gamma)."""
    with np.errstate(over="ignore"):
        i = np.arange(1, n + 1, dtype=np.uint64)
        z = np.uint64(seed & _MASK64) + i * np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def gaussian_stream(seed: int, n: int) -> np.ndarray:
    """``n`` standard normal draws from the SplitMix64 stream of ``seed`` by the Box-Muller transform
    (Box & Muller 1958).

    The pages derive a dense rotation from a seed (weight-reservoir page, the QR
    fallback) without naming the generator; the reading taken: draws 2p and 2p+1
    come from outputs 2p and 2p+1, u = (output >> 11) / 2^53 in [0, 1), and
    r = sqrt(-2 ln(1 - u_2p)), z_2p = r cos(2 pi u_2p+1), z_2p+1 = r sin(2 pi u_2p+1).
    """
    m = n + (n & 1)
    x = splitmix64_array(seed, m)
    u = (x >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    z = np.empty(m)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n]


def rotation_dense(seed: int, dim: int) -> np.ndarray:
    """Dense Haar-random rotation R [dim, dim] for the QR fallback.

    Weight-reservoir page: a rotation for a dimension the fast transform cannot
    take is derived from the seed by a QR decomposition (numpy.linalg.qr of a
    random matrix).  Reading: G[i, j] = gaussian_stream(seed)[i * dim + j], G = Q U
    with the diagonal of U made positive (the unique factorisation, which makes Q
    Haar-distributed), R = Q; x_rot = R x and W_rot = W R^T as for Hadamard layers.
    """
    G = gaussian_stream(seed, dim * dim).reshape(dim, dim)
    Q, U = np.linalg.qr(G)  # library primitive (LAPACK Householder)
    return Q * np.sign(np.diag(U))[None, :]


def rotation_matrix(signs: np.ndarray, block: int) -> np.ndarray:
    """Dense R = blockdiag(H_b, ..., H_b) . diag(signs) / sqrt(b).

    "How it works", section "Quantizing a weight, with no data", step
    "Randomized Hadamard rotation": multiply by a Hadamard matrix with random
    +-1 signs.  Reading: the signs act first (on the input), then H, then the
    1/sqrt(b) normalisation of the Sylvester construction.
    """
    d = len(signs)
    if d % block:
        raise ValueError("block must divide dim")
    H = hadamard(block) / math.sqrt(block)
    R = np.zeros((d, d))
    for j in range(d // block):
        R[j * block:(j + 1) * block, j * block:(j + 1) * block] = H
    return R * np.asarray(signs, np.float64)[None, :]


# ---------------------------------------------------------------------------
# Encode: group RMS, snap, pack
# ---------------------------------------------------------------------------


def codes_per_word(levels: int) -> int:
    """Codes per 32-bit word for a self-describing codebook size.

    "How it works", section "The ternary tier": 3 entries means trit-packed,
    20 trits per word in base 3; 2^b entries means bit-packed b bits per code
    (section "Quantizing a weight", step "Pack").  3-bit codes go 10 to a word
    (top two bits zero).
    """
    if levels == 3:
        return 20
    b = int(levels).bit_length() - 1
    if levels != (1 << b) or b < 1 or b > 8:
        raise ValueError("levels must be 3 or a power of two up to 256")
    return 32 // b


def bits_per_code(levels: int) -> int:
    return int(levels).bit_length() - 1


def row_words(levels: int, cols: int) -> int:
    """Words holding one row of ``cols`` codes (each row starts a fresh word)."""
    cw = codes_per_word(levels)
    return -(-cols // cw)


def snap(u, thresholds):
    """Nearest-centroid index of each normalised value u.

    "How it works", step "Snap to a codebook": replace each scaled weight by
    its nearest centroid.  With ascending centroids and midpoint thresholds,
    the nearest centroid's index is the number of thresholds strictly below u
    (a value exactly on a threshold goes to the lower cell).  The decision is
    taken in fp32, the GPU kernels' precision: u and the thresholds are
    rounded to fp32 before comparing.
    """
    u32 = np.asarray(u, dtype=np.float64).astype(np.float32)
    t32 = np.asarray(thresholds, dtype=np.float64).astype(np.float32)
    return np.searchsorted(t32, u32, side="left").astype(np.int64)


def group_rms_scales(v: np.ndarray, group: int):
    """Per-group RMS of rotated rows ``v`` [rows, K] (fp64) and its fp16 copy.

    "How it works", step "Group and scale": groups run along the input
    dimension and each group is divided by its root-mean-square.  Readings: the
    RMS divides by the group size; the stored scale is the fp16 rounding
    (round to nearest even) of the exact RMS, and the exact RMS (not the stored
    copy) is what the group is divided by.
    """
    rows, K = v.shape
    g = v.reshape(rows, K // group, group)
    s = np.sqrt(np.mean(g * g, axis=2))
    return s, s.astype(np.float16)


def encode_rotated(v: np.ndarray, group: int, thresholds) -> tuple[np.ndarray, np.ndarray]:
    """Codes and fp16 scales of already-rotated rows ``v`` [rows, K].

    An all-zero group has RMS 0; its values are taken as u = 0 (reading: the
    pages are silent), so they snap to the cell holding 0 and dequantize to 0.
    """
    rows, K = v.shape
    if K % group:
        raise ValueError("group must divide K")
    s, s16 = group_rms_scales(v, group)
    g = v.reshape(rows, K // group, group)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(s[:, :, None] > 0, g / s[:, :, None], 0.0)
    codes = snap(u.reshape(rows, K), thresholds)
    return codes, s16


def quantize(W: np.ndarray, signs: np.ndarray, block: int, group: int, thresholds):
    """Full encode of weight rows W [rows, K] (any float dtype, taken as fp64).

    "How it works", section "Quantizing a weight, with no data": rotate along
    the input dimension, group and scale, snap, (pack with ``pack``).  Rows are
    rotated as w_rot = R w, i.e. W_rot = W R^T, so that W x = W_rot (R x).
    """
    R = rotation_matrix(signs, block)
    v = np.asarray(W, np.float64) @ R.T
    return encode_rotated(v, group, thresholds)


def pack(codes: np.ndarray, levels: int, stride_words: int | None = None) -> np.ndarray:
    """Pack code rows [rows, K] into uint32 words [rows, stride_words].

    "How it works", step "Pack" (bit-packing into 32-bit words) and section
    "The ternary tier" (20 trits per word in base 3).  Readings: within a word,
    bit-packed code j sits at bits [b*j, b*j + b) (little-endian order); trit j
    is the base-3 digit of weight 3^j.  Each row starts a fresh word; unused
    slots and padding words are zero.
    """
    codes = np.asarray(codes, dtype=np.int64)
    rows, K = codes.shape
    cw = codes_per_word(levels)
    nw = -(-K // cw)
    stride = nw if stride_words is None else int(stride_words)
    if stride < nw:
        raise ValueError("stride too small")
    full = np.zeros((rows, nw * cw), dtype=np.int64)
    full[:, :K] = codes
    full = full.reshape(rows, nw, cw)
    words = np.zeros((rows, stride), dtype=np.uint64)
    if levels == 3:
        acc = np.zeros((rows, nw), dtype=np.uint64)
        for j in range(cw):
            acc += full[:, :, j].astype(np.uint64) * np.uint64(3 ** j)
    else:
        b = bits_per_code(levels)
        acc = np.zeros((rows, nw), dtype=np.uint64)
        for j in range(cw):
            acc |= full[:, :, j].astype(np.uint64) << np.uint64(b * j)
    words[:, :nw] = acc
    if np.any(words > 0xFFFFFFFF):
        raise AssertionError("word overflow")
    return words.astype(np.uint32)


def unpack(words: np.ndarray, levels: int, K: int) -> np.ndarray:
    """Inverse of ``pack``: uint32 words [rows, >= row_words] -> codes [rows, K]."""
    words = np.asarray(words, dtype=np.uint64)
    rows = words.shape[0]
    cw = codes_per_word(levels)
    nw = -(-K // cw)
    w = words[:, :nw]
    out = np.zeros((rows, nw, cw), dtype=np.int64)
    if levels == 3:
        rem = w.copy()
        for j in range(cw):
            out[:, :, j] = (rem % np.uint64(3)).astype(np.int64)
            rem //= np.uint64(3)
    else:
        b = bits_per_code(levels)
        m = np.uint64((1 << b) - 1)
        for j in range(cw):
            out[:, :, j] = ((w >> np.uint64(b * j)) & m).astype(np.int64)
    return out.reshape(rows, nw * cw)[:, :K]


def dequantize(codes: np.ndarray, scales16: np.ndarray, centroids, group: int) -> np.ndarray:
    """Rotated-domain weights W_rot_hat[n, k] = fp16 scale[n, k/g] * c[code[n, k]]."""
    c = np.asarray(centroids, np.float64)
    s = np.asarray(scales16, np.float16).astype(np.float64)
    return c[codes] * np.repeat(s, group, axis=1)


# ---------------------------------------------------------------------------
# Decode: rotate the input, multiply by the (dequantized) packed weights
# ---------------------------------------------------------------------------


def rotate(x: np.ndarray, signs: np.ndarray, block: int) -> np.ndarray:
    """x_rot = R x for each row of x [rows, K].

    "How it works", section "Running a quantized layer": the rotation is
    orthonormal, so the layer rotates its input instead of un-rotating W.
    """
    R = rotation_matrix(signs, block)
    return np.asarray(x, np.float64) @ R.T


def qmv(W_rot_hat: np.ndarray, x_rot: np.ndarray) -> np.ndarray:
    """y[t, n] = sum_k W_rot_hat[n, k] x_rot[t, k]   (dense quantized linear).

    "How it works", section "Running a quantized layer": multiply the rotated
    input by the packed weights (here, in the oracle, by their dequantized
    values: the reference dequantize-and-multiply the pages test against).
    """
    return np.asarray(x_rot, np.float64) @ np.asarray(W_rot_hat, np.float64).T


def gather_qmv(Wbank_rot_hat, ids: np.ndarray, x_rot: np.ndarray) -> np.ndarray:
    """y[t, j, :] = W_{ids[t, j]} x_rot[t]: every routed expert reads the shared input.

    "How it works", section "Running a quantized layer", table row "Decoding one
    token" (polar_gather_qmv).  ``Wbank_rot_hat(e)`` returns expert e's
    dequantized rotated weights [N, K].
    """
    T, k = ids.shape
    out = []
    for t in range(T):
        out.append([qmv(Wbank_rot_hat(int(ids[t, j])), x_rot[t:t + 1])[0] for j in range(k)])
    return np.array(out)


def multi_gather_qmv(Wbank_rot_hat, ids: np.ndarray, x_rot: np.ndarray) -> np.ndarray:
    """y[p] = W_{ids[p]} x_rot[p]: a different input for each (expert, input) pair.

    "How it works", table row "Prefill with a different input per expert"
    (polar_multi_gather_qmv).
    """
    return np.array([qmv(Wbank_rot_hat(int(e)), x_rot[p:p + 1])[0] for p, e in enumerate(ids)])


# ---------------------------------------------------------------------------
# Mixture-of-Experts glue
# ---------------------------------------------------------------------------


def route(logits: np.ndarray, k: int):
    """Top-k routing with softmax over the selected logits.

    "Running a 1T-Parameter Model on a Laptop": a router picks the 8 best of
    384 experts per token.  Readings: ties go to the lower expert id; the
    weights are a softmax over the k selected (fp32) logits, computed in fp64.
    Returns ids [T, k] (descending logit), probs [T, k].
    """
    logits = np.asarray(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), dtype=np.int64)
    probs = np.zeros((T, k))
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        ids[t] = order
        z = np.array([float(logits[t, e]) for e in order], np.float64)
        z = np.exp(z - z.max())
        probs[t] = z / z.sum()
    return ids, probs


def sort_pairs(ids: np.ndarray, n_experts: int):
    """Expert-sorted order of the (token, slot) pairs.

    "How it works", table row "A large batch sorted by expert".  Pair index
    f = t*k + j; pairs are ordered by (expert, f).  Returns perm [T*k] (the
    pair index at each sorted position) and offsets [E+1] (first sorted
    position of each expert).
    """
    flat = np.asarray(ids).reshape(-1)
    perm = np.array(sorted(range(len(flat)), key=lambda f: (int(flat[f]), f)), dtype=np.int64)
    counts = np.bincount(flat, minlength=n_experts)
    offsets = np.concatenate(([0], np.cumsum(counts))).astype(np.int64)
    return perm, offsets


def silu(x):
    return x / (1.0 + np.exp(-x))


def swiglu(gate_up: np.ndarray, inter: int) -> np.ndarray:
    """h = silu(gate) * up, with gate = first ``inter`` outputs and up = the rest.

    The SwiGLU between the gate/up and down projections of each expert
    (reading: the gate and up projections are stored stacked, gate first).
    """
    g = gate_up[..., :inter]
    u = gate_up[..., inter:2 * inter]
    return silu(g) * u


def combine(y: np.ndarray, probs: np.ndarray) -> np.ndarray:
    """out[t] = sum_j probs[t, j] * y[t, j]: the router-weighted sum of expert outputs."""
    return np.einsum("tj,tjn->tn", probs, y)


def gather_qmm(Wbank_rot_hat, x_rot_tokens: np.ndarray, perm: np.ndarray, offsets: np.ndarray, k: int,
               per_pair_input: bool = False) -> np.ndarray:
    """Expert-sorted batched gather-GEMM: Y[i] = W_{e(i)} x[src(i)] for sorted position i.

    "How it works", table row "A large batch sorted by expert": polar_gather_qmm,
    a batched gather-GEMM.  The input of sorted position i is the rotated token
    perm[i] // k (shared input) or, with ``per_pair_input``, row i of the
    sorted per-pair inputs.
    """
    E = len(offsets) - 1
    P = len(perm)
    out = None
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        W = Wbank_rot_hat(e)
        if per_pair_input:
            X = x_rot_tokens[lo:hi]
        else:
            X = x_rot_tokens[np.asarray(perm[lo:hi]) // k]
        Y = qmv(W, X)
        if out is None:
            out = np.zeros((P, W.shape[0]))
        out[lo:hi] = Y
    return out


def dequant_experts(Wbank_rot_hat, ids) -> np.ndarray:
    """Dense rotated-domain weights of the selected experts, [n, N, K].

    "How it works", table row "Anything else": polar_dequant_experts, then a
    regular matmul (reading: the output stays in the rotated domain and the
    caller multiplies it by the rotated input).
    """
    return np.array([Wbank_rot_hat(int(e)) for e in ids])


# ---------------------------------------------------------------------------
# KV cache
# ---------------------------------------------------------------------------


def kv_quantize(X: np.ndarray, signs: np.ndarray, group: int, thresholds):
    """Quantize cache vectors X [T, H, D] with one rotation shared by all heads.

    "How it works", section "The KV cache": the same rotation and codebook
    compress the cache at run time.  "Running a 1T-Parameter Model on a
    Laptop", update_and_fetch: rotate, then quantize each new key/value.
    Readings: each (token, head) vector of D is rotated by R_D (Hadamard of
    order D with the seeded signs), then encoded like a weight row with group
    RMS scales.  Returns codes [H, T, D] and fp16 scales [H, T, D/group].
    """
    T, H, D = X.shape
    R = rotation_matrix(signs, D)
    v = np.asarray(X, np.float64).reshape(T * H, D) @ R.T
    codes, s16 = encode_rotated(v, group, thresholds)
    codes = codes.reshape(T, H, D).transpose(1, 0, 2)
    s16 = s16.reshape(T, H, D // group).transpose(1, 0, 2)
    return codes, s16


def kv_attend(q: np.ndarray, K_rot_hat: np.ndarray, V_rot_hat: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """One decode step of attention over a rotated, dequantized cache.

    "Running a 1T-Parameter Model on a Laptop", update_and_fetch: dequantize
    the cache, de-rotate it with R^T, and hand full keys/values to attention
    softmax(q K^T / sqrt(D)) V.  Inputs: q [Hq, D]; K_rot_hat, V_rot_hat
    [Hkv, T, D] in the rotated domain.  Query head h reads kv head
    h // (Hq / Hkv) (grouped-query attention).  Returns o [Hq, D] (fp64).
    """
    Hq, D = q.shape
    Hkv, T, _ = K_rot_hat.shape
    R = rotation_matrix(signs, D)
    Kh = np.asarray(K_rot_hat, np.float64) @ R  # de-rotate: k = R^T k_rot (row form k_rot R)
    Vh = np.asarray(V_rot_hat, np.float64) @ R
    out = np.zeros((Hq, D))
    grp = Hq // Hkv
    for h in range(Hq):
        kv = h // grp
        s = Kh[kv] @ np.asarray(q[h], np.float64) / math.sqrt(D)
        s = np.exp(s - s.max())
        p = s / s.sum()
        out[h] = p @ Vh[kv]
    return out
