"""Comparison rules shared by the parity tests.

Parity bar: codes, packed words and indices bit-exact, except a code may differ
from the oracle's by one cell where the oracle's normalised value lies within
1e-6 (relative, floor 1) of the threshold between the two cells (counted and
reported); an fp16 scale may differ by one ulp only where the oracle's fp64 RMS
lies within 1e-6 (relative) of an fp16 rounding midpoint (counted);
floating-point outputs within 2e-3 relative L2 of the oracle.
"""
from __future__ import annotations

import numpy as np

from oracle import tq_oracle as o

REL_L2 = 2e-3
TIE_REL = 1e-6


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    d = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (d if d > 0 else 1.0))


def u32(t) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32)


def f16_from_bits(t) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.float16)


def oracle_u(v_rot: np.ndarray, group: int) -> np.ndarray:
    """The oracle's normalised values u = v / RMS (0 for a zero group)."""
    rows, K = v_rot.shape
    s, _ = o.group_rms_scales(v_rot, group)
    g = v_rot.reshape(rows, K // group, group)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(s[:, :, None] > 0, g / s[:, :, None], 0.0)
    return u.reshape(rows, K), s


def compare_codes(gpu_words, oracle_words, levels, K, u, thresholds, what="codes"):
    """Words bit-exact except in words that hold a counted threshold tie. Returns the tie count."""
    gw = np.asarray(gpu_words, np.uint32)
    ow = np.asarray(oracle_words, np.uint32)
    assert gw.shape == ow.shape, (gw.shape, ow.shape)
    diff_rows = np.nonzero(np.any(gw != ow, axis=1))[0]
    ties = 0
    if len(diff_rows):
        gc = o.unpack(gw[diff_rows], levels, K)
        oc = o.unpack(ow[diff_rows], levels, K)
        r, c = np.nonzero(gc != oc)
        t = np.asarray(thresholds, np.float64)
        for rr, cc in zip(r, c):
            a, b = int(gc[rr, cc]), int(oc[rr, cc])
            assert abs(a - b) == 1, f"{what}: code {a} vs oracle {b} at row {diff_rows[rr]} col {cc}"
            uu = u[diff_rows[rr], cc]
            thr = t[min(a, b)]
            assert abs(uu - thr) <= TIE_REL * max(1.0, abs(uu)), \
                f"{what}: mismatch away from a tie: u={uu!r} threshold={thr!r} (row {diff_rows[rr]}, col {cc})"
            ties += 1
        # words that differ must differ only through those codes (padding identical)
        pad_g = gw[diff_rows][:, o.row_words(levels, K):]
        pad_o = ow[diff_rows][:, o.row_words(levels, K):]
        np.testing.assert_array_equal(pad_g, pad_o)
    return ties


def compare_scales(gpu_f16, oracle_f16, rms64, what="scales"):
    """fp16 scales equal except one-ulp differences at counted rounding midpoints."""
    g = np.asarray(gpu_f16, np.float16)
    ref = np.asarray(oracle_f16, np.float16)
    bad = np.nonzero(g.view(np.uint16) != ref.view(np.uint16))
    near = 0
    for idx in zip(*bad):
        gv, ov = g[idx], ref[idx]
        assert abs(int(gv.view(np.uint16)) - int(ov.view(np.uint16))) == 1, f"{what}: {gv} vs {ov} at {idx}"
        mid = (float(gv) + float(ov)) / 2
        assert abs(rms64[idx] - mid) <= TIE_REL * abs(mid), f"{what}: {gv} vs {ov} not at a midpoint ({rms64[idx]})"
        near += 1
    return near
