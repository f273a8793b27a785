"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Both sides take identical seeded inputs from the workload generators and
compute independently.  Sizes are small enough for the oracle to finish in
seconds but span several row tiles, several column steps and a ragged tail.
"""
import math

import numpy as np
import pytest

from oracle import tq_oracle as o
from rotated_codebook_quantized_gb300 import workloads as wl
from tests.helpers import REL_L2, compare_codes, compare_scales, f16_from_bits, oracle_u, rel_l2, u32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def test_trit_decoder_exhaustive(lib):
    """Every word below 3^20: the divide-free digit decoder equals plain division."""
    assert lib.selftest_trit_decode(0, 3 ** 20) == 0


def test_host_codebook_and_signs_match_oracle(lib):
    for L in (2, 3, 4, 8, 16, 256):
        c, t = lib.codebook(L)
        oc, ot = o.lloyd_max_gaussian(L)
        # The 256-level fixed point is ill-conditioned (the Lloyd map contracts by
        # about 1 - O(1/L^2)), so two converged solvers agree to ~1e-12, not 1e-15;
        # the fp32 tables the kernels use must agree exactly.
        tol = 1e-10 if L == 256 else 1e-12
        np.testing.assert_allclose(c, oc, rtol=0, atol=tol)
        np.testing.assert_allclose(t, ot, rtol=0, atol=tol)
        np.testing.assert_array_equal(c.astype(np.float32), oc.astype(np.float32))
        np.testing.assert_array_equal(t.astype(np.float32), ot.astype(np.float32))
    np.testing.assert_array_equal(lib.rotation_signs(4001, 4096), o.rotation_signs(4001, 4096))


@pytest.mark.parametrize("dim,block,rows,xdt", [(512, 512, 3, "f32"), (7168, 1024, 2, "bf16"), (1536, 512, 5, "bf16"),
                                                (128, 128, 33, "f32"), (4096, 4096, 1, "bf16"), (2048, 2048, 4, "f32"),
                                                (576, 64, 3, "f32"), (1280, 256, 2, "bf16"), (16384, 8192, 1, "f32")])
def test_rotate(lib, dim, block, rows, xdt):
    x = wl.rng(1, dim).normal(size=(rows, dim)).astype(np.float32)
    if xdt == "bf16":
        bits, x = wl.to_bf16(x)
        xd = _bf16_dev(bits)
    else:
        xd = _dev(x)
    rot = lib.Rotation(dim, block, seed=7)
    got = lib.rotate(xd, rot).cpu().numpy()
    ref = o.rotate(x, o.rotation_signs(7, dim), block)
    assert rel_l2(got, ref) < 1e-6


# (levels, group, K, block, rows, wdtype)
QCASES = [
    (16, 64, 512, 512, 512, "f32"),     # dense tiny (full size)
    (8, 128, 4096, 4096, 300, "bf16"),  # dense decode rows, ragged row tail
    (3, 16, 7168, 1024, 70, "bf16"),    # ternary experts, gate/up shape
    (3, 16, 2048, 2048, 96, "bf16"),    # ternary experts, down shape
    (8, 64, 1536, 512, 45, "bf16"),     # 3-bit group 64, three Hadamard blocks
    (4, 32, 1024, 256, 40, "f32"),      # 2-bit
    (3, 32, 640, 128, 33, "f32"),       # ternary group 32
    (3, 128, 1280, 256, 20, "f32"),     # ternary group 128
    (16, 16, 96, 32, 65, "f32"),        # 4-bit group 16, K not a multiple of the step
    (8, 32, 160, 32, 9, "f32"),         # 3-bit group 32, one ragged step
]


def _weights(levels, K, rows, wdt, seed):
    if levels == 16 and K == 512 and rows == 512:
        W, _ = wl.dense_tiny()
        return W, _dev(W)
    W = wl.heavy_rows(wl.rng(seed, rows, K), rows, K)
    if wdt == "bf16":
        bits, W = wl.to_bf16(W)
        return W, _bf16_dev(bits)
    return W, _dev(W)


def _encode_both(lib, levels, group, K, block, rows, wdt, seed=11):
    W, Wd = _weights(levels, K, rows, wdt, seed)
    signs = o.rotation_signs(seed, K)
    rot = lib.Rotation(K, block, signs=signs)
    cb = lib.Codebook(levels)
    codes, scales = lib.quantize(Wd, group, rot, cb)
    oc, ot = o.lloyd_max_gaussian(levels)
    v = W.astype(np.float64) @ o.rotation_matrix(signs, block).T
    ocodes, os16 = o.encode_rotated(v, group, ot)
    stride = lib.row_stride_words(levels, K)
    owords = o.pack(ocodes, levels, stride)
    u, rms = oracle_u(v, group)
    return dict(W=W, Wd=Wd, signs=signs, rot=rot, cb=cb, codes=codes, scales=scales, oc=oc, ot=ot, ocodes=ocodes,
                os16=os16, owords=owords, u=u, rms=rms, stride=stride)


@pytest.mark.parametrize("levels,group,K,block,rows,wdt", QCASES)
def test_quantize_codes_and_scales(lib, levels, group, K, block, rows, wdt):
    e = _encode_both(lib, levels, group, K, block, rows, wdt)
    ties = compare_codes(u32(e["codes"]), e["owords"], levels, K, e["u"], e["ot"])
    near = compare_scales(f16_from_bits(e["scales"]), e["os16"], e["rms"])
    n = rows * K
    assert ties <= max(3, n // 20000), f"{ties} ties of {n}"
    assert near <= max(3, (n // group) // 500)


@pytest.mark.parametrize("levels,group,K,block,rows,wdt", QCASES)
@pytest.mark.parametrize("T", [1, 3])
def test_quantize_then_qmv(lib, levels, group, K, block, rows, wdt, T):
    """End to end on a dense layer: GPU encode + GPU qmv vs oracle encode + oracle qmv."""
    e = _encode_both(lib, levels, group, K, block, rows, wdt)
    x = wl.rng(5, T, K).normal(size=(T, K)).astype(np.float32)
    xr = lib.rotate(_dev(x), e["rot"])
    qw = lib.QWeight(e["codes"], e["scales"], 1, rows, K, group, e["cb"])
    ref = o.qmv(o.dequantize(e["ocodes"], e["os16"], e["oc"], group), o.rotate(x, e["signs"], block))
    assert rel_l2(lib.qmv(qw, xr).cpu().numpy(), ref) < REL_L2  # the tensor-core form where it applies
    y = lib.qmv(qw, xr, tensor_cores=False).cpu().numpy()
    assert rel_l2(y, ref) < REL_L2
    # bf16 output: the kernel's own fp32 result rounded once (nearest even), and
    # within the bar of the oracle rounded to bf16 the same way.
    ybf = lib.qmv(qw, xr, out_dtype=torch.bfloat16).float().cpu().numpy()
    np.testing.assert_array_equal(ybf, wl.to_bf16(y)[1])
    assert rel_l2(ybf, wl.to_bf16(ref)[1]) < REL_L2


def _decode_tol(levels):
    """Decode-only tolerance.  Bit-packed books: fp32 arithmetic only (1e-5).  The
    three-level table-lookup kernel holds the input as integers per group of 16 columns,
    |xq| <= 8191 (rounding error uniform in +-max_g/16382 per element: for Gaussian inputs
    about 7e-5 of the output's RMS); the single-pass kernel as 16-bit integers per vector
    (about 4e-5).  Bar: 2.5e-4."""
    return 2.5e-4 if levels == 3 else 1e-5


def _random_bank(levels, experts, rows, K, group, seed):
    """Random valid packed words and fp16 scales (timing-style bank), uint32 / float16 numpy."""
    g = wl.rng(seed, 99)
    stride = o.row_words(levels, K)
    stride4 = (stride + 3) // 4 * 4
    if levels == 3:
        words = g.integers(0, 3 ** 20, size=(experts, rows, stride), dtype=np.int64)
    else:
        b = o.bits_per_code(levels)
        cw = 32 // b
        words = g.integers(0, 1 << (b * cw), size=(experts, rows, stride), dtype=np.int64)
    # zero the unused slots of each row's last word
    cw = o.codes_per_word(levels)
    used = K - (stride - 1) * cw
    if used < cw:
        if levels == 3:
            words[..., -1] %= 3 ** used
        else:
            words[..., -1] &= (1 << (o.bits_per_code(levels) * used)) - 1
    full = np.zeros((experts, rows, stride4), dtype=np.uint32)
    full[..., :stride] = words.astype(np.uint32)
    scales = (np.exp(g.normal(-3.5, 0.5, size=(experts, rows, K // group)))).astype(np.float16)
    return full, scales


def _bank_dev(lib, levels, experts, rows, K, group, seed):
    words, scales = _random_bank(levels, experts, rows, K, group, seed)
    cb = lib.Codebook(levels)
    qw = lib.QWeight(_dev(words.view(np.int32)), _dev(scales.view(np.int16)), experts, rows, K, group, cb,
                     row_stride=words.shape[-1])
    oc, _ = o.lloyd_max_gaussian(levels)

    def Wh(e):
        return o.dequantize(o.unpack(words[e], levels, K), scales[e], oc, group)

    return qw, Wh


@pytest.mark.parametrize("levels,group,K,rows", [(3, 16, 7168, 200), (8, 128, 4096, 130), (16, 64, 512, 64),
                                                 (4, 16, 640, 40), (3, 64, 2048, 33), (8, 16, 320, 31)])
def test_qmv_decode_exact(lib, levels, group, K, rows):
    """Decode of the same random words on both sides: only fp32 rounding separates them."""
    qw, Wh = _bank_dev(lib, levels, 1, rows, K, group, seed=levels * 100 + group)
    x = wl.rng(3, K).normal(size=(4, K))
    for T in (1, 2, 4):
        y = lib.qmv(qw, _dev(x[:T].astype(np.float32)), tensor_cores=False).cpu().numpy()
        ref = o.qmv(Wh(0), x[:T].astype(np.float32))
        assert rel_l2(y, ref) < _decode_tol(levels), T


# Tensor-core dense matvec: fp16 operands (unit roundoff u = 2^-11 each for the
# scaled input and the decoded weight), fp32 sums.  Per product the relative error
# has a standard deviation of about sqrt(2/3) u = 4e-4 and the errors are
# independent, so the relative L2 error of y stays near that; 1e-3 is the bar.
TC_TOL = 1e-3


@pytest.mark.parametrize("levels,group,K,rows,Ts", [
    (8, 128, 4096, 256, (1, 3, 16, 17, 64)),  # the dense decode shape, 2 row tiles, both pair tiles
    (8, 128, 4096, 2048, (4,)),               # 208 units over the SMs: CTA ranges cross row tiles
    (8, 32, 1344, 128, (2, 13)),              # 21 stages: the last code chunk holds one stage
    (16, 64, 1024, 384, (5,)),                # 4-bit, 3 row tiles
    (4, 32, 2048, 128, (1, 8)),               # 2-bit, 64 groups a row
    (8, 16, 1024, 256, (16,)),                # group 16
])
def test_qmv_tensor_cores(lib, levels, group, K, rows, Ts):
    qw, Wh = _bank_dev(lib, levels, 1, rows, K, group, seed=levels * 7 + group)
    W = Wh(0)
    for T in Ts:
        x = wl.rng(8, T, K).normal(size=(T, K)).astype(np.float32)
        y = lib.qmv_tc(qw, _dev(x)).cpu().numpy()
        assert rel_l2(y, o.qmv(W, x)) < TC_TOL, T


def test_qmv_tensor_cores_input_range(lib):
    """Rows of very different magnitude, and a zero row: each row is scaled by its own power of two
    (fp16 alone would overflow at 1e6 and flush 1e-7 to zero)."""
    qw, Wh = _bank_dev(lib, 8, 1, 256, 1024, 64, seed=3)
    W = Wh(0)
    x = wl.rng(9, 4).normal(size=(4, 1024)).astype(np.float32)
    x[0] *= 1e6
    x[2] *= 1e-7
    x[3] = 0.0
    y = lib.qmv_tc(qw, _dev(x)).cpu().numpy()
    ref = o.qmv(W, x)
    for t in range(3):
        assert rel_l2(y[t], ref[t]) < TC_TOL, t
    assert not np.any(y[3])


def test_qmv_tensor_cores_unsupported_shapes(lib):
    """Shapes outside the form raise (nothing launched); qmv() then takes tq_qmv."""
    qw, Wh = _bank_dev(lib, 8, 1, 130, 1024, 64, seed=4)  # rows not a multiple of 128
    x = wl.rng(10, 2).normal(size=(2, 1024)).astype(np.float32)
    with pytest.raises(lib.TQError):
        lib.qmv_tc(qw, _dev(x))
    assert rel_l2(lib.qmv(qw, _dev(x)).cpu().numpy(), o.qmv(Wh(0), x)) < 1e-5
    qw3, _ = _bank_dev(lib, 3, 1, 128, 1024, 64, seed=4)  # ternary book
    with pytest.raises(lib.TQError):
        lib.qmv_tc(qw3, _dev(x))


def test_gather_qmv_and_bad_ids(lib):
    E, rows, K, group = 12, 96, 7168, 16
    qw, Wh = _bank_dev(lib, 3, E, rows, K, group, seed=5)
    T, k = 2, 4
    ids = np.array([[3, 11, 0, 3], [7, 5, 11, 2]], dtype=np.int32)
    x = wl.rng(4).normal(size=(T, K)).astype(np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = lib.gather_qmv(qw, _dev(x), _dev(ids), err=err).cpu().numpy()
    ref = o.gather_qmv(Wh, ids, x)
    assert rel_l2(y, ref) < _decode_tol(3)
    assert lib.check_error(err) == 0
    # without scratch the single-pass kernel takes the 7168-wide rows
    y1 = lib.gather_qmv(qw, _dev(x), _dev(ids), err=err, use_ws=False).cpu().numpy()
    assert rel_l2(y1, ref) < _decode_tol(3)
    assert lib.check_error(err) == 0
    bad = ids.copy()
    bad[1, 2] = 12
    y = lib.gather_qmv(qw, _dev(x), _dev(bad), err=err).cpu().numpy()
    assert lib.check_error(err) == lib.TQ_DEVERR_BAD_ID
    assert np.all(y[1, 2] == 0)
    assert rel_l2(y[0], ref[0]) < _decode_tol(3)


def test_multi_gather_qmv(lib):
    E, rows, K, group = 9, 7168 // 32, 2048, 16
    qw, Wh = _bank_dev(lib, 3, E, rows, K, group, seed=6)
    ids = np.array([8, 0, 8, 4, 4, 1, 2], dtype=np.int32)
    x = wl.rng(6).normal(size=(len(ids), K)).astype(np.float32)
    y = lib.multi_gather_qmv(qw, _dev(x), _dev(ids)).cpu().numpy()
    assert rel_l2(y, o.multi_gather_qmv(Wh, ids, x)) < _decode_tol(3)


def test_dequant_experts(lib):
    qw, Wh = _bank_dev(lib, 8, 5, 40, 1536, 64, seed=8)
    ids = np.array([4, 1, 4], dtype=np.int32)
    out = lib.dequant_experts(qw, _dev(ids)).cpu().numpy()
    ref = o.dequant_experts(Wh, ids)
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-12)
    outh = lib.dequant_experts(qw, _dev(ids), out_dtype=torch.float16).float().cpu().numpy()
    np.testing.assert_allclose(outh, ref, rtol=1e-3, atol=1e-7)


@pytest.mark.parametrize("T,E,k,zipf", [(1, 384, 8, None), (37, 128, 8, 1.1), (300, 64, 4, None), (5, 16, 16, None),
                                        (3, 1000, 8, None), (9, 200, 6, 1.1)])
def test_route(lib, T, E, k, zipf):
    logits = wl.router_logits(9, T, E, zipf=zipf)
    if T == 5:
        logits[:, :] = np.round(logits * 2) / 2  # many exact ties
    ids, probs, perm, pos, off = lib.moe_route(_dev(logits), k)
    oids, oprobs = o.route(logits, k)
    operm, ooff = o.sort_pairs(oids, E)
    np.testing.assert_array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(probs.cpu().numpy(), oprobs, rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(perm.cpu().numpy(), operm)
    np.testing.assert_array_equal(off.cpu().numpy(), ooff)
    inv = np.empty_like(operm)
    inv[operm] = np.arange(len(operm))
    np.testing.assert_array_equal(pos.cpu().numpy(), inv)
    # without the sorted order (the one-token decode form): the same ids and weights
    ids2, probs2, perm2, _, _ = lib.moe_route(_dev(logits), k, sort=False)
    assert perm2 is None
    np.testing.assert_array_equal(ids2.cpu().numpy(), oids)
    np.testing.assert_allclose(probs2.cpu().numpy(), oprobs, rtol=2e-6, atol=1e-7)


def test_route_signed_zero_ties(lib):
    """-0.0 and +0.0 are one value: the tie goes to the lower expert id whatever the sign bits."""
    E, k = 64, 6
    logits = np.full((2, E), -1.0, np.float32)
    logits[0, [3, 9, 20, 41, 50, 63]] = [-0.0, 0.0, -0.0, 0.0, -0.0, 0.0]
    logits[1, [5, 6]] = [0.0, -0.0]
    logits[1, [30, 31, 32, 33]] = 0.5
    ids, probs, _, _, _ = lib.moe_route(_dev(logits), k, sort=False)
    oids, oprobs = o.route(logits, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(probs.cpu().numpy(), oprobs, rtol=2e-6, atol=1e-7)


def test_swiglu_rotate_and_combine(lib):
    P, inter = 19, 1536
    gu = wl.rng(10).normal(size=(P, 2 * inter)).astype(np.float32)
    rot = lib.Rotation(inter, 512, seed=3)
    h = lib.swiglu_rotate(_dev(gu), inter, rot).cpu().numpy()
    ref = o.rotate(o.swiglu(gu.astype(np.float64), inter), o.rotation_signs(3, inter), 512)
    assert rel_l2(h, ref) < 1e-6
    T, k, H = 4, 3, 700
    y = wl.rng(11).normal(size=(T * k, H)).astype(np.float32)
    p = wl.rng(12).random(size=(T, k)).astype(np.float32)
    out = lib.moe_combine(_dev(y), _dev(p), k).cpu().numpy()
    assert rel_l2(out, o.combine(y.reshape(T, k, H).astype(np.float64), p)) < 1e-6
    pos = np.array([5, 0, 11, 3, 1, 7, 2, 10, 4, 9, 6, 8], dtype=np.int32)
    ys = np.empty_like(y)
    ys[pos] = y
    out2 = lib.moe_combine(_dev(ys), _dev(p), k, pair_pos=_dev(pos)).cpu().numpy()
    assert rel_l2(out2, o.combine(y.reshape(T, k, H).astype(np.float64), p)) < 1e-6


def test_moe_decode_layer(lib):
    """Router -> rotate -> gate/up gather_qmv -> SwiGLU + rotate -> down multi_gather_qmv -> combine."""
    E, k, H, I = 16, 4, 1024, 512
    seed = wl.SEED_MOE_DECODE
    logits = wl.router_logits(seed, 1, E)
    _, x = wl.activations(seed, 1, H)
    gu_bank = [wl.expert_weights(seed, e, 0, 2 * I, H)[1] for e in range(E)]
    dn_bank = [wl.expert_weights(seed, e, 1, H, I)[1] for e in range(E)]
    sH, sI = o.rotation_signs(wl.sign_seed(seed, 0), H), o.rotation_signs(wl.sign_seed(seed, 1), I)
    bH, bI = o.rotation_block(H), o.rotation_block(I)
    ct, tt = o.lloyd_max_gaussian(3)
    # GPU side: encode both banks, run the layer
    rotH, rotI = lib.Rotation(H, bH, signs=sH), lib.Rotation(I, bI, signs=sI)
    cb = lib.Codebook(3)
    gu_codes, gu_scales = lib.quantize(_dev(np.concatenate(gu_bank)), 16, rotH, cb)
    dn_codes, dn_scales = lib.quantize(_dev(np.concatenate(dn_bank)), 16, rotI, cb)
    qgu = lib.QWeight(gu_codes, gu_scales, E, 2 * I, H, 16, cb)
    qdn = lib.QWeight(dn_codes, dn_scales, E, H, I, 16, cb)
    ids, probs, _, _, _ = lib.moe_route(_dev(logits), k)
    xr = lib.rotate(_dev(x), rotH)
    gu = lib.gather_qmv(qgu, xr, ids)
    hr = lib.swiglu_rotate(gu, I, rotI)
    yd = lib.multi_gather_qmv(qdn, hr, ids.reshape(-1))
    out = lib.moe_combine(yd, probs, k).cpu().numpy()
    # oracle side
    oids, oprobs = o.route(logits, k)
    RH, RI = o.rotation_matrix(sH, bH), o.rotation_matrix(sI, bI)

    def bank(ws, R, e):
        c, s16 = o.encode_rotated(ws[e].astype(np.float64) @ R.T, 16, tt)
        return o.dequantize(c, s16, ct, 16)

    gu_o = o.gather_qmv(lambda e: bank(gu_bank, RH, e), oids, o.rotate(x, sH, bH))
    h_o = o.rotate(o.swiglu(gu_o.reshape(k, 2 * I), I), sI, bI)
    yd_o = o.multi_gather_qmv(lambda e: bank(dn_bank, RI, e), oids.reshape(-1), h_o)
    ref = o.combine(yd_o.reshape(1, k, H), oprobs)
    assert rel_l2(out, ref) < REL_L2


@pytest.mark.parametrize("E,k,H,I", [(16, 4, 1024, 512), (4, 2, 2048, 256)])
def test_moe_decode_fused_stages(lib, E, k, H, I):
    """The decode layer with the input rotation inside gate/up and SwiGLU + rotation inside down:
    against the oracle, and the gate/up outputs against the separate rotate + gather_qmv calls."""
    seed = wl.SEED_MOE_DECODE + 7
    logits = wl.router_logits(seed, 1, E)
    xb, x = wl.activations(seed, 1, H)
    gu_bank = [wl.expert_weights(seed, e, 0, 2 * I, H)[1] for e in range(E)]
    dn_bank = [wl.expert_weights(seed, e, 1, H, I)[1] for e in range(E)]
    sH, sI = o.rotation_signs(wl.sign_seed(seed, 0), H), o.rotation_signs(wl.sign_seed(seed, 1), I)
    bH, bI = o.rotation_block(H), o.rotation_block(I)
    ct, tt = o.lloyd_max_gaussian(3)
    rotH, rotI = lib.Rotation(H, bH, signs=sH), lib.Rotation(I, bI, signs=sI)
    cb = lib.Codebook(3)
    gu_codes, gu_scales = lib.quantize(_dev(np.concatenate(gu_bank)), 16, rotH, cb)
    dn_codes, dn_scales = lib.quantize(_dev(np.concatenate(dn_bank)), 16, rotI, cb)
    qgu = lib.QWeight(gu_codes, gu_scales, E, 2 * I, H, 16, cb)
    qdn = lib.QWeight(dn_codes, dn_scales, E, H, I, 16, cb)
    ids, probs, _, _, _ = lib.moe_route(_dev(logits), k)
    gu_f = lib.gather_qmv_rotate(qgu, _dev(x), rotH, ids)
    gu_s = lib.gather_qmv(qgu, lib.rotate(_dev(x), rotH), ids)
    assert rel_l2(gu_f.cpu().numpy(), gu_s.cpu().numpy()) < 2.5e-4  # two integer input forms (see _decode_tol)
    gu_b = lib.gather_qmv_rotate(qgu, _bf16_dev(xb), rotH, ids)  # bf16 input, the same values
    assert rel_l2(gu_b.cpu().numpy(), gu_f.cpu().numpy()) < 1e-6
    yd = lib.multi_gather_qmv_swiglu(qdn, gu_f.reshape(k, 2 * I), rotI, ids.reshape(-1))
    out = lib.moe_combine(yd, probs, k).cpu().numpy()
    oids, oprobs = o.route(logits, k)
    RH, RI = o.rotation_matrix(sH, bH), o.rotation_matrix(sI, bI)

    def bank(ws, R, e):
        c, s16 = o.encode_rotated(ws[e].astype(np.float64) @ R.T, 16, tt)
        return o.dequantize(c, s16, ct, 16)

    gu_o = o.gather_qmv(lambda e: bank(gu_bank, RH, e), oids, o.rotate(x, sH, bH))
    h_o = o.rotate(o.swiglu(gu_o.reshape(k, 2 * I), I), sI, bI)
    yd_o = o.multi_gather_qmv(lambda e: bank(dn_bank, RI, e), oids.reshape(-1), h_o)
    ref = o.combine(yd_o.reshape(1, k, H), oprobs)
    assert rel_l2(out, ref) < REL_L2


@pytest.mark.parametrize("T,klev,vlev,group", [(300, 256, 8, 32), (2100, 256, 8, 32), (65, 16, 16, 16)])
def test_kv_quantize_and_attend(lib, T, klev, vlev, group):
    Hkv, D, Hq = 8, 128, 32
    kb, k = wl.kv_cache(tokens=T, which=0)
    vb, v = wl.kv_cache(tokens=T, which=1)
    qb, q = wl.kv_query()
    signs = o.rotation_signs(wl.sign_seed(wl.SEED_KV, 0), D)
    rot = lib.Rotation(D, D, signs=signs)
    kcb, vcb = lib.Codebook(klev), lib.Codebook(vlev)
    cache = lib.KVCache(T + 5, Hkv, D, group, kcb, vcb, rot)
    half = T // 2
    lib.kv_quantize(cache, _bf16_dev(kb[:half]), _bf16_dev(vb[:half]))
    lib.kv_quantize(cache, _bf16_dev(kb[half:]), _bf16_dev(vb[half:]))
    assert cache.length == T
    # codes and scales against the oracle
    kc, kt = o.lloyd_max_gaussian(klev)
    vc, vt = o.lloyd_max_gaussian(vlev)
    R = o.rotation_matrix(signs, D)
    outs = {}
    for name, X, c, t, lev, codes_d, scales_d in (("k", k, kc, kt, klev, cache.kcodes, cache.kscales),
                                                  ("v", v, vc, vt, vlev, cache.vcodes, cache.vscales)):
        ocodes, os16 = o.kv_quantize(X, signs, group, t)
        vrot = X.reshape(T * Hkv, D).astype(np.float64) @ R.T
        u, rms = oracle_u(vrot, group)
        u = u.reshape(T, Hkv, D).transpose(1, 0, 2).reshape(Hkv * T, D)
        rms = rms.reshape(T, Hkv, -1).transpose(1, 0, 2).reshape(Hkv * T, -1)
        ow = o.pack(ocodes.reshape(Hkv * T, D), lev)
        gw = u32(codes_d[:, :T]).reshape(Hkv * T, -1)
        ties = compare_codes(gw, ow, lev, D, u, t, what=name)
        near = compare_scales(f16_from_bits(scales_d[:, :T]).reshape(Hkv * T, -1), os16.reshape(Hkv * T, -1), rms)
        # each counted case was checked above to sit at a tie / rounding midpoint;
        # the counts only guard against a systematic shift
        assert ties <= max(3, T * Hkv * D // 20000) and near <= max(3, T * Hkv * (D // group) // 500)
        outs[name] = o.dequantize(ocodes.reshape(Hkv * T, D), os16.reshape(Hkv * T, -1), c, group).reshape(Hkv, T, D)
    o_gpu = lib.kv_attend(cache, _bf16_dev(qb)).cpu().numpy()
    ref = o.kv_attend(q, outs["k"], outs["v"], signs)
    assert rel_l2(o_gpu, ref) < REL_L2


def _qmm_case(lib, levels, group, E, rows, K, T, k, xt, seed):
    """Encode an expert bank on both sides, route T tokens, run the gather-GEMM."""
    bank = [wl.expert_weights(seed, e, 0, rows, K)[1] for e in range(E)]
    signs = o.rotation_signs(wl.sign_seed(seed, 0), K)
    blk = o.rotation_block(K)
    rot = lib.Rotation(K, blk, signs=signs)
    cb = lib.Codebook(levels)
    codes, scales = lib.quantize(_dev(np.concatenate(bank)), group, rot, cb)
    qw = lib.QWeight(codes, scales, E, rows, K, group, cb)
    logits = wl.router_logits(seed, T, E, zipf=1.1)
    _, x = wl.activations(seed, T, K)
    ids, probs, perm, pos, off = lib.moe_route(_dev(logits), k)
    dt = torch.float16 if xt == "f16" else torch.bfloat16
    xr = lib.rotate(_dev(x), rot, out_dtype=dt)
    y = lib.gather_qmm(qw, xr, perm, off, k).cpu().numpy()
    oids, _ = o.route(logits, k)
    operm, ooff = o.sort_pairs(oids, E)
    oc, ot = o.lloyd_max_gaussian(levels)
    R = o.rotation_matrix(signs, blk)
    Wh = {}

    def bankf(e):
        if e not in Wh:
            c, s16 = o.encode_rotated(bank[e].astype(np.float64) @ R.T, group, ot)
            Wh[e] = o.dequantize(c, s16, oc, group)
        return Wh[e]

    ref = o.gather_qmm(bankf, o.rotate(x, signs, blk), operm, ooff, k)
    return y, ref, ooff


@pytest.mark.parametrize("levels,group,E,rows,K,T,k", [(8, 64, 12, 256, 1024, 300, 8), (16, 64, 6, 128, 512, 70, 2),
                                                       (4, 32, 5, 128, 640, 40, 3), (8, 128, 3, 384, 1536, 9, 2),
                                                       (16, 16, 4, 128, 512, 50, 2), (8, 16, 3, 128, 64, 20, 2),
                                                       # more than 64 or an odd number of groups per row
                                                       (8, 16, 3, 128, 1280, 40, 2), (4, 64, 4, 128, 576, 33, 2)])
def test_gather_qmm_tensor_core(lib, levels, group, E, rows, K, T, k):
    y, ref, off = _qmm_case(lib, levels, group, E, rows, K, T, k, "f16", seed=4)
    assert rel_l2(y, ref) < REL_L2
    for e in range(E):  # every expert's block of sorted rows on its own
        lo, hi = off[e], off[e + 1]
        if hi > lo:
            assert rel_l2(y[lo:hi], ref[lo:hi]) < REL_L2, e


def test_gather_qmm_skew_spans_several_tiles(lib):
    y, ref, off = _qmm_case(lib, 8, 64, 16, 128, 512, 700, 8, "f16", seed=41)
    counts = np.diff(off)
    assert counts.max() > 256
    assert rel_l2(y, ref) < REL_L2


def test_gather_qmm_bf16_operands(lib):
    """bf16 operands: A and B rounded to 8-bit mantissas, error budget about 2 x 2^-9 / sqrt(3)."""
    y, ref, _ = _qmm_case(lib, 8, 64, 6, 128, 512, 64, 4, "bf16", seed=43)
    assert rel_l2(y, ref) < 4e-3


def test_gather_qmm_per_pair_input(lib):
    """Down-projection form: row i of x is sorted pair i's own input."""
    E, rows, K, group, levels = 7, 256, 1536, 64, 8
    bank = [wl.expert_weights(5, e, 1, rows, K)[1] for e in range(E)]
    signs = o.rotation_signs(77, K)
    rot = lib.Rotation(K, 512, signs=signs)
    cb = lib.Codebook(levels)
    codes, scales = lib.quantize(_dev(np.concatenate(bank)), group, rot, cb)
    qw = lib.QWeight(codes, scales, E, rows, K, group, cb)
    counts = np.array([0, 300, 5, 17, 0, 64, 1])
    off = np.concatenate(([0], np.cumsum(counts))).astype(np.int32)
    P = int(off[-1])
    h = wl.rng(6, P).normal(size=(P, K)).astype(np.float16)
    y = lib.gather_qmm(qw, _dev(h), _dev(np.zeros(P, np.int32)), _dev(off), 1, per_pair_input=True).cpu().numpy()
    oc, ot = o.lloyd_max_gaussian(levels)
    R = o.rotation_matrix(signs, 512)
    Wh = [o.dequantize(*o.encode_rotated(bank[e].astype(np.float64) @ R.T, group, ot), oc, group) for e in range(E)]
    ref = o.gather_qmm(lambda e: Wh[e], h.astype(np.float64), np.arange(P), off, 1, per_pair_input=True)
    assert rel_l2(y, ref) < REL_L2
