"""GPU parity of the paths and shapes the first parity file leaves out.

* bit-packed books (3-bit group 64, 4-bit group 64, 2-bit group 32) through
  tq_gather_qmv and tq_multi_gather_qmv, with repeated experts and a bad id;
* the gather-GEMM at 64 groups per row (K = 4096, group 64: the prefill
  gate||up shape and the edge of the staged kernel's rule) and with sorted
  positions whose perm entry is out of range;
* tq_dequant_experts with bf16 output, a ternary bank and a bad id.

The weights are random valid packed words and fp16 scales drawn on the host
(inputs, never library results); the oracle decodes them and multiplies in
fp64.
"""
import numpy as np
import pytest

from oracle import tq_oracle as o
from rotated_codebook_quantized_gb300 import workloads as wl
from tests.helpers import REL_L2, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# Bit-packed decode: fp32 products and sums on both sides' inputs, so only fp32 rounding
# separates the library from the fp64 oracle.
BITS_TOL = 1e-5


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _random_bank(levels, experts, rows, K, group, seed, scale_mu=-3.5):
    """Random valid packed words (unused slots and padding zero) and fp16 scales."""
    g = wl.rng(seed, 199)
    nw = o.row_words(levels, K)
    stride = (nw + 3) // 4 * 4
    cw = o.codes_per_word(levels)
    if levels == 3:
        words = g.integers(0, 3 ** 20, size=(experts, rows, nw), dtype=np.int64)
    else:
        words = g.integers(0, 1 << (o.bits_per_code(levels) * cw), size=(experts, rows, nw), dtype=np.int64)
    used = K - (nw - 1) * cw
    if used < cw:
        if levels == 3:
            words[..., -1] %= 3 ** used
        else:
            words[..., -1] &= (1 << (o.bits_per_code(levels) * used)) - 1
    full = np.zeros((experts, rows, stride), dtype=np.uint32)
    full[..., :nw] = words.astype(np.uint32)
    scales = np.exp(g.normal(scale_mu, 0.5, size=(experts, rows, K // group))).astype(np.float16)
    return full, scales


def _bank(lib, levels, experts, rows, K, group, seed, scale_mu=-3.5):
    words, scales = _random_bank(levels, experts, rows, K, group, seed, scale_mu)
    cb = lib.Codebook(levels)
    qw = lib.QWeight(_dev(words.view(np.int32)), _dev(scales.view(np.int16)), experts, rows, K, group, cb,
                     row_stride=words.shape[-1])
    oc, _ = o.lloyd_max_gaussian(levels)
    cache = {}

    def Wh(e):
        if e not in cache:
            cache[e] = o.dequantize(o.unpack(words[e], levels, K), scales[e], oc, group)
        return cache[e]

    return qw, Wh


@pytest.mark.parametrize("levels,group,K,rows", [(8, 64, 1536, 96), (16, 64, 1024, 70), (4, 32, 640, 40),
                                                 (8, 128, 4096, 33)])
def test_gather_qmv_bitpacked(lib, levels, group, K, rows):
    """Shared input per token, bit-packed books; expert 3 appears twice in token 0."""
    E = 9
    qw, Wh = _bank(lib, levels, E, rows, K, group, seed=levels * 10 + group)
    ids = np.array([[3, 8, 3, 0], [6, 2, 8, 5]], dtype=np.int32)
    x = wl.rng(41, levels).normal(size=(2, K)).astype(np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = lib.gather_qmv(qw, _dev(x), _dev(ids), err=err).cpu().numpy()
    ref = o.gather_qmv(Wh, ids, x)
    assert rel_l2(y, ref) < BITS_TOL
    assert lib.check_error(err) == 0
    bad = ids.copy()
    bad[1, 1] = E  # one past the bank
    bad[0, 3] = -2
    y = lib.gather_qmv(qw, _dev(x), _dev(bad), err=err).cpu().numpy()
    assert lib.check_error(err) == lib.TQ_DEVERR_BAD_ID
    assert np.all(y[1, 1] == 0) and np.all(y[0, 3] == 0)
    keep = [(0, 0), (0, 1), (0, 2), (1, 0), (1, 2), (1, 3)]
    assert rel_l2(np.array([y[t, j] for t, j in keep]), np.array([ref[t, j] for t, j in keep])) < BITS_TOL


@pytest.mark.parametrize("levels,group,K,rows", [(8, 64, 1536, 128), (16, 64, 512, 65), (4, 32, 640, 40)])
def test_multi_gather_qmv_bitpacked(lib, levels, group, K, rows):
    """A different input per pair; repeated experts (the prefill-at-8-tokens pattern) and a bad id."""
    E = 12
    qw, Wh = _bank(lib, levels, E, rows, K, group, seed=levels * 20 + group)
    ids = np.array([5, 11, 5, 0, 5, 7, 11, 2, 2, 9, 5, 1, 3, 3, 10, 5, 0, 4, 6, 8], dtype=np.int32)
    x = wl.rng(42, levels).normal(size=(len(ids), K)).astype(np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = lib.multi_gather_qmv(qw, _dev(x), _dev(ids), err=err).cpu().numpy()
    ref = o.multi_gather_qmv(Wh, ids, x)
    assert rel_l2(y, ref) < BITS_TOL
    assert lib.check_error(err) == 0
    # without scratch the column chunks' partial sums are added with atomics: the same sums in
    # another order
    ypp = lib.multi_gather_qmv(qw, _dev(x), _dev(ids), use_ws=False).cpu().numpy()
    np.testing.assert_allclose(y, ypp, rtol=1e-5, atol=1e-6 * np.abs(ref).max())
    bad = ids.copy()
    bad[4] = 99
    y = lib.multi_gather_qmv(qw, _dev(x), _dev(bad), err=err).cpu().numpy()
    assert lib.check_error(err) == lib.TQ_DEVERR_BAD_ID
    assert np.all(y[4] == 0)
    keep = np.arange(len(ids)) != 4
    assert rel_l2(y[keep], ref[keep]) < BITS_TOL


def test_multi_gather_qmv_grouped_prefill_shape(lib):
    """8 tokens x top-8 of 128 experts under a Zipf(1.1) router (64 pairs, many repeats), 3-bit
    group 64 over K = 1536: every pair against the oracle, and equal to the per-pair kernel."""
    E, K, rows, T, k = 128, 1536, 256, 8, 8
    qw, Wh = _bank(lib, 8, E, rows, K, 64, seed=77)
    logits = wl.router_logits(77, T, E, zipf=1.1)
    oids, _ = o.route(logits, k)
    ids = oids.reshape(-1).astype(np.int32)
    assert len(set(ids.tolist())) < len(ids)
    x = wl.rng(77, 3).normal(size=(T * k, K)).astype(np.float32)
    y = lib.multi_gather_qmv(qw, _dev(x), _dev(ids)).cpu().numpy()
    assert rel_l2(y, o.multi_gather_qmv(Wh, ids, x)) < BITS_TOL
    ypp = lib.multi_gather_qmv(qw, _dev(x), _dev(ids), use_ws=False).cpu().numpy()
    np.testing.assert_allclose(y, ypp, rtol=1e-5, atol=1e-6 * np.abs(y).max())


def test_multi_gather_qmv_grouped_record_sizes(lib):
    """Experts with 1..9 pairs each: records of four pairs, then a remainder of three, two or one
    (each kind run by its own instance), shuffled pair order; against the oracle and bit-equal
    to the per-pair kernel."""
    E, K, rows = 10, 640, 96
    qw, Wh = _bank(lib, 16, E, rows, K, 32, seed=78)
    ids = np.concatenate([np.full(c, e, np.int32) for e, c in zip(range(E), [1, 2, 3, 4, 5, 6, 7, 8, 9, 0])])
    ids = ids[np.random.default_rng(78).permutation(len(ids))]
    x = wl.rng(78, 4).normal(size=(len(ids), K)).astype(np.float32)
    y = lib.multi_gather_qmv(qw, _dev(x), _dev(ids)).cpu().numpy()
    assert rel_l2(y, o.multi_gather_qmv(Wh, ids, x)) < BITS_TOL
    ypp = lib.multi_gather_qmv(qw, _dev(x), _dev(ids), use_ws=False).cpu().numpy()
    np.testing.assert_allclose(y, ypp, rtol=1e-5, atol=1e-6 * np.abs(y).max())


@pytest.mark.parametrize("levels,group,K,rows", [(8, 128, 1280, 200), (4, 16, 512, 37), (16, 64, 768, 70)])
def test_qmv_bitpacked_ragged_batches(lib, levels, group, K, rows):
    """tq_qmv at T = 1 .. 16 (vectors taken four, two and one to a task): every batch against the
    oracle, and each row equal to the one-vector call up to the order of the column chunks' sums."""
    qw, Wh = _bank(lib, levels, 1, rows, K, group, seed=90 + levels)
    W = Wh(0)
    x = wl.rng(90, levels).normal(size=(16, K)).astype(np.float32)
    singles = np.stack([lib.qmv(qw, _dev(x[t:t + 1]), tensor_cores=False).cpu().numpy()[0] for t in range(16)])
    assert rel_l2(singles, o.qmv(W, x)) < BITS_TOL
    for T in (2, 3, 5, 6, 7, 9, 13, 16):
        y = lib.qmv(qw, _dev(x[:T]), tensor_cores=False).cpu().numpy()
        assert rel_l2(y, o.qmv(W, x[:T])) < BITS_TOL, T
        np.testing.assert_allclose(y, singles[:T], rtol=1e-5, atol=1e-6 * np.abs(singles).max())


def test_multi_gather_qmv_grouped_bf16_and_bad_ids(lib):
    """Grouped pairs with a bf16 output (one column chunk: direct stores) and with an f32 output
    over several chunks (partial sums in scratch): bad ids give zero rows and BAD_ID, the rest
    match the oracle (bf16: to its rounding)."""
    E = 7
    for K, group in ((320, 64), (2560, 64)):
        qw, Wh = _bank(lib, 8, E, 100, K, group, seed=91 + K)
        ids = np.array([2, 2, 6, 2, 2, 2, 9, 0, 6, 2, -1, 3, 3, 3], dtype=np.int32)
        x = wl.rng(91, K).normal(size=(len(ids), K)).astype(np.float32)
        good = (ids >= 0) & (ids < E)
        ref = np.zeros((len(ids), 100))
        ref[good] = o.multi_gather_qmv(Wh, ids[good], x[good])
        for dt, tol in ((torch.float32, BITS_TOL), (torch.bfloat16, 8e-3)):
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            y = lib.multi_gather_qmv(qw, _dev(x), _dev(ids), out_dtype=dt, err=err).float().cpu().numpy()
            assert lib.check_error(err) == lib.TQ_DEVERR_BAD_ID
            assert np.all(y[~good] == 0)
            assert rel_l2(y[good], ref[good]) < tol


def test_gather_qmv_bitpacked_grouped_tokens(lib):
    """Eight tokens, top-4 of 24 experts under a skewed router (shared input per token, experts
    repeated across tokens, grouped by expert): against the oracle and the one-token calls."""
    E, K, rows, T, k = 24, 1536, 160, 8, 4
    qw, Wh = _bank(lib, 8, E, rows, K, 64, seed=92)
    oids, _ = o.route(wl.router_logits(92, T, E, zipf=1.3), k)
    ids = oids.astype(np.int32)
    x = wl.rng(92, 8).normal(size=(T, K)).astype(np.float32)
    y = lib.gather_qmv(qw, _dev(x), _dev(ids)).cpu().numpy()
    assert rel_l2(y, o.gather_qmv(Wh, ids, x)) < BITS_TOL
    one = np.stack([lib.gather_qmv(qw, _dev(x[t:t + 1]), _dev(ids[t:t + 1])).cpu().numpy()[0] for t in range(T)])
    np.testing.assert_allclose(y, one, rtol=1e-5, atol=1e-6 * np.abs(one).max())


def test_multi_gather_qmv_ternary_repeats_and_bad_id(lib):
    """Ternary book, per-pair inputs with repeated experts and a bad id (integer input per group: 2.5e-4)."""
    E, rows, K, group = 10, 96, 2048, 16
    qw, Wh = _bank(lib, 3, E, rows, K, group, seed=77)
    ids = np.array([4, 4, 9, 0, 4, 2, 9, 7], dtype=np.int32)
    x = wl.rng(43).normal(size=(len(ids), K)).astype(np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = ids.copy()
    bad[2] = 10
    y = lib.multi_gather_qmv(qw, _dev(x), _dev(bad), err=err).cpu().numpy()
    ref = o.multi_gather_qmv(Wh, ids, x)
    assert lib.check_error(err) == lib.TQ_DEVERR_BAD_ID
    assert np.all(y[2] == 0)
    keep = np.arange(len(ids)) != 2
    assert rel_l2(y[keep], ref[keep]) < 2.5e-4


def _qmm_random(lib, levels, group, E, rows, K, T, k, seed, zipf=1.1):
    """Gather-GEMM over random valid words: routing by the library (compared with the oracle's),
    fp16 token rows, the oracle's decode-and-multiply in fp64."""
    qw, Wh = _bank(lib, levels, E, rows, K, group, seed)
    logits = wl.router_logits(seed, T, E, zipf=zipf)
    ids, probs, perm, pos, off = lib.moe_route(_dev(logits), k)
    oids, _ = o.route(logits, k)
    operm, ooff = o.sort_pairs(oids, E)
    np.testing.assert_array_equal(perm.cpu().numpy(), operm)
    np.testing.assert_array_equal(off.cpu().numpy(), ooff)
    x = wl.rng(seed, 5).normal(size=(T, K)).astype(np.float16)
    return qw, Wh, x, perm, off, operm, ooff


def test_gather_qmm_64_groups_per_row(lib):
    """K = 4096 at group 64: the prefill gate||up shape, 64 groups per row (the staged kernel's limit)."""
    levels, group, E, rows, K, T, k = 8, 64, 6, 256, 4096, 96, 4
    qw, Wh, x, perm, off, operm, ooff = _qmm_random(lib, levels, group, E, rows, K, T, k, seed=51)
    y = lib.gather_qmm(qw, _dev(x), perm, off, k).cpu().numpy()
    ref = o.gather_qmm(Wh, x.astype(np.float64), operm, ooff, k)
    assert rel_l2(y, ref) < REL_L2
    for e in range(E):
        lo, hi = ooff[e], ooff[e + 1]
        if hi > lo:
            assert rel_l2(y[lo:hi], ref[lo:hi]) < REL_L2, e


@pytest.mark.parametrize("K,group", [(1024, 64), (1280, 16)])  # the staged kernel and the first one
def test_gather_qmm_bad_perm(lib, K, group):
    """Sorted positions whose perm entry is outside [0, P) read a zero input row and raise BAD_ID."""
    levels, E, rows, T, k = 8, 5, 128, 40, 2
    qw, Wh, x, perm, off, operm, ooff = _qmm_random(lib, levels, group, E, rows, K, T, k, seed=52)
    P = T * k
    bad = perm.clone()
    bad_pos = [3, P // 2, P - 1]
    bad[bad_pos[0]] = P
    bad[bad_pos[1]] = -1
    bad[bad_pos[2]] = 1 << 30
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = lib.gather_qmm(qw, _dev(x), bad, off, k, err=err).cpu().numpy()
    assert lib.check_error(err) == lib.TQ_DEVERR_BAD_ID
    ref = o.gather_qmm(Wh, x.astype(np.float64), operm, ooff, k)
    for i in bad_pos:
        assert np.all(y[i] == 0), i
    keep = np.ones(P, bool)
    keep[bad_pos] = False
    assert rel_l2(y[keep], ref[keep]) < REL_L2


def test_dequant_experts_bf16_ternary_and_bad_id(lib):
    """bf16 output (the benchmarked form), a ternary bank, and an out-of-range id (zeros + BAD_ID)."""
    qw, Wh = _bank(lib, 8, 5, 40, 1536, 64, seed=61)
    ids = np.array([4, 1, 4, 0], dtype=np.int32)
    ref = o.dequant_experts(Wh, ids)
    out = lib.dequant_experts(qw, _dev(ids), out_dtype=torch.bfloat16).float().cpu().numpy()
    np.testing.assert_allclose(out, ref, rtol=2.0 ** -8, atol=0)  # one bf16 rounding: half an ulp, 2^-9
    q3, W3 = _bank(lib, 3, 4, 24, 2048, 16, seed=62)
    ids3 = np.array([3, 0, 2], dtype=np.int32)
    out3 = lib.dequant_experts(q3, _dev(ids3)).cpu().numpy()
    np.testing.assert_allclose(out3, o.dequant_experts(W3, ids3), rtol=1e-6, atol=1e-12)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    badids = np.array([1, 5, -1, 2], dtype=np.int32)
    outb = lib.dequant_experts(qw, _dev(badids), out_dtype=torch.bfloat16, err=err).float().cpu().numpy()
    assert lib.check_error(err) == lib.TQ_DEVERR_BAD_ID
    assert not np.any(outb[1]) and not np.any(outb[2])
    np.testing.assert_allclose(outb[[0, 3]], o.dequant_experts(Wh, np.array([1, 2])), rtol=2.0 ** -8, atol=0)


@pytest.mark.parametrize("levels,group,rows,K,odt", [(4, 16, 37, 1024, "f32"), (16, 32, 13, 2080, "f16"),
                                                     (3, 16, 9, 7168, "bf16"), (8, 128, 6, 23040, "f32")])
def test_dequant_experts_books_and_ragged_rows(lib, levels, group, rows, K, odt):
    """2- and 4-bit books, rows that do not fill the last run of a CTA, a code row wider than one CTA's
    staging of several rows (K = 23040 takes one row per CTA), each output type."""
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[odt]
    qw, Wh = _bank(lib, levels, 3, rows, K, group, seed=70 + levels)
    ids = np.array([2, 0, 2, 1], dtype=np.int32)
    out = lib.dequant_experts(qw, _dev(ids), out_dtype=dt).float().cpu().numpy()
    ref = o.dequant_experts(Wh, ids)
    tol = {"f32": 1e-6, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}[odt]
    np.testing.assert_allclose(out, ref, rtol=tol, atol=1e-12 if odt == "f32" else 1e-7)
