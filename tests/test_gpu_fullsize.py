"""Full-size parity in the launch configurations the benchmark times, on sampled outputs.

Decode layer: 384 ternary experts (gate||up 4096 x 7168, down 7168 x 2048, group 16), one
token routed top-8, the same calls as the benchmark's step.  Dense layer: 11008 x 4096,
3-bit, group 128, T = 1, 4, 16.  The weight words and scales are random valid ones drawn
by a seeded torch generator on the device (inputs, not results of the library); the oracle
decodes each sampled row on the host from the same words and multiplies it in fp64.  Every
oracle input comes from the workload generators or those draws, never from the library's
own outputs, so each call is checked on inputs of its own.
"""
import numpy as np
import pytest

from oracle import tq_oracle as o
from rotated_codebook_quantized_gb300 import workloads as wl
from tests.helpers import REL_L2, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

E, TOPK, H, I, G = 384, 8, 7168, 2048, 16
SAMPLES = 96

# The ternary table-lookup kernel holds the input as integers per group of 16 columns
# (|xq| <= 8191): about 7e-5 relative error per dot product (rms) for Gaussian inputs; a
# sample of 96 outputs stays under 2.5e-4.
TRIT_TOL = 2.5e-4


def _trit_bank(lib, experts, rows, cols, seed):
    """Random valid trit words (3^20 per word; the last word holds cols mod 20 trits) + fp16 scales."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    nw = -(-cols // 20)
    stride = lib.row_stride_words(3, cols)
    codes = torch.zeros((experts, rows, stride), dtype=torch.int32, device="cuda")
    used = cols - (nw - 1) * 20
    for e0 in range(0, experts, 32):
        w = torch.randint(0, 3 ** 20, (min(32, experts - e0), rows, nw), generator=g, device="cuda",
                          dtype=torch.int64)
        w[..., -1] %= 3 ** used
        codes[e0:e0 + 32, :, :nw] = (w - (w >= 2 ** 31).long() * 2 ** 32).to(torch.int32)
    sc = (torch.exp(torch.randn((experts, rows, cols // G), generator=g, device="cuda") * 0.5 - 3.5)).half()
    return codes, sc


def _rows(codes, sc, e, rows, levels, cols, group, oc):
    """Oracle weights of the given rows of expert e, decoded on the host."""
    w = codes[e, rows].cpu().numpy().view(np.uint32)
    s = sc[e, rows].cpu().numpy()
    return o.dequantize(o.unpack(w, levels, cols), s, oc, group)


def test_full_size_moe_decode_layer_sampled(lib):
    rs = np.random.default_rng(20261202)
    seed = wl.SEED_MOE_DECODE
    oc, _ = o.lloyd_max_gaussian(3)
    cb = lib.Codebook(3)
    gu_codes, gu_sc = _trit_bank(lib, E, 2 * I, H, 1101)
    dn_codes, dn_sc = _trit_bank(lib, E, H, I, 1102)
    qgu = lib.QWeight(gu_codes, gu_sc.view(torch.int16), E, 2 * I, H, G, cb, row_stride=gu_codes.shape[-1])
    qdn = lib.QWeight(dn_codes, dn_sc.view(torch.int16), E, H, I, G, cb, row_stride=dn_codes.shape[-1])

    # routing of one token over 384 experts
    logits = wl.router_logits(seed, 1, E)
    ids, probs, _, _, _ = lib.moe_route(torch.from_numpy(logits).cuda(), TOPK, sort=False)
    oids, oprobs = o.route(logits, TOPK)
    np.testing.assert_array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(probs.cpu().numpy(), oprobs, rtol=1e-5, atol=1e-7)

    # input rotation (7168 = 7 x 1024) and the gate||up gather over the 8 routed experts
    bits, x = wl.activations(seed, 1, H)
    sH = o.rotation_signs(wl.sign_seed(seed, 0), H)
    rotH = lib.Rotation(H, 1024, signs=sH)
    xb = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    gu = lib.gather_qmv(qgu, lib.rotate(xb, rotH), ids).cpu().numpy()  # [1, 8, 4096]
    xr_o = o.rotate(x, sH, 1024)[0]
    got, ref = [], []
    for j, r in zip(rs.integers(0, TOPK, SAMPLES), rs.integers(0, 2 * I, SAMPLES)):
        ref.append(float(_rows(gu_codes, gu_sc, int(oids[0, j]), [int(r)], 3, H, G, oc)[0] @ xr_o))
        got.append(gu[0, j, r])
    assert rel_l2(np.array(got), np.array(ref)) < TRIT_TOL

    # SwiGLU + rotation of the 2048-wide intermediate, on a seeded gate||up input
    gin = rs.normal(size=(TOPK, 2 * I)).astype(np.float32)
    sI = o.rotation_signs(wl.sign_seed(seed, 1), I)
    rotI = lib.Rotation(I, 2048, signs=sI)
    hr = lib.swiglu_rotate(torch.from_numpy(gin).cuda(), I, rotI).cpu().numpy()
    assert rel_l2(hr, o.rotate(o.swiglu(gin.astype(np.float64), I), sI, 2048)) < 1e-5

    # down multi-gather over the same 8 experts, on seeded per-pair inputs
    hin = rs.normal(size=(TOPK, I)).astype(np.float32)
    yd = lib.multi_gather_qmv(qdn, torch.from_numpy(hin).cuda(), torch.from_numpy(oids.reshape(-1).astype(np.int32)).cuda())
    yd = yd.cpu().numpy()
    got, ref = [], []
    for p, r in zip(rs.integers(0, TOPK, SAMPLES), rs.integers(0, H, SAMPLES)):
        ref.append(float(_rows(dn_codes, dn_sc, int(oids[0, p]), [int(r)], 3, I, G, oc)[0] @ hin[p].astype(np.float64)))
        got.append(yd[p, r])
    assert rel_l2(np.array(got), np.array(ref)) < TRIT_TOL

    # router-weighted combine of seeded expert outputs
    yin = rs.normal(size=(TOPK, H)).astype(np.float32)
    out = lib.moe_combine(torch.from_numpy(yin).cuda(), torch.from_numpy(oprobs.astype(np.float32)).cuda(), TOPK)
    assert rel_l2(out.cpu().numpy(), o.combine(yin[None].astype(np.float64), oprobs)) < 1e-6


def _bit_bank(lib, rows, cols, levels, group, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    b = {4: 2, 8: 3, 16: 4}[levels]
    cw = o.codes_per_word(levels)
    nw = -(-cols // cw)
    stride = lib.row_stride_words(levels, cols)
    w = torch.randint(0, 1 << (b * cw), (1, rows, nw), generator=g, device="cuda", dtype=torch.int64)
    w[..., -1] &= (1 << (b * (cols - (nw - 1) * cw))) - 1
    codes = torch.zeros((1, rows, stride), dtype=torch.int32, device="cuda")
    codes[..., :nw] = (w - (w >= 2 ** 31).long() * 2 ** 32).to(torch.int32)
    sc = (torch.exp(torch.randn((1, rows, cols // group), generator=g, device="cuda") * 0.5 - 3.5)).half()
    return codes, sc


@pytest.mark.parametrize("T", [1, 4, 16])
def test_full_size_dense_qmv_sampled(lib, T):
    """11008 x 4096, 3-bit, group 128: tq_qmv (fp32 decode, 1e-5) and tq_qmv_tc (fp16 operands, 1e-3)."""
    N, K, Gd, L = 11008, 4096, 128, 8
    rs = np.random.default_rng(T)
    oc, _ = o.lloyd_max_gaussian(L)
    codes, sc = _bit_bank(lib, N, K, L, Gd, 1201)
    qw = lib.QWeight(codes, sc.view(torch.int16), 1, N, K, Gd, lib.Codebook(L), row_stride=codes.shape[-1])
    x = wl.rng(wl.SEED_DENSE_DECODE, 7, T).normal(size=(T, K)).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    y32 = lib.qmv(qw, xd, tensor_cores=False).cpu().numpy()
    ytc = lib.qmv_tc(qw, xd).cpu().numpy()
    rows = np.sort(rs.choice(N, SAMPLES, replace=False))
    ref = _rows(codes, sc, 0, rows, L, K, Gd, oc) @ x.astype(np.float64).T  # [samples, T]
    assert rel_l2(y32[:, rows].T, ref) < 1e-5
    assert rel_l2(ytc[:, rows].T, ref) < 1e-3
    assert rel_l2(lib.qmv(qw, xd).cpu().numpy()[:, rows].T, ref) < REL_L2  # the form qmv() picks at this T


def _bit_bank_experts(lib, experts, rows, cols, levels, group, seed):
    """Random valid bit-packed words and fp16 scales of an expert bank, drawn on the device."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    b = {4: 2, 8: 3, 16: 4}[levels]
    cw = o.codes_per_word(levels)
    nw = -(-cols // cw)
    stride = lib.row_stride_words(levels, cols)
    codes = torch.zeros((experts, rows, stride), dtype=torch.int32, device="cuda")
    for e0 in range(0, experts, 16):
        n = min(16, experts - e0)
        w = torch.randint(0, 1 << (b * cw), (n, rows, nw), generator=g, device="cuda", dtype=torch.int64)
        w[..., -1] &= (1 << (b * (cols - (nw - 1) * cw))) - 1
        codes[e0:e0 + n, :, :nw] = (w - (w >= 2 ** 31).long() * 2 ** 32).to(torch.int32)
    sc = (torch.exp(torch.randn((experts, rows, cols // group), generator=g, device="cuda") * 0.5 - 3.5)).half()
    return codes, sc


def test_full_size_prefill_gather_qmm_sampled(lib):
    """MoE prefill at full size in the benchmark's launch configuration: 4096 tokens routed top-8
    of 128 experts (N(0,1) + Zipf(1.1) logits), gate||up 3072 x 4096 and per-pair down 4096 x 1536,
    3-bit group 64, fp16 operands.  32 sampled outputs from each of the hottest, the median and the
    coldest expert of each projection (96 per projection) against the oracle's decode of those rows."""
    PE, PT, PK, PH, PI, PG, L = 128, 4096, 8, 4096, 1536, 64, 8
    rs = np.random.default_rng(20261203)
    oc, _ = o.lloyd_max_gaussian(L)
    cb = lib.Codebook(L)
    gu_codes, gu_sc = _bit_bank_experts(lib, PE, 2 * PI, PH, L, PG, 1301)
    dn_codes, dn_sc = _bit_bank_experts(lib, PE, PH, PI, L, PG, 1302)
    qgu = lib.QWeight(gu_codes, gu_sc.view(torch.int16), PE, 2 * PI, PH, PG, cb, row_stride=gu_codes.shape[-1])
    qdn = lib.QWeight(dn_codes, dn_sc.view(torch.int16), PE, PH, PI, PG, cb, row_stride=dn_codes.shape[-1])
    logits = wl.router_logits(wl.SEED_MOE_PREFILL, PT, PE, zipf=1.1)
    _, _, perm, _, off = lib.moe_route(torch.from_numpy(logits).cuda(), PK)
    oids, _ = o.route(logits, PK)
    operm, ooff = o.sort_pairs(oids, PE)
    np.testing.assert_array_equal(perm.cpu().numpy(), operm)
    np.testing.assert_array_equal(off.cpu().numpy(), ooff)
    g = torch.Generator(device="cuda")
    g.manual_seed(1303)
    x = torch.randn((PT, PH), generator=g, device="cuda").half()
    h = torch.randn((PT * PK, PI), generator=g, device="cuda").half()
    ygu = lib.gather_qmm(qgu, x, perm, off, PK).cpu().numpy()
    ydn = lib.gather_qmm(qdn, h, perm, off, 1, per_pair_input=True).cpu().numpy()
    counts = np.diff(ooff)
    order = [e for e in np.argsort(-counts, kind="stable") if counts[e] > 0]
    picks = [order[0], order[len(order) // 2], order[-1]]  # hottest, median, coldest routed expert
    assert counts[picks[0]] > 1000 and counts[picks[2]] < counts[picks[0]]
    xh = x.cpu().numpy().astype(np.float64)
    hh = h.cpu().numpy().astype(np.float64)
    for codes, sc, y, rows, K, inp, by_token in ((gu_codes, gu_sc, ygu, 2 * PI, PH, xh, True),
                                                 (dn_codes, dn_sc, ydn, PH, PI, hh, False)):
        got, ref = [], []
        for e in picks:
            lo, hi = int(ooff[e]), int(ooff[e + 1])
            pos = rs.integers(lo, hi, 32)
            rws = rs.integers(0, rows, 32)
            W = _rows(codes, sc, int(e), rws, L, K, PG, oc)  # [32, K]
            for i, (ps, r) in enumerate(zip(pos, rws)):
                src = inp[int(operm[ps]) // PK] if by_token else inp[int(ps)]
                ref.append(float(W[i] @ src))
                got.append(float(y[ps, r]))
        assert rel_l2(np.array(got), np.array(ref)) < REL_L2


def test_full_size_kv_attend_sampled(lib):
    """KV decode read at full size: 131072 cached tokens x 8 kv heads x 128 (8-bit keys, 3-bit values,
    group 32), 32 query heads, 128 split-context partials merged.  The cache is random valid codes
    and fp16 scales drawn on the device; the oracle dequantizes kv heads 2 and 7, de-rotates, and
    runs softmax attention for the 8 query heads that read them."""
    ctx, Hkv, D, Hq, KG = 131072, 8, 128, 32, 32
    g = torch.Generator(device="cuda")
    g.manual_seed(1401)
    signs = o.rotation_signs(wl.sign_seed(wl.SEED_KV, 0), D)
    rot = lib.Rotation(D, D, signs=signs)
    cache = lib.KVCache(ctx, Hkv, D, KG, lib.Codebook(256), lib.Codebook(8), rot)
    kw = cache.kw
    k_words = torch.randint(0, 2 ** 32, (Hkv, ctx, kw), generator=g, device="cuda", dtype=torch.int64)
    cache.kcodes.copy_((k_words - (k_words >= 2 ** 31).long() * 2 ** 32).to(torch.int32))
    del k_words
    v_words = torch.randint(0, 2 ** 30, (Hkv, ctx, cache.vw), generator=g, device="cuda", dtype=torch.int64)
    v_words[..., -1] &= (1 << (3 * (D - (cache.vw - 1) * 10))) - 1
    cache.vcodes.copy_(v_words.to(torch.int32))
    del v_words
    cache.kscales.copy_(torch.exp(torch.randn((Hkv, ctx, D // KG), generator=g, device="cuda") * 0.5).half()
                        .view(torch.int16))
    cache.vscales.copy_(torch.exp(torch.randn((Hkv, ctx, D // KG), generator=g, device="cuda") * 0.5).half()
                        .view(torch.int16))
    cache.length = ctx
    qb, q = wl.kv_query()
    qd = torch.from_numpy(np.ascontiguousarray(qb).view(np.int16)).cuda().view(torch.bfloat16)
    out = lib.kv_attend(cache, qd).cpu().numpy()
    kc, _ = o.lloyd_max_gaussian(256)
    vc, _ = o.lloyd_max_gaussian(8)
    grp = Hq // Hkv
    for kvh in (2, 7):
        Kh = o.dequantize(o.unpack(cache.kcodes[kvh].cpu().numpy().view(np.uint32), 256, D),
                          cache.kscales[kvh].cpu().numpy().view(np.float16), kc, KG)
        Vh = o.dequantize(o.unpack(cache.vcodes[kvh].cpu().numpy().view(np.uint32), 8, D),
                          cache.vscales[kvh].cpu().numpy().view(np.float16), vc, KG)
        heads = list(range(kvh * grp, (kvh + 1) * grp))
        ref = o.kv_attend(q[heads], Kh[None], Vh[None], signs)
        assert rel_l2(out[heads], ref) < REL_L2, kvh
