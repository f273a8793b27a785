"""One token through the MoE decode layer in one launch (tq_moe_decode_layer).

"How it works", "Running a quantized layer", and the router of "Running a 1T-Parameter Model on a
Laptop": route, rotate the input, gate||up gather, SwiGLU + the intermediate rotation, down gather,
router-weighted combine.  The fused launch does each phase with the arithmetic of the separate entry
points, in the same order, so its output must equal theirs bit for bit; and the oracle's layer
(its routing, dequantized banks in the rotated domain, SwiGLU, rotations, combine) within the
ternary decode tolerance.  At wait budget 0 the grid barriers give up and the call reports
TQ_ERR_TIMEOUT; the next call is again bit-identical.
"""
import ctypes

import numpy as np
import pytest

from oracle import tq_oracle as o
from rotated_codebook_quantized_gb300 import workloads as wl
from tests.helpers import rel_l2
from tests.test_gpu_coverage import _bank, _dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _chain(lib, qgu, qdn, rotH, rotI, logits, x, k, I):
    ids, probs, _, _, _ = lib.moe_route(logits.view(1, -1), k, sort=False)
    xr = lib.rotate(x.view(1, -1), rotH)
    gu = lib.gather_qmv(qgu, xr, ids)
    hr = lib.swiglu_rotate(gu.reshape(k, 2 * I).contiguous(), I, rotI)
    yd = lib.multi_gather_qmv(qdn, hr, ids.view(-1))
    return lib.moe_combine(yd, probs, k), ids


@pytest.mark.parametrize("E,H,I,k,xbf16", [(16, 3072, 2048, 8, True), (12, 5120, 2048, 4, False)])
def test_decode_layer_matches_chain_and_oracle(lib, E, H, I, k, xbf16):
    qgu, Wgu = _bank(lib, 3, E, 2 * I, H, 16, seed=E + H)
    qdn, Wdn = _bank(lib, 3, E, H, I, 16, seed=E + I + 1)
    sH, sI = o.rotation_signs(7 + H, H), o.rotation_signs(8 + I, I)
    rotH, rotI = lib.Rotation(H, 1024, signs=sH), lib.Rotation(I, 2048, signs=sI)
    logits = wl.router_logits(E + k, 1, E)[0]
    x = wl.rng(E, H).normal(size=H).astype(np.float32)
    xd = _dev(x).to(torch.bfloat16) if xbf16 else _dev(x)
    ld = _dev(logits)
    out = lib.moe_decode_layer(qgu, qdn, rotH, rotI, ld, xd, k)
    ref_chain, ids = _chain(lib, qgu, qdn, rotH, rotI, ld, xd, k, I)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_chain)
    # the oracle's layer
    oids, oprobs = o.route(logits[None], k)
    np.testing.assert_array_equal(ids.cpu().numpy(), oids)
    xo = xd.float().cpu().numpy().astype(np.float64)[None]
    xr = o.rotate(xo, sH, 1024)[0]
    y = np.zeros(H)
    for j in range(k):
        e = int(oids[0, j])
        gu = Wgu(e) @ xr
        h = o.rotate(o.swiglu(gu[None], I), sI, 2048)[0]
        y += oprobs[0, j] * (Wdn(e) @ h)
    assert rel_l2(out.cpu().numpy()[0], y) < 5e-4


def test_decode_layer_wait_budget_and_unsupported(lib):
    E, H, I, k = 10, 3072, 2048, 8
    qgu, _ = _bank(lib, 3, E, 2 * I, H, 16, seed=5)
    qdn, _ = _bank(lib, 3, E, H, I, 16, seed=6)
    rotH, rotI = lib.Rotation(H, 1024, seed=1), lib.Rotation(I, 2048, seed=2)
    ld = _dev(wl.router_logits(3, 1, E)[0])
    xd = _dev(wl.rng(4, H).normal(size=H).astype(np.float32))
    good = lib.moe_decode_layer(qgu, qdn, rotH, rotI, ld, xd, k)
    torch.cuda.synchronize()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.set_wait_budget(0)
    try:
        lib.moe_decode_layer(qgu, qdn, rotH, rotI, ld, xd, k, err=err)
    finally:
        lib.set_wait_budget(-1)
    assert lib.check_error(err) & lib.TQ_DEVERR_TIMEOUT
    for _ in range(2):
        again = lib.moe_decode_layer(qgu, qdn, rotH, rotI, ld, xd, k, err=err)
        assert lib.check_error(err) == 0
        assert torch.equal(again, good)
    # a bank the launch does not take (bit-packed): the separate entry points serve it
    q8, _ = _bank(lib, 8, E, 2 * I, H, 64, seed=7)
    with pytest.raises(lib.TQError):
        lib.moe_decode_layer(q8, qdn, rotH, rotI, ld, xd, k)
