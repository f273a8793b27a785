"""GPU parity of the dense (QR-fallback) rotation: the rotation of rows, the encode through it
and the quantized matvec of a layer whose input dimension takes it.

Weight-reservoir page: dimensions the fast transform cannot take get a dense rotation derived
from a seed by QR.  The oracle builds the same rotation with numpy's QR from its own Gaussian
stream; codes are compared with the parity rule of the other encodes (bit-exact up to counted
ties within 1e-6), outputs within 2e-3 relative L2.
"""
import numpy as np
import pytest

from oracle import tq_oracle as o
from rotated_codebook_quantized_gb300 import workloads as wl
from tests.helpers import REL_L2, compare_codes, compare_scales, f16_from_bits, oracle_u, rel_l2, u32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("dim,rows,precise", [(400, 33, True), (400, 3, False), (1040, 70, True), (50, 5, False),
                                             (2000, 1, False), (2000, 6, True), (1040, 9, False), (1996, 2, True)])
def test_rotate_dense(lib, dim, rows, precise):
    seed = 40 + dim
    x = wl.rng(seed, rows).normal(size=(rows, dim)).astype(np.float32)
    rot = lib.DenseRotation(dim, seed=seed)
    y = lib.rotate_dense(torch.from_numpy(x).cuda(), rot, precise=precise).cpu().numpy()
    ref = x.astype(np.float64) @ o.rotation_dense(seed, dim).T
    # fp32 operands: R and x exact inputs, sums in fp64 (precise) or fp32
    assert rel_l2(y, ref) < (1e-7 if precise else 2e-6)


@pytest.mark.parametrize("levels,group,dim,rows", [(8, 16, 400, 96), (3, 16, 1040, 64), (16, 16, 208, 40)])
def test_quantize_dense_and_qmv(lib, levels, group, dim, rows):
    seed = 70 + dim
    W = wl.heavy_rows(wl.rng(seed, rows, dim), rows, dim)
    rot = lib.DenseRotation(dim, seed=seed)
    cb = lib.Codebook(levels)
    codes, scales = lib.quantize_dense(torch.from_numpy(W).cuda(), group, rot, cb)
    oc, ot = o.lloyd_max_gaussian(levels)
    R = o.rotation_dense(seed, dim)
    v = W.astype(np.float64) @ R.T
    ocodes, os16 = o.encode_rotated(v, group, ot)
    owords = o.pack(ocodes, levels, lib.row_stride_words(levels, dim))
    u, rms = oracle_u(v, group)
    ties = compare_codes(u32(codes), owords, levels, dim, u, ot)
    near = compare_scales(f16_from_bits(scales), os16, rms)
    assert ties <= max(3, rows * dim // 20000) and near <= max(3, rows * (dim // group) // 500)
    # decode: rotate the input with the dense rotation, multiply by the packed codes
    x = wl.rng(seed, 9).normal(size=(2, dim)).astype(np.float32)
    xr = lib.rotate_dense(torch.from_numpy(x).cuda(), rot)
    qw = lib.QWeight(codes, scales, 1, rows, dim, group, cb)
    y = lib.qmv(qw, xr, tensor_cores=False).cpu().numpy()
    ref = o.qmv(o.dequantize(ocodes, os16, oc, group), x.astype(np.float64) @ R.T)
    assert rel_l2(y, ref) < REL_L2
    # the layer computes W x up to the quantization error: the rotation cancels
    assert rel_l2(y, x.astype(np.float64) @ W.astype(np.float64).T) < 0.5
