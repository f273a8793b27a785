"""The C-ABI library without a GPU: it builds, loads, exports every declared
symbol, and its host-only entry points agree with the oracle.  No device work
is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import tq_oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def clib():
    from rotated_codebook_quantized_gb300 import _build

    path = _build.build()
    return ctypes.CDLL(path)


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\*?\s+\*?(tq_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("tq_codebook", "tq_quantize", "tq_qmv", "tq_gather_qmv", "tq_multi_gather_qmv", "tq_gather_qmm",
                 "tq_dequant_experts", "tq_kv_quantize", "tq_kv_attend", "tq_rotate", "tq_moe_route"):
        assert must in names


def test_every_declared_symbol_is_exported(clib):
    for name in declared_functions():
        assert hasattr(clib, name), name


def test_binding_signatures_cover_the_header():
    import rotated_codebook_quantized_gb300 as tq

    assert sorted(tq._SIGS) == declared_functions()


def test_host_codebook_matches_oracle():
    import rotated_codebook_quantized_gb300 as tq

    for L in (2, 3, 4, 8, 16, 256):
        c, t = tq.codebook(L)
        oc, ot = o.lloyd_max_gaussian(L)
        # The 256-level fixed point is ill-conditioned (the Lloyd map contracts by
        # about 1 - O(1/L^2)), so two converged solvers agree to ~1e-12, not 1e-15;
        # the fp32 tables the kernels use must agree exactly.
        tol = 1e-10 if L == 256 else 1e-12
        np.testing.assert_allclose(c, oc, rtol=0, atol=tol)
        np.testing.assert_allclose(t, ot, rtol=0, atol=tol)
        np.testing.assert_array_equal(c.astype(np.float32), oc.astype(np.float32))
        np.testing.assert_array_equal(t.astype(np.float32), ot.astype(np.float32))
        np.testing.assert_array_equal(c, -c[::-1])


def test_host_signs_match_oracle():
    import rotated_codebook_quantized_gb300 as tq

    for seed, dim in ((0, 17), (1234567, 5), (4001, 7168)):
        np.testing.assert_array_equal(tq.rotation_signs(seed, dim), o.rotation_signs(seed, dim))


def test_format_helpers_match_oracle():
    import rotated_codebook_quantized_gb300 as tq

    for L in (2, 3, 4, 8, 16, 256):
        assert tq.codes_per_word(L) == o.codes_per_word(L)
        for K in (1, 20, 21, 4096, 7168):
            assert tq.row_words(L, K) == o.row_words(L, K)
            assert tq.row_stride_words(L, K) == (o.row_words(L, K) + 3) // 4 * 4
    assert tq.codes_per_word(5) == 0


def test_host_validation_rejects_bad_arguments():
    """Argument checks run on the host and return before any CUDA call."""
    import rotated_codebook_quantized_gb300 as tq

    lib = tq.load()
    fake = ctypes.c_void_p(0x1000)
    cb = tq.tq_codebook_t(8, fake.value, fake.value)
    rot = tq.tq_rotation_t(512, 512, fake.value)
    # group 48 is not a supported group size
    assert lib.tq_quantize(fake, 0, 4, 512, 48, ctypes.byref(rot), ctypes.byref(cb), fake, fake, 52, None) == \
        tq.TQ_ERR_INVALID
    # rotation block that does not divide the dimension
    bad_rot = tq.tq_rotation_t(512, 384, fake.value)
    assert lib.tq_quantize(fake, 0, 4, 512, 64, ctypes.byref(bad_rot), ctypes.byref(cb), fake, fake, 52, None) == \
        tq.TQ_ERR_INVALID
    # row stride below the packed row length
    assert lib.tq_quantize(fake, 0, 4, 512, 64, ctypes.byref(rot), ctypes.byref(cb), fake, fake, 12, None) == \
        tq.TQ_ERR_INVALID
    qw = tq.tq_qweight_t(fake.value, fake.value, 1, 64, 512, 64, 51, 0, 0, cb)  # stride not a multiple of 4
    assert lib.tq_qmv(ctypes.byref(qw), fake, 1, fake, 0, None) == tq.TQ_ERR_INVALID
    assert lib.tq_moe_route(fake, 1, 2000, 8, fake, fake, fake, fake, fake, fake, 1 << 20, None) == tq.TQ_ERR_INVALID
    assert lib.tq_codebook(5, None, None) == tq.TQ_ERR_INVALID
    assert lib.tq_status_string(tq.TQ_ERR_TIMEOUT) == b"device wait timed out"


def test_qmv_tc_host_checks_and_workspace():
    """tq_qmv_tc: the shapes it refuses, the workspace rule and the size formula, all decided on the
    host before any CUDA call; a NULL error word is accepted (the device simply does not report)."""
    import rotated_codebook_quantized_gb300 as tq

    lib = tq.load()
    fake = ctypes.c_void_p(0x1000)
    cb8 = tq.tq_codebook_t(8, fake.value, fake.value)
    cb3 = tq.tq_codebook_t(3, fake.value, fake.value)
    stride = o.row_words(8, 4096) + 2  # 412: padded to a multiple of 4 words
    need = lib.tq_qmv_tc_workspace_bytes(3, 4096)
    assert need == 3 * 4096 * 2 + 16  # fp16 rows, then 3 row scales in one 16-byte piece
    assert lib.tq_qmv_tc_workspace_bytes(0, 4096) == 0
    ok = tq.tq_qweight_t(fake.value, fake.value, 1, 256, 4096, 128, stride, 0, 0, cb8)
    assert lib.tq_qmv_tc(ctypes.byref(ok), fake, 0, fake, None, 0, None, None) == tq.TQ_OK  # nothing to do
    assert lib.tq_qmv_tc(ctypes.byref(ok), fake, -1, fake, fake, need, None, None) == tq.TQ_ERR_INVALID
    assert lib.tq_qmv_tc(ctypes.byref(ok), None, 3, fake, fake, need, None, None) == tq.TQ_ERR_INVALID
    assert lib.tq_qmv_tc(ctypes.byref(ok), fake, 3, fake, fake, need - 16, None, None) == tq.TQ_ERR_INVALID
    assert lib.tq_qmv_tc(ctypes.byref(ok), fake, 3, fake, ctypes.c_void_p(0x1008), need, None, None) == tq.TQ_ERR_INVALID
    assert lib.tq_qmv_tc(ctypes.byref(ok), fake, 65, fake, fake, 1 << 30, None, None) == tq.TQ_ERR_UNSUPPORTED
    tern = tq.tq_qweight_t(fake.value, fake.value, 1, 256, 4096, 128, 208, 0, 0, cb3)
    assert lib.tq_qmv_tc(ctypes.byref(tern), fake, 3, fake, fake, need, None, None) == tq.TQ_ERR_UNSUPPORTED
    rows130 = tq.tq_qweight_t(fake.value, fake.value, 1, 130, 4096, 128, stride, 0, 0, cb8)
    assert lib.tq_qmv_tc(ctypes.byref(rows130), fake, 3, fake, fake, need, None, None) == tq.TQ_ERR_UNSUPPORTED
    cols96 = tq.tq_qweight_t(fake.value, fake.value, 1, 256, 96, 32, 12, 0, 0, cb8)
    assert lib.tq_qmv_tc(ctypes.byref(cols96), fake, 3, fake, fake, need, None, None) == tq.TQ_ERR_UNSUPPORTED


def test_gather_workspace_sizes_cover_grouping():
    """Scratch sizes of the bit-packed gathers (host only): with more than one token, or per-pair
    inputs, the size adds the record lists of the grouping (whole 256-byte pieces, at least a
    count per expert and an id per pair) to the per-pair partial sums; one token, and ternary
    books, need no lists."""
    import rotated_codebook_quantized_gb300 as tq

    lib = tq.load()
    fake = ctypes.c_void_p(0x1000)
    E, rows, cols, group = 128, 4096, 1536, 64
    stride = (o.row_words(8, cols) + 3) // 4 * 4
    cb8 = tq.tq_codebook_t(8, fake.value, fake.value)
    qw = tq.tq_qweight_t(fake.value, fake.value, E, rows, cols, group, stride, rows * stride,
                         rows * (cols // group), cb8)
    P = 64
    one_token = lib.tq_gather_qmv_workspace_bytes(ctypes.byref(qw), 1, P)
    eight_tokens = lib.tq_gather_qmv_workspace_bytes(ctypes.byref(qw), 8, P // 8)
    multi = lib.tq_multi_gather_qmv_workspace_bytes(ctypes.byref(qw), P)
    lists = eight_tokens - one_token
    assert multi == eight_tokens
    assert lists > 0 and lists % 256 == 0 and lists >= 4 * (E + 2 * P)
    assert lib.tq_gather_qmv_workspace_bytes(ctypes.byref(qw), 0, 8) == 0
    assert lib.tq_multi_gather_qmv_workspace_bytes(ctypes.byref(qw), 0) == 0
    cb3 = tq.tq_codebook_t(3, fake.value, fake.value)
    stride3 = (o.row_words(3, 7168) + 3) // 4 * 4
    tw = tq.tq_qweight_t(fake.value, fake.value, 16, 2048, 7168, 16, stride3, 2048 * stride3, 2048 * 448, cb3)
    assert lib.tq_gather_qmv_workspace_bytes(ctypes.byref(tw), 8, 8) == \
        lib.tq_gather_qmv_workspace_bytes(ctypes.byref(tw), 1, 64)
    assert lib.tq_multi_gather_qmv_workspace_bytes(ctypes.byref(tw), 64) == \
        lib.tq_gather_qmv_workspace_bytes(ctypes.byref(tw), 1, 64)
