"""Bounded waits of the tensor-core kernels, made to run out on purpose.

Every wait of one pipeline role on another (an mbarrier phase) in the gather-GEMM and the
tensor-core matvec is bounded; on expiry the kernel raises TQ_DEVERR_TIMEOUT, drains what it
has in flight, frees its TMEM and returns.  With the wait budget set to 0 cycles through the
library's test hook, nearly every wait runs out at once: the call must report TQ_ERR_TIMEOUT,
and once the default budget is back, the next call on the same context must give the same
result as before (nothing left allocated or half-written in the library's state).
"""
import ctypes

import numpy as np
import pytest

from tests.test_gpu_coverage import _dev, _qmm_random

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _expire(lib, fn):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.set_wait_budget(0)
    try:
        fn(err)
    finally:
        lib.set_wait_budget(-1)
    bits = ctypes.c_uint32(0)
    st = lib.load().tq_check_error(ctypes.c_void_p(err.data_ptr()), ctypes.byref(bits),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, bits.value


@pytest.mark.parametrize("K,group", [(1024, 64), (1280, 16)])  # the staged kernel and the first one
def test_gather_qmm_wait_budget_zero(lib, K, group):
    levels, E, rows, T, k = 8, 5, 256, 48, 2
    qw, Wh, x, perm, off, operm, ooff = _qmm_random(lib, levels, group, E, rows, K, T, k, seed=61)
    xd = _dev(x)
    good = lib.gather_qmm(qw, xd, perm, off, k)
    torch.cuda.synchronize()
    st, bits = _expire(lib, lambda err: lib.gather_qmm(qw, xd, perm, off, k, err=err))
    assert st == lib.TQ_ERR_TIMEOUT and bits & lib.TQ_DEVERR_TIMEOUT, (st, bits)
    for _ in range(2):  # TMEM was freed: the next calls allocate it again and finish
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        again = lib.gather_qmm(qw, xd, perm, off, k, err=err)
        assert lib.check_error(err) == 0
        assert torch.equal(again, good)


def test_qmv_tc_wait_budget_zero(lib):
    from tests.test_gpu_coverage import _bank

    qw, Wh = _bank(lib, 8, 1, 512, 2048, 64, 62)
    x = torch.from_numpy(np.random.default_rng(62).normal(size=(4, 2048)).astype(np.float32)).cuda()
    good = lib.qmv_tc(qw, x)
    torch.cuda.synchronize()
    st, bits = _expire(lib, lambda err: lib.qmv_tc(qw, x, err=err))
    assert st == lib.TQ_ERR_TIMEOUT and bits & lib.TQ_DEVERR_TIMEOUT, (st, bits)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    again = lib.qmv_tc(qw, x, err=err)
    assert lib.check_error(err) == 0
    torch.testing.assert_close(again, good, rtol=1e-5, atol=1e-6)  # split-K partial sums: any order


def test_ternary_tensor_copy_matvec_wait_budget_zero(lib):
    """The ternary tensor-copy matvec (tq_gather_qmv_rotate: the input rotation in its prologue,
    then a producer warp feeding 15 decoder warps through mbarrier rings), with enough stages per
    decoder (8 experts x 4096 rows x 7168 columns) that producer and decoders wait on each other:
    at budget 0 the waits give up and the call reports TQ_ERR_TIMEOUT; the next call at the default
    budget gives the earlier result."""
    from tests.test_gpu_coverage import _random_bank

    E, rows, K, T, k = 8, 4096, 7168, 1, 8
    words, scales = _random_bank(3, E, rows, K, 16, seed=64)
    cb = lib.Codebook(3)
    qw = lib.QWeight(_dev(words.view(np.int32)), _dev(scales.view(np.int16)), E, rows, K, 16, cb,
                     row_stride=words.shape[-1])
    rot = lib.Rotation(K, 1024, seed=64)
    ids = np.array([[4, 0, 5, 2, 7, 1, 6, 3]], dtype=np.int32)
    x = np.random.default_rng(64).normal(size=(T, K)).astype(np.float32)
    xd, idd = _dev(x), _dev(ids)
    good = lib.gather_qmv_rotate(qw, xd, rot, idd)
    torch.cuda.synchronize()
    st, bits = _expire(lib, lambda err: lib.gather_qmv_rotate(qw, xd, rot, idd, err=err))
    assert st == lib.TQ_ERR_TIMEOUT and bits & lib.TQ_DEVERR_TIMEOUT, (st, bits)
    for _ in range(2):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        again = lib.gather_qmv_rotate(qw, xd, rot, idd, err=err)
        assert lib.check_error(err) == 0
        torch.testing.assert_close(again, good, rtol=1e-5, atol=1e-6 * float(good.abs().max()))  # atomics


def test_wait_budget_default_is_restored(lib):
    """With the default budget a long gather-GEMM raises nothing."""
    levels, group, E, rows, K, T, k = 8, 64, 8, 512, 2048, 256, 4
    qw, Wh, x, perm, off, operm, ooff = _qmm_random(lib, levels, group, E, rows, K, T, k, seed=63)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gather_qmm(qw, _dev(x), perm, off, k, err=err)
    assert lib.check_error(err) == 0
