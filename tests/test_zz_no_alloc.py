"""The allocation-free KV attention entry point against the ordinary one.

tq_kv_attend_noalloc is for callers that cannot allocate device memory where
they attend (a process whose device memory is all pre-assigned to its own
pool, a plug-in that is given no allocator).  It keeps its split-context
partials in a fixed array in the library instead of a caller workspace.  This
file is collected last on purpose, and must pass both alone and after the
rest of the suite.
"""
import ctypes

import numpy as np
import pytest

from rotated_codebook_quantized_gb300 import workloads as wl
from tests.helpers import REL_L2, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def test_noalloc_matches_workspace_entry_point_twice(lib):
    T, Hkv, D, Hq, group = 3000, 8, 128, 32, 32
    kb, _ = wl.kv_cache(tokens=T, which=0)
    vb, _ = wl.kv_cache(tokens=T, which=1)
    rot = lib.Rotation(D, D, seed=wl.sign_seed(wl.SEED_KV, 0))
    cache = lib.KVCache(T, Hkv, D, group, lib.Codebook(256), lib.Codebook(8), rot)
    lib.kv_quantize(cache, _bf16_dev(kb), _bf16_dev(vb))
    c = lib.load()
    for call in range(2):  # two calls in a row share (and overwrite) the fixed scratch
        qb, _ = wl.to_bf16(wl.rng(wl.SEED_KV, 90, call).normal(size=(Hq, D)))
        q = _bf16_dev(qb)
        ctx = T - 517 * call
        ref = lib.kv_attend(cache, q, ctx=ctx)
        o = torch.empty((Hq, D), dtype=torch.float32, device="cuda")
        r, kcb, vcb = rot.c(), cache.kcb.c(), cache.vcb.c()
        st = c.tq_kv_attend_noalloc(ctypes.c_void_p(q.data_ptr()), lib.TQ_BF16, Hq, Hkv, D, ctx, cache.capacity,
                                    ctypes.byref(r), ctypes.byref(kcb), ctypes.byref(vcb), group,
                                    ctypes.c_void_p(cache.kcodes.data_ptr()),
                                    ctypes.c_void_p(cache.kscales.data_ptr()),
                                    ctypes.c_void_p(cache.vcodes.data_ptr()),
                                    ctypes.c_void_p(cache.vscales.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == lib.TQ_OK
        torch.cuda.synchronize()
        assert rel_l2(o.cpu().numpy(), ref.cpu().numpy()) < REL_L2


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    c = lib.load()
    cap = int(c.tq_kv_attend_noalloc_max_scratch_bytes())
    assert cap == 4 << 20
    # 64 query heads over 2^20 tokens need 1024 * 64 * 130 * 4 bytes of partials: more than the array
    need = int(c.tq_kv_attend_workspace_bytes(64, 128, 1 << 20))
    assert need > cap
    r = lib.tq_rotation_t(128, 128, 0x1000)
    b = lib.tq_codebook_t(256, 0x1000, 0x1000)
    fake = ctypes.c_void_p(0x1000)
    st = c.tq_kv_attend_noalloc(fake, lib.TQ_BF16, 64, 8, 128, 1 << 20, 1 << 20, ctypes.byref(r), ctypes.byref(b),
                                ctypes.byref(b), 32, fake, fake, fake, fake, fake, None)
    assert st == lib.TQ_ERR_INVALID
