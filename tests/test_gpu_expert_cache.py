"""Expert streaming from host memory through a device LRU of slots.

"How it works", "Expert streaming": only the routed experts are brought in, through an LRU
cache, and the result is bit-identical to running the whole bank resident.  A bank encoded on
the device is moved to pinned host memory; every step maps its routing into a few slots
(one pair of host-to-device copies per missing expert) and runs gather_qmv on the slot bank.
Each step's output must equal, bit for bit, gather_qmv of the resident bank with the original
ids, and every cached slot must hold its expert's bytes.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _bank(lib, E, rows, cols, group, levels, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    W = torch.randn(E * rows, cols, generator=g, device="cuda") * 0.02
    block = 1024 if cols % 1024 == 0 else cols
    rot = lib.Rotation(cols, block, seed=seed)
    cb = lib.Codebook(levels)
    codes, scales = lib.quantize(W, group, rot, cb)
    w = lib.QWeight(codes.reshape(E, rows, -1), scales.reshape(E, rows, -1), E, rows, cols, group, cb)
    return w


@pytest.mark.parametrize("levels,group,E,rows,cols,slots,T,k", [
    (3, 16, 48, 256, 2048, 12, 1, 8),     # ternary (table-lookup gather)
    (3, 16, 40, 128, 1024, 10, 2, 4),
    (8, 64, 32, 192, 1024, 8, 2, 3),      # 3-bit
    (16, 128, 24, 128, 512, 6, 1, 6),     # 4-bit
])
def test_streamed_gather_is_bit_identical(lib, levels, group, E, rows, cols, slots, T, k):
    w = _bank(lib, E, rows, cols, group, levels, seed=E * 7 + levels)
    hc = w.codes.cpu().pin_memory()
    hs = w.scales.cpu().pin_memory()
    cache = lib.ExpertCache(hc, hs, E, rows, cols, group, w.cb, slots, row_stride=w.row_stride)
    g = np.random.default_rng(levels * 100 + E)
    hot = g.choice(E, size=max(k, slots // 2), replace=False)  # a hot set, so that some steps hit
    total_distinct = 0
    for step in range(24):
        rows_ids = []
        for _ in range(T):
            pool = hot if g.random() < 0.6 else np.arange(E)
            rows_ids.append(g.choice(pool, size=k, replace=False))
        ids = np.stack(rows_ids).astype(np.int32)
        if len(set(ids.reshape(-1).tolist())) > slots:
            ids = np.stack([ids[0]] * T)
        total_distinct += len(set(ids.reshape(-1).tolist()))
        x = torch.randn(T, cols, device="cuda", generator=torch.Generator(device="cuda").manual_seed(step))
        ids_d = torch.from_numpy(ids).cuda()
        want = lib.gather_qmv(w, x, ids_d)
        got = cache.gather_qmv(x, ids_d)
        torch.cuda.synchronize()
        assert torch.equal(got, want), step
    hits, misses, nbytes = cache.stats()
    assert hits + misses == total_distinct
    per_expert = rows * w.row_stride * 4 + rows * (cols // group) * 2
    assert nbytes == misses * per_expert
    assert misses < total_distinct  # the hot set hit at least once
    # every slot that holds an expert holds its bytes
    last = cache.map(np.unique(ids.reshape(-1)))  # all cached already: no copies
    torch.cuda.synchronize()
    assert cache.stats()[2] == nbytes
    for e, s in zip(np.unique(ids.reshape(-1)), last):
        assert torch.equal(cache.view.codes[s].cpu(), hc[e])
        assert torch.equal(cache.view.scales[s].cpu(), hs[e])


def test_streamed_bank_larger_than_slots_end_to_end(lib):
    """A bank 8x the slot budget, routed by moe_route from seeded logits each step."""
    E, rows, cols, group, slots, T, k = 64, 128, 1024, 16, 8, 1, 8
    w = _bank(lib, E, rows, cols, group, 3, seed=99)
    cache = lib.ExpertCache(w.codes.cpu().pin_memory(), w.scales.cpu().pin_memory(), E, rows, cols, group, w.cb,
                            slots, row_stride=w.row_stride)
    g = torch.Generator(device="cuda").manual_seed(5)
    for step in range(10):
        logits = torch.randn(T, E, device="cuda", generator=g)
        routed = lib.moe_route(logits, k)
        ids = routed[0]
        x = torch.randn(T, cols, device="cuda", generator=g)
        got = cache.gather_qmv(x, ids)
        want = lib.gather_qmv(w, x, ids)
        torch.cuda.synchronize()
        assert torch.equal(got, want), step
