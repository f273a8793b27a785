"""Expert streaming bookkeeping (host code, no GPU).

"How it works", "Expert streaming": the experts a step routes to are brought in through a
least-recently-used cache.  The library's plan is checked here against a plain model of the
policy stated in the header (lowest empty slot first, else the least recently used slot not
used by the step, lowest of equals), over long random routings with repeats.
"""
import numpy as np
import pytest

tq = pytest.importorskip("rotated_codebook_quantized_gb300")


def _lib():
    try:
        return tq.load()
    except RuntimeError:
        pytest.skip("libtq.so not built")


class ModelLRU:
    def __init__(self, slots):
        self.slot_expert = [-1] * slots
        self.last = [0] * slots
        self.step = 0
        self.hits = self.misses = 0

    def plan(self, ids):
        self.step += 1
        now = self.step
        where = {e: k for k, e in enumerate(self.slot_expert) if e >= 0}
        order = list(dict.fromkeys(ids))
        for e in order:
            if e in where:
                self.last[where[e]] = now
        slots, miss = [], []
        placed = {}
        for e in ids:
            if e in placed:
                slots.append(placed[e])
                miss.append(0)
                continue
            if e in where:
                self.hits += 1
                placed[e] = where[e]
                slots.append(where[e])
                miss.append(0)
                continue
            cand = [k for k in range(len(self.slot_expert)) if self.last[k] != now]
            empty = [k for k in cand if self.slot_expert[k] < 0]
            v = empty[0] if empty else min(cand, key=lambda k: (self.last[k], k))
            self.slot_expert[v] = e
            self.last[v] = now
            placed[e] = v
            self.misses += 1
            slots.append(v)
            miss.append(1)
        return slots, miss


def _cache(experts, slots, rows=4, cols=64, group=16, levels=3):
    _lib()
    cb = tq.Codebook(levels, device="cpu")
    stride = tq.row_stride_words(levels, cols)
    codes = np.zeros((experts, rows, stride), np.uint32)
    scales = np.zeros((experts, rows, cols // group), np.uint16)
    return tq.ExpertCache(codes, scales, experts, rows, cols, group, cb, slots, device=None)


@pytest.mark.parametrize("experts,slots,k,zipf", [(64, 16, 8, 0.0), (384, 32, 8, 1.1), (20, 8, 8, 0.0),
                                                   (10, 3, 2, 0.5)])
def test_plan_matches_model(experts, slots, k, zipf):
    c = _cache(experts, slots)
    m = ModelLRU(slots)
    g = np.random.default_rng(experts * 31 + slots)
    p = 1.0 / np.arange(1, experts + 1) ** zipf
    p /= p.sum()
    for step in range(300):
        T = int(g.integers(1, 4))
        ids = []
        for _ in range(T):  # each token: k distinct experts; tokens may share experts
            ids += list(g.choice(experts, size=min(k, experts), replace=False, p=p))
        if len(set(ids)) > slots:
            ids = list(dict.fromkeys(ids))[:slots] + ids[: len(ids) // 2]
            ids = [e for e in ids if e in set(list(dict.fromkeys(ids))[:slots])]
        got_s, got_m = c.plan(ids)
        want_s, want_m = m.plan(ids)
        assert list(got_s) == want_s, step
        assert list(got_m) == want_m, step
        # every id's slot holds it: equal ids share a slot, distinct ids do not
        pairs = {}
        for e, s in zip(ids, got_s):
            assert pairs.setdefault(e, s) == s
        assert len(set(pairs.values())) == len(pairs)
    h, mi, b = c.stats()
    assert (h, mi) == (m.hits, m.misses)
    assert b == 0  # plan copies nothing


def test_lru_eviction_order():
    c = _cache(8, 3)
    s, mi = c.plan([0, 1, 2])
    assert list(s) == [0, 1, 2] and list(mi) == [1, 1, 1]
    s, mi = c.plan([0])            # 0 used at step 2: 1 and 2 are the oldest
    assert list(mi) == [0]
    s, mi = c.plan([3])            # evicts the lowest of the oldest (slot 1, expert 1)
    assert list(s) == [1] and list(mi) == [1]
    s, mi = c.plan([1, 0])         # 1 is gone again; the victim is slot 2 (expert 2, step 1)
    assert list(s) == [2, 0] and list(mi) == [1, 0]
    assert c.stats()[:2] == (2, 5)


def test_repeats_share_one_copy():
    c = _cache(16, 4)
    s, mi = c.plan([5, 5, 7, 5, 7])
    assert list(mi) == [1, 0, 1, 0, 0]
    assert s[0] == s[1] == s[3] and s[2] == s[4] and s[0] != s[2]
    assert c.stats()[:2] == (0, 2)


def test_errors_leave_contents():
    c = _cache(16, 2)
    c.plan([1, 2])
    with pytest.raises(tq.TQError):
        c.plan([3, 16])            # id out of range
    with pytest.raises(tq.TQError):
        c.plan([-1])
    with pytest.raises(tq.TQError):
        c.plan([3, 4, 5])          # three distinct misses, two slots
    with pytest.raises(tq.TQError):
        c.plan([1, 3, 4])          # 1 keeps its slot: one left for two misses
    s, mi = c.plan([1, 2])         # still cached
    assert list(mi) == [0, 0]
    s, mi = c.plan([])
    assert len(s) == 0


def test_create_rejects_bad_bank():
    lib = _lib()
    import ctypes
    cb = tq.Codebook(3, device="cpu")
    codes = np.zeros((4, 2, 4), np.uint32)
    scales = np.zeros((4, 2, 4), np.uint16)
    h = ctypes.c_void_p()
    good = tq.tq_qweight_t(codes.ctypes.data, scales.ctypes.data, 4, 2, 64, 16, 4, 8, 8, cb.c())
    assert lib.tq_expert_cache_create(ctypes.byref(good), 2, None, None, ctypes.byref(h)) == tq.TQ_OK
    lib.tq_expert_cache_destroy(h)
    assert lib.tq_expert_cache_create(ctypes.byref(good), 0, None, None, ctypes.byref(h)) == tq.TQ_ERR_INVALID
    gapped = tq.tq_qweight_t(codes.ctypes.data, scales.ctypes.data, 4, 2, 64, 16, 4, 16, 8, cb.c())
    assert lib.tq_expert_cache_create(ctypes.byref(gapped), 2, None, None, ctypes.byref(h)) == \
        tq.TQ_ERR_UNSUPPORTED
    short = tq.tq_qweight_t(codes.ctypes.data, scales.ctypes.data, 4, 2, 128, 16, 4, 8, 8, cb.c())
    assert lib.tq_expert_cache_create(ctypes.byref(short), 2, None, None, ctypes.byref(h)) == tq.TQ_ERR_INVALID
    # map with no device slots is refused on the host
    c = _cache(4, 2)
    ids = np.array([0], np.int32)
    out = np.zeros(1, np.int32)
    assert lib.tq_expert_cache_map(c._h, ids.ctypes.data, 1, out.ctypes.data, None) == tq.TQ_ERR_INVALID
    lib.tq_expert_cache_destroy(None)
