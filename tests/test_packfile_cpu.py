"""Per-layer tiers and the persisted packed format (host code, no GPU).

"How it works", "The ternary tier (1.58 bits)" and "Configuration that converter and loader
share": a layer's bit width is chosen from its name and recovered from the size of its saved
codebook; the weight-reservoir page: a flat, page-aligned file that loads byte-identical to what
was written.
"""
import ctypes
import os

import numpy as np
import pytest

from oracle import tq_oracle as o

tq = pytest.importorskip("rotated_codebook_quantized_gb300")


def _lib():
    try:
        return tq.load()
    except RuntimeError:
        pytest.skip("libtq.so not built")


def _random_layer(name, levels, experts, rows, cols, group, block, seed):
    g = np.random.default_rng(seed)
    cw = o.codes_per_word(levels)
    nw = -(-cols // cw)
    stride = (nw + 3) // 4 * 4
    codes = np.zeros((experts, rows, stride), np.uint32)
    if levels == 3:
        codes[..., :nw] = g.integers(0, 3 ** 20, size=(experts, rows, nw), dtype=np.int64)
    else:
        b = o.bits_per_code(levels)
        codes[..., :nw] = g.integers(0, 1 << (b * cw), size=(experts, rows, nw), dtype=np.int64)
    scales = np.exp(g.normal(-3, 0.5, size=(experts, rows, cols // group))).astype(np.float16)
    c, _ = o.lloyd_max_gaussian(levels)
    return tq.PackedLayer(name, codes, scales, c, group, block, 1000 * seed + 7)


LAYERS = [("model.embed_tokens", 16, 1, 24, 256, 64, 256),
          ("layers.0.self_attn.q_proj", 8, 1, 40, 512, 64, 512),
          ("layers.0.mlp.experts.gate_up_proj", 3, 4, 32, 640, 16, 128),
          ("layers.0.mlp.experts.down_proj", 16, 4, 64, 320, 16, 64),
          ("layers.0.self_attn.k_cache_probe", 256, 1, 8, 128, 32, 128)]


def test_round_trip_is_byte_identical(tmp_path):
    _lib()
    layers = [_random_layer(n, lv, e, r, c, gr, b, i) for i, (n, lv, e, r, c, gr, b) in enumerate(LAYERS)]
    p1, p2 = str(tmp_path / "a.tqpack"), str(tmp_path / "b.tqpack")
    tq.save_packed(p1, layers)
    back = tq.load_packed(p1)
    assert [L.name for L in back] == [L.name for L in layers]
    for L, B in zip(layers, back):
        assert B.levels == L.levels  # recovered from the stored codebook's size
        np.testing.assert_array_equal(B.centroids, L.centroids)
        np.testing.assert_array_equal(B.codes, L.codes)
        np.testing.assert_array_equal(B.scales, L.scales)
        assert (B.group, B.cols, B.rot_block, B.rot_seed) == (L.group, L.cols, L.rot_block, L.rot_seed)
    tq.save_packed(p2, back)
    a, b = open(p1, "rb").read(), open(p2, "rb").read()
    assert a == b
    assert len(a) % 4096 == 0 and a[:8] == b"TQPACK\x00\x01"


def test_blobs_are_page_aligned(tmp_path):
    _lib()
    layers = [_random_layer(n, lv, e, r, c, gr, b, i) for i, (n, lv, e, r, c, gr, b) in enumerate(LAYERS[:3])]
    p = str(tmp_path / "a.tqpack")
    tq.save_packed(p, layers)
    raw = open(p, "rb").read()
    n = int.from_bytes(raw[12:16], "little")
    assert n == 3
    for i in range(n):
        rec = raw[64 + 256 * i:64 + 256 * (i + 1)]
        offs = [int.from_bytes(rec[104 + 16 * k:112 + 16 * k], "little") for k in range(3)]
        sizes = [int.from_bytes(rec[112 + 16 * k:120 + 16 * k], "little") for k in range(3)]
        assert all(off % 4096 == 0 for off in offs)
        L = layers[i]
        assert sizes == [8 * L.levels, L.codes.nbytes, L.scales.nbytes]
        np.testing.assert_array_equal(np.frombuffer(raw[offs[1]:offs[1] + sizes[1]], np.uint32), L.codes.reshape(-1))


def test_damaged_files_are_rejected(tmp_path):
    lib = _lib()
    layers = [_random_layer(*LAYERS[1][:1], *LAYERS[1][1:], 3)]
    p = str(tmp_path / "a.tqpack")
    tq.save_packed(p, layers)
    raw = bytearray(open(p, "rb").read())
    n = ctypes.c_int32(0)
    bad = str(tmp_path / "bad.tqpack")
    for damage in ("magic", "version", "truncate", "codebook_size"):
        d = bytearray(raw)
        if damage == "magic":
            d[0] = ord("X")
        elif damage == "version":
            d[8] = 9
        elif damage == "truncate":
            d = d[:len(d) // 2]
        else:
            d[64 + 112:64 + 120] = (8 * 5).to_bytes(8, "little")  # a 5-entry codebook is no book
        open(bad, "wb").write(bytes(d))
        assert lib.tq_pack_file_info(bad.encode(), ctypes.byref(n), None, 0) == tq.TQ_ERR_INVALID, damage
    assert lib.tq_pack_file_info(str(tmp_path / "missing").encode(), ctypes.byref(n), None, 0) == tq.TQ_ERR_INVALID
    # an inconsistent layer is refused before anything is written
    L = _random_layer(*LAYERS[2][:1], *LAYERS[2][1:], 4)
    L.rot_block = 48  # does not divide cols = 640
    with pytest.raises(tq.TQError):
        tq.save_packed(str(tmp_path / "c.tqpack"), [L])


def test_tiers_follow_layer_names():
    _lib()
    assert tq.layer_tier("layers.3.mlp.experts.gate_up_proj") == (3, 16)
    assert tq.layer_tier("layers.3.mlp.experts.down_proj") == (16, 16)  # down projections before experts
    assert tq.layer_tier("layers.3.mlp.shared_expert.up_proj") == (3, 16)
    assert tq.layer_tier("layers.3.mlp.up_proj") == (8, 16)
    assert tq.layer_tier("layers.3.self_attn.o_proj") == (8, 64)
    assert tq.layer_tier("lm_head") == (8, 64)
    pol = tq.tier_policy({"other": (16, 128), "attn": (4, 32)})
    assert tq.layer_tier("lm_head", pol) == (16, 128)
    assert tq.layer_tier("layers.0.self_attn.q_proj", pol) == (4, 32)
    with pytest.raises(tq.TQError):
        tq.layer_tier("lm_head", tq.tier_policy({"other": (5, 64)}))
