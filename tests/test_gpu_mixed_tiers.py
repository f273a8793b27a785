"""A synthetic model with mixed tiers, encoded on the GPU, persisted, loaded and run.

"How it works", "The ternary tier (1.58 bits)": a model mixes tiers layer by layer (ternary
experts, 4-bit down projections, 3-bit protected layers) with no extra configuration, because
the codebook size marks the packing; "Configuration that converter and loader share": each layer's
width is chosen from its name and recovered from its saved codebook.  Every layer is encoded by
tq_quantize at its tier, written to a packed file, read back (codes, scales and codebook equal
bit for bit, the file byte-identical when written again) and multiplied through the kernels,
against the oracle's own encode + dequantize + matmul of the same weights.
"""
import numpy as np
import pytest

from oracle import tq_oracle as o
from rotated_codebook_quantized_gb300 import workloads as wl
from tests.helpers import REL_L2, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# name, experts, rows, cols
MODEL = [("model.embed_proj", 1, 192, 512),
         ("model.layers.0.self_attn.q_proj", 1, 256, 512),
         ("model.layers.0.mlp.experts.gate_up_proj", 4, 128, 1024),
         ("model.layers.0.mlp.experts.down_proj", 4, 512, 256),
         ("model.layers.0.mlp.up_proj", 1, 256, 512)]


def test_mixed_tier_model_round_trip_and_run(lib, tmp_path):
    pol = lib.tier_policy()
    packed, enc = [], {}
    for li, (name, E, rows, cols) in enumerate(MODEL):
        levels, group = lib.layer_tier(name, pol)
        W = np.concatenate([wl.expert_weights(20 + li, e, 0, rows, cols)[1] for e in range(E)])  # [E*rows, cols]
        seed = 5000 + li
        block = o.rotation_block(cols)
        signs = o.rotation_signs(seed, cols)
        rot = lib.Rotation(cols, block, signs=signs)
        cb = lib.Codebook(levels)
        codes, scales = lib.quantize(torch.from_numpy(np.ascontiguousarray(W)).cuda(), group, rot, cb)
        c64, t64 = lib.codebook(levels)
        L = lib.PackedLayer(name, codes.cpu().numpy().view(np.uint32).reshape(E, rows, -1),
                            scales.cpu().numpy().view(np.float16).reshape(E, rows, -1), c64, group, block, seed)
        packed.append(L)
        enc[name] = (W, signs, block, levels, group)
    p1, p2 = str(tmp_path / "model.tqpack"), str(tmp_path / "again.tqpack")
    lib.save_packed(p1, packed)
    back = lib.load_packed(p1)
    lib.save_packed(p2, back)
    assert open(p1, "rb").read() == open(p2, "rb").read()
    for L, B in zip(packed, back):
        assert (B.name, B.levels, B.group) == (L.name, L.levels, L.group)
        assert (B.levels, B.group) == lib.layer_tier(B.name, pol)  # the loader recomputes the same choice
        np.testing.assert_array_equal(B.codes, L.codes)
        np.testing.assert_array_equal(B.scales, L.scales)
    # run each loaded layer: bit-identical to the layer as encoded, and against the oracle
    for L, B in zip(packed, back):
        W, signs, block, levels, group = enc[L.name]
        E, rows, cols = L.experts, L.rows, L.cols
        x = wl.rng(77, len(L.name)).normal(size=(2, cols)).astype(np.float32)
        xr = lib.rotate(torch.from_numpy(x).cuda(), lib.Rotation(cols, block, signs=signs))
        qa, qb = L.qweight(), B.qweight()
        oc, ot = o.lloyd_max_gaussian(levels)
        R = o.rotation_matrix(signs, block)
        Wo = [o.dequantize(*o.encode_rotated(W[e * rows:(e + 1) * rows].astype(np.float64) @ R.T, group, ot), oc,
                           group) for e in range(E)]
        xro = o.rotate(x, signs, block)
        if E == 1:
            ya, yb = lib.qmv(qa, xr).cpu().numpy(), lib.qmv(qb, xr).cpu().numpy()
            ref = o.qmv(Wo[0], xro)
        else:
            ids = torch.tensor([[3, 1], [0, 3]], dtype=torch.int32, device="cuda")
            ya, yb = lib.gather_qmv(qa, xr, ids).cpu().numpy(), lib.gather_qmv(qb, xr, ids).cpu().numpy()
            ref = o.gather_qmv(lambda e: Wo[e], ids.cpu().numpy(), xro)
        np.testing.assert_array_equal(ya, yb)
        assert rel_l2(yb, ref) < REL_L2, L.name
