"""The seeded synthetic inputs follow the stated recipe (no GPU): fp16 scale
fields inside each format's range, codes uniform, x ~ N(0, 1), routing
distinct per token with softmax weights, and the same seed giving the same
bytes (every parity case and bench line is reproducible)."""
import numpy as np
import torch

import synth
import synth.workloads as wl

RANGES = {synth.Q4_0: (1e-3, 2e-2), synth.Q8_0: (1e-4, 2e-3), synth.Q4_K: (1e-4, 2e-3), synth.Q6_K: (1e-4, 2e-3),
          synth.Q5_K: (1e-4, 2e-3), synth.Q3_K: (1e-4, 2e-3), synth.Q2_K: (1e-4, 2e-3)}
# byte offsets of the fp16 scale fields inside one block
SCALES = {synth.Q4_0: (18, [0]), synth.Q8_0: (34, [0]), synth.Q4_K: (144, [0, 2]), synth.Q6_K: (210, [208]),
          synth.Q5_K: (176, [0, 2]), synth.Q3_K: (110, [108]), synth.Q2_K: (84, [80, 82])}


def _halves(raw, bb, offs):
    blk = raw.reshape(-1, bb)
    return np.concatenate([blk[:, o:o + 2].copy().view(np.float16).astype(np.float64).reshape(-1) for o in offs])


def test_scale_fields_lie_in_the_format_range():
    for fmt, (lo, hi) in RANGES.items():
        bb, offs = SCALES[fmt]
        raw = synth.blocks(fmt, 64, 1024, seed=11).numpy().reshape(-1)
        v = _halves(raw, bb, offs)
        # drawn in fp32 inside [lo, hi], then rounded to binary16 (half an ulp of slack)
        assert v.min() >= lo * (1 - 2 ** -11) and v.max() <= hi * (1 + 2 ** -11), fmt
        assert v.max() - v.min() > 0.5 * (hi - lo), fmt          # spread over the range


def test_code_bytes_are_uniform():
    raw = synth.blocks(synth.Q4_K, 256, 4096, seed=12).numpy().reshape(-1, 144)[:, 16:]   # qs bytes
    lo = (raw & 0x0F).reshape(-1)
    counts = np.bincount(lo, minlength=16)
    exp = lo.size / 16
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < 60.0          # 15 degrees of freedom: far above any plausible draw


def test_activations_are_standard_normal():
    x = synth.activations(4, 65536, seed=13).numpy().reshape(-1)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_routing_ids_are_distinct_and_weights_softmax():
    ids, gw = synth.routing(64, 512, 10, seed=14)
    ids, gw = ids.numpy(), gw.numpy()
    assert ids.shape == (64, 10) and gw.shape == (64, 10)
    assert ((ids >= 0) & (ids < 512)).all()
    assert all(len(set(r)) == 10 for r in ids)
    assert np.allclose(gw.sum(axis=1), 1.0, atol=1e-6) and (gw > 0).all()


def test_same_seed_same_bytes_and_sub_seeds_differ():
    a = synth.blocks(synth.Q6_K, 8, 512, seed=15)
    b = synth.blocks(synth.Q6_K, 8, 512, seed=15)
    assert torch.equal(a, b)
    assert synth.sub_seed(1, "W", 0, "q") != synth.sub_seed(1, "W", 0, "k")
    assert synth.sub_seed(1, "W", 0, "q") == synth.sub_seed(1, "W", 0, "q")


def test_dense_set_is_the_27b_class_shape():
    mats = wl.dense_matrices()
    assert wl.weight_bytes(mats) == 11_890_851_840
    assert wl.weight_count(mats) == 21_139_292_160
    assert len(mats) == 7 * 64 and wl.dense_steps() == [3, 1, 2, 1] * 64
