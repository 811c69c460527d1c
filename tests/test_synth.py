"""The seeded input generator: shapes, value ranges, routing rules and
reproducibility of per-expert streams."""
import numpy as np

import synth


def test_hidden_is_bf16_normal():
    x = synth.hidden(64, 512, seed=0)
    assert x.dtype == np.uint16 and x.shape == (64, 512)
    f = synth.bf16_bits_to_f32(x)
    assert abs(f.mean()) < 0.02 and abs(f.std() - 1.0) < 0.02
    assert np.array_equal(synth.f32_to_bf16_bits(f), x)       # already bf16
    assert np.array_equal(x, synth.hidden(64, 512, seed=0))


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], np.float32)
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(vals))
    assert got.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 0.0]


def test_routing_topk_and_weights():
    layer = synth.DECODE.layer
    lg = synth.logits(90, layer.E, seed=0)
    ids, w = synth.route(lg, layer.k)
    assert ids.shape == (90, 8) and w.shape == (90, 8) and w.dtype == np.float32
    for t in range(90):
        row = lg[t]
        assert len(set(ids[t].tolist())) == 8
        thresh = row[ids[t]].min()
        assert np.all(row[np.setdiff1d(np.arange(layer.E), ids[t])] <= thresh)
        assert np.all(np.diff(row[ids[t]]) <= 0)           # descending logit order
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_routing_tie_goes_to_lower_index():
    lg = np.array([[0.5, 2.0, 2.0, 1.0]], np.float32)
    ids, w = synth.route(lg, 2)
    assert ids.tolist() == [[1, 2]] and w[0, 0] == w[0, 1]


def test_zipf_prefill_is_skewed():
    layer = synth.PREFILL.layer
    ids, _ = synth.routing(4096, layer, seed=0, zipf_s=synth.PREFILL.zipf_s)
    c = np.bincount(ids.ravel(), minlength=layer.E)
    assert c.max() / c.mean() >= 8


def test_expert_weights_reproducible_and_uniform():
    layer = synth.TOY.layer
    w13, s13, w2, s2 = synth.expert_weights(layer, 3, seed=0)
    assert w13.shape == (256, 128) and s13.shape == (256, 8)
    assert w2.shape == (256, 64) and s2.shape == (256, 4)
    again = synth.expert_weights(layer, 3, seed=0)
    assert all(np.array_equal(a, b) for a, b in zip((w13, s13, w2, s2), again))
    other = synth.expert_weights(layer, 4, seed=0)
    assert not np.array_equal(w13, other[0])
    codes = np.concatenate([(w13 & 15).ravel(), (w13 >> 4).ravel()])
    hist = np.bincount(codes, minlength=16) / codes.size
    assert np.all(np.abs(hist - 1 / 16) < 0.01)
    s = synth.bf16_bits_to_f32(s13)
    assert s.min() >= 0.002 * (1 - 2 ** -8) and s.max() <= 0.02 * (1 + 2 ** -8)
    full = synth.layer_weights(layer, seed=0)
    assert np.array_equal(full[0][3], w13) and np.array_equal(full[3][3], s2)
