"""Variants beyond the pages' layer, against the oracle with the usual layer
tolerance: scale groups of 64 and 128 elements along K (prepack repeats each
scale into the 32-element slots of the packed layout), a 256-expert layer of
the decode width, and a shared expert every token routes to (one more slot
per token, weight 1)."""
import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _run(dl, M, seed=0, zipf=None, rows=None, ids=None, w=None):
    import quantized_moe_expert_align_gb300 as moe
    L = dl.layer
    x = synth.hidden(M, L.H, seed)
    if ids is None:
        ids, w = synth.routing(M, L, seed, zipf_s=zipf)
    out, ws = dl.forward(x, ids, w)
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    got = gu.bf16_dev_to_f64(out)
    ref = dl.oracle(x, ids, w, rows)
    return gu.parity(got if rows is None else got[rows], ref, f"E{L.E} g{L.group} M={M}")


@pytest.mark.parametrize("group", [64, 128])
def test_toy_wide_groups(gpu, group):
    L = synth.Layer(8, 256, 128, 2, group)
    dl = gu.DeviceLayer(L, seed=0)
    assert dl.s13.shape == (8, 256, 256 // group)
    for M in (4, 37):
        _run(dl, M)


@pytest.fixture(scope="module")
def group128_layer(gpu):
    return gu.DeviceLayer(synth.GROUP128.layer, seed=0)


@pytest.mark.parametrize("M", [1, 32, 256])
def test_second_shape_group128(group128_layer, M):
    _run(group128_layer, M, rows=None if M <= 32 else gu.sample_rows(M, 16))


def test_group_repeat_equals_group32(gpu):
    """A group-64 layer equals the group-32 layer whose scales repeat each
    value twice: both prepacked buffers must give bit-identical outputs."""
    L64 = synth.Layer(8, 256, 128, 2, 64)
    w13, s13, w2, s2 = synth.layer_weights(L64, 0)
    L32 = synth.Layer(8, 256, 128, 2, 32)
    d64 = gu.DeviceLayer(L64, weights=(w13, s13, w2, s2))
    d32 = gu.DeviceLayer(L32, weights=(w13, np.repeat(s13, 2, axis=2), w2, np.repeat(s2, 2, axis=2)))
    x = synth.hidden(16, 256, 4)
    ids, w = synth.routing(16, L64, 4)
    a, _ = d64.forward(x, ids, w)
    b, _ = d32.forward(x, ids, w)
    assert bool((a.view(-1) == b.view(-1)).all())


@pytest.fixture(scope="module")
def e256_layer(gpu):
    return gu.DeviceLayer(synth.E256.layer, seed=0)


@pytest.mark.parametrize("M", [1, 9, 90])
def test_e256(e256_layer, M):
    _run(e256_layer, M, rows=None if M <= 9 else gu.sample_rows(M, 16))


def test_shared_expert_slot(e128_layer):
    """Expert 127 serves every token with weight 1 next to the routed top-8:
    k = 9 slots per token (the router's 8 among experts 0..126)."""
    L = synth.SECOND.layer
    M = 48
    lg = synth.logits(M, L.E - 1, seed=6)
    rids, rw = synth.route(lg, L.k)
    ids = np.concatenate([rids, np.full((M, 1), L.E - 1, np.int32)], axis=1)
    w = np.concatenate([rw, np.ones((M, 1), np.float32)], axis=1)
    x = synth.hidden(M, L.H, 6)
    import quantized_moe_expert_align_gb300 as moe
    torch = gu.torch_mod()
    xd = gu.to_dev(x.view(np.int16)).view(torch.bfloat16)
    out = moe.forward(xd, gu.to_dev(ids), gu.to_dev(w), e128_layer.p13, e128_layer.p2, L.E, L.I)
    got = gu.bf16_dev_to_f64(out)
    gu.parity(got, e128_layer.oracle(x, ids, w), "shared expert")
