"""GPU layer forward against the oracle, within |d| <= 1e-2 + 1e-2*|ref|
elementwise and relative L2 <= 5e-3, on the workloads' seeded inputs.

Every workload up to M = 2048 is compared in full: the layer output of every
token, and the two GEMMs' sorted intermediates (act = silu(gate)*up and the
down projection y) of every slot, element by element, against the oracle's.
The Zipf prefill batches (M = 4096 and 16384) are checked on slots chosen
from the tile structure -- the first and last row of every token tile of both
GEMMs, every row of the heaviest expert (M = 4096), the first and last token
tile of the four heaviest experts -- plus the full output rows of sampled
tokens."""
import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _inputs(wl, M, seed=0):
    L = wl.layer
    x = synth.hidden(M, L.H, seed)
    ids, w = synth.routing(M, L, seed, zipf_s=wl.zipf_s)
    return x, ids, w


def _forward_ok(dl, x, ids, w):
    import quantized_moe_expert_align_gb300 as moe
    out, ws = dl.forward(x, ids, w)
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    return out, ws


def _full(dl, wl, M, stages=True):
    """The whole batch: output of every token; with ``stages`` also act and
    y of every slot (one oracle run gives both)."""
    x, ids, w = _inputs(wl, M)
    out, ws = _forward_ok(dl, x, ids, w)
    got = gu.bf16_dev_to_f64(out)
    what = f"{wl.name} M={M}"
    if stages:
        ref, toks = gu.check_stages(dl, x, ids, w, ws.buf, np.arange(M * wl.layer.k), what)
        assert len(toks) == M
        return gu.parity(got, ref["out"], what)
    return gu.parity(got, dl.oracle(x, ids, w), what)


def test_toy_full(toy_layer):
    _full(toy_layer, synth.TOY, 4)


@pytest.mark.parametrize("M", [1, 9, 90])
def test_decode_e384(e384_layer, M):
    _full(e384_layer, synth.DECODE, M)


@pytest.mark.parametrize("M", [1, 32, 256, 2048])
def test_second_shape(e128_layer, M):
    """M = 2048: 160-row token tiles of the gate+up GEMM (80 for the down
    GEMM), round-robin whole tiles."""
    import quantized_moe_expert_align_gb300 as moe
    _full(e128_layer, synth.SECOND, M)
    if M == 2048:
        d = moe.moe_w4a16_get_diag()
        assert d["token_tile"] == 160 and d["token_tile2"] == 80


@pytest.mark.parametrize("M", [256, 512, 1024])
def test_plateau_e384(e384_layer, M):
    _full(e384_layer, synth.PLATEAU, M)


def test_token_tile_64(e128_layer):
    """A batch whose rows per expert select 64-row token tiles."""
    import quantized_moe_expert_align_gb300 as moe
    _full(e128_layer, synth.SECOND, 800)
    assert moe.moe_w4a16_get_diag()["token_tile"] == 64


@pytest.mark.parametrize("M", [4, 32])
def test_deterministic(e128_layer, M):
    # two calls on the same inputs give bit-identical outputs (split tiles are
    # reduced in a fixed order, whichever CTA finishes last)
    x, ids, w = _inputs(synth.SECOND, M)
    a, _ = e128_layer.forward(x, ids, w)
    b, _ = e128_layer.forward(x, ids, w)
    assert bool((a.view(-1) == b.view(-1)).all())


def test_duplicate_ids_and_ragged(toy_layer):
    L = synth.TOY.layer
    rng = np.random.default_rng(3)
    M = 37
    x = synth.hidden(M, L.H, seed=5)
    ids = rng.integers(0, L.E, size=(M, L.k)).astype(np.int32)
    ids[::3, 1] = ids[::3, 0]                      # duplicate ids in some rows
    w = rng.random((M, L.k)).astype(np.float32)
    out, ws = toy_layer.forward(x, ids, w)
    ref, _ = gu.check_stages(toy_layer, x, ids, w, ws.buf, np.arange(M * L.k), "toy duplicates")
    gu.parity(gu.bf16_dev_to_f64(out), ref["out"], "toy duplicates")


def _bf16(v):
    return synth.f32_to_bf16_bits(np.array([v], np.float32))[0]


@pytest.mark.parametrize("which", ["w13", "w2"])
def test_wide_and_zero_scales(gpu, which):
    """A scale above 65504/24 (here 2800, on a group whose only nonzero
    weight is one code 9, so the activations stay in fp16 range) moves that
    matrix to the two-step dequantisation; zero scales give zero weights.
    Both against the oracle."""
    L = synth.TOY.layer
    w13, s13, w2, s2 = (a.copy() for a in synth.layer_weights(L, 0))
    codes, sc = (w13, s13) if which == "w13" else (w2, s2)
    for e in range(L.E):
        sc[e, 3, 0] = _bf16(2800.0)
        codes[e, 3, :16] = np.array([0x89] + [0x88] * 15, np.uint8)  # q - 8 = 1, 0, 0, ...
        sc[e, 5, :] = 0
    dl = gu.DeviceLayer(L, 0, weights=(w13, s13, w2, s2))
    M = 16
    x = synth.hidden(M, L.H, seed=2)
    ids, w = synth.routing(M, L, seed=2)
    out, ws = _forward_ok(dl, x, ids, w)
    gu.parity(gu.bf16_dev_to_f64(out), dl.oracle(x, ids, w), f"wide scale in {which}")


# ---- Zipf prefill: the 32-CTA alignment (more than 2048 slots), 128- and
# 160-row token tiles, experts spanning many token tiles
@pytest.mark.parametrize("M,heavy_full,tile", [(4096, 1, 128), (16384, 0, 160)])
def test_prefill_zipf_e384(e384_layer, M, heavy_full, tile):
    import quantized_moe_expert_align_gb300 as moe
    wl = synth.PREFILL
    L = wl.layer
    x, ids, w = _inputs(wl, M)
    out, ws = _forward_ok(e384_layer, x, ids, w)
    d = moe.moe_w4a16_get_diag()
    nt, nt2 = d["token_tile"], d["token_tile2"]
    assert nt == tile and nt2 == 80
    slots = gu.tile_sample(ids, L.E, nt, nt2, heavy_full=heavy_full)
    gu.check_stages(e384_layer, x, ids, w, ws.buf, slots, f"{wl.name} M={M}")
    # output rows of sampled tokens (each depends only on its own row, ids
    # and weights)
    rows = gu.sample_rows(M, 16)
    gu.parity(gu.bf16_dev_to_f64(out)[rows], e384_layer.oracle(x, ids, w, rows),
              f"{wl.name} M={M} sampled tokens")


def test_small_batch_path(e128_layer):
    """Batches of at most 128 slots run four kernels (one aligns in every
    CTA and gathers), larger ones five; both match the oracle in full."""
    import quantized_moe_expert_align_gb300 as moe
    for M, kernels in ((16, 4), (17, 5)):
        _full(e128_layer, synth.SECOND, M)
        assert moe.moe_w4a16_get_diag()["kernels_launched"] == kernels
