"""GPU layer forward against the oracle, within |d| <= 1e-2 + 1e-2*|ref|
elementwise and relative L2 <= 5e-3, on the workloads' seeded inputs.  Small
batches are compared in full; large ones on sampled token rows (the forward
still runs on the whole batch; each token's output depends only on its own
row, ids and weights)."""
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


def _check(dl, wl, M, sample=None):
    x, ids, w = _inputs(wl, M)
    out, ws = dl.forward(x, ids, w)
    import quantized_moe_expert_align_gb300 as moe
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    got = gu.bf16_dev_to_f64(out)
    rows = None if sample is None else gu.sample_rows(M, sample)
    ref = dl.oracle(x, ids, w, rows)
    return gu.parity(got if rows is None else got[rows], ref, f"{wl.name} M={M}")


def test_toy_full(toy_layer):
    _check(toy_layer, synth.TOY, 4)


@pytest.mark.parametrize("M", [1, 9, 90])
def test_decode_e384(e384_layer, M):
    _check(e384_layer, synth.DECODE, M)


@pytest.mark.parametrize("M", [1, 32])
def test_second_shape_small(e128_layer, M):
    _check(e128_layer, synth.SECOND, M)


@pytest.mark.parametrize("M", [4, 32])
def test_deterministic(e128_layer, M):
    # M = 4: gather inside the alignment and combine inside the down GEMM
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
    out, _ = toy_layer.forward(x, ids, w)
    gu.parity(gu.bf16_dev_to_f64(out), toy_layer.oracle(x, ids, w), "toy duplicates")


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
    out, ws = dl.forward(x, ids, w)
    import quantized_moe_expert_align_gb300 as moe
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    gu.parity(gu.bf16_dev_to_f64(out), dl.oracle(x, ids, w), f"wide scale in {which}")


# ---- larger batches: the forward runs on the whole batch, the oracle on a sample
@pytest.mark.parametrize("M", [256, 512, 1024])
def test_plateau_e384_sampled(e384_layer, M):
    _check(e384_layer, synth.PLATEAU, M, sample=24)


@pytest.mark.parametrize("M", [4096, 16384])
def test_prefill_zipf_e384_sampled(e384_layer, M):
    _check(e384_layer, synth.PREFILL, M, sample=16)


@pytest.mark.parametrize("M", [256, 2048])
def test_second_shape_sampled(e128_layer, M):
    _check(e128_layer, synth.SECOND, M, sample=24)


def test_token_tile_64(e128_layer):
    """A batch whose rows per expert select 64-row token tiles."""
    import quantized_moe_expert_align_gb300 as moe
    _check(e128_layer, synth.SECOND, 800, sample=24)
    assert moe.moe_w4a16_get_diag()["token_tile"] == 64


# ---- stage-level checks: the sorted intermediates against the oracle's
def _stages(dl, wl, M, rows_cap=None):
    import quantized_moe_expert_align_gb300 as moe
    L = wl.layer
    x, ids, w = _inputs(wl, M)
    out, ws = dl.forward(x, ids, w)
    inter = moe.intermediates(ws, M, L.k, L.E, L.H, L.I)
    import oracle
    ref = oracle.forward(x, ids, w, dl.w13, dl.s13, dl.w2, dl.s2, L.E, L.H, L.I,
                         want_intermediates=True)
    assert np.array_equal(inter["offsets"], ref["offsets"])
    n = int(ref["offsets"][-1])
    assert np.array_equal(inter["perm"][:n], ref["perm"][:n])
    for name, got, exp in [("act", inter["act"], ref["act"]), ("y", inter["y"], ref["y"])]:
        d = np.abs(got - exp)
        tol = 1e-3 + 1e-3 * np.abs(exp)
        assert np.all(d <= tol), f"{name}: {int(np.sum(d > tol))} bad, max d/tol {float(np.max(d / tol)):.3f}"


def test_stages_toy(toy_layer):
    _stages(toy_layer, synth.TOY, 4)


@pytest.mark.parametrize("M", [1, 9])
def test_stages_decode(e384_layer, M):
    _stages(e384_layer, synth.DECODE, M)
