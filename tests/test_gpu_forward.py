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


def test_deterministic(e128_layer):
    x, ids, w = _inputs(synth.SECOND, 32)
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
