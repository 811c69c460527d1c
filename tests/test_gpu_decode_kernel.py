"""Small batches (at most 128 routed slots, 16-row token tiles) run the whole
layer as one cooperative kernel: alignment in every CTA, the hidden-row
gather, both GEMMs through one pipeline with per-chunk activation-ready
flags between them, and the combine by the last tile of each output slice.
These tests check that small batches take that path, that it matches the
oracle (output of every token, act and y of every slot) on the edges of its
range, and that the five-kernel path still does on the same batches when the
single kernel is switched off (MOE_W4A16_DECODE_FUSED=0, read once per
process, so in a child)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _full(dl, M, seed=0, ids=None, w=None):
    import quantized_moe_expert_align_gb300 as moe
    L = dl.layer
    x = synth.hidden(M, L.H, seed)
    if ids is None:
        ids, w = synth.routing(M, L, seed)
    out, ws = dl.forward(x, ids, w)
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    kernels = moe.moe_w4a16_get_diag()["kernels_launched"]
    what = f"E{L.E} H{L.H} I{L.I} k{L.k} M{M}"
    ref, _ = gu.check_stages(dl, x, ids, w, ws.buf, np.arange(M * L.k), what)
    gu.parity(gu.bf16_dev_to_f64(out), ref["out"], what)
    return kernels


@pytest.mark.parametrize("M", [1, 9, 16])
def test_one_kernel_decode_e384(e384_layer, M):
    assert _full(e384_layer, M) == 1


@pytest.mark.parametrize("M", [1, 16])
def test_one_kernel_second_shape(e128_layer, M):
    assert _full(e128_layer, M) == 1


def test_largest_one_kernel_batch_and_the_next(e128_layer):
    """k = 8: M = 16 is 128 slots (one kernel), M = 17 is 136 (five)."""
    import quantized_moe_expert_align_gb300 as moe
    assert _full(e128_layer, 16, seed=4) == 1
    assert _full(e128_layer, 17, seed=4) == 5


def test_every_expert_of_a_small_layer(gpu):
    """k = E = 64, two tokens: 128 slots over 64 experts of 2 rows each, one
    token tile per expert."""
    dl = gu.DeviceLayer(synth.Layer(64, 256, 128, 64), 0)
    assert _full(dl, 2) == 1


def test_one_expert_many_token_tiles(gpu):
    """64 of 120 slots on one expert of 64 (the token tile is chosen from the
    mean rows per expert, so it stays 16): that expert spans four token
    tiles, and the down GEMM waits on the gate+up tiles of each of them."""
    L = synth.Layer(64, 256, 256, 1)
    dl = gu.DeviceLayer(L, 0)
    M = 120
    ids = (np.arange(M) % 64).astype(np.int32).reshape(M, 1)
    ids[::2] = 5
    w = np.ones((M, 1), np.float32)
    assert _full(dl, M, ids=ids, w=w) == 1


def test_invalid_ids_only(toy_layer):
    """No slot has a valid id: the output is zero and the status says so."""
    import quantized_moe_expert_align_gb300 as moe
    L = synth.TOY.layer
    x = synth.hidden(3, L.H, seed=2)
    ids = np.array([[-1, 8], [9, -5], [100, 8]], np.int32)
    w = np.full((3, 2), 0.5, np.float32)
    out, ws = toy_layer.forward(x, ids, w)
    st, detail = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_ERR_DEVICE_BAD_EXPERT_ID and detail == -1
    assert bool((out.float() == 0).all())


def test_repeated_calls_reuse_the_workspace(e128_layer):
    """Back-to-back one-kernel calls on one workspace (the kernel zeroes its
    own tickets and flags each call) give bit-identical results, also after
    a call with other inputs in between."""
    import quantized_moe_expert_align_gb300 as moe
    L = synth.SECOND.layer
    ws = moe.Workspace(16, L.k, L.E, L.H, L.I, "cuda")
    x, (ids, w) = synth.hidden(16, L.H, 1), synth.routing(16, L, 1)
    a, _ = e128_layer.forward(x, ids, w, workspace=ws)
    a = a.clone()
    x2, (ids2, w2) = synth.hidden(5, L.H, 2), synth.routing(5, L, 2)
    e128_layer.forward(x2, ids2, w2, workspace=ws)
    b, _ = e128_layer.forward(x, ids, w, workspace=ws)
    assert bool((a.view(-1) == b.view(-1)).all())


_CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import synth
from tests import gpu_util as gu
import quantized_moe_expert_align_gb300 as moe
res = []
for L, M in ((synth.TOY.layer, 4), (synth.SECOND.layer, 1), (synth.SECOND.layer, 16)):
    dl = gu.DeviceLayer(L, 0)
    x = synth.hidden(M, L.H, 0)
    ids, w = synth.routing(M, L, 0)
    out, ws = dl.forward(x, ids, w)
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    kernels = moe.moe_w4a16_get_diag()["kernels_launched"]
    ref, _ = gu.check_stages(dl, x, ids, w, ws.buf, np.arange(M * L.k), f"E{L.E} M{M}")
    ratio, rel = gu.parity(gu.bf16_dev_to_f64(out), ref["out"], f"E{L.E} M{M} five kernels")
    res.append({"E": L.E, "M": M, "status": st, "kernels": kernels, "ratio": ratio})
print(json.dumps(res))
"""


def test_five_kernel_path_on_small_batches(gpu):
    env = dict(os.environ, MOE_W4A16_DECODE_FUSED="0")
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    for row in res:
        assert row["status"] == 0 and row["kernels"] == 5, row
