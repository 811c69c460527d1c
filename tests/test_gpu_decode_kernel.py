"""The single small-batch kernel (opt-in, MOE_W4A16_DECODE_FUSED=1, read once
per process, so every check here runs in a child process with the switch
set): batches of at most 128 routed slots with 16-row token tiles run the
whole layer as one cooperative kernel -- alignment in every CTA, the
hidden-row gather, both GEMMs through one pipeline with per-chunk
activation-ready flags between them, and the combine by the last tile of
each output slice.

The child checks, against the oracle (output of every token, act and y of
every slot), that small batches take the one-kernel path and larger ones
the five kernels; the edges of the path's range; a batch with no valid slot;
back-to-back calls on one workspace; the allocation-free entry point and a
CUDA-graph replay on that path (both bit-identical to the plain call)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
import synth
from tests import gpu_util as gu
import quantized_moe_expert_align_gb300 as moe

res = {}


def full(dl, M, seed=0, ids=None, w=None):
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
    ratio, _ = gu.parity(gu.bf16_dev_to_f64(out), ref["out"], what)
    return {"kernels": kernels, "ratio": ratio}


def case(name, fn):
    try:
        res[name] = fn()
    except Exception as e:  # reported to the parent, which fails the test
        res[name] = {"error": repr(e)[:400]}


e128 = gu.DeviceLayer(synth.SECOND.layer, 0)
for M in (1, 16):
    case(f"e128_M{M}", lambda M=M: full(e128, M))
case("e128_M17", lambda: full(e128, 17, seed=4))
small = gu.DeviceLayer(synth.Layer(64, 256, 128, 64), 0)
case("every_expert", lambda: full(small, 2))


def many_tiles():
    L = synth.Layer(64, 256, 256, 1)
    dl = gu.DeviceLayer(L, 0)
    M = 120
    ids = (np.arange(M) % 64).astype(np.int32).reshape(M, 1)
    ids[::2] = 5          # 62 slots on expert 5: four 16-row token tiles
    return full(dl, M, ids=ids, w=np.ones((M, 1), np.float32))


case("one_expert_many_tiles", many_tiles)
toy = gu.DeviceLayer(synth.TOY.layer, 0)


def invalid_only():
    L = synth.TOY.layer
    x = synth.hidden(3, L.H, seed=2)
    ids = np.array([[-1, 8], [9, -5], [100, 8]], np.int32)
    out, ws = toy.forward(x, ids, np.full((3, 2), 0.5, np.float32))
    st, detail = moe.moe_w4a16_get_device_status(ws.buf)
    return {"status": st, "detail": detail, "zero": bool((out.float() == 0).all())}


case("invalid_only", invalid_only)


def repeated():
    L = synth.SECOND.layer
    ws = moe.Workspace(16, L.k, L.E, L.H, L.I, "cuda")
    x, (ids, w) = synth.hidden(16, L.H, 1), synth.routing(16, L, 1)
    a, _ = e128.forward(x, ids, w, workspace=ws)
    a = a.clone()
    x2, (ids2, w2) = synth.hidden(5, L.H, 2), synth.routing(5, L, 2)
    e128.forward(x2, ids2, w2, workspace=ws)
    b, _ = e128.forward(x, ids, w, workspace=ws)
    return {"same": bool((a.view(-1) == b.view(-1)).all())}


case("repeated", repeated)


def static_and_graph():
    L = synth.SECOND.layer
    M = 4
    x = gu.to_dev(synth.hidden(M, L.H, 3).view(np.int16)).view(torch.bfloat16)
    ids, w = synth.routing(M, L, 3)
    idd, wd = gu.to_dev(ids), gu.to_dev(w)
    ref = moe.forward(x, idd, wd, e128.p13, e128.p2, L.E, L.I)
    torch.cuda.synchronize()
    out = torch.empty_like(ref)
    st = moe.moe_w4a16_forward_static(x, idd, wd, e128.p13, e128.p2, out, M, L.k, L.E, L.H, L.I)
    torch.cuda.synchronize()
    same_static = st == moe.MOE_OK and bool((out.view(-1) == ref.view(-1)).all())
    ws = moe.Workspace(M, L.k, L.E, L.H, L.I, "cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        moe.moe_w4a16_forward(x, idd, wd, e128.p13, e128.p2, out, M, L.k, L.E, L.H, L.I, ws.buf)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st_c = moe.moe_w4a16_forward(x, idd, wd, e128.p13, e128.p2, out, M, L.k, L.E, L.H, L.I, ws.buf)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    st_g, _ = moe.moe_w4a16_get_device_status(ws.buf)
    return {"static": same_static, "capture": st_c, "status": st_g,
            "graph": bool((out.view(-1) == ref.view(-1)).all())}


case("static_and_graph", static_and_graph)
e384 = gu.DeviceLayer(synth.DECODE.layer, 0)
for M in (1, 9, 16):
    case(f"e384_M{M}", lambda M=M: full(e384, M))
print(json.dumps(res))
"""


@pytest.fixture(scope="module")
def one_kernel_results(gpu):
    env = dict(os.environ, MOE_W4A16_DECODE_FUSED="1")
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def _ok(res, name, kernels):
    row = res[name]
    assert "error" not in row, row
    assert row["kernels"] == kernels, row


@pytest.mark.parametrize("M", [1, 9, 16])
def test_one_kernel_decode_e384(one_kernel_results, M):
    _ok(one_kernel_results, f"e384_M{M}", 1)


@pytest.mark.parametrize("M", [1, 16])
def test_one_kernel_second_shape(one_kernel_results, M):
    _ok(one_kernel_results, f"e128_M{M}", 1)


def test_largest_one_kernel_batch_and_the_next(one_kernel_results):
    """k = 8: M = 16 is 128 slots (one kernel), M = 17 is 136 (five)."""
    _ok(one_kernel_results, "e128_M16", 1)
    _ok(one_kernel_results, "e128_M17", 5)


def test_every_expert_of_a_small_layer(one_kernel_results):
    """k = E = 64, two tokens: 128 slots, 64 experts of 2 rows each."""
    _ok(one_kernel_results, "every_expert", 1)


def test_one_expert_many_token_tiles(one_kernel_results):
    """62 of 120 slots on one expert of 64: four token tiles, so the down
    GEMM waits on the gate+up tiles of each of them."""
    _ok(one_kernel_results, "one_expert_many_tiles", 1)


def test_invalid_ids_only(one_kernel_results):
    """No slot has a valid id: the output is zero and the status says so."""
    import quantized_moe_expert_align_gb300 as moe
    row = one_kernel_results["invalid_only"]
    assert "error" not in row, row
    assert row["status"] == moe.MOE_ERR_DEVICE_BAD_EXPERT_ID and row["detail"] == -1
    assert row["zero"]


def test_repeated_calls_reuse_the_workspace(one_kernel_results):
    """The kernel zeroes its own tickets and flags each call: back-to-back
    calls on one workspace give bit-identical results."""
    row = one_kernel_results["repeated"]
    assert row.get("same") is True, row


def test_static_entry_point_and_graph_replay(one_kernel_results):
    """The allocation-free entry point and a CUDA-graph replay of the
    one-kernel forward equal the plain call bit for bit."""
    import quantized_moe_expert_align_gb300 as moe
    row = one_kernel_results["static_and_graph"]
    assert "error" not in row, row
    assert row["static"] and row["capture"] == moe.MOE_OK
    assert row["status"] == moe.MOE_OK and row["graph"]
