"""Device-side error reporting: out-of-range expert ids, mismatched prepacked
buffers, fp16 range; and M = 0.  None of these faults or traps the GPU: the
kernels record a status word and skip the affected work."""
import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_invalid_ids_contribute_zero(toy_layer):
    import quantized_moe_expert_align_gb300 as moe
    L = synth.TOY.layer
    x = synth.hidden(3, L.H, seed=2)
    ids = np.array([[0, 9], [-3, 2], [1, 3]], np.int32)
    w = np.full((3, 2), 0.5, np.float32)
    out, ws = toy_layer.forward(x, ids, w)
    st, detail = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_ERR_DEVICE_BAD_EXPERT_ID and detail in (9, -3)
    gu.parity(gu.bf16_dev_to_f64(out), toy_layer.oracle(x, ids, w), "invalid ids")
    # the next clean call on the same workspace reports OK again
    ids2 = np.array([[0, 1], [2, 3], [4, 5]], np.int32)
    out, ws = toy_layer.forward(x, ids2, w, workspace=ws)
    assert moe.moe_w4a16_get_device_status(ws.buf)[0] == moe.MOE_OK


def test_swapped_buffers_report_bad_layout(toy_layer):
    import torch
    import quantized_moe_expert_align_gb300 as moe
    L = synth.TOY.layer
    x = gu.to_dev(synth.hidden(4, L.H).view(np.int16)).view(torch.bfloat16)
    ids, w = synth.routing(4, L)
    ws = moe.Workspace(4, L.k, L.E, L.H, L.I, "cuda")
    p13, p2 = toy_layer.p13, toy_layer.p2
    moe.forward(x, gu.to_dev(ids), gu.to_dev(w), p2, p13, L.E, L.I,
                workspace=ws)
    assert moe.moe_w4a16_get_device_status(ws.buf)[0] == moe.MOE_ERR_BAD_LAYOUT


def test_hidden_beyond_fp16_range(toy_layer):
    import quantized_moe_expert_align_gb300 as moe
    L = synth.TOY.layer
    x = synth.hidden(4, L.H)
    x[1, 7] = synth.f32_to_bf16_bits(np.array([1.0e5], np.float32))[0]
    ids, w = synth.routing(4, L)
    _, ws = toy_layer.forward(x, ids, w)
    assert moe.moe_w4a16_get_device_status(ws.buf)[0] == moe.MOE_ERR_DEVICE_FP16_RANGE


def test_prepack_rejects_scales_outside_fp16(gpu):
    import quantized_moe_expert_align_gb300 as moe
    L = synth.TOY.layer
    w13, s13, _, _ = synth.layer_weights(L)
    s13 = s13.copy()
    s13[2, 5, 1] = synth.f32_to_bf16_bits(np.array([1.0e-6], np.float32))[0]
    with pytest.raises(moe.MoeError) as ei:
        moe.prepack(moe.MOE_PACK_W13, gu.to_dev(w13), gu.to_dev(s13.view(np.int16)))
    assert ei.value.status == moe.MOE_ERR_DEVICE_FP16_RANGE


def test_m_zero_is_a_noop(toy_layer):
    import torch
    import quantized_moe_expert_align_gb300 as moe
    L = synth.TOY.layer
    ws = moe.Workspace(1, L.k, L.E, L.H, L.I, "cuda")
    out = torch.full((0, L.H), 1.0, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((0, L.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((0, L.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((0, L.k), dtype=torch.float32, device="cuda")
    moe.forward(x, ids, w, toy_layer.p13, toy_layer.p2,
                L.E, L.I, out=out, workspace=ws)
    torch.cuda.synchronize()


_STALL_CHILD = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
import synth
from tests import gpu_util as gu
import quantized_moe_expert_align_gb300 as moe
L = synth.TOY.layer
M = int(sys.argv[2]) if len(sys.argv) > 2 else 4
dl = gu.DeviceLayer(L, 0)
x = synth.hidden(M, L.H, 0)
ids, w = synth.routing(M, L, 0)
t0 = time.time()
out, ws = dl.forward(x, ids, w)
st, detail = moe.moe_w4a16_get_device_status(ws.buf)
secs = time.time() - t0
tile = moe.moe_w4a16_get_diag()["token_tile"]
# the context is still usable afterwards
y = (torch.arange(1024, device="cuda", dtype=torch.float32) * 2).sum().item()
print(json.dumps({"status": st, "detail": detail, "secs": secs, "y": y, "tile": tile}))
"""


def test_bounded_wait_runs_out(gpu):
    """With the failure-path switch the gate+up GEMM issues no copies: its
    waits give up after about a second, the status word says
    MOE_ERR_DEVICE_TIMEOUT (detail: the role whose wait gave up), the kernel
    winds down without hanging, and the CUDA context stays usable.  The
    switch is read once per process, so in a child."""
    import json
    import os
    import subprocess
    import sys

    import quantized_moe_expert_align_gb300 as moe
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MOE_W4A16_TEST_NO_COPIES="1")
    r = subprocess.run([sys.executable, "-c", _STALL_CHILD, root], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["status"] == moe.MOE_ERR_DEVICE_TIMEOUT, res
    assert 1 <= res["detail"] <= 6
    assert res["y"] == float(sum(2 * i for i in range(1024)))
    assert res["secs"] < 60


def test_bounded_wait_runs_out_cta_pairs(gpu):
    """The same with the GEMMs on CTA pairs (M = 300 on the toy layer:
    128-row gate+up and 80-row down tiles): every wait of both CTAs of a
    pair still gives up, the pair meets at its closing cluster barrier and
    the context stays usable."""
    import json
    import os
    import subprocess
    import sys

    import quantized_moe_expert_align_gb300 as moe
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MOE_W4A16_TEST_NO_COPIES="1")
    r = subprocess.run([sys.executable, "-c", _STALL_CHILD, root, "300"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["tile"] == 128, res
    assert res["status"] == moe.MOE_ERR_DEVICE_TIMEOUT, res
    assert 1 <= res["detail"] <= 6
    assert res["y"] == float(sum(2 * i for i in range(1024)))
    assert res["secs"] < 60


def test_bounded_wait_runs_out_one_kernel(gpu):
    """The same in the single small-batch kernel (opt-in switch set): no
    weight copy is issued, and the first wait to give up may also be a
    producer's wait for activation rows that another CTA never finishes
    (detail 7)."""
    import json
    import os
    import subprocess
    import sys

    import quantized_moe_expert_align_gb300 as moe
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MOE_W4A16_TEST_NO_COPIES="1", MOE_W4A16_DECODE_FUSED="1")
    r = subprocess.run([sys.executable, "-c", _STALL_CHILD, root], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["status"] == moe.MOE_ERR_DEVICE_TIMEOUT, res
    assert 1 <= res["detail"] <= 7
    assert res["y"] == float(sum(2 * i for i in range(1024)))
    assert res["secs"] < 60
