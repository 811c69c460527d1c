"""The allocation-free forward, moe_w4a16_forward_static.

It serves callers that cannot allocate device memory (a host framework that
owns every device allocation, a decode loop where cudaMalloc would
synchronise the device): instead of a caller-provided workspace it uses one
static device array inside the library.  Here it is called through the C ABI
twice in a row and must match the regular entry point, moe_w4a16_forward,
bit for bit: both run the same kernels on the same sizes, and the forward is
deterministic (split tiles are reduced in a fixed order), so any difference
would come from the static scratch itself.  A size whose workspace exceeds
the static array must be rejected before any launch.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""
import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _static_matches_regular(dl, wl, M):
    import torch
    import quantized_moe_expert_align_gb300 as moe
    L = wl.layer
    x = synth.hidden(M, L.H, seed=3)
    ids, w = synth.routing(M, L, seed=3, zipf_s=wl.zipf_s)
    ref, _ = dl.forward(x, ids, w)
    torch.cuda.synchronize()
    xd = gu.to_dev(x.view(np.int16)).view(torch.bfloat16)
    idd, wd = gu.to_dev(ids), gu.to_dev(w)
    for _ in range(2):
        out = torch.full((M, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = moe.moe_w4a16_forward_static(xd, idd, wd, dl.p13, dl.p2,
                                          out, M, L.k, L.E, L.H, L.I)
        assert st == moe.MOE_OK, moe.moe_status_string(st)
        torch.cuda.synchronize()
        same = out.view(torch.int16) == ref.view(torch.int16)
        assert bool(same.all()), (f"static scratch {wl.name} M={M}: "
                                  f"{int((~same).sum())} outputs differ from moe_w4a16_forward")


def test_static_toy(toy_layer):
    _static_matches_regular(toy_layer, synth.TOY, 4)


@pytest.mark.parametrize("M", [1, 9])
def test_static_decode_e384(e384_layer, M):
    _static_matches_regular(e384_layer, synth.DECODE, M)


def test_static_second_shape(e128_layer):
    _static_matches_regular(e128_layer, synth.SECOND, 32)


def test_static_rejects_sizes_beyond_the_array(e384_layer):
    import torch
    import quantized_moe_expert_align_gb300 as moe
    L = synth.DECODE.layer
    M = 256
    assert moe.moe_w4a16_workspace_size(M, L.k, L.E, L.H, L.I) > moe.MOE_W4A16_STATIC_SCRATCH_BYTES
    x = torch.zeros((M, L.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((M, L.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((M, L.k), dtype=torch.float32, device="cuda")
    out = torch.zeros((M, L.H), dtype=torch.bfloat16, device="cuda")
    dl = e384_layer
    st = moe.moe_w4a16_forward_static(x, ids, w, dl.p13, dl.p2, out,
                                      M, L.k, L.E, L.H, L.I)
    assert st == moe.MOE_ERR_WORKSPACE_TOO_SMALL
