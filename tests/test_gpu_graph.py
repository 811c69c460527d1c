"""The forward is stream-ordered and capturable in a CUDA graph: a captured
forward, replayed, gives bit-identical outputs to the eager call, also
after new inputs are copied into the captured buffers."""
import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


# (M = 2048: the 32-CTA alignment and both GEMMs on CTA pairs, cluster launches
# inside the captured graph)
@pytest.mark.parametrize("wl,M", [(synth.TOY, 4), (synth.SECOND, 1), (synth.SECOND, 32),
                                  (synth.SECOND, 2048)])
def test_forward_in_cuda_graph(request, wl, M):
    import quantized_moe_expert_align_gb300 as moe
    torch = gu.torch_mod()
    dl = request.getfixturevalue("toy_layer" if wl is synth.TOY else "e128_layer")
    L = wl.layer

    def inputs(seed):
        x = synth.hidden(M, L.H, seed)
        ids, w = synth.routing(M, L, seed)
        return (gu.to_dev(x.view(np.int16)).view(torch.bfloat16), gu.to_dev(ids), gu.to_dev(w))

    x, ids, w = inputs(0)
    out = torch.empty((M, L.H), dtype=torch.bfloat16, device="cuda")
    ws = moe.Workspace(M, L.k, L.E, L.H, L.I, "cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up off the default stream, as capture wants
        assert moe.moe_w4a16_forward(x, ids, w, dl.p13, dl.p2, out, M, L.k, L.E, L.H, L.I,
                                     ws.buf) == moe.MOE_OK
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = out.clone()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = moe.moe_w4a16_forward(x, ids, w, dl.p13, dl.p2, out, M, L.k, L.E, L.H, L.I, ws.buf)
    assert st == moe.MOE_OK
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert bool((out.view(-1) == eager.view(-1)).all())

    # new inputs through the captured buffers
    x2, ids2, w2 = inputs(7)
    x.copy_(x2)
    ids.copy_(ids2)
    w.copy_(w2)
    g.replay()
    torch.cuda.synchronize()
    ref = torch.empty_like(out)
    assert moe.moe_w4a16_forward(x2, ids2, w2, dl.p13, dl.p2, ref, M, L.k, L.E, L.H, L.I,
                                 ws.buf) == moe.MOE_OK
    torch.cuda.synchronize()
    assert bool((out.view(-1) == ref.view(-1)).all())
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_OK
