"""Router front-end on the GPU (moe_route_align, moe_w4a16_forward_routed)
against the oracle's router.

* ids: bit-exact.  Both sides decide the order by comparing the same fp32
  logits (no arithmetic is involved), so the selection is unique.
* weights: the GPU computes exp(l_j - l_0) / sum_i exp(l_i - l_0) in fp32
  (one rounded subtraction, expf within 2 ulp, a 6-level sum, one division),
  the oracle the renormalised full softmax in double.  With x_j = l_j - l_0
  the fp32 result is within (|x_j| + k + 16) * 2^-24 relative of the exact
  value (the rounding of x_j contributes |x_j| * 2^-24 through exp; the
  k-term sum of values <= 1, whose largest is 1, at most (k/e + 10) * 2^-24;
  expf, the division and the oracle's own fp32 rounding 4 * 2^-24), plus
  2^-120 absolute for results in the subnormal range.
* the alignment of the routed ids: bit-exact against the oracle's alignment.
"""
import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _weight_tol(lg, ids, w_ref):
    lg = lg.astype(np.float64)
    sel = np.take_along_axis(lg, ids.astype(np.int64), axis=1)
    x = sel - sel[:, :1]
    x = np.where(np.isfinite(x), x, 0.0)
    k = ids.shape[1]
    return (np.abs(x) + k + 16) * 2.0 ** -24 * np.abs(w_ref.astype(np.float64)) + 2.0 ** -120


def _route_gpu(lg, k):
    import quantized_moe_expert_align_gb300 as moe
    torch = gu.torch_mod()
    ids, w, counts, offsets, perm, inv_perm, ws = moe.route_align(gu.to_dev(lg), k)
    torch.cuda.synchronize()
    st, detail = moe.moe_w4a16_get_device_status(ws)
    return ({"ids": ids.cpu().numpy(), "w": w.cpu().numpy(), "counts": counts.cpu().numpy(),
             "offsets": offsets.cpu().numpy(), "perm": perm.cpu().numpy(),
             "inv_perm": inv_perm.cpu().numpy()}, st, detail)


def _check_route(lg, k, expect_bad_rows=()):
    import oracle
    import quantized_moe_expert_align_gb300 as moe
    M, E = lg.shape
    got, st, detail = _route_gpu(lg, k)
    ids, w, bad = oracle.route(lg, k)
    assert np.array_equal(got["ids"], ids), "ids differ"
    tol = _weight_tol(lg, ids, w)
    d = np.abs(got["w"].astype(np.float64) - w.astype(np.float64))
    assert np.all(d <= tol), f"weights: {int(np.sum(d > tol))} out of tolerance, max d/tol {float(np.max(d / tol)):.3f}"
    counts, offsets, perm, inv_perm, n_bad = oracle.align(ids, E)
    assert n_bad == 0
    assert np.array_equal(got["counts"], counts) and np.array_equal(got["offsets"], offsets)
    n = M * k
    assert np.array_equal(got["perm"][:n], perm) and np.array_equal(got["inv_perm"][:n], inv_perm)
    if expect_bad_rows:
        assert bad == len(expect_bad_rows)
        assert st == moe.MOE_ERR_DEVICE_BAD_LOGIT and detail in expect_bad_rows
    else:
        assert bad == 0 and st == moe.MOE_OK, moe.moe_status_string(st)
    return got


# batches up to 64 tokens are routed inside the alignment kernel, larger ones
# by the separate routing kernel: both sides of that boundary are covered
@pytest.mark.parametrize("wl,M", [(synth.TOY, 4), (synth.DECODE, 1), (synth.DECODE, 9),
                                  (synth.DECODE, 64), (synth.DECODE, 65), (synth.DECODE, 90),
                                  (synth.PLATEAU, 1024), (synth.PREFILL, 4096),
                                  (synth.PREFILL, 16384), (synth.SECOND, 1), (synth.SECOND, 32),
                                  (synth.SECOND, 2048)])
def test_route_workload_logits(gpu, wl, M):
    L = wl.layer
    lg = synth.logits(M, L.E, seed=0, zipf_s=wl.zipf_s)
    got = _check_route(lg, L.k)
    # the routed ids are the ones the layer workloads are generated with
    ids_ref, _ = synth.route(lg, L.k)
    assert np.array_equal(got["ids"], ids_ref)


@pytest.mark.parametrize("M,E,k", [(5, 1024, 8), (100, 1024, 8), (3, 64, 64), (70, 64, 64),
                                   (50, 100, 7), (200, 100, 7), (33, 1, 1), (40, 33, 33)])
def test_route_shapes_and_ties(gpu, M, E, k):
    """E that is not a multiple of 32 (padded lanes), E = 1024 (32 logits a
    lane, always the routing kernel), k = E and k > 32 (two slots a lane),
    and tie-heavy logits with signed zeros (the lower index first)."""
    rng = np.random.default_rng(M * 131 + E)
    vals = np.array([-2.0, -0.0, 0.0, 0.5, 0.5, 1.25], np.float32)
    lg = vals[rng.integers(0, len(vals), size=(M, E))]
    lg[::2] += rng.standard_normal((lg[::2].shape)).astype(np.float32)   # some rows untied
    _check_route(lg.astype(np.float32), k)


@pytest.mark.parametrize("M", [6, 80])
def test_route_special_values(gpu, M):
    """NaN and +inf rows: reported, zero weights, NaN ranked last and +inf
    first; -inf: weight 0, ranked after every number; all -inf: zero weights."""
    rng = np.random.default_rng(5)
    E, k = 40, 6
    lg = rng.standard_normal((M, E)).astype(np.float32)
    lg[1, 3] = np.nan
    lg[2, 7] = np.inf
    lg[3, :30] = -np.inf
    lg[4, :] = -np.inf
    lg[5, [0, 9]] = np.nan
    got = _check_route(lg, k, expect_bad_rows=(1, 2, 5))
    assert np.all(got["w"][[1, 2, 4, 5]] == 0)
    assert got["ids"][2, 0] == 7
    assert np.all(got["w"][3, :] > 0)   # 10 finite logits left, k = 6


def test_route_empty_batch(gpu):
    import quantized_moe_expert_align_gb300 as moe
    torch = gu.torch_mod()
    lg = torch.empty((0, 16), dtype=torch.float32, device="cuda")
    ids, w, counts, offsets, perm, inv_perm, ws = moe.route_align(lg, 2)
    torch.cuda.synchronize()
    assert int(counts.sum()) == 0 and int(offsets[-1]) == 0


def _routed_forward(dl, wl, M, rows=None):
    import oracle
    import quantized_moe_expert_align_gb300 as moe
    torch = gu.torch_mod()
    L = wl.layer
    x = synth.hidden(M, L.H, seed=0)
    lg = synth.logits(M, L.E, seed=0, zipf_s=wl.zipf_s)
    xd = gu.to_dev(x.view(np.int16)).view(torch.bfloat16)
    ws = moe.Workspace(M, L.k, L.E, L.H, L.I, "cuda")
    out, ids_d, w_d = moe.forward_routed(xd, gu.to_dev(lg), L.k, dl.p13, dl.p2, L.E, L.I,
                                         workspace=ws)
    torch.cuda.synchronize()
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    ids, w, _ = oracle.route(lg, L.k)
    assert np.array_equal(ids_d.cpu().numpy(), ids)
    d = np.abs(w_d.cpu().numpy().astype(np.float64) - w)
    assert np.all(d <= _weight_tol(lg, ids, w))
    # the layer against the oracle fed with the oracle's own routing
    got = gu.bf16_dev_to_f64(out)
    ref = dl.oracle(x, ids, w, rows)
    gu.parity(got if rows is None else got[rows], ref, f"routed {wl.name} M={M}")
    return moe.moe_w4a16_get_diag()


def _launches(M, k):
    """Kernels of a forward from logits: the five kernels, the alignment
    kernel routing first up to 64 tokens, else a router kernel first."""
    return 5 if M <= 64 else 6


def test_forward_routed_toy(toy_layer):
    d = _routed_forward(toy_layer, synth.TOY, 4)
    assert d["kernels_launched"] == _launches(4, synth.TOY.layer.k)


@pytest.mark.parametrize("M", [1, 9, 90])
def test_forward_routed_decode(e384_layer, M):
    d = _routed_forward(e384_layer, synth.DECODE, M, rows=None if M < 90 else gu.sample_rows(M, 24))
    assert d["kernels_launched"] == _launches(M, synth.DECODE.layer.k)


def test_forward_routed_second_shape(e128_layer):
    _routed_forward(e128_layer, synth.SECOND, 32)


def test_forward_routed_small_batch_bad_logit(toy_layer):
    """A small routed batch (the alignment kernel routes it): a row with a
    NaN logit gets zero weights and is reported (its index as the detail),
    the other rows are routed as the oracle routes them."""
    import oracle
    import quantized_moe_expert_align_gb300 as moe
    torch = gu.torch_mod()
    L = synth.TOY.layer
    M = 6
    x = synth.hidden(M, L.H, seed=1)
    lg = synth.logits(M, L.E, seed=1)
    lg[2, 5] = np.nan
    ws = moe.Workspace(M, L.k, L.E, L.H, L.I, "cuda")
    xd = gu.to_dev(x.view(np.int16)).view(torch.bfloat16)
    out, ids_d, w_d = moe.forward_routed(xd, gu.to_dev(lg), L.k, toy_layer.p13, toy_layer.p2,
                                         L.E, L.I, workspace=ws)
    torch.cuda.synchronize()
    st, detail = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_ERR_DEVICE_BAD_LOGIT and detail == 2
    assert moe.moe_w4a16_get_diag()["kernels_launched"] == _launches(M, L.k)
    ids, w, _ = oracle.route(lg, L.k)
    assert np.array_equal(ids_d.cpu().numpy(), ids)
    assert np.all(w_d.cpu().numpy()[2] == 0)
    ok = [r for r in range(M) if r != 2]
    d = np.abs(w_d.cpu().numpy()[ok].astype(np.float64) - w[ok])
    assert np.all(d <= _weight_tol(lg[ok], ids[ok], w[ok]))


def test_forward_routed_wide_router_small_batch(gpu):
    """E = 1024 (32 logits a lane, beyond the alignment kernel's router):
    small batches run the router kernel ahead of the five kernels."""
    L = synth.Layer(1024, 256, 128, 8)
    dl = gu.DeviceLayer(L, 0)
    wl = synth.Workload("e1024 routed", L, (2,))
    d = _routed_forward(dl, wl, 2)
    assert d["kernels_launched"] == 6
