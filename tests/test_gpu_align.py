"""GPU alignment (moe_align) against the oracle: bit-exact counts, offsets,
permutation and inverse permutation on every workload's routing, plus edge
cases (M = 0, one slot, duplicate ids, out-of-range ids, all slots on one
expert)."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


def _run(ids, E):
    import torch
    import quantized_moe_expert_align_gb300 as moe
    idd = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    counts, offsets, perm, inv_perm, ws = moe.align(idd, E)
    st, detail = moe.moe_w4a16_get_device_status(ws)
    return (counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy(),
            inv_perm.cpu().numpy(), st, detail)


def _check(ids, E):
    c, o, p, ip, st, detail = _run(ids, E)
    rc, ro, rp, rip, bad = oracle.align(ids, E)
    assert np.array_equal(c, rc), "counts"
    assert np.array_equal(o, ro), "offsets"
    n = ro[E]
    assert np.array_equal(p[:n], rp[:n]), "perm"
    assert np.all(p[n:] == -1), "perm tail"
    assert np.array_equal(ip, rip), "inv_perm"
    return st, detail, bad


CASES = [(w.name, M) for w in synth.WORKLOADS.values() for M in w.Ms]


@pytest.mark.parametrize("name,M", CASES, ids=[f"{n}-M{m}" for n, m in CASES])
def test_align_bit_exact(gpu, name, M):
    import quantized_moe_expert_align_gb300 as moe
    wl = synth.WORKLOADS[name]
    ids, _ = synth.routing(M, wl.layer, seed=0, zipf_s=wl.zipf_s)
    st, _, bad = _check(ids, wl.layer.E)
    assert st == moe.MOE_OK and bad == 0


def test_align_edge_cases(gpu):
    import quantized_moe_expert_align_gb300 as moe
    rng = np.random.default_rng(0)
    # one slot; every slot on one expert; duplicates; E = 1; E = 1024
    for ids, E in [(np.array([[5]]), 8), (np.full((300, 8), 3), 384),
                   (rng.integers(0, 4, size=(77, 6)), 4), (np.zeros((50, 2)), 1),
                   (rng.integers(0, 1024, size=(999, 8)), 1024),
                   (rng.integers(0, 384, size=(16384, 8)), 384),
                   (rng.integers(0, 384, size=(256, 8)), 384),      # the one-CTA maximum
                   (rng.integers(0, 5, size=(1111, 3)), 5)]:
        st, _, bad = _check(np.asarray(ids, np.int32), E)
        assert st == moe.MOE_OK and bad == 0
    # M = 0 writes zero counts/offsets
    c, o, p, ip, st, _ = _run(np.zeros((0, 8), np.int32), 16)
    assert np.all(c == 0) and np.all(o == 0) and st == moe.MOE_OK


def test_align_out_of_range_ids(gpu):
    import quantized_moe_expert_align_gb300 as moe
    ids = np.array([[0, 4], [-1, 2], [2, 0], [3, 1 << 30]], np.int32)
    st, detail, bad = _check(ids, 4)
    assert bad == 3
    assert st == moe.MOE_ERR_DEVICE_BAD_EXPERT_ID and detail in (4, -1, 1 << 30)
    # one CTA, segments of several 8-step batches with a ragged end
    rng = np.random.default_rng(3)
    ids = rng.integers(0, 200, size=(1500, 8)).astype(np.int32)
    ids[::37, 2] = -3
    ids[1499, 7] = 200
    st, detail, bad = _check(ids, 200)
    assert bad == len(range(0, 1500, 37)) + 1
    assert st == moe.MOE_ERR_DEVICE_BAD_EXPERT_ID and detail in (-3, 200)


def test_align_large_batches(gpu):
    """More than 2048 slots take the multi-CTA path (per-segment counts,
    one scan, per-segment placement): still the same stable counting sort,
    out-of-range ids included."""
    import quantized_moe_expert_align_gb300 as moe
    rng = np.random.default_rng(11)
    for ids, E in [(rng.integers(0, 384, size=(2049, 1)), 384),       # just above the switch
                   (rng.integers(0, 384, size=(16385, 1)), 384),
                   (rng.integers(0, 1024, size=(3000, 8)), 1024),
                   (np.zeros((5000, 4)), 1),
                   (np.full((2100, 8), 17), 64),                      # one expert takes all
                   (rng.integers(0, 7, size=(4099, 5)), 7)]:
        st, _, bad = _check(np.asarray(ids, np.int32), E)
        assert st == moe.MOE_OK and bad == 0
    ids = rng.integers(0, 96, size=(2500, 8)).astype(np.int32)
    ids[::97, 3] = -5
    ids[5, 0] = 96
    st, detail, bad = _check(ids, 96)
    assert bad == 26 + 1
    assert st == moe.MOE_ERR_DEVICE_BAD_EXPERT_ID and detail in (-5, 96)


@pytest.mark.parametrize("M,k,E", [(37, 8, 384), (2500, 8, 96)])
def test_align_without_inv_perm(gpu, M, k, E):
    """inv_perm may be NULL (one CTA and the 32-CTA path): the rest is
    unchanged."""
    import torch
    import quantized_moe_expert_align_gb300 as moe
    rng = np.random.default_rng(M)
    ids = rng.integers(0, E, size=(M, k)).astype(np.int32)
    idd = torch.from_numpy(ids).cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(M * k, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(moe.moe_align_workspace_size(M, k, E), 256), dtype=torch.uint8,
                     device="cuda")
    assert moe.moe_align(idd, M, k, E, counts, offsets, perm, None, ws) == moe.MOE_OK
    torch.cuda.synchronize()
    rc, ro, rp, _, _ = oracle.align(ids, E)
    assert np.array_equal(counts.cpu().numpy(), rc) and np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
