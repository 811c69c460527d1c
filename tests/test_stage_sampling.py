"""The machinery behind the GPU stage-level checks, on the CPU: the oracle
run restricted to chosen slots (other slots' ids set to -1) gives exactly the
act and y rows of the unrestricted run for those slots, and the tile-structure
sample covers the rows it promises."""
import types

import numpy as np

import oracle
import synth
from tests import gpu_util as gu


def _layer(L, seed=0):
    w13, s13, w2, s2 = synth.layer_weights(L, seed)
    return types.SimpleNamespace(layer=L, w13=w13, s13=s13, w2=w2, s2=s2)


def test_restricted_oracle_equals_full_run():
    L = synth.Layer(16, 256, 128, 4)
    dl = _layer(L)
    M = 40
    x = synth.hidden(M, L.H, 1)
    ids, w = synth.routing(M, L, 1)
    full = oracle.forward(x, ids, w, dl.w13, dl.s13, dl.w2, dl.s2, L.E, L.H, L.I,
                          want_intermediates=True)
    rng = np.random.default_rng(0)
    slots = rng.choice(M * L.k, size=37, replace=False)
    s, ref, ref_pos, toks = gu.oracle_on_slots(dl, x, ids, w, slots)
    assert np.array_equal(s, np.unique(slots))
    pos = full["inv_perm"][s]
    assert np.array_equal(ref["act"][ref_pos], full["act"][pos])
    assert np.array_equal(ref["y"][ref_pos], full["y"][pos])
    # tokens whose every slot was kept have their full output
    s_all, ref_all, _, toks_all = gu.oracle_on_slots(dl, x, ids, w, np.arange(M * L.k))
    assert np.array_equal(toks_all, np.arange(M))
    assert np.array_equal(ref_all["out"], full["out"])


def test_tile_sample_covers_tile_edges_and_heavy_experts():
    L = synth.Layer(32, 256, 128, 8)
    M = 700
    ids, _ = synth.routing(M, L, 0, zipf_s=1.1)
    nt, nt2 = 128, 64
    slots = gu.tile_sample(ids, L.E, nt, nt2, heavy_full=1, heavy_edges=4)
    counts, offsets, perm, inv_perm, _ = oracle.align(ids, L.E)
    rows = set(inv_perm[slots].tolist())
    order = np.argsort(-counts, kind="stable")
    heavy = int(order[0])
    assert set(range(offsets[heavy], offsets[heavy + 1])) <= rows
    for e in range(L.E):
        c, o = int(counts[e]), int(offsets[e])
        for width in (nt, nt2):
            for s in range(0, c, width):
                assert o + s in rows and o + min(s + width, c) - 1 in rows
    for e in order[:4]:
        c, o = int(counts[e]), int(offsets[e])
        assert set(range(o + (c - 1) // nt * nt, o + c)) <= rows   # last (partial) tile
    assert len(rows) < M * L.k
