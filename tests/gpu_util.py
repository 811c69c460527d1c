"""Helpers for the GPU parity tests: device copies of the seeded inputs,
prepacked layers, the parity criterion, and oracle runs on sampled tokens."""
from __future__ import annotations

import numpy as np

import synth

ATOL = 1e-2      # |gpu - oracle| <= ATOL + RTOL * |oracle|, elementwise
RTOL = 1e-2
REL_L2 = 5e-3    # ||gpu - oracle|| / ||oracle|| <= REL_L2


def torch_mod():
    import torch
    return torch


def to_dev(a: np.ndarray, dtype=None):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev_to_f64(t) -> np.ndarray:
    """bf16 device tensor -> float64 numpy (exact)."""
    return t.float().cpu().numpy().astype(np.float64)


class DeviceLayer:
    """Host canonical weights of one layer plus their prepacked device copies."""

    def __init__(self, layer: synth.Layer, seed: int = 0, weights=None):
        """``weights``: canonical (w13, s13, w2, s2) to use instead of the
        seeded ones."""
        import quantized_moe_expert_align_gb300 as moe
        self.layer = layer
        self.seed = seed
        self.w13, self.s13, self.w2, self.s2 = (weights if weights is not None
                                                else synth.layer_weights(layer, seed))
        torch = torch_mod()
        q = to_dev(self.w13)
        s = to_dev(self.s13.view(np.int16))
        self.p13 = moe.prepack(moe.MOE_PACK_W13, q, s)
        del q, s
        q = to_dev(self.w2)
        s = to_dev(self.s2.view(np.int16))
        self.p2 = moe.prepack(moe.MOE_PACK_W2, q, s)
        del q, s
        torch.cuda.synchronize()

    def forward(self, x_bits, ids, w, workspace=None, stream=None):
        """Run the library forward on host inputs; returns (out_dev, ws)."""
        import quantized_moe_expert_align_gb300 as moe
        torch = torch_mod()
        L = self.layer
        xd = to_dev(x_bits.view(np.int16)).view(torch.bfloat16)
        idd = to_dev(ids)
        wd = to_dev(w)
        M = ids.shape[0]
        ws = workspace if workspace is not None else moe.Workspace(M, L.k, L.E, L.H, L.I, "cuda")
        out = moe.forward(xd, idd, wd, self.p13, self.p2,
                          L.E, L.I, workspace=ws, stream=stream)
        return out, ws

    def oracle(self, x_bits, ids, w, rows=None):
        import oracle
        L = self.layer
        if rows is not None:
            x_bits, ids, w = x_bits[rows], ids[rows], w[rows]
        return oracle.forward(x_bits, ids, w, self.w13, self.s13, self.w2, self.s2,
                              L.E, L.H, L.I)


def parity(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    """Assert the layer-output parity criterion; returns (max d/tol, relL2)."""
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    d = np.abs(gpu - ref)
    tol = ATOL + RTOL * np.abs(ref)
    ratio = float(np.max(d / tol)) if d.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(gpu - ref) / denom) if denom > 0 else float(np.linalg.norm(gpu))
    bad = int(np.sum(d > tol))
    assert bad == 0, f"{what}: {bad} elements out of tolerance, max d/tol {ratio:.3f}"
    assert rel <= REL_L2, f"{what}: relative L2 {rel:.3e} > {REL_L2}"
    return ratio, rel


def sample_rows(M: int, count: int, seed: int = 1) -> np.ndarray:
    """A sorted sample of token rows that always includes the first and last."""
    if M <= count:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, M - 1), size=count - 2, replace=False)
    return np.sort(np.concatenate([[0, M - 1], mid]))


# ---------------------------------------------------------------------------
# Stage-level checks: the sorted intermediates a finished forward leaves in its
# workspace (act = silu(gate)*up as an fp16 hi + lo pair, y the down
# projection, both per expert-sorted row) against the oracle's, slot by slot.
# ---------------------------------------------------------------------------
# |gpu - oracle| <= STAGE_ATOL + STAGE_RTOL * |oracle| for act and y.  Each
# slot's y enters the output multiplied by its routing weight (the k weights
# sum to 1), so a y within half the layer's absolute tolerance keeps its
# share of the output error inside the layer's bound; the relative part is
# ten times tighter than the layer's.  Measured: the largest absolute y error
# over the whole suite is 1.1e-3 (E=384, Zipf M = 4096, at y ~ 0.01: the
# tensor core's fp32 accumulation over 2 x 2048 K steps of products up to
# ~40, plus the fast exp/divide of SiLU inside act); a wrong row, chunk,
# scale or slot gives errors of order |y| ~ 25.
STAGE_ATOL = 5e-3
STAGE_RTOL = 1e-3


def workspace_rows(ws_buf, M, k, E, H, I, rows):
    """Copies from a finished forward's workspace: the alignment arrays
    (counts, offsets, perm, inv_perm, whole) and the sorted rows ``rows`` of
    act_hi, act_lo and y, as float64 numpy arrays (rows picked on the device,
    so a large batch's intermediates are never copied whole)."""
    import quantized_moe_expert_align_gb300 as moe
    torch = torch_mod()
    v = moe.moe_w4a16_workspace_views(M, k, E, H, I)
    n = M * k
    torch.cuda.synchronize()

    def whole(off, count, dtype):
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return ws_buf[off:off + nbytes].view(dtype)

    idx = torch.from_numpy(np.ascontiguousarray(rows, dtype=np.int64)).to(ws_buf.device)

    def pick(off, cols, dtype):
        t = whole(off, n * cols, dtype).view(n, cols)
        return t.index_select(0, idx).cpu().numpy().astype(np.float64)

    return {"counts": whole(v["counts"], E, torch.int32).cpu().numpy(),
            "offsets": whole(v["offsets"], E + 1, torch.int32).cpu().numpy(),
            "perm": whole(v["perm"], n, torch.int32).cpu().numpy(),
            "inv_perm": whole(v["inv_perm"], n, torch.int32).cpu().numpy(),
            "act_hi": pick(v["act_hi"], I, torch.float16),
            "act_lo": pick(v["act_lo"], I, torch.float16),
            "y": pick(v["y"], H, torch.float32)}


def oracle_on_slots(dl, x, ids, w, slots):
    """The oracle's forward restricted to the flat slots ``slots`` (t*k + j):
    it runs on the tokens that own them, with every other slot's id set to
    -1 (such a slot is left out of the alignment and of every stage), so it
    computes act and y of exactly those slots.  Returns (slots sorted,
    oracle dict, the oracle's sorted row of each slot)."""
    import oracle
    L = dl.layer
    k = L.k
    slots = np.unique(np.asarray(slots, np.int64))
    toks, tpos = np.unique(slots // k, return_inverse=True)
    keep = np.zeros((len(toks), k), bool)
    keep[tpos, slots % k] = True
    ids_m = np.where(keep, ids[toks], -1).astype(np.int32)
    ref = oracle.forward(x[toks], ids_m, w[toks], dl.w13, dl.s13, dl.w2, dl.s2,
                         L.E, L.H, L.I, want_intermediates=True)
    ref_pos = ref["inv_perm"].reshape(len(toks), k)[tpos, slots % k]
    assert np.all(ref_pos >= 0)
    return slots, ref, ref_pos, toks


def check_stages(dl, x, ids, w, ws_buf, slots, what=""):
    """Alignment bit-exact against the oracle's (whole batch), then act and y
    of every slot in ``slots`` element by element.  Returns the oracle dict
    of the restricted run (its ``out`` holds the tokens that own the slots,
    complete only for tokens whose every slot is in ``slots``)."""
    import oracle
    L = dl.layer
    M, k = ids.shape
    rc, ro, rp, rip, _ = oracle.align(ids, L.E)
    slots, ref, ref_pos, toks = oracle_on_slots(dl, x, ids, w, slots)
    gpu_pos = rip[slots]
    g = workspace_rows(ws_buf, M, k, L.E, L.H, L.I, gpu_pos)
    assert np.array_equal(g["counts"], rc), f"{what}: counts"
    assert np.array_equal(g["offsets"], ro), f"{what}: offsets"
    n = int(ro[L.E])
    assert np.array_equal(g["perm"][:n], rp[:n]), f"{what}: perm"
    assert np.array_equal(g["inv_perm"], rip), f"{what}: inv_perm"
    for name, got, exp in [("act", g["act_hi"] + g["act_lo"], ref["act"][ref_pos]),
                           ("y", g["y"], ref["y"][ref_pos])]:
        assert np.all(np.isfinite(got)), f"{what}: non-finite {name}"
        d = np.abs(got - exp)
        tol = STAGE_ATOL + STAGE_RTOL * np.abs(exp)
        bad = d > tol
        if np.any(bad):
            r, c = np.argwhere(bad)[0]
            raise AssertionError(
                f"{what}: {name}: {int(bad.sum())} elements out of tolerance in "
                f"{int(bad.any(axis=1).sum())} of {len(slots)} slots; first at slot "
                f"{int(slots[r])} (sorted row {int(gpu_pos[r])}), column {int(c)}: "
                f"{got[r, c]!r} vs {exp[r, c]!r}; max d/tol {float(np.max(d / tol)):.3f}")
    return ref, toks


def tile_sample(ids, E, nt, nt2, heavy_full=1, heavy_edges=4):
    """Slots chosen from the token-tile structure of both GEMMs: the first and
    last sorted row of every token tile (tiles of ``nt`` rows for the gate+up
    GEMM and ``nt2`` for the down GEMM, per expert segment), every row of the
    ``heavy_full`` heaviest experts, and every row of the first and last
    token tile of the ``heavy_edges`` heaviest experts (the last being the
    partial one).  Returns flat slot indices."""
    import oracle
    counts, offsets, perm, _, _ = oracle.align(ids, E)
    rows = set()
    for e in np.nonzero(counts)[0]:
        c, o = int(counts[e]), int(offsets[e])
        for width in (nt, nt2):
            for s in range(0, c, width):
                rows.add(o + s)
                rows.add(o + min(s + width, c) - 1)
    order = np.argsort(-counts, kind="stable")
    for e in order[:heavy_full]:
        rows.update(range(int(offsets[e]), int(offsets[e + 1])))
    for e in order[:heavy_edges]:
        c, o = int(counts[e]), int(offsets[e])
        last = (c - 1) // nt * nt
        rows.update(range(o, o + min(nt, c)))
        rows.update(range(o + last, o + c))
    return perm[np.array(sorted(rows), np.int64)]
