"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself.

Each ``check_*`` function takes an ``oracle.Oracle`` and raises
AssertionError on a mismatch.  ``test_oracle_pins.py`` runs them against the
real oracle; ``test_oracle_mutants.py`` runs them against copies of the
oracle with planted mistakes and requires every mistake to be caught.

What each pin rests on:
  * worked bytes  -- the packed-code convention and the dequantisation rule
    (value = (q - 8) * scale, group of 32 along K; 64 and 128 for the
    wider-group variant), evaluated by hand;
  * stable sort   -- the alignment is a stable counting sort, so it must equal
    numpy's stable argsort and bincount/cumsum;
  * closed form   -- weights whose codes are constant along K make every
    projection a multiple of sum(x); the layer output then has a closed form;
  * brute force   -- an independent dense per-token path (no alignment, no
    grouping, numpy matmul) on tiny random layers;
  * special cases -- all-zero codes give exactly zero, k = 1 with weight 1 is a
    single-expert MLP, outputs are linear in topk_w and equivariant under
    token permutation, unused experts are never read;
  * router        -- the selection equals a Python sort by (-logit, index) on
    tie-heavy inputs; the weights equal a full numpy softmax renormalised
    over the selection, and closed forms (equal logits give 1/k; logits
    -e ln 2 give 2^-j / (2 - 2^(1-k))); NaN / +inf / -inf rows follow the
    stated rules.
"""
from __future__ import annotations

import math

import numpy as np

import synth

BF16_ONE_QUARTER = 0x3E80   # 0.25
BF16_THREE = 0x4040         # 3.0
BF16_NAN = 0x7FC0


# ----------------------------------------------------------------------------
# independent helpers (numpy; no code shared with the oracle)
# ----------------------------------------------------------------------------
def _bf16(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def dense_weight(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Unpack one canonical [N][K/2] code matrix with [N][K/group] scales into
    a dense fp64 [N][K]."""
    N, half = q.shape
    codes = np.empty((N, 2 * half), np.int64)
    codes[:, 0::2] = q & 0x0F
    codes[:, 1::2] = q >> 4
    group = 2 * half // s.shape[1]
    return (codes - 8).astype(np.float64) * np.repeat(_bf16(s), group, axis=1)


def brute_force(hidden, ids, topk_w, w13, s13, w2, s2, E, H, I):
    """Dense per-token reference: no sort, no grouping."""
    x = _bf16(hidden)
    M, k = ids.shape
    out = np.zeros((M, H), np.float64)
    cache = {}
    for t in range(M):
        for j in range(k):
            e = int(ids[t, j])
            if not 0 <= e < E:
                continue
            if e not in cache:
                cache[e] = (dense_weight(w13[e], s13[e]), dense_weight(w2[e], s2[e]))
            W13, W2 = cache[e]
            h = W13 @ x[t]
            g, u = h[:I], h[I:]
            a = g / (1.0 + np.exp(-g)) * u
            out[t] += float(topk_w[t, j]) * (W2 @ a)
    return out


def _random_layer(rng, E, H, I, group=32):
    w13 = rng.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8)
    w2 = rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    s13 = synth.f32_to_bf16_bits(
        rng.uniform(0.002, 0.02, (E, 2 * I, H // group)).astype(np.float32))
    s2 = synth.f32_to_bf16_bits(rng.uniform(0.002, 0.02, (E, H, I // group)).astype(np.float32))
    return w13, s13, w2, s2


def _random_inputs(rng, M, E, H, k):
    hidden = synth.f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    w = rng.random((M, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    return hidden, ids, w.astype(np.float32)


def _close(a, b, rtol=1e-10):
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= rtol * scale, f"max abs diff {err:.3e} > {rtol * scale:.3e}"


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------
def check_dequant_worked_bytes(orc):
    """Hand-evaluated codes: row 0 uses scale 0.25 for group 0 and 3.0 for
    group 1; row 1 swaps them.  Byte b holds element 2b in its low nibble."""
    K = 64
    q = np.full((2, K // 2), 0x88, np.uint8)             # every code 8 -> 0.0
    q[0, 0], q[0, 1], q[0, 2], q[0, 3] = 0x9A, 0x0F, 0x80, 0x7F
    q[0, 16] = 0x1C
    q[1, 0] = 0x9A
    s = np.array([[BF16_ONE_QUARTER, BF16_THREE], [BF16_THREE, BF16_ONE_QUARTER]], np.uint16)
    expect = {
        (0, 0): (10 - 8) * 0.25, (0, 1): (9 - 8) * 0.25,
        (0, 2): (15 - 8) * 0.25, (0, 3): (0 - 8) * 0.25,
        (0, 4): (0 - 8) * 0.25, (0, 5): (8 - 8) * 0.25,
        (0, 6): (15 - 8) * 0.25, (0, 7): (7 - 8) * 0.25,
        (0, 32): (12 - 8) * 3.0, (0, 33): (1 - 8) * 3.0,
        (0, 31): 0.0, (0, 63): 0.0,
        (1, 0): (10 - 8) * 3.0, (1, 1): (9 - 8) * 3.0, (1, 32): 0.0,
    }
    for (n, kk), v in expect.items():
        got = orc.dequant_element(q, s, n, kk)
        assert got == v, f"W[{n}][{kk}] = {got}, expected {v}"


def check_align_matches_stable_sort(orc):
    rng = np.random.default_rng(11)
    for (M, k, E) in [(1, 1, 1), (1, 8, 384), (9, 8, 384), (37, 3, 5), (200, 4, 16),
                      (64, 2, 8), (5, 6, 3)]:
        ids = rng.integers(0, E, size=(M, k)).astype(np.int32)   # duplicates allowed
        counts, offsets, perm, inv_perm, bad = orc.align(ids, E)
        flat = ids.ravel()
        ref_perm = np.argsort(flat, kind="stable").astype(np.int32)
        ref_counts = np.bincount(flat, minlength=E).astype(np.int32)
        assert bad == 0
        assert np.array_equal(counts, ref_counts)
        assert offsets[0] == 0 and np.array_equal(offsets[1:], np.cumsum(ref_counts))
        assert np.array_equal(perm, ref_perm)
        ref_inv = np.empty_like(ref_perm)
        ref_inv[ref_perm] = np.arange(M * k, dtype=np.int32)
        assert np.array_equal(inv_perm, ref_inv)


def check_align_invalid_ids(orc):
    E = 4
    ids = np.array([[0, 4], [-1, 2], [2, 0], [3, 1 << 30]], np.int32)
    counts, offsets, perm, inv_perm, bad = orc.align(ids, E)
    assert bad == 3
    assert counts.tolist() == [2, 0, 2, 1] and offsets.tolist() == [0, 2, 2, 4, 5]
    assert perm.tolist()[:5] == [0, 5, 3, 4, 6]
    assert inv_perm.tolist() == [0, -1, -1, 2, 3, 1, 4, -1]


def check_forward_closed_form(orc):
    """Codes constant along K, one scale per matrix: gate row n has code
    8 + cg[n] and scale sg, up row n has 8 + cu[n] and su, w2 row h has code
    8 + d[h][n] (constant inside each group of 32 along n... here I = 32) and
    scale s2.  With S = sum(x): g = cg*sg*S, u = cu*su*S, a = silu(g)*u,
    y[h] = s2 * sum_n d[h][n]*a[n], out = sum_j w_j * y_j."""
    E, H, I, M, k = 2, 64, 32, 3, 2
    rng = np.random.default_rng(5)
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    s13 = np.zeros((E, 2 * I, H // 32), np.uint16)
    w2 = np.zeros((E, H, I // 2), np.uint8)
    s2 = np.zeros((E, H, I // 32), np.uint16)
    cg = rng.integers(-8, 8, size=(E, I))
    cu = rng.integers(-8, 8, size=(E, I))
    d = rng.integers(-8, 8, size=(E, H, I))
    sg, su, sd = 0.03125, 0.0625, 0.125                  # exact in bf16
    sg_b, su_b, sd_b = 0x3D00, 0x3D80, 0x3E00
    for e in range(E):
        for n in range(I):
            c = int(cg[e, n]) + 8
            w13[e, n, :] = c | (c << 4)
            c = int(cu[e, n]) + 8
            w13[e, I + n, :] = c | (c << 4)
        s13[e, :I, :] = sg_b
        s13[e, I:, :] = su_b
        for h in range(H):
            codes = d[e, h] + 8
            w2[e, h, :] = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
        s2[e, :, :] = sd_b
    x = synth.f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    ids = np.array([[0, 1], [1, 0], [1, 1]], np.int32)
    w = np.array([[0.75, 0.25], [0.5, 0.5], [0.125, 0.875]], np.float32)
    out = orc.forward(x, ids, w, w13, s13, w2, s2, E, H, I)
    xs = synth.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(M):
        S = math.fsum(xs[t])
        ref = np.zeros(H)
        for j in range(k):
            e = ids[t, j]
            a = np.array([(cg[e, n] * sg * S) / (1.0 + math.exp(-cg[e, n] * sg * S))
                          * (cu[e, n] * su * S) for n in range(I)])
            y = sd * (d[e].astype(np.float64) @ a)
            ref += float(w[t, j]) * y
        _close(out[t], ref, 1e-9)


def check_dequant_wide_groups(orc):
    """Hand-evaluated scale indexing for groups of 64 and 128: element kk
    takes scale kk // group."""
    K = 256
    q = np.full((1, K // 2), 0x88, np.uint8)
    q[0, 31] = 0xA8      # element 63 -> code 10, element 62 -> 8
    q[0, 32] = 0x89      # element 64 -> code 9
    q[0, 63] = 0xB8      # element 127 -> code 11
    q[0, 64] = 0x8F      # element 128 -> code 15
    q[0, 127] = 0x08     # element 255 -> code 0
    s64 = np.array([[BF16_ONE_QUARTER, BF16_THREE, BF16_ONE_QUARTER, BF16_THREE]], np.uint16)
    expect64 = {63: 2 * 0.25, 64: 1 * 3.0, 127: 3 * 3.0, 128: 7 * 0.25, 255: -8 * 3.0, 62: 0.0}
    for kk, v in expect64.items():
        got = orc.dequant_element(q, s64, 0, kk)
        assert got == v, f"group 64, element {kk}: {got} != {v}"
    s128 = np.array([[BF16_THREE, BF16_ONE_QUARTER]], np.uint16)
    expect128 = {63: 2 * 3.0, 64: 1 * 3.0, 127: 3 * 3.0, 128: 7 * 0.25, 255: -8 * 0.25}
    for kk, v in expect128.items():
        got = orc.dequant_element(q, s128, 0, kk)
        assert got == v, f"group 128, element {kk}: {got} != {v}"


def check_forward_brute_force_wide_groups(orc):
    rng = np.random.default_rng(31)
    for group in (64, 128):
        for (M, E, H, I, k) in [(4, 6, 256, 128, 2), (3, 3, 128, 128, 3)]:
            w13, s13, w2, s2 = _random_layer(rng, E, H, I, group)
            hidden, ids, w = _random_inputs(rng, M, E, H, k)
            out = orc.forward(hidden, ids, w, w13, s13, w2, s2, E, H, I)
            _close(out, brute_force(hidden, ids, w, w13, s13, w2, s2, E, H, I))


def check_forward_brute_force(orc):
    rng = np.random.default_rng(7)
    for (M, E, H, I, k) in [(4, 8, 256, 128, 2), (3, 2, 64, 32, 2), (6, 5, 96, 64, 3),
                            (2, 4, 32, 32, 1)]:
        w13, s13, w2, s2 = _random_layer(rng, E, H, I)
        hidden, ids, w = _random_inputs(rng, M, E, H, k)
        out = orc.forward(hidden, ids, w, w13, s13, w2, s2, E, H, I)
        _close(out, brute_force(hidden, ids, w, w13, s13, w2, s2, E, H, I))
    # duplicates inside a row are independent slots
    E, H, I, M, k = 3, 64, 32, 2, 3
    w13, s13, w2, s2 = _random_layer(rng, E, H, I)
    hidden = synth.f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    ids = np.array([[1, 1, 2], [0, 0, 0]], np.int32)
    w = np.array([[0.5, 0.25, 0.25], [0.125, 0.5, 0.375]], np.float32)
    out = orc.forward(hidden, ids, w, w13, s13, w2, s2, E, H, I)
    _close(out, brute_force(hidden, ids, w, w13, s13, w2, s2, E, H, I))


def check_forward_zero_codes(orc):
    E, H, I, M, k = 4, 64, 32, 5, 2
    rng = np.random.default_rng(3)
    _, s13, _, s2 = _random_layer(rng, E, H, I)
    w13 = np.full((E, 2 * I, H // 2), 0x88, np.uint8)
    w2 = np.full((E, H, I // 2), 0x88, np.uint8)
    hidden, ids, w = _random_inputs(rng, M, E, H, k)
    out = orc.forward(hidden, ids, w, w13, s13, w2, s2, E, H, I)
    assert np.all(out == 0.0)
    # zero gate alone also zeroes the output (silu(0) = 0), whatever up holds
    w13 = rng.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8)
    w13[:, :I, :] = 0x88
    w2 = rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    out = orc.forward(hidden, ids, w, w13, s13, w2, s2, E, H, I)
    assert np.all(out == 0.0)


def check_forward_single_expert_mlp(orc):
    """k = 1 with weight 1 is one expert's MLP: W2 (silu(Wg x) * (Wu x))."""
    rng = np.random.default_rng(9)
    E, H, I, M = 3, 128, 64, 4
    w13, s13, w2, s2 = _random_layer(rng, E, H, I)
    hidden = synth.f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    ids = np.array([[2], [0], [2], [1]], np.int32)
    w = np.ones((M, 1), np.float32)
    out = orc.forward(hidden, ids, w, w13, s13, w2, s2, E, H, I)
    x = _bf16(hidden)
    for t in range(M):
        e = int(ids[t, 0])
        Wg = dense_weight(w13[e], s13[e])[:I]
        Wu = dense_weight(w13[e], s13[e])[I:]
        W2 = dense_weight(w2[e], s2[e])
        g = Wg @ x[t]
        ref = W2 @ (g / (1.0 + np.exp(-g)) * (Wu @ x[t]))
        _close(out[t], ref)


def check_forward_linearity_and_permutation(orc):
    rng = np.random.default_rng(13)
    E, H, I, M, k = 6, 64, 64, 7, 3
    w13, s13, w2, s2 = _random_layer(rng, E, H, I)
    hidden, ids, w = _random_inputs(rng, M, E, H, k)
    base = orc.forward(hidden, ids, w, w13, s13, w2, s2, E, H, I)
    doubled = orc.forward(hidden, ids, (2 * w).astype(np.float32), w13, s13, w2, s2, E, H, I)
    assert np.array_equal(doubled, 2 * base)
    # one slot's weight set to zero removes exactly that expert's term
    w0 = w.copy()
    w0[:, 1] = 0
    part = orc.forward(hidden, ids, w0, w13, s13, w2, s2, E, H, I)
    only = np.zeros_like(w)
    only[:, 1] = w[:, 1]
    rest = orc.forward(hidden, ids, only, w13, s13, w2, s2, E, H, I)
    _close(part + rest, base)
    pi = rng.permutation(M)
    perm_out = orc.forward(hidden[pi], ids[pi], w[pi], w13, s13, w2, s2, E, H, I)
    assert np.array_equal(perm_out, base[pi])


def check_unused_expert_not_read(orc):
    rng = np.random.default_rng(17)
    E, H, I, M, k = 5, 64, 32, 4, 2
    w13, s13, w2, s2 = _random_layer(rng, E, H, I)
    hidden = synth.f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    ids = np.array([[0, 1], [1, 3], [3, 0], [4, 1]], np.int32)   # expert 2 unused
    w = np.full((M, k), 0.5, np.float32)
    base = orc.forward(hidden, ids, w, w13, s13, w2, s2, E, H, I)
    s13p, s2p = s13.copy(), s2.copy()
    s13p[2] = BF16_NAN
    s2p[2] = BF16_NAN
    poisoned = orc.forward(hidden, ids, w, w13, s13p, w2, s2p, E, H, I)
    assert np.all(np.isfinite(poisoned)) and np.array_equal(poisoned, base)


def check_forward_invalid_slot_contributes_zero(orc):
    rng = np.random.default_rng(19)
    E, H, I, M, k = 4, 64, 32, 3, 2
    w13, s13, w2, s2 = _random_layer(rng, E, H, I)
    hidden = synth.f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    ids = np.array([[0, 7], [-3, 2], [1, 3]], np.int32)
    w = np.full((M, k), 0.5, np.float32)
    out = orc.forward(hidden, ids, w, w13, s13, w2, s2, E, H, I)
    _close(out, brute_force(hidden, ids, w, w13, s13, w2, s2, E, H, I))
    assert np.all(out[2] != 0.0)


def _py_topk(row, k):
    """Order by descending logit, lower index first on ties, NaN last."""
    def key(e):
        v = float(row[e])
        return (1, 0.0, e) if math.isnan(v) else (0, -v, e)
    return sorted(range(len(row)), key=key)[:k]


def check_route_selection_brute_force(orc):
    rng = np.random.default_rng(23)
    for trial in range(60):
        E = int(rng.integers(1, 41))
        k = int(rng.integers(1, E + 1))
        M = int(rng.integers(1, 6))
        # few distinct values, so ties are common; signed zeros compare equal
        vals = np.array([-1.5, -0.0, 0.0, 0.25, 1.0, 1.0], np.float32)
        lg = vals[rng.integers(0, len(vals), size=(M, E))]
        ids, _, bad = orc.route(lg, k)
        assert bad == 0
        for t in range(M):
            assert list(ids[t]) == _py_topk(lg[t], k), (trial, t)


def check_route_weights_full_softmax(orc):
    rng = np.random.default_rng(29)
    for E, k, M in [(8, 2, 5), (64, 8, 7), (384, 8, 4), (17, 17, 3), (128, 1, 3)]:
        lg = (rng.standard_normal((M, E)) * 3).astype(np.float32)
        ids, w, bad = orc.route(lg, k)
        assert bad == 0
        x = lg.astype(np.float64)
        p = np.exp(x - x.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        for t in range(M):
            assert list(ids[t]) == _py_topk(lg[t], k)
            sel = p[t, ids[t]]
            ref = sel / sel.sum()
            assert np.all(np.abs(w[t] - ref) <= 2.0 ** -23 * ref), (E, k, t)
            assert np.all(np.diff(w[t].astype(np.float64)) <= 0)


def check_route_closed_forms(orc):
    # equal logits: the first k experts, each 1/k
    for E, k in [(8, 2), (384, 8), (5, 5), (3, 1)]:
        ids, w, _ = orc.route(np.full((2, E), 0.75, np.float32), k)
        assert np.array_equal(ids, np.tile(np.arange(k, dtype=np.int32), (2, 1)))
        assert np.all(w == np.float32(1.0 / k))
    # logits -e ln 2: p_e proportional to 2^-e, so w_j = 2^-j / (2 - 2^(1-k))
    E = 40
    lg = (-np.arange(E) * math.log(2.0)).astype(np.float32)[None, :]
    for k in (1, 2, 8, 20):
        ids, w, _ = orc.route(lg, k)
        assert np.array_equal(ids[0], np.arange(k))
        ref = np.array([2.0 ** -j / (2.0 - 2.0 ** (1 - k)) for j in range(k)])
        assert np.all(np.abs(w[0] - ref) <= 1e-6 * ref), k
    # one dominant logit: weight 1 on it, 0 elsewhere (exp underflows)
    lg = np.zeros((1, 16), np.float32)
    lg[0, 11] = 1000.0
    ids, w, _ = orc.route(lg, 3)
    assert list(ids[0]) == [11, 0, 1] and list(w[0]) == [1.0, 0.0, 0.0]


def check_route_special_values(orc):
    inf, nan = np.inf, np.nan
    lg = np.array([[0.5, -inf, 2.0, -inf, 1.0],     # -inf: weight 0, ranked after numbers
                   [nan, 1.0, nan, 0.0, -inf],      # NaN: bad row, ranked last
                   [0.0, inf, 1.0, 2.0, 3.0],       # +inf: bad row, ranked first
                   [-inf, -inf, -inf, -inf, -inf]], # all -inf: zero weights, not bad
                  np.float32)
    ids, w, bad = orc.route(lg, 4)
    assert bad == 2
    assert list(ids[0]) == [2, 4, 0, 1] and w[0, 3] == 0.0 and w[0, 2] > 0
    assert abs(float(w[0].astype(np.float64).sum()) - 1.0) <= 4 * 2.0 ** -24
    assert list(ids[1]) == [1, 3, 4, 0] and np.all(w[1] == 0)
    assert list(ids[2]) == [1, 4, 3, 2] and np.all(w[2] == 0)
    assert list(ids[3]) == [0, 1, 2, 3] and np.all(w[3] == 0)


def check_route_matches_input_generator(orc):
    # synth.route draws the workloads' routing with numpy (stable argsort,
    # softmax over the selected logits): an independent implementation
    for M, E, k, zipf in [(64, 384, 8, None), (64, 384, 8, 1.1), (16, 8, 2, None)]:
        lg = synth.logits(M, E, seed=3, zipf_s=zipf)
        ids, w, bad = orc.route(lg, k)
        ids_ref, w_ref = synth.route(lg, k)
        assert bad == 0 and np.array_equal(ids, ids_ref)
        assert np.all(np.abs(w - w_ref) <= 2.0 ** -23 * w_ref)


ALL_PINS = [check_dequant_wide_groups, check_forward_brute_force_wide_groups,
            check_route_selection_brute_force, check_route_weights_full_softmax,
            check_route_closed_forms, check_route_special_values,
            check_route_matches_input_generator,
            check_dequant_worked_bytes, check_align_matches_stable_sort,
            check_align_invalid_ids, check_forward_closed_form,
            check_forward_brute_force, check_forward_zero_codes,
            check_forward_single_expert_mlp, check_forward_linearity_and_permutation,
            check_unused_expert_not_read, check_forward_invalid_slot_contributes_zero]
