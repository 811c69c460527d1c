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
