"""Python binding of ``libmoe_w4a16.so`` -- the GB300 W4A16 MoE layer forward.

Argument marshalling only: every function below forwards to the C entry
point of the same name in ``include/moe_w4a16.h``; all work runs in the CUDA
kernels of that library.  PyTorch supplies device memory and streams.  If
the compiled library is missing, loading raises -- there is no fallback.

Helpers at the bottom (``prepack``, ``align``, ``forward``) allocate outputs
and workspaces with torch and raise ``MoeError`` on a non-OK status.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LIB_PATH = _build.LIB_PATH

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_MISALIGNED = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_BAD_LAYOUT = 4
MOE_ERR_UNSUPPORTED_DEVICE = 5
MOE_ERR_CUDA = 6
MOE_ERR_DEVICE_BAD_EXPERT_ID = 7
MOE_ERR_DEVICE_TIMEOUT = 8
MOE_ERR_DEVICE_FP16_RANGE = 9
MOE_ERR_DEVICE_BAD_LOGIT = 10
MOE_PACK_W13 = 1
MOE_PACK_W2 = 2


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")
        self.status = status


class moe_ws_views_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("counts", "offsets", "perm", "inv_perm", "act_hi", "act_lo", "y")]


class moe_diag_t(ctypes.Structure):
    _fields_ = [("version", ctypes.c_int32), ("M", ctypes.c_int32), ("k", ctypes.c_int32),
                ("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("token_tile", ctypes.c_int32), ("grid_gemm1", ctypes.c_int32),
                ("grid_gemm2", ctypes.c_int32), ("kernels_launched", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("calls", ctypes.c_int64),
                ("token_tile2", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load the compiled library (raises OSError/RuntimeError if absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run quantized_moe_expert_align_gb300.build.build()")
        lib = ctypes.CDLL(path)
        i, p, sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        sig = {
            "moe_status_string": (ctypes.c_char_p, [i]),
            "moe_w4a16_prepack_size": (i, [i, i, i, i, i, ctypes.POINTER(sz)]),
            "moe_w4a16_prepack": (i, [i, p, p, i, i, i, i, p, sz, p]),
            "moe_align_workspace_size": (sz, [i, i, i]),
            "moe_align": (i, [p, i, i, i, p, p, p, p, p, sz, p]),
            "moe_route_align": (i, [p, i, i, i, p, p, p, p, p, p, p, sz, p]),
            "moe_w4a16_workspace_size": (sz, [i, i, i, i, i]),
            "moe_w4a16_forward_routed": (i, [p, p, p, p, p, p, p, i, i, i, i, i, p, sz, p]),
            "moe_w4a16_forward": (i, [p, p, p, p, p, p, i, i, i, i, i, p, sz, p]),
            "moe_w4a16_forward_profiled": (i, [p, p, p, p, p, p, i, i, i, i, i, p, sz, p,
                                               ctypes.POINTER(p), i]),
            "moe_w4a16_forward_static": (i, [p, p, p, p, p, p, i, i, i, i, i, p]),
            "moe_w4a16_get_device_status": (i, [p, p, ctypes.POINTER(ctypes.c_int32)]),
            "moe_w4a16_get_diag": (i, [ctypes.POINTER(moe_diag_t)]),
            "moe_w4a16_workspace_views": (i, [i, i, i, i, i, ctypes.POINTER(moe_ws_views_t)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(t):
    """Device (or host) address of a tensor, or None."""
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# ---------------------------------------------------------------------------
# 1:1 wrappers of the C entry points (tensors -> pointers, return the status)
# ---------------------------------------------------------------------------
def moe_status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def moe_w4a16_prepack_size(kind, E, N, K, group=32):
    b = ctypes.c_size_t(0)
    st = load().moe_w4a16_prepack_size(kind, E, N, K, group, ctypes.byref(b))
    return st, b.value


def moe_w4a16_prepack(kind, q_canon, scales, E, N, K, group, dst, stream=None):
    return load().moe_w4a16_prepack(kind, _p(q_canon), _p(scales), E, N, K, group,
                                    _p(dst), dst.numel() * dst.element_size(), _stream(stream))


def moe_align_workspace_size(M, k, E):
    return load().moe_align_workspace_size(M, k, E)


def moe_align(topk_ids, M, k, E, counts, offsets, perm, inv_perm, workspace, stream=None):
    return load().moe_align(_p(topk_ids), M, k, E, _p(counts), _p(offsets), _p(perm),
                            _p(inv_perm), _p(workspace), workspace.numel() * workspace.element_size(),
                            _stream(stream))


def moe_route_align(logits, M, k, E, topk_ids, topk_w, counts, offsets, perm, inv_perm,
                    workspace, stream=None):
    return load().moe_route_align(_p(logits), M, k, E, _p(topk_ids), _p(topk_w), _p(counts),
                                  _p(offsets), _p(perm), _p(inv_perm), _p(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))


def moe_w4a16_workspace_size(M, k, E, H, I):
    return load().moe_w4a16_workspace_size(M, k, E, H, I)


def moe_w4a16_forward_routed(hidden, logits, w13, w2, out, topk_ids, topk_w, M, k, E, H, I,
                             workspace, stream=None):
    return load().moe_w4a16_forward_routed(
        _p(hidden), _p(logits), _p(w13), _p(w2), _p(out), _p(topk_ids), _p(topk_w), M, k, E, H,
        I, _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream))


def moe_w4a16_forward(hidden, topk_ids, topk_w, w13, w2, out, M, k, E, H, I, workspace,
                      stream=None):
    return load().moe_w4a16_forward(_p(hidden), _p(topk_ids), _p(topk_w), _p(w13), _p(w2),
                                    _p(out), M, k, E, H, I, _p(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))


def moe_w4a16_forward_profiled(hidden, topk_ids, topk_w, w13, w2, out, M, k, E, H, I,
                               workspace, events, stream=None):
    """``events``: six torch.cuda.Event(enable_timing=True) objects."""
    for e in events:
        if not e.cuda_event:   # torch creates the event lazily on first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return load().moe_w4a16_forward_profiled(
        _p(hidden), _p(topk_ids), _p(topk_w), _p(w13), _p(w2), _p(out), M, k, E, H, I,
        _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream), arr,
        len(events))


def moe_w4a16_forward_static(hidden, topk_ids, topk_w, w13, w2, out, M, k, E, H, I,
                             stream=None):
    """The forward on the library's static device scratch (no workspace)."""
    return load().moe_w4a16_forward_static(_p(hidden), _p(topk_ids), _p(topk_w), _p(w13), _p(w2),
                                           _p(out), M, k, E, H, I, _stream(stream))


MOE_W4A16_STATIC_SCRATCH_BYTES = 16 << 20


def moe_w4a16_get_device_status(workspace, stream=None):
    d = ctypes.c_int32(0)
    st = load().moe_w4a16_get_device_status(_p(workspace), _stream(stream), ctypes.byref(d))
    return st, d.value


def moe_w4a16_workspace_views(M, k, E, H, I):
    v = moe_ws_views_t()
    st = load().moe_w4a16_workspace_views(M, k, E, H, I, ctypes.byref(v))
    if st != MOE_OK:
        raise MoeError(st, "moe_w4a16_workspace_views")
    return {name: getattr(v, name) for name, _ in moe_ws_views_t._fields_}


def moe_w4a16_get_diag():
    d = moe_diag_t()
    st = load().moe_w4a16_get_diag(ctypes.byref(d))
    if st != MOE_OK:
        raise MoeError(st, "moe_w4a16_get_diag")
    return {name: getattr(d, name) for name, _ in moe_diag_t._fields_}


# ---------------------------------------------------------------------------
# torch conveniences (allocation with torch, then the C entry points)
# ---------------------------------------------------------------------------
def _check(st, where):
    if st != MOE_OK:
        raise MoeError(st, where)


def _empty_bytes(nbytes, device):
    import torch
    # torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def prepack(kind, q_canon, scales, stream=None):
    """Prepack canonical codes [E][N][K/2] (uint8) and bf16 scales
    [E][N][K/group] (int16/uint16/bfloat16 bits; group 32, 64 or 128, taken
    from the shapes) that live on the GPU; returns the packed uint8 buffer."""
    import torch
    E, N, half = q_canon.shape
    K = half * 2
    group = K // scales.shape[2]
    st, nb = moe_w4a16_prepack_size(kind, E, N, K, group)
    _check(st, "moe_w4a16_prepack_size")
    packed = _empty_bytes(nb, q_canon.device)
    if scales.dtype == torch.bfloat16:
        scales = scales.view(torch.int16)
    _check(moe_w4a16_prepack(kind, q_canon.contiguous(), scales.contiguous(), E, N, K, group,
                             packed, stream), "moe_w4a16_prepack")
    return packed


def align(topk_ids, E, stream=None):
    """Returns (counts, offsets, perm, inv_perm, workspace) on topk_ids' device."""
    import torch
    M, k = topk_ids.shape
    dev = topk_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(M * k, 1), dtype=torch.int32, device=dev)
    inv_perm = torch.empty(max(M * k, 1), dtype=torch.int32, device=dev)
    ws = _empty_bytes(moe_align_workspace_size(M, k, E), dev)
    _check(moe_align(topk_ids.contiguous(), M, k, E, counts, offsets, perm, inv_perm, ws, stream),
           "moe_align")
    return counts, offsets, perm[:M * k], inv_perm[:M * k], ws


def route_align(logits, k, stream=None):
    """Router front-end + alignment from fp32 logits [M][E].  Returns
    (topk_ids, topk_w, counts, offsets, perm, inv_perm, workspace)."""
    import torch
    M, E = logits.shape
    dev = logits.device
    ids = torch.empty((M, k), dtype=torch.int32, device=dev)
    w = torch.empty((M, k), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(M * k, 1), dtype=torch.int32, device=dev)
    inv_perm = torch.empty(max(M * k, 1), dtype=torch.int32, device=dev)
    ws = _empty_bytes(moe_align_workspace_size(M, k, E), dev)
    _check(moe_route_align(logits.contiguous(), M, k, E, ids, w, counts, offsets, perm, inv_perm,
                           ws, stream), "moe_route_align")
    return ids, w, counts, offsets, perm[:M * k], inv_perm[:M * k], ws


class Workspace:
    """A reusable forward workspace sized for up to ``max_M`` tokens."""

    def __init__(self, max_M, k, E, H, I, device):
        self.nbytes = moe_w4a16_workspace_size(max_M, k, E, H, I)
        if self.nbytes == 0:
            raise MoeError(MOE_ERR_INVALID_ARG, "moe_w4a16_workspace_size")
        self.buf = _empty_bytes(self.nbytes, device)


def forward(hidden, topk_ids, topk_w, w13, w2, E, I, out=None, workspace=None, stream=None):
    """out[M][H] bf16 = MoE layer forward; raises MoeError on a host-side error."""
    import torch
    M, H = hidden.shape
    k = topk_ids.shape[1]
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=hidden.device)
    ws = workspace.buf if isinstance(workspace, Workspace) else workspace
    if ws is None:
        ws = Workspace(M, k, E, H, I, hidden.device).buf
    _check(moe_w4a16_forward(hidden, topk_ids, topk_w, w13, w2, out, M, k, E, H, I, ws, stream),
           "moe_w4a16_forward")
    return out


def forward_routed(hidden, logits, k, w13, w2, E, I, out=None, workspace=None, stream=None):
    """The layer from router logits [M][E] fp32: returns (out [M][H] bf16,
    topk_ids [M][k], topk_w [M][k]); raises MoeError on a host-side error."""
    import torch
    M, H = hidden.shape
    dev = hidden.device
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    ids = torch.empty((M, k), dtype=torch.int32, device=dev)
    w = torch.empty((M, k), dtype=torch.float32, device=dev)
    ws = workspace.buf if isinstance(workspace, Workspace) else workspace
    if ws is None:
        ws = Workspace(M, k, E, H, I, dev).buf
    _check(moe_w4a16_forward_routed(hidden, logits.contiguous(), w13, w2, out, ids, w, M, k, E,
                                    H, I, ws, stream), "moe_w4a16_forward_routed")
    return out, ids, w
