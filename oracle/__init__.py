"""CPU oracle of the W4A16 MoE layer forward -- TEST INFRASTRUCTURE ONLY.

This package wraps ``moe_oracle.c`` (plain C, IEEE double, OpenMP over
independent output rows) with numpy-facing helpers.  Only the test-suite, the
smoke check and the benchmark's CPU-baseline leg may import it; the CUDA
library and its Python binding never do.  It shares no code with them.

What it computes, and the readings behind it, is documented at the top of
``moe_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoe_oracle.so")
_lock = threading.Lock()
_default = None

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
          "-fno-fast-math", "-ffp-contract=off"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle source file into a shared library with gcc."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` unless an up-to-date build exists."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


class Oracle:
    """numpy front end of one compiled oracle library."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_dequant_element.restype = ctypes.c_double
        lib.oracle_dequant_element.argtypes = [p, p, i64, i64, i64, i64]
        lib.oracle_align.restype = i64
        lib.oracle_align.argtypes = [p, i64, i64, i64, p, p, p, p]
        lib.oracle_route.restype = i64
        lib.oracle_route.argtypes = [p, i64, i64, i64, p, p]
        lib.oracle_forward.restype = i64
        lib.oracle_forward.argtypes = [p, p, p, p, p, p, p,
                                       i64, i64, i64, i64, i64, i64,
                                       p, p, p, p, p, p, p, p, i64]
        self.lib = lib
        self.path = so_path

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def dequant_element(self, q, s, n: int, kk: int) -> float:
        """Dequantised element (n, kk) of one packed [N][K/2] matrix with
        [N][K/group] scales (the group size follows from the shapes)."""
        q = np.ascontiguousarray(q, dtype=np.uint8)
        s = np.ascontiguousarray(s, dtype=np.uint16)
        K = q.shape[1] * 2
        group = K // s.shape[1]
        assert group * s.shape[1] == K
        return float(self.lib.oracle_dequant_element(_ptr(q), _ptr(s), K, group, n, kk))

    def align(self, ids, E: int):
        """Stable counting sort of the flat slot indices by expert.

        Returns (counts[E], offsets[E+1], perm[M*k], inv_perm[M*k], n_invalid);
        only the first offsets[E] entries of ``perm`` are defined (rest -1).
        """
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        M, k = ids.shape
        counts = np.zeros(E, np.int32)
        offsets = np.zeros(E + 1, np.int32)
        perm = np.full(max(M * k, 1), -1, np.int32)
        inv_perm = np.full(max(M * k, 1), -1, np.int32)
        bad = self.lib.oracle_align(_ptr(ids), M, k, E, _ptr(counts), _ptr(offsets),
                                    _ptr(perm), _ptr(inv_perm))
        n = M * k
        return counts, offsets, perm[:n], inv_perm[:n], int(bad)

    def route(self, logits, k: int):
        """Softmax top-k router with renormalised weights.

        ``logits`` [M][E] fp32.  Returns (ids [M][k] int32, topk_w [M][k]
        fp32, bad_rows); a bad row (NaN or +inf logit) has zero weights.
        """
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        M, E = logits.shape
        assert 1 <= k <= E
        ids = np.full((M, k), -1, np.int32)
        w = np.zeros((M, k), np.float32)
        bad = self.lib.oracle_route(_ptr(logits), M, E, k, _ptr(ids), _ptr(w))
        return ids, w, int(bad)

    def forward(self, hidden, ids, topk_w, w13, s13, w2, s2, E: int, H: int, I: int,
                want_intermediates: bool = False):
        """Layer forward in double.  ``hidden`` and the scales are bf16 bit
        patterns (uint16); packed weights are canonical [E][N][K/2] bytes.

        The scale group size (32 on the pages; 64 and 128 also work) follows
        from the scale shapes [E][N][K/group].

        Returns ``out`` [M][H] float64, or with ``want_intermediates`` a dict
        with ``out``, ``act`` ([n_valid][I], sorted order), ``y``
        ([n_valid][H], sorted order) and the alignment, n_valid being the
        number of slots whose id lies in [0, E) (the rows the alignment
        places; slots with other ids are left out of every stage).
        """
        hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        topk_w = np.ascontiguousarray(topk_w, dtype=np.float32)
        M, k = ids.shape
        assert hidden.shape == (M, H) and topk_w.shape == (M, k)
        group = H // s13.shape[2]
        assert group * s13.shape[2] == H and I % group == 0
        assert w13.shape == (E, 2 * I, H // 2) and s13.shape == (E, 2 * I, H // group)
        assert w2.shape == (E, H, I // 2) and s2.shape == (E, H, I // group)
        assert w13.dtype == np.uint8 and w2.dtype == np.uint8
        assert s13.dtype == np.uint16 and s2.dtype == np.uint16
        n = M * k
        # only the placed slots get sorted rows: size y and act by them
        n_valid = int(np.count_nonzero((ids >= 0) & (ids < E)))
        out = np.zeros((M, H), np.float64)
        y = np.zeros((max(n_valid, 1), H), np.float64)
        act = np.zeros((max(n_valid, 1), I), np.float64) if want_intermediates else None
        nt = self.num_threads()
        scratch = np.zeros(nt * I, np.float64)
        counts = np.zeros(E, np.int32)
        offsets = np.zeros(E + 1, np.int32)
        perm = np.full(max(n, 1), -1, np.int32)
        inv_perm = np.full(max(n, 1), -1, np.int32)
        bad = self.lib.oracle_forward(
            _ptr(hidden), _ptr(ids), _ptr(topk_w), _ptr(w13), _ptr(s13), _ptr(w2),
            _ptr(s2), M, k, E, H, I, group, _ptr(out), _ptr(act), _ptr(y), _ptr(counts),
            _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(scratch), nt * I)
        if bad < 0:
            raise RuntimeError("oracle_forward: scratch too small")
        if not want_intermediates:
            return out
        return {"out": out, "act": act[:n_valid], "y": y[:n_valid], "counts": counts,
                "offsets": offsets, "perm": perm[:n], "inv_perm": inv_perm[:n],
                "n_invalid": int(bad)}


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def num_threads() -> int:
    return default().num_threads()


def dequant_element(q, s, n, kk):
    return default().dequant_element(q, s, n, kk)


def align(ids, E):
    return default().align(ids, E)


def route(logits, k):
    return default().route(logits, k)


def forward(*args, **kwargs):
    return default().forward(*args, **kwargs)
