"""Seeded synthetic inputs for the W4A16 MoE layer.

This module is shared by the tests, the benchmark and the oracle harness.  It
holds none of the layer's arithmetic: it only draws inputs (hidden states,
router logits and the routing derived from them, packed INT4 codes, bf16
scales) with the shapes and distributions of the workloads below, each from a
counter-keyed numpy stream so that any one expert's weights can be rebuilt on
its own.

Recipe (every tensor from ``np.random.Generator(PCG64(SeedSequence([seed,
tag, index])))``):
  hidden   [M][H]  N(0,1) rounded to bf16 (round-to-nearest-even)
  logits   [M][E]  N(0,1) fp32, plus ln p_e for a Zipf(s) prior p_e ~ (e+1)^-s
  routing  top-k by descending logit (lower expert index first on ties);
           weights = softmax over the k selected logits (the renormalised
           softmax top-k), computed in fp64 and stored as fp32
  w13/w2   canonical packed codes [E][N][K/2] uint8 taken from the raw 64-bit
           PCG64 output, so each nibble is uniform on {0..15}; element kk of a
           row sits in byte kk/2, low nibble when kk is even
  s13/s2   [E][N][K/32] bf16 uniform on [0.002, 0.02]

The workloads are those of the MoE GEMM sweep in "The MoE Throughput Lever:
Quantifying the INT4 Marlin GEMM on Blackwell PRO 6000" (section "The
Benchmark: What Was Measured": E=384, hidden 7168, intermediate 2048, top-8,
INT4 group 32, M = 1..1024), extended with skewed prefill batches and a
second, smaller layer shape, plus a toy layer for quick checks.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

TAG_HIDDEN, TAG_LOGITS, TAG_W13, TAG_S13, TAG_W2, TAG_S2 = 1, 2, 3, 4, 5, 6
SCALE_LO, SCALE_HI = 0.002, 0.02
GROUP = 32


@dataclass(frozen=True)
class Layer:
    E: int
    H: int
    I: int
    k: int
    group: int = GROUP   # elements of K per scale (32 on the pages; 64, 128 variants)


@dataclass(frozen=True)
class Workload:
    name: str
    layer: Layer
    Ms: Sequence[int]
    zipf_s: Optional[float] = None


TOY = Workload("toy_e8_h256_i128_top2", Layer(8, 256, 128, 2), (4,))
DECODE = Workload("decode_e384_h7168_i2048_top8", Layer(384, 7168, 2048, 8), (1, 9, 90))
PLATEAU = Workload("plateau_e384_h7168_i2048_top8", Layer(384, 7168, 2048, 8), (256, 512, 1024))
PREFILL = Workload("prefill_zipf1.1_e384_h7168_i2048_top8", Layer(384, 7168, 2048, 8),
                   (4096, 16384), zipf_s=1.1)
SECOND = Workload("second_e128_h4096_i1536_top8", Layer(128, 4096, 1536, 8), (1, 32, 256, 2048))
# Variants beyond the pages' layer: 256 experts of the same width, and scale
# groups of 128 elements on the second shape.
E256 = Workload("e256_h7168_i2048_top8", Layer(256, 7168, 2048, 8), (1, 9, 90))
GROUP128 = Workload("second_group128_e128_h4096_i1536_top8", Layer(128, 4096, 1536, 8, 128),
                    (1, 32, 256))
WORKLOADS = {w.name: w for w in (TOY, DECODE, PLATEAU, PREFILL, SECOND, E256, GROUP128)}


def _rng(seed: int, tag: int, index: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, index])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def hidden(M: int, H: int, seed: int = 0) -> np.ndarray:
    """bf16 bit patterns [M][H], N(0,1)."""
    x = _rng(seed, TAG_HIDDEN).standard_normal((M, H), dtype=np.float32)
    return f32_to_bf16_bits(x)


def logits(M: int, E: int, seed: int = 0, zipf_s: Optional[float] = None) -> np.ndarray:
    lg = _rng(seed, TAG_LOGITS).standard_normal((M, E), dtype=np.float32)
    if zipf_s is not None:
        p = np.arange(1, E + 1, dtype=np.float64) ** (-zipf_s)
        p /= p.sum()
        lg = (lg + np.log(p).astype(np.float32)).astype(np.float32)
    return lg


def route(lg: np.ndarray, k: int):
    """Top-k by descending logit, ties to the lower expert index; weights are
    the softmax over the selected logits (fp64 -> fp32)."""
    M, E = lg.shape
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    ids = order.astype(np.int32)
    sel = np.take_along_axis(lg, order, axis=1).astype(np.float64)
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    w = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return np.ascontiguousarray(ids), np.ascontiguousarray(w)


def routing(M: int, layer: Layer, seed: int = 0, zipf_s: Optional[float] = None):
    return route(logits(M, layer.E, seed, zipf_s), layer.k)


def packed_codes(N: int, K: int, seed: int, tag: int, e: int) -> np.ndarray:
    """[N][K/2] uint8: two uniform 4-bit codes per byte (raw PCG64 output)."""
    nbytes = N * (K // 2)
    assert nbytes % 8 == 0
    bg = np.random.PCG64(np.random.SeedSequence([seed, tag, e]))
    return bg.random_raw(nbytes // 8).view(np.uint8).reshape(N, K // 2)


def scales(N: int, K: int, seed: int, tag: int, e: int, group: int = GROUP) -> np.ndarray:
    """[N][K/group] bf16 bit patterns, uniform on [0.002, 0.02]."""
    g = _rng(seed, tag, e)
    s = g.uniform(SCALE_LO, SCALE_HI, size=(N, K // group)).astype(np.float32)
    return f32_to_bf16_bits(s)


def expert_weights(layer: Layer, e: int, seed: int = 0):
    """(w13[2I][H/2], s13[2I][H/32], w2[H][I/2], s2[H][I/32]) of expert e."""
    H, I, g = layer.H, layer.I, layer.group
    return (packed_codes(2 * I, H, seed, TAG_W13, e), scales(2 * I, H, seed, TAG_S13, e, g),
            packed_codes(H, I, seed, TAG_W2, e), scales(H, I, seed, TAG_S2, e, g))


def layer_weights(layer: Layer, seed: int = 0, experts: Optional[Sequence[int]] = None):
    """Full canonical arrays [E][...] for every expert.  When ``experts`` is
    given, only those experts are drawn and the others are left zero (codes
    0 and scale 0), which is enough for an oracle restricted to them."""
    from concurrent.futures import ThreadPoolExecutor
    import os

    E, H, I = layer.E, layer.H, layer.I
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    s13 = np.zeros((E, 2 * I, H // layer.group), np.uint16)
    w2 = np.zeros((E, H, I // 2), np.uint8)
    s2 = np.zeros((E, H, I // layer.group), np.uint16)

    def fill(e):
        w13[e], s13[e], w2[e], s2[e] = expert_weights(layer, int(e), seed)

    todo = list(range(E) if experts is None else experts)
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, todo))
    return w13, s13, w2, s2


def expected_active(layer: Layer, M: int) -> float:
    """Expected number of distinct experts under uniform routing."""
    return layer.E * (1.0 - (1.0 - layer.k / layer.E) ** M)
