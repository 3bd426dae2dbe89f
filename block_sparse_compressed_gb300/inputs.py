"""Seeded synthetic inputs for HCA attention.

This module holds only input generation -- random tensors and packed-document
segment layouts -- and none of the attention arithmetic.  Both the CUDA tests
and the CPU oracle draw their inputs from here, so the two sides always see
identical bytes.

The pages measure on the DeepSeek-V4 model, whose weights and data are not
available; the shapes below (batch, heads, sequence length, head dim, window,
compression ratio, document-length mix) stand in for those workloads, with
q, kv, ckv and dO drawn i.i.d. N(0,1) in fp32 and cast to the compute dtype.

Seeds: tensor k of a workload uses ``seed + k`` with q=0, kv=1, ckv=2, dO=3
and the document lengths 4.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

SEED = 1234


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    W: int
    m: int
    dtype: torch.dtype
    layout: str = "single"            # single | halves | docs | lengths
    lengths: Optional[Sequence[int]] = None   # per-row valid lengths (layout=lengths)
    doc_range: Sequence[int] = (512, 8192)    # layout=docs: uniform doc-length range
    backward: bool = True

    @property
    def Sc(self) -> int:
        return -(-self.S // self.m)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# The five workloads of the benchmark description, by what they are.
TINY_F32 = Workload("tiny-f32 B1 H4 S512 D64 W64 m16", 1, 4, 512, 64, 64, 16, torch.float32)
FWD_S4096_2DOC = Workload("fwd bf16 B1 H16 S4096 D128 W128 m128 2x2048 docs", 1, 16, 4096, 128, 128, 128,
                          torch.bfloat16, layout="halves", backward=False)
DOCS_S16384 = Workload("fwd+bwd bf16 B2 H64 S16384 D128 W128 m128 docs U[512,8192]", 2, 64, 16384, 128, 128, 128,
                       torch.bfloat16, layout="docs")
UNALIGNED = Workload("fwd+bwd bf16 B4 H64 D128 W128 m128 lengths 489/3001/12345/32768", 4, 64, 32768, 128, 128, 128,
                     torch.bfloat16, layout="lengths", lengths=(489, 3001, 12345, 32768))
LONG_S131072 = Workload("fwd+bwd bf16 B1 H64 S131072 D128 W128 m128", 1, 64, 131072, 128, 128, 128, torch.bfloat16)
LONG_S65536 = Workload("fwd+bwd bf16 B1 H64 S65536 D128 W128 m128", 1, 64, 65536, 128, 128, 128, torch.bfloat16)

ALL = (TINY_F32, FWD_S4096_2DOC, DOCS_S16384, UNALIGNED, LONG_S131072, LONG_S65536)


def doc_lengths(S: int, lo: int, hi: int, seed: int) -> List[int]:
    """Document lengths drawn uniformly from [lo, hi] (inclusive) until they
    fill S; the last document is truncated so the lengths sum to S."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out, total = [], 0
    while total < S:
        L = int(rng.integers(lo, hi + 1))
        L = min(L, S - total)
        out.append(L)
        total += L
    return out


def segments(w: Workload, seed: int = SEED) -> Optional[torch.Tensor]:
    """int32 [B,S] segment ids (0,1,2,... per row; -1 = padding) or None for
    one unpadded segment per row."""
    B, S = w.B, w.S
    if w.layout == "single":
        return None
    seg = torch.empty(B, S, dtype=torch.int32)
    if w.layout == "halves":
        seg[:, : S // 2] = 0
        seg[:, S // 2:] = 1
    elif w.layout == "docs":
        for b in range(B):
            lens = doc_lengths(S, w.doc_range[0], w.doc_range[1], seed + 4 + 1000 * b)
            ids = np.repeat(np.arange(len(lens), dtype=np.int32), lens)
            seg[b] = torch.from_numpy(ids)
    elif w.layout == "lengths":
        assert w.lengths is not None and len(w.lengths) == B
        seg.fill_(-1)
        for b, L in enumerate(w.lengths):
            seg[b, :L] = 0
    else:
        raise ValueError(w.layout)
    return seg


def segments_from_lengths(lengths: Sequence[int], S: int, pad: int = 0) -> torch.Tensor:
    """One row of ids for documents of the given lengths, then ``pad``
    padding positions (-1); sum(lengths) + pad must equal S."""
    assert sum(lengths) + pad == S
    ids = np.concatenate([np.full(L, k, dtype=np.int32) for k, L in enumerate(lengths)] +
                         [np.full(pad, -1, dtype=np.int32)])
    return torch.from_numpy(ids).reshape(1, S)


def normal(shape, seed: int, dtype: torch.dtype, device="cpu") -> torch.Tensor:
    """i.i.d. N(0,1) drawn in fp32 from a seeded generator, then cast."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=device).to(dtype)


def tensors(w: Workload, device="cpu", seed: int = SEED, with_dout: bool = True):
    """(q[B,H,S,D], kv[B,S,D], ckv[B,Sc,D], seg[B,S]|None, dO[B,H,S,D]|None)."""
    q = normal((w.B, w.H, w.S, w.D), seed + 0, w.dtype, device)
    kv = normal((w.B, w.S, w.D), seed + 1, w.dtype, device)
    ckv = normal((w.B, w.Sc, w.D), seed + 2, w.dtype, device)
    dout = normal((w.B, w.H, w.S, w.D), seed + 3, w.dtype, device) if with_dout else None
    seg = segments(w, seed)
    if seg is not None:
        seg = seg.to(device)
    return q, kv, ckv, seg, dout


def small(B, H, S, D, W, m, dtype=torch.float64, seg=None, seed: int = SEED, device="cpu"):
    """Inputs for an ad-hoc small case (tests)."""
    Sc = -(-S // m)
    q = normal((B, H, S, D), seed + 0, dtype, device)
    kv = normal((B, S, D), seed + 1, dtype, device)
    ckv = normal((B, Sc, D), seed + 2, dtype, device)
    dout = normal((B, H, S, D), seed + 3, dtype, device)
    return q, kv, ckv, seg, dout


def random_layout(S: int, rng: np.random.Generator, max_docs: int = 6, allow_pad: bool = True) -> np.ndarray:
    """A random packed layout for tests: a few documents of random lengths
    (ids 0,1,2,...) optionally followed by padding (-1)."""
    pad = int(rng.integers(0, max(1, S // 4))) if (allow_pad and S > 1 and rng.random() < 0.5) else 0
    n = S - pad
    ndocs = int(rng.integers(1, max_docs + 1))
    if n <= 0:
        return np.full(S, -1, dtype=np.int32)
    cuts = np.sort(rng.choice(np.arange(1, n), size=min(ndocs - 1, max(0, n - 1)), replace=False)) if n > 1 else []
    bounds = [0] + list(cuts) + [n]
    ids = np.empty(S, dtype=np.int32)
    for k in range(len(bounds) - 1):
        ids[bounds[k]:bounds[k + 1]] = k
    ids[n:] = -1
    return ids


def random_selection(B: int, S: int, m: int, k: int, seed: int, extra: int = 2) -> torch.Tensor:
    """int32 [B,S,k] per-query compressed-entry selections for CSA tests and
    benchmarks (a stand-in for the indexer's top-k): entries drawn uniformly
    from [0, (i+1)//m + extra) for query i, so a few are not yet complete (the
    attention must ignore them), with repeats; the first and last slot of
    every fifth query are -1 (padding)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    hi = (np.arange(S) + 1) // m + extra
    u = rng.random((B, S, k))
    sel = np.floor(u * hi[None, :, None]).astype(np.int32)
    sel[:, ::5, 0] = -1
    sel[:, ::5, -1] = -1
    return torch.from_numpy(sel)
