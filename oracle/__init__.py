"""fp64 CPU oracle for Heavily Compressed Attention (HCA) and for its sparse
variant (CSA: the same sets, compressed entries also selected per query by an
indexer keep mask that is an input here).

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the
product library never imports, links or calls it, and it shares no code with
the CUDA path.  The arithmetic lives in ``hca_oracle.c`` (plain C, doubles,
one visibility predicate evaluated per (query, key) element); this module only
compiles it with gcc and marshals numpy arrays through ctypes.

Definitions followed (see the header of ``hca_oracle.c`` for the full text):
"Add HCA Static Compilation for Splash Attention [Deepseek v4]", Description
(sliding window plus completed compression windows; segment ids; unaligned
lengths), "DSV4: Route compressed and sliding train attention onto the splash
kernels", review suggestion on the segment mask (equal ids), and
"[DeepSeek-V4] Implement Compressed Attention Layers", review suggestions on
the einsums (k = v = the single shared kv head).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hca_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, F32, F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``hca_oracle.c`` into ``liboracle.so`` (gcc, portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lpthread", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i, d = ctypes.c_int, ctypes.c_double
            lib.hca_oracle_fwd.argtypes = [P, P, P, P, i, i, i, i, i, i, i, d, i, i, P, P, i]
            lib.hca_oracle_bwd.argtypes = [P, P, P, P, P, i, i, i, i, i, i, i, d, i, i, P, P, P, i]
            lib.hca_oracle_bwd_keys.argtypes = [P, P, P, P, P, i, i, i, i, i, i, i, d, P, i, P, i, P, P, i]
            lib.hca_oracle_visible_pairs.argtypes = [P, i, i, i, i, P, P]
            lib.hca_oracle_tile_ranges.argtypes = [P, i, i, i, i, i, P]
            lib.hca_oracle_num_threads.argtypes = [i]
            lib.hca_oracle_csa_fwd.argtypes = [P, P, P, P, P, i, i, i, i, i, i, i, d, i, i, P, P, i]
            lib.hca_oracle_csa_bwd.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, i, d, i, i, P, P, P, i]
            lib.hca_oracle_csa_visible_pairs.argtypes = [P, P, i, i, i, i, P, P]
            for f in ("hca_oracle_fwd", "hca_oracle_bwd", "hca_oracle_bwd_keys",
                      "hca_oracle_visible_pairs", "hca_oracle_tile_ranges", "hca_oracle_num_threads",
                      "hca_oracle_csa_fwd", "hca_oracle_csa_bwd", "hca_oracle_csa_visible_pairs"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads(nthreads: int = 0) -> int:
    return _load().hca_oracle_num_threads(nthreads)


def _arr(x):
    """Return (contiguous array, dtype code) for an input tensor.

    Accepts numpy arrays (float64 / float32) or torch tensors (bfloat16,
    float32, float64 on the CPU); bf16 is passed as its raw 16-bit pattern.
    """
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, BF16
    if x.dtype == np.float32:
        return x, F32
    return np.ascontiguousarray(x, dtype=np.float64), F64


def _seg(seg, B, S):
    if seg is None:
        return None
    try:
        import torch
        if isinstance(seg, torch.Tensor):
            seg = seg.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    s = np.ascontiguousarray(seg, dtype=np.int32)
    assert s.shape == (B, S), s.shape
    return s


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _inputs(q, kv, ckv, dout=None):
    qa, dt = _arr(q)
    kva, dt2 = _arr(kv)
    ca, dt3 = _arr(ckv)
    if not (dt == dt2 == dt3):
        raise TypeError("q, kv and ckv must share one dtype")
    da = None
    if dout is not None:
        da, dt4 = _arr(dout)
        if dt4 != dt:
            raise TypeError("dout must have the dtype of q")
    return qa, kva, ca, da, dt


def fwd(q, kv, ckv, seg, W: int, m: int, scale: float, rows=None, nthreads: int = 0):
    """out[B,H,S,D], lse[B,H,S] (float64).  ``rows=(lo,hi)`` restricts the
    query positions evaluated (others are NaN)."""
    qa, kva, ca, _, dt = _inputs(q, kv, ckv)
    B, H, S, D = qa.shape
    sg = _seg(seg, B, S)
    lo, hi = rows if rows is not None else (0, S)
    out = np.full((B, H, S, D), np.nan)
    lse = np.full((B, H, S), np.nan)
    rc = _load().hca_oracle_fwd(_ptr(qa), _ptr(kva), _ptr(ca), _ptr(sg), dt, B, H, S, D, W, m, float(scale),
                                lo, hi, _ptr(out), _ptr(lse), nthreads)
    if rc != 0:
        raise RuntimeError(f"hca_oracle_fwd failed ({rc})")
    return out, lse


def bwd(q, kv, ckv, seg, dout, W: int, m: int, scale: float, rows=None, nthreads: int = 0):
    """dq[B,H,S,D], dkv[B,S,D], dckv[B,Sc,D] (float64).  With ``rows=(lo,hi)``
    dq covers only those query positions and dkv/dckv hold only their
    contributions."""
    qa, kva, ca, da, dt = _inputs(q, kv, ckv, dout)
    B, H, S, D = qa.shape
    Sc = -(-S // m)
    sg = _seg(seg, B, S)
    lo, hi = rows if rows is not None else (0, S)
    dq = np.full((B, H, S, D), np.nan)
    dkv = np.zeros((B, S, D))
    dckv = np.zeros((B, Sc, D))
    rc = _load().hca_oracle_bwd(_ptr(qa), _ptr(kva), _ptr(ca), _ptr(sg), _ptr(da), dt, B, H, S, D, W, m,
                                float(scale), lo, hi, _ptr(dq), _ptr(dkv), _ptr(dckv), nthreads)
    if rc != 0:
        raise RuntimeError(f"hca_oracle_bwd failed ({rc})")
    return dq, dkv, dckv


def bwd_keys(q, kv, ckv, seg, dout, W: int, m: int, scale: float, raw_ids=(), comp_ids=(), nthreads: int = 0):
    """Exact gradients of selected keys over all queries.

    raw_ids: flat ids b*S+t of kv rows; comp_ids: flat ids b*Sc+j of ckv
    entries.  Returns (draw[n_raw,D], dcomp[n_comp,D]) in float64."""
    qa, kva, ca, da, dt = _inputs(q, kv, ckv, dout)
    B, H, S, D = qa.shape
    sg = _seg(seg, B, S)
    r = np.ascontiguousarray(np.asarray(raw_ids, dtype=np.int64).reshape(-1))
    c = np.ascontiguousarray(np.asarray(comp_ids, dtype=np.int64).reshape(-1))
    draw = np.zeros((len(r), D))
    dcomp = np.zeros((len(c), D))
    rc = _load().hca_oracle_bwd_keys(_ptr(qa), _ptr(kva), _ptr(ca), _ptr(sg), _ptr(da), dt, B, H, S, D, W, m,
                                     float(scale), _ptr(r), len(r), _ptr(c), len(c), _ptr(draw), _ptr(dcomp),
                                     nthreads)
    if rc != 0:
        raise RuntimeError(f"hca_oracle_bwd_keys failed ({rc})")
    return draw, dcomp


def visible_pairs(seg, B: int, S: int, W: int, m: int):
    """(raw_pairs[B], comp_pairs[B]) int64, counted per element (per head)."""
    sg = _seg(seg, B, S)
    raw = np.zeros(B, dtype=np.int64)
    comp = np.zeros(B, dtype=np.int64)
    rc = _load().hca_oracle_visible_pairs(_ptr(sg), B, S, W, m, _ptr(raw), _ptr(comp))
    if rc != 0:
        raise RuntimeError(f"hca_oracle_visible_pairs failed ({rc})")
    return raw, comp


def tile_ranges(seg, B: int, S: int, W: int, m: int, Pq: int):
    """int32[B, ceil(S/Pq), 4]: per query tile of Pq positions the half-open
    key ranges {raw_lo, raw_hi, comp_lo, comp_hi} holding all visible pairs."""
    sg = _seg(seg, B, S)
    nt = -(-S // Pq)
    out = np.zeros((B, nt, 4), dtype=np.int32)
    rc = _load().hca_oracle_tile_ranges(_ptr(sg), B, S, W, m, Pq, _ptr(out))
    if rc != 0:
        raise RuntimeError(f"hca_oracle_tile_ranges failed ({rc})")
    return out


# --------------------------------------------------------------------------
# compressed sparse attention (CSA): the HCA sets with an indexer selection
# --------------------------------------------------------------------------

def topk_mask(topk, Sc: int):
    """Dense keep mask uint8[B,S,Sc] from per-query index lists int[B,S,k]
    (entries outside [0, Sc), e.g. -1 padding, select nothing)."""
    try:
        import torch
        if isinstance(topk, torch.Tensor):
            topk = topk.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    t = np.asarray(topk, dtype=np.int64)
    B, S, _ = t.shape
    sel = np.zeros((B, S, Sc), dtype=np.uint8)
    b, i, _k = np.nonzero((t >= 0) & (t < Sc))
    sel[b, i, t[b, i, _k]] = 1
    return sel


def _sel(sel, B, S, Sc):
    s = np.ascontiguousarray(np.asarray(sel) != 0, dtype=np.uint8)
    assert s.shape == (B, S, Sc), s.shape
    return s


def csa_fwd(q, kv, ckv, seg, sel, W: int, m: int, scale: float, rows=None, nthreads: int = 0):
    """CSA out[B,H,S,D], lse[B,H,S] (float64); sel[B,S,Sc] keeps (query,
    compressed entry) pairs (see ``topk_mask``)."""
    qa, kva, ca, _, dt = _inputs(q, kv, ckv)
    B, H, S, D = qa.shape
    sg = _seg(seg, B, S)
    sl = _sel(sel, B, S, -(-S // m))
    lo, hi = rows if rows is not None else (0, S)
    out = np.full((B, H, S, D), np.nan)
    lse = np.full((B, H, S), np.nan)
    rc = _load().hca_oracle_csa_fwd(_ptr(qa), _ptr(kva), _ptr(ca), _ptr(sg), _ptr(sl), dt, B, H, S, D, W, m,
                                    float(scale), lo, hi, _ptr(out), _ptr(lse), nthreads)
    if rc != 0:
        raise RuntimeError(f"hca_oracle_csa_fwd failed ({rc})")
    return out, lse


def csa_bwd(q, kv, ckv, seg, sel, dout, W: int, m: int, scale: float, rows=None, nthreads: int = 0):
    """CSA dq[B,H,S,D], dkv[B,S,D], dckv[B,Sc,D] (float64)."""
    qa, kva, ca, da, dt = _inputs(q, kv, ckv, dout)
    B, H, S, D = qa.shape
    Sc = -(-S // m)
    sg = _seg(seg, B, S)
    sl = _sel(sel, B, S, Sc)
    lo, hi = rows if rows is not None else (0, S)
    dq = np.full((B, H, S, D), np.nan)
    dkv = np.zeros((B, S, D))
    dckv = np.zeros((B, Sc, D))
    rc = _load().hca_oracle_csa_bwd(_ptr(qa), _ptr(kva), _ptr(ca), _ptr(sg), _ptr(sl), _ptr(da), dt, B, H, S, D,
                                    W, m, float(scale), lo, hi, _ptr(dq), _ptr(dkv), _ptr(dckv), nthreads)
    if rc != 0:
        raise RuntimeError(f"hca_oracle_csa_bwd failed ({rc})")
    return dq, dkv, dckv


def csa_visible_pairs(seg, sel, B: int, S: int, W: int, m: int):
    """CSA (raw_pairs[B], comp_pairs[B]) int64, counted per element."""
    sg = _seg(seg, B, S)
    sl = _sel(sel, B, S, -(-S // m))
    raw = np.zeros(B, dtype=np.int64)
    comp = np.zeros(B, dtype=np.int64)
    rc = _load().hca_oracle_csa_visible_pairs(_ptr(sg), _ptr(sl), B, S, W, m, _ptr(raw), _ptr(comp))
    if rc != 0:
        raise RuntimeError(f"hca_oracle_csa_visible_pairs failed ({rc})")
    return raw, comp
