"""Thin Python binding of libhca (the C ABI declared in include/hca.h).

Argument marshalling only: every entry point checks tensor dtypes/shapes,
allocates outputs and workspace through PyTorch (device memory is torch's),
passes raw pointers, sizes and torch's current CUDA stream to the C function
of the same name, and turns a non-zero status into an exception.  All of the
computation runs in libhca's CUDA kernels; there is no fallback of any kind,
and a missing library is an error.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhca.so")

HCA_BF16, HCA_F32 = 0, 1
_DTYPES = {torch.bfloat16: HCA_BF16, torch.float32: HCA_F32}

_lock = threading.Lock()
_lib = None

EXPORTS = ("hca_status_string", "hca_version", "hca_workspace_size", "hca_query_tile_positions", "hca_attn_fwd",
           "hca_attn_bwd", "hca_visible_pairs", "hca_tile_map", "hca_workspace_status", "hca_profile_enable",
           "hca_profile_read", "hca_num_kernels", "hca_kernel_name", "hca_attn_fwd_noalloc",
           "hca_local_workspace_size", "hca_local_attn_fwd", "hca_local_attn_bwd", "hca_test_inject",
           "hca_compress_fwd", "hca_compress_workspace_size", "hca_compress_bwd", "hca_indexer_workspace_size",
           "hca_indexer_topk", "hca_csa_workspace_size", "hca_csa_attn_fwd", "hca_csa_attn_bwd")

# failure-path test hooks (hca_test_inject)
INJECT_RESET, INJECT_LAUNCH_FAILURE, INJECT_STALL, INJECT_WAIT_LIMIT_NS, INJECT_CSA_UNION = 0, 1, 2, 3, 4


class HCAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {hca_status_string(status)}")


def load(path: str = LIB_PATH):
    """Load libhca.so and declare the C signatures (no CUDA call is made)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libhca.so is not built ({path}); run "
                                   "`python -m block_sparse_compressed_gb300.build`")
            lib = ctypes.CDLL(path)
            P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            lib.hca_status_string.argtypes = [I]
            lib.hca_status_string.restype = ctypes.c_char_p
            lib.hca_version.argtypes = []
            lib.hca_version.restype = I
            lib.hca_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
            lib.hca_workspace_size.restype = Z
            lib.hca_query_tile_positions.argtypes = [I, I, I]
            lib.hca_query_tile_positions.restype = I
            lib.hca_attn_fwd.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, Z, P]
            lib.hca_attn_fwd.restype = I
            lib.hca_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, Z, P]
            lib.hca_attn_bwd.restype = I
            lib.hca_visible_pairs.argtypes = [P, I, I, I, I, P, P, P, Z, P]
            lib.hca_visible_pairs.restype = I
            lib.hca_tile_map.argtypes = [P, I, I, I, I, I, P, P, Z, P]
            lib.hca_tile_map.restype = I
            lib.hca_workspace_status.argtypes = [P, P]
            lib.hca_workspace_status.restype = I
            lib.hca_profile_enable.argtypes = [I]
            lib.hca_profile_enable.restype = I
            lib.hca_profile_read.argtypes = [I, ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_double)]
            lib.hca_profile_read.restype = I
            lib.hca_num_kernels.argtypes = []
            lib.hca_num_kernels.restype = I
            lib.hca_kernel_name.argtypes = [I]
            lib.hca_kernel_name.restype = ctypes.c_char_p
            lib.hca_attn_fwd_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, I, P]
            lib.hca_attn_fwd_noalloc.restype = I
            lib.hca_local_workspace_size.argtypes = [I, I, I, I, I, I, I]
            lib.hca_local_workspace_size.restype = Z
            lib.hca_local_attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P, Z, P]
            lib.hca_local_attn_fwd.restype = I
            lib.hca_local_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, F, I, P, Z, P]
            lib.hca_local_attn_bwd.restype = I
            lib.hca_test_inject.argtypes = [I, ctypes.c_longlong]
            lib.hca_test_inject.restype = I
            lib.hca_compress_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
            lib.hca_compress_fwd.restype = I
            lib.hca_compress_workspace_size.argtypes = [I, I, I]
            lib.hca_compress_workspace_size.restype = Z
            lib.hca_compress_bwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, Z, P]
            lib.hca_compress_bwd.restype = I
            lib.hca_indexer_workspace_size.argtypes = [I, I, I]
            lib.hca_indexer_workspace_size.restype = Z
            lib.hca_indexer_topk.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, Z, P]
            lib.hca_indexer_topk.restype = I
            lib.hca_csa_workspace_size.argtypes = [I, I, I, I, I, I, I, I, I]
            lib.hca_csa_workspace_size.restype = Z
            lib.hca_csa_attn_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, Z, P]
            lib.hca_csa_attn_fwd.restype = I
            lib.hca_csa_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, Z, P]
            lib.hca_csa_attn_bwd.restype = I
            _lib = lib
    return _lib


def hca_status_string(status: int) -> str:
    return load().hca_status_string(int(status)).decode()


def hca_version() -> int:
    return load().hca_version()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")
    return _DTYPES[t.dtype]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _on(device):
    """Make `device` the current CUDA device for the C call: the library
    resolves per-device state (kernel attributes, the built-in scratch of the
    no-allocation entry point) on the current device."""
    device = torch.device(device)
    return torch.cuda.device(device) if device.type == "cuda" else contextlib.nullcontext()


def _check(rc: int, where: str):
    if rc != 0:
        raise HCAError(rc, where)


def _need(t: torch.Tensor, name: str, shape, dtype, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def hca_workspace_size(B: int, H: int, S: int, D: int, W: int, m: int, dtype: torch.dtype,
                       for_backward: bool) -> int:
    return load().hca_workspace_size(B, H, S, D, W, m, _DTYPES[dtype], int(for_backward))


def hca_query_tile_positions(H: int, D: int, dtype: torch.dtype) -> int:
    return load().hca_query_tile_positions(H, D, _DTYPES[dtype])


def workspace(B, H, S, D, W, m, dtype, for_backward, device) -> torch.Tensor:
    n = hca_workspace_size(B, H, S, D, W, m, dtype, for_backward)
    if n == 0:
        raise ValueError("invalid sizes for hca_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def hca_workspace_status(ws: torch.Tensor) -> int:
    """Synchronise the current stream and return the device-recorded status."""
    with _on(ws.device):
        return load().hca_workspace_status(_ptr(ws), _stream(ws.device))


def hca_test_inject(what: int, value: int = 0) -> None:
    """Failure-path test hook (include/hca.h, hca_test_inject)."""
    _check(load().hca_test_inject(int(what), int(value)), "hca_test_inject")


def _shapes(q, kv, ckv, seg, m):
    if q.dim() != 4:
        raise ValueError("q must be [B,H,S,D]")
    B, H, S, D = q.shape
    Sc = -(-S // m)
    dev = q.device
    _need(kv, "kv", (B, S, D), q.dtype, dev)
    _need(ckv, "ckv", (B, Sc, D), q.dtype, dev)
    if seg is not None:
        _need(seg, "seg", (B, S), torch.int32, dev)
    return B, H, S, D, Sc


def hca_attn_fwd(q: torch.Tensor, kv: torch.Tensor, ckv: torch.Tensor, seg: Optional[torch.Tensor], W: int,
                 m: int, scale: float, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 ws: Optional[torch.Tensor] = None, check: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """HCA forward: returns (out[B,H,S,D], lse[B,H,S] fp32)."""
    lib = load()
    if m < 1:
        raise ValueError("m must be >= 1")
    B, H, S, D, Sc = _shapes(q, kv, ckv, seg, m)
    _need(q, "q", q.shape, q.dtype, q.device)
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, S, dtype=torch.float32, device=q.device)
    _need(out, "out", q.shape, q.dtype, q.device)
    _need(lse, "lse", (B, H, S), torch.float32, q.device)
    if ws is None:
        ws = workspace(B, H, S, D, W, m, q.dtype, False, q.device)
    with _on(q.device):
        rc = lib.hca_attn_fwd(_ptr(q), _ptr(kv), _ptr(ckv), _ptr(seg), _ptr(out), _ptr(lse), B, H, S, D, W, m,
                              float(scale), dt, _ptr(ws), ws.numel(), _stream(q.device))
    _check(rc, "hca_attn_fwd")
    if check:
        _check(hca_workspace_status(ws), "hca_attn_fwd (device)")
    return out, lse


def hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, W: int, m: int, scale: float, dq=None, dkv=None, dckv=None,
                 ws=None, check: bool = False):
    """HCA backward: returns (dq[B,H,S,D], dkv[B,S,D], dckv[B,Sc,D])."""
    lib = load()
    if m < 1:
        raise ValueError("m must be >= 1")
    B, H, S, D, Sc = _shapes(q, kv, ckv, seg, m)
    _need(q, "q", q.shape, q.dtype, q.device)
    _need(out, "out", q.shape, q.dtype, q.device)
    _need(dout, "dout", q.shape, q.dtype, q.device)
    _need(lse, "lse", (B, H, S), torch.float32, q.device)
    dt = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dkv = torch.empty_like(kv) if dkv is None else dkv
    dckv = torch.empty_like(ckv) if dckv is None else dckv
    _need(dq, "dq", q.shape, q.dtype, q.device)
    _need(dkv, "dkv", kv.shape, q.dtype, q.device)
    _need(dckv, "dckv", ckv.shape, q.dtype, q.device)
    if ws is None:
        ws = workspace(B, H, S, D, W, m, q.dtype, True, q.device)
    with _on(q.device):
        rc = lib.hca_attn_bwd(_ptr(q), _ptr(kv), _ptr(ckv), _ptr(seg), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                              _ptr(dkv), _ptr(dckv), B, H, S, D, W, m, float(scale), dt, _ptr(ws), ws.numel(),
                              _stream(q.device))
    _check(rc, "hca_attn_bwd")
    if check:
        _check(hca_workspace_status(ws), "hca_attn_bwd (device)")
    return dq, dkv, dckv


def hca_local_workspace_size(B: int, H: int, S: int, D: int, W: int, dtype: torch.dtype, for_backward: bool) -> int:
    return load().hca_local_workspace_size(B, H, S, D, W, _DTYPES[dtype], int(for_backward))


def local_workspace(B, H, S, D, W, dtype, for_backward, device) -> torch.Tensor:
    n = hca_local_workspace_size(B, H, S, D, W, dtype, for_backward)
    if n == 0:
        raise ValueError("invalid sizes for hca_local_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _local_shapes(q, kv, seg):
    if q.dim() != 4:
        raise ValueError("q must be [B,H,S,D]")
    B, H, S, D = q.shape
    _need(kv, "kv", (B, S, D), q.dtype, q.device)
    if seg is not None:
        _need(seg, "seg", (B, S), torch.int32, q.device)
    return B, H, S, D


def hca_local_attn_fwd(q, kv, seg, W: int, scale: float, out=None, lse=None, ws=None, check: bool = False):
    """Local sliding-window attention forward: returns (out, lse)."""
    lib = load()
    B, H, S, D = _local_shapes(q, kv, seg)
    dt = _dtype_code(q)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(B, H, S, dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, "out", q.shape, q.dtype, q.device)
    _need(lse, "lse", (B, H, S), torch.float32, q.device)
    if ws is None:
        ws = local_workspace(B, H, S, D, W, q.dtype, False, q.device)
    with _on(q.device):
        rc = lib.hca_local_attn_fwd(_ptr(q), _ptr(kv), _ptr(seg), _ptr(out), _ptr(lse), B, H, S, D, W, float(scale), dt,
                                    _ptr(ws), ws.numel(), _stream(q.device))
    _check(rc, "hca_local_attn_fwd")
    if check:
        _check(hca_workspace_status(ws), "hca_local_attn_fwd (device)")
    return out, lse


def hca_local_attn_bwd(q, kv, seg, out, lse, dout, W: int, scale: float, dq=None, dkv=None, ws=None,
                       check: bool = False):
    """Local sliding-window attention backward: returns (dq, dkv)."""
    lib = load()
    B, H, S, D = _local_shapes(q, kv, seg)
    _need(out, "out", q.shape, q.dtype, q.device)
    _need(dout, "dout", q.shape, q.dtype, q.device)
    _need(lse, "lse", (B, H, S), torch.float32, q.device)
    dt = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dkv = torch.empty_like(kv) if dkv is None else dkv
    _need(dq, "dq", q.shape, q.dtype, q.device)
    _need(dkv, "dkv", kv.shape, q.dtype, q.device)
    if ws is None:
        ws = local_workspace(B, H, S, D, W, q.dtype, True, q.device)
    with _on(q.device):
        rc = lib.hca_local_attn_bwd(_ptr(q), _ptr(kv), _ptr(seg), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dkv),
                                    B, H, S, D, W, float(scale), dt, _ptr(ws), ws.numel(), _stream(q.device))
    _check(rc, "hca_local_attn_bwd")
    if check:
        _check(hca_workspace_status(ws), "hca_local_attn_bwd (device)")
    return dq, dkv


def hca_visible_pairs(seg: Optional[torch.Tensor], B: int, S: int, W: int, m: int, device=None):
    """(raw_pairs[B], comp_pairs[B]) int64 device tensors."""
    lib = load()
    device = seg.device if seg is not None else torch.device(device or "cuda")
    raw = torch.empty(B, dtype=torch.int64, device=device)
    comp = torch.empty(B, dtype=torch.int64, device=device)
    ws = workspace(B, 1, S, 16, W, m, torch.float32, False, device)
    with _on(device):
        rc = lib.hca_visible_pairs(_ptr(seg), B, S, W, m, _ptr(raw), _ptr(comp), _ptr(ws), ws.numel(), _stream(device))
    _check(rc, "hca_visible_pairs")
    return raw, comp


def hca_tile_map(seg: Optional[torch.Tensor], B: int, S: int, W: int, m: int, Pq: int, device=None):
    """int32 [B, ceil(S/Pq), 4] device tensor of per-tile key ranges."""
    lib = load()
    device = seg.device if seg is not None else torch.device(device or "cuda")
    nt = -(-S // Pq)
    out = torch.empty(B, nt, 4, dtype=torch.int32, device=device)
    ws = workspace(B, 1, S, 16, W, m, torch.float32, False, device)
    with _on(device):
        rc = lib.hca_tile_map(_ptr(seg), B, S, W, m, Pq, _ptr(out), _ptr(ws), ws.numel(), _stream(device))
    _check(rc, "hca_tile_map")
    return out


def hca_profile_enable(on: bool = True) -> None:
    _check(load().hca_profile_enable(int(on)), "hca_profile_enable")


def hca_profile_read() -> dict:
    """{kernel name: (launches, total_ms)} since the last enable (syncs)."""
    lib = load()
    res = {}
    for k in range(lib.hca_num_kernels()):
        n, ms = ctypes.c_longlong(0), ctypes.c_double(0.0)
        _check(lib.hca_profile_read(k, ctypes.byref(n), ctypes.byref(ms)), "hca_profile_read")
        res[lib.hca_kernel_name(k).decode()] = (int(n.value), float(ms.value))
    return res


NOALLOC_MAX_POSITIONS = 1 << 20


def hca_attn_fwd_noalloc(q, kv, ckv, seg, W: int, m: int, scale: float, out=None, lse=None):
    """Forward through the entry point that uses the library's built-in
    scratch instead of a workspace (for callers that cannot allocate device
    memory; B*S <= NOALLOC_MAX_POSITIONS).  Returns (out, lse)."""
    lib = load()
    if m < 1:
        raise ValueError("m must be >= 1")
    B, H, S, D, Sc = _shapes(q, kv, ckv, seg, m)
    _need(q, "q", q.shape, q.dtype, q.device)
    dt = _dtype_code(q)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(B, H, S, dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, "out", q.shape, q.dtype, q.device)
    _need(lse, "lse", (B, H, S), torch.float32, q.device)
    with _on(q.device):
        rc = lib.hca_attn_fwd_noalloc(_ptr(q), _ptr(kv), _ptr(ckv), _ptr(seg), _ptr(out), _ptr(lse), B, H, S, D, W, m,
                                      float(scale), dt, _stream(q.device))
    _check(rc, "hca_attn_fwd_noalloc")
    return out, lse


def hca_compress_fwd(x: torch.Tensor, g: torch.Tensor, bias: torch.Tensor, seg: Optional[torch.Tensor], m: int,
                     ckv: Optional[torch.Tensor] = None) -> torch.Tensor:
    """HCA compressor: ckv[B, ceil(S/m), D] from x[B,S,D], gates g[B,S] fp32,
    block bias[m] fp32 (include/hca.h, hca_compress_fwd)."""
    lib = load()
    B, S, D = x.shape
    Sc = -(-S // m)
    dev = x.device
    _need(x, "x", (B, S, D), x.dtype, dev)
    _need(g, "g", (B, S), torch.float32, dev)
    _need(bias, "bias", (m,), torch.float32, dev)
    if seg is not None:
        _need(seg, "seg", (B, S), torch.int32, dev)
    ckv = torch.empty(B, Sc, D, dtype=x.dtype, device=dev) if ckv is None else ckv
    _need(ckv, "ckv", (B, Sc, D), x.dtype, dev)
    with _on(dev):
        rc = lib.hca_compress_fwd(_ptr(x), _ptr(g), _ptr(bias), _ptr(seg), _ptr(ckv), B, S, D, m, _dtype_code(x),
                                  _stream(dev))
    _check(rc, "hca_compress_fwd")
    return ckv


def hca_compress_bwd(x, g, bias, seg, m: int, dckv, dx=None, dg=None, dbias=None, ws=None):
    """Backward of the compressor: (dx[B,S,D], dg[B,S] fp32, dbias[m] fp32)."""
    lib = load()
    B, S, D = x.shape
    Sc = -(-S // m)
    dev = x.device
    _need(dckv, "dckv", (B, Sc, D), x.dtype, dev)
    dx = torch.empty_like(x) if dx is None else dx
    dg = torch.empty(B, S, dtype=torch.float32, device=dev) if dg is None else dg
    dbias = torch.empty(m, dtype=torch.float32, device=dev) if dbias is None else dbias
    if ws is None:
        ws = torch.empty(lib.hca_compress_workspace_size(B, S, m), dtype=torch.uint8, device=dev)
    with _on(dev):
        rc = lib.hca_compress_bwd(_ptr(x), _ptr(g), _ptr(bias), _ptr(seg), _ptr(dckv), _ptr(dx), _ptr(dg),
                                  _ptr(dbias), B, S, D, m, _dtype_code(x), _ptr(ws), ws.numel(), _stream(dev))
    _check(rc, "hca_compress_bwd")
    return dx, dg, dbias


def hca_indexer_topk(qi: torch.Tensor, ki: torch.Tensor, w: torch.Tensor, seg: Optional[torch.Tensor], m: int,
                     k: int, with_scores: bool = False, ws: Optional[torch.Tensor] = None, check: bool = False):
    """Lightning Indexer top-k: (sel[B,S,k] int32, scores[B,S,Sc] fp32 or
    None) from qi[B,S,Hi,128], ki[B,ceil(S/m),128] (bf16), w[B,S,Hi] fp32."""
    lib = load()
    B, S, Hi, Di = qi.shape
    Sc = -(-S // m)
    dev = qi.device
    _need(qi, "qi", (B, S, Hi, Di), torch.bfloat16, dev)
    _need(ki, "ki", (B, Sc, Di), torch.bfloat16, dev)
    _need(w, "w", (B, S, Hi), torch.float32, dev)
    if seg is not None:
        _need(seg, "seg", (B, S), torch.int32, dev)
    sel = torch.empty(B, S, k, dtype=torch.int32, device=dev)
    scores = torch.empty(B, S, Sc, dtype=torch.float32, device=dev) if with_scores else None
    if ws is None:
        ws = torch.empty(lib.hca_indexer_workspace_size(B, S, m), dtype=torch.uint8, device=dev)
    with _on(dev):
        rc = lib.hca_indexer_topk(_ptr(qi), _ptr(ki), _ptr(w), _ptr(seg), _ptr(sel), _ptr(scores), B, S, Hi, Di, m, k,
                                  _ptr(ws), ws.numel(), _stream(dev))
    _check(rc, "hca_indexer_topk")
    if check:
        _check(hca_workspace_status(ws), "hca_indexer_topk (device)")
    return sel, scores


def csa_workspace(B, H, S, D, W, m, k, dtype, for_backward, device) -> torch.Tensor:
    n = load().hca_csa_workspace_size(B, H, S, D, W, m, k, _DTYPES[dtype], int(for_backward))
    if n == 0:
        raise HCAError(8, "hca_csa_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def hca_csa_attn_fwd(q, kv, ckv, seg, sel, W: int, m: int, scale: float, out=None, lse=None, ws=None,
                     check: bool = False):
    """CSA forward: (out, lse); sel[B,S,k] int32 selected compressed entries."""
    lib = load()
    B, H, S, D, Sc = _shapes(q, kv, ckv, seg, m)
    k = sel.shape[-1]
    _need(sel, "sel", (B, S, k), torch.int32, q.device)
    dt = _dtype_code(q)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(B, H, S, dtype=torch.float32, device=q.device) if lse is None else lse
    ws = csa_workspace(B, H, S, D, W, m, k, q.dtype, False, q.device) if ws is None else ws
    with _on(q.device):
        rc = lib.hca_csa_attn_fwd(_ptr(q), _ptr(kv), _ptr(ckv), _ptr(seg), _ptr(sel), _ptr(out), _ptr(lse), B, H, S,
                                  D, W, m, k, float(scale), dt, _ptr(ws), ws.numel(), _stream(q.device))
    _check(rc, "hca_csa_attn_fwd")
    if check:
        _check(hca_workspace_status(ws), "hca_csa_attn_fwd (device)")
    return out, lse


def hca_csa_attn_bwd(q, kv, ckv, seg, sel, out, lse, dout, W: int, m: int, scale: float, dq=None, dkv=None,
                     dckv=None, ws=None, check: bool = False):
    """CSA backward: (dq, dkv, dckv)."""
    lib = load()
    B, H, S, D, Sc = _shapes(q, kv, ckv, seg, m)
    k = sel.shape[-1]
    _need(sel, "sel", (B, S, k), torch.int32, q.device)
    dt = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dkv = torch.empty_like(kv) if dkv is None else dkv
    dckv = torch.empty_like(ckv) if dckv is None else dckv
    ws = csa_workspace(B, H, S, D, W, m, k, q.dtype, True, q.device) if ws is None else ws
    with _on(q.device):
        rc = lib.hca_csa_attn_bwd(_ptr(q), _ptr(kv), _ptr(ckv), _ptr(seg), _ptr(sel), _ptr(out), _ptr(lse),
                                  _ptr(dout), _ptr(dq), _ptr(dkv), _ptr(dckv), B, H, S, D, W, m, k, float(scale), dt,
                                  _ptr(ws), ws.numel(), _stream(q.device))
    _check(rc, "hca_csa_attn_bwd")
    if check:
        _check(hca_workspace_status(ws), "hca_csa_attn_bwd (device)")
    return dq, dkv, dckv
