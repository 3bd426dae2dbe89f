"""hca_attn_fwd_noalloc: the forward for callers that cannot allocate device
memory (runtime plugin hooks, real-time loops, hosts without an allocator).

It runs with the library's built-in scratch array instead of a caller
workspace.  This file is collected last on purpose: it must pass both alone in
a fresh process and after every other test, and two calls in a row must each
match the ordinary entry point (the shared array keeps the previous call's
contents, so the second call checks that nothing stale leaks through).
"""
import ctypes
import math

import pytest
import torch

from block_sparse_compressed_gb300 import hca
from block_sparse_compressed_gb300 import inputs as I

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, H, S, D, W, m, lens=None, seed=0):
    q, kv, ckv, _, _ = I.small(B, H, S, D, W, m, dtype=torch.bfloat16, seed=seed)
    seg = None
    if lens is not None:
        seg = torch.cat([I.segments_from_lengths(l, S, pad=S - sum(l)) for l in lens]).to(DEV)
    return q.to(DEV), kv.to(DEV), ckv.to(DEV), seg


def _noalloc_c_abi(q, kv, ckv, seg, W, m, scale):
    """Call the C entry point directly through ctypes."""
    lib = hca.load()
    B, H, S, D = q.shape
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=q.device)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.hca_attn_fwd_noalloc(P(q), P(kv), P(ckv), P(seg), P(out), P(lse), B, H, S, D, W, m, scale, 0, stream)
    assert rc == 0, hca.hca_status_string(rc)
    return out, lse


def _compare(q, kv, ckv, seg, W, m):
    scale = 1.0 / math.sqrt(q.shape[-1])
    ref_out, ref_lse = hca.hca_attn_fwd(q, kv, ckv, seg, W, m, scale, check=True)
    out, lse = _noalloc_c_abi(q, kv, ckv, seg, W, m, scale)
    torch.cuda.synchronize()
    # the same kernels on the same inputs: any difference at all would be
    # stale state leaking out of the shared scratch array
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)


def test_noalloc_matches_workspace_entry_point_twice():
    # first call: two batch rows with documents and padding
    q, kv, ckv, seg = _case(2, 16, 700, 128, 128, 64, lens=[[300, 250], [699]], seed=1)
    _compare(q, kv, ckv, seg, 128, 64)
    # second call right after, different sizes and layout, on the same array
    q, kv, ckv, seg = _case(1, 64, 1500, 128, 96, 32, lens=[[40, 1000, 200]], seed=2)
    _compare(q, kv, ckv, seg, 96, 32)


def test_noalloc_without_segments_and_fp32():
    q, kv, ckv, _ = _case(1, 4, 333, 128, 50, 16, seed=3)
    _compare(q, kv, ckv, None, 50, 16)
    q32, kv32, ckv32, _, _ = I.small(1, 4, 200, 64, 30, 8, dtype=torch.float32, seed=4)
    q32, kv32, ckv32 = q32.to(DEV), kv32.to(DEV), ckv32.to(DEV)
    ref_out, ref_lse = hca.hca_attn_fwd(q32, kv32, ckv32, None, 30, 8, 0.125)
    out, lse = hca.hca_attn_fwd_noalloc(q32, kv32, ckv32, None, 30, 8, 0.125)
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = hca.load()
    B, S = 2, hca.NOALLOC_MAX_POSITIONS // 2 + 1
    # rejected on the host before any pointer is touched or work enqueued
    fake = ctypes.c_void_p(256)
    rc = lib.hca_attn_fwd_noalloc(fake, fake, fake, None, fake, fake, B, 4, S, 128, 16, 16, 0.1, 0, None)
    assert rc == 7, hca.hca_status_string(rc)
