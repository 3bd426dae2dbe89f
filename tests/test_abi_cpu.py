"""Host-side checks of the C ABI: the library loads without a GPU, exports
every entry point declared in include/hca.h, and rejects bad arguments on the
host before any CUDA call.  No compute call is made here."""
import ctypes
import os
import re

import pytest
import torch

from block_sparse_compressed_gb300 import hca

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hca.h")

OK, E_NULL, E_SHAPE, E_DTYPE, E_ALIGN, E_ARG, E_SEG, E_WS, E_UNSUP, E_CUDA = range(10)


@pytest.fixture(scope="module")
def lib():
    from block_sparse_compressed_gb300 import build
    build.build()
    return hca.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"HCA_API[^;]*?\b(hca_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert set(declared_symbols()) == set(hca.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for s in range(11):
        assert hca.hca_status_string(s).startswith("HCA_")
    assert "UNKNOWN" in hca.hca_status_string(99)
    assert hca.hca_version() >= 1


def test_workspace_is_linear_not_quadratic(lib):
    f = lambda S, bwd: lib.hca_workspace_size(1, 64, S, 128, 128, 128, 0, bwd)  # noqa: E731
    for bwd in (0, 1):
        a, b = f(65536, bwd), f(131072, bwd)
        assert 0 < a < b <= 2 * a + 4096 * 1024, (a, b)
        # far below one byte per (query, key) pair (the backward keeps fp32
        # partial sums per key block: a fixed number of slots per row)
        assert b < 131072 * 131072 // 32
    assert lib.hca_workspace_size(1, 64, 1024, 128, 0, 128, 0, 0) == 0   # W < 1
    assert lib.hca_workspace_size(1, 64, 1024, 128, 128, 0, 0, 0) == 0   # m < 1
    assert lib.hca_workspace_size(1, 64, 1024, 128, 128, 128, 7, 0) == 0  # dtype


def _fwd(lib, **kw):
    a = dict(q=16, kv=16, ckv=16, seg=None, out=16, lse=16, B=1, H=4, S=64, D=128, W=8, m=4, scale=0.1, dt=0,
             ws=256, wsb=1 << 20, stream=None)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731
    return lib.hca_attn_fwd(P(a["q"]), P(a["kv"]), P(a["ckv"]), P(a["seg"]), P(a["out"]), P(a["lse"]), a["B"], a["H"],
                            a["S"], a["D"], a["W"], a["m"], a["scale"], a["dt"], P(a["ws"]), a["wsb"], a["stream"])


def test_argument_errors_are_caught_on_the_host(lib):
    # every case below returns before any CUDA call, so fake addresses are fine
    assert _fwd(lib, dt=5) == E_DTYPE
    assert _fwd(lib, W=0) == E_ARG
    assert _fwd(lib, m=0) == E_ARG
    assert _fwd(lib, scale=float("nan")) == E_ARG
    assert _fwd(lib, scale=float("inf")) == E_ARG
    assert _fwd(lib, H=0) == E_SHAPE
    assert _fwd(lib, D=0) == E_SHAPE
    assert _fwd(lib, D=1024) == E_SHAPE
    assert _fwd(lib, S=-1) == E_SHAPE
    assert _fwd(lib, D=12) == E_ALIGN              # 12 bf16 = 24 bytes
    assert _fwd(lib, q=None) == E_NULL
    assert _fwd(lib, lse=None) == E_NULL
    assert _fwd(lib, kv=24) == E_ALIGN
    assert _fwd(lib, seg=20) == E_ALIGN
    assert _fwd(lib, ws=None) == E_WS
    assert _fwd(lib, ws=128) == E_WS               # not 256-aligned
    assert _fwd(lib, wsb=16) == E_WS               # too small
    assert _fwd(lib, B=0) == OK                     # empty problem: nothing to do
    assert _fwd(lib, S=0) == OK
    # bf16 runs on the tensor-core kernels only (D = 64 or 128): other head
    # dims are rejected before anything is enqueued, never sent to CUDA cores
    assert _fwd(lib, D=32) == E_UNSUP
    assert _fwd(lib, D=256) == E_UNSUP
    # supported shapes pass that check and stop at the (too small) workspace,
    # still before any CUDA call
    assert _fwd(lib, D=64, wsb=16) == E_WS
    assert _fwd(lib, D=128, wsb=16) == E_WS
    assert _fwd(lib, D=256, dt=1, wsb=16) == E_WS   # fp32 runs every D


def test_backward_argument_errors(lib):
    P = ctypes.c_void_p
    args = [P(16)] * 10
    base = dict(B=1, H=4, S=64, D=128, W=8, m=4, scale=0.1, dt=0)

    def call(ptrs=None, ws=256, wsb=1 << 24, **kw):
        a = dict(base); a.update(kw)
        p = list(args if ptrs is None else ptrs)
        return lib.hca_attn_bwd(*p, a["B"], a["H"], a["S"], a["D"], a["W"], a["m"], a["scale"], a["dt"],
                                P(ws) if ws else None, wsb, None)

    assert call(W=0) == E_ARG
    p = list(args); p[7] = None            # dkv
    assert call(ptrs=p) == E_NULL
    p = list(args); p[9] = P(8)            # dckv misaligned
    assert call(ptrs=p) == E_ALIGN
    assert call(wsb=64) == E_WS
    p = list(args); p[3] = None            # seg = NULL is allowed: one segment
    assert call(ptrs=p, wsb=64) == E_WS


def test_test_hooks_argument_checks(lib):
    # the failure-path hooks validate their arguments on the host
    assert lib.hca_test_inject(0, 0) == OK
    assert lib.hca_test_inject(1, -1) == E_ARG
    assert lib.hca_test_inject(2, 8) == E_ARG       # not a mask of the three kernels
    assert lib.hca_test_inject(99, 0) == E_ARG
    assert lib.hca_test_inject(3, 1000) == OK
    assert lib.hca_test_inject(4, 1) == OK          # CSA union: sorting kernel
    assert lib.hca_test_inject(4, 128) == OK        # byte-mask kernel, 128-entry chunks
    assert lib.hca_test_inject(4, 63) == E_ARG      # chunks are multiples of 64
    assert lib.hca_test_inject(4, 16384 + 64) == E_ARG
    assert lib.hca_test_inject(0, 0) == OK


def test_head_packing_covers_every_head_count(lib):
    # Pq = 128 / (largest power of two dividing H and 128)
    for H, pq in ((1, 128), (3, 128), (6, 64), (48, 8), (64, 2), (96, 4), (128, 1), (256, 1), (384, 1)):
        assert lib.hca_query_tile_positions(H, 128, 0) == pq, H
    assert lib.hca_query_tile_positions(64, 64, 1) == 1   # fp32: one row per warp


def test_local_attention_host_checks(lib):
    # the local entry points are the HCA calls with an empty compressed set:
    # same argument checks, a workspace that exists for every valid size
    P = ctypes.c_void_p
    for bwd in (0, 1):
        assert lib.hca_local_workspace_size(1, 64, 65536, 128, 128, 0, bwd) > 0
        assert lib.hca_local_workspace_size(1, 64, 65536, 128, 0, 0, bwd) == 0   # W < 1
    rc = lib.hca_local_attn_fwd(P(16), P(16), None, P(16), P(16), 1, 4, 64, 128, 0, 0.1, 0, P(256), 1 << 20, None)
    assert rc == E_ARG
    rc = lib.hca_local_attn_fwd(P(16), P(16), None, P(16), P(16), 1, 4, 64, 128, 8, 0.1, 0, P(256), 16, None)
    assert rc == E_WS
    rc = lib.hca_local_attn_bwd(P(16), P(16), None, P(16), P(16), P(16), P(16), P(16), 1, 4, 64, 128, 8, 0.1, 0,
                                P(256), 64, None)
    assert rc == E_WS
    rc = lib.hca_local_attn_bwd(P(16), P(16), None, P(16), P(16), P(16), None, P(16), 1, 4, 64, 128, 8, 0.1, 0,
                                P(256), 1 << 26, None)
    assert rc == E_NULL


@pytest.mark.skipif(torch.cuda.is_available(), reason="uses fake device addresses; only meaningful without a GPU")
def test_valid_call_without_a_device_reports_cuda_error(lib):
    # with no GPU the first CUDA call fails: the ABI reports HCA_ERR_CUDA and
    # returns instead of aborting
    assert _fwd(lib) == E_CUDA
