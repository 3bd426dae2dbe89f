"""GPU parity of the local sliding-window attention entry points
(hca_local_attn_fwd / hca_local_attn_bwd) against the fp64 oracle.

Local sliding attention is HCA without the compressed set: the oracle runs
with a compression ratio longer than the sequence (no window completes), so
its compressed set is empty and only the raw window and the segment rule
remain.  Same tolerances as the HCA parity tests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_compressed_gb300 import hca
from block_sparse_compressed_gb300 import inputs as I
from _util import assert_close, to_np, valid_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_local(B, H, S, D, W, dtype, seg=None, seed=77):
    scale = 1.0 / math.sqrt(D)
    m = S + 1  # no compression window completes: empty compressed set
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, dtype=dtype, seed=seed)
    seg_t = None if seg is None else torch.as_tensor(np.asarray(seg, dtype=np.int32)).reshape(B, S)
    sg = None if seg_t is None else seg_t.to(DEV)
    gq, gkv, gdo = q.to(DEV), kv.to(DEV), dout.to(DEV)
    out, lse = hca.hca_local_attn_fwd(gq, gkv, sg, W, scale, check=True)
    ro, rl = oracle.fwd(q, kv, ckv, seg_t, W, m, scale)
    v = valid_rows(seg_t, B, H, S)
    assert_close("out", out, ro, dtype, v)
    assert_close("lse", lse, rl, dtype, v)
    assert np.all(to_np(out)[~v] == 0)
    dq, dkv = hca.hca_local_attn_bwd(gq, gkv, sg, out, lse, gdo, W, scale, check=True)
    rdq, rdkv, rdckv = oracle.bwd(q, kv, ckv, seg_t, dout, W, m, scale)
    assert np.all(np.asarray(rdckv) == 0)  # the oracle agrees the compressed set is empty
    assert_close("dq", dq, rdq, dtype, v)
    assert np.all(to_np(dq)[~v] == 0)
    assert_close("dkv", dkv, rdkv, dtype)


@pytest.mark.parametrize("W", [1, 64, 128, 300])
def test_local_bf16_documents(W):
    rng = np.random.Generator(np.random.PCG64(W))
    S = 1000
    seg = np.stack([I.random_layout(S, rng, allow_pad=True) for _ in range(2)])
    run_local(2, 64, S, 128, W, torch.bfloat16, seg)


@pytest.mark.parametrize("H", [1, 16, 128])
def test_local_bf16_heads_ragged(H):
    run_local(1, H, 489, 128, 128, torch.bfloat16)


def test_local_long_window_is_causal_attention():
    # W >= S: plain causal softmax attention over one document
    run_local(1, 16, 700, 128, 700, torch.bfloat16)


def test_local_f32():
    rng = np.random.Generator(np.random.PCG64(3))
    S = 300
    seg = np.stack([I.random_layout(S, rng)])
    run_local(1, 4, S, 64, 48, torch.float32, seg)


def test_local_s8192_one_document():
    run_local(1, 64, 8192, 128, 128, torch.bfloat16)


def test_local_full_size_sampled_rows():
    # the local bench workload, B1 H64 S65536 D128 W128: out, lse and dq on
    # sampled rows; dkv exactly for a few key ranges (key j is seen by the W
    # queries [j, j + W) alone, so those rows give its whole gradient)
    B, H, S, D, W = 1, 64, 65536, 128, 128
    m = S + 1
    scale = 1.0 / math.sqrt(D)
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, dtype=torch.bfloat16, seed=31, device=DEV)
    out, lse = hca.hca_local_attn_fwd(q, kv, None, W, scale, check=True)
    dq, dkv = hca.hca_local_attn_bwd(q, kv, None, out, lse, dout, W, scale, check=True)
    torch.cuda.synchronize()
    qc, kvc, ckvc, dc = q.cpu(), kv.cpu(), ckv.cpu(), dout.cpu()
    out_c, lse_c, dq_c, dkv_c = to_np(out)[0], to_np(lse)[0], to_np(dq)[0], to_np(dkv)[0]
    for lo in (0, 127, 33000, S - 2):
        hi = lo + 2
        ro, rl = oracle.fwd(qc, kvc, ckvc, None, W, m, scale, rows=(lo, hi))
        assert_close(f"out [{lo},{hi})", out_c[:, lo:hi], ro[0][:, lo:hi], torch.bfloat16)
        assert_close(f"lse [{lo},{hi})", lse_c[:, lo:hi], rl[0][:, lo:hi], torch.bfloat16)
        rdq, _, _ = oracle.bwd(qc, kvc, ckvc, None, dc, W, m, scale, rows=(lo, hi))
        assert_close(f"dq [{lo},{hi})", dq_c[:, lo:hi], rdq[0][:, lo:hi], torch.bfloat16)
    for j0 in (0, 40000, S - 4):
        _, rdkv, _ = oracle.bwd(qc, kvc, ckvc, None, dc, W, m, scale, rows=(j0, min(S, j0 + 3 + W)))
        assert_close(f"dkv [{j0},{j0 + 4})", dkv_c[j0:j0 + 4], rdkv[0][j0:j0 + 4], torch.bfloat16)
