"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times, against the fp64 oracle on sampled rows.

The oracle evaluates, per batch row, windows of consecutive query positions:
the first and last query tiles, every segment boundary +-2, and seeded random
windows.  Tolerance: max|err| <= 1e-2*max|ref| + 1e-3 per tensor (bf16).
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_compressed_gb300 import hca
from block_sparse_compressed_gb300 import inputs as I
from _util import assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def sample_windows(seg_row, S, Pq, n_random=24, width=4, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    wins = [(0, min(S, 2 * Pq)), (max(0, S - 2 * Pq), S)]
    if seg_row is not None:
        starts = np.flatnonzero(np.diff(seg_row) != 0) + 1
        for s in starts[:64]:
            wins.append((max(0, s - 2), min(S, s + 2)))
    for x in rng.integers(0, max(1, S - width), size=n_random):
        wins.append((int(x), int(min(S, x + width))))
    return wins


def check_fwd_sampled(w, seed=1234):
    q, kv, ckv, seg, _ = I.tensors(w, device=DEV, seed=seed, with_dout=False)
    out, lse = hca.hca_attn_fwd(q, kv, ckv, seg, w.W, w.m, w.scale, check=True)
    torch.cuda.synchronize()
    qc, kvc, ckvc = q.cpu(), kv.cpu(), ckv.cpu()
    segc = None if seg is None else seg.cpu()
    seg_np = None if segc is None else segc.numpy()
    Pq = hca.hca_query_tile_positions(w.H, w.D, w.dtype)
    out_c, lse_c = to_np(out), to_np(lse)
    for b in range(w.B):
        wins = sample_windows(None if seg_np is None else seg_np[b], w.S, Pq, seed=b)
        for lo, hi in wins:
            ro, rl = oracle.fwd(qc[b:b + 1], kvc[b:b + 1], ckvc[b:b + 1],
                                None if segc is None else segc[b:b + 1], w.W, w.m, w.scale, rows=(lo, hi))
            valid = np.ones(hi - lo, bool) if seg_np is None else seg_np[b, lo:hi] >= 0
            sl = slice(lo, hi)
            ref_o, ref_l = ro[0][:, sl], rl[0][:, sl]
            got_o, got_l = out_c[b][:, sl], lse_c[b][:, sl]
            assert_close(f"out b{b} [{lo},{hi})", got_o[:, valid], ref_o[:, valid], w.dtype)
            assert_close(f"lse b{b} [{lo},{hi})", got_l[:, valid], ref_l[:, valid], w.dtype)
            assert np.all(got_o[:, ~valid] == 0) and np.all(got_l[:, ~valid] == -np.inf)


def test_fwd_docs_16384():
    check_fwd_sampled(I.DOCS_S16384)


def test_fwd_unaligned_lengths():
    check_fwd_sampled(I.UNALIGNED)


def test_fwd_long_131072():
    check_fwd_sampled(I.LONG_S131072)


def test_fwd_long_65536():
    check_fwd_sampled(I.LONG_S65536)


def test_fwd_489_alone():
    # S = 3*128 + 105: ragged against both the tile and m
    w = I.Workload("S489", 1, 64, 489, 128, 128, 128, torch.bfloat16)
    q, kv, ckv, seg, _ = I.tensors(w, with_dout=False)
    out, lse = hca.hca_attn_fwd(q.to(DEV), kv.to(DEV), ckv.to(DEV), None, w.W, w.m, w.scale, check=True)
    ro, rl = oracle.fwd(q, kv, ckv, None, w.W, w.m, w.scale)
    assert_close("out", out, ro, w.dtype)
    assert_close("lse", lse, rl, w.dtype)
