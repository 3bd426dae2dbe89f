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


def cheap_comp_ids(seg_row, S, m, max_queries=1500, count=6, seed=0):
    """Compressed entries whose exact gradient needs few queries (entries
    near the end of their document), plus entry ids spread over the row."""
    Sc = -(-S // m)
    seg_row = np.zeros(S, np.int32) if seg_row is None else seg_row
    ends = np.empty(S, np.int64)
    e = S - 1
    for x in range(S - 1, -1, -1):
        if x < S - 1 and seg_row[x] != seg_row[x + 1]:
            e = x
        ends[x] = e
    cands = []
    for j in range(Sc):
        lo, hi = j * m, (j + 1) * m - 1
        if hi >= S or seg_row[lo] < 0 or seg_row[lo] != seg_row[hi]:
            continue
        nq = ends[lo] - hi + 1
        if nq <= max_queries:
            cands.append(j)
    rng = np.random.Generator(np.random.PCG64(seed))
    if len(cands) > count:
        cands = sorted(rng.choice(cands, size=count, replace=False).tolist())
    return cands


def check_bwd_sampled(w, seed=1234, n_raw=24):
    q, kv, ckv, seg, dout = I.tensors(w, device=DEV, seed=seed)
    out, lse = hca.hca_attn_fwd(q, kv, ckv, seg, w.W, w.m, w.scale, check=True)
    dq, dkv, dckv = hca.hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, w.W, w.m, w.scale, check=True)
    torch.cuda.synchronize()
    qc, kvc, ckvc, dc = q.cpu(), kv.cpu(), ckv.cpu(), dout.cpu()
    segc = None if seg is None else seg.cpu()
    seg_np = None if segc is None else segc.numpy()
    Pq = hca.hca_query_tile_positions(w.H, w.D, w.dtype)
    dq_c, dkv_c, dckv_c = to_np(dq), to_np(dkv), to_np(dckv)
    rng = np.random.Generator(np.random.PCG64(seed))
    for b in range(w.B):
        sb = None if segc is None else segc[b:b + 1]
        srow = None if seg_np is None else seg_np[b]
        args = (qc[b:b + 1], kvc[b:b + 1], ckvc[b:b + 1], sb)
        # dq on sampled windows
        for lo, hi in sample_windows(srow, w.S, Pq, n_random=8, seed=b)[:24]:
            rdq, _, _ = oracle.bwd(*args, dc[b:b + 1], w.W, w.m, w.scale, rows=(lo, hi))
            valid = np.ones(hi - lo, bool) if srow is None else srow[lo:hi] >= 0
            got = dq_c[b][:, lo:hi]
            assert_close(f"dq b{b} [{lo},{hi})", got[:, valid], rdq[0][:, lo:hi][:, valid], w.dtype)
            assert np.all(got[:, ~valid] == 0)
        # dkv rows: document starts, the row ends and random rows
        n_valid = w.S if srow is None else int((srow >= 0).sum())
        raw = [0, 1, n_valid - 1, max(0, n_valid - 2)]
        if srow is not None:
            raw += (np.flatnonzero(np.diff(srow) != 0) + 1)[:8].tolist()
        raw += rng.integers(0, n_valid, size=n_raw).tolist()
        raw = sorted(set(int(x) for x in raw if 0 <= x < n_valid))
        comp = cheap_comp_ids(srow, w.S, w.m, seed=b)
        draw, dcomp = oracle.bwd_keys(*args, dc[b:b + 1], w.W, w.m, w.scale, raw_ids=raw, comp_ids=comp)
        assert_close(f"dkv b{b}", dkv_c[b][raw], draw, w.dtype)
        if comp:
            assert_close(f"dckv b{b}", dckv_c[b][comp], dcomp, w.dtype)
        # any size: the gradients of all keys sum to the sum of dO over valid rows
        valid = np.ones(w.S, bool) if srow is None else srow >= 0
        total = dkv_c[b].sum(0) + dckv_c[b].sum(0)
        expect = to_np(dout[b][:, torch.from_numpy(valid).to(DEV)].sum((0, 1)))
        assert_close(f"sum identity b{b}", total, expect, w.dtype)


def test_bwd_docs_16384():
    check_bwd_sampled(I.DOCS_S16384)


def test_bwd_unaligned_lengths():
    check_bwd_sampled(I.UNALIGNED)


def test_bwd_long_65536():
    check_bwd_sampled(I.LONG_S65536)


def test_bwd_long_131072():
    check_bwd_sampled(I.LONG_S131072, n_raw=12)


def test_backward_is_deterministic():
    w = I.DOCS_S16384
    q, kv, ckv, seg, dout = I.tensors(w, device=DEV)
    out, lse = hca.hca_attn_fwd(q, kv, ckv, seg, w.W, w.m, w.scale)
    a = hca.hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, w.W, w.m, w.scale)
    b = hca.hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, w.W, w.m, w.scale)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    o2, l2 = hca.hca_attn_fwd(q, kv, ckv, seg, w.W, w.m, w.scale)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_fwd_489_alone():
    # S = 3*128 + 105: ragged against both the tile and m
    w = I.Workload("S489", 1, 64, 489, 128, 128, 128, torch.bfloat16)
    q, kv, ckv, _, dout = I.tensors(w)
    g = [x.to(DEV) for x in (q, kv, ckv, dout)]
    out, lse = hca.hca_attn_fwd(g[0], g[1], g[2], None, w.W, w.m, w.scale, check=True)
    ro, rl = oracle.fwd(q, kv, ckv, None, w.W, w.m, w.scale)
    assert_close("out", out, ro, w.dtype)
    assert_close("lse", lse, rl, w.dtype)
    dq, dkv, dckv = hca.hca_attn_bwd(g[0], g[1], g[2], None, out, lse, g[3], w.W, w.m, w.scale, check=True)
    rdq, rdkv, rdckv = oracle.bwd(q, kv, ckv, None, dout, w.W, w.m, w.scale)
    assert_close("dq", dq, rdq, w.dtype)
    assert_close("dkv", dkv, rdkv, w.dtype)
    assert_close("dckv", dckv, rdckv, w.dtype)


def visible_comp_ids(seg_row, S, m):
    """Compressed entries that some query sees: the window lies in one
    document and completes before that document ends."""
    Sc = -(-S // m)
    out = []
    for j in range(Sc):
        lo, hi = j * m, (j + 1) * m - 1
        if hi >= S or seg_row[lo] < 0 or seg_row[lo] != seg_row[hi]:
            continue
        out.append(j)
    return out


def test_bwd_dckv_entries_exact_16384():
    # compressed entries 0, 1, the last visible one and random ones, each
    # exact over every query that sees it (no cap on the query count)
    w = I.DOCS_S16384
    q, kv, ckv, seg, dout = I.tensors(w, device=DEV)
    out, lse = hca.hca_attn_fwd(q, kv, ckv, seg, w.W, w.m, w.scale, check=True)
    _, _, dckv = hca.hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, w.W, w.m, w.scale, check=True)
    qc, kvc, ckvc, dc, segc = q.cpu(), kv.cpu(), ckv.cpu(), dout.cpu(), seg.cpu()
    dckv_c = to_np(dckv)
    rng = np.random.Generator(np.random.PCG64(7))
    for b in range(w.B):
        vis = visible_comp_ids(segc[b].numpy(), w.S, w.m)
        assert len(vis) >= 3
        ids = {vis[0], vis[1], vis[-1]} | set(rng.choice(vis, size=min(4, len(vis)), replace=False).tolist())
        ids = sorted(int(x) for x in ids)
        _, ref = oracle.bwd_keys(qc[b:b + 1], kvc[b:b + 1], ckvc[b:b + 1], segc[b:b + 1], dc[b:b + 1], w.W, w.m,
                                 w.scale, comp_ids=ids)
        assert_close(f"dckv b{b} entries {ids}", dckv_c[b][ids], ref, w.dtype)


def check_dckv_high_fan_in(w, seed=1234):
    """dckv entries that collect gradient from the most queries, each exact
    over every query that sees it: entry 0 (all queries from m - 1 on), entry
    1, the middle entry and the last visible one.  At this size those entries
    are summed through the split partial slots and the fixed-order reduce."""
    q, kv, ckv, seg, dout = I.tensors(w, device=DEV, seed=seed)
    assert seg is None or bool((seg >= 0).all())
    out, lse = hca.hca_attn_fwd(q, kv, ckv, seg, w.W, w.m, w.scale, check=True)
    _, _, dckv = hca.hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, w.W, w.m, w.scale, check=True)
    torch.cuda.synchronize()
    Sc = w.Sc
    last = w.S // w.m - 1                       # last window that completes
    ids = sorted({0, 1, Sc // 2, last})
    _, ref = oracle.bwd_keys(q.cpu(), kv.cpu(), ckv.cpu(), None if seg is None else seg.cpu(), dout.cpu(), w.W,
                             w.m, w.scale, comp_ids=ids)
    got = to_np(dckv)[0][ids]
    err = assert_close(f"dckv entries {ids}", got, ref, w.dtype)
    tol = 1e-2 * float(np.max(np.abs(ref))) + 1e-3
    per_entry = [float(np.max(np.abs(got[k] - ref[k]))) for k in range(len(ids))]
    print(f"{w.name}: dckv entries {ids} max|err| {err:.3e} of bound {tol:.3e} ({100 * err / tol:.1f} %); "
          f"per entry {[f'{e:.2e}' for e in per_entry]}")


def test_bwd_dckv_high_fan_in_65536():
    check_dckv_high_fan_in(I.LONG_S65536)


def test_bwd_dckv_high_fan_in_131072():
    check_dckv_high_fan_in(I.LONG_S131072)
