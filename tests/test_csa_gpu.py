"""GPU parity of compressed sparse attention (hca_csa_attn_fwd / _bwd,
through the C ABI binding) against the fp64 oracle's CSA mode
(oracle.csa_fwd / csa_bwd with the selection as a keep mask).  Tolerance per
tensor over valid positions: bf16 max|err| <= 1e-2*max|ref| + 1e-3."""
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


def run_csa(B, H, S, W, m, k, seg=None, seed=7, backward=True, sel=None):
    D = 128
    scale = 1.0 / math.sqrt(D)
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, dtype=torch.bfloat16, seed=seed)
    Sc = -(-S // m)
    sel = I.random_selection(B, S, m, k, seed + 50) if sel is None else sel
    keep = oracle.topk_mask(sel, Sc)
    g = [x.to(DEV) for x in (q, kv, ckv, dout)]
    sg = None if seg is None else seg.to(DEV)
    out, lse = hca.hca_csa_attn_fwd(g[0], g[1], g[2], sg, sel.to(DEV), W, m, scale, check=True)
    ro, rl = oracle.csa_fwd(q, kv, ckv, seg, keep, W, m, scale)
    v = valid_rows(seg, B, H, S)
    assert_close("out", out, ro, torch.bfloat16, v)
    assert_close("lse", lse, rl, torch.bfloat16, v)
    if not backward:
        return
    dq, dkv, dckv = hca.hca_csa_attn_bwd(g[0], g[1], g[2], sg, sel.to(DEV), out, lse, g[3], W, m, scale, check=True)
    rdq, rdkv, rdckv = oracle.csa_bwd(q, kv, ckv, seg, keep, dout, W, m, scale)
    assert_close("dq", dq, rdq, torch.bfloat16, v)
    assert np.all(to_np(dq)[~v] == 0)
    assert_close("dkv", dkv, rdkv, torch.bfloat16)
    assert_close("dckv", dckv, rdckv, torch.bfloat16)


@pytest.mark.parametrize("B,H,S,W,m,k", [
    (1, 64, 600, 64, 4, 16),      # H=64: two positions per tile, four per forward pair
    (2, 32, 333, 128, 4, 40),     # H=32: four positions per tile, ragged
    (1, 128, 400, 32, 8, 8),      # one position per tile
    (1, 64, 1100, 128, 4, 96),    # several compressed blocks per tile
])
def test_csa_matches_oracle(B, H, S, W, m, k):
    run_csa(B, H, S, W, m, k)


@pytest.fixture
def union_setting():
    yield lambda v: hca.hca_test_inject(hca.INJECT_CSA_UNION, v)
    hca.hca_test_inject(hca.INJECT_RESET)


@pytest.mark.parametrize("setting", [1, 64, 0])
def test_csa_union_kernels_agree(union_setting, setting):
    # the per-group union of selections comes from a bitonic sort (1) or from
    # byte masks over the group's entry range (64: 64-entry chunks, so a
    # group's range spans several); both against the oracle, and the
    # forward and dq (no atomics) bit-identical to the automatic choice
    B, H, S, W, m, k = 1, 64, 1100, 128, 4, 96
    seed = 11
    q, kv, ckv, _, dout = I.small(B, H, S, 128, W, m, dtype=torch.bfloat16, seed=seed)
    sel = I.random_selection(B, S, m, k, seed + 50).to(DEV)
    g = [x.to(DEV) for x in (q, kv, ckv, dout)]
    scale = 1 / math.sqrt(128)

    def call():
        o, l = hca.hca_csa_attn_fwd(g[0], g[1], g[2], None, sel, W, m, scale, check=True)
        d = hca.hca_csa_attn_bwd(g[0], g[1], g[2], None, sel, o, l, g[3], W, m, scale, check=True)
        return o, l, d[0]

    ref = call()
    union_setting(setting)
    got = call()
    for name, a, b in zip(("out", "lse", "dq"), got, ref):
        assert torch.equal(a, b), name
    run_csa(B, H, S, W, m, k, seed=seed)


def test_csa_union_chunks_with_documents(union_setting):
    union_setting(64)
    S = 700
    seg = torch.cat([I.segments_from_lengths([250, 300, 100], S, pad=50),
                     I.segments_from_lengths([699], S, pad=1)])
    run_csa(2, 64, S, 96, 4, 24, seg=seg)


def test_csa_documents_and_padding():
    S = 700
    seg = torch.cat([I.segments_from_lengths([250, 300, 100], S, pad=50),
                     I.segments_from_lengths([699], S, pad=1)])
    run_csa(2, 64, S, 96, 4, 24, seg=seg)


def test_csa_selecting_everything_is_hca():
    # every completed entry selected: CSA reduces to HCA (the oracle pins the
    # same reduction on the CPU)
    B, H, S, W, m = 1, 64, 300, 64, 4
    Sc = -(-S // m)
    sel = torch.arange(Sc, dtype=torch.int32).expand(B, S, Sc).contiguous()
    q, kv, ckv, _, dout = I.small(B, H, S, 128, W, m, dtype=torch.bfloat16, seed=3)
    g = [x.to(DEV) for x in (q, kv, ckv, dout)]
    scale = 1 / math.sqrt(128)
    o1, l1 = hca.hca_csa_attn_fwd(g[0], g[1], g[2], None, sel.to(DEV), W, m, scale, check=True)
    o2, l2 = hca.hca_attn_fwd(g[0], g[1], g[2], None, W, m, scale, check=True)
    assert_close("out", o1, to_np(o2), torch.bfloat16)
    assert_close("lse", l1, to_np(l2), torch.bfloat16)
    d1 = hca.hca_csa_attn_bwd(g[0], g[1], g[2], None, sel.to(DEV), o1, l1, g[3], W, m, scale, check=True)
    d2 = hca.hca_attn_bwd(g[0], g[1], g[2], None, o2, l2, g[3], W, m, scale, check=True)
    for name, a, b in zip(("dq", "dkv", "dckv"), d1, d2):
        assert_close(name, a, to_np(b), torch.bfloat16)


def test_csa_full_size_sampled_rows():
    # the CSA bench workload, B1 H64 S65536 D128 W128 m4 k256 with random
    # selections: out, lse and dq on sampled rows; exactly, the gradients of
    # the last 32 raw keys and the last 8 compressed entries (only the last 64
    # positions see them, and those positions are made to select the 8
    # entries); and, over every key, the sum identity (the gradients of all
    # keys add up to the sum of dO, since each row's softmax sums to one and
    # its dS sums to zero)
    B, H, S, D, W, m, k = 1, 64, 65536, 128, 128, 4, 256
    Sc = S // m
    scale = 1.0 / math.sqrt(D)
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, dtype=torch.bfloat16, seed=21, device=DEV)
    sel = I.random_selection(B, S, m, k, 71)
    sel[0, S - 64:, :8] = torch.arange(Sc - 8, Sc, dtype=torch.int32)
    out, lse = hca.hca_csa_attn_fwd(q, kv, ckv, None, sel.to(DEV), W, m, scale, check=True)
    dq, dkv, dckv = hca.hca_csa_attn_bwd(q, kv, ckv, None, sel.to(DEV), out, lse, dout, W, m, scale, check=True)
    torch.cuda.synchronize()
    keep = oracle.topk_mask(sel, Sc)
    qc, kvc, ckvc, dc = q.cpu(), kv.cpu(), ckv.cpu(), dout.cpu()
    out_c, lse_c, dq_c = to_np(out)[0], to_np(lse)[0], to_np(dq)[0]
    for lo in (0, 1022, 20000, 40962, S - 66):
        hi = lo + 2
        ro, rl = oracle.csa_fwd(qc, kvc, ckvc, None, keep, W, m, scale, rows=(lo, hi))
        assert_close(f"out [{lo},{hi})", out_c[:, lo:hi], ro[0][:, lo:hi], torch.bfloat16)
        assert_close(f"lse [{lo},{hi})", lse_c[:, lo:hi], rl[0][:, lo:hi], torch.bfloat16)
        rdq, _, _ = oracle.csa_bwd(qc, kvc, ckvc, None, keep, dc, W, m, scale, rows=(lo, hi))
        assert_close(f"dq [{lo},{hi})", dq_c[:, lo:hi], rdq[0][:, lo:hi], torch.bfloat16)
    _, rdkv, rdckv = oracle.csa_bwd(qc, kvc, ckvc, None, keep, dc, W, m, scale, rows=(S - 64, S))
    dkv_c, dckv_c = to_np(dkv)[0], to_np(dckv)[0]
    assert_close("dkv, last 32 keys", dkv_c[S - 32:], rdkv[0][S - 32:], torch.bfloat16)
    assert np.abs(rdckv[0][Sc - 8:]).max() > 0
    assert_close("dckv, last 8 entries", dckv_c[Sc - 8:], rdckv[0][Sc - 8:], torch.bfloat16)
    total = dkv_c.astype(np.float64).sum(0) + dckv_c.astype(np.float64).sum(0)
    assert_close("sum identity", total, to_np(dout[0].float().sum((0, 1))), torch.bfloat16)


def test_csa_fed_by_the_indexer():
    # the indexer's top-k selection drives the attention (the CSA chain)
    B, H, S, W, m, k = 1, 64, 512, 64, 4, 12
    q, kv, ckv, _, dout = I.small(B, H, S, 128, W, m, dtype=torch.bfloat16, seed=5)
    qi = I.normal((B, S, 4, 128), 60, torch.bfloat16)
    w = I.normal((B, S, 4), 61, torch.float32)
    sel, _ = hca.hca_indexer_topk(qi.to(DEV), ckv.to(DEV), w.to(DEV), None, m, k, check=True)
    run_csa(B, H, S, W, m, k, seed=5, sel=sel.cpu())


def test_csa_unsupported_shapes():
    q, kv, ckv, _, _ = I.small(1, 16, 64, 128, 16, 4, dtype=torch.bfloat16)
    sel = I.random_selection(1, 64, 4, 4, 1)
    with pytest.raises(hca.HCAError) as e:
        hca.hca_csa_attn_fwd(q.to(DEV), kv.to(DEV), ckv.to(DEV), None, sel.to(DEV), 16, 4, 0.1)
    assert e.value.status == 8   # H = 16: more than four positions per tile
