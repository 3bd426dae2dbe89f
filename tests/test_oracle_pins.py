"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test fixes the oracle to something independent of its own code: a
hand-derived table, a closed form derived from the definition, a library
routine on a special case (PyTorch's scaled-dot-product attention and
autograd), central finite differences, or an invariant of softmax attention.
They run on the CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_compressed_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# closed form of the visible-pair count
# --------------------------------------------------------------------------

def closed_form_pairs(seg_row, W, m):
    """Per-head visible pairs of one batch row from the segment layout.

    Derivation (own, from the definition): a document of length L sees
    sum_{x<L} min(x+1, W) raw pairs = L(L+1)/2 if L <= W else W*L - W(W-1)/2.
    Compressed windows start at multiples of m; the first one inside the
    document starts at c0 = m*ceil(a/m).  The query c0+x (x = 0..N-1, with
    N = a+L-c0) sees floor((x+1)/m) completed windows, so the total is
    sum_{y=1..N} floor(y/m) = m*q(q-1)/2 + q(r+1) for N = q*m + r.
    """
    seg_row = np.asarray(seg_row)
    S = len(seg_row)
    raw = comp = 0
    i = 0
    while i < S:
        j = i
        while j < S and seg_row[j] == seg_row[i]:
            j += 1
        if seg_row[i] >= 0:
            a, L = i, j - i
            raw += L * (L + 1) // 2 if L <= W else W * L - W * (W - 1) // 2
            c0 = m * (-(-a // m))
            N = max(0, a + L - c0)
            q, r = divmod(N, m)
            comp += m * q * (q - 1) // 2 + q * (r + 1)
        i = j
    return raw, comp


def test_closed_form_matches_enumeration_random_layouts():
    rng = np.random.Generator(np.random.PCG64(7))
    for _ in range(300):
        S = int(rng.integers(1, 90))
        W = int(rng.integers(1, 40))
        m = int(rng.integers(1, 20))
        seg = I.random_layout(S, rng)[None, :]
        raw, comp = oracle.visible_pairs(seg, 1, S, W, m)
        cr, cc = closed_form_pairs(seg[0], W, m)
        assert (raw[0], comp[0]) == (cr, cc), (S, W, m, seg)


@pytest.mark.parametrize("w", [I.TINY_F32, I.FWD_S4096_2DOC, I.UNALIGNED, I.LONG_S65536])
def test_closed_form_matches_enumeration_workloads(w):
    seg = I.segments(w)
    raw, comp = oracle.visible_pairs(seg, w.B, w.S, w.W, w.m)
    seg_np = np.zeros((w.B, w.S), np.int32) if seg is None else seg.numpy()
    for b in range(w.B):
        assert (raw[b], comp[b]) == closed_form_pairs(seg_np[b], w.W, w.m)


def test_closed_form_workload_totals():
    # pairs x heads of the benchmark workloads, from the closed form alone
    def total(w):
        seg = I.segments(w)
        seg_np = np.zeros((w.B, w.S), np.int32) if seg is None else seg.numpy()
        return sum(sum(closed_form_pairs(seg_np[b], w.W, w.m)) for b in range(w.B)) * w.H
    assert total(I.TINY_F32) == 154880
    assert total(I.FWD_S4096_2DOC) == 8620544
    assert total(I.UNALIGNED) == 703393024
    assert total(I.LONG_S65536) == 1608028160
    assert total(I.LONG_S131072) == 5364060160


# --------------------------------------------------------------------------
# hand-derived golden table
# --------------------------------------------------------------------------

def _read_golden(name):
    g = {"q": {}, "tile": {}}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, rest = line.split(None, 1)
            if key in ("S", "W", "m"):
                g[key] = int(rest)
            elif key == "seg":
                g["seg"] = [int(x) for x in rest.split()]
            elif key == "pairs":
                g["pairs"] = tuple(int(x) for x in rest.split())
            elif key == "q":
                idx, body = rest.split(":")
                raw, comp = body.split("|")
                g["q"][int(idx)] = ([int(x) for x in raw.split()], [int(x) for x in comp.split()])
            elif key == "tile":
                idx, body = rest.split(":")
                g["tile"][int(idx)] = [int(x) for x in body.split()]
    return g


def test_golden_visibility_table():
    g = _read_golden("visibility_S10_W3_m2.txt")
    S, W, m = g["S"], g["W"], g["m"]
    Sc = -(-S // m)
    seg = np.array([g["seg"]], dtype=np.int32)
    # one-hot keys and zero queries: every visible key gets weight 1/n, so the
    # support of out[i] is exactly the visible set of query i
    D = S + Sc
    kv = np.eye(D)[None, :S, :]
    ckv = np.eye(D)[None, S:, :]
    q = np.zeros((1, 1, S, D))
    out, lse = oracle.fwd(q, kv, ckv, seg, W, m, 1.0)
    for i in range(S):
        raw, comp = g["q"][i]
        n = len(raw) + len(comp)
        expect = np.zeros(D)
        for t in raw:
            expect[t] = 1.0 / n
        for j in comp:
            expect[S + j] = 1.0 / n
        if n == 0:
            assert lse[0, 0, i] == -np.inf
            assert np.all(out[0, 0, i] == 0)
        else:
            np.testing.assert_allclose(out[0, 0, i], expect, atol=1e-15)
            assert abs(lse[0, 0, i] - math.log(n)) < 1e-14
    raw, comp = oracle.visible_pairs(seg, 1, S, W, m)
    assert (raw[0], comp[0]) == g["pairs"]
    assert closed_form_pairs(seg[0], W, m) == g["pairs"]
    tiles = oracle.tile_ranges(seg, 1, S, W, m, 2)
    for k, e in g["tile"].items():
        assert list(tiles[0, k]) == e, (k, tiles[0, k], e)


# --------------------------------------------------------------------------
# special case: plain causal attention (library routine)
# --------------------------------------------------------------------------

def _torch_reference(q, kv, ckv, mask_raw, mask_comp, scale, dout):
    """Dense MQA attention over [kv ; ckv] with a boolean mask, through
    PyTorch's scaled_dot_product_attention and autograd (fp64, CPU)."""
    q = q.clone().requires_grad_(True)
    kv = kv.clone().requires_grad_(True)
    ckv = ckv.clone().requires_grad_(True)
    keys = torch.cat([kv, ckv], dim=1)[:, None]               # [B,1,S+Sc,D]
    mask = torch.cat([mask_raw, mask_comp], dim=-1)[:, None]   # [B,1,S,S+Sc]
    H = q.shape[1]
    k = keys.expand(-1, H, -1, -1)
    out = torch.nn.functional.scaled_dot_product_attention(q, k, k, attn_mask=mask, scale=scale)
    logits = (q @ k.transpose(-1, -2)) * scale
    lse = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)
    out.backward(dout)
    return out.detach(), lse.detach(), q.grad, kv.grad, ckv.grad


def test_causal_special_case_matches_sdpa():
    B, H, S, D = 2, 3, 37, 8
    W, m = S, S + 1            # window covers everything, no window completes
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m)
    scale = 0.37
    causal = torch.ones(S, S, dtype=torch.bool).tril()[None].expand(B, -1, -1)
    comp = torch.zeros(B, S, ckv.shape[1], dtype=torch.bool)
    ro, rl, rdq, rdkv, rdckv = _torch_reference(q, kv, ckv, causal, comp, scale, dout)
    out, lse = oracle.fwd(q, kv, ckv, None, W, m, scale)
    np.testing.assert_allclose(out, ro.numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, rl.numpy(), atol=1e-12)
    # plain is_causal path of the library as a second reading of the same case
    k = kv[:, None].expand(-1, H, -1, -1)
    o2 = torch.nn.functional.scaled_dot_product_attention(q, k, k, is_causal=True, scale=scale)
    np.testing.assert_allclose(out, o2.numpy(), atol=1e-12)
    dq, dkv, dckv = oracle.bwd(q, kv, ckv, None, dout, W, m, scale)
    np.testing.assert_allclose(dq, rdq.numpy(), atol=1e-11)
    np.testing.assert_allclose(dkv, rdkv.numpy(), atol=1e-11)
    np.testing.assert_allclose(dckv, 0.0, atol=0)


def _interval_masks(seg, S, W, m):
    """Dense masks from the interval reading (contiguous documents):
    raw t in [max(i-W+1, start_i), i], compressed j in [ceil(start_i/m),
    floor((i+1)/m)-1].  Written independently of the oracle's predicate."""
    B = seg.shape[0]
    Sc = -(-S // m)
    mr = torch.zeros(B, S, S, dtype=torch.bool)
    mc = torch.zeros(B, S, Sc, dtype=torch.bool)
    for b in range(B):
        start = 0
        for i in range(S):
            if i > 0 and seg[b, i] != seg[b, i - 1]:
                start = i
            if seg[b, i] < 0:
                continue
            mr[b, i, max(i - W + 1, start): i + 1] = True
            lo, hi = -(-start // m), (i + 1) // m - 1
            if hi >= lo:
                mc[b, i, lo: hi + 1] = True
    return mr, mc


@pytest.mark.parametrize("S,W,m,H,D", [(23, 4, 3, 2, 5), (40, 7, 5, 3, 4), (31, 1, 1, 1, 6), (29, 40, 2, 2, 3)])
def test_masked_case_matches_sdpa_autograd(S, W, m, H, D):
    rng = np.random.Generator(np.random.PCG64(S * 100 + W))
    B = 2
    seg = np.stack([I.random_layout(S, rng), I.random_layout(S, rng)])
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, seed=S + W)
    scale = 1.0 / math.sqrt(D)
    mr, mc = _interval_masks(seg, S, W, m)
    valid = torch.from_numpy(seg >= 0)
    # padded query rows have an empty mask: give them a dummy key so SDPA
    # stays finite, then ignore them (their dO is zeroed)
    mr_safe = mr.clone()
    for b in range(B):
        for i in range(S):
            if not valid[b, i]:
                mr_safe[b, i, i] = True
    d_eff = dout * valid[:, None, :, None]
    ro, rl, rdq, rdkv, rdckv = _torch_reference(q, kv, ckv, mr_safe, mc, scale, d_eff)
    out, lse = oracle.fwd(q, kv, ckv, seg, W, m, scale)
    v = valid[:, None, :].expand(-1, H, -1).numpy()
    np.testing.assert_allclose(out[v], ro.numpy()[v], atol=1e-12)
    np.testing.assert_allclose(lse[v], rl.numpy()[v], atol=1e-12)
    assert np.all(out[~v] == 0) and np.all(lse[~v] == -np.inf)
    dq, dkv, dckv = oracle.bwd(q, kv, ckv, seg, dout, W, m, scale)
    np.testing.assert_allclose(dq[v], rdq.numpy()[v], atol=1e-11)
    assert np.all(dq[~v] == 0)
    np.testing.assert_allclose(dkv, rdkv.numpy(), atol=1e-11)
    np.testing.assert_allclose(dckv, rdckv.numpy(), atol=1e-11)


# --------------------------------------------------------------------------
# gradients: central finite differences
# --------------------------------------------------------------------------

def test_gradients_match_finite_differences():
    B, H, S, D, W, m = 1, 2, 11, 3, 4, 2
    seg = np.array([[0, 0, 0, 0, 0, 1, 1, 1, 1, 1, -1]], dtype=np.int32)
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, seed=99)
    q, kv, ckv, dout = (x.numpy() for x in (q, kv, ckv, dout))
    scale = 0.61

    def loss(qq, kk, cc):
        out, _ = oracle.fwd(qq, kk, cc, seg, W, m, scale)
        return float(np.sum(out * dout))

    dq, dkv, dckv = oracle.bwd(q, kv, ckv, seg, dout, W, m, scale)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("kv", kv, dkv), ("ckv", ckv, dckv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args = {"q": (q, kv, ckv), "kv": (q, kv, ckv), "ckv": (q, kv, ckv)}[name]
            args_p = [a if nm != name else xp for a, nm in zip(args, ("q", "kv", "ckv"))]
            args_m = [a if nm != name else xm for a, nm in zip(args, ("q", "kv", "ckv"))]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(g, num, atol=2e-8, err_msg=name)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_identical_rows_give_that_row():
    B, H, S, D, W, m = 2, 3, 30, 6, 5, 4
    rng = np.random.Generator(np.random.PCG64(3))
    seg = np.stack([I.random_layout(S, rng), I.random_layout(S, rng)])
    q, _, _, _, dout = I.small(B, H, S, D, W, m, seed=5)
    r = torch.randn(D, dtype=torch.float64, generator=torch.Generator().manual_seed(11))
    Sc = -(-S // m)
    kv = r.expand(B, S, D).contiguous()
    ckv = r.expand(B, Sc, D).contiguous()
    out, _ = oracle.fwd(q, kv, ckv, seg, W, m, 0.4)
    valid = seg >= 0
    for b in range(B):
        for i in range(S):
            if valid[b, i]:
                np.testing.assert_allclose(out[b, :, i], np.broadcast_to(r.numpy(), (H, D)), atol=1e-13)
    dq, dkv, dckv = oracle.bwd(q, kv, ckv, seg, dout, W, m, 0.4)
    np.testing.assert_allclose(dq, 0.0, atol=1e-12)
    for b in range(B):
        total = dkv[b].sum(0) + dckv[b].sum(0)
        expect = (dout.numpy()[b] * valid[b][None, :, None]).sum((0, 1))
        np.testing.assert_allclose(total, expect, atol=1e-11)


def test_gradient_sum_identity_general_inputs():
    # sum over all keys of d r_k = sum over valid (h,i) of dO: the dS terms
    # cancel because sum_k dS_k = Delta - Delta = 0 and sum_k P_k = 1.
    B, H, S, D, W, m = 2, 4, 45, 5, 6, 4
    rng = np.random.Generator(np.random.PCG64(21))
    seg = np.stack([I.random_layout(S, rng), I.random_layout(S, rng)])
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, seed=8)
    dq, dkv, dckv = oracle.bwd(q, kv, ckv, seg, dout, W, m, 0.45)
    valid = seg >= 0
    for b in range(B):
        np.testing.assert_allclose(dkv[b].sum(0) + dckv[b].sum(0),
                                   (dout.numpy()[b] * valid[b][None, :, None]).sum((0, 1)), atol=1e-11)


def test_zero_queries_average_visible_keys():
    # q = 0: every visible logit is 0, so lse = log(n_i) and out = mean of the
    # visible key rows; n_i summed over the row equals the closed form.
    B, H, S, D, W, m = 1, 1, 64, 4, 9, 5
    rng = np.random.Generator(np.random.PCG64(4))
    seg = I.random_layout(S, rng)[None]
    _, kv, ckv, _, _ = I.small(B, H, S, D, W, m, seed=1)
    q = np.zeros((B, H, S, D))
    out, lse = oracle.fwd(q, kv, ckv, seg, W, m, 1.0)
    n = np.where(np.isfinite(lse[0, 0]), np.exp(lse[0, 0]), 0.0)
    assert abs(n.sum() - sum(closed_form_pairs(seg[0], W, m))) < 1e-6


def test_softmax_weights_sum_to_one():
    B, H, S, D, W, m = 1, 2, 40, 6, 7, 3
    rng = np.random.Generator(np.random.PCG64(9))
    seg = I.random_layout(S, rng)[None]
    q, kv, ckv, _, _ = I.small(B, H, S, D, W, m, seed=2)
    kv = kv.clone(); ckv = ckv.clone()
    kv[..., 2] = 1.0
    ckv[..., 2] = 1.0
    out, _ = oracle.fwd(q, kv, ckv, seg, W, m, 0.5)
    valid = (seg[0] >= 0)
    np.testing.assert_allclose(out[0, :, valid, 2], 1.0, atol=1e-13)


def test_packing_invariance_on_window_boundaries():
    # documents starting on a multiple of m: packed == each alone
    H, D, W, m = 2, 4, 5, 4
    lens = [12, 20]
    S = sum(lens)
    seg = I.segments_from_lengths(lens, S).numpy()
    q, kv, ckv, _, dout = I.small(1, H, S, D, W, m, seed=12)
    out, lse = oracle.fwd(q, kv, ckv, seg, W, m, 0.5)
    dq, dkv, dckv = oracle.bwd(q, kv, ckv, seg, dout, W, m, 0.5)
    a = 0
    for L in lens:
        sl = slice(a, a + L)
        csl = slice(a // m, (a + L) // m)
        q1, kv1, ckv1, d1 = q[:, :, sl], kv[:, sl], ckv[:, csl], dout[:, :, sl]
        o1, l1 = oracle.fwd(q1, kv1, ckv1, None, W, m, 0.5)
        g1 = oracle.bwd(q1, kv1, ckv1, None, d1, W, m, 0.5)
        np.testing.assert_allclose(out[:, :, sl], o1, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, sl], l1, atol=1e-13)
        np.testing.assert_allclose(dq[:, :, sl], g1[0], atol=1e-12)
        np.testing.assert_allclose(dkv[:, sl], g1[1], atol=1e-12)
        np.testing.assert_allclose(dckv[:, csl], g1[2], atol=1e-12)
        a += L


def test_packing_off_boundary_start_differs():
    # a document starting off a multiple of m loses the window straddling its
    # start, so it differs from the same document run alone (absolute windows)
    H, D, W, m = 1, 4, 5, 4
    lens = [6, 14]
    S = sum(lens)
    seg = I.segments_from_lengths(lens, S).numpy()
    raw, comp = oracle.visible_pairs(seg, 1, S, W, m)
    alone_raw, alone_comp = oracle.visible_pairs(None, 1, 14, W, m)
    first_raw, first_comp = oracle.visible_pairs(None, 1, 6, W, m)
    assert raw[0] == alone_raw[0] + first_raw[0]
    assert comp[0] < alone_comp[0] + first_comp[0]


def test_head_permutation_equivariance():
    B, H, S, D, W, m = 1, 4, 26, 5, 6, 3
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, seed=31)
    perm = torch.tensor([2, 0, 3, 1])
    o, l = oracle.fwd(q, kv, ckv, None, W, m, 0.5)
    op, lp = oracle.fwd(q[:, perm], kv, ckv, None, W, m, 0.5)
    np.testing.assert_array_equal(op, o[:, perm.numpy()])
    np.testing.assert_array_equal(lp, l[:, perm.numpy()])


# --------------------------------------------------------------------------
# consistency of the sampling entry points used at large sizes
# --------------------------------------------------------------------------

def test_row_ranges_and_key_lists_agree_with_full():
    B, H, S, D, W, m = 2, 3, 50, 4, 6, 5
    rng = np.random.Generator(np.random.PCG64(17))
    seg = np.stack([I.random_layout(S, rng), I.random_layout(S, rng)])
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, seed=40)
    out, lse = oracle.fwd(q, kv, ckv, seg, W, m, 0.3)
    o2, l2 = oracle.fwd(q, kv, ckv, seg, W, m, 0.3, rows=(13, 29))
    np.testing.assert_array_equal(o2[:, :, 13:29], out[:, :, 13:29])
    np.testing.assert_array_equal(l2[:, :, 13:29], lse[:, :, 13:29])
    dq, dkv, dckv = oracle.bwd(q, kv, ckv, seg, dout, W, m, 0.3)
    a = oracle.bwd(q, kv, ckv, seg, dout, W, m, 0.3, rows=(0, 21))
    b = oracle.bwd(q, kv, ckv, seg, dout, W, m, 0.3, rows=(21, S))
    np.testing.assert_allclose(a[1] + b[1], dkv, atol=1e-12)
    np.testing.assert_allclose(a[2] + b[2], dckv, atol=1e-12)
    np.testing.assert_array_equal(a[0][:, :, :21], dq[:, :, :21])
    Sc = -(-S // m)
    raw_ids = [0, 7, S + 3, 2 * S - 1]
    comp_ids = [0, 4, Sc + 2, 2 * Sc - 1]
    draw, dcomp = oracle.bwd_keys(q, kv, ckv, seg, dout, W, m, 0.3, raw_ids, comp_ids)
    np.testing.assert_allclose(draw, dkv.reshape(-1, D)[raw_ids], atol=1e-13)
    np.testing.assert_allclose(dcomp, dckv.reshape(-1, D)[comp_ids], atol=1e-13)


def test_bf16_inputs_are_widened_exactly():
    B, H, S, D, W, m = 1, 2, 20, 8, 5, 3
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, dtype=torch.bfloat16, seed=3)
    o1, l1 = oracle.fwd(q, kv, ckv, None, W, m, 0.35)
    o2, l2 = oracle.fwd(q.double(), kv.double(), ckv.double(), None, W, m, 0.35)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
