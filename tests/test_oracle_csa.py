"""Pins of the oracle's compressed sparse attention (CSA) mode.

CSA keeps HCA's raw window and its completed, same-document compressed
entries, but a compressed entry counts for a query only when the indexer's
selection keeps that (query, entry) pair ("Add HCA Static Compilation for
Splash Attention [Deepseek v4]", Description: CSA has compression ratio 4 and
a top-k step; the selection is an input here).  The masks below are built in
Python from that definition, independently of the oracle's predicate, and the
attention itself comes from PyTorch's scaled-dot-product attention with
autograd.  CPU only.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_compressed_gb300 import inputs as I
from test_oracle_pins import _interval_masks, _torch_reference


def _random_sel(rng, B, S, Sc, density):
    return (rng.random((B, S, Sc)) < density).astype(np.uint8)


def _check_against_sdpa(B, H, S, D, W, m, seg, sel, seed):
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, seed=seed)
    scale = 1.0 / math.sqrt(D)
    mr, mc = _interval_masks(seg, S, W, m)
    mc = mc & torch.from_numpy(sel.astype(bool))
    valid = torch.from_numpy(seg >= 0)
    mr_safe = mr.clone()
    for b in range(B):
        for i in range(S):
            if not valid[b, i]:
                mr_safe[b, i, i] = True
    d_eff = dout * valid[:, None, :, None]
    ro, rl, rdq, rdkv, rdckv = _torch_reference(q, kv, ckv, mr_safe, mc, scale, d_eff)
    out, lse = oracle.csa_fwd(q, kv, ckv, seg, sel, W, m, scale)
    v = valid[:, None, :].expand(-1, H, -1).numpy()
    np.testing.assert_allclose(out[v], ro.numpy()[v], atol=1e-12)
    np.testing.assert_allclose(lse[v], rl.numpy()[v], atol=1e-12)
    assert np.all(out[~v] == 0) and np.all(lse[~v] == -np.inf)
    dq, dkv, dckv = oracle.csa_bwd(q, kv, ckv, seg, sel, dout, W, m, scale)
    np.testing.assert_allclose(dq[v], rdq.numpy()[v], atol=1e-11)
    assert np.all(dq[~v] == 0)
    np.testing.assert_allclose(dkv, rdkv.numpy(), atol=1e-11)
    np.testing.assert_allclose(dckv, rdckv.numpy(), atol=1e-11)
    raw, comp = oracle.csa_visible_pairs(seg, sel, B, S, W, m)
    np.testing.assert_array_equal(raw, mr.sum(dim=(1, 2)).numpy())
    np.testing.assert_array_equal(comp, mc.sum(dim=(1, 2)).numpy())


@pytest.mark.parametrize("S,W,m,H,D,density", [(29, 5, 4, 2, 5, 0.5), (40, 8, 4, 3, 4, 0.2), (33, 3, 2, 1, 6, 0.8),
                                               (26, 30, 1, 2, 3, 0.5)])
def test_csa_matches_sdpa_autograd(S, W, m, H, D, density):
    rng = np.random.Generator(np.random.PCG64(S * 31 + W))
    B = 2
    seg = np.stack([I.random_layout(S, rng), I.random_layout(S, rng)])
    sel = _random_sel(rng, B, S, -(-S // m), density)
    _check_against_sdpa(B, H, S, D, W, m, seg, sel, seed=S + m)


def test_csa_selecting_nothing_is_the_sliding_window():
    # no compressed entry survives: the raw window alone, and dckv is exactly 0
    B, H, S, D, W, m = 1, 2, 30, 4, 6, 4
    seg = np.zeros((B, S), dtype=np.int32)
    sel = np.zeros((B, S, -(-S // m)), dtype=np.uint8)
    _check_against_sdpa(B, H, S, D, W, m, seg, sel, seed=3)
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, seed=3)
    _, _, dckv = oracle.csa_bwd(q, kv, ckv, seg, sel, dout, W, m, 0.5)
    assert np.all(dckv == 0)


def test_csa_selecting_everything_is_hca():
    B, H, S, D, W, m = 2, 2, 37, 4, 5, 4
    rng = np.random.Generator(np.random.PCG64(11))
    seg = np.stack([I.random_layout(S, rng), I.random_layout(S, rng)])
    sel = np.ones((B, S, -(-S // m)), dtype=np.uint8)
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, seed=5)
    a = oracle.csa_fwd(q, kv, ckv, seg, sel, W, m, 0.4)
    b = oracle.fwd(q, kv, ckv, seg, W, m, 0.4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    a = oracle.csa_bwd(q, kv, ckv, seg, sel, dout, W, m, 0.4)
    b = oracle.bwd(q, kv, ckv, seg, dout, W, m, 0.4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_topk_lists_order_duplicates_and_padding():
    # the selection is a set: list order, repeats and -1 / out-of-range
    # padding do not change it
    rng = np.random.Generator(np.random.PCG64(2))
    B, S, Sc, k = 2, 17, 5, 3
    base = np.stack([[rng.choice(Sc, size=k, replace=False) for _ in range(S)] for _ in range(B)])
    shuffled = base[..., ::-1].copy()
    padded = np.concatenate([base, base[..., :1], np.full((B, S, 2), -1), np.full((B, S, 1), Sc)], axis=-1)
    a = oracle.topk_mask(base, Sc)
    np.testing.assert_array_equal(a, oracle.topk_mask(shuffled, Sc))
    np.testing.assert_array_equal(a, oracle.topk_mask(padded, Sc))
    assert np.all(a.sum(-1) == k)
