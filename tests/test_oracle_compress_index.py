"""CPU pins of the compressor and Lightning Indexer oracle
(oracle/compress_index.py) against closed forms, library routines and
invariants, chosen so that a dropped term, a wrong sign or a transposed
operand fails one of them."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import compress_index as CI


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# --------------------------------------------------------------------------
# compressor
# --------------------------------------------------------------------------

def test_zero_gates_and_bias_give_mean_pooling():
    r = _rng(1)
    B, S, D, m = 2, 23, 5, 4
    x = r.standard_normal((B, S, D))
    ckv = CI.compress_fwd(x, np.zeros((B, S)), np.zeros(m), None, m)
    for j in range(-(-S // m)):
        np.testing.assert_allclose(ckv[:, j], x[:, j * m:min(S, (j + 1) * m)].mean(1), rtol=1e-13, atol=1e-14)


def test_bias_only_two_position_window_by_hand():
    # m = 2, bias = (0, ln 3): weights 1/4 and 3/4 in every window
    x = np.array([[[1.0, 2.0], [5.0, -1.0], [0.5, 0.5], [3.0, 7.0]]])
    ckv = CI.compress_fwd(x, np.zeros((1, 4)), np.array([0.0, math.log(3.0)]), None, 2)
    np.testing.assert_allclose(ckv[0, 0], [0.25 * 1 + 0.75 * 5, 0.25 * 2 - 0.75 * 1], rtol=1e-14)
    np.testing.assert_allclose(ckv[0, 1], [0.25 * 0.5 + 0.75 * 3, 0.25 * 0.5 + 0.75 * 7], rtol=1e-14)


def test_dominant_gate_selects_its_row_and_constant_rows_pass_through():
    r = _rng(2)
    B, S, D, m = 1, 16, 3, 8
    x = r.standard_normal((B, S, D))
    g = np.zeros((B, S))
    g[0, 5] = 80.0
    g[0, 8 + 7] = 80.0
    ckv = CI.compress_fwd(x, g, r.standard_normal(m), None, m)
    np.testing.assert_allclose(ckv[0, 0], x[0, 5], rtol=1e-12)
    np.testing.assert_allclose(ckv[0, 1], x[0, 15], rtol=1e-12)
    xc = np.broadcast_to(np.array([1.5, -2.0, 0.25]), (B, S, D))
    np.testing.assert_allclose(CI.compress_fwd(xc, r.standard_normal((B, S)), r.standard_normal(m), None, m)[0],
                               np.broadcast_to([1.5, -2.0, 0.25], (2, 3)), rtol=1e-13)


def test_padding_is_left_out_and_an_all_padding_window_is_zero():
    r = _rng(3)
    B, S, D, m = 1, 12, 4, 4
    x = r.standard_normal((B, S, D))
    seg = np.zeros((B, S), np.int32)
    seg[0, 6:] = -1
    ckv = CI.compress_fwd(x, np.zeros((B, S)), np.zeros(m), seg, m)
    np.testing.assert_allclose(ckv[0, 1], x[0, 4:6].mean(0), rtol=1e-13)
    assert np.all(ckv[0, 2] == 0)


def test_compressor_backward_matches_finite_differences():
    r = _rng(4)
    B, S, D, m = 2, 11, 3, 4
    x = r.standard_normal((B, S, D))
    g = r.standard_normal((B, S))
    bias = r.standard_normal(m)
    seg = np.zeros((B, S), np.int32)
    seg[1, 9:] = -1
    dck = r.standard_normal((B, -(-S // m), D))
    dx, dg, db = CI.compress_bwd(x, g, bias, seg, m, dck)

    def loss(x_, g_, b_):
        return float((CI.compress_fwd(x_, g_, b_, seg, m) * dck).sum())

    h = 1e-6
    for arr, grad in ((x, dx), (g, dg), (bias, db)):
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            k = it.multi_index
            ap, am = arr.copy(), arr.copy()
            ap[k] += h
            am[k] -= h
            args_p = [ap if arr is a else a for a in (x, g, bias)]
            args_m = [am if arr is a else a for a in (x, g, bias)]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[k]) < 1e-6, (k, fd, grad[k])
    # adding a constant to every logit of a window changes nothing
    assert abs(db.sum() - dg.sum()) < 1e-12 and abs(dg.sum()) < 1e-10


# --------------------------------------------------------------------------
# Lightning Indexer
# --------------------------------------------------------------------------

def _idx_inputs(B, S, Hi, Di, m, seed):
    r = _rng(seed)
    Sc = -(-S // m)
    return (r.standard_normal((B, S, Hi, Di)), r.standard_normal((B, Sc, Di)), r.standard_normal((B, S, Hi)))


def test_one_head_unit_weight_is_a_masked_matmul():
    B, S, Di, m = 2, 40, 8, 4
    qi, ki, _ = _idx_inputs(B, S, 1, Di, m, 5)
    w = np.ones((B, S, 1))
    sc = CI.index_scores(qi, ki, w, None, m)
    ref = torch.matmul(torch.from_numpy(qi[:, :, 0]), torch.from_numpy(ki).transpose(1, 2)).numpy()
    for i in range(S):
        for j in range(ki.shape[1]):
            if (j + 1) * m <= i + 1:
                assert abs(sc[0, i, j] - ref[0, i, j]) < 1e-12 and abs(sc[1, i, j] - ref[1, i, j]) < 1e-12
            else:
                assert sc[0, i, j] == -np.inf


def test_head_weights_and_relu():
    B, S, Hi, Di, m = 1, 24, 3, 6, 4
    qi, ki, _ = _idx_inputs(B, S, Hi, Di, m, 6)
    onehot = np.zeros((B, S, Hi))
    onehot[..., 2] = 1.0
    sc = CI.index_scores(qi, ki, onehot, None, m)
    sc2 = CI.index_scores(qi[:, :, 2:3], ki, np.ones((B, S, 1)), None, m)
    np.testing.assert_array_equal(sc, sc2)
    # with every per-head score positive the ReLU changes nothing; with
    # opposite signs it removes the negative heads
    qp, kp = np.abs(qi), np.abs(ki)
    w = np.abs(_idx_inputs(B, S, Hi, Di, m, 7)[2])
    np.testing.assert_allclose(CI.index_scores(qp, kp, w, None, m, relu=True), CI.index_scores(qp, kp, w, None, m))
    qn = qp.copy()
    qn[:, :, 1] *= -1
    a = CI.index_scores(qn, kp, w, None, m, relu=True)
    b = CI.index_scores(qn[:, :, [0, 2]], kp, w[:, :, [0, 2]], None, m)
    np.testing.assert_allclose(a, b, rtol=1e-13)


def test_visibility_count_matches_the_attention_oracle():
    r = _rng(8)
    from block_sparse_compressed_gb300 import inputs as I
    for _ in range(6):
        S = int(r.integers(20, 150))
        m = int(r.integers(1, 9))
        seg = np.stack([I.random_layout(S, r), I.random_layout(S, r)])
        vis = CI.comp_visible(seg, 2, S, m)
        _, comp = oracle.visible_pairs(seg, 2, S, 4, m)
        assert vis.sum(axis=(1, 2)).tolist() == comp.tolist()


def test_topk_matches_torch_topk_on_distinct_scores():
    r = _rng(9)
    B, S, Sc, k = 2, 30, 17, 5
    sc = r.standard_normal((B, S, Sc))
    sc[:, :3, 10:] = -np.inf      # some rows see few entries
    sel = CI.topk_select(sc, k)
    for b in range(B):
        for s in range(S):
            n = int(np.isfinite(sc[b, s]).sum())
            kk = min(k, n)
            ref = torch.topk(torch.from_numpy(sc[b, s]), kk).indices.sort().values.tolist()
            assert sel[b, s, :kk].tolist() == ref
            assert np.all(sel[b, s, kk:] == -1)


def test_topk_ties_go_to_the_smaller_index():
    sc = np.array([[[1.0, 2.0, 2.0, 2.0, 0.0, -np.inf]]])
    assert CI.topk_select(sc, 2)[0, 0].tolist() == [1, 2]
    assert CI.topk_select(sc, 4)[0, 0].tolist() == [0, 1, 2, 3]
    assert CI.topk_select(sc, 7)[0, 0].tolist() == [0, 1, 2, 3, 4, -1, -1]


def test_selection_respects_documents_and_completion():
    B, S, Hi, Di, m, k = 1, 64, 2, 4, 4, 8
    qi, ki, w = _idx_inputs(B, S, Hi, Di, m, 10)
    seg = np.zeros((B, S), np.int32)
    seg[0, 30:] = 1          # second document starts mid-window (window 7 = 28..31 spans both)
    sel, sc = CI.indexer_topk(qi, ki, w, seg, m, k)
    for i in range(S):
        for j in sel[0, i]:
            if j < 0:
                continue
            assert (j + 1) * m <= i + 1
            assert np.all(seg[0, j * m:(j + 1) * m] == seg[0, i])
    # queries of the second document see nothing before window 8
    assert np.all(sel[0, 30:35] == -1)
