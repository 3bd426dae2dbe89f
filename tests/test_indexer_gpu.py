"""GPU parity of the Lightning Indexer (hca_indexer_topk, through the C ABI
binding) against the fp64 oracle in oracle/compress_index.py.

- scores: fp32 GPU scores against the fp64 definition over the visible
  entries, bf16 bound max|err| <= 1e-2*max|ref| + 1e-3; the sentinel (-inf)
  exactly where an entry is not visible;
- selection, bit-exact where the precision is the same: the GPU selection
  equals the oracle's top-k rule applied to the GPU's own fp32 scores (the
  decision taken in the kernel's precision);
- selection against the fp64 scores: any entry that differs from the
  oracle's selection is a near tie, within the score tolerance of the
  oracle's k-th score."""
import numpy as np
import pytest
import torch

from oracle import compress_index as CI
from block_sparse_compressed_gb300 import hca
from block_sparse_compressed_gb300 import inputs as I
from _util import bound

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(B, S, Hi, m, seed):
    Sc = -(-S // m)
    qi = I.normal((B, S, Hi, 128), seed, torch.bfloat16)
    ki = I.normal((B, Sc, 128), seed + 1, torch.bfloat16)
    w = I.normal((B, S, Hi), seed + 2, torch.float32)
    return qi, ki, w


def _check_rows(sel, got_sc, ref_sc, k):
    """sel [R,k], got_sc/ref_sc [R,Sc] for the same query rows."""
    finite = np.isfinite(ref_sc)
    assert np.array_equal(np.isfinite(got_sc), finite), "sentinel placement differs"
    tol = bound(ref_sc[finite], torch.bfloat16)
    err = float(np.max(np.abs(got_sc[finite] - ref_sc[finite]))) if finite.any() else 0.0
    assert err <= tol, f"scores: max|err| {err:.3e} > {tol:.3e}"
    # the kernel's decision in its own precision: exactly the top-k rule
    own = CI.topk_select(got_sc[None], k)[0]
    np.testing.assert_array_equal(sel, own)
    # against the fp64 scores: differences are near ties only
    ref_sel = CI.topk_select(ref_sc[None], k)[0]
    for r in range(sel.shape[0]):
        a = set(sel[r][sel[r] >= 0].tolist())
        b = set(ref_sel[r][ref_sel[r] >= 0].tolist())
        assert len(a) == len(b)
        if a == b:
            continue
        kth = np.sort(ref_sc[r][finite[r]])[::-1][len(b) - 1]
        for j in a ^ b:
            assert abs(ref_sc[r, j] - kth) <= 2 * tol, (r, j, ref_sc[r, j], kth)


@pytest.mark.parametrize("B,S,Hi,m,k,docs", [
    (1, 1000, 4, 4, 16, False),
    (2, 777, 8, 4, 64, True),      # documents and padding, ragged
    (1, 600, 16, 8, 5, True),
    (1, 300, 2, 1, 300, False),    # k above every row's visible count
])
def test_indexer_matches_oracle(B, S, Hi, m, k, docs):
    qi, ki, w = _inputs(B, S, Hi, m, 31)
    seg = None
    if docs:
        rng = np.random.Generator(np.random.PCG64(S))
        seg = torch.from_numpy(np.stack([I.random_layout(S, rng) for _ in range(B)]))
    sel, sc = hca.hca_indexer_topk(qi.to(DEV), ki.to(DEV), w.to(DEV), None if seg is None else seg.to(DEV), m, k,
                                   with_scores=True, check=True)
    ref = CI.index_scores(qi, ki, w, seg, m)
    sel, sc = sel.cpu().numpy(), sc.cpu().numpy().astype(np.float64)
    for b in range(B):
        _check_rows(sel[b], sc[b], ref[b], k)


def test_indexer_full_size_sampled_rows():
    # the CSA workload's indexer: S = 65536, m = 4 (16384 entries), k = 512,
    # 8 index heads; rows sampled at both ends and in the middle
    B, S, Hi, m, k = 1, 65536, 8, 4, 512
    qi, ki, w = _inputs(B, S, Hi, m, 41)
    sel, sc = hca.hca_indexer_topk(qi.to(DEV), ki.to(DEV), w.to(DEV), None, m, k, with_scores=True, check=True)
    sel_c, sc_c = sel.cpu().numpy(), sc.cpu().numpy()
    for r0 in (0, 2040, 32768, S - 8):
        rows = (r0, r0 + 8)
        ref = CI.index_scores(qi, ki, w, None, m, rows=rows)
        _check_rows(sel_c[0, r0:r0 + 8], sc_c[0, r0:r0 + 8].astype(np.float64), ref[0], k)


def test_indexer_ties():
    # the entries repeat three key vectors, so every row's scores take three
    # values: the k-th largest is a heavy tie (smaller entry index first);
    # early rows resolve it from the list of keys sharing the k-th key's top
    # digit, late rows (more than the list holds) from passes over every key
    B, S, Hi, m, k = 1, 8192, 2, 1, 100
    qi, ki, w = _inputs(B, S, Hi, m, 51)
    pick = torch.from_numpy(np.random.Generator(np.random.PCG64(5)).integers(0, 3, S))
    ki = ki[:, :3][:, pick].contiguous()
    sel, sc = hca.hca_indexer_topk(qi.to(DEV), ki.to(DEV), w.to(DEV), None, m, k, with_scores=True, check=True)
    sel_c, sc_c = sel.cpu().numpy(), sc.cpu().numpy()
    for r0 in (0, 96, 3000, 5500, 5600, 6000, S - 8):
        rows = (r0, r0 + 8)
        ref = CI.index_scores(qi, ki, w, None, m, rows=rows)
        _check_rows(sel_c[0, r0:r0 + 8], sc_c[0, r0:r0 + 8].astype(np.float64), ref[0], k)


def test_indexer_bad_segments_select_nothing():
    qi, ki, w = _inputs(1, 64, 2, 4, 3)
    seg = torch.zeros(1, 64, dtype=torch.int32)
    seg[0, 20:] = 1
    seg[0, 40:] = 0
    ws = torch.empty(hca.load().hca_indexer_workspace_size(1, 64, 4), dtype=torch.uint8, device=DEV)
    sel, _ = hca.hca_indexer_topk(qi.to(DEV), ki.to(DEV), w.to(DEV), seg.to(DEV), 4, 3, ws=ws)
    assert hca.hca_workspace_status(ws) == 6
    assert bool((sel == -1).all())
