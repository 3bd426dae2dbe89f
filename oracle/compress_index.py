"""fp64 CPU oracle for the two steps that produce HCA's and CSA's compressed
entries and CSA's selection: the HCA compressor (pooling of kv into ckv over
length-m windows) and the Lightning Indexer (index scores of compressed
entries per query, sentinel masking, top-k).

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/`` and by ``bench.py``'s CPU
baseline; the product library never imports or calls it and shares no code
with it.  Plain numpy in float64, one definition per function, written from
the pages:

- "[DeepSeek-V4] Implement Compressed Attention Layers", Description: the
  CSA/HCA compressors pool with a causal block bias; the LightningIndexer
  implements sentinel masking; review suggestion on the indexer: scores are
  the matmul of the indexer queries with the (transposed) compressed kv,
  giving [B, S, H, W] per-head scores against the compressed entries.
- "Add HCA Static Compilation for Splash Attention [Deepseek v4]",
  Description: compressed entries are length-m windows (the HCA compressor's
  window boundaries); CSA (compress ratio 4) needs a top-k step.

Readings where the pages are silent (each listed in the design notes):
- Compressor: within window j the positions' gate logits g plus a bias per
  offset inside the block (the "causal block bias") are softmax-normalised
  over the window's non-padding positions, and the entry is the weighted sum
  of those rows.  A window without such positions gives a zero row.
- Indexer: the per-head scores are combined by a weighted sum over heads with
  per-(query, head) weights (all-ones gives the plain sum); an optional ReLU
  on each per-head score is a flag (the pages name no activation).  Entries a
  query may not see (not completed, or outside its document; the HCA
  compressed rule) get the sentinel -inf and are never selected.  top-k keeps
  the k largest scores, ties going to the smaller entry index; the result is
  the selected entry ids in ascending order, padded with -1 when fewer than k
  entries are visible.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _seg(seg, B, S):
    if seg is None:
        return np.zeros((B, S), dtype=np.int64)
    try:
        import torch
        if isinstance(seg, torch.Tensor):
            seg = seg.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    s = np.asarray(seg, dtype=np.int64)
    assert s.shape == (B, S), s.shape
    return s


# --------------------------------------------------------------------------
# HCA compressor
# --------------------------------------------------------------------------

def compress_weights(g, bias, seg, m: int):
    """Pooling weights a[B, Sc, m] of every window (0 outside the sequence and
    at padding positions)."""
    g = _f64(g)
    bias = _f64(bias)
    B, S = g.shape
    assert bias.shape == (m,)
    sg = _seg(seg, B, S)
    Sc = -(-S // m)
    a = np.zeros((B, Sc, m))
    for b in range(B):
        for j in range(Sc):
            pos = [j * m + r for r in range(m) if j * m + r < S and sg[b, j * m + r] >= 0]
            if not pos:
                continue
            z = np.array([g[b, x] + bias[x - j * m] for x in pos])
            e = np.exp(z - z.max())
            for x, v in zip(pos, e / e.sum()):
                a[b, j, x - j * m] = v
    return a


def compress_fwd(x, g, bias, seg, m: int):
    """ckv[B, Sc, D] = per window, the softmax(g + bias)-weighted sum of its
    rows of x[B, S, D]."""
    x = _f64(x)
    B, S, D = x.shape
    a = compress_weights(g, bias, seg, m)
    Sc = a.shape[1]
    ckv = np.zeros((B, Sc, D))
    for j in range(Sc):
        for r in range(m):
            t = j * m + r
            if t < S:
                ckv[:, j, :] += a[:, j, r, None] * x[:, t, :]
    return ckv


def compress_bwd(x, g, bias, seg, m: int, dckv):
    """(dx[B,S,D], dg[B,S], dbias[m]) for the cotangent dckv[B,Sc,D]."""
    x = _f64(x)
    dckv = _f64(dckv)
    B, S, D = x.shape
    a = compress_weights(g, bias, seg, m)
    Sc = a.shape[1]
    dx = np.zeros((B, S, D))
    dg = np.zeros((B, S))
    dbias = np.zeros(m)
    sg = _seg(seg, B, S)
    for b in range(B):
        for j in range(Sc):
            idx = [r for r in range(m) if j * m + r < S and sg[b, j * m + r] >= 0]
            if not idx:
                continue
            da = np.array([dckv[b, j] @ x[b, j * m + r] for r in idx])
            w = np.array([a[b, j, r] for r in idx])
            dz = w * (da - (w * da).sum())
            for k, r in enumerate(idx):
                t = j * m + r
                dx[b, t] = w[k] * dckv[b, j]
                dg[b, t] = dz[k]
                dbias[r] += dz[k]
    return dx, dg, dbias


# --------------------------------------------------------------------------
# Lightning Indexer: scores, sentinel masking, top-k
# --------------------------------------------------------------------------

def comp_visible(seg, B: int, S: int, m: int, rows=None):
    """bool [B, R, Sc]: compressed entry j may be seen by query i (its window
    [j*m, (j+1)*m - 1] has completed at i and lies in i's document), for the
    query positions i in rows = (r0, r1) (default: all S)."""
    sg = _seg(seg, B, S)
    Sc = -(-S // m)
    r0, r1 = rows if rows is not None else (0, S)
    vis = np.zeros((B, r1 - r0, Sc), dtype=bool)
    for b in range(B):
        for j in range(Sc):
            lo, hi = j * m, (j + 1) * m - 1
            if hi >= S:
                continue
            d = sg[b, lo]
            if d < 0 or not np.all(sg[b, lo:hi + 1] == d):
                continue
            for i in range(max(hi, r0), r1):
                if sg[b, i] == d:
                    vis[b, i - r0, j] = True
    return vis


def index_scores(qi, ki, w, seg, m: int, relu: bool = False, rows=None):
    """float64 [B, R, Sc]: sum_h w[b,s,h] * act(<qi[b,s,h,:], ki[b,j,:]>) for
    visible entries, -inf (the sentinel) elsewhere; query positions s in
    rows = (r0, r1) (default: all)."""
    B, S = qi.shape[0], qi.shape[1]
    r0, r1 = rows if rows is not None else (0, S)
    qi = _f64(qi[:, r0:r1])
    ki = _f64(ki)
    w = _f64(w[:, r0:r1])
    Hi, Di = qi.shape[2], qi.shape[3]
    Sc = ki.shape[1]
    assert ki.shape == (B, Sc, Di) and w.shape == (B, r1 - r0, Hi)
    per_head = np.einsum("bshd,bjd->bshj", qi, ki)
    if relu:
        per_head = np.maximum(per_head, 0.0)
    sc = np.einsum("bsh,bshj->bsj", w, per_head)
    vis = comp_visible(seg, B, S, m, rows=(r0, r1))
    assert vis.shape == sc.shape
    return np.where(vis, sc, -np.inf)


def topk_select(scores, k: int):
    """int64 [B, S, k]: per query, the k entries with the largest finite
    score (ties: smaller entry index first), in ascending entry order, -1
    where fewer than k entries are visible."""
    sc = np.asarray(scores, dtype=np.float64)
    B, S, Sc = sc.shape
    out = np.full((B, S, k), -1, dtype=np.int64)
    for b in range(B):
        for s in range(S):
            row = sc[b, s]
            vis = np.flatnonzero(np.isfinite(row))
            # larger score first, then smaller index
            order = sorted(vis.tolist(), key=lambda j: (-row[j], j))
            sel = sorted(order[:k])
            out[b, s, :len(sel)] = sel
    return out


def indexer_topk(qi, ki, w, seg, m: int, k: int, relu: bool = False):
    """(selection int64 [B,S,k], scores float64 [B,S,Sc])."""
    sc = index_scores(qi, ki, w, seg, m, relu)
    return topk_select(sc, k), sc
