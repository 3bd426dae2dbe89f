"""GPU parity: libhca (through the C ABI binding) against the fp64 oracle.

Tolerance per tensor over valid positions: bf16 max|err| <= 1e-2*max|ref| +
1e-3; fp32 max|err| <= 1e-5.  Visible-pair counts and tile ranges are
compared bit-exactly.
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


def run_case(B, H, S, D, W, m, dtype, seg=None, backward=True, seed=1234, scale=None):
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, dtype=dtype, seed=seed)
    seg_t = None if seg is None else torch.as_tensor(np.asarray(seg, dtype=np.int32)).reshape(B, S)
    g = [x.to(DEV) for x in (q, kv, ckv, dout)]
    sg = None if seg_t is None else seg_t.to(DEV)
    out, lse = hca.hca_attn_fwd(g[0], g[1], g[2], sg, W, m, scale, check=True)
    ro, rl = oracle.fwd(q, kv, ckv, seg_t, W, m, scale)
    v = valid_rows(seg_t, B, H, S)
    assert_close("out", out, ro, dtype, v)
    assert_close("lse", lse, rl, dtype, v)
    got_out, got_lse = to_np(out), to_np(lse)
    assert np.all(got_out[~v] == 0)
    assert np.all(got_lse[~v] == -np.inf)
    if not backward:
        return
    dq, dkv, dckv = hca.hca_attn_bwd(g[0], g[1], g[2], sg, out, lse, g[3], W, m, scale, check=True)
    rdq, rdkv, rdckv = oracle.bwd(q, kv, ckv, seg_t, dout, W, m, scale)
    assert_close("dq", dq, rdq, dtype, v)
    assert np.all(to_np(dq)[~v] == 0)
    assert_close("dkv", dkv, rdkv, dtype)
    assert_close("dckv", dckv, rdckv, dtype)


def test_tiny_f32_workload():
    w = I.TINY_F32
    seg = I.segments(w)
    run_case(w.B, w.H, w.S, w.D, w.W, w.m, torch.float32, seg)


@pytest.mark.parametrize("S", [1, 15, 16, 17, 127, 128, 129, 489])
def test_edge_lengths_bf16(S):
    run_case(1, 4, S, 128, 128, 128, torch.bfloat16)


@pytest.mark.parametrize("W,m", [(1, 128), (1, 1), (300, 16), (128, 1000), (5, 3)])
def test_edge_windows_bf16(W, m):
    run_case(1, 8, 300, 128, W, m, torch.bfloat16)


@pytest.mark.parametrize("H,W,m", [(64, 16, 1), (64, 113, 2), (64, 128, 8), (64, 200, 1), (128, 128, 1), (16, 48, 2)])
def test_key_list_block_boundaries_bf16(H, W, m):
    # a tile's key list is its compressed entries (padded to 16) then its raw
    # keys, cut into 128-column blocks: over 700 positions the compressed
    # count takes every residue mod 16 and mod 128, so blocks hold compressed
    # rows only, raw rows only, or both (16-row loads), and last blocks are short
    run_case(1, H, 700, 128, W, m, torch.bfloat16)


@pytest.mark.parametrize("scale", [2.0, -1.0 / math.sqrt(128)])
def test_rescale_and_negative_scale_bf16(scale):
    # scale 2 spreads the logits (std ~ 23), so a row's running max grows by
    # more than 2^8 between key blocks and O is rescaled; a negative scale
    # runs the forward's min-based instantiation
    run_case(1, 64, 600, 128, 128, 16, torch.bfloat16, scale=scale)


@pytest.mark.parametrize("H", [1, 4, 16, 64, 128, 256])
def test_heads_bf16(H):
    run_case(1, H, 260, 128, 64, 32, torch.bfloat16)


@pytest.mark.parametrize("H", [3, 6, 48, 96, 24])
def test_any_head_count_on_tensor_cores(H):
    # a tile packs the largest power of two dividing H and 128 (H = 3: one
    # head x 128 positions; 48: 16 heads x 8 positions; 96: 32 x 4)
    assert hca.hca_query_tile_positions(H, 128, torch.bfloat16) == 128 // math.gcd(H, 128)
    run_case(1, H, 300, 128, 48, 16, torch.bfloat16)


@pytest.mark.parametrize("H,S,W,m,layout", [(64, 700, 128, 16, False), (16, 489, 333, 64, True),
                                             (48, 300, 48, 1, False), (128, 260, 600, 8, True)])
def test_head_dim_64_bf16(H, S, W, m, layout):
    # D = 64 runs its own instantiation of the tensor-core kernels (one
    # 128-byte half per row instead of two): several query tiles and key
    # blocks with a ragged tail, multi-block windows, the atomic raw partials
    # (W = 600) and documents with padding
    seg = None
    if layout:
        rng = np.random.Generator(np.random.PCG64(S))
        seg = I.random_layout(S, rng, allow_pad=True)[None]
    assert hca.hca_query_tile_positions(H, 64, torch.bfloat16) == 128 // math.gcd(H, 128)
    run_case(1, H, S, 64, W, m, torch.bfloat16, seg)


@pytest.mark.parametrize("D", [32, 256])
def test_bf16_head_dims_without_a_tensor_core_tile_are_rejected(D):
    # bf16 runs on the tensor-core kernels only: other head dims are an
    # error, never a silent CUDA-core fallback
    q, kv, ckv, _, dout = I.small(1, 4, 64, D, 16, 8, dtype=torch.bfloat16)
    q, kv, ckv, dout = (x.to(DEV) for x in (q, kv, ckv, dout))
    with pytest.raises(hca.HCAError) as e:
        hca.hca_attn_fwd(q, kv, ckv, None, 16, 8, 0.1)
    assert e.value.status == 8
    out = torch.zeros_like(q)
    lse = torch.zeros(q.shape[:3], dtype=torch.float32, device=DEV)
    with pytest.raises(hca.HCAError) as e:
        hca.hca_attn_bwd(q, kv, ckv, None, out, lse, dout, 16, 8, 0.1)
    assert e.value.status == 8


@pytest.mark.parametrize("B", [1, 3])
def test_long_window_multiple_raw_blocks(B):
    # W > 128: a tile's raw range spans several 128-key blocks
    rng = np.random.Generator(np.random.PCG64(B))
    S = 700
    seg = np.stack([I.random_layout(S, rng, allow_pad=True) for _ in range(B)])
    run_case(B, 16, S, 128, 333, 64, torch.bfloat16, seg)


@pytest.mark.parametrize("W", [390, 600])
def test_long_window_atomic_raw_partials(W):
    # windows longer than four 128-key blocks: the key-major backward sums the
    # raw blocks' partials with fp32 atomics instead of per-range slots
    rng = np.random.Generator(np.random.PCG64(W))
    S = 900
    seg = np.stack([I.random_layout(S, rng, allow_pad=True) for _ in range(2)])
    run_case(2, 16, S, 128, W, 64, torch.bfloat16, seg)


def test_segments_off_boundary_and_short_docs_bf16():
    # documents starting off an m-boundary, one shorter than W and than m,
    # and padding at the end
    lens = [70, 5, 200, 31]
    S = sum(lens) + 30
    seg = I.segments_from_lengths(lens, S, pad=30)
    run_case(1, 8, S, 128, 64, 16, torch.bfloat16, seg)


def test_random_layouts_bf16():
    rng = np.random.Generator(np.random.PCG64(5))
    for k in range(4):
        S = int(rng.integers(50, 400))
        seg = np.stack([I.random_layout(S, rng), I.random_layout(S, rng)])
        run_case(2, 4, S, 128, int(rng.integers(1, 100)), int(rng.integers(1, 40)), torch.bfloat16, seg, seed=k)


def test_random_layouts_f32():
    rng = np.random.Generator(np.random.PCG64(6))
    for k in range(3):
        S = int(rng.integers(20, 200))
        seg = np.stack([I.random_layout(S, rng)])
        run_case(1, 3, S, 64, int(rng.integers(1, 50)), int(rng.integers(1, 20)), torch.float32, seg, seed=k)


def test_many_documents_bf16():
    # more documents than compressed splits need; W > 128 and m < 128
    lens = [40, 300, 129, 1, 700, 256, 77]
    S = sum(lens)
    seg = I.segments_from_lengths(lens, S)
    run_case(1, 4, S, 128, 200, 32, torch.bfloat16, seg)


def test_fwd_4096_two_documents():
    w = I.FWD_S4096_2DOC
    q, kv, ckv, seg, _ = I.tensors(w, with_dout=False)
    out, lse = hca.hca_attn_fwd(q.to(DEV), kv.to(DEV), ckv.to(DEV), seg.to(DEV), w.W, w.m, w.scale, check=True)
    ro, rl = oracle.fwd(q, kv, ckv, seg, w.W, w.m, w.scale)
    assert_close("out", out, ro, w.dtype)
    assert_close("lse", lse, rl, w.dtype)


# --------------------------------------------------------------------------
# visibility enumeration: bit-exact
# --------------------------------------------------------------------------

def _layouts():
    rng = np.random.Generator(np.random.PCG64(11))
    cases = []
    for _ in range(12):
        S = int(rng.integers(1, 700))
        cases.append((S, int(rng.integers(1, 200)), int(rng.integers(1, 150)),
                      np.stack([I.random_layout(S, rng) for _ in range(2)])))
    return cases


def test_visible_pairs_bit_exact():
    for S, W, m, seg in _layouts():
        raw, comp = hca.hca_visible_pairs(torch.from_numpy(seg).to(DEV), 2, S, W, m)
        oraw, ocomp = oracle.visible_pairs(seg, 2, S, W, m)
        assert raw.cpu().numpy().tolist() == oraw.tolist()
        assert comp.cpu().numpy().tolist() == ocomp.tolist()


@pytest.mark.parametrize("Pq", [1, 2, 8, 128])
def test_tile_map_bit_exact(Pq):
    for S, W, m, seg in _layouts():
        got = hca.hca_tile_map(torch.from_numpy(seg).to(DEV), 2, S, W, m, Pq).cpu().numpy()
        exp = oracle.tile_ranges(seg, 2, S, W, m, Pq)
        np.testing.assert_array_equal(got, exp)


@pytest.mark.parametrize("w", [I.TINY_F32, I.FWD_S4096_2DOC, I.DOCS_S16384, I.UNALIGNED, I.LONG_S65536])
def test_workload_pair_counts_bit_exact(w):
    seg = I.segments(w)
    raw, comp = hca.hca_visible_pairs(None if seg is None else seg.to(DEV), w.B, w.S, w.W, w.m, device=DEV)
    oraw, ocomp = oracle.visible_pairs(seg, w.B, w.S, w.W, w.m)
    assert raw.cpu().numpy().tolist() == oraw.tolist()
    assert comp.cpu().numpy().tolist() == ocomp.tolist()
    Pq = hca.hca_query_tile_positions(w.H, w.D, w.dtype)
    if w.S <= 16384:
        got = hca.hca_tile_map(None if seg is None else seg.to(DEV), w.B, w.S, w.W, w.m, Pq, device=DEV)
        np.testing.assert_array_equal(got.cpu().numpy(), oracle.tile_ranges(seg, w.B, w.S, w.W, w.m, Pq))


def test_bad_segment_order_is_reported_and_poisons_outputs():
    B, H, S, D, W, m = 1, 2, 64, 128, 16, 8
    q, kv, ckv, _, _ = I.small(B, H, S, D, W, m, dtype=torch.bfloat16)
    seg = torch.zeros(B, S, dtype=torch.int32)
    seg[0, 20:] = 1
    seg[0, 40:] = 0          # id decreases: not a packed layout
    with pytest.raises(hca.HCAError) as e:
        hca.hca_attn_fwd(q.to(DEV), kv.to(DEV), ckv.to(DEV), seg.to(DEV), W, m, 0.1, check=True)
    assert e.value.status == 6
    seg2 = torch.zeros(B, S, dtype=torch.int32)
    seg2[0, 30:40] = -1      # padding in the middle
    ws = hca.workspace(B, H, S, D, W, m, torch.bfloat16, False, DEV)
    out, lse = hca.hca_attn_fwd(q.to(DEV), kv.to(DEV), ckv.to(DEV), seg2.to(DEV), W, m, 0.1, ws=ws)
    assert hca.hca_workspace_status(ws) == 6
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
