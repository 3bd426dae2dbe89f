"""The head-sharding split on one GPU.  With the query heads partitioned
across devices, each device runs the library on its own head slice: q, out,
lse and dq are sharded, kv and ckv replicated, and the only exchange step is
a sum of the per-slice dkv and dckv (one all-reduce).  This test runs the
slices in one process and does that sum on the host in fp32, then compares
with the call over all heads and with the fp64 oracle.  (Key and value share
the one kv head for all query heads: "[DeepSeek-V4] Implement Compressed
Attention Layers", einsum review suggestions.)"""
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


@pytest.mark.parametrize("group", [16, 32])
def test_head_slices_sum_to_the_full_call(group):
    B, H, S, D, W, m = 2, 64, 1100, 128, 128, 64
    scale = 1.0 / math.sqrt(D)
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, dtype=torch.bfloat16, seed=11)
    seg = torch.cat([I.segments_from_lengths([500, 560], S, pad=40),
                     I.segments_from_lengths([1100], S)])
    g = [x.to(DEV) for x in (q, kv, ckv, seg, dout)]
    # full call over all heads
    out, lse = hca.hca_attn_fwd(g[0], g[1], g[2], g[3], W, m, scale, check=True)
    dq, dkv, dckv = hca.hca_attn_bwd(g[0], g[1], g[2], g[3], out, lse, g[4], W, m, scale, check=True)
    # one call per head slice, as one device of a head-sharded layer would make
    outs, lses, dqs = [], [], []
    dkv_sum = torch.zeros(B, S, D, dtype=torch.float32, device=DEV)
    dckv_sum = torch.zeros(ckv.shape, dtype=torch.float32, device=DEV)
    for h0 in range(0, H, group):
        qs = g[0][:, h0:h0 + group].contiguous()
        dos = g[4][:, h0:h0 + group].contiguous()
        o, l = hca.hca_attn_fwd(qs, g[1], g[2], g[3], W, m, scale, check=True)
        a, b, c = hca.hca_attn_bwd(qs, g[1], g[2], g[3], o, l, dos, W, m, scale, check=True)
        outs.append(o)
        lses.append(l)
        dqs.append(a)
        dkv_sum += b.float()
        dckv_sum += c.float()
    v = valid_rows(seg, B, H, S)
    # the forward and dq of a head do not depend on the other heads (a slice
    # packs its heads into tiles differently, so only rounding may differ)
    assert_close("out (slices) vs full call", torch.cat(outs, 1), to_np(out), torch.bfloat16, v)
    assert_close("lse (slices) vs full call", torch.cat(lses, 1), to_np(lse), torch.bfloat16, v)
    assert_close("dq (slices) vs full call", torch.cat(dqs, 1), to_np(dq), torch.bfloat16, v)
    # the summed slices match the full call and the oracle
    rdq, rdkv, rdckv = oracle.bwd(q, kv, ckv, seg, dout, W, m, scale)
    assert_close("dkv (slices summed) vs full call", dkv_sum, to_np(dkv), torch.bfloat16)
    assert_close("dckv (slices summed) vs full call", dckv_sum, to_np(dckv), torch.bfloat16)
    assert_close("dkv (slices summed) vs oracle", dkv_sum, rdkv, torch.bfloat16)
    assert_close("dckv (slices summed) vs oracle", dckv_sum, rdckv, torch.bfloat16)
    assert_close("dq vs oracle", dq, rdq, torch.bfloat16, v)
