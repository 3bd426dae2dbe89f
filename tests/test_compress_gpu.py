"""GPU parity of the HCA compressor (hca_compress_fwd / hca_compress_bwd,
through the C ABI binding) against the fp64 oracle in
oracle/compress_index.py.  Tolerance per tensor: bf16 max|err| <=
1e-2*max|ref| + 1e-3; fp32 max|err| <= 1e-5."""
import numpy as np
import pytest
import torch

from oracle import compress_index as CI
from block_sparse_compressed_gb300 import hca
from block_sparse_compressed_gb300 import inputs as I
from _util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(B, S, D, m, dtype, seed):
    x = I.normal((B, S, D), seed, dtype)
    g = I.normal((B, S), seed + 1, torch.float32)
    bias = I.normal((m,), seed + 2, torch.float32)
    dck = I.normal((B, -(-S // m), D), seed + 3, dtype)
    return x, g, bias, dck


@pytest.mark.parametrize("B,S,D,m,dtype", [
    (2, 1000, 128, 128, torch.bfloat16),   # HCA ratio, ragged last window
    (1, 777, 128, 4, torch.bfloat16),      # CSA ratio
    (2, 300, 64, 7, torch.float32),
    (1, 129, 32, 40, torch.float32),       # m > 32: logits in two lane passes
    (1, 65, 256, 1, torch.bfloat16),
])
def test_compressor_matches_oracle(B, S, D, m, dtype):
    x, g, bias, dck = _inputs(B, S, D, m, dtype, 21)
    rng = np.random.Generator(np.random.PCG64(S))
    seg = torch.from_numpy(np.stack([I.random_layout(S, rng) for _ in range(B)]))
    gd = [t.to(DEV) for t in (x, g, bias, seg, dck)]
    ckv = hca.hca_compress_fwd(gd[0], gd[1], gd[2], gd[3], m)
    dx, dg, db = hca.hca_compress_bwd(gd[0], gd[1], gd[2], gd[3], m, gd[4])
    torch.cuda.synchronize()
    assert_close("ckv", ckv, CI.compress_fwd(x, g, bias, seg, m), dtype)
    rdx, rdg, rdb = CI.compress_bwd(x, g, bias, seg, m, dck)
    assert_close("dx", dx, rdx, dtype)
    assert_close("dg", dg, rdg, dtype)
    assert_close("dbias", db, rdb, dtype)
    # the backward is deterministic (fixed-order bias reduction)
    dx2, dg2, db2 = hca.hca_compress_bwd(gd[0], gd[1], gd[2], gd[3], m, gd[4])
    assert torch.equal(dx, dx2) and torch.equal(dg, dg2) and torch.equal(db, db2)


def test_compressor_bench_size_exact():
    # the bench workload, B16 S65536 D128 m128 bf16 with the bench's seeds:
    # every output against the oracle (the windows are independent, so the
    # whole tensor is cheap to check)
    B, S, D, m = 16, 65536, 128, 128
    x = I.normal((B, S, D), 1, torch.bfloat16)
    g = I.normal((B, S), 2, torch.float32)
    bias = I.normal((m,), 3, torch.float32)
    dck = I.normal((B, S // m, D), 4, torch.bfloat16)
    gd = [t.to(DEV) for t in (x, g, bias, dck)]
    ckv = hca.hca_compress_fwd(gd[0], gd[1], gd[2], None, m)
    dx, dg, db = hca.hca_compress_bwd(gd[0], gd[1], gd[2], None, m, gd[3])
    torch.cuda.synchronize()
    assert_close("ckv", ckv, CI.compress_fwd(x, g, bias, None, m), torch.bfloat16)
    rdx, rdg, rdb = CI.compress_bwd(x, g, bias, None, m, dck)
    assert_close("dx", dx, rdx, torch.bfloat16)
    assert_close("dg", dg, rdg, torch.bfloat16)
    assert_close("dbias", db, rdb, torch.bfloat16)


def test_compressor_without_segments_and_unsupported_dim():
    x, g, bias, _ = _inputs(1, 512, 128, 16, torch.bfloat16, 5)
    ckv = hca.hca_compress_fwd(x.to(DEV), g.to(DEV), bias.to(DEV), None, 16)
    assert_close("ckv", ckv, CI.compress_fwd(x, g, bias, None, 16), torch.bfloat16)
    x2 = I.normal((1, 64, 48), 1, torch.bfloat16).to(DEV)
    with pytest.raises(hca.HCAError) as e:
        hca.hca_compress_fwd(x2, g[:, :64].contiguous().to(DEV), bias.to(DEV), None, 16)
    assert e.value.status == 8


def test_compressor_feeds_the_attention():
    # ckv produced on the GPU by the compressor, then HCA attention over it,
    # against the oracle chain (compressor then attention) in fp64
    import math
    import oracle
    B, H, S, D, W, m = 1, 16, 600, 128, 64, 32
    x, g, bias, _ = _inputs(B, S, D, m, torch.bfloat16, 8)
    q = I.normal((B, H, S, D), 9, torch.bfloat16)
    ckv = hca.hca_compress_fwd(x.to(DEV), g.to(DEV), bias.to(DEV), None, m)
    out, lse = hca.hca_attn_fwd(q.to(DEV), x.to(DEV), ckv, None, W, m, 1 / math.sqrt(D), check=True)
    # the attention oracle on the GPU's bf16 ckv (the compressor itself is
    # checked above); out must match within the bf16 bound
    ro, _ = oracle.fwd(q, x, ckv.cpu(), None, W, m, 1 / math.sqrt(D))
    assert_close("out", out, ro, torch.bfloat16)


def test_compressor_ignores_values_at_padding():
    # padding positions may hold anything (here NaN); they must not leak into
    # any output of the forward or the backward
    B, S, D, m = 1, 300, 128, 16
    x, g, bias, dck = _inputs(B, S, D, m, torch.bfloat16, 12)
    seg = I.segments_from_lengths([120, 130], S, pad=50)
    xn = x.clone()
    xn[0, 250:] = float("nan")
    gn = g.clone()
    gn[0, 250:] = float("nan")
    gd = [t.to(DEV) for t in (xn, gn, bias, seg, dck)]
    ckv = hca.hca_compress_fwd(gd[0], gd[1], gd[2], gd[3], m)
    dx, dg, db = hca.hca_compress_bwd(gd[0], gd[1], gd[2], gd[3], m, gd[4])
    torch.cuda.synchronize()
    assert_close("ckv", ckv, CI.compress_fwd(x, g, bias, seg, m), torch.bfloat16)
    rdx, rdg, rdb = CI.compress_bwd(x, g, bias, seg, m, dck)
    assert_close("dx", dx, rdx, torch.bfloat16)
    assert_close("dg", dg, rdg, torch.bfloat16)
    assert_close("dbias", db, rdb, torch.bfloat16)
