"""Failure paths on the GPU, made without faulting it ("Add HCA Static
Compilation for Splash Attention [Deepseek v4]", Description, validation-guard
bullet: unsupported or failing cases are reported as errors, not crashes).

- An injected launch failure: the call returns HCA_ERR_CUDA after checking its
  arguments and before enqueuing anything; the next call is unaffected.
- An injected stall: a kernel's MMA warp first waits on a barrier that nothing
  arrives at, with the bounded-wait limit shortened to 30 ms.  The wait gives
  up, every CTA drains its own copies and MMAs, frees its tensor memory and
  exits; the workspace status reads HCA_ERR_TIMEOUT, the context stays usable
  and the next ordinary call matches the oracle.  The CSA instantiations of
  the forward and dq kernels are stalled the same way.
"""
import math

import pytest
import torch

import oracle
from block_sparse_compressed_gb300 import hca
from block_sparse_compressed_gb300 import inputs as I
from _util import assert_close, valid_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT, CUDA_ERR = 10, 9
STALL_FWD, STALL_DQ, STALL_DKV = 1, 2, 4


@pytest.fixture(autouse=True)
def _reset_hooks():
    hca.hca_test_inject(hca.INJECT_RESET)
    yield
    hca.hca_test_inject(hca.INJECT_RESET)


def _case(S=700, H=16, W=128, m=64, seed=3):
    B, D = 1, 128
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, dtype=torch.bfloat16, seed=seed)
    seg = I.segments_from_lengths([S // 2, S - S // 2 - 30], S, pad=30)
    return (q, kv, ckv, seg, dout), W, m, 1.0 / math.sqrt(D)


def _check_ordinary_call(cpu, W, m, scale, backward):
    q, kv, ckv, seg, dout = cpu
    g = [x.to(DEV) for x in (q, kv, ckv, seg, dout)]
    out, lse = hca.hca_attn_fwd(g[0], g[1], g[2], g[3], W, m, scale, check=True)
    ro, rl = oracle.fwd(q, kv, ckv, seg, W, m, scale)
    v = valid_rows(seg, *q.shape[:3])
    assert_close("out", out, ro, torch.bfloat16, v)
    assert_close("lse", lse, rl, torch.bfloat16, v)
    if backward:
        dq, dkv, dckv = hca.hca_attn_bwd(g[0], g[1], g[2], g[3], out, lse, g[4], W, m, scale, check=True)
        rdq, rdkv, rdckv = oracle.bwd(q, kv, ckv, seg, dout, W, m, scale)
        assert_close("dq", dq, rdq, torch.bfloat16, v)
        assert_close("dkv", dkv, rdkv, torch.bfloat16)
        assert_close("dckv", dckv, rdckv, torch.bfloat16)


def test_injected_launch_failure_returns_cuda_error_and_enqueues_nothing():
    cpu, W, m, scale = _case()
    q, kv, ckv, seg, dout = (x.to(DEV) for x in cpu)
    out = torch.full_like(q, 7.0)
    lse = torch.full(q.shape[:3], 7.0, dtype=torch.float32, device=DEV)
    hca.hca_test_inject(hca.INJECT_LAUNCH_FAILURE, 2)
    with pytest.raises(hca.HCAError) as e:
        hca.hca_attn_fwd(q, kv, ckv, seg, W, m, scale, out=out, lse=lse)
    assert e.value.status == CUDA_ERR
    with pytest.raises(hca.HCAError) as e:
        hca.hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, W, m, scale)
    assert e.value.status == CUDA_ERR
    torch.cuda.synchronize()
    # nothing was enqueued: the outputs still hold what the caller put there
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
    # the injection is used up; the next calls run normally
    _check_ordinary_call(cpu, W, m, scale, backward=True)


@pytest.mark.parametrize("mask", [STALL_FWD])
def test_forward_wait_gives_up_and_context_stays_usable(mask):
    cpu, W, m, scale = _case()
    q, kv, ckv, seg, _ = (x.to(DEV) for x in cpu)
    ws = hca.workspace(1, q.shape[1], q.shape[2], 128, W, m, torch.bfloat16, False, DEV)
    hca.hca_test_inject(hca.INJECT_WAIT_LIMIT_NS, 30_000_000)
    hca.hca_test_inject(hca.INJECT_STALL, mask)
    hca.hca_attn_fwd(q, kv, ckv, seg, W, m, scale, ws=ws)
    assert hca.hca_workspace_status(ws) == TIMEOUT
    hca.hca_test_inject(hca.INJECT_RESET)
    # the context is intact and the same workspace serves an ordinary call
    out, lse = hca.hca_attn_fwd(q, kv, ckv, seg, W, m, scale, ws=ws)
    assert hca.hca_workspace_status(ws) == 0
    ro, rl = oracle.fwd(*cpu[:4], W, m, scale)
    v = valid_rows(cpu[3], *cpu[0].shape[:3])
    assert_close("out", out, ro, torch.bfloat16, v)
    assert_close("lse", lse, rl, torch.bfloat16, v)


@pytest.mark.parametrize("mask", [STALL_DQ, STALL_DKV])
def test_backward_wait_gives_up_and_context_stays_usable(mask):
    cpu, W, m, scale = _case(seed=4)
    q, kv, ckv, seg, dout = (x.to(DEV) for x in cpu)
    out, lse = hca.hca_attn_fwd(q, kv, ckv, seg, W, m, scale, check=True)
    ws = hca.workspace(1, q.shape[1], q.shape[2], 128, W, m, torch.bfloat16, True, DEV)
    hca.hca_test_inject(hca.INJECT_WAIT_LIMIT_NS, 30_000_000)
    hca.hca_test_inject(hca.INJECT_STALL, mask)
    hca.hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, W, m, scale, ws=ws)
    assert hca.hca_workspace_status(ws) == TIMEOUT
    hca.hca_test_inject(hca.INJECT_RESET)
    _check_ordinary_call(cpu, W, m, scale, backward=True)


@pytest.mark.parametrize("mask", [STALL_FWD, STALL_DQ])
def test_csa_wait_gives_up_and_context_stays_usable(mask):
    # the CSA instantiations give up the same way; their TMA warp has TMA
    # gather4 loads of the selected rows in flight, which land before the CTA
    # exits and frees its tensor memory
    B, H, S, W, m, k, D = 1, 64, 600, 64, 4, 16, 128
    scale = 1.0 / math.sqrt(D)
    q, kv, ckv, _, dout = I.small(B, H, S, D, W, m, dtype=torch.bfloat16, seed=11)
    sel = I.random_selection(B, S, m, k, 61)
    g = [x.to(DEV) for x in (q, kv, ckv, dout, sel)]
    hca.hca_test_inject(hca.INJECT_WAIT_LIMIT_NS, 30_000_000)
    if mask == STALL_FWD:
        ws = hca.csa_workspace(B, H, S, D, W, m, k, torch.bfloat16, False, DEV)
        hca.hca_test_inject(hca.INJECT_STALL, mask)
        hca.hca_csa_attn_fwd(g[0], g[1], g[2], None, g[4], W, m, scale, ws=ws)
    else:
        out, lse = hca.hca_csa_attn_fwd(g[0], g[1], g[2], None, g[4], W, m, scale, check=True)
        ws = hca.csa_workspace(B, H, S, D, W, m, k, torch.bfloat16, True, DEV)
        hca.hca_test_inject(hca.INJECT_STALL, mask)
        hca.hca_csa_attn_bwd(g[0], g[1], g[2], None, g[4], out, lse, g[3], W, m, scale, ws=ws)
    assert hca.hca_workspace_status(ws) == TIMEOUT
    hca.hca_test_inject(hca.INJECT_RESET)
    # ordinary calls afterwards match the oracle
    keep = oracle.topk_mask(sel, -(-S // m))
    out, lse = hca.hca_csa_attn_fwd(g[0], g[1], g[2], None, g[4], W, m, scale, check=True)
    ro, rl = oracle.csa_fwd(q, kv, ckv, None, keep, W, m, scale)
    assert_close("out", out, ro, torch.bfloat16)
    assert_close("lse", lse, rl, torch.bfloat16)
    dq, dkv, dckv = hca.hca_csa_attn_bwd(g[0], g[1], g[2], None, g[4], out, lse, g[3], W, m, scale, check=True)
    rdq, rdkv, rdckv = oracle.csa_bwd(q, kv, ckv, None, keep, dout, W, m, scale)
    assert_close("dq", dq, rdq, torch.bfloat16)
    assert_close("dkv", dkv, rdkv, torch.bfloat16)
    assert_close("dckv", dckv, rdckv, torch.bfloat16)


def test_stall_mask_is_consumed_by_one_call():
    cpu, W, m, scale = _case(S=300, H=4)
    q, kv, ckv, seg, _ = (x.to(DEV) for x in cpu)
    hca.hca_test_inject(hca.INJECT_WAIT_LIMIT_NS, 30_000_000)
    hca.hca_test_inject(hca.INJECT_STALL, STALL_FWD)
    ws = hca.workspace(1, q.shape[1], q.shape[2], 128, W, m, torch.bfloat16, False, DEV)
    hca.hca_attn_fwd(q, kv, ckv, seg, W, m, scale, ws=ws)
    assert hca.hca_workspace_status(ws) == TIMEOUT
    # no reset: the second call runs normally with the short limit still set
    hca.hca_attn_fwd(q, kv, ckv, seg, W, m, scale, ws=ws)
    assert hca.hca_workspace_status(ws) == 0
