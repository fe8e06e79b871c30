"""Failure detection without a GPU fault.

attn_fwd_test_skip_load makes the producer warp of every CTA never issue one
K/V load.  The consumers' bounded mbarrier waits run out (about 2 s), the
kernel records ATTN_ERR_DEVICE_TIMEOUT in the device error word, every CTA
unwinds (frees its TMEM, lets its own copies land) and exits.  The host reads
the status; the context stays usable and the next call is correct.
Nothing traps, faults or hangs.
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
import online_softmax_attention_attn_gb300 as pkg
from online_softmax_attention_attn_gb300.inputs import mha_inputs

pytestmark = pytest.mark.gpu


def test_stuck_pipeline_reports_timeout_and_context_survives():
    dev = torch.device("cuda")
    q, k, v = mha_inputs(1, 1, 512, 128, torch.bfloat16, seed=80)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(dq)
    lse = torch.empty(1, 1, 512, dtype=torch.float32, device=dev)
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
    t0 = time.time()
    # load 3 is V_1: the second KV block's values never arrive
    pkg.attn_fwd_test_skip_load(dq, dk, dv, o, lse, True, 1.0 / math.sqrt(128), 3)
    code = pkg.attn_device_status(raise_on_error=False)
    elapsed = time.time() - t0
    assert code == pkg.ATTN_ERR_DEVICE_TIMEOUT, pkg.attn_last_error()
    assert "wait ran out" in pkg.attn_last_error()
    assert elapsed < 30
    # the error word was cleared and the context is healthy
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
    o2, lse2 = pkg.attn_fwd(dq, dk, dv, causal=True)
    pkg.attn_device_status()
    ro, rl = oracle.mha(q, k, v, True, 1.0 / math.sqrt(128))
    assert np.abs(o2.float().cpu().numpy() - ro).max() <= 2e-2
    assert np.abs(lse2.cpu().numpy() - rl).max() <= 1e-3


def test_skip_hook_rejects_bad_index():
    dev = torch.device("cuda")
    q = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(pkg.AttnError):
        pkg.attn_fwd_test_skip_load(q, q, q, q.clone(), torch.empty(1, 1, 128, device=dev),
                                    False, 0.1, 0)


def test_stuck_tf32x3_pipeline_reports_timeout_and_context_survives():
    """attn_fwd_tf32x3 with block 1 never loaded: the S issuer's bounded wait
    runs out in every CTA, the CTAs unwind, and the next call is correct."""
    dev = torch.device("cuda")
    q, k, v = mha_inputs(1, 1, 512, 64, torch.float32, seed=81)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(dq)
    lse = torch.empty(1, 1, 512, dtype=torch.float32, device=dev)
    ws = torch.empty(pkg.attn_fwd_tf32x3_workspace_size(1, 1, 512, 64), dtype=torch.uint8,
                     device=dev)
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
    t0 = time.time()
    pkg.attn_fwd_tf32x3_test_skip_load(dq, dk, dv, o, lse, True, 0.125, ws, 1)
    code = pkg.attn_device_status(raise_on_error=False)
    elapsed = time.time() - t0
    assert code == pkg.ATTN_ERR_DEVICE_TIMEOUT, pkg.attn_last_error()
    assert "wait ran out" in pkg.attn_last_error()
    assert elapsed < 30
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
    o2, lse2 = pkg.attn_fwd_tf32x3(dq, dk, dv, causal=True, scale=0.125, workspace=ws)
    pkg.attn_device_status()
    ro, rl = oracle.mha(q, k, v, True, 0.125)
    assert np.abs(o2.cpu().numpy() - ro).max() <= 1e-4
    assert np.abs(lse2.cpu().numpy() - rl).max() <= 1e-4


@pytest.mark.parametrize("skip_block,N,B,H", [(0, 256, 1, 2), (2, 512, 1, 20)])
def test_stuck_f32_pipeline_reports_timeout_and_context_survives(skip_block, N, B, H):
    """fp32 attn_fwd (CUDA cores) with one K/V block never loaded, with the
    32-row and the 128-row blocks: every CTA's bounded wait on that block runs
    out (for block 0 also the second half's wait for the first half to start),
    the CTAs unwind, and the next call is correct."""
    dev = torch.device("cuda")
    q, k, v = mha_inputs(B, H, N, 64, torch.float32, seed=83 + skip_block)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(dq)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
    t0 = time.time()
    pkg.attn_fwd_f32_test_skip_load(dq, dk, dv, o, lse, False, 0.125, skip_block)
    code = pkg.attn_device_status(raise_on_error=False)
    elapsed = time.time() - t0
    assert code == pkg.ATTN_ERR_DEVICE_TIMEOUT, pkg.attn_last_error()
    assert "wait ran out" in pkg.attn_last_error()
    assert elapsed < 30
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
    o2, lse2 = pkg.attn_fwd(dq, dk, dv, causal=False, scale=0.125)
    pkg.attn_device_status()
    ro, rl = oracle.mha(q, k, v, False, 0.125)
    assert np.abs(o2.cpu().numpy() - ro).max() <= 1e-4
    assert np.abs(lse2.cpu().numpy() - rl).max() <= 1e-4


def test_f32_skip_hook_rejects_bad_index():
    dev = torch.device("cuda")
    z = torch.zeros(1, 1, 128, 64, dtype=torch.float32, device=dev)
    with pytest.raises(pkg.AttnError):
        pkg.attn_fwd_f32_test_skip_load(z, z, z, z.clone(), torch.empty(1, 1, 128, device=dev),
                                        False, 0.1, -1)


def test_stuck_decode_cluster_reports_timeout_and_context_survives():
    """mla_decode in which rank 1 of every cluster never loads its fourth
    step: rank 1 times out waiting for the page, rank 0 times out waiting for
    rank 1's partial scores, both CTAs of every pair meet at the final cluster
    barrier and free their tensor memory, and the next call is correct."""
    from online_softmax_attention_attn_gb300.inputs import mla_inputs
    dev = torch.device("cuda")
    lens = [512] * 64  # one chunk of 8 pages per sequence
    scale = 1.0 / math.sqrt(192.0)
    q, kv, table, sl = mla_inputs(len(lens), 128, lens, seed=82, paged_random=True)
    dq, dkv, dt, dsl = q.to(dev), kv.to(dev), table.to(dev), sl.to(dev)
    o = torch.empty(len(lens), 128, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(len(lens), 128, dtype=torch.float32, device=dev)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    ws = torch.empty(pkg.mla_decode_workspace_size(len(lens), 128, table.shape[1], nsm),
                     dtype=torch.uint8, device=dev)
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
    t0 = time.time()
    pkg.mla_decode_test_skip_load(dq, dkv, dt, dsl, o, lse, scale, ws, 3)
    code = pkg.attn_device_status(raise_on_error=False)
    elapsed = time.time() - t0
    assert code == pkg.ATTN_ERR_DEVICE_TIMEOUT, pkg.attn_last_error()
    assert "wait ran out" in pkg.attn_last_error()
    assert elapsed < 30
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
    o2, lse2 = pkg.mla_decode(dq, dkv, dt, dsl, scale=scale, workspace=ws)
    pkg.attn_device_status()
    ro, rl = oracle.mla(q, kv, table, sl, scale)
    assert np.abs(o2.float().cpu().numpy() - ro).max() <= 2e-2
    assert np.abs(lse2.cpu().numpy() - rl).max() <= 1e-3


def test_decode_and_tf32x3_skip_hooks_reject_bad_index():
    dev = torch.device("cuda")
    z = torch.zeros(1, 1, 128, 64, dtype=torch.float32, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    with pytest.raises(pkg.AttnError):
        pkg.attn_fwd_tf32x3_test_skip_load(z, z, z, z.clone(),
                                           torch.empty(1, 1, 128, device=dev), False, 0.1, ws,
                                           -1)
    qm = torch.zeros(1, 128, 576, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(1, 64, 576, dtype=torch.bfloat16, device=dev)
    table = torch.zeros(1, 1, dtype=torch.int32, device=dev)
    sl = torch.full((1,), 64, dtype=torch.int32, device=dev)
    with pytest.raises(pkg.AttnError):
        pkg.mla_decode_test_skip_load(qm, kv, table, sl,
                                      torch.empty(1, 128, 512, dtype=torch.bfloat16, device=dev),
                                      torch.empty(1, 128, device=dev), 0.1, ws, -1)
