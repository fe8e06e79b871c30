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
