"""GPU checks of the host-buffer entry points.

attn_fwd_host and mla_decode_host run the same kernels on the same inputs as
attn_fwd and mla_decode, so their outputs must be bit-for-bit the device
entry points' (the host path only adds copies and chunking by whole heads),
and within the oracle's tolerances.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_attention_attn_gb300 as pkg
from online_softmax_attention_attn_gb300.inputs import mha_inputs, mla_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,D,dtype,causal", [
    (2, 3, 300, 128, torch.bfloat16, True),    # 6 heads -> 3 chunks of 2
    (1, 1, 200, 128, torch.bfloat16, False),   # one chunk
    (3, 3, 129, 64, torch.bfloat16, True),     # 9 heads -> 3 chunks of 3
    (1, 5, 200, 64, torch.float32, True),      # fp32, 5 heads -> 3 chunks of 2
])
def test_attn_fwd_host_matches_device_entry(B, H, N, D, dtype, causal):
    q, k, v = mha_inputs(B, H, N, D, torch.float32, seed=400 + N)
    q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    hq, hk, hv = (t.contiguous().pin_memory() for t in (q, k, v))
    scale = 1.0 / math.sqrt(D)
    ho, hl = pkg.attn_fwd_host(hq, hk, hv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    pkg.attn_device_status()
    dev = torch.device("cuda")
    do, dl = pkg.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    pkg.attn_device_status()
    assert torch.equal(ho, do.cpu()) and torch.equal(hl, dl.cpu())
    ro, rl = oracle.mha(q, k, v, causal, scale)
    to, tl = (1e-4, 1e-4) if dtype == torch.float32 else (2e-2, 1e-3)
    assert np.abs(ho.float().numpy() - ro).max() <= to
    assert np.abs(hl.numpy() - rl).max() <= tl


def test_attn_fwd_host_repeated_calls_reuse_one_workspace():
    q, k, v = mha_inputs(2, 4, 256, 128, torch.bfloat16, seed=41)
    hq, hk, hv = (t.contiguous().pin_memory() for t in (q, k, v))
    need = pkg.attn_fwd_host_workspace_size(2, 4, 256, 128, pkg.ATTN_DTYPE_BF16)
    raw = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    off = (-raw.data_ptr()) % 256
    ws = raw[off:off + need]
    outs = []
    for _ in range(3):
        o, l = pkg.attn_fwd_host(hq, hk, hv, causal=True, workspace=ws)
        outs.append((o, l))
    torch.cuda.synchronize()
    pkg.attn_device_status()
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_mla_decode_host_matches_device_entry():
    lens = [64, 100, 1, 0, 4096, 777]
    q, kv, table, sl = mla_inputs(len(lens), 128, lens, seed=44, paged_random=True)
    scale = 1.0 / math.sqrt(192.0)
    hq, hkv, ht, hs = (t.contiguous().pin_memory() for t in (q, kv, table, sl))
    ho, hl = pkg.mla_decode_host(hq, hkv, ht, hs, scale=scale)
    torch.cuda.synchronize()
    pkg.attn_device_status()
    dev = torch.device("cuda")
    do, dl = pkg.mla_decode(q.to(dev), kv.to(dev), table.to(dev), sl.to(dev), scale=scale)
    pkg.attn_device_status()
    assert torch.equal(ho, do.cpu()) and torch.equal(hl, dl.cpu())
