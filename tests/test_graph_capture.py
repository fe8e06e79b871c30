"""The bf16 prefill inside a captured CUDA graph.

The persistent prefill kernel draws its work items from a counter that the
call zeroes on its stream.  A call made while the stream is being captured
gets a counter no other call uses, so replays of the graph stay correct
while ordinary launches (which take the shared counters in turn) run at the
same time on another stream.  Checked against the fp64 oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_attention_attn_gb300 as pkg
from online_softmax_attention_attn_gb300.inputs import mha_inputs

pytestmark = pytest.mark.gpu

TOL_O, TOL_L = 2e-2, 1e-3


def _err(o, lse, ro, rl):
    return (float(np.abs(o.float().cpu().numpy() - ro).max()),
            float(np.abs(lse.cpu().numpy() - rl).max()))


def test_captured_prefill_replays_beside_ordinary_launches():
    dev = torch.device("cuda")
    q, k, v = mha_inputs(2, 4, 700, 128, torch.bfloat16, seed=90)
    q2, k2, v2 = mha_inputs(1, 8, 1000, 128, torch.bfloat16, seed=91)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    dq2, dk2, dv2 = q2.to(dev), k2.to(dev), v2.to(dev)
    o = torch.empty_like(dq)
    lse = torch.empty(2, 4, 700, dtype=torch.float32, device=dev)
    o2 = torch.empty_like(dq2)
    lse2 = torch.empty(1, 8, 1000, dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(128)

    # warm-up outside the capture (first-call set-up of the library)
    pkg.attn_fwd(dq, dk, dv, o, lse, causal=True, scale=scale)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        pkg.attn_fwd(dq, dk, dv, o, lse, causal=True, scale=scale)
    ro, rl = oracle.mha(q, k, v, True, scale)
    ro2, rl2 = oracle.mha(q2, k2, v2, False, scale)

    other = torch.cuda.Stream()
    for _ in range(3):
        o.zero_()
        o2.zero_()
        torch.cuda.synchronize()
        graph.replay()
        with torch.cuda.stream(other):
            # ordinary launches drawing the shared counters in turn, enqueued
            # while the replay may still run
            for _ in range(3):
                pkg.attn_fwd(dq2, dk2, dv2, o2, lse2, causal=False, scale=scale)
        torch.cuda.synchronize()
        assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
        eo, el = _err(o, lse, ro, rl)
        assert eo <= TOL_O and el <= TOL_L, (eo, el)
        eo2, el2 = _err(o2, lse2, ro2, rl2)
        assert eo2 <= TOL_O and el2 <= TOL_L, (eo2, el2)
