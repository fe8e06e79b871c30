"""mla_decode_noalloc: the decode entry point for callers that cannot allocate.

Some callers may not allocate device memory at the moment they call (their
device memory is all handed to their own pool, or an allocation would
synchronise the device at a bad time), so they cannot pass mla_decode a
workspace.  mla_decode_noalloc runs the same kernels with the plan and split
partials in a fixed device array inside the library.  This test calls it
through the C ABI, twice in a row, and checks it against mla_decode (which
uses a caller workspace) and against the fp64 oracle, within the decode
tolerance.  It sits in its own
file, collected last, and passes alone in a fresh process or after the rest
of the suite.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_attention_attn_gb300 as pkg
from online_softmax_attention_attn_gb300.inputs import mla_inputs

pytestmark = pytest.mark.gpu

TOL_O, TOL_L = 2e-2, 1e-3


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice():
    L = pkg.lib()
    dev = torch.device("cuda")
    lens = [1, 64, 300, 1000, 4096, 2048, 0, 777]
    q, kv, table, sl = mla_inputs(len(lens), 128, lens, seed=70, paged_random=True)
    q, kv, table, sl = q.to(dev), kv.to(dev), table.to(dev), sl.to(dev)
    scale = 1.0 / math.sqrt(192.0)
    ref_o, ref_l = pkg.mla_decode(q, kv, table, sl, scale=scale)
    pkg.attn_device_status()
    ref_o, ref_l = ref_o.float().cpu().numpy(), ref_l.cpu().numpy()
    oro, orl = oracle.mla(q.cpu(), kv.cpu(), table.cpu(), sl.cpu(), scale)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        o = torch.full((len(lens), 128, 512), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((len(lens), 128), float("nan"), dtype=torch.float32, device=dev)
        rc = L.mla_decode_noalloc(_p(q), _p(kv), _p(table), _p(sl), _p(o), _p(lse),
                                  len(lens), 128, ctypes.c_float(scale), table.shape[1],
                                  kv.shape[0], stream)
        assert rc == pkg.ATTN_OK, pkg.attn_last_error()
        assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK
        go, gl = o.float().cpu().numpy(), lse.cpu().numpy()
        assert np.abs(go - ref_o).max() <= TOL_O
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isneginf(gl), np.isneginf(ref_l))
        assert np.abs(gl[fin] - ref_l[fin]).max() <= TOL_L
        # and against the fp64 oracle itself
        assert np.abs(go - oro).max() <= TOL_O
        assert np.array_equal(np.isneginf(gl), np.isneginf(orl))
        ofin = np.isfinite(orl)
        assert np.abs(gl[ofin] - orl[ofin]).max() <= TOL_L


def test_noalloc_calls_allocate_no_device_memory():
    """After a first call (which only looks up the scratch array's address),
    further calls leave the device's free memory unchanged: nothing is
    allocated per call, by the library or on its behalf."""
    L = pkg.lib()
    dev = torch.device("cuda")
    lens = [4096, 300, 0, 2000, 64, 1, 3000, 777]
    q, kv, table, sl = mla_inputs(len(lens), 128, lens, seed=71, paged_random=True)
    q, kv, table, sl = q.to(dev), kv.to(dev), table.to(dev), sl.to(dev)
    o = torch.empty(len(lens), 128, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(len(lens), 128, dtype=torch.float32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (_p(q), _p(kv), _p(table), _p(sl), _p(o), _p(lse), len(lens), 128,
            ctypes.c_float(1.0 / math.sqrt(192.0)), table.shape[1], kv.shape[0], stream)
    assert L.mla_decode_noalloc(*args) == pkg.ATTN_OK, pkg.attn_last_error()
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        assert L.mla_decode_noalloc(*args) == pkg.ATTN_OK, pkg.attn_last_error()
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after >= free_before, (free_before, free_after)
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK


def test_noalloc_rejects_batches_beyond_the_fixed_scratch():
    L = pkg.lib()
    dev = torch.device("cuda")
    buf = torch.empty(1024, dtype=torch.uint8, device=dev)
    p = _p(buf)
    rc = L.mla_decode_noalloc(p, p, p, p, p, p, 8193, 128, ctypes.c_float(0.1), 1, 1, None)
    assert rc == pkg.ATTN_ERR_UNSUPPORTED
    assert "8192" in pkg.attn_last_error()
