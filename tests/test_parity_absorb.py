"""GPU parity of the projections around MLA decode against the fp64 oracle.

mla_absorb_q and mla_project_out are per-head bf16 GEMMs with fp32
accumulation and a bf16 result: each output may differ from the exact value
by its own bf16 rounding (2^-9 relative) plus accumulation-order noise, so the
bound is 2^-8 |ref| + 1e-4 max|ref|.  The rotary part of the absorbed query is
copied, so it must match bit for bit.  The whole layer (absorb -> mla_decode ->
project) is checked against attention over explicitly decompressed keys and
values (the absorption identity), with the bf16 tolerances of the decode
widened for the rounded absorbed query: O within 2e-2 of max |ref|, LSE
within 5e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_attention_attn_gb300 as pkg
from online_softmax_attention_attn_gb300.inputs import mla_layer_inputs

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192.0)


def _close_gemm(got, ref):
    got = got.float().cpu().numpy().astype(np.float64)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * np.abs(ref).max()
    worst = float((np.abs(got - ref) - bound).max())
    assert worst <= 0.0, f"exceeds the bound by {worst:.3g}"


def test_absorb_q_matches_oracle():
    qn, qr, wk, _, _, _, _ = mla_layer_inputs(64, 128, [64] * 64, seed=51)
    dev = torch.device("cuda")
    qa = pkg.mla_absorb_q(qn.to(dev), qr.to(dev), wk.to(dev))
    pkg.attn_device_status()
    ref = oracle.mla_absorb_q(qn, qr, wk)
    _close_gemm(qa[:, :, :512], ref[:, :, :512])
    assert torch.equal(qa[:, :, 512:].cpu(), qr)


def test_project_out_matches_oracle():
    _, _, _, wv, _, _, _ = mla_layer_inputs(64, 128, [64] * 64, seed=52)
    g = torch.Generator().manual_seed(53)
    ol = (torch.randn(64, 128, 512, generator=g) * 0.5).to(torch.bfloat16)
    dev = torch.device("cuda")
    out = pkg.mla_project_out(ol.to(dev), wv.to(dev))
    pkg.attn_device_status()
    _close_gemm(out, oracle.mla_project_out(ol, wv))


def test_into_caller_buffers_and_odd_batch():
    """Outputs written into given tensors; a batch that is no multiple of anything."""
    qn, qr, wk, wv, _, _, _ = mla_layer_inputs(7, 128, [64] * 7, seed=54)
    dev = torch.device("cuda")
    qa = torch.full((7, 128, 576), float("nan"), dtype=torch.bfloat16, device=dev)
    pkg.mla_absorb_q(qn.to(dev), qr.to(dev), wk.to(dev), q_out=qa)
    out = torch.full((7, 128, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    ol = qa[:, :, :512].contiguous()
    pkg.mla_project_out(ol, wv.to(dev), out=out)
    pkg.attn_device_status()
    _close_gemm(qa[:, :, :512], oracle.mla_absorb_q(qn, qr, wk)[:, :, :512])
    _close_gemm(out, oracle.mla_project_out(ol.cpu(), wv))


def test_layer_matches_decompressed_attention():
    """absorb -> latent attention -> value projection equals attention over the
    decompressed keys [c W_UK^T | k_rope] and values c W_UV (article's identity)."""
    lens = [1, 65, 200, 377]
    qn, qr, wk, wv, kv, table, sl = mla_layer_inputs(4, 128, lens, seed=55, paged_random=True)
    dev = torch.device("cuda")
    qa = pkg.mla_absorb_q(qn.to(dev), qr.to(dev), wk.to(dev))
    ol, lse = pkg.mla_decode(qa, kv.to(dev), table.to(dev), sl.to(dev), scale=SCALE)
    out = pkg.mla_project_out(ol, wv.to(dev))
    pkg.attn_device_status()
    ref, rlse = oracle.mla_decompressed(qn, qr, wk, wv, kv, table, sl, SCALE)
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max()
    assert np.abs(lse.cpu().numpy() - rlse).max() <= 5e-3
