"""GPU parity of attn_fwd_tf32x3 (fp32 attention on tcgen05 kind::tf32 with
the three-product split) against the fp64 oracle.

The bound is the fp32 one: O and LSE within 1e-4 (max abs error against the
unrounded fp64 oracle).  A single TF32 product would miss it (10 explicit
mantissa bits: relative errors near 5e-4 in every score); with the split the
dropped terms are below 2^-21 of each product.  Element by element on small
and ragged shapes that span several tiles and a ragged tail; at the blog's
full workload on sampled rows, plus properties that hold at any size.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_attention_attn_gb300 as pkg
from online_softmax_attention_attn_gb300.inputs import (FP32_PAGE2, FP32_SMALL_CAUSAL,
                                                         mha_config_inputs, mha_inputs)

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 1e-4, 1e-4


def _run(q, k, v, causal, scale, workspace=None):
    dev = torch.device("cuda")
    o, lse = pkg.attn_fwd_tf32x3(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale,
                                 workspace=workspace)
    pkg.attn_device_status()
    return o.cpu().numpy(), lse.cpu().numpy()


def _check_full(q, k, v, causal, scale):
    o, lse = _run(q, k, v, causal, scale)
    ro, rl = oracle.mha(q, k, v, causal, scale)
    eo, el = np.abs(o - ro).max(), np.abs(lse - rl).max()
    assert eo <= TOL_O and el <= TOL_LSE, f"O err {eo:.3g}, LSE err {el:.3g}"


def _sample_rows(B, H, N, n, seed):
    rng = np.random.default_rng(seed)
    rows = set()
    for bh in (0, B * H - 1):
        for i in (0, 1, 63, 64, 127, 128, N // 2, N - 129, N - 128, N - 1):
            if 0 <= i < N:
                rows.add(bh * N + i)
    rows.update(rng.integers(0, B * H * N, size=n).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def test_small_causal_workload():
    cfg = FP32_SMALL_CAUSAL
    q, k, v = mha_config_inputs(cfg)
    _check_full(q, k, v, cfg.causal, cfg.scale)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 64, 65, 128, 200, 321, 700])
def test_ragged(N, causal):
    q, k, v = mha_inputs(2, 3, N, 64, torch.float32, seed=300 + N)
    _check_full(q, k, v, causal, 0.125)


def test_scale_zero_gives_prefix_means():
    q, k, v = mha_inputs(1, 2, 300, 64, torch.float32, seed=6)
    o, lse = _run(q, k, v, True, 0.0)
    ref = (torch.cumsum(v.double(), 2) / torch.arange(1, 301).double()[None, None, :, None])
    assert np.abs(o - ref.numpy()).max() <= 1e-5
    assert np.abs(lse - np.log(np.arange(1, 301))[None, None]).max() <= 1e-5


def test_negative_scale():
    q, k, v = mha_inputs(1, 2, 260, 64, torch.float32, seed=7)
    for causal in (False, True):
        _check_full(q, k, v, causal, -0.1)


def test_long_rows_exercise_lazy_rescale():
    """Scores with a growing trend force the running max up many times."""
    q, k, v = mha_inputs(1, 2, 1024, 64, torch.float32, seed=10)
    k = k + torch.linspace(0, 6, 1024)[None, None, :, None] * q.mean(2, keepdim=True).sign()
    _check_full(q, k, v, True, 0.5)
    _check_full(q, k, v, False, 0.5)


def test_sudden_max_jump_in_a_later_block():
    """Keys 192..255 score far above the earlier ones: O, holding blocks 0-2,
    is rescaled once PV of block 2 has landed."""
    q, k, v = mha_inputs(1, 2, 512, 64, torch.float32, seed=22)
    q = q + 0.5
    k[:, :, 192:256, :] += 1.5
    for causal in (False, True):
        _check_full(q, k, v, causal, 1.0 / math.sqrt(64))


def test_large_magnitude_inputs_keep_fp32_accuracy():
    """|q|, |k| ~ 8: scores reach hundreds, so the split's low parts matter."""
    q, k, v = mha_inputs(1, 2, 384, 64, torch.float32, seed=23)
    _check_full(q * 8, k * 8, v, False, 1.0 / 64)


def test_repeat_calls_with_one_workspace_are_bitwise_identical():
    q, k, v = mha_inputs(2, 2, 333, 64, torch.float32, seed=24)
    dev = torch.device("cuda")
    ws = torch.empty(pkg.attn_fwd_tf32x3_workspace_size(2, 2, 333, 64), dtype=torch.uint8,
                     device=dev)
    ws.fill_(0xFF)  # NaN bit patterns: every byte the kernel reads must be written first
    a = _run(q, k, v, True, 0.125, workspace=ws)
    b = _run(q, k, v, True, 0.125, workspace=ws)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.isfinite(a[0]).all()


def test_too_small_workspace_is_refused():
    q, k, v = mha_inputs(1, 1, 64, 64, torch.float32, seed=25)
    dev = torch.device("cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device=dev)
    with pytest.raises(pkg.AttnError) as e:
        pkg.attn_fwd_tf32x3(q.to(dev), k.to(dev), v.to(dev), workspace=ws)
    assert e.value.code == pkg.ATTN_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("causal", [False, True])
def test_blog_workload_sampled(causal):
    """B4 H8 N8192 D64 fp32 (the blog's section 4.1 workload), sampled rows."""
    cfg = FP32_PAGE2
    q, k, v = mha_config_inputs(cfg)
    o, lse = _run(q, k, v, causal, cfg.scale)
    B, H, N, D = q.shape
    rows = _sample_rows(B, H, N, 384, seed=10 + int(causal))
    ro, rl = oracle.mha(q, k, v, causal, cfg.scale, rows=rows)
    eo = np.abs(o.reshape(-1, D)[rows] - ro).max()
    el = np.abs(lse.reshape(-1)[rows] - rl).max()
    assert eo <= TOL_O and el <= TOL_LSE, f"O err {eo:.3g}, LSE err {el:.3g}"
    # every row: finite, and O inside the hull of the V rows
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    vmin = v.amin(dim=2).numpy()[:, :, None, :]
    vmax = v.amax(dim=2).numpy()[:, :, None, :]
    assert (o >= vmin - TOL_O).all() and (o <= vmax + TOL_O).all()


@pytest.mark.parametrize("causal", [False, True])
def test_heads_in_a_ragged_last_group(causal):
    """15 heads: tiles are scheduled in groups of 8 heads, the last group has 7."""
    q, k, v = mha_inputs(3, 5, 200, 64, torch.float32, seed=26)
    _check_full(q, k, v, causal, 0.125)
