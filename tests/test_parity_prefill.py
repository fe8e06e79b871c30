"""GPU parity of attn_fwd (fp32 and bf16 paths) against the fp64 oracle.

Element-by-element on small and ragged shapes that span several tiles; at the
full workload sizes on sampled rows the oracle computes one by one, plus
properties that hold at any size (finite, convex combination of V rows).
Tolerances: fp32 path O and LSE within 1e-4; bf16 path O within 2e-2 and
LSE within 1e-3 (max abs error against the unrounded fp64 oracle).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_attention_attn_gb300 as pkg
from online_softmax_attention_attn_gb300.inputs import (BF16_PREFILL, FP32_PAGE2,
                                                         FP32_SMALL_CAUSAL, mha_inputs,
                                                         mha_config_inputs)

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-4, 1e-4), torch.bfloat16: (2e-2, 1e-3)}


def _run(q, k, v, causal, scale):
    dev = torch.device("cuda")
    o, lse = pkg.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    pkg.attn_device_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _check_full(q, k, v, causal, scale):
    o, lse = _run(q, k, v, causal, scale)
    ro, rl = oracle.mha(q, k, v, causal, scale)
    to, tl = TOL[q.dtype]
    eo, el = np.abs(o - ro).max(), np.abs(lse - rl).max()
    assert eo <= to and el <= tl, f"O err {eo:.3g}, LSE err {el:.3g}"
    return eo, el


def _sample_rows(B, H, N, n, seed):
    rng = np.random.default_rng(seed)
    rows = set()
    for bh in (0, B * H - 1):
        for i in (0, 1, 127, 128, N // 2, N - 129, N - 128, N - 1):
            if 0 <= i < N:
                rows.add(bh * N + i)
    rows.update(rng.integers(0, B * H * N, size=n).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def _check_sampled(q, k, v, causal, scale, o, lse, nrows=384, seed=0):
    B, H, N, D = q.shape
    rows = _sample_rows(B, H, N, nrows, seed)
    ro, rl = oracle.mha(q, k, v, causal, scale, rows=rows)
    go = o.reshape(-1, D)[rows]
    gl = lse.reshape(-1)[rows]
    to, tl = TOL[q.dtype]
    eo, el = np.abs(go - ro).max(), np.abs(gl - rl).max()
    assert eo <= to and el <= tl, f"O err {eo:.3g}, LSE err {el:.3g}"
    # properties at every row: finite, and O inside the hull of the V rows
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    vmin = v.float().amin(dim=2).numpy()[:, :, None, :]
    vmax = v.float().amax(dim=2).numpy()[:, :, None, :]
    slack = to
    assert (o.reshape(B, H, N, D) >= vmin - slack).all()
    assert (o.reshape(B, H, N, D) <= vmax + slack).all()


# ------------------------------------------------------------------ fp32

def test_fp32_small_causal_workload():
    cfg = FP32_SMALL_CAUSAL
    q, k, v = mha_config_inputs(cfg)
    _check_full(q, k, v, cfg.causal, cfg.scale)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 64, 200, 321])
def test_fp32_ragged(N, causal):
    q, k, v = mha_inputs(2, 3, N, 64, torch.float32, seed=200 + N)
    _check_full(q, k, v, causal, 0.125)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [200, 321])
def test_fp32_ragged_large_grid(N, causal):
    """Enough (head, 128-row block) pairs to fill half the SMs, so the kernel
    runs with 128-row blocks (the small cases above get 32-row blocks)."""
    q, k, v = mha_inputs(4, 20, N, 64, torch.float32, seed=250 + N)
    _check_full(q, k, v, causal, 0.125)


def test_fp32_scale_zero_gives_prefix_means():
    q, k, v = mha_inputs(1, 2, 300, 64, torch.float32, seed=5)
    o, lse = _run(q, k, v, True, 0.0)
    ref = (torch.cumsum(v.double(), 2) / torch.arange(1, 301).double()[None, None, :, None])
    assert np.abs(o - ref.numpy()).max() <= 1e-5
    assert np.abs(lse - np.log(np.arange(1, 301))[None, None]).max() <= 1e-5


@pytest.mark.parametrize("causal", [False, True])
def test_fp32_page2_workload_sampled(causal):
    cfg = FP32_PAGE2
    q, k, v = mha_config_inputs(cfg)
    o, lse = _run(q, k, v, causal, cfg.scale)
    _check_sampled(q, k, v, causal, cfg.scale, o, lse, seed=int(causal))


# ------------------------------------------------------------------ bf16

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 256, 300, 513])
def test_bf16_d128_small_and_ragged(N, causal):
    q, k, v = mha_inputs(2, 2, N, 128, torch.bfloat16, seed=300 + N)
    _check_full(q, k, v, causal, 1.0 / math.sqrt(128))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [64, 256, 389])
def test_bf16_d64(N, causal):
    q, k, v = mha_inputs(2, 3, N, 64, torch.bfloat16, seed=400 + N)
    _check_full(q, k, v, causal, 0.125)


def test_bf16_long_rows_exercise_lazy_rescale():
    """Scores with a growing trend force the running max up many times."""
    B, H, N, D = 1, 2, 1024, 128
    q, k, v = mha_inputs(B, H, N, D, torch.float32, seed=9)
    k = k + torch.linspace(0, 6, N)[None, None, :, None] * q.mean(2, keepdim=True).sign()
    _check_full(q.bfloat16(), k.bfloat16(), v.bfloat16(), True, 0.5)


def test_bf16_sudden_max_jump_inside_a_block():
    """Keys 192..255 score far above everything before them: the second half of
    KV block 1 moves the running reference, so O (holding block 0 and the
    first half of block 1) is rescaled after that half's PV has landed."""
    B, H, N, D = 1, 2, 512, 128
    q, k, v = mha_inputs(B, H, N, D, torch.float32, seed=21)
    q = q + 0.5                   # a component every query shares ...
    k[:, :, 192:256, :] += 1.5    # ... lifts these keys by ~12 in log2 units
    for causal in (False, True):
        _check_full(q.bfloat16(), k.bfloat16(), v.bfloat16(), causal, 1.0 / math.sqrt(D))


@pytest.mark.parametrize("scale", [0.0, -0.05])
def test_bf16_zero_and_negative_scale(scale):
    """A zero scale gives plain means; a negative one flips the max to a min:
    both bypass the fast path's assumptions."""
    q, k, v = mha_inputs(1, 2, 300, 128, torch.bfloat16, seed=23)
    for causal in (False, True):
        _check_full(q, k, v, causal, scale)


def test_bf16_prefill_workload_sampled():
    cfg = BF16_PREFILL
    q, k, v = mha_config_inputs(cfg)
    o, lse = _run(q, k, v, cfg.causal, cfg.scale)
    _check_sampled(q, k, v, cfg.causal, cfg.scale, o, lse, nrows=512, seed=3)


def test_bf16_repeat_calls_are_bitwise_identical():
    q, k, v = mha_inputs(2, 4, 700, 128, torch.bfloat16, seed=11)
    a = _run(q, k, v, True, 0.09)
    b = _run(q, k, v, True, 0.09)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------------ persistent schedule

@pytest.mark.parametrize("causal", [False, True])
def test_bf16_many_items_per_cta(causal):
    """192 heads x 2 Q-tile pairs = 384 work items on ~150 persistent CTAs; the
    second pair of every head has no second tile (N = 3 tiles of 128)."""
    B, H, N, D = 4, 48, 384, 128
    q, k, v = mha_inputs(B, H, N, D, torch.bfloat16, seed=31 + int(causal))
    o, lse = _run(q, k, v, causal, 1.0 / math.sqrt(D))
    _check_sampled(q, k, v, causal, 1.0 / math.sqrt(D), o, lse, nrows=768, seed=7)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_item_boundaries_every_row(causal):
    """200 heads (full head groups plus a short last one) x 2 Q-tile pairs
    with a ragged last tile (N = 500): 400 work items, two or three per
    persistent CTA, so the next item's Q_0 load, the early claim and the L2
    prefetch of K/V all cross item boundaries; every output row is checked."""
    q, k, v = mha_inputs(2, 100, 500, 128, torch.bfloat16, seed=61 + int(causal))
    _check_full(q, k, v, causal, 1.0 / math.sqrt(128))


def test_bf16_more_launches_than_ticket_slots():
    """Each launch draws its items from one of a fixed set of counters; many
    launches in a row reuse them and every result stays the same."""
    q, k, v = mha_inputs(2, 8, 640, 128, torch.bfloat16, seed=41)
    dev = torch.device("cuda")
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    o0, l0 = pkg.attn_fwd(dq, dk, dv, causal=True, scale=0.1)
    o, l = torch.empty_like(o0), torch.empty_like(l0)
    for _ in range(150):
        pkg.attn_fwd(dq, dk, dv, o, l, causal=True, scale=0.1)
    pkg.attn_device_status()
    assert torch.equal(o, o0) and torch.equal(l, l0)
    ro, rl = oracle.mha(q, k, v, True, 0.1, rows=np.arange(0, 2 * 8 * 640, 97))
    assert np.abs(o0.float().cpu().numpy().reshape(-1, 128)[::97] - ro).max() <= 2e-2
    assert np.abs(l0.cpu().numpy().reshape(-1)[::97] - rl).max() <= 1e-3


def test_bf16_two_streams_at_once():
    """Launches on two streams may run together; each has its own counter."""
    dev = torch.device("cuda")
    qa, ka, va = (t.to(dev) for t in mha_inputs(2, 16, 1024, 128, torch.bfloat16, seed=43))
    qb, kb, vb = (t.to(dev) for t in mha_inputs(2, 16, 1024, 128, torch.bfloat16, seed=44))
    ra = pkg.attn_fwd(qa, ka, va, causal=True)
    rb = pkg.attn_fwd(qb, kb, vb, causal=False)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(5):
        with torch.cuda.stream(sa):
            oa = pkg.attn_fwd(qa, ka, va, causal=True)
        with torch.cuda.stream(sb):
            ob = pkg.attn_fwd(qb, kb, vb, causal=False)
        torch.cuda.synchronize()
        pkg.attn_device_status()
        assert torch.equal(oa[0], ra[0]) and torch.equal(oa[1], ra[1])
        assert torch.equal(ob[0], rb[0]) and torch.equal(ob[1], rb[1])
