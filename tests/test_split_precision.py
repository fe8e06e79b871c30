"""The precision premise of fp32 attention on the tensor cores, checked on the CPU.

attn_fwd_tf32x3 rounds its operands to TF32 (10 explicit mantissa bits) and
recovers fp32 accuracy with a three-product split: x = hi + lo,
hi = x rounded to TF32, lo = x - hi, x*y ~ lo*hi + hi*lo + hi*hi.  In Q K^T all
three products are TF32; in P V the two cross terms run on bf16 operands.
These tests replay that arithmetic in numpy (products exact in float64, the
operands rounded as the kernel rounds them) against exact float64 attention
on inputs whose scores reach tens of units, and check the claims the design
rests on: one TF32 product misses the fp32 bound of 1e-4 on O and LSE, the
split meets it, and the bf16 cross terms in P V cost far less than the bound.
"""
import numpy as np
import pytest
import torch

from online_softmax_attention_attn_gb300.inputs import mha_inputs


def tf32(x):
    """Nearest TF32 value, ties away from zero (add half a TF32 unit to the
    bits, clear the 13 low ones), as the kernels round."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x1000) & 0xFFFFE000).astype(np.uint32).view(np.float32)


def bf16(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.bfloat16().float().numpy()


def f64(x):
    return np.asarray(x, dtype=np.float64)


def scores(q, k, mode):
    if mode == "exact":
        return f64(q) @ f64(k).T
    qh, kh = tf32(q), tf32(k)
    if mode == "tf32":
        return f64(qh) @ f64(kh).T
    ql, kl = tf32(q - qh), tf32(k - kh)
    return f64(ql) @ f64(kh).T + f64(qh) @ f64(kl).T + f64(qh) @ f64(kh).T


def attention(s, v, scale, causal, pv_mode):
    n = s.shape[0]
    t = s * scale
    if causal:
        t = np.where(np.tril(np.ones((n, n), dtype=bool)), t, -np.inf)
    m = t.max(axis=1, keepdims=True)
    p = np.exp(t - m).astype(np.float32)  # P in fp32, as the kernel holds it
    l = f64(p).sum(axis=1, keepdims=True)
    if pv_mode == "exact":
        pv = f64(p) @ f64(v)
    elif pv_mode == "tf32":
        pv = f64(tf32(p)) @ f64(tf32(v))
    else:  # the kernel: hi x hi in TF32, the cross terms on bf16 operands
        ph, vh = tf32(p), tf32(v)
        pv = (f64(ph) @ f64(vh) + f64(bf16(p - ph)) @ f64(bf16(v))
              + f64(bf16(p)) @ f64(bf16(v - vh)))
    return pv / l, (m + np.log(l))[:, 0]


@pytest.fixture(scope="module")
def large_inputs():
    """Scores of tens of units: |q|, |k| ~ 8, D = 64, scale 1/64."""
    q, k, v = mha_inputs(1, 1, 256, 64, torch.float32, seed=23)
    return (q[0, 0].numpy() * 8, k[0, 0].numpy() * 8, v[0, 0].numpy(), 1.0 / 64)


@pytest.mark.parametrize("causal", [False, True])
def test_one_tf32_product_misses_the_fp32_bound(large_inputs, causal):
    q, k, v, scale = large_inputs
    oe, le = attention(scores(q, k, "exact"), v, scale, causal, "exact")
    o1, l1 = attention(scores(q, k, "tf32"), v, scale, causal, "tf32")
    assert max(np.abs(o1 - oe).max(), np.abs(l1 - le).max()) > 1e-4


@pytest.mark.parametrize("causal", [False, True])
def test_the_split_meets_the_fp32_bound(large_inputs, causal):
    q, k, v, scale = large_inputs
    oe, le = attention(scores(q, k, "exact"), v, scale, causal, "exact")
    o3, l3 = attention(scores(q, k, "split"), v, scale, causal, "split")
    # a tenth of the bound: the margin the kernel's own fp32 sums draw on
    assert np.abs(o3 - oe).max() <= 1e-5
    assert np.abs(l3 - le).max() <= 1e-5


def test_bf16_cross_terms_in_pv_cost_far_below_the_bound(large_inputs):
    q, k, v, scale = large_inputs
    s = scores(q, k, "exact")
    oe, _ = attention(s, v, scale, False, "exact")
    ob, _ = attention(s, v, scale, False, "split")
    assert np.abs(ob - oe).max() <= 1e-5


def test_tf32_rounding_is_nearest_on_the_tf32_grid():
    """The rounding rule itself: a value already on the grid is unchanged, the
    result differs from x by at most half a TF32 unit, and halfway cases go
    away from zero."""
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * 10.0 ** rng.uniform(-3, 3, 100000)).astype(np.float32)
    h = tf32(x)
    assert np.array_equal(tf32(h), h)
    assert (h.view(np.uint32) & 0x1FFF == 0).all()
    ulp = np.ldexp(np.ones_like(x, dtype=np.float64), np.frexp(np.abs(f64(x)))[1] - 11)
    assert (np.abs(f64(h) - f64(x)) <= 0.5 * ulp * (1 + 1e-12)).all()
    half = np.float32(1.0 + 2.0 ** -11)  # exactly halfway between 1 and 1 + 2^-10
    assert tf32(np.array([half]))[0] == np.float32(1.0 + 2.0 ** -10)
    assert tf32(np.array([-half]))[0] == np.float32(-(1.0 + 2.0 ** -10))
