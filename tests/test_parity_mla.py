"""GPU parity of mla_decode against the fp64 oracle, plus paging, split and
edge-case properties.  Tolerance: O within 2e-2, LSE within 1e-3 (max abs
error against the unrounded fp64 oracle)."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_attention_attn_gb300 as pkg
from online_softmax_attention_attn_gb300.inputs import (MLA_B16, MLA_B64, MLA_B128, MLA_B256,
                                                         MLA_B256_PAGED,
                                                         mla_config_inputs, mla_inputs)

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192.0)
TOL_O, TOL_L = 2e-2, 1e-3


def _gpu(q, kv, table, sl, pages_per_split=0, scale=SCALE):
    d = torch.device("cuda")
    o, lse = pkg.mla_decode_split(q.to(d), kv.to(d), table.to(d), sl.to(d), scale=scale,
                                  pages_per_split=pages_per_split)
    pkg.attn_device_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _check(q, kv, table, sl, o, lse, rows=None, scale=SCALE):
    ro, rl = oracle.mla(q, kv, table, sl, scale, rows=rows)
    if rows is not None:
        o = o.reshape(-1, 512)[rows]
        lse = lse.reshape(-1)[rows]
    fin = np.isfinite(rl)
    eo = np.abs(o - ro).max()
    el = np.abs(lse[fin] - rl[fin]).max() if fin.any() else 0.0
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl))
    assert eo <= TOL_O and el <= TOL_L, f"O err {eo:.3g}, LSE err {el:.3g}"


@pytest.mark.parametrize("paged", [False, True])
def test_small_uniform(paged):
    q, kv, table, sl = mla_inputs(2, 128, [64, 128], seed=50, paged_random=paged)
    o, lse = _gpu(q, kv, table, sl)
    _check(q, kv, table, sl, o, lse)


def test_ragged_lengths_and_page_tails():
    lens = [1, 31, 32, 33, 63, 64, 65, 100, 200, 257]
    q, kv, table, sl = mla_inputs(len(lens), 128, lens, seed=51, paged_random=True,
                                  max_blocks=6, num_blocks=80)
    o, lse = _gpu(q, kv, table, sl)
    _check(q, kv, table, sl, o, lse)


@pytest.mark.parametrize("pps", [1, 2, 3, 5])
def test_forced_splits(pps):
    lens = [1, 64, 130, 300, 511, 64 * 9]
    q, kv, table, sl = mla_inputs(len(lens), 128, lens, seed=52, paged_random=True,
                                  max_blocks=9, num_blocks=64)
    o, lse = _gpu(q, kv, table, sl, pages_per_split=pps)
    _check(q, kv, table, sl, o, lse)
    o0, l0 = _gpu(q, kv, table, sl, pages_per_split=0)
    assert np.abs(o - o0).max() <= 2 * TOL_O
    assert np.abs(lse - l0).max() <= 2 * TOL_L


def test_empty_sequences():
    q, kv, table, sl = mla_inputs(4, 128, [0, 50, 0, 64], seed=53, paged_random=True)
    o, lse = _gpu(q, kv, table, sl)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(o[2] == 0) and np.all(np.isneginf(lse[2]))
    _check(q, kv, table, sl, o, lse)


def test_all_empty():
    q, kv, table, sl = mla_inputs(3, 128, [0, 0, 0], seed=54, max_blocks=1)
    o, lse = _gpu(q, kv, table, sl)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_page_permutation_is_bitwise_invariant():
    """Moving pages in the pool with a matching block table changes no bit."""
    lens = [70, 200, 129]
    q, kv, table, sl = mla_inputs(3, 128, lens, seed=55, max_blocks=4, num_blocks=12)
    perm = torch.randperm(kv.shape[0], generator=torch.Generator().manual_seed(4))
    inv = torch.argsort(perm)
    kv2 = kv[perm].contiguous()
    table2 = inv[table.long()].to(torch.int32).contiguous()
    a = _gpu(q, kv, table, sl)
    b = _gpu(q, kv2, table2, sl)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_non_finite_page_tail_is_ignored():
    """Tokens past the end weigh exactly zero even if the tail holds NaN/Inf."""
    lens = [40, 100]
    q, kv, table, sl = mla_inputs(2, 128, lens, seed=56, max_blocks=2)
    clean = _gpu(q, kv, table, sl)
    kv2 = kv.clone()
    kv2[table[0, 0], 40:] = float("nan")
    kv2[table[1, 1], 100 - 64:] = float("inf")
    dirty = _gpu(q, kv2, table, sl)
    assert np.array_equal(clean[0], dirty[0]) and np.array_equal(clean[1], dirty[1])


def test_scale_zero_is_mean_of_latent_prefix():
    q, kv, table, sl = mla_inputs(2, 128, [64, 150], seed=57, paged_random=True)
    o, lse = _gpu(q, kv, table, sl, scale=0.0)
    for b, L in enumerate([64, 150]):
        idx = torch.arange(L)
        C = kv[table[b, idx // 64].long(), idx % 64].double()
        ref = C[:, :512].mean(0).numpy()
        assert np.abs(o[b] - ref[None]).max() <= 2e-3
        assert np.abs(lse[b] - math.log(L)).max() <= 1e-4


def test_bad_block_table_is_reported_not_faulted():
    q, kv, table, sl = mla_inputs(2, 128, [64, 64], seed=58, max_blocks=1)
    bad = table.clone()
    bad[1, 0] = 10_000
    d = torch.device("cuda")
    pkg.mla_decode(q.to(d), kv.to(d), bad.to(d), sl.to(d), scale=SCALE)
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_ERR_BAD_BLOCK_TABLE
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_OK  # cleared


def test_bad_seqlen_is_reported():
    q, kv, table, sl = mla_inputs(2, 128, [64, 64], seed=59, max_blocks=1)
    sl2 = torch.tensor([64, 65], dtype=torch.int32)
    d = torch.device("cuda")
    pkg.mla_decode(q.to(d), kv.to(d), table.to(d), sl2.to(d), scale=SCALE)
    assert pkg.attn_device_status(raise_on_error=False) == pkg.ATTN_ERR_BAD_SEQLEN


def test_repeat_calls_bitwise_identical():
    q, kv, table, sl = mla_inputs(5, 128, [300, 7, 64, 128, 1000], seed=60, paged_random=True)
    a = _gpu(q, kv, table, sl)
    b = _gpu(q, kv, table, sl)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def _sampled(cfg, n, seed):
    q, kv, table, sl = mla_config_inputs(cfg)
    o, lse = _gpu(q, kv, table, sl)
    rng = np.random.default_rng(seed)
    total = cfg.batch * cfg.Hq
    rows = np.unique(np.concatenate([[0, 127, total - 1], rng.integers(0, total, n)]))
    _check(q, kv, table, sl, o, lse, rows=rows)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    # O is a convex combination of latent rows: inside their per-column hull
    assert np.abs(o).max() <= float(kv.float().abs().max())


def test_scores_jump_on_a_later_page():
    """One late page scores far above the rest: the decode's per-half fast
    path must fall back, move the reference and rescale O in TMEM."""
    q, kv, table, sl = mla_inputs(3, 128, [1000, 640, 1500], seed=31)
    q = (q.float() + 0.3).to(q.dtype)  # a component every head shares ...
    for b in range(3):
        page = int(table[b, 7])          # ... lifts page 7 by ~18 in log2 units
        kv[page] = (kv[page].float() + 1.0).to(kv.dtype)
    o, lse = _gpu(q, kv, table, sl)
    _check(q, kv, table, sl, o, lse)


def test_heads_of_each_cta_jump_at_different_steps():
    """The two CTAs of a decode cluster run the softmax of heads 0-63 and
    64-127.  Heads 0-63 get a large score jump on page 5 (an odd step), heads
    64-127 on page 8 and again on page 9 (even, then odd): each CTA moves its
    references at its own steps, on both step parities, and the peer must
    apply those factors to its O columns of the same heads."""
    q, kv, table, sl = mla_inputs(3, 128, [1000, 640, 1500], seed=37)
    q = q.float()
    kv = kv.float()
    q[:, :64, 0:64] += 2.0      # heads 0-63 see columns 0-63 ...
    q[:, 64:, 64:128] += 2.0    # ... heads 64-127 columns 64-127
    for b in range(3):
        kv[int(table[b, 5]), :, 0:64] += 2.0     # ~27 log2 units up for heads 0-63
        kv[int(table[b, 8]), :, 64:128] += 1.5   # ~20 up for heads 64-127 ...
        kv[int(table[b, 9]), :, 64:128] += 3.0   # ... and ~20 more on the next page
    q, kv = q.to(torch.bfloat16), kv.to(torch.bfloat16)
    o, lse = _gpu(q, kv, table, sl)
    _check(q, kv, table, sl, o, lse)


def _all_rows(cfg):
    q, kv, table, sl = mla_config_inputs(cfg)
    o, lse = _gpu(q, kv, table, sl)
    _check(q, kv, table, sl, o, lse)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_decode_batch64_workload_every_row():
    """Every (sequence, head) row of the batch-64, seq-4096 workload."""
    _all_rows(MLA_B64)


def test_decode_batch256_paged_workload_every_row():
    """Every row of the batch-256 paged workload (ragged lengths 1024-4096,
    random page permutation, split-KV partials merged by the combine)."""
    _all_rows(MLA_B256_PAGED)


@pytest.mark.parametrize("cfg", [MLA_B16, MLA_B128, MLA_B256], ids=lambda c: str(c.batch))
def test_decode_batch_sweep_sampled(cfg):
    """The batch sweep at seq 4096: batch 16 runs through the split-KV plan
    (fewer sequences than clusters), 128 and 256 through whole chunks."""
    _sampled(cfg, 128, 3)


def test_few_uneven_sequences_split_into_their_own_chunks():
    """Fewer sequences than clusters with very different lengths: long ones are
    cut into several chunks of their own, short ones stay whole, empty ones
    are finished by the combine kernel."""
    lens = [4096, 100, 0, 2000, 64, 1, 3000, 4096, 500, 77]
    q, kv, table, sl = mla_inputs(len(lens), 128, lens, seed=61, paged_random=True)
    o, lse = _gpu(q, kv, table, sl)
    _check(q, kv, table, sl, o, lse)
