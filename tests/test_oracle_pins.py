"""Pins for the fp64 oracle, each against something other than the oracle.

Every check here is fixed by mathematics or by an independent routine, not by
re-typing the oracle's formula:
  * closed forms (one key, identical keys, scale = 0, causal row 0);
  * invariants (permutation of unmasked keys, rows of P sum to 1,
    sum_j exp(s_j - LSE) = 1, split-and-merge by LSE equals the whole);
  * brute force on tiny inputs against torch's scaled_dot_product_attention in
    float64 (a library routine) and against a pure-Python loop;
  * the large-scale limit (softmax tends to the argmax row).
test_mutants_are_caught plants plausible mistakes into copies of the oracle's
C source and checks that these pins catch every one.
"""
import math
import shutil

import numpy as np
import pytest
import torch

import oracle
from online_softmax_attention_attn_gb300.inputs import mha_inputs, mla_inputs


def _sdpa64(q, k, v, causal, scale):
    q, k, v = (t.to(torch.float64) for t in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(
        q, k, v, is_causal=causal, scale=scale)


def _lse64(q, k, causal, scale):
    s = torch.einsum("bhid,bhjd->bhij", q.double(), k.double()) * scale
    if causal:
        n = s.shape[-1]
        mask = torch.ones(n, n, dtype=torch.bool).triu(1)
        s = s.masked_fill(mask, float("-inf"))
    return torch.logsumexp(s, dim=-1)


# ---------------------------------------------------------------- MHA pins

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 4), (2, 3, 5, 8), (1, 2, 8, 3),
                                   (1, 1, 37, 16)])
def test_mha_matches_sdpa_float64(oracle_lib, shape, causal):
    B, H, N, D = shape
    q, k, v = mha_inputs(B, H, N, D, seed=11 + N + D)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.mha(q, k, v, causal, scale)
    ref = _sdpa64(q, k, v, causal, scale).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, _lse64(q, k, causal, scale).numpy(),
                               rtol=0, atol=1e-12)


def test_mha_matches_python_loops(oracle_lib):
    """Independent pure-Python fp64 formula (math.exp, math.fsum) on tiny data."""
    B, H, N, Dk, Dv = 1, 2, 6, 3, 5
    g = torch.Generator().manual_seed(5)
    q = torch.randn(B, H, N, Dk, generator=g)
    k = torch.randn(B, H, N, Dk, generator=g)
    v = torch.randn(B, H, N, Dv, generator=g)
    scale = 0.7
    for causal in (False, True):
        o, lse = oracle.mha(q, k, v, causal, scale)
        for h in range(H):
            for i in range(N):
                keys = range(i + 1) if causal else range(N)
                s = [scale * math.fsum(float(q[0, h, i, d]) * float(k[0, h, j, d])
                                       for d in range(Dk)) for j in keys]
                w = [math.exp(x) for x in s]
                z = math.fsum(w)
                for d in range(Dv):
                    ref = math.fsum(w[n] * float(v[0, h, j, d])
                                    for n, j in enumerate(keys)) / z
                    assert abs(o[0, h, i, d] - ref) < 1e-12
                assert abs(lse[0, h, i] - math.log(z)) < 1e-12


def test_one_key_gives_v_row(oracle_lib):
    """N = 1: the only key has weight 1, so O = V[0] and LSE = s_00."""
    q, k, v = mha_inputs(2, 3, 1, 16, seed=3)
    o, lse = oracle.mha(q, k, v, False, 0.25)
    np.testing.assert_array_equal(o, v.double().numpy())
    s00 = (q.double() * k.double()).sum(-1) * 0.25
    np.testing.assert_allclose(lse, s00.numpy(), rtol=0, atol=1e-13)


def test_causal_row0_is_v0(oracle_lib):
    q, k, v = mha_inputs(1, 2, 33, 8, seed=4)
    o, lse = oracle.mha(q, k, v, True, 0.3)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0].double().numpy())
    s00 = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) * 0.3
    np.testing.assert_allclose(lse[:, :, 0], s00.numpy(), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_v(oracle_lib, causal):
    """All keys equal -> uniform weights: O_i = mean of visible V rows and
    LSE_i = s + ln(#visible)."""
    B, H, N, D = 1, 2, 19, 8
    q, _, v = mha_inputs(B, H, N, D, seed=6)
    k = torch.randn(B, H, 1, D).expand(B, H, N, D).contiguous()
    scale = 0.4
    o, lse = oracle.mha(q, k, v, causal, scale)
    vd = v.double()
    s = (q.double() * k.double()).sum(-1) * scale
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(o[:, :, i], vd[:, :, :n].mean(2).numpy(),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], (s[:, :, i] + math.log(n)).numpy(),
                                   rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_scale_zero_closed_form(oracle_lib, causal):
    """scale = 0: every visible score is 0, O = mean(V visible), LSE = ln|V(i)|."""
    B, H, N, D = 2, 1, 23, 4
    q, k, v = mha_inputs(B, H, N, D, seed=7)
    o, lse = oracle.mha(q, k, v, causal, 0.0)
    csum = torch.cumsum(v.double(), dim=2)
    for i in range(N):
        n = i + 1 if causal else N
        ref = (csum[:, :, i] / n) if causal else v.double().mean(2)
        np.testing.assert_allclose(o[:, :, i], ref.numpy(), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), rtol=0, atol=1e-14)


def test_permuting_keys_with_values_is_invariant(oracle_lib):
    B, H, N, D = 1, 2, 31, 16
    q, k, v = mha_inputs(B, H, N, D, seed=8)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(1))
    o1, l1 = oracle.mha(q, k, v, False, 0.25)
    o2, l2 = oracle.mha(q, k[:, :, perm], v[:, :, perm], False, 0.25)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows(oracle_lib, causal):
    """Rows of P sum to 1, masked entries are 0, and P = exp(s - LSE)."""
    B, H, N, D = 1, 2, 12, 8
    q, k, v = mha_inputs(B, H, N, D, seed=9)
    scale = 0.5
    P = oracle.mha_probs(q, k, causal, scale)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-14)
    if causal:
        assert np.all(P[..., np.triu_indices(N, 1)[0], np.triu_indices(N, 1)[1]] == 0)
    _, lse = oracle.mha(q, k, v, causal, scale)
    s = (torch.einsum("bhid,bhjd->bhij", q.double(), k.double()) * scale).numpy()
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(np.exp(s[:, :, i, :n] - lse[:, :, i, None]).sum(-1),
                                   1.0, rtol=0, atol=1e-13)
    # O equals P @ V with P from the separate export
    o, _ = oracle.mha(q, k, v, causal, scale)
    np.testing.assert_allclose(o, P @ v.double().numpy(), rtol=0, atol=1e-13)


def test_direct_logsumexp_small_scores(oracle_lib):
    """For small scores no max shift is needed: LSE = log(fsum exp(s_j))."""
    B, H, N, D = 1, 1, 9, 4
    q, k, v = mha_inputs(B, H, N, D, seed=10, std=0.3)
    scale = 0.5
    _, lse = oracle.mha(q, k, v, False, scale)
    for i in range(N):
        s = [scale * sum(float(q[0, 0, i, d]) * float(k[0, 0, j, d]) for d in range(D))
             for j in range(N)]
        assert abs(lse[0, 0, i] - math.log(math.fsum(math.exp(x) for x in s))) < 1e-13


def test_split_and_merge_by_lse_equals_whole(oracle_lib):
    """Attention over disjoint key sets merged with LSE weights equals the
    attention over their union: L = log(sum_s e^{L_s}), O = sum_s e^{L_s-L} O_s."""
    B, H, N, D = 1, 2, 40, 8
    q, k, v = mha_inputs(B, H, N, D, seed=12)
    scale = 0.35
    o_all, l_all = oracle.mha(q, k, v, False, scale)
    cuts = [0, 7, 8, 29, 40]
    Os, Ls = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        n = b - a
        o_p = np.zeros((B, H, N, D))
        l_p = np.zeros((B, H, N))
        for i in range(N):
            # query i alone against keys [a, b): n copies of the query, row 0
            qi = q[:, :, i:i + 1].expand(B, H, n, D).contiguous()
            o_i, l_i = oracle.mha(qi, k[:, :, a:b].contiguous(),
                                  v[:, :, a:b].contiguous(), False, scale)
            o_p[:, :, i] = o_i[:, :, 0]
            l_p[:, :, i] = l_i[:, :, 0]
        Os.append(o_p)
        Ls.append(l_p)
    Ls = np.stack(Ls)
    L = np.logaddexp.reduce(Ls, axis=0)
    O = sum(np.exp(Ls[s] - L)[..., None] * Os[s] for s in range(len(Os)))
    np.testing.assert_allclose(O, o_all, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, l_all, rtol=0, atol=1e-13)


def test_large_scale_is_stable_and_tends_to_argmax(oracle_lib):
    """scale x100 with distinct maxima: finite, and O -> V[argmax_j s_j]."""
    B, H, N, D = 1, 1, 16, 8
    q, k, v = mha_inputs(B, H, N, D, seed=13)
    scale = 100.0
    o, lse = oracle.mha(q, k, v, False, scale)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    s = torch.einsum("bhid,bhjd->bhij", q.double(), k.double())
    top2 = torch.topk(s, 2, dim=-1).values
    arg = s.argmax(-1)
    for i in range(N):
        gap = float(top2[0, 0, i, 0] - top2[0, 0, i, 1]) * scale
        if gap > 40:  # the runner-up weighs < e^-40
            np.testing.assert_allclose(o[0, 0, i], v[0, 0, arg[0, 0, i]].double().numpy(),
                                       rtol=0, atol=1e-12)


def test_row_subset_equals_full(oracle_lib):
    B, H, N, D = 2, 2, 17, 8
    q, k, v = mha_inputs(B, H, N, D, seed=14)
    o, lse = oracle.mha(q, k, v, True, 0.3)
    rows = [0, 5, 33, 67, 50]
    o2, l2 = oracle.mha(q, k, v, True, 0.3, rows=rows)
    np.testing.assert_array_equal(o2, o.reshape(-1, D)[rows])
    np.testing.assert_array_equal(l2, lse.reshape(-1)[rows])


def test_thread_count_does_not_change_result(oracle_lib):
    q, k, v = mha_inputs(1, 4, 64, 16, seed=15)
    a = oracle.mha(q, k, v, True, 0.25, threads=1)
    b = oracle.mha(q, k, v, True, 0.25, threads=4)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------- MLA pins

def _mla_sdpa_ref(q, kv, table, seqlens, scale, dv=512):
    """Gather + torch sdpa (float64): K = C, V = C[:, :dv], shared by all heads."""
    B, Hq, Dk = q.shape
    page = kv.shape[1]
    outs, lses = [], []
    for b in range(B):
        L = int(seqlens[b])
        if L == 0:
            outs.append(torch.zeros(Hq, dv, dtype=torch.float64))
            lses.append(torch.full((Hq,), float("-inf"), dtype=torch.float64))
            continue
        idx = torch.arange(L)
        C = kv[table[b, idx // page].long(), idx % page].double()
        qq = q[b].double()[None]                         # [1, Hq, Dk]
        o = torch.nn.functional.scaled_dot_product_attention(
            qq[:, :, None], C[None, None].expand(1, Hq, L, Dk),
            C[None, None, :, :dv].expand(1, Hq, L, dv), scale=scale)
        outs.append(o[0, :, 0])
        lses.append(torch.logsumexp(qq[0] @ C.T * scale, dim=-1))
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


@pytest.mark.parametrize("paged", [False, True])
def test_mla_matches_gather_plus_sdpa(oracle_lib, paged):
    seqlens = [1, 64, 65, 200]
    q, kv, table, sl = mla_inputs(4, 8, seqlens, seed=21, paged_random=paged,
                                  dtype=torch.float32)
    scale = 1.0 / math.sqrt(192.0)
    o, lse = oracle.mla(q, kv, table, sl, scale)
    ref_o, ref_l = _mla_sdpa_ref(q, kv, table, sl, scale)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_mla_bf16_inputs_are_widened_exactly(oracle_lib):
    q, kv, table, sl = mla_inputs(2, 4, [70, 3], seed=22, paged_random=True)
    assert q.dtype == torch.bfloat16
    o1, l1 = oracle.mla(q, kv, table, sl, 0.1)
    o2, l2 = oracle.mla(q.float(), kv.float(), table, sl, 0.1)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_mla_scale_zero_is_mean_of_latent_prefix(oracle_lib):
    q, kv, table, sl = mla_inputs(3, 4, [1, 64, 130], seed=23, paged_random=True,
                                  dtype=torch.float32)
    o, lse = oracle.mla(q, kv, table, sl, 0.0)
    for b in range(3):
        L = int(sl[b])
        idx = torch.arange(L)
        C = kv[table[b, idx // 64].long(), idx % 64].double()
        np.testing.assert_allclose(o[b], C[:, :512].mean(0).expand(4, 512).numpy(),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], math.log(L), rtol=0, atol=1e-14)


def test_mla_page_permutation_is_exactly_invariant(oracle_lib):
    """Moving pages in the pool with a matching block table changes nothing."""
    q, kv, table, sl = mla_inputs(2, 4, [150, 90], seed=24, dtype=torch.float32)
    perm = torch.randperm(kv.shape[0], generator=torch.Generator().manual_seed(2))
    inv = torch.argsort(perm)
    kv2 = kv[perm]                       # new slot s holds old page perm[s]
    table2 = inv[table.long()].to(torch.int32)
    a = oracle.mla(q, kv, table, sl, 0.2)
    b = oracle.mla(q, kv2, table2, sl, 0.2)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_mla_token_permutation_invariant_and_tail_ignored(oracle_lib):
    """Permuting the visible tokens, or changing data past seqlen, leaves O."""
    q, kv, table, sl = mla_inputs(1, 4, [100], seed=25, dtype=torch.float32)
    o, lse = oracle.mla(q, kv, table, sl, 0.2)
    kv2 = kv.clone()
    kv2[1, 100 - 64:] = 1e3               # past the end of the sequence
    o2, l2 = oracle.mla(q, kv2, table, sl, 0.2)
    np.testing.assert_array_equal(o, o2)
    flat = torch.cat([kv[0], kv[1, :36]])
    perm = torch.randperm(100, generator=torch.Generator().manual_seed(3))
    kv3 = kv.clone()
    kv3[0] = flat[perm[:64]]
    kv3[1, :36] = flat[perm[64:]]
    o3, l3 = oracle.mla(q, kv3, table, sl, 0.2)
    np.testing.assert_allclose(o3, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l3, lse, rtol=0, atol=1e-13)


def test_mla_equals_mha_with_shared_latent_head(oracle_lib):
    """MLA = MHA with every query head on one shared K = C, V = C[:, :512]."""
    L, Hq = 70, 4
    q, kv, table, sl = mla_inputs(1, Hq, [L], seed=26, dtype=torch.float32)
    o, lse = oracle.mla(q, kv, table, sl, 0.15)
    C = torch.cat([kv[0], kv[1]])[:L]
    for h in range(Hq):
        qh = q[0, h][None, None, None].expand(1, 1, L, 576).contiguous()
        om, lm = oracle.mha(qh, C[None, None].contiguous(),
                            C[None, None, :, :512].contiguous(), False, 0.15)
        np.testing.assert_allclose(o[0, h], om[0, 0, 0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, h], lm[0, 0, 0], rtol=0, atol=1e-13)


def test_mla_empty_sequence(oracle_lib):
    q, kv, table, sl = mla_inputs(2, 4, [0, 5], seed=27, dtype=torch.float32)
    o, lse = oracle.mla(q, kv, table, sl, 0.2)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_mla_rejects_bad_table(oracle_lib):
    q, kv, table, sl = mla_inputs(1, 2, [10], seed=28, dtype=torch.float32)
    bad = table.clone()
    bad[0, 0] = kv.shape[0]
    with pytest.raises(RuntimeError):
        oracle.mla(q, kv, bad, sl, 0.2)
    with pytest.raises(RuntimeError):
        oracle.mla(q, kv, table, torch.tensor([65], dtype=torch.int32), 0.2)


# ------------------------------------------------------------ mutation check

_MUTANTS = [
    ("causal j<i", "int64_t nkeys = causal ? (i + 1) : N;",
     "int64_t nkeys = causal ? (i > 0 ? i : 1) : N;"),
    ("scale dropped", "s[j] = scale * acc;", "s[j] = acc;"),
    ("max not subtracted in lse", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("no normalisation", "o_out[d] /= l;", "o_out[d] /= 1.0;"),
    ("value index transposed", "vr[j] = v + (bh * N + j) * Dv;",
     "vr[j] = v + (bh * N + (N - 1 - j)) * Dv;"),
    ("key row off by one", "kr[j] = k + (bh * N + j) * Dk;",
     "kr[j] = k + (bh * N + (j + 1) % N) * Dk;"),
    ("V taken from the end of the row", "const float* vr = vrows[j];",
     "const float* vr = vrows[j] + (dk - dv);"),
    ("mla page index", "cr[t] = kv + (blk * page + t % page) * Dk;",
     "cr[t] = kv + (blk * page + (t + 1) % page) * Dk;"),
    ("mla table row", "int64_t blk = block_table[b * max_blocks + t / page];",
     "int64_t blk = block_table[t / page];"),
]


def _pins_pass(lib) -> bool:
    """A compact re-run of the pins above against a given oracle build."""
    try:
        for (B, H, N, D) in [(2, 3, 5, 8), (1, 2, 9, 4)]:
            q, k, v = mha_inputs(B, H, N, D, seed=100 + N)
            for causal in (False, True):
                o, lse = oracle.mha(q, k, v, causal, 0.45, lib=lib)
                if not np.allclose(o, _sdpa64(q, k, v, causal, 0.45).numpy(), atol=1e-12):
                    return False
                if not np.allclose(lse, _lse64(q, k, causal, 0.45).numpy(), atol=1e-12):
                    return False
        for paged in (False, True):
            q, kv, table, sl = mla_inputs(3, 4, [1, 64, 130], seed=31,
                                          paged_random=paged, dtype=torch.float32)
            o, lse = oracle.mla(q, kv, table, sl, 0.1, lib=lib)
            ro, rl = _mla_sdpa_ref(q, kv, table, sl, 0.1)
            if not (np.allclose(o, ro, atol=1e-12) and np.allclose(lse, rl, atol=1e-12)):
                return False
        return True
    except RuntimeError:
        return False


def test_mutants_are_caught(oracle_lib, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(oracle._SRC).read()
    assert _pins_pass(oracle_lib), "the real oracle must pass the compact pins"
    mutants = list(_MUTANTS)
    checked = 0
    for name, old, new in mutants:
        assert src.count(old) >= 1, f"mutation anchor for {name!r} missing"
        mutated = src.replace(old, new)  # the same slip at every site
        c = tmp_path / f"m{checked}.c"
        so = tmp_path / f"m{checked}.so"
        c.write_text(mutated)
        oracle.build(str(c), str(so))
        lib = oracle.load(str(so))
        assert not _pins_pass(lib), f"pins missed the planted mistake: {name}"
        checked += 1
    assert checked >= 8


# ---------------------------------------------------------------- MLA projections

def _layer(seed=3, B=2, Hq=4, lens=(37, 70), dn=16, dr=8, dl=32, dv=16):
    from online_softmax_attention_attn_gb300.inputs import mla_layer_inputs
    return mla_layer_inputs(B, Hq, list(lens), seed=seed, d_nope=dn, d_rope=dr, d_latent=dl,
                            d_v=dv, paged_random=True)


def test_absorption_identity_matches_decompressed_attention(oracle_lib):
    """The article's absorption identity: folding W_UK into the query and W_UV
    after the latent attention gives exactly the attention over explicitly
    decompressed keys [c W_UK^T | k_rope] and values c W_UV (fp64; the only
    residue is the fp32 rounding of the absorbed query fed to the C oracle)."""
    qn, qr, wk, wv, kv, table, sl = _layer()
    qa = oracle.mla_absorb_q(qn, qr, wk)
    ol, lse = oracle.mla(qa, kv, table, sl, 0.2, dv=32, lib=oracle_lib)
    out = oracle.mla_project_out(ol, wv)
    ref, rlse = oracle.mla_decompressed(qn, qr, wk, wv, kv, table, sl, 0.2)
    assert np.abs(out - ref).max() <= 1e-6 * np.abs(ref).max()
    assert np.abs(lse - rlse).max() <= 1e-6
    # a planted slip: the rotary part left out of the absorbed query
    qa_bad = qa.copy()
    qa_bad[:, :, 32:] = 0.0
    ol_bad, _ = oracle.mla(qa_bad, kv, table, sl, 0.2, dv=32, lib=oracle_lib)
    assert np.abs(oracle.mla_project_out(ol_bad, wv) - ref).max() > 1e-3


def test_absorb_and_project_with_identity_weights():
    """W_UK = [I | 0] copies q_nope into the leading latent columns (rest zero,
    q_rope appended); W_UV = [I; 0] keeps the leading latent columns."""
    qn, qr, _, _, _, _, _ = _layer()
    wk = np.zeros((4, 16, 32))
    wk[:, :, :16] = np.eye(16)
    qa = oracle.mla_absorb_q(qn, qr, wk)
    assert np.array_equal(qa[:, :, :16], qn.float().numpy())
    assert not qa[:, :, 16:32].any()
    assert np.array_equal(qa[:, :, 32:], qr.float().numpy())
    ol = np.random.default_rng(1).standard_normal((2, 4, 32))
    wv = np.zeros((4, 32, 16))
    wv[:, :16, :] = np.eye(16)
    assert np.array_equal(oracle.mla_project_out(ol, wv), ol[:, :, :16])


def test_decompressed_single_token_gives_its_value_row():
    """One visible token: the attention output is that token's value row
    c_0 W_UV_h and the LSE is the scaled score itself."""
    qn, qr, wk, wv, kv, table, _ = _layer(lens=(1, 1))
    sl = torch.tensor([1, 1], dtype=torch.int32)
    out, lse = oracle.mla_decompressed(qn, qr, wk, wv, kv, table, sl, 0.3)
    for b in range(2):
        row = kv[int(table[b, 0]), 0].double().numpy()
        for h in range(4):
            assert np.allclose(out[b, h], row[:32] @ wv[h].double().numpy(), rtol=1e-12)
            k = np.concatenate([row[:32] @ wk[h].double().numpy().T, row[32:]])
            q = np.concatenate([qn[b, h].double().numpy(), qr[b, h].double().numpy()])
            assert abs(lse[b, h] - 0.3 * float(k @ q)) <= 1e-9
