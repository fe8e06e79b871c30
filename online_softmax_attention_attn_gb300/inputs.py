"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws numbers: it holds none of the attention arithmetic.
Every tensor is drawn on the CPU from a seeded ``torch.Generator`` as float32
and, for bf16 workloads, rounded once with round-to-nearest-even
(``.to(torch.bfloat16)``).  The same host bytes then feed both the CUDA path
and the fp64 oracle.

Workload shapes follow the two pages' benchmarks:
  * MHA prefill shapes of the FP32 FlashAttention-2 blog (section 4.1:
    N=8192, B=4, H=8, D=64) plus a small case and a bf16 D=128 case;
  * MLA decode shapes of the MLA x FlashAttention-3 article (its benchmark
    table: batch 16..256, sequence 4096, 512-d latent + 64-d RoPE key).
No dataset or model is involved; the article's "67B MLA variant" is stood in
for by these shapes with random data.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

MLA_DK = 576      # [c_kv 512 | k_rope 64]
MLA_DV = 512      # V = the c_kv slice of the same row
MLA_PAGE = 64     # tokens per paged block


@dataclass(frozen=True)
class MHAConfig:
    name: str
    B: int
    H: int
    N: int
    D: int
    causal: bool
    dtype: torch.dtype
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclass(frozen=True)
class MLAConfig:
    name: str
    batch: int
    Hq: int
    seq_min: int
    seq_max: int
    paged_random: bool
    seed: int
    q_std: float = 1.0
    cache_std: float = 0.5
    scale: float = 1.0 / math.sqrt(192.0)
    extra: dict = field(default_factory=dict)


# The five workloads.  Seeds are 1000 + workload number.
FP32_SMALL_CAUSAL = MHAConfig("fp32 MHA causal B1 H2 N256 D64", 1, 2, 256, 64,
                              True, torch.float32, 1001)
FP32_PAGE2 = MHAConfig("fp32 MHA B4 H8 N8192 D64", 4, 8, 8192, 64, False,
                       torch.float32, 1002)
FP32_PAGE2_CAUSAL = MHAConfig("fp32 MHA causal B4 H8 N8192 D64", 4, 8, 8192,
                              64, True, torch.float32, 1002)
BF16_PREFILL = MHAConfig("bf16 MHA causal prefill B4 H16 N4096 D128", 4, 16,
                         4096, 128, True, torch.bfloat16, 1003)
BF16_PREFILL_NONCAUSAL = MHAConfig("bf16 MHA prefill B4 H16 N4096 D128", 4, 16, 4096,
                                   128, False, torch.bfloat16, 1003)
MLA_B64 = MLAConfig("bf16 MLA decode batch64 Hq128 seq4096", 64, 128, 4096,
                    4096, False, 1004)
MLA_B256_PAGED = MLAConfig("bf16 MLA decode batch256 Hq128 seq1024-4096 paged",
                           256, 128, 1024, 4096, True, 1005)
# The decode batch sweep at seq 4096 (batch 64 is MLA_B64 above).
MLA_B16 = MLAConfig("bf16 MLA decode batch16 Hq128 seq4096", 16, 128, 4096, 4096, False, 1006)
MLA_B128 = MLAConfig("bf16 MLA decode batch128 Hq128 seq4096", 128, 128, 4096, 4096, False, 1007)
MLA_B256 = MLAConfig("bf16 MLA decode batch256 Hq128 seq4096", 256, 128, 4096, 4096, False, 1008)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def mha_inputs(B: int, H: int, N: int, D: int, dtype=torch.float32,
               seed: int = 0, std: float = 1.0, Dv: int | None = None):
    """q, k, v ~ N(0, std^2) i.i.d., shape [B,H,N,D] (v: [B,H,N,Dv]), CPU."""
    g = _gen(seed)
    Dv = D if Dv is None else Dv
    q = torch.randn(B, H, N, D, generator=g, dtype=torch.float32) * std
    k = torch.randn(B, H, N, D, generator=g, dtype=torch.float32) * std
    v = torch.randn(B, H, N, Dv, generator=g, dtype=torch.float32) * std
    return q.to(dtype), k.to(dtype), v.to(dtype)


def mha_config_inputs(cfg: MHAConfig):
    return mha_inputs(cfg.B, cfg.H, cfg.N, cfg.D, cfg.dtype, cfg.seed)


def mla_inputs(batch: int, Hq: int, seqlens, seed: int = 0,
               paged_random: bool = False, q_std: float = 1.0,
               cache_std: float = 0.5, num_blocks: int | None = None,
               max_blocks: int | None = None, dtype=torch.bfloat16, width: int = MLA_DK):
    """Absorbed queries, a paged latent pool, a block table and lengths (CPU).

    q [batch, Hq, 576]; kv_cache [num_blocks, 64, 576] filled over the whole
    pool (unused page tails hold random data, so masking is exercised);
    block_table [batch, max_blocks] int32: identity b*max_blocks + j, or a
    seeded random permutation of the pool when ``paged_random``.
    """
    g = _gen(seed)
    seqlens = torch.as_tensor(seqlens, dtype=torch.int32).reshape(batch)
    need = int(math.ceil(int(seqlens.max().item() if batch else 0) / MLA_PAGE))
    max_blocks = max(need, 1) if max_blocks is None else max_blocks
    num_blocks = batch * max_blocks if num_blocks is None else num_blocks
    q = torch.randn(batch, Hq, width, generator=g, dtype=torch.float32) * q_std
    kv = torch.randn(num_blocks, MLA_PAGE, width, generator=g,
                     dtype=torch.float32) * cache_std
    if paged_random:
        perm = torch.randperm(num_blocks, generator=g)[: batch * max_blocks]
        table = perm.view(batch, max_blocks).to(torch.int32)
    else:
        table = torch.arange(batch * max_blocks, dtype=torch.int32).view(
            batch, max_blocks)
    return (q.to(dtype).contiguous(), kv.to(dtype).contiguous(),
            table.contiguous(), seqlens.contiguous())


# Widths of the projections around the latent attention (DeepSeek-style MLA):
# per head a 128-wide non-rotary query part, a 64-wide rotary part, a
# 512-wide latent and a 128-wide value.
MLA_DNOPE, MLA_DROPE, MLA_DLATENT, MLA_DVHEAD = 128, 64, 512, 128


def mla_layer_inputs(batch: int, Hq: int, seqlens, seed: int = 0, d_nope: int = MLA_DNOPE,
                     d_rope: int = MLA_DROPE, d_latent: int = MLA_DLATENT,
                     d_v: int = MLA_DVHEAD, paged_random: bool = False,
                     cache_std: float = 0.5, dtype=torch.bfloat16):
    """Un-absorbed query parts, per-head up-projections and a paged latent pool (CPU).

    q_nope [batch,Hq,d_nope], q_rope [batch,Hq,d_rope] ~ N(0,1);
    w_uk [Hq,d_nope,d_latent] ~ N(0,1/d_nope), w_uv [Hq,d_latent,d_v] ~ N(0,1/d_latent)
    (so projected entries stay of order one); the cache, block table and lengths
    are those of ``mla_inputs`` (rows of d_latent + d_rope).
    """
    g = _gen(seed + 104729)
    q_nope = torch.randn(batch, Hq, d_nope, generator=g, dtype=torch.float32)
    q_rope = torch.randn(batch, Hq, d_rope, generator=g, dtype=torch.float32)
    w_uk = torch.randn(Hq, d_nope, d_latent, generator=g, dtype=torch.float32) / math.sqrt(d_nope)
    w_uv = torch.randn(Hq, d_latent, d_v, generator=g, dtype=torch.float32) / math.sqrt(d_latent)
    _, kv, table, sl = mla_inputs(batch, Hq, seqlens, seed=seed, paged_random=paged_random,
                                  cache_std=cache_std, dtype=dtype, width=d_latent + d_rope)
    return (q_nope.to(dtype), q_rope.to(dtype), w_uk.to(dtype), w_uv.to(dtype), kv, table, sl)


def mla_seqlens(cfg: MLAConfig) -> torch.Tensor:
    """Per-sequence lengths: fixed, or uniform integers in [seq_min, seq_max]."""
    if cfg.seq_min == cfg.seq_max:
        return torch.full((cfg.batch,), cfg.seq_max, dtype=torch.int32)
    g = _gen(cfg.seed + 7919)
    return torch.randint(cfg.seq_min, cfg.seq_max + 1, (cfg.batch,),
                         generator=g, dtype=torch.int32)


def mla_config_inputs(cfg: MLAConfig):
    sl = mla_seqlens(cfg)
    max_blocks = cfg.seq_max // MLA_PAGE
    return mla_inputs(cfg.batch, cfg.Hq, sl, seed=cfg.seed,
                      paged_random=cfg.paged_random, q_std=cfg.q_std,
                      cache_std=cfg.cache_std, max_blocks=max_blocks,
                      num_blocks=cfg.batch * max_blocks)
