"""Work accounting for the roofline: algorithmic FLOPs and bytes per call.

FLOP convention of the FP32 FlashAttention-2 blog's timing table (section
4.1): a non-causal forward counts 4*B*H*N^2*D (two GEMMs of 2*N^2*D each per
head); a causal forward counts only the visible pairs, 4*B*H*D*N(N+1)/2.  The
page's own numbers pin this (38 ms -> 14.45 TFLOPS, 21.4 ms -> 12.87 TFLOPS
at B=4, H=8, N=8192, D=64).

Bytes are algorithmic: every input element read once and every output
element written once.  For MLA decode each visible latent row (576 bf16) is
read once, plus q in and O + LSE out, plus the block table and lengths; split
partials and L2 re-reads are implementation overhead and are not counted.
"""
from __future__ import annotations


def mha_flops(B: int, H: int, N: int, D: int, causal: bool) -> float:
    if causal:
        return 4.0 * B * H * D * N * (N + 1) / 2.0
    return 4.0 * B * H * N * N * D


def mha_bytes(B: int, H: int, N: int, D: int, elem_bytes: int) -> float:
    """q, k, v read once, o written once (elem_bytes each), lse fp32 written."""
    return 4.0 * B * H * N * D * elem_bytes + 4.0 * B * H * N


def mla_bytes(seqlens, Hq: int = 128, dk: int = 576, dv: int = 512,
              max_blocks: int | None = None) -> float:
    """Algorithmic HBM bytes of one MLA decode call (bf16 data, fp32 LSE)."""
    seqlens = [int(x) for x in seqlens]
    B = len(seqlens)
    kv = sum(seqlens) * dk * 2
    q = B * Hq * dk * 2
    o = B * Hq * dv * 2
    lse = B * Hq * 4
    table = B * (max_blocks if max_blocks is not None else 0) * 4
    lens = B * 4
    return float(kv + q + o + lse + table + lens)


def mla_flops(seqlens, Hq: int = 128, dk: int = 576, dv: int = 512) -> float:
    return float(sum(int(x) for x in seqlens)) * Hq * 2.0 * (dk + dv)
