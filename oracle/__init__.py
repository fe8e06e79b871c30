"""fp64 CPU oracle for attention forward (MHA prefill and MLA absorbed decode).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
timed CPU baseline of ``bench.py`` may import this module.  The CUDA library
never calls it and shares no code with it; see ``attn_oracle.c`` for the
definitions it writes out and the passages they follow.

The C source is compiled with gcc into ``liboracle.so`` next to this file
(``build()``); ``load()`` builds it on first use if it is missing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, strict IEEE: no fast-math)."""
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _bind(lib):
    lib.oracle_mha.argtypes = [_ptr, _ptr, _ptr, _i64, _i64, _i64, _i64, _i64,
                               ctypes.c_int, ctypes.c_double, _ptr, _i64, _ptr,
                               _ptr, ctypes.c_int]
    lib.oracle_mha.restype = ctypes.c_int
    lib.oracle_mha_probs.argtypes = [_ptr, _ptr, _i64, _i64, _i64, _i64,
                                     ctypes.c_int, ctypes.c_double, _ptr]
    lib.oracle_mha_probs.restype = ctypes.c_int
    lib.oracle_mla.argtypes = [_ptr, _ptr, _ptr, _ptr, _i64, _i64, _i64, _i64,
                               _i64, _i64, _i64, ctypes.c_double, _ptr, _i64,
                               _ptr, _ptr, ctypes.c_int]
    lib.oracle_mla.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; a path loads a variant."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(_LIB) or (
                os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
            build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _f32(x) -> np.ndarray:
    """Exact widening to a contiguous float32 numpy array (bf16 -> fp32 is exact)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu")
            if x.dtype != torch.float32:
                x = x.to(torch.float32)
            return np.ascontiguousarray(x.numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _i32(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu").to(torch.int32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads(nthreads: int = 0) -> int:
    return load().oracle_num_threads(nthreads)


def mha(q, k, v, causal: bool, scale: float, rows=None, threads: int = 0,
        lib=None):
    """fp64 MHA forward.  q,k: [B,H,N,Dk]; v: [B,H,N,Dv].

    Returns (O, LSE) in float64: full shapes [B,H,N,Dv] and [B,H,N] when
    ``rows`` is None, else [len(rows), Dv] and [len(rows)] for the flat row
    ids (b*H + h)*N + i.
    """
    lib = lib or load()
    qa, ka, va = _f32(q), _f32(k), _f32(v)
    B, H, N, Dk = qa.shape
    Dv = va.shape[-1]
    assert ka.shape == (B, H, N, Dk) and va.shape == (B, H, N, Dv)
    if rows is None:
        nrows, rp = B * H * N, None
    else:
        ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows, rp = ra.size, _p(ra)
    o = np.zeros((nrows, Dv), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    rc = lib.oracle_mha(_p(qa), _p(ka), _p(va), B, H, N, Dk, Dv, int(causal),
                        float(scale), rp, nrows, _p(o), _p(lse), threads)
    if rc != 0:
        raise RuntimeError(f"oracle_mha failed: {rc}")
    if rows is None:
        return o.reshape(B, H, N, Dv), lse.reshape(B, H, N)
    return o, lse


def mha_probs(q, k, causal: bool, scale: float, lib=None) -> np.ndarray:
    """Softmax probabilities [B,H,N,N] (tiny inputs only)."""
    lib = lib or load()
    qa, ka = _f32(q), _f32(k)
    B, H, N, Dk = qa.shape
    P = np.zeros((B, H, N, N), dtype=np.float64)
    rc = lib.oracle_mha_probs(_p(qa), _p(ka), B, H, N, Dk, int(causal),
                              float(scale), _p(P))
    if rc != 0:
        raise RuntimeError(f"oracle_mha_probs failed: {rc}")
    return P


def mla(q, kv_cache, block_table, seqlens, scale: float, dv: int = 512,
        rows=None, threads: int = 0, lib=None):
    """fp64 MLA absorbed decode.

    q: [B,Hq,Dk]; kv_cache: [num_blocks, page, Dk]; block_table:
    [B, max_blocks] int; seqlens: [B] int.  Returns (O, LSE) float64, full
    [B,Hq,dv] / [B,Hq] or per requested flat id b*Hq + h.
    """
    lib = lib or load()
    qa, ca = _f32(q), _f32(kv_cache)
    bt, sl = _i32(block_table), _i32(seqlens)
    B, Hq, Dk = qa.shape
    num_blocks, page, Dk2 = ca.shape
    assert Dk2 == Dk and bt.shape[0] == B and sl.shape == (B,)
    max_blocks = bt.shape[1]
    if rows is None:
        nrows, rp = B * Hq, None
    else:
        ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows, rp = ra.size, _p(ra)
    o = np.zeros((nrows, dv), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    rc = lib.oracle_mla(_p(qa), _p(ca), _p(bt), _p(sl), B, Hq, Dk, dv, page,
                        max_blocks, num_blocks, float(scale), rp, nrows, _p(o),
                        _p(lse), threads)
    if rc != 0:
        raise RuntimeError(f"oracle_mla failed: {rc}")
    if rows is None:
        return o.reshape(B, Hq, dv), lse.reshape(B, Hq)
    return o, lse


# ----------------------------------------------------------------------------
# The projections around the latent attention ("MLA x FlashAttention-3
# fusion" article: absorption identity Q K^T = (Q W_UK) c^T + Q_R k_R^T, and
# the value up-projection W_UV after the latent attention).  Plain fp64
# definitions; numpy's matrix product is the library step.

def _f64(x) -> np.ndarray:
    """Exact widening to a contiguous float64 numpy array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu").to(torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def mla_absorb_q(q_nope, q_rope, w_uk) -> np.ndarray:
    """[q_nope_h W_UK_h | q_rope_h] for every sequence and head, fp64.

    q_nope [B,Hq,Dn], q_rope [B,Hq,Dr], w_uk [Hq,Dn,L] -> [B,Hq,L+Dr].
    """
    qn, qr, w = _f64(q_nope), _f64(q_rope), _f64(w_uk)
    B, Hq, _ = qn.shape
    L = w.shape[2]
    out = np.empty((B, Hq, L + qr.shape[2]), dtype=np.float64)
    for h in range(Hq):
        out[:, h, :L] = qn[:, h, :] @ w[h]
    out[:, :, L:] = qr
    return out


def mla_project_out(o_latent, w_uv) -> np.ndarray:
    """o_latent_h W_UV_h for every sequence and head, fp64: [B,Hq,L] x [Hq,L,Dv]."""
    ol, w = _f64(o_latent), _f64(w_uv)
    out = np.empty((ol.shape[0], ol.shape[1], w.shape[2]), dtype=np.float64)
    for h in range(ol.shape[1]):
        out[:, h, :] = ol[:, h, :] @ w[h]
    return out


def mla_decompressed(q_nope, q_rope, w_uk, w_uv, kv_cache, block_table, seqlens,
                     scale: float):
    """MLA attention with every head's keys and values decompressed, fp64.

    Per sequence b and head h, over the visible tokens t of its pages:
    K_h[t] = [c_t W_UK_h^T | k_rope_t], V_h[t] = c_t W_UV_h, and
    out = softmax(scale * [q_nope_h | q_rope_h] K_h^T) V_h, with its natural-log
    LSE.  This is attention as first defined, before any absorption; the
    absorbed path (mla_absorb_q, mla, mla_project_out) must reproduce it.
    Returns (out [B,Hq,Dv], lse [B,Hq]).
    """
    qn, qr, wk, wv = _f64(q_nope), _f64(q_rope), _f64(w_uk), _f64(w_uv)
    cache = _f64(kv_cache)
    bt, sl = _i32(block_table), _i32(seqlens)
    B, Hq, _ = qn.shape
    L = wk.shape[2]
    page = cache.shape[1]
    out = np.zeros((B, Hq, wv.shape[2]), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf, dtype=np.float64)
    for b in range(B):
        n = int(sl[b])
        if n == 0:
            continue
        rows = np.concatenate([cache[bt[b, j]] for j in range((n + page - 1) // page)])[:n]
        c, kr = rows[:, :L], rows[:, L:]
        for h in range(Hq):
            k_h = np.concatenate([c @ wk[h].T, kr], axis=1)
            v_h = c @ wv[h]
            s = scale * (k_h @ np.concatenate([qn[b, h], qr[b, h]]))
            m = s.max()
            p = np.exp(s - m)
            out[b, h] = (p @ v_h) / p.sum()
            lse[b, h] = m + np.log(p.sum())
    return out, lse
