"""Python binding of libattn.so (GB300 / sm_103a attention forward).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/attn.h``.  PyTorch is used for
device memory and streams.  There is no fallback: if the library is missing
or cannot be loaded, every call raises.

Entry points (same names as the C ABI):
  attn_fwd(q, k, v, o=None, lse=None, causal=False, scale=None, stream=None)
  attn_fwd_tf32x3(q, k, v, o=None, lse=None, causal=False, scale=None,
                  workspace=None, stream=None)
  attn_fwd_tf32x3_workspace_size(B, H, N, D)
  attn_fwd_host(q, k, v, o=None, lse=None, causal=False, scale=None,
                workspace=None, stream=None)          # host tensors in and out
  mla_decode_host(q, kv_cache, block_table, seqlens, o=None, lse=None,
                  scale=..., workspace=None, stream=None)
  mla_decode(q, kv_cache, block_table, seqlens, o=None, lse=None, scale=...,
             workspace=None, stream=None)
  mla_decode_split(..., pages_per_split=...)
  mla_decode_workspace_size(B, Hq, max_blocks_per_seq, num_sms)
  mla_decode_split_workspace_size(B, Hq, max_blocks_per_seq, num_sms, pages_per_split=0)
  attn_device_status(stream=None)
  attn_last_error()
"""
from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "AttnError", "lib", "attn_fwd", "attn_fwd_tf32x3", "attn_fwd_tf32x3_workspace_size",
    "attn_fwd_host", "attn_fwd_host_workspace_size", "mla_decode_host",
    "mla_decode_host_workspace_size",
    "mla_decode", "mla_decode_split",
    "mla_decode_workspace_size", "mla_decode_split_workspace_size", "mla_decode_noalloc", "mla_absorb_q", "mla_project_out",
    "attn_device_status", "attn_last_error",
    "attn_kv_tiles", "attn_kernel_info", "attn_fwd_test_skip_load",
    "attn_fwd_f32_test_skip_load",
    "attn_fwd_tf32x3_test_skip_load", "mla_decode_test_skip_load",
    "LIB_PATH", "ATTN_DTYPE_F32", "ATTN_DTYPE_BF16",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_MISALIGNED = -3
ATTN_ERR_WORKSPACE_TOO_SMALL = -4
ATTN_ERR_CUDA = -5
ATTN_ERR_BAD_BLOCK_TABLE = -6
ATTN_ERR_BAD_SEQLEN = -7
ATTN_ERR_DEVICE_TIMEOUT = -8
ATTN_DTYPE_F32 = 0
ATTN_DTYPE_BF16 = 1

MLA_DK, MLA_DV, MLA_PAGE = 576, 512, 64


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


_lib = None
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libattn.so not found at {LIB_PATH}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        L.attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]
        L.attn_fwd.restype = _i
        L.attn_fwd_test_skip_load.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                              _f, _vp, _i]
        L.attn_fwd_test_skip_load.restype = _i
        L.attn_fwd_f32_test_skip_load.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                                  _f, _vp, _i]
        L.attn_fwd_f32_test_skip_load.restype = _i
        L.attn_fwd_tf32x3_test_skip_load.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i,
                                                     _i, _i, _f, _vp, _sz, _vp, _i]
        L.attn_fwd_tf32x3_test_skip_load.restype = _i
        L.mla_decode_test_skip_load.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _f, _i,
                                                _i, _vp, _sz, _vp, _i]
        L.mla_decode_test_skip_load.restype = _i
        L.attn_fwd_tf32x3_workspace_size.argtypes = [_i, _i, _i, _i]
        L.attn_fwd_tf32x3_workspace_size.restype = _sz
        L.attn_fwd_tf32x3.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp,
                                      _sz, _vp]
        L.attn_fwd_tf32x3.restype = _i
        L.attn_fwd_host_workspace_size.argtypes = [_i, _i, _i, _i, _i]
        L.attn_fwd_host_workspace_size.restype = _sz
        L.attn_fwd_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp,
                                    _sz, _vp]
        L.attn_fwd_host.restype = _i
        L.mla_decode_host_workspace_size.argtypes = [_i, _i, _i, _i, _i]
        L.mla_decode_host_workspace_size.restype = _sz
        L.mla_decode_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _f, _i, _i, _vp,
                                      _sz, _vp]
        L.mla_decode_host.restype = _i
        L.mla_decode_workspace_size.argtypes = [_i, _i, _i, _i]
        L.mla_decode_workspace_size.restype = _sz
        L.mla_decode_split_workspace_size.argtypes = [_i, _i, _i, _i, _i]
        L.mla_decode_split_workspace_size.restype = _sz
        L.mla_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _f, _i, _i, _vp, _sz,
                                 _vp]
        L.mla_decode.restype = _i
        L.mla_decode_split.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _f, _i, _i, _vp,
                                       _sz, _i, _vp]
        L.mla_decode_split.restype = _i
        L.mla_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _f, _i, _i, _vp]
        L.mla_decode_noalloc.restype = _i
        L.mla_absorb_q.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]
        L.mla_absorb_q.restype = _i
        L.mla_project_out.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp]
        L.mla_project_out.restype = _i
        L.attn_device_status.argtypes = [_vp]
        L.attn_device_status.restype = _i
        L.attn_last_error.argtypes = []
        L.attn_last_error.restype = ctypes.c_char_p
        L.attn_kv_tiles.argtypes = [_i, _i, _i, _i, _i]
        L.attn_kv_tiles.restype = _i
        L.attn_kernel_info.argtypes = [_i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i),
                                       ctypes.POINTER(_i), ctypes.POINTER(_i)]
        L.attn_kernel_info.restype = _i
        _lib = L
    return _lib


def attn_last_error() -> str:
    return lib().attn_last_error().decode()


def _check(code: int):
    if code != ATTN_OK:
        raise AttnError(code, attn_last_error())


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _require(t, name, dtype, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def attn_fwd(q, k, v, o=None, lse=None, causal: bool = False, scale: float | None = None,
             stream=None):
    """Attention forward. q,k,v: [B,H,N,D] fp32 or bf16 CUDA tensors.

    Returns (o, lse): o like q, lse float32 [B,H,N].
    """
    import torch
    B, H, N, D = q.shape
    dt = q.dtype
    if dt == torch.float32:
        code = ATTN_DTYPE_F32
    elif dt == torch.bfloat16:
        code = ATTN_DTYPE_BF16
    else:
        raise ValueError(f"unsupported dtype {dt}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, dt, (B, H, N, D))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    _require(o, "o", dt, (B, H, N, D))
    _require(lse, "lse", torch.float32, (B, H, N))
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D,
                          int(bool(causal)), scale, code, _stream_ptr(stream)))
    return o, lse


def attn_fwd_tf32x3_workspace_size(B: int, H: int, N: int, D: int = 64) -> int:
    return int(lib().attn_fwd_tf32x3_workspace_size(B, H, N, D))


def attn_fwd_tf32x3(q, k, v, o=None, lse=None, causal: bool = False,
                    scale: float | None = None, workspace=None, stream=None):
    """fp32 attention forward on the tensor cores (three-product TF32 split).

    q, k, v: [B,H,N,64] float32 CUDA tensors.  Returns (o, lse) as attn_fwd.
    `workspace` (uint8, >= attn_fwd_tf32x3_workspace_size bytes) is allocated
    when not given.
    """
    import torch
    B, H, N, D = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, torch.float32, (B, H, N, D))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    _require(o, "o", torch.float32, (B, H, N, D))
    _require(lse, "lse", torch.float32, (B, H, N))
    if workspace is None:
        need = attn_fwd_tf32x3_workspace_size(B, H, N, D)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _require(workspace, "workspace", torch.uint8)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib().attn_fwd_tf32x3(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D,
                                 int(bool(causal)), scale, _ptr(workspace), workspace.numel(),
                                 _stream_ptr(stream)))
    return o, lse


def _require_host(t, name, dtype, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _device_workspace(workspace, need, device):
    import torch
    if workspace is None:
        # 256 bytes of slack for the alignment the library asks for
        raw = torch.empty(need + 256, dtype=torch.uint8, device=device)
        off = (-raw.data_ptr()) % 256
        workspace = raw[off:off + need]
    _require(workspace, "workspace", torch.uint8)
    return workspace


def attn_fwd_host_workspace_size(B: int, H: int, N: int, D: int, dtype: int) -> int:
    return int(lib().attn_fwd_host_workspace_size(B, H, N, D, dtype))


def attn_fwd_host(q, k, v, o=None, lse=None, causal: bool = False, scale: float | None = None,
                  workspace=None, stream=None):
    """attn_fwd on HOST tensors (page-locked ones overlap the copies).

    q, k, v: [B,H,N,D] fp32 or bf16 CPU tensors; returns (o, lse) on the host,
    valid once `stream` has reached the end of the call.
    """
    import torch
    B, H, N, D = q.shape
    dt = q.dtype
    code = ATTN_DTYPE_F32 if dt == torch.float32 else ATTN_DTYPE_BF16
    if dt not in (torch.float32, torch.bfloat16):
        raise ValueError(f"unsupported dtype {dt}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require_host(t, name, dt, (B, H, N, D))
    if o is None:
        o = torch.empty(B, H, N, D, dtype=dt, pin_memory=True)
    if lse is None:
        lse = torch.empty(B, H, N, dtype=torch.float32, pin_memory=True)
    _require_host(o, "o", dt, (B, H, N, D))
    _require_host(lse, "lse", torch.float32, (B, H, N))
    need = attn_fwd_host_workspace_size(B, H, N, D, code)
    workspace = _device_workspace(workspace, max(need, 16), torch.cuda.current_device())
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D,
                               int(bool(causal)), scale, code, _ptr(workspace),
                               workspace.numel(), _stream_ptr(stream)))
    return o, lse


def mla_decode_host_workspace_size(B: int, Hq: int, max_blocks_per_seq: int, num_blocks: int,
                                   num_sms: int) -> int:
    return int(lib().mla_decode_host_workspace_size(B, Hq, max_blocks_per_seq, num_blocks,
                                                    num_sms))


def mla_decode_host(q, kv_cache, block_table, seqlens, o=None, lse=None,
                    scale: float = 1.0 / math.sqrt(192.0), workspace=None, stream=None):
    """mla_decode on HOST tensors: q [B,128,576] bf16, pool [nb,64,576] bf16,
    block_table [B,max_blocks] int32, seqlens [B] int32; returns (o, lse) on the host."""
    import torch
    B, Hq, _ = q.shape
    _require_host(q, "q", torch.bfloat16, (B, Hq, MLA_DK))
    nb = kv_cache.shape[0]
    _require_host(kv_cache, "kv_cache", torch.bfloat16, (nb, MLA_PAGE, MLA_DK))
    _require_host(block_table, "block_table", torch.int32)
    _require_host(seqlens, "seqlens", torch.int32, (B,))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks_per_seq]")
    max_blocks = block_table.shape[1]
    if o is None:
        o = torch.empty(B, Hq, MLA_DV, dtype=torch.bfloat16, pin_memory=True)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, pin_memory=True)
    _require_host(o, "o", torch.bfloat16, (B, Hq, MLA_DV))
    _require_host(lse, "lse", torch.float32, (B, Hq))
    dev = torch.cuda.current_device()
    need = mla_decode_host_workspace_size(B, Hq, max_blocks, nb, _num_sms(dev))
    workspace = _device_workspace(workspace, max(need, 16), dev)
    _check(lib().mla_decode_host(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seqlens),
                                 _ptr(o), _ptr(lse), B, Hq, float(scale), max_blocks, nb,
                                 _ptr(workspace), workspace.numel(), _stream_ptr(stream)))
    return o, lse


def attn_fwd_test_skip_load(q, k, v, o, lse, causal: bool, scale: float, skip_load_index: int,
                            stream=None):
    """Test hook: bf16 attn_fwd whose producer never issues one K/V load."""
    B, H, N, D = q.shape
    _check(lib().attn_fwd_test_skip_load(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                         N, D, int(bool(causal)), float(scale),
                                         _stream_ptr(stream), int(skip_load_index)))


def attn_fwd_f32_test_skip_load(q, k, v, o, lse, causal: bool, scale: float, skip_block: int,
                                stream=None):
    """Test hook: fp32 attn_fwd (CUDA cores) in which no CTA loads one K/V block."""
    B, H, N, D = q.shape
    _check(lib().attn_fwd_f32_test_skip_load(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B,
                                             H, N, D, int(bool(causal)), float(scale),
                                             _stream_ptr(stream), int(skip_block)))


def attn_fwd_tf32x3_test_skip_load(q, k, v, o, lse, causal: bool, scale: float,
                                   workspace, skip_block: int, stream=None):
    """Test hook: attn_fwd_tf32x3 whose producers never load one K/V block."""
    B, H, N, D = q.shape
    _check(lib().attn_fwd_tf32x3_test_skip_load(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D, int(bool(causal)),
        float(scale), _ptr(workspace), workspace.numel(), _stream_ptr(stream), int(skip_block)))


def mla_decode_test_skip_load(q, kv_cache, block_table, seqlens, o, lse, scale: float,
                              workspace, skip_step: int, stream=None):
    """Test hook: mla_decode in which rank 1 of every cluster never loads one step."""
    B, Hq, _ = q.shape
    _check(lib().mla_decode_test_skip_load(
        _ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seqlens), _ptr(o), _ptr(lse), B, Hq,
        float(scale), block_table.shape[1], kv_cache.shape[0], _ptr(workspace),
        workspace.numel(), _stream_ptr(stream), int(skip_step)))


def mla_decode_workspace_size(B: int, Hq: int, max_blocks_per_seq: int, num_sms: int) -> int:
    return int(lib().mla_decode_workspace_size(B, Hq, max_blocks_per_seq, num_sms))


def mla_decode_split_workspace_size(B: int, Hq: int, max_blocks_per_seq: int, num_sms: int,
                                    pages_per_split: int = 0) -> int:
    return int(lib().mla_decode_split_workspace_size(B, Hq, max_blocks_per_seq, num_sms,
                                                     pages_per_split))


def _num_sms(device) -> int:
    import torch
    return torch.cuda.get_device_properties(device).multi_processor_count


def mla_decode_split(q, kv_cache, block_table, seqlens, o=None, lse=None,
                     scale: float = 1.0 / math.sqrt(192.0), workspace=None,
                     pages_per_split: int = 0, stream=None):
    """MLA absorbed decode with an explicit split length (0 = automatic)."""
    import torch
    B, Hq, Dk = q.shape
    _require(q, "q", torch.bfloat16, (B, Hq, MLA_DK))
    nb, page, dk2 = kv_cache.shape
    _require(kv_cache, "kv_cache", torch.bfloat16, (nb, MLA_PAGE, MLA_DK))
    _require(block_table, "block_table", torch.int32)
    _require(seqlens, "seqlens", torch.int32, (B,))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks_per_seq]")
    max_blocks = block_table.shape[1]
    if o is None:
        o = torch.empty(B, Hq, MLA_DV, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    _require(o, "o", torch.bfloat16, (B, Hq, MLA_DV))
    _require(lse, "lse", torch.float32, (B, Hq))
    need = mla_decode_split_workspace_size(B, Hq, max_blocks, _num_sms(q.device),
                                           pages_per_split)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _require(workspace, "workspace", torch.uint8)
    _check(lib().mla_decode_split(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seqlens),
                                  _ptr(o), _ptr(lse), B, Hq, float(scale), max_blocks, nb,
                                  _ptr(workspace), workspace.numel(), int(pages_per_split),
                                  _stream_ptr(stream)))
    return o, lse


def mla_decode(q, kv_cache, block_table, seqlens, o=None, lse=None,
               scale: float = 1.0 / math.sqrt(192.0), workspace=None, stream=None):
    """MLA absorbed decode: q [B,128,576] bf16, paged latent pool [nb,64,576] bf16."""
    return mla_decode_split(q, kv_cache, block_table, seqlens, o, lse, scale, workspace, 0,
                            stream)


def mla_decode_noalloc(q, kv_cache, block_table, seqlens, o=None, lse=None,
                       scale: float = 1.0 / math.sqrt(192.0), stream=None):
    """MLA decode without a workspace: the library's fixed device scratch is used.

    For callers that may not allocate device memory when they call, so this
    wrapper allocates nothing either: o ([B,Hq,512] bf16) and lse ([B,Hq]
    float32) must be passed in.  Calls that can overlap on the GPU share the
    one scratch array and must be serialised by the caller.
    """
    import torch
    B, Hq, _ = q.shape
    _require(q, "q", torch.bfloat16, (B, Hq, MLA_DK))
    nb = kv_cache.shape[0]
    _require(kv_cache, "kv_cache", torch.bfloat16, (nb, MLA_PAGE, MLA_DK))
    _require(block_table, "block_table", torch.int32)
    _require(seqlens, "seqlens", torch.int32, (B,))
    if o is None or lse is None:
        raise ValueError("mla_decode_noalloc allocates nothing: pass o and lse")
    _require(o, "o", torch.bfloat16, (B, Hq, MLA_DV))
    _require(lse, "lse", torch.float32, (B, Hq))
    _check(lib().mla_decode_noalloc(_ptr(q), _ptr(kv_cache), _ptr(block_table),
                                    _ptr(seqlens), _ptr(o), _ptr(lse), B, Hq, float(scale),
                                    block_table.shape[1], nb, _stream_ptr(stream)))
    return o, lse


def mla_absorb_q(q_nope, q_rope, w_uk, q_out=None, stream=None):
    """The absorbed query [q_nope_h W_UK_h | q_rope_h] that mla_decode takes.

    q_nope [B,Hq,d_nope], q_rope [B,Hq,d_rope], w_uk [Hq,d_nope,d_latent], bf16.
    Returns q_out [B,Hq,d_latent+d_rope] bf16.
    """
    import torch
    B, Hq, d_nope = q_nope.shape
    d_rope = q_rope.shape[2]
    d_latent = w_uk.shape[2]
    _require(q_nope, "q_nope", torch.bfloat16, (B, Hq, d_nope))
    _require(q_rope, "q_rope", torch.bfloat16, (B, Hq, d_rope))
    _require(w_uk, "w_uk", torch.bfloat16, (Hq, d_nope, d_latent))
    if q_out is None:
        q_out = torch.empty(B, Hq, d_latent + d_rope, dtype=torch.bfloat16, device=q_nope.device)
    _require(q_out, "q_out", torch.bfloat16, (B, Hq, d_latent + d_rope))
    _check(lib().mla_absorb_q(_ptr(q_nope), _ptr(q_rope), _ptr(w_uk), _ptr(q_out), B, Hq,
                              d_nope, d_rope, d_latent, _stream_ptr(stream)))
    return q_out


def mla_project_out(o_latent, w_uv, out=None, stream=None):
    """Each head's output o_latent_h W_UV_h.  o_latent [B,Hq,d_latent], w_uv
    [Hq,d_latent,d_v], bf16; returns out [B,Hq,d_v] bf16."""
    import torch
    B, Hq, d_latent = o_latent.shape
    d_v = w_uv.shape[2]
    _require(o_latent, "o_latent", torch.bfloat16, (B, Hq, d_latent))
    _require(w_uv, "w_uv", torch.bfloat16, (Hq, d_latent, d_v))
    if out is None:
        out = torch.empty(B, Hq, d_v, dtype=torch.bfloat16, device=o_latent.device)
    _require(out, "out", torch.bfloat16, (B, Hq, d_v))
    _check(lib().mla_project_out(_ptr(o_latent), _ptr(w_uv), _ptr(out), B, Hq, d_latent, d_v,
                                 _stream_ptr(stream)))
    return out


def attn_device_status(stream=None, raise_on_error: bool = True) -> int:
    code = lib().attn_device_status(_stream_ptr(stream))
    if raise_on_error:
        _check(code)
    return code


def attn_kv_tiles(N: int, Br: int, Bc: int, causal: bool, q_tile: int) -> int:
    return lib().attn_kv_tiles(N, Br, Bc, int(bool(causal)), q_tile)


def attn_kernel_info(dtype: int, D: int):
    vals = [ctypes.c_int() for _ in range(4)]
    _check(lib().attn_kernel_info(dtype, D, *[ctypes.byref(x) for x in vals]))
    return dict(zip(("Br", "Bc", "threads", "smem_bytes"), (x.value for x in vals)))
