"""The C ABI library loads on any host and exports what include/attn.h declares.

These checks make no compute call: invalid arguments are rejected by host
validation before any CUDA call, and the helpers are pure host arithmetic.
"""
import ctypes
import os
import re
import subprocess

import pytest

import online_softmax_attention_attn_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"^#.*$", "", text, flags=re.M)
    return sorted(set(re.findall(r"^ATTN_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(pkg.LIB_PATH):
        from online_softmax_attention_attn_gb300 import _build
        _build.build()
    return pkg.lib()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ["attn_fwd", "mla_decode", "mla_decode_split", "mla_decode_workspace_size",
              "mla_decode_split_workspace_size",
              "attn_device_status", "attn_last_error", "attn_kv_tiles", "attn_kernel_info",
              "attn_fwd_test_skip_load", "attn_fwd_f32_test_skip_load", "mla_absorb_q",
              "mla_project_out",
              "attn_fwd_tf32x3", "attn_fwd_tf32x3_workspace_size", "attn_fwd_host",
              "attn_fwd_host_workspace_size", "mla_decode_host",
              "mla_decode_host_workspace_size"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", pkg.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _declared_functions():
        assert name in exported, f"{name} declared in attn.h but not exported"
        assert hasattr(L, name)


def test_only_the_boundary_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", pkg.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {n for n in exported if n.startswith(("attn_", "mla_"))}
    assert ours == set(_declared_functions())


def test_null_pointers_are_rejected_before_any_cuda_call(L):
    rc = L.attn_fwd(None, None, None, None, None, 1, 1, 16, 64, 0, 0.125, 0, None)
    assert rc == pkg.ATTN_ERR_INVALID_ARG
    assert "null" in pkg.attn_last_error()


def test_bad_sizes_dtype_and_head_dim(L):
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    assert L.attn_fwd(p, p, p, p, p, 0, 1, 16, 64, 0, 0.1, 0, None) == pkg.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd(p, p, p, p, p, 1, 1, 16, 64, 0, float("nan"), 0, None) == \
        pkg.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd(p, p, p, p, p, 1, 1, 16, 96, 0, 0.1, 1, None) == pkg.ATTN_ERR_UNSUPPORTED
    assert L.attn_fwd(p, p, p, p, p, 1, 1, 16, 128, 0, 0.1, 0, None) == pkg.ATTN_ERR_UNSUPPORTED
    assert L.attn_fwd(p, p, p, p, p, 1, 1, 16, 64, 0, 0.1, 7, None) == pkg.ATTN_ERR_UNSUPPORTED
    q = ctypes.c_void_p(24)  # not 16-byte aligned
    assert L.attn_fwd(q, p, p, p, p, 1, 1, 16, 64, 0, 0.1, 0, None) == pkg.ATTN_ERR_MISALIGNED


def test_mla_argument_checks(L):
    p = ctypes.c_void_p(16)
    args = [p, p, p, p, p, p]
    assert L.mla_decode(*args, 1, 128, 0.1, 4, 4, None, 0, None) == pkg.ATTN_ERR_INVALID_ARG
    assert L.mla_decode(*args, 1, 64, 0.1, 4, 4, p, 1 << 20, None) == pkg.ATTN_ERR_UNSUPPORTED
    assert L.mla_decode(*args, 0, 128, 0.1, 4, 4, p, 1 << 20, None) == pkg.ATTN_ERR_INVALID_ARG
    assert L.mla_decode(*args, 1, 128, float("inf"), 4, 4, p, 1 << 20, None) == \
        pkg.ATTN_ERR_INVALID_ARG


def test_workspace_size_is_host_arithmetic(L):
    assert pkg.mla_decode_workspace_size(0, 128, 64, 152) == 0
    assert pkg.mla_decode_workspace_size(4, 128, 64, 1) == 0
    a = pkg.mla_decode_workspace_size(64, 128, 64, 152)
    b = pkg.mla_decode_split_workspace_size(64, 128, 64, 152, pages_per_split=1)
    assert a > 0 and b >= a
    assert pkg.mla_decode_split_workspace_size(64, 128, 64, 152, pages_per_split=0) == a
    assert pkg.mla_decode_split_workspace_size(64, 128, 64, 152, pages_per_split=-1) == 0


def test_kernel_info(L):
    f32 = pkg.attn_kernel_info(pkg.ATTN_DTYPE_F32, 64)
    assert f32["Br"] == 128 and f32["threads"] == 256
    bf = pkg.attn_kernel_info(pkg.ATTN_DTYPE_BF16, 128)
    assert bf["Br"] == 128 and bf["Bc"] == 128 and bf["smem_bytes"] <= 232448
    with pytest.raises(pkg.AttnError):
        pkg.attn_kernel_info(pkg.ATTN_DTYPE_F32, 80)


def test_projection_arguments_are_checked_before_any_cuda_call(L):
    """The absorption GEMMs reject bad arguments on the host (no GPU needed)."""
    rc = L.mla_absorb_q(None, None, None, None, 4, 128, 128, 64, 512, None)
    assert rc == pkg.ATTN_ERR_INVALID_ARG and "null pointer" in pkg.attn_last_error()
    import ctypes
    buf = ctypes.create_string_buffer(256)
    p = ctypes.cast(ctypes.addressof(buf), ctypes.c_void_p)
    aligned = ctypes.c_void_p((p.value + 15) & ~15)
    rc = L.mla_absorb_q(aligned, aligned, aligned, aligned, 4, 128, 100, 64, 512, None)
    assert rc == pkg.ATTN_ERR_INVALID_ARG and "multiples of 8" in pkg.attn_last_error()
    rc = L.mla_project_out(aligned, aligned, aligned, 0, 128, 512, 128, None)
    assert rc == pkg.ATTN_ERR_INVALID_ARG
    odd = ctypes.c_void_p(aligned.value + 2)
    rc = L.mla_project_out(odd, aligned, aligned, 4, 128, 512, 128, None)
    assert rc == pkg.ATTN_ERR_MISALIGNED


def test_tf32x3_workspace_and_argument_checks(L):
    """attn_fwd_tf32x3: workspace arithmetic and host-side rejections."""
    # split K: 2 x BH*N*64 floats; split V^T: 2 x BH*64*ceil64(N) floats
    assert pkg.attn_fwd_tf32x3_workspace_size(4, 8, 8192, 64) == 4 * 32 * 8192 * 64 * 4
    assert pkg.attn_fwd_tf32x3_workspace_size(1, 2, 100, 64) == \
        2 * 2 * 100 * 256 + 2 * 2 * 64 * 128 * 4
    assert pkg.attn_fwd_tf32x3_workspace_size(1, 1, 16, 128) == 0
    assert pkg.attn_fwd_tf32x3_workspace_size(0, 1, 16, 64) == 0
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    rc = L.attn_fwd_tf32x3(None, p, p, p, p, 1, 1, 16, 64, 0, 0.1, p, 1 << 20, None)
    assert rc == pkg.ATTN_ERR_INVALID_ARG and "null" in pkg.attn_last_error()
    rc = L.attn_fwd_tf32x3(p, p, p, p, p, 1, 1, 16, 64, 0, float("nan"), p, 1 << 20, None)
    assert rc == pkg.ATTN_ERR_INVALID_ARG
    rc = L.attn_fwd_tf32x3(p, p, p, p, p, 1, 1, 16, 128, 0, 0.1, p, 1 << 20, None)
    assert rc == pkg.ATTN_ERR_UNSUPPORTED
    rc = L.attn_fwd_tf32x3(p, p, p, p, ctypes.c_void_p(20), 1, 1, 16, 64, 0, 0.1, p, 1 << 20,
                           None)
    assert rc == pkg.ATTN_ERR_MISALIGNED
    need = pkg.attn_fwd_tf32x3_workspace_size(1, 1, 16, 64)
    rc = L.attn_fwd_tf32x3(p, p, p, p, p, 1, 1, 16, 64, 0, 0.1, p, need - 1, None)
    assert rc == pkg.ATTN_ERR_WORKSPACE_TOO_SMALL


def test_host_entry_workspace_and_argument_checks(L):
    """attn_fwd_host / mla_decode_host: workspace arithmetic, host-side rejections."""
    # 4 chunks of ceil(6/4) = 2 heads: two buffers of [q|k|v|o] + lse
    per = 2 * 300 * 128 * 2
    lse = 2 * 300 * 4
    r256 = lambda x: (x + 255) // 256 * 256
    assert pkg.attn_fwd_host_workspace_size(2, 3, 300, 128, pkg.ATTN_DTYPE_BF16) == \
        2 * (4 * r256(per) + r256(lse))
    # a single head is one chunk: one buffer
    assert pkg.attn_fwd_host_workspace_size(1, 1, 64, 64, pkg.ATTN_DTYPE_F32) == \
        4 * r256(64 * 64 * 4) + r256(64 * 4)
    assert pkg.attn_fwd_host_workspace_size(1, 1, 64, 128, pkg.ATTN_DTYPE_F32) == 0
    assert pkg.attn_fwd_host_workspace_size(1, 1, 64, 64, 7) == 0
    assert pkg.mla_decode_host_workspace_size(4, 128, 8, 32, 152) > 32 * 64 * 576 * 2
    assert pkg.mla_decode_host_workspace_size(4, 64, 8, 32, 152) == 0
    p = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    assert L.attn_fwd_host(None, p, p, p, p, 1, 1, 16, 64, 0, 0.1, 0, p, 1 << 20, None) == \
        pkg.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_host(p, p, p, p, p, 1, 1, 16, 96, 0, 0.1, 1, p, 1 << 20, None) == \
        pkg.ATTN_ERR_UNSUPPORTED
    assert L.attn_fwd_host(p, p, p, p, p, 1, 1, 16, 64, 0, 0.1, 0, ctypes.c_void_p(272),
                           1 << 20, None) == pkg.ATTN_ERR_MISALIGNED
    assert L.attn_fwd_host(p, p, p, p, p, 1, 1, 16, 64, 0, 0.1, 0, p, 16, None) == \
        pkg.ATTN_ERR_WORKSPACE_TOO_SMALL
    args = [p] * 6
    assert L.mla_decode_host(*args, 1, 128, 0.1, 4, 4, None, 0, None) == pkg.ATTN_ERR_INVALID_ARG
    assert L.mla_decode_host(*args, 1, 64, 0.1, 4, 4, p, 1 << 20, None) == \
        pkg.ATTN_ERR_UNSUPPORTED
