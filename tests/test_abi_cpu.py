"""CPU-only checks of the C ABI: the library builds and loads, exports every
symbol include/linear_logp.h declares, sizes workspaces, and rejects bad
arguments with the documented status codes before touching any device.

No call here launches work: every call either is a pure host query or fails
validation (or is the N == 0 no-op) before the first CUDA runtime call.
"""
import ctypes
import os
import re

import pytest

from lm_head_selected_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "linear_logp.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**(linear_logp_[a-z_0-9]+)\s*\(", text, re.M)))


def test_header_declares_the_abi():
    names = _declared_functions()
    assert "linear_logp_fwd" in names and "linear_logp_bwd" in names
    assert set(names) == set(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(-7, 1):
        assert len(_lib.status_string(code)) > 0
    assert _lib.status_string(0) == "ok"


def test_workspace_queries(lib):
    fwd = lib.linear_logp_fwd_workspace_bytes
    bwd = lib.linear_logp_bwd_workspace_bytes
    assert fwd(0, 256, 4096) == 0
    S = (131072 + 511) // 512
    n = 16384
    assert fwd(n, 2688, 131072) >= 2 * S * n * 4 + n * 4
    # dlogits bf16 [N, round_up(V, 64)] dominates the backward workspace
    assert bwd(n, 2688, 131072, 0) >= n * 131072 * 2
    assert bwd(n, 2688, 131072, 1) > bwd(n, 2688, 131072, 0)
    # grad_weight partials appear once N exceeds one 32768-token segment
    assert bwd(65600, 2688, 131072, 0) >= 65600 * 131072 * 2 + 3 * 131072 * 2688 * 4
    # V = 1000 pads the dlogits rows to 1024 columns
    assert bwd(10, 64, 1000, 0) >= 10 * 1024 * 2
    # invalid shapes report 0
    assert fwd(4, 12, 10) == 0 and bwd(4, 0, 10, 0) == 0


P = ctypes.c_void_p


def _fwd(lib, hidden=0x1000, weight=0x2000, bias=None, targets=0x3000, temp=None, N=4, D=64, V=100,
         logp=0x4000, lse=0x5000, ws=0x6000, wsb=1 << 30):
    return lib.linear_logp_fwd(P(hidden) if hidden else None, P(weight) if weight else None,
                               P(bias) if bias else None, P(targets) if targets else None,
                               P(temp) if temp else None, N, D, V, -100,
                               P(logp) if logp else None, P(lse) if lse else None,
                               P(ws) if ws else None, wsb, None)


def test_fwd_rejects_bad_arguments_on_host(lib):
    assert _fwd(lib, hidden=0) == _lib.LLP_ERR_NULL_POINTER
    assert _fwd(lib, weight=0) == _lib.LLP_ERR_NULL_POINTER
    assert _fwd(lib, targets=0) == _lib.LLP_ERR_NULL_POINTER
    assert _fwd(lib, logp=0) == _lib.LLP_ERR_NULL_POINTER
    assert _fwd(lib, lse=0) == _lib.LLP_ERR_NULL_POINTER
    assert _fwd(lib, ws=0) == _lib.LLP_ERR_NULL_POINTER
    assert _fwd(lib, D=12) == _lib.LLP_ERR_BAD_SHAPE
    assert _fwd(lib, D=0) == _lib.LLP_ERR_BAD_SHAPE
    assert _fwd(lib, V=0) == _lib.LLP_ERR_BAD_SHAPE
    assert _fwd(lib, N=-1) == _lib.LLP_ERR_BAD_SHAPE
    assert _fwd(lib, N=1 << 31) == _lib.LLP_ERR_BAD_SHAPE
    assert _fwd(lib, hidden=0x1008) == _lib.LLP_ERR_MISALIGNED
    assert _fwd(lib, weight=0x2004) == _lib.LLP_ERR_MISALIGNED
    assert _fwd(lib, targets=0x3004) == _lib.LLP_ERR_MISALIGNED
    assert _fwd(lib, bias=0x7002) == _lib.LLP_ERR_MISALIGNED
    assert _fwd(lib, temp=0x7002) == _lib.LLP_ERR_MISALIGNED
    assert _fwd(lib, ws=0x6008) == _lib.LLP_ERR_MISALIGNED
    need = lib.linear_logp_fwd_workspace_bytes(4, 64, 100)
    assert _fwd(lib, wsb=need - 1) == _lib.LLP_ERR_WORKSPACE_TOO_SMALL
    # N == 0 is a no-op that succeeds without touching the device
    assert _fwd(lib, N=0, ws=0, wsb=0) == _lib.LLP_OK


def _bwd(lib, g=0x1000, lse=0x1100, hidden=0x2000, weight=0x3000, bias=None, targets=0x4000, temp=None,
         N=4, D=64, V=100, gh=0x5000, gw=0x6000, gb=None, ws=0x7000, wsb=1 << 30):
    f = lambda x: P(x) if x else None  # noqa: E731
    return lib.linear_logp_bwd(f(g), f(lse), f(hidden), f(weight), f(bias), f(targets), f(temp), N, D, V, -100,
                               f(gh), f(gw), f(gb), f(ws), wsb, None)


def test_bwd_rejects_bad_arguments_on_host(lib):
    assert _bwd(lib, g=0) == _lib.LLP_ERR_NULL_POINTER
    assert _bwd(lib, lse=0) == _lib.LLP_ERR_NULL_POINTER
    assert _bwd(lib, hidden=0) == _lib.LLP_ERR_NULL_POINTER
    assert _bwd(lib, gb=0x8000) == _lib.LLP_ERR_NULL_POINTER  # grad_bias without bias
    assert _bwd(lib, ws=0) == _lib.LLP_ERR_NULL_POINTER
    assert _bwd(lib, D=20) == _lib.LLP_ERR_BAD_SHAPE
    assert _bwd(lib, gh=0x5008) == _lib.LLP_ERR_MISALIGNED
    assert _bwd(lib, gw=0x6002) == _lib.LLP_ERR_MISALIGNED
    assert _bwd(lib, g=0x1002) == _lib.LLP_ERR_MISALIGNED
    need = lib.linear_logp_bwd_workspace_bytes(4, 64, 100, 0)
    assert _bwd(lib, wsb=need - 1) == _lib.LLP_ERR_WORKSPACE_TOO_SMALL
    # nothing requested: no-op
    assert _bwd(lib, gh=0, gw=0, gb=0) == _lib.LLP_OK


def test_fused_header_and_exports(lib):
    with open(os.path.join(ROOT, "include", "fused_logp.h")) as f:
        text = f.read()
    names = set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**(fused_logp_[a-z_0-9]+)\s*\(", text, re.M))
    assert names == set(_lib.EXPORTED_FUSED)
    for n in names:
        assert hasattr(lib, n)


def test_fused_rejects_bad_arguments_on_host(lib):
    f = lambda x: P(x) if x else None  # noqa: E731
    fwd = lambda **k: lib.fused_logp_fwd(  # noqa: E731
        f(k.get("z", 0x1000)), k.get("dt", 0), k.get("N", 4), k.get("V", 100), f(k.get("t", 0x2000)), -100,
        f(k.get("lp", 0x3000)), f(k.get("m", 0x4000)), f(k.get("ls", 0x5000)), f(k.get("ws", 0x6000)),
        k.get("wsb", 1 << 20), None)
    assert fwd(dt=3) == _lib.LLP_ERR_BAD_SHAPE  # dtypes: 0 bf16, 1 fp32, 2 fp16
    assert fwd(V=0) == _lib.LLP_ERR_BAD_SHAPE
    assert fwd(z=0) == _lib.LLP_ERR_NULL_POINTER
    assert fwd(t=0) == _lib.LLP_ERR_NULL_POINTER
    assert fwd(lp=0) == _lib.LLP_ERR_NULL_POINTER
    assert fwd(z=0x1001) == _lib.LLP_ERR_MISALIGNED
    assert fwd(dt=1, z=0x1002) == _lib.LLP_ERR_MISALIGNED
    assert fwd(wsb=lib.fused_logp_workspace_bytes(4, 100) - 1) == _lib.LLP_ERR_WORKSPACE_TOO_SMALL
    assert fwd(N=0, z=0, t=0, lp=0, m=0, ls=0, ws=0) == _lib.LLP_OK
    assert lib.fused_logp_workspace_bytes(16384, 131072) == 2 * 8 * 16384 * 4
    assert lib.fused_logp_bwd(None, f(0x10), f(0x20), f(0x1000), 0, 4, 100, f(0x2000), -100, f(0x3000),
                              None) == _lib.LLP_ERR_NULL_POINTER
    assert lib.fused_logp_bwd(f(0x10), f(0x20), f(0x30), f(0x1000), 0, 4, 100, f(0x2000), -100, f(0x3001),
                              None) == _lib.LLP_ERR_MISALIGNED


def test_selftest_limit_is_checked_on_host(lib):
    assert lib.linear_logp_selftest_wait_timeout(0, None) == _lib.LLP_ERR_BAD_SHAPE
    assert lib.linear_logp_selftest_wait_timeout(2_000_000_000, None) == _lib.LLP_ERR_BAD_SHAPE


def test_noalloc_limits_are_checked_on_host(lib):
    f = lambda x: P(x) if x else None  # noqa: E731
    # 9000 tokens at V = 131072 need about 18.4 MB > 16 MiB of scratch: refused before any device call
    st = lib.linear_logp_fwd_noalloc(f(0x1000), f(0x2000), None, f(0x3000), None, 9000, 2688, 131072, -100,
                                     f(0x4000), f(0x5000), None)
    assert st == _lib.LLP_ERR_SCRATCH_LIMIT
    assert lib.linear_logp_fwd_noalloc(None, f(0x2000), None, f(0x3000), None, 4, 64, 100, -100, f(0x4000),
                                       f(0x5000), None) == _lib.LLP_ERR_NULL_POINTER
    assert lib.linear_logp_fwd_noalloc(None, None, None, None, None, 0, 64, 100, -100, None, None,
                                       None) == _lib.LLP_OK


def test_python_wrapper_fails_closed_without_gpu():
    import torch
    import lm_head_selected_gb300 as llp
    h = torch.zeros(4, 64, dtype=torch.bfloat16)
    w = torch.zeros(10, 64, dtype=torch.bfloat16)
    t = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError):
        llp.linear_logp_fwd(h, w, t)
