"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any CUDA call.
"""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from online_softmax_fa_gb300.build import build_library
    from online_softmax_fa_gb300 import fa
    build_library()
    return fa.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", src, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fa_fwd", "fa_fwd_gqa", "fa_decode", "fa_decode_workspace_bytes", "fa_fwd_host", "fa_fwd_host_workspace_bytes", "fa_device_error",
                 "fa_status_string", "fa_selftest_bounded_wait", "fa_version"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    from online_softmax_fa_gb300 import fa
    for code in range(0, -13, -1):
        s = fa.fa_status_string(code)
        assert s and s != "unknown status"
    assert fa.fa_status_string(-999) == "unknown status"
    assert fa.fa_version() >= 100


def _call(lib, Q=16, K=32, V=48, O=4096, L=8192, B=1, H=1, N=8, d=64, causal=0,
          scale=0.125):
    return lib.fa_fwd(Q, K, V, O, L, B, H, N, d, causal, scale, None)


# Fake, never-dereferenced addresses: the checks below must reject each
# request on the host before any pointer is touched.
def test_null_pointers(lib):
    assert _call(lib, Q=None) == -1
    assert _call(lib, L=None) == -1


def test_bad_shapes(lib):
    assert _call(lib, B=0) == -2
    assert _call(lib, N=0) == -2
    assert _call(lib, H=-1) == -2
    assert _call(lib, B=1 << 16, H=1 << 16) == -2
    assert _call(lib, d=96) == -3
    assert _call(lib, d=512) == -3


def test_head_dim_256(lib):
    # the forward, the backward and decoding take d = 256 (checks pass up to
    # the device check); other head dimensions are rejected
    assert _call(lib, Q=1 << 20, K=2 << 20, V=3 << 20, O=4 << 20, L=5 << 20, d=256) in (0, -5)
    # the backward's workspace does not depend on d: two fp32 per padded row
    assert lib.fa_bwd_workspace_bytes(1, 1, 8, 256) == lib.fa_bwd_workspace_bytes(1, 1, 8, 128) > 0
    assert lib.fa_decode_workspace_bytes(1, 1, 1, 8, 256) > 0
    assert lib.fa_bwd_workspace_bytes(1, 1, 8, 96) == 0
    assert _call(lib, d=96) == -3


def test_bad_scale(lib):
    assert _call(lib, scale=0.0) == -9
    assert _call(lib, scale=-1.0) == -9
    assert _call(lib, scale=float("inf")) == -9
    assert _call(lib, scale=float("nan")) == -9


def test_alignment(lib):
    assert _call(lib, Q=17) == -4
    assert _call(lib, O=4104) == -4
    assert _call(lib, L=8194) == -4


def test_aliasing(lib):
    # [1,1,8,64] bf16 = 1024 bytes per tensor
    assert _call(lib, Q=1 << 20, O=(1 << 20) + 512) == -10
    assert _call(lib, V=1 << 20, L=(1 << 20) + 1020) == -10
    assert _call(lib, O=1 << 20, L=(1 << 20) + 4) == -10


def test_host_variant_checks(lib):
    need = lib.fa_fwd_host_workspace_bytes(1, 2, 300, 64)
    assert need >= 4 * 2 * 300 * 64 * 2 + 2 * 300 * 4
    assert need % 256 == 0
    assert lib.fa_fwd_host_workspace_bytes(1, 1, 8, 96) == 0
    args = (16, 32, 48, 64, 80)
    assert lib.fa_fwd_host(*args, None, need, 1, 2, 300, 64, 0, 0.1, None) == -11
    assert lib.fa_fwd_host(*args, 1 << 20, need - 1, 1, 2, 300, 64, 0, 0.1, None) == -11
    assert lib.fa_fwd_host(*args, (1 << 20) + 16, need, 1, 2, 300, 64, 0, 0.1, None) == -11
    assert lib.fa_fwd_host(None, 32, 48, 64, 80, 1 << 20, need, 1, 2, 300, 64, 0, 0.1,
                           None) == -1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_request_without_gpu_reports_arch(lib):
    # valid arguments, but no sm_103 device: nothing may be enqueued
    assert _call(lib, Q=1 << 20, K=2 << 20, V=3 << 20, O=4 << 20, L=5 << 20) == -5
    assert lib.fa_selftest_bounded_wait(1000, None) == -5
    assert lib.fa_selftest_bounded_wait(0, None) == -2


def declared_debug_functions():
    src = open(os.path.join(ROOT, "include", "fa_debug.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", src, re.M)))


def test_debug_library_exports(lib):
    """The debug build exports fa.h and fa_debug.h; the release build only fa.h."""
    from online_softmax_fa_gb300 import fa
    dbg = fa.load_debug_library()
    assert declared_debug_functions() == ["fa_debug_arm"]
    for name in declared_functions() + declared_debug_functions():
        assert hasattr(dbg, name), name
    assert not hasattr(lib, "fa_debug_arm")


def test_debug_arm_checks(lib):
    from online_softmax_fa_gb300 import fa
    dbg = fa.load_debug_library()
    assert dbg.fa_debug_arm(3, 0, 0, 0) == -8
    assert dbg.fa_debug_arm(fa.FA_DEBUG_LOSE_K_ARRIVAL, -1, 0, 0) == -2
    assert dbg.fa_debug_arm(fa.FA_DEBUG_LOSE_K_ARRIVAL, 0, -1, 0) == -2
    assert dbg.fa_debug_arm(fa.FA_DEBUG_SHRINK_OUTPUT, 5, 0, 1000001) == -2
    assert dbg.fa_debug_arm(fa.FA_DEBUG_SHRINK_OUTPUT, 5, 0, 1000) == 0
    assert dbg.fa_debug_arm(fa.FA_DEBUG_NONE, 0, 0, 0) == 0  # disarm
    # no device status was read on this thread: nothing to report
    assert dbg.fa_last_device_status() == 0
    assert fa.fa_status_string(-12) != "unknown status"


def test_binding_fails_loudly_without_library(tmp_path):
    from online_softmax_fa_gb300 import fa
    saved = fa._lib
    try:
        fa._lib = None
        with pytest.raises(RuntimeError, match="not found"):
            fa.load_library(str(tmp_path / "missing.so"))
    finally:
        fa._lib = saved


def test_gqa_argument_checks(lib):
    base = (16, 32, 48, 4096, 8192)
    # H_kv must divide H and be >= 1
    assert lib.fa_fwd_gqa(*base, 1, 8, 3, 8, 64, 0, 0.125, None) == -2
    assert lib.fa_fwd_gqa(*base, 1, 8, 0, 8, 64, 0, 0.125, None) == -2
    assert lib.fa_fwd_gqa(None, 32, 48, 4096, 8192, 1, 8, 2, 8, 64, 0, 0.125, None) == -1
    assert lib.fa_fwd_gqa(*base, 1, 8, 2, 8, 96, 0, 0.125, None) == -3


def test_bwd_gqa_argument_checks(lib):
    # Q K V O dO LSE dQ dK dV workspace bytes
    base = (16, 32, 48, 64, 80, 96, 4096, 8192, 12288, 65536, 1 << 30)
    # H_kv must divide H and be >= 1; head dimension 64, 128 or 256; null pointers
    assert lib.fa_bwd_gqa(*base, 1, 8, 3, 8, 64, 0, 0.125, None) == -2
    assert lib.fa_bwd_gqa(*base, 1, 8, 0, 8, 64, 0, 0.125, None) == -2
    assert lib.fa_bwd_gqa(*base, 1, 8, 2, 8, 96, 0, 0.125, None) == -3
    assert lib.fa_bwd_gqa(None, *base[1:], 1, 8, 2, 8, 64, 0, 0.125, None) == -1


def test_decode_argument_checks(lib):
    need = lib.fa_decode_workspace_bytes(2, 8, 2, 1000, 128)
    assert need > 0 and need % 256 == 0
    assert lib.fa_decode_workspace_bytes(2, 12, 1, 1000, 128) == 0  # group 12 unsupported
    assert lib.fa_decode_workspace_bytes(2, 8, 3, 1000, 128) == 0   # 3 does not divide 8
    ws = 1 << 24
    args = (16, 1 << 20, 2 << 20, 4096, 8192)
    assert lib.fa_decode(*args, ws, need, 2, 12, 1, 1000, 128, 0.1, None) == -8
    assert lib.fa_decode(*args, ws, need, 2, 8, 2, 1000, 96, 0.1, None) == -3
    assert lib.fa_decode(*args, None, need, 2, 8, 2, 1000, 128, 0.1, None) == -11
    assert lib.fa_decode(*args, ws, need - 1, 2, 8, 2, 1000, 128, 0.1, None) == -11
    assert lib.fa_decode(*args, ws + 16, need, 2, 8, 2, 1000, 128, 0.1, None) == -11
    assert lib.fa_decode(None, 1 << 20, 2 << 20, 4096, 8192, ws, need, 2, 8, 2, 1000, 128,
                         0.1, None) == -1
    assert lib.fa_decode(*args, ws, need, 2, 8, 2, 1000, 128, 0.0, None) == -9
