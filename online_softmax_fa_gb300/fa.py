"""ctypes binding of the C ABI in ``include/fa.h`` -- argument marshalling only.

Every step of the attention forward pass runs in the CUDA library
``_build/libfa_gb300.so``; this module passes pointers, sizes and the
current torch stream.  There is no fallback: if the library is missing or a
call fails, it raises.
"""
from __future__ import annotations

import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfa_gb300.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "_build", "libfa_gb300_debug.so")

FA_OK = 0
FA_ERR_TIMEOUT = -7
FA_ERR_CHECK = -12
# include/fa_debug.h
FA_DEBUG_NONE = 0
FA_DEBUG_LOSE_K_ARRIVAL = 1
FA_DEBUG_SHRINK_OUTPUT = 2

_lib = None
_debug_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = load_library().fa_last_error_detail().decode()
        super().__init__(f"{where}: {fa_status_string(status)} (status {status})"
                         + (f" [{detail}]" if detail else ""))


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load (once) the in-tree CUDA library; raise if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = _open(path or LIB_PATH)
    return _lib


def load_debug_library() -> ctypes.CDLL:
    """Load (once) the debug build (include/fa_debug.h): a handle of its own,
    with every fa.h function plus fa_debug_arm.  The module-level functions
    below keep using the release library."""
    global _debug_lib
    if _debug_lib is None:
        lib = _open(DEBUG_LIB_PATH)
        lib.fa_debug_arm.argtypes = [ctypes.c_int, ctypes.c_longlong, ctypes.c_longlong,
                                     ctypes.c_int]
        lib.fa_debug_arm.restype = ctypes.c_int
        _debug_lib = lib
    return _debug_lib


def _open(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P]
    lib.fa_fwd.restype = I
    lib.fa_fwd_gqa.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
    lib.fa_fwd_gqa.restype = I
    lib.fa_fwd_host_workspace_bytes.argtypes = [I, I, I, I]
    lib.fa_fwd_host_workspace_bytes.restype = S
    lib.fa_fwd_host.argtypes = [P, P, P, P, P, P, S, I, I, I, I, I, F, P]
    lib.fa_fwd_host.restype = I
    lib.fa_fwd_host_gqa_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.fa_fwd_host_gqa_workspace_bytes.restype = S
    lib.fa_fwd_host_gqa.argtypes = [P, P, P, P, P, P, S, I, I, I, I, I, I, F, P]
    lib.fa_fwd_host_gqa.restype = I
    lib.fa_bwd_workspace_bytes.argtypes = [I, I, I, I]
    lib.fa_bwd_workspace_bytes.restype = S
    lib.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, S, I, I, I, I, I, F, P]
    lib.fa_bwd.restype = I
    lib.fa_bwd_gqa.argtypes = [P, P, P, P, P, P, P, P, P, P, S, I, I, I, I, I, I, F, P]
    lib.fa_bwd_gqa.restype = I
    lib.fa_decode_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.fa_decode_workspace_bytes.restype = S
    lib.fa_decode.argtypes = [P, P, P, P, P, P, S, I, I, I, I, I, F, P]
    lib.fa_decode.restype = I
    lib.fa_decode_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P]
    lib.fa_decode_noalloc.restype = I
    lib.fa_device_error.argtypes = [P]
    lib.fa_device_error.restype = I
    lib.fa_selftest_bounded_wait.argtypes = [I, P]
    lib.fa_selftest_bounded_wait.restype = I
    lib.fa_status_string.argtypes = [I]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_last_error_detail.argtypes = []
    lib.fa_last_error_detail.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = I
    lib.fa_last_device_status.argtypes = []
    lib.fa_last_device_status.restype = I
    return lib


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_qkv(q, k, v):
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, N, d]")
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    return tuple(int(x) for x in q.shape)


def fa_fwd(q, k, v, o=None, lse=None, causal: bool = False, scale: float | None = None,
           stream=None):
    """O = softmax(scale * q k^T [+causal]) v and LSE, on the current stream.

    q, k, v: contiguous CUDA bf16 [B, H, N, d].  o (bf16 [B,H,N,d]) and lse
    (fp32 [B,H,N]) are allocated when not given.  Returns (o, lse).
    """
    import torch
    B, H, N, d = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    rc = load_library().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, H, N, d, 1 if causal else 0,
                               float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return o, lse


def fa_fwd_gqa(q, k, v, o=None, lse=None, causal: bool = False, scale: float | None = None,
               stream=None):
    """Grouped-query attention: q [B, H, N, d]; k, v [B, H_kv, N, d] with
    H_kv dividing H.  Returns (o [B, H, N, d] bf16, lse [B, H, N] fp32)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda \
                or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 [B, H, N, d] tensor")
    B, H, N, d = (int(x) for x in q.shape)
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError(f"k/v shape {tuple(k.shape)} does not match q {tuple(q.shape)}")
    H_kv = int(k.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    rc = load_library().fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, H_kv, N, d, 1 if causal else 0,
                                   float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_gqa")
    return o, lse


def fa_fwd_host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa_fwd_host_workspace_bytes(B, H, N, d))


def fa_fwd_host(q_host, k_host, v_host, o_host, lse_host, workspace,
                causal: bool = False, scale: float | None = None, stream=None):
    """Host-buffer variant: H2D copies, the kernel and D2H copies, overlapped
    across chunks of heads on the library's own streams and ordered after the
    work already on ``stream``.  Tensors are CPU (ideally pinned);
    ``workspace`` is a CUDA uint8 tensor of at least
    fa_fwd_host_workspace_bytes bytes.  Asynchronous: synchronise the stream
    before reading o_host/lse_host."""
    B, H, N, d = (int(x) for x in q_host.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = load_library().fa_fwd_host(
        q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), o_host.data_ptr(),
        lse_host.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        B, H, N, d, 1 if causal else 0, float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_host")


def fa_fwd_host_gqa_workspace_bytes(B: int, H: int, H_kv: int, N: int, d: int) -> int:
    return int(load_library().fa_fwd_host_gqa_workspace_bytes(B, H, H_kv, N, d))


def fa_fwd_host_gqa(q_host, k_host, v_host, o_host, lse_host, workspace,
                    causal: bool = False, scale: float | None = None, stream=None):
    """fa_fwd_host for grouped-query attention: q_host, o_host [B, H, N, d];
    k_host, v_host [B, H_kv, N, d] with H_kv dividing H; lse_host [B, H, N].
    ``workspace``: CUDA uint8 tensor of at least
    fa_fwd_host_gqa_workspace_bytes bytes.  Asynchronous, as fa_fwd_host."""
    B, H, N, d = (int(x) for x in q_host.shape)
    H_kv = int(k_host.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = load_library().fa_fwd_host_gqa(
        q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), o_host.data_ptr(),
        lse_host.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        B, H, H_kv, N, d, 1 if causal else 0, float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_host_gqa")


def fa_bwd(q, k, v, o, lse, do, dq=None, dk=None, dv=None, workspace=None,
           causal: bool = False, scale: float | None = None, stream=None):
    """Gradients (dq, dk, dv) of fa_fwd for the output gradient ``do``.
    q, k, v, o, do: contiguous CUDA bf16 [B, H, N, d]; lse: fp32 [B, H, N]
    from the same forward call.  Outputs are allocated when not given."""
    import torch
    B, H, N, d = _check_qkv(q, k, v)
    for name, t in (("o", o), ("do", do)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8,
                                device=q.device)
    rc = load_library().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), B, H, N, d,
                               1 if causal else 0, float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


def fa_bwd_gqa(q, k, v, o, lse, do, dq=None, dk=None, dv=None, workspace=None,
               causal: bool = False, scale: float | None = None, stream=None):
    """Gradients of fa_fwd_gqa: q, o, do [B, H, N, d]; k, v [B, H_kv, N, d]
    with H_kv dividing H; lse [B, H, N].  Returns (dq [B, H, N, d],
    dk, dv [B, H_kv, N, d]), allocated when not given."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda \
                or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 [B, H, N, d] tensor")
    B, H, N, d = (int(x) for x in q.shape)
    if o.shape != q.shape or do.shape != q.shape:
        raise ValueError("o and do must be shaped like q")
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError(f"k/v shape {tuple(k.shape)} does not match q {tuple(q.shape)}")
    H_kv = int(k.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8,
                                device=q.device)
    rc = load_library().fa_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), B, H, H_kv, N,
                                   d, 1 if causal else 0, float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_gqa")
    return dq, dk, dv


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, N, d))


def fa_decode_workspace_bytes(B: int, H: int, H_kv: int, N: int, d: int) -> int:
    return int(load_library().fa_decode_workspace_bytes(B, H, H_kv, N, d))


def fa_decode(q, k, v, workspace=None, o=None, lse=None, scale: float | None = None,
              stream=None):
    """Decoding step: q [B, H, d] (newest token), k/v cache [B, H_kv, N, d].
    Returns (o [B, H, d] bf16, lse [B, H] fp32).  ``workspace``: CUDA uint8
    tensor of at least fa_decode_workspace_bytes(...) bytes (allocated when
    not given)."""
    import torch
    if q.dim() != 3 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B, H, d] and k, v [B, H_kv, N, d]")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    B, H, d = (int(x) for x in q.shape)
    H_kv, N = int(k.shape[1]), int(k.shape[2])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        need = fa_decode_workspace_bytes(B, H, H_kv, N, d)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    rc = load_library().fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), B, H, H_kv,
                                  N, d, float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_decode")
    return o, lse


def fa_device_error(stream=None) -> int:
    return int(load_library().fa_device_error(_stream_handle(stream)))


def fa_last_device_status() -> int:
    """(kernel << 8) | code behind this thread's last fa_device_error; 0 if clean."""
    return int(load_library().fa_last_device_status())


def fa_selftest_bounded_wait(limit_us: int, stream=None) -> int:
    return int(load_library().fa_selftest_bounded_wait(int(limit_us), _stream_handle(stream)))


def fa_version() -> int:
    return int(load_library().fa_version())
