"""fp64 CPU oracle for the exact attention forward pass -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares nothing with it (no code, header, helper or table).

The arithmetic lives in ``fa_oracle.c`` (plain C, fp64, POSIX threads); this
module only compiles it with gcc and marshals numpy arrays through ctypes.

Every function is pinned by ``tests/test_oracle_pins.py`` against values the
pages print, closed forms, invariants and a high-precision brute force; none
is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfa_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``fa_oracle.c`` into ``_build/libfa_oracle.so`` (gcc, -O2).

    ``-ffp-contract=off`` keeps a*b+c unfused so x86 and Arm round alike.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.fa_oracle_bf16_to_f64.argtypes = [p, p, i64]
        lib.fa_oracle_bf16_to_f64.restype = ctypes.c_int
        lib.fa_oracle_fwd.argtypes = [p, p, p, p, p, i64, i64, i64, i64,
                                      ctypes.c_int, ctypes.c_double, p, i64,
                                      ctypes.c_int]
        lib.fa_oracle_fwd.restype = ctypes.c_int
        lib.fa_oracle_fwd_q.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64,
                                        ctypes.c_int, ctypes.c_double, p, i64,
                                        ctypes.c_int]
        lib.fa_oracle_fwd_q.restype = ctypes.c_int
        lib.fa_oracle_bwd.argtypes = [p, p, p, p, p, p, p, p, p, i64, i64, i64, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_int]
        lib.fa_oracle_bwd.restype = ctypes.c_int
        lib.fa_oracle_fwd_blockwise.argtypes = [
            p, p, p, p, p, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double,
            p, i64, p, i64, ctypes.c_int, p, p, p, ctypes.c_int]
        lib.fa_oracle_fwd_blockwise.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16 array, or a torch bfloat16 tensor) -> fp64."""
    if not isinstance(bits, np.ndarray):  # torch tensor
        import torch
        bits = bits.detach().cpu().contiguous().view(torch.int16).numpy()
    bits = np.ascontiguousarray(bits).view(np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    rc = _load().fa_oracle_bf16_to_f64(_ptr(bits), _ptr(out), bits.size)
    if rc != 0:
        raise ValueError(f"fa_oracle_bf16_to_f64 failed ({rc})")
    return out


def _as_f64(x, name: str) -> np.ndarray:
    if isinstance(x, np.ndarray):
        if x.dtype == np.uint16:
            return bf16_bits_to_f64(x)
        return np.ascontiguousarray(x, dtype=np.float64)
    import torch
    if isinstance(x, torch.Tensor):
        if x.dtype == torch.bfloat16:
            return bf16_bits_to_f64(x)
        return np.ascontiguousarray(x.detach().cpu().double().numpy())
    raise TypeError(f"{name}: unsupported type {type(x)}")


def _shapes(q, k, v):
    if q.ndim < 2 or q.shape != k.shape or q.shape[:-1] != v.shape[:-1]:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    lead = q.shape[:-2]
    N, d = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    return lead, BH, N, d, dv


def attention_fwd(q, k, v, causal: bool = False, scale: float | None = None,
                  rows=None, nthreads: int | None = None):
    """Dense materialised attention in fp64.

    q, k: [..., N, d]; v: [..., N, dv] (numpy fp64 / uint16 bf16 bits, or
    torch tensors).  ``rows``: optional [..., R] int64 query indices per head.
    Returns (O [..., R or N, dv], LSE [..., R or N]) as fp64 numpy arrays.
    """
    q, k, v = _as_f64(q, "q"), _as_f64(k, "k"), _as_f64(v, "v")
    lead, BH, N, d, dv = _shapes(q, k, v)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows_arr = None
    R = N
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        if rows_arr.ndim == 1:
            rows_arr = np.ascontiguousarray(np.broadcast_to(rows_arr, (BH, rows_arr.size)))
        rows_arr = rows_arr.reshape(BH, -1)
        R = rows_arr.shape[1]
    O = np.empty((BH, R, dv), dtype=np.float64)
    LSE = np.empty((BH, R), dtype=np.float64)
    rc = _load().fa_oracle_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(O), _ptr(LSE), BH, N, d, dv,
        1 if causal else 0, float(scale),
        _ptr(rows_arr) if rows_arr is not None else None, R,
        nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"fa_oracle_fwd failed ({rc})")
    return O.reshape(*lead, R, dv), LSE.reshape(*lead, R)


def attention_fwd_gqa(q, k, v, causal: bool = False, scale: float | None = None,
                      rows=None, nthreads: int | None = None):
    """Grouped-query attention by its definition ("Understanding
    FlashAttention Pt 1", section 4.1): q [B, H, N, d], k/v [B, H_kv, N, d]
    with H_kv dividing H; query head h uses K/V head h // (H / H_kv).  Each
    K/V head is repeated for its group and the dense oracle runs on the
    result.  Returns (O [B, H, R, dv], LSE [B, H, R])."""
    q, k, v = _as_f64(q, "q"), _as_f64(k, "k"), _as_f64(v, "v")
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape[:3] + (k.shape[3],):
        raise ValueError("expected q [B,H,N,d] and k, v [B,H_kv,N,*]")
    H, H_kv = q.shape[1], k.shape[1]
    if H_kv < 1 or H % H_kv:
        raise ValueError(f"H_kv={H_kv} does not divide H={H}")
    group = H // H_kv
    k_full = np.repeat(k, group, axis=1)  # head h -> K/V head h // group
    v_full = np.repeat(v, group, axis=1)
    return attention_fwd(q, k_full, v_full, causal=causal, scale=scale, rows=rows,
                         nthreads=nthreads)


def attention_decode(q, k, v, causal: bool = True, scale: float | None = None,
                     nthreads: int | None = None):
    """Attention of the newest query rows against a key/value cache, by the
    definition: q [B, H, Nq, d] are the last Nq positions of a sequence whose
    keys and values are k, v [B, H_kv, N, d] (H_kv divides H; query head h
    uses K/V head h // (H / H_kv)).  Causal keeps key j for query row i iff
    j <= i + (N - Nq); with Nq = 1 every key is kept.
    Returns (O [B, H, Nq, dv], LSE [B, H, Nq])."""
    q, k, v = _as_f64(q, "q"), _as_f64(k, "k"), _as_f64(v, "v")
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4 or k.shape[:3] != v.shape[:3]:
        raise ValueError("expected q [B,H,Nq,d] and k, v [B,H_kv,N,*]")
    B, H, Nq, d = q.shape
    H_kv, N = k.shape[1], k.shape[2]
    if k.shape[0] != B or k.shape[3] != d or H_kv < 1 or H % H_kv:
        raise ValueError("shape mismatch")
    group = H // H_kv
    k_full = np.ascontiguousarray(np.repeat(k, group, axis=1))
    v_full = np.ascontiguousarray(np.repeat(v, group, axis=1))
    dv = v.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q = np.ascontiguousarray(q)
    O = np.empty((B * H, Nq, dv), dtype=np.float64)
    LSE = np.empty((B * H, Nq), dtype=np.float64)
    rc = _load().fa_oracle_fwd_q(_ptr(q), _ptr(k_full), _ptr(v_full), _ptr(O), _ptr(LSE),
                                 B * H, Nq, N, d, dv, 1 if causal else 0, float(scale),
                                 None, Nq, nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"fa_oracle_fwd_q failed ({rc})")
    return O.reshape(B, H, Nq, dv), LSE.reshape(B, H, Nq)


def attention_bwd(q, k, v, do, causal: bool = False, scale: float | None = None,
                  nthreads: int | None = None, return_D: bool = False, D=None):
    """Gradients (dQ, dK, dV) of the forward pass for the output gradient
    dO, by the definition (fp64, S, P, dP, dS materialised per head).
    q, k, v, do: [..., N, d].  With ``return_D`` also D_i = sum_r dO_ir O_ir.
    ``D`` ([..., N], optional) replaces the D_i of the exact O: the same
    gradients with D taken from another O (e.g. the forward's bf16 output)."""
    q, k, v, do = (_as_f64(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (do, "do")))
    if not (q.shape == k.shape == v.shape == do.shape) or q.ndim < 2:
        raise ValueError("q, k, v, do must share one shape [..., N, d]")
    lead = q.shape[:-2]
    N, d = q.shape[-2], q.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq, dk, dv = (np.empty((BH, N, d)) for _ in range(3))
    D_in = None
    if D is not None:
        D_in = np.ascontiguousarray(np.asarray(D, dtype=np.float64).reshape(BH, N))
    D = np.empty((BH, N))
    q, k, v, do = (np.ascontiguousarray(x) for x in (q, k, v, do))
    rc = _load().fa_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(D), _ptr(D_in) if D_in is not None else None,
                               BH, N, d, 1 if causal else 0, float(scale),
                               nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"fa_oracle_bwd failed ({rc})")
    out = (dq.reshape(q.shape), dk.reshape(q.shape), dv.reshape(q.shape))
    if return_D:
        out = out + (D.reshape(*lead, N),)
    return out


def attention_bwd_gqa(q, k, v, do, causal: bool = False, scale: float | None = None,
                      nthreads: int | None = None, D=None):
    """Gradients (dQ, dK, dV) of grouped-query attention ("Understanding
    FlashAttention Pt 1", section 4.1: query head h uses K/V head
    h // (H / H_kv)) for the output gradient dO.  q, do [B, H, N, d]; k, v
    [B, H_kv, N, d].  Grouped-query attention is the dense forward pass on
    K/V heads repeated for their group, so by the chain rule a K/V head's
    gradient is the sum of the dense gradients of its repeats; dQ is the
    dense one.  Returns dQ [B, H, N, d], dK and dV [B, H_kv, N, d]."""
    q, k, v, do = (_as_f64(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (do, "do")))
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape or do.shape != q.shape:
        raise ValueError("expected q, do [B,H,N,d] and k, v [B,H_kv,N,d]")
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if k.shape[0] != B or k.shape[2:] != (N, d) or H_kv < 1 or H % H_kv:
        raise ValueError("shape mismatch")
    group = H // H_kv
    k_full = np.repeat(k, group, axis=1)
    v_full = np.repeat(v, group, axis=1)
    dq, dk_full, dv_full = attention_bwd(q, k_full, v_full, do, causal=causal, scale=scale,
                                         nthreads=nthreads, D=D)
    dk = dk_full.reshape(B, H_kv, group, N, d).sum(axis=2)
    dv = dv_full.reshape(B, H_kv, group, N, d).sum(axis=2)
    return dq, dk, dv


def attention_fwd_blockwise(q, k, v, bounds, causal: bool = False,
                            scale: float | None = None, reverse: bool = False,
                            rows=None, nthreads: int | None = None,
                            return_state: bool = False):
    """Online-softmax blockwise recurrence in fp64 (oracle self-tests only).

    ``bounds``: ascending key-block boundaries, first 0, last N.  ``reverse``
    visits the blocks last-to-first.  With ``return_state`` also returns the
    final running state (m, l, a) before the division.
    """
    q, k, v = _as_f64(q, "q"), _as_f64(k, "k"), _as_f64(v, "v")
    lead, BH, N, d, dv = _shapes(q, k, v)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    b = np.ascontiguousarray(np.asarray(bounds, dtype=np.int64))
    rows_arr = None
    R = N
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        if rows_arr.ndim == 1:
            rows_arr = np.ascontiguousarray(np.broadcast_to(rows_arr, (BH, rows_arr.size)))
        rows_arr = rows_arr.reshape(BH, -1)
        R = rows_arr.shape[1]
    O = np.empty((BH, R, dv), dtype=np.float64)
    LSE = np.empty((BH, R), dtype=np.float64)
    M = np.empty((BH, R), dtype=np.float64)
    L = np.empty((BH, R), dtype=np.float64)
    A = np.empty((BH, R, dv), dtype=np.float64)
    rc = _load().fa_oracle_fwd_blockwise(
        _ptr(q), _ptr(k), _ptr(v), _ptr(O), _ptr(LSE), BH, N, d, dv,
        1 if causal else 0, float(scale),
        _ptr(rows_arr) if rows_arr is not None else None, R,
        _ptr(b), b.size - 1, 1 if reverse else 0, _ptr(M), _ptr(L), _ptr(A),
        nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"fa_oracle_fwd_blockwise failed ({rc})")
    out = (O.reshape(*lead, R, dv), LSE.reshape(*lead, R))
    if return_state:
        out = out + (M.reshape(*lead, R), L.reshape(*lead, R), A.reshape(*lead, R, dv))
    return out
