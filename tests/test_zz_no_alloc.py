"""fa_decode_noalloc: decoding for callers that cannot allocate device memory.

The entry point keeps its split states in a library-owned area instead of a
caller workspace.  These tests call it through the C ABI and check its
output against the fp64 oracle and against fa_decode (the caller-workspace
entry point) within the tolerances the other tests use, on two calls in a
row with different inputs (so a second call cannot pass on what the first
one left behind).  The file
sorts last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_softmax_fa_gb300 import fa
    from online_softmax_fa_gb300.build import build_library
    build_library()
    lib = fa.load_library()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_decode_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P]
    lib.fa_decode_noalloc.restype = I
    return lib


def _inputs(seed, B, H, H_kv, N, d):
    from online_softmax_fa_gb300.inputs import make_decode
    dev = torch.device("cuda")
    return tuple(t.to(dev) for t in make_decode(B, H, H_kv, N, d, seed))


def _noalloc(lib, q, k, v, scale):
    B, H, d = q.shape
    H_kv, N = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.fa_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, H, H_kv, N, d, scale, stream)
    assert rc == 0, lib.fa_last_error_detail()
    return o, lse


@pytest.mark.parametrize("B,H,H_kv,N,d", [(4, 8, 2, 3000, 128), (2, 16, 16, 1000, 64)])
def test_noalloc_matches_oracle_and_workspace_decode_twice(lib, B, H, H_kv, N, d):
    import oracle
    from online_softmax_fa_gb300 import fa
    from online_softmax_fa_gb300.inputs import make_decode
    scale = float(np.float32(1 / np.sqrt(d)))
    for seed in (101, 202):  # two calls in a row, different inputs
        q_h, k_h, v_h = make_decode(B, H, H_kv, N, d, seed)
        q, k, v = _inputs(seed, B, H, H_kv, N, d)
        o_na, l_na = _noalloc(lib, q, k, v, scale)
        o_ws, l_ws = fa.fa_decode(q, k, v, scale=scale)
        torch.cuda.synchronize()
        assert fa.fa_device_error() == 0
        O_ref, L_ref = oracle.attention_decode(q_h.unsqueeze(2), k_h, v_h, scale=scale)
        eo = np.abs(o_na.float().cpu().numpy() - O_ref[:, :, 0])
        el = np.abs(l_na.cpu().numpy() - L_ref[:, :, 0])
        assert eo.max() <= O_MAX and eo.mean() <= O_MEAN and el.max() <= LSE_MAX
        assert (o_na.float() - o_ws.float()).abs().max().item() <= O_MAX
        assert (l_na - l_ws).abs().max().item() <= LSE_MAX
        assert torch.isfinite(l_na).all()


def test_noalloc_rejects_requests_beyond_its_area(lib):
    # 2048 sequences x 64 query heads of 128-wide states need more than the
    # 16 MiB area: rejected on the host before any buffer is touched
    from online_softmax_fa_gb300 import fa
    B, H, H_kv, N, d = 2048, 64, 8, 1024, 128
    need = fa.fa_decode_workspace_bytes(B, H, H_kv, N, d)
    assert need > (16 << 20)
    dummy = torch.empty(64, dtype=torch.bfloat16, device="cuda")  # never read
    lse = torch.empty(16, dtype=torch.float32, device="cuda")
    p = dummy.data_ptr()
    rc = lib.fa_decode_noalloc(p, p, p, p, lse.data_ptr(), B, H, H_kv, N, d, 0.088, None)
    assert rc == -11  # FA_ERR_WORKSPACE
    assert b"16 MiB" in lib.fa_last_error_detail()
