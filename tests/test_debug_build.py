"""The debug build (include/fa_debug.h) on the GPU.

- Its device index checks (forward and backward kernels) pass on valid
  requests, and its outputs are bit-identical to the release build's.
- A failed check is recorded (FA_ERR_CHECK, with the check's number) and its
  store skipped.  The fault shrinks the extent that the checks use, so every
  skipped store lay inside the real buffer.
- A lost barrier arrival ends the launch with FA_ERR_TIMEOUT, not a hang,
  and the context stays usable afterwards.
"""
import time

import pytest
import torch

from online_softmax_fa_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

SENT_O, SENT_L = 1000.0, -1000.0  # outside any O or LSE these inputs can give
CHK_STORE_O = 6


def kernel_of(d):
    """The forward kernel's number in fa_last_device_status."""
    return 2 if d == 256 else 1


# each kernel's bounded-wait sites (the numbers it records on a timeout)
WAIT_SITES = {1: range(1, 14), 2: range(0x41, 0x4F)}


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_softmax_fa_gb300 import fa
    from online_softmax_fa_gb300.build import build_library
    build_library()
    return fa, fa.load_library(), fa.load_debug_library()


def _inputs(B, H, Hkv, N, d, seed):
    q, k, v = make_qkv(B, H, N, d, seed=seed, H_kv=Hkv)
    dev = torch.device("cuda")
    return q.to(dev), k.to(dev), v.to(dev)


def _outputs(q, o_offset=0):
    """O (bf16, optionally starting o_offset elements into a larger buffer)
    and LSE, filled with sentinels."""
    B, H, N, d = q.shape
    buf = torch.full((B * H * N * d + o_offset,), SENT_O, dtype=torch.bfloat16, device=q.device)
    o = buf[o_offset:].view(B, H, N, d)
    lse = torch.full((B, H, N), SENT_L, dtype=torch.float32, device=q.device)
    return o, lse


def _launch(lib, q, k, v, o, lse, causal):
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    scale = float(d) ** -0.5
    rc = lib.fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, H, Hkv, N, d, int(causal), scale, stream)
    assert rc == 0
    return lib.fa_device_error(stream)


CLEAN_CASES = [
    # B, H, H_kv, N, d, causal, O offset (8 elements: 16- but not 32-byte aligned)
    (1, 2, 2, 300, 64, False, 0),
    (1, 2, 2, 300, 64, True, 0),
    (2, 3, 3, 1000, 128, True, 0),
    (1, 4, 1, 777, 128, False, 0),
    (1, 8, 2, 2048, 128, True, 0),
    (1, 1, 1, 1, 128, True, 0),
    (1, 2, 2, 129, 64, True, 8),
    (2, 2, 2, 640, 128, False, 8),
    (1, 2, 2, 700, 256, True, 0),
    (2, 4, 2, 333, 256, False, 8),
    (1, 1, 1, 1, 256, True, 0),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,off", CLEAN_CASES)
def test_checks_pass_and_match_release(libs, B, H, Hkv, N, d, causal, off):
    fa, rel, dbg = libs
    q, k, v = _inputs(B, H, Hkv, N, d, seed=40 + N)
    o_r, l_r = _outputs(q, off)
    o_d, l_d = _outputs(q, off)
    assert _launch(rel, q, k, v, o_r, l_r, causal) == 0
    assert _launch(dbg, q, k, v, o_d, l_d, causal) == 0
    assert dbg.fa_last_device_status() == 0
    assert torch.equal(o_r, o_d) and torch.equal(l_r, l_d)
    assert not (o_d == SENT_O).any()  # every row was written


@pytest.mark.parametrize("d", [64, 256])
def test_failed_store_check_is_recorded_and_skipped(libs, d):
    fa, rel, dbg = libs
    B, H, N = 1, 2, 300
    q, k, v = _inputs(B, H, H, N, d, seed=7)
    o_r, l_r = _outputs(q)
    assert _launch(rel, q, k, v, o_r, l_r, False) == 0
    rows = B * H * N
    # the checks take the output to end one row early: the last row's stores
    # fail their check and are skipped
    assert dbg.fa_debug_arm(fa.FA_DEBUG_SHRINK_OUTPUT, rows - 1, 0, 20000) == 0
    o, lse = _outputs(q)
    assert _launch(dbg, q, k, v, o, lse, False) == fa.FA_ERR_CHECK
    assert dbg.fa_last_device_status() == (kernel_of(d) << 8) | 0x80 | CHK_STORE_O
    assert (o[0, 1, N - 1] == SENT_O).all() and lse[0, 1, N - 1] == SENT_L
    # every other row holds the release result, or the sentinel where the
    # aborted CTA stopped early
    o_rows, r_rows = o.reshape(rows, d)[:-1], o_r.reshape(rows, d)[:-1]
    written = ~(o_rows == SENT_O).all(dim=1)
    assert torch.equal(o_rows[written], r_rows[written])
    # an extent of zero rows: no store at all
    assert dbg.fa_debug_arm(fa.FA_DEBUG_SHRINK_OUTPUT, 0, 0, 20000) == 0
    o, lse = _outputs(q)
    assert _launch(dbg, q, k, v, o, lse, False) == fa.FA_ERR_CHECK
    assert (o == SENT_O).all() and (lse == SENT_L).all()
    # the fault was one-shot: the next launch is clean again
    o, lse = _outputs(q)
    assert _launch(dbg, q, k, v, o, lse, False) == 0
    assert torch.equal(o, o_r) and torch.equal(lse, l_r)


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_lost_arrival_times_out_and_context_survives(libs, causal, d):
    fa, rel, dbg = libs
    B, H, N = 1, 2, 1024
    q, k, v = _inputs(B, H, H, N, d, seed=9)
    o_r, l_r = _outputs(q)
    assert _launch(rel, q, k, v, o_r, l_r, causal) == 0
    # work item 0 (the first CTA's own, 8 key tiles long in both orders and
    # at both head dimensions) loses the arrival of its key tile 1; every
    # wait is limited to 20 ms
    assert dbg.fa_debug_arm(fa.FA_DEBUG_LOSE_K_ARRIVAL, 0, 1, 20000) == 0
    o, lse = _outputs(q)
    t0 = time.monotonic()
    assert _launch(dbg, q, k, v, o, lse, causal) == fa.FA_ERR_TIMEOUT
    assert time.monotonic() - t0 < 10.0
    st = dbg.fa_last_device_status()
    assert st >> 8 == kernel_of(d) and (st & 0xFF) in WAIT_SITES[st >> 8], hex(st)
    assert dbg.fa_device_error(None) == 0  # cleared
    # the context is usable: a clean launch of both builds matches
    o, lse = _outputs(q)
    assert _launch(dbg, q, k, v, o, lse, causal) == 0
    assert torch.equal(o, o_r) and torch.equal(lse, l_r)
    o2, l2 = _outputs(q)
    assert _launch(rel, q, k, v, o2, l2, causal) == 0
    assert torch.equal(o2, o_r)


BWD_CASES = [
    # B, H, H_kv, N, d, causal
    (1, 2, 2, 300, 64, True),
    (1, 4, 2, 640, 128, False),
    (2, 2, 2, 129, 128, True),
    (1, 1, 1, 1, 128, True),
    (1, 2, 1, 333, 256, True),
    (1, 2, 2, 256, 256, False),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", BWD_CASES)
def test_backward_checks_pass_and_match_release(libs, B, H, Hkv, N, d, causal):
    """The backward kernels' checks (debug build) pass, and the gradients are
    bit-identical to the release build's."""
    fa, rel, dbg = libs
    q, k, v = _inputs(B, H, Hkv, N, d, seed=80 + N)
    o, lse = _outputs(q)
    assert _launch(rel, q, k, v, o, lse, causal) == 0
    g = torch.Generator(device="cpu").manual_seed(81 + N)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16).to(q.device)
    stream = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=q.device)
    got = []
    for lib in (rel, dbg):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rc = lib.fa_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                            dv.data_ptr(), ws.data_ptr(), ws.numel(), B, H, Hkv, N, d,
                            int(causal), float(d) ** -0.5, stream)
        assert rc == 0
        assert lib.fa_device_error(stream) == 0
        got.append((dq, dk, dv))
    assert dbg.fa_last_device_status() == 0
    for a, b in zip(*got):
        assert torch.equal(a, b)


DEC_CASES = [
    # B, H, H_kv, N, d
    (2, 8, 2, 1000, 128),
    (1, 4, 4, 100, 64),
    (2, 8, 1, 4097, 256),
    (3, 16, 2, 1, 128),
]


@pytest.mark.parametrize("B,H,Hkv,N,d", DEC_CASES)
def test_decode_checks_pass_and_match_release(libs, B, H, Hkv, N, d):
    """The decoding kernels' checks (debug build) pass, and the output is
    bit-identical to the release build's."""
    fa, rel, dbg = libs
    dev = torch.device("cuda")
    g = torch.Generator(device="cpu").manual_seed(90 + N)
    q = torch.randn(B, H, d, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(B, Hkv, N, d, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(B, Hkv, N, d, generator=g).to(torch.bfloat16).to(dev)
    need = fa.fa_decode_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    got = []
    for lib in (rel, dbg):
        o = torch.empty_like(q)
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
        rc = lib.fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), ws.data_ptr(), need, B, H, Hkv, N, d,
                           float(d) ** -0.5, stream)
        assert rc == 0
        assert lib.fa_device_error(stream) == 0
        got.append((o, lse))
    assert dbg.fa_last_device_status() == 0
    assert torch.equal(got[0][0], got[1][0]) and torch.equal(got[0][1], got[1][1])
