"""Concurrent calls from several host threads, each on its own CUDA stream.

The C ABI promises that calls on different streams are independent: the
library's host state (per-device caches, the host-buffer pipeline, error
details) is safe to use from several threads at once.  Each thread repeats
its call a few times while the others run theirs.  Every result must be
bit-identical to the same call made alone, since all kernels are
deterministic.
"""
import threading

import pytest
import torch

from online_softmax_fa_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_softmax_fa_gb300 import fa as fa_mod
    from online_softmax_fa_gb300.build import build_library
    build_library()
    fa_mod.load_library()
    return fa_mod


def _cases(fa):
    """(name, call(stream) -> tuple of output tensors) with inputs resident."""
    dev = torch.device("cuda")
    cases = []

    def fwd_case(B, H, Hkv, N, d, causal, seed):
        q, k, v = (t.to(dev) for t in make_qkv(B, H, N, d, seed=seed, H_kv=Hkv))
        if Hkv == H:
            return lambda s: fa.fa_fwd(q, k, v, causal=causal, stream=s)
        return lambda s: fa.fa_fwd_gqa(q, k, v, causal=causal, stream=s)

    cases.append(("fwd d128 causal", fwd_case(1, 4, 4, 1000, 128, True, 61)))
    cases.append(("fwd d64", fwd_case(2, 2, 2, 300, 64, False, 62)))
    cases.append(("fwd d256 causal", fwd_case(1, 2, 2, 700, 256, True, 63)))
    cases.append(("fwd gqa", fwd_case(1, 8, 2, 640, 128, True, 64)))

    q, k, v = (t.to(dev) for t in make_qkv(1, 2, 500, 128, seed=65))
    o, lse = fa.fa_fwd(q, k, v, causal=True)
    do = torch.randn_like(q.float()).to(torch.bfloat16)
    cases.append(("bwd d128 causal",
                  lambda s: fa.fa_bwd(q, k, v, o, lse, do, causal=True, stream=s)))

    qd = torch.randn(2, 8, 128, device=dev).to(torch.bfloat16)
    _, kd, vd = (t.to(dev) for t in make_qkv(2, 2, 1000, 128, seed=66))
    cases.append(("decode", lambda s: fa.fa_decode(qd, kd, vd, stream=s)))

    qh, kh, vh = (t.pin_memory() for t in make_qkv(1, 3, 600, 128, seed=67))
    ws_bytes = fa.fa_fwd_host_workspace_bytes(1, 3, 600, 128)

    def host_call(s):
        # a workspace of its own: calls in flight at the same time may not
        # share one
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        oh = torch.empty_like(qh).pin_memory()
        lh = torch.empty((1, 3, 600), dtype=torch.float32).pin_memory()
        fa.fa_fwd_host(qh, kh, vh, oh, lh, ws, causal=True, stream=s)
        return oh, lh
    cases.append(("fwd host buffers", host_call))
    torch.cuda.synchronize()
    return cases


def _run(call, stream):
    with torch.cuda.stream(stream):
        out = call(stream)
    stream.synchronize()
    return tuple(t.detach().cpu().clone() for t in out)


def test_concurrent_calls_match_serial(fa):
    cases = _cases(fa)
    serial = {name: _run(call, torch.cuda.Stream()) for name, call in cases}
    assert fa.fa_device_error() == 0
    # host-buffer calls share one pipeline per device, so two workers use it
    work = cases + [cases[-1]]
    got, errors = {}, []

    def worker(i, name, call):
        try:
            stream = torch.cuda.Stream()
            for _ in range(4):
                out = _run(call, stream)
                got.setdefault(i, []).append(out)
        except Exception as e:  # reported on the main thread
            errors.append(f"{name}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i, name, call))
               for i, (name, call) in enumerate(work)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a worker did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    for i, (name, _) in enumerate(work):
        assert len(got[i]) == 4, name
        for out in got[i]:
            for a, b in zip(out, serial[name]):
                assert torch.equal(a, b), name
