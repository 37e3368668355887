"""Seeded input generator: deterministic, right shapes, right structure."""
import numpy as np
import torch

from online_softmax_fa_gb300.inputs import (WORKLOADS, fixed_edge_rows, make_qkv,
                                            sample_rows)


def test_deterministic_and_shaped():
    a = make_qkv(2, 3, 17, 64, seed=7)
    b = make_qkv(2, 3, 17, 64, seed=7)
    c = make_qkv(2, 3, 17, 64, seed=8)
    for x, y, z in zip(a, b, c):
        assert x.shape == (2, 3, 17, 64) and x.dtype == torch.bfloat16
        assert x.is_contiguous()
        assert torch.equal(x, y)
        assert not torch.equal(x, z)


def test_draw_order_q_k_v():
    g = torch.Generator().manual_seed(5)
    q = torch.randn((1, 1, 9, 8), generator=g).to(torch.bfloat16)
    k = torch.randn((1, 1, 9, 8), generator=g).to(torch.bfloat16)
    v = torch.randn((1, 1, 9, 8), generator=g).to(torch.bfloat16)
    Q, K, V = make_qkv(1, 1, 9, 8, seed=5)
    assert torch.equal(Q, q) and torch.equal(K, k) and torch.equal(V, v)


def test_k_row_ramp():
    Q0, K0, V0 = make_qkv(1, 2, 64, 8, seed=3)
    Q1, K1, V1 = make_qkv(1, 2, 64, 8, seed=3, k_row_ramp=True)
    assert torch.equal(Q0, Q1) and torch.equal(V0, V1)
    g = torch.Generator().manual_seed(3)
    torch.randn((1, 2, 64, 8), generator=g)
    k = torch.randn((1, 2, 64, 8), generator=g)
    want = (k * (1 + 4 * torch.arange(64.0) / 64).view(1, 1, 64, 1)).to(torch.bfloat16)
    assert torch.equal(K1, want)


def test_workload_table():
    w = WORKLOADS["llama"]
    assert (w.B, w.H, w.N, w.d, w.causal) == (1, 32, 8192, 128, (True,))
    assert abs(w.flops(True) - 4 * 32 * 8192 ** 2 * 128 / 2) < 1
    assert WORKLOADS["long"].N == 256 * 128 + 3
    assert np.float32(WORKLOADS["batch"].scale) == np.float32(1 / np.sqrt(128))


def test_row_sampler():
    N = 32771
    t = sample_rows(N, 8, 512, seed=5)
    assert t.shape[0] == 8 and t.shape[1] >= 512
    for h in range(8):
        assert set(fixed_edge_rows(N)) <= set(t[h].tolist())
        assert t[h].min() >= 0 and t[h].max() < N
    assert {32768, 32769, 32770, 0, 127, 128}.issubset(fixed_edge_rows(N))
    assert np.array_equal(t, sample_rows(N, 8, 512, seed=5))
