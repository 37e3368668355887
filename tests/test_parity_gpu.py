"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerance (bf16 output, fp32 accumulation): O max-abs <= 2e-2 and mean-abs
<= 2e-3, LSE abs <= 1e-3, compared element by element on the same seeded
inputs.  Small shapes and the llama (B1 H32 N8192 d128 causal) and batch (B16 H16
N2048 d128) workloads are compared in full; the long ragged workload and
the wider-path workloads on sampled query rows (the oracle computes them
one by one) plus properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_fa_gb300.inputs import WORKLOADS, make_qkv, make_workload, sample_rows

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_softmax_fa_gb300 import fa as fa_mod
    from online_softmax_fa_gb300.build import build_library
    build_library()
    fa_mod.load_library()
    return fa_mod


def run(fa, q, k, v, causal, scale):
    dev = torch.device("cuda")
    o, lse = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(o, lse, O_ref, L_ref, what=""):
    eo = np.abs(o - O_ref)
    el = np.abs(lse - L_ref)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    assert eo.max() <= O_MAX, f"{what}: O max-abs {eo.max():.3e}"
    assert eo.mean() <= O_MEAN, f"{what}: O mean-abs {eo.mean():.3e}"
    assert el.max() <= LSE_MAX, f"{what}: LSE max-abs {el.max():.3e}"
    return eo.max(), eo.mean(), el.max()


def scale_of(d):
    return float(np.float32(1 / np.sqrt(d)))


# --------------------------------------------------------- small, in full
def test_tiny_workload(fa):
    w = WORKLOADS["tiny"]
    q, k, v = make_workload(w)
    o, lse = run(fa, q, k, v, False, w.scale)
    O_ref, L_ref = oracle.attention_fwd(q, k, v, causal=False, scale=w.scale)
    check(o, lse, O_ref, L_ref, "tiny")


@pytest.mark.parametrize("seed", [2, 12, 22, 32])
@pytest.mark.parametrize("causal", [False, True])
def test_late_max_workload(fa, causal, seed):
    """The late-maximum workload on its own seed (2) and three more: K row j
    grows by (1 + 4j/N), so rows are peaked and the running max moves late;
    rounding P to bf16 sets most of the O error here, so the margin to the
    bound is printed."""
    w = WORKLOADS["late"]
    q, k, v = make_qkv(w.B, w.H, w.N, w.d, seed, k_row_ramp=True)
    o, lse = run(fa, q, k, v, causal, w.scale)
    O_ref, L_ref = oracle.attention_fwd(q, k, v, causal=causal, scale=w.scale)
    mx, mean, lmx = check(o, lse, O_ref, L_ref, f"late causal={causal} seed={seed}")
    print(f"late causal={causal} seed={seed}: O max {mx:.4e} mean {mean:.4e} LSE max {lmx:.4e}")


EDGE_N = [1, 2, 63, 127, 128, 129, 255, 256, 257, 300, 383, 512, 640, 1000]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_sweep(fa, N, d, causal):
    """Single tile, tile edges, ragged tails, odd block counts."""
    q, k, v = make_qkv(1, 2, N, d, seed=1000 + N + d)
    o, lse = run(fa, q, k, v, causal, scale_of(d))
    O_ref, L_ref = oracle.attention_fwd(q, k, v, causal=causal, scale=scale_of(d))
    check(o, lse, O_ref, L_ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("scale", [0.02, 0.5, 1.0])
def test_scales_and_large_scores(fa, scale):
    """Scores up to ~|40|: the running max moves by large steps."""
    q, k, v = make_qkv(2, 3, 700, 64, seed=77)
    q = (q.float() * 2).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = run(fa, q, k, v, causal, scale)
        O_ref, L_ref = oracle.attention_fwd(q, k, v, causal=causal, scale=scale)
        check(o, lse, O_ref, L_ref, f"scale={scale} causal={causal}")


def test_batch_and_heads_layout(fa):
    """B > 1 and H > 1 with a ragged N: heads must not bleed into each other."""
    q, k, v = make_qkv(3, 5, 333, 128, seed=9)
    for causal in (False, True):
        o, lse = run(fa, q, k, v, causal, scale_of(128))
        O_ref, L_ref = oracle.attention_fwd(q, k, v, causal=causal, scale=scale_of(128))
        check(o, lse, O_ref, L_ref, f"layout causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_256_layout_and_late_max(fa, causal):
    """d = 256 (its own kernel): B, H > 1, ragged N, and keys whose scores
    grow along the row, so the reference max moves and O is rescaled."""
    q, k, v = make_qkv(2, 3, 777, 256, seed=31, k_row_ramp=True)
    o, lse = run(fa, q, k, v, causal, scale_of(256))
    O_ref, L_ref = oracle.attention_fwd(q, k, v, causal=causal, scale=scale_of(256))
    check(o, lse, O_ref, L_ref, f"d256 late causal={causal}")


@pytest.mark.parametrize("scale", [0.02, 0.3])
def test_head_dim_256_large_scores(fa, scale):
    q, k, v = make_qkv(1, 2, 640, 256, seed=33)
    q = (q.float() * 2).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = run(fa, q, k, v, causal, scale)
        O_ref, L_ref = oracle.attention_fwd(q, k, v, causal=causal, scale=scale)
        check(o, lse, O_ref, L_ref, f"d256 scale={scale} causal={causal}")


def test_head_dim_256_workload_sampled(fa):
    _sampled_check(fa, WORKLOADS["d256"], 24, True)


def test_head_dim_256_gqa(fa):
    q, k, v = make_qkv(2, 8, 600, 256, seed=35, H_kv=2)
    dev = torch.device("cuda")
    for causal in (False, True):
        o, lse = fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), causal=causal,
                               scale=scale_of(256))
        torch.cuda.synchronize()
        assert fa.fa_device_error() == 0
        O_ref, L_ref = oracle.attention_fwd_gqa(q, k, v, causal=causal, scale=scale_of(256))
        check(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref,
              f"d256 gqa causal={causal}")


# ----------------------------------------------- one dominant key per row
# Column positions that a 128-key tile (64 at d = 256 in decoding) treats
# differently: first and last key, the edges of 8-, 16- and 64-key groups,
# the last eight keys of a tile, and keys of later tiles.
SPIKE_COLS = [0, 5, 15, 16, 63, 64, 119, 120, 121, 127, 128, 250, 255, 383]


def _spike(q_rows, k, h_kv, col, scale, margin=150.0):
    """Make key ``col`` of K/V head ``h_kv`` score ``margin`` (natural-log
    units) for a query direction u = mean of ``q_rows``: k_col = alpha * u
    with alpha * scale * |u|^2 = margin.  Every other score stays O(1), so
    the running reference max must take this key, or exp of the gap
    overflows fp32."""
    u = q_rows.reshape(-1, q_rows.shape[-1]).mean(dim=0)
    alpha = margin / (scale * float(u @ u))
    k[:, h_kv, col] = alpha * u


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_dominant_key_anywhere_in_a_tile(fa, d, causal):
    H, N = len(SPIKE_COLS), 384
    q, k, v = make_qkv(1, H, N, d, seed=90 + d)
    g = torch.Generator(device="cpu")
    g.manual_seed(91 + d)
    u = torch.randn(H, d, generator=g, dtype=torch.float32)
    qf = u.view(1, H, 1, d) + 0.1 * q.float()  # every row of head h near u_h
    kf = k.float()
    scale = scale_of(d)
    for h, c in enumerate(SPIKE_COLS):
        _spike(qf[:, h], kf, h, c, scale)
    q, k = qf.to(torch.bfloat16), kf.to(torch.bfloat16)
    o, lse = run(fa, q, k, v, causal, scale)
    O_ref, L_ref = oracle.attention_fwd(q, k, v, causal=causal, scale=scale)
    # rows that see their head's dominant key return (nearly) its value row
    assert L_ref[0, 0, -1] > 100
    check(o, lse, O_ref, L_ref, f"dominant key d={d} causal={causal}")


# ------------------------------------------------------------ closed forms
def test_closed_forms(fa):
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(3)
    # identical keys -> mean of V, LSE = s + log N
    N, d = 520, 128
    q = torch.randn(1, 2, N, d, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 2, 1, d, generator=g).to(torch.bfloat16).expand(1, 2, N, d).contiguous()
    v = torch.randn(1, 2, N, d, generator=g).to(torch.bfloat16)
    o, lse = run(fa, q, k, v, False, 0.1)
    mean_v = v.double().mean(dim=2, keepdim=True).numpy()
    assert np.abs(o - mean_v).max() <= O_MAX
    s = 0.1 * np.einsum("bhnd,bhd->bhn", q.double().numpy(), k[:, :, 0].double().numpy())
    assert np.abs(lse - (s + np.log(N))).max() <= LSE_MAX
    # N = 1: O = V, LSE = scale q.k
    q1, k1, v1 = make_qkv(2, 3, 1, 64, seed=4)
    o, lse = run(fa, q1, k1, v1, True, 0.125)
    assert np.array_equal(o, v1.float().numpy())
    s = 0.125 * (q1.double() * k1.double()).sum(-1).numpy()
    assert np.abs(lse - s).max() <= LSE_MAX
    # causal row 0 returns V_0 exactly (one key, weight 1)
    q2, k2, v2 = make_qkv(1, 4, 700, 128, seed=5)
    o, _ = run(fa, q2, k2, v2, True, scale_of(128))
    assert np.array_equal(o[:, :, 0], v2[:, :, 0].float().numpy())


def test_determinism(fa):
    q, k, v = make_workload(WORKLOADS["late"])
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    for causal in (False, True):
        o1, l1 = fa.fa_fwd(q, k, v, causal=causal)
        o2, l2 = fa.fa_fwd(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


# --------------------------------------------------- full-size workloads
def _sampled_check(fa, w, rows_per_head, causal):
    q, k, v = make_workload(w)
    dev = torch.device("cuda")
    o_d, lse_d = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    BH = w.B * w.H
    # properties at full size: finite everywhere, LSE >= the row's own score
    assert torch.isfinite(lse_d).all()
    assert torch.isfinite(o_d.float()).all()
    rows = sample_rows(w.N, BH, rows_per_head, seed=w.seed)
    o = o_d.float().reshape(BH, w.N, w.d).cpu().numpy()
    lse = lse_d.reshape(BH, w.N).cpu().numpy()
    idx = np.arange(BH)[:, None]
    O_ref, L_ref = oracle.attention_fwd(q.reshape(BH, w.N, w.d), k.reshape(BH, w.N, w.d),
                                        v.reshape(BH, w.N, w.d), causal=causal,
                                        scale=w.scale, rows=rows)
    mx, mean, lmx = check(o[idx, rows], lse[idx, rows], O_ref, L_ref, w.name)
    print(f"{w.name} sampled ({rows.size} rows): O max {mx:.4e} mean {mean:.4e} "
          f"LSE max {lmx:.4e}")
    return mx, mean, lmx


def _full_check(fa, w, causal):
    """Every row of O and LSE against the oracle (the oracle takes about
    half a minute for these shapes on 16 host cores)."""
    q, k, v = make_workload(w)
    dev = torch.device("cuda")
    o_d, lse_d = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    o = o_d.float().cpu().numpy()
    lse = lse_d.cpu().numpy()
    del o_d, lse_d
    O_ref, L_ref = oracle.attention_fwd(q, k, v, causal=causal, scale=w.scale)
    mx, mean, lmx = check(o, lse, O_ref, L_ref, w.name)
    print(f"{w.name} full ({o.shape[0] * o.shape[1] * o.shape[2]} rows): O max {mx:.4e} "
          f"mean {mean:.4e} LSE max {lmx:.4e}")


def test_llama_workload_full(fa):
    _full_check(fa, WORKLOADS["llama"], True)


def test_batch_workload_full(fa):
    _full_check(fa, WORKLOADS["batch"], False)


def test_long_ragged_workload_sampled(fa):
    w = WORKLOADS["long"]
    _sampled_check(fa, w, w.sampled_rows, True)


# --------------------------------------------- host-buffer entry point
def test_host_buffer_variant_matches(fa):
    q, k, v = make_qkv(2, 3, 300, 128, seed=21)
    B, H, N, d = q.shape
    dev = torch.device("cuda")
    need = fa.fa_fwd_host_workspace_bytes(B, H, N, d)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty_like(q).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    for causal in (False, True):
        fa.fa_fwd_host(qh, kh, vh, oh, lh, ws, causal=causal)
        torch.cuda.synchronize()
        o_d, l_d = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(oh, o_d.cpu()) and torch.equal(lh, l_d.cpu())


# ------------------------------------------------------ failure detection
def test_bounded_wait_expires_with_status(fa):
    """A wait nothing signals ends with FA_ERR_TIMEOUT, not a hang, and the
    context stays usable afterwards."""
    assert fa.fa_selftest_bounded_wait(20000) == fa.FA_ERR_TIMEOUT
    assert fa.fa_last_device_status() == (1 << 8) | 0x7F  # forward word, the test's wait
    assert fa.fa_device_error() == 0  # the status word was cleared
    assert fa.fa_last_device_status() == 0
    q, k, v = make_qkv(1, 1, 256, 64, seed=1)
    o, lse = run(fa, q, k, v, False, 0.125)
    O_ref, L_ref = oracle.attention_fwd(q, k, v, scale=0.125)
    check(o, lse, O_ref, L_ref, "after selftest")


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 40, 2048, 64, True), (1, 100, 8192, 64, False),
                                         (1, 20, 4096, 256, True)])
def test_host_buffer_chunked_pipeline_is_bit_identical(fa, B, H, N, d, causal):
    """Shapes that the host path cuts into several (uneven) chunks of heads:
    the outputs must equal one fa_fwd call on device buffers, bit for bit."""
    q, k, v = make_qkv(B, H, N, d, seed=60 + H + d)
    dev = torch.device("cuda")
    o_ref, l_ref = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale_of(d))
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty(fa.fa_fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    fa.fa_fwd_host(qh, kh, vh, oh, lh, ws, causal=causal, scale=scale_of(d))
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    assert torch.equal(oh, o_ref.cpu()) and torch.equal(lh, l_ref.cpu())


@pytest.mark.parametrize("B,H,H_kv,N,d,causal", [(1, 32, 8, 2048, 128, True),
                                                 (2, 12, 3, 700, 64, False),
                                                 (1, 16, 1, 1000, 256, True)])
def test_host_buffer_gqa_is_bit_identical(fa, B, H, H_kv, N, d, causal):
    """Grouped-query heads through host buffers (chunks of whole K/V groups)
    equal one fa_fwd_gqa call on device buffers, bit for bit."""
    q, k, v = make_qkv(B, H, N, d, seed=65 + H + H_kv + d, H_kv=H_kv)
    dev = torch.device("cuda")
    o_ref, l_ref = fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), causal=causal,
                                 scale=scale_of(d))
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty(fa.fa_fwd_host_gqa_workspace_bytes(B, H, H_kv, N, d), dtype=torch.uint8,
                     device=dev)
    fa.fa_fwd_host_gqa(qh, kh, vh, oh, lh, ws, causal=causal, scale=scale_of(d))
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    assert torch.equal(oh, o_ref.cpu()) and torch.equal(lh, l_ref.cpu())


# ------------------------------------------------- grouped-query attention
@pytest.mark.parametrize("H,H_kv,N,d,causal", [
    (8, 2, 1000, 128, True), (8, 2, 1000, 128, False), (6, 1, 300, 64, True),
    (4, 4, 257, 64, False), (32, 8, 520, 128, True)])
def test_gqa_parity(fa, H, H_kv, N, d, causal):
    q, k, v = make_qkv(2, H, N, d, seed=40 + H + H_kv + N, H_kv=H_kv)
    dev = torch.device("cuda")
    o, lse = fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale_of(d))
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    O_ref, L_ref = oracle.attention_fwd_gqa(q, k, v, causal=causal, scale=scale_of(d))
    check(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref,
          f"gqa H={H} H_kv={H_kv} N={N} d={d} causal={causal}")


def test_gqa_with_equal_heads_is_fa_fwd(fa):
    q, k, v = make_qkv(1, 4, 700, 128, seed=50)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = fa.fa_fwd_gqa(q, k, v, causal=True)
    o2, l2 = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_llama_gqa_workload_sampled(fa):
    w = WORKLOADS["llama_gqa"]
    q, k, v = make_workload(w)
    dev = torch.device("cuda")
    o_d, lse_d = fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    assert torch.isfinite(lse_d).all() and torch.isfinite(o_d.float()).all()
    rows = sample_rows(w.N, w.H, 32, seed=w.seed)
    O_ref, L_ref = oracle.attention_fwd_gqa(q, k, v, causal=True, scale=w.scale,
                                            rows=rows)
    idx = np.arange(w.H)[:, None]
    o = o_d.float()[0].cpu().numpy()
    lse = lse_d[0].cpu().numpy()
    check(o[idx, rows][None], lse[idx, rows][None], O_ref, L_ref, "llama_gqa")


# ------------------------------------------------------------ decoding
from online_softmax_fa_gb300.inputs import DECODE_WORKLOADS, make_decode  # noqa: E402


def _decode_check(fa, q, k, v, scale, what):
    dev = torch.device("cuda")
    o, lse = fa.fa_decode(q.to(dev), k.to(dev), v.to(dev), scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    O_ref, L_ref = oracle.attention_decode(q.unsqueeze(2), k, v, scale=scale)
    return check(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref[:, :, 0], L_ref[:, :, 0],
                 what)


@pytest.mark.parametrize("N", [1, 7, 63, 64, 65, 1000, 4097])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("H,H_kv", [(8, 8), (8, 4), (8, 2), (8, 1)])
def test_decode_parity(fa, N, d, H, H_kv):
    q, k, v = make_decode(2, H, H_kv, N, d, seed=60 + N + H_kv)
    _decode_check(fa, q, k, v, scale_of(d), f"decode N={N} d={d} H={H} H_kv={H_kv}")


def test_decode_closed_form_identical_keys(fa):
    q, k, v = make_decode(1, 4, 2, 3000, 128, seed=70)
    k = k[:, :, :1].expand(-1, -1, 3000, -1).contiguous()
    dev = torch.device("cuda")
    o, lse = fa.fa_decode(q.to(dev), k.to(dev), v.to(dev), scale=0.1)
    torch.cuda.synchronize()
    mean_v = v.double().mean(dim=2).repeat_interleave(2, dim=1).numpy()
    assert np.abs(o.float().cpu().numpy() - mean_v).max() <= O_MAX


def test_decode_workload(fa):
    w = DECODE_WORKLOADS["decode"]
    q, k, v = make_decode(w.B, w.H, w.kv_heads, w.N, w.d, w.seed)
    _decode_check(fa, q, k, v, w.scale, "decode workload")


def test_decode_matches_forward_last_row(fa):
    """The newest row decoded against the cache equals the last row of the
    causal forward pass over the whole sequence."""
    q, k, v = make_qkv(1, 8, 777, 128, seed=71, H_kv=2)
    dev = torch.device("cuda")
    o_f, l_f = fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), causal=True)
    o_d, l_d = fa.fa_decode(q[:, :, -1].contiguous().to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    assert (o_f[:, :, -1].float() - o_d.float()).abs().max().item() <= 2 * O_MAX
    assert (l_f[:, :, -1] - l_d).abs().max().item() <= 2 * LSE_MAX


@pytest.mark.parametrize("d", [64, 128, 256])
def test_decode_dominant_key_anywhere_in_a_tile(fa, d):
    cols = [0, 15, 16, 31, 32, 63, 64, 120, 127, 128, 1000, 4095, 4096]
    H = len(cols)
    q, k, v = make_decode(1, H, H, 4097, d, seed=92 + d)
    kf = k.float()
    scale = scale_of(d)
    for h, c in enumerate(cols):
        _spike(q[:, h].float(), kf, h, c, scale)
    _decode_check(fa, q, kf.to(torch.bfloat16), v, scale, f"decode dominant key d={d}")


# ------------------------------------------------------------ backward pass
from online_softmax_fa_gb300.inputs import make_grad  # noqa: E402

# Bounds for the bf16 gradients, relative to the size of each reference
# gradient (max |ref| for the max error, mean |ref| for the mean error):
# outputs are rounded to bf16 (<= 2^-9 relative each), P and dS are rounded
# to bf16 for the tensor cores (<= 2^-9 per term), and dQ, dK are sums of dS
# terms that cancel (each row of dS sums to zero), which amplifies those
# roundings relative to the result (measured up to ~7e-3 mean at N = 2).
# Gradients below G_FLOOR in size (N = 1 gives exact zeros) use the floor.
# Each bound also takes the effect of forming D from the bf16 O, measured
# with the oracle (_bwd_refs).
G_MAX_REL, G_MEAN_REL, G_FLOOR = 2e-2, 1e-2, 1e-3


@pytest.mark.parametrize("d", [64, 128])
def test_output_only_16_byte_aligned(fa, d):
    """O 16-byte but not 32-byte aligned (the API's minimum): the epilogue
    takes its 16-byte stores and writes the same bits as with an aligned O."""
    q, k, v = make_qkv(1, 3, 300, d, seed=90 + d)
    dev = torch.device("cuda")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o_ref, l_ref = fa.fa_fwd(qd, kd, vd, causal=True)
    flat = torch.empty(o_ref.numel() + 8, dtype=torch.bfloat16, device=dev)
    o_off = flat[8:].view(o_ref.shape)  # 16 bytes past a 256-byte aligned base
    assert o_off.data_ptr() % 32 == 16
    o2, l2 = fa.fa_fwd(qd, kd, vd, o=o_off, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    assert torch.equal(o2, o_ref) and torch.equal(l2, l_ref)


def _bwd_run(fa, q, k, v, do, causal, scale):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fa_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    return tuple(t.float().cpu().numpy() for t in (dq, dk, dv))


def _bwd_refs(q, k, v, do, causal, scale, gqa=False):
    """The oracle's gradients, and the same gradients with D_i = sum_r dO_ir
    O_ir formed from the oracle's own O rounded to bf16.  The kernels form D
    from the bf16 O the forward returned (section 3.6 gives D in that form);
    the difference between the two references is the part of the error that
    rounding alone adds (it does not cancel in dQ = scale dS K, where the
    reference itself can be a small difference of terms), and the bound
    includes it."""
    fwd = oracle.attention_fwd_gqa if gqa else oracle.attention_fwd
    bwd = oracle.attention_bwd_gqa if gqa else oracle.attention_bwd
    ref = bwd(q, k, v, do, causal=causal, scale=scale)
    O, _ = fwd(q, k, v, causal=causal, scale=scale)
    O_b = torch.from_numpy(O).to(torch.bfloat16).double().numpy()
    D_b = (oracle.bf16_bits_to_f64(do) * O_b).sum(-1)
    ref_b = bwd(q, k, v, do, causal=causal, scale=scale, D=D_b)
    return ref, ref_b


def _grad_check(got, ref, what, ref_b=None):
    """max-abs <= G_MAX_REL * max|ref| and mean-abs <= G_MEAN_REL * mean|ref|
    per gradient (floor G_FLOOR), each plus the max / mean of |ref_b - ref|
    (the effect of D formed from the bf16 O, see _bwd_refs) when given."""
    errs = []
    for i, (name, g, r) in enumerate(zip(("dQ", "dK", "dV"), got, ref)):
        assert np.isfinite(g).all(), f"{what} {name} not finite"
        e = np.abs(g - r)
        scale_max = max(np.abs(r).max(), G_FLOOR)
        scale_mean = max(np.abs(r).mean(), G_FLOOR)
        x = np.abs(ref_b[i] - r) if ref_b is not None else np.zeros(1)
        errs.append((name, e.max() / scale_max, e.mean() / scale_mean))
        assert e.max() <= G_MAX_REL * scale_max + x.max(), \
            f"{what} {name}: max {e.max():.3e} ref {scale_max:.3e} D-rounding {x.max():.3e}"
        assert e.mean() <= G_MEAN_REL * scale_mean + x.mean(), \
            f"{what} {name}: mean {e.mean():.3e} ref {scale_mean:.3e} D-rounding {x.mean():.3e}"
    return errs


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 300, 640])
def test_backward_parity(fa, N, d, causal):
    q, k, v = make_qkv(1, 2, N, d, seed=500 + N + d)
    do = make_grad(1, 2, N, d, seed=500 + N + d)
    got = _bwd_run(fa, q, k, v, do, causal, scale_of(d))
    ref, ref_b = _bwd_refs(q, k, v, do, causal, scale_of(d))
    errs = _grad_check(got, ref, f"bwd N={N} d={d} causal={causal}", ref_b)
    print(f"bwd N={N} d={d} causal={causal}: " + ", ".join(
        f"{n} max {a:.2e} mean {b:.2e}" for n, a, b in errs))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_late_max_workload(fa, causal):
    w = WORKLOADS["late"]
    q, k, v = make_workload(w)
    do = make_grad(w.B, w.H, w.N, w.d, w.seed)
    got = _bwd_run(fa, q, k, v, do, causal, w.scale)
    ref, ref_b = _bwd_refs(q, k, v, do, causal, w.scale)
    errs = _grad_check(got, ref, f"bwd late causal={causal}", ref_b)
    print(f"bwd late causal={causal}: " + ", ".join(
        f"{n} max {a:.2e} mean {b:.2e}" for n, a, b in errs))


def _bwd_gqa_run(fa, q, k, v, do, causal, scale):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fa_fwd_gqa(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_bwd_gqa(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    return tuple(t.float().cpu().numpy() for t in (dq, dk, dv))


@pytest.mark.parametrize("B,H,H_kv,N,d,causal", [
    (1, 4, 2, 300, 64, True),
    (1, 4, 2, 300, 64, False),
    (2, 8, 1, 257, 128, True),   # multi-query, ragged last block
    (1, 8, 2, 640, 128, True),
    (1, 6, 3, 129, 128, False),
    (1, 16, 2, 384, 128, True),  # groups of 8
    (1, 4, 4, 200, 128, True),   # H_kv = H: the dense backward
    (1, 8, 2, 300, 256, True),   # head dimension 256
    (2, 4, 1, 200, 256, False),
])
def test_backward_gqa_parity(fa, B, H, H_kv, N, d, causal):
    seed = 700 + H * 10 + N
    q, k, v = make_qkv(B, H, N, d, seed=seed, H_kv=H_kv)
    do = make_grad(B, H, N, d, seed=seed)
    got = _bwd_gqa_run(fa, q, k, v, do, causal, scale_of(d))
    ref, ref_b = _bwd_refs(q, k, v, do, causal, scale_of(d), gqa=True)
    assert got[1].shape == (B, H_kv, N, d) and got[2].shape == (B, H_kv, N, d)
    errs = _grad_check(got, ref, f"bwd gqa B={B} H={H} H_kv={H_kv} N={N} d={d} causal={causal}",
                       ref_b)
    print(f"bwd gqa H={H} H_kv={H_kv} N={N} d={d} causal={causal}: " + ", ".join(
        f"{n} max {a:.2e} mean {b:.2e}" for n, a, b in errs))


@pytest.mark.parametrize("B,H,H_kv,N", [(1, 128, 128, 384), (2, 160, 80, 256)])
def test_backward_grouped_cost_order(fa, B, H, H_kv, N):
    """Enough heads that the causal CTA order of both backward kernels runs
    over several groups of heads, the last one smaller (on 152 SMs: groups
    of 114 heads at N = 384, of 152 at N = 256): every head's gradients
    still match the oracle."""
    d = 64
    seed = 900 + H + N
    q, k, v = make_qkv(B, H, N, d, seed=seed, H_kv=H_kv)
    do = make_grad(B, H, N, d, seed=seed)
    got = _bwd_gqa_run(fa, q, k, v, do, True, scale_of(d))
    ref, ref_b = _bwd_refs(q, k, v, do, True, scale_of(d), gqa=True)
    # per head, so that a head left out or written twice cannot hide in a mean
    for b in range(B):
        for hq in range(H):
            hk = hq * H_kv // H
            _grad_check((got[0][b, hq], got[1][b, hk], got[2][b, hk]),
                        (ref[0][b, hq], ref[1][b, hk], ref[2][b, hk]),
                        f"bwd grouped order B={B} H={H} H_kv={H_kv} N={N} head {b},{hq}",
                        (ref_b[0][b, hq], ref_b[1][b, hk], ref_b[2][b, hk]))


def test_backward_gqa_deterministic(fa):
    """The group sum of dK / dV runs in a fixed order: two calls agree bit
    for bit."""
    q, k, v = make_qkv(1, 8, 500, 128, seed=81, H_kv=2)
    do = make_grad(1, 8, 500, 128, seed=81)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fa_fwd_gqa(qd, kd, vd, causal=True)
    a = fa.fa_bwd_gqa(qd, kd, vd, o, lse, dod, causal=True)
    b = fa.fa_bwd_gqa(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_backward_head_dim_256_deterministic_and_late_max(fa):
    """d = 256 (its own kernels): bit-identical repeats, and keys whose
    scores grow along the row (peaked probabilities) against the oracle."""
    q, k, v = make_qkv(2, 3, 333, 256, seed=83, k_row_ramp=True)
    do = make_grad(2, 3, 333, 256, seed=83)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fa_fwd(qd, kd, vd, causal=True)
    a = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=True)
    b = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == 0
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    ref, ref_b = _bwd_refs(q, k, v, do, True, scale_of(256))
    _grad_check(tuple(t.float().cpu().numpy() for t in a), ref, "bwd d256 late", ref_b)


def test_backward_deterministic(fa):
    q, k, v = make_qkv(2, 3, 700, 128, seed=77)
    do = make_grad(2, 3, 700, 128, seed=77)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fa_fwd(qd, kd, vd, causal=True)
    a = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=True)
    b = fa.fa_bwd(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
