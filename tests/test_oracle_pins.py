"""Pins for the fp64 oracle, checked against what the pages and mathematics fix.

Nothing here compares the oracle with itself or retypes its formula: each
check is a value the pages print, a closed form, an invariant of the exact
function, or a separately written high-precision brute force (Python
``decimal`` at 40 digits, softmax taken without max subtraction).  A dropped
term, a wrong sign or index, a transposed operand or a wrong causal direction
in the oracle fails at least one of them.
"""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
from tests.conftest import read_golden


# ---------------------------------------------------------------- page values
def test_worked_example_dense_and_blockwise():
    """wpnews.pro "Understanding FlashAttention Pt 1", section 2.5."""
    g = read_golden("wpnews_s2_5_worked_example.txt")
    s = np.array(g["scores"])
    v = np.array(g["v"])
    tol = g["tol"][0]
    # d = 1, q = [1], k_j = [s_j], scale 1: the scaled score row is s itself.
    q = np.ones((1, 1, 1))[:, :, :].repeat(len(s), axis=1)  # every query row = [1]
    k = s.reshape(1, -1, 1)
    vv = v.reshape(1, len(s), 2)
    O, L = oracle.attention_fwd(q, k, vv, causal=False, scale=1.0, rows=[0])
    np.testing.assert_allclose(O[0, 0], g["o"], atol=tol, rtol=0)
    # LSE = m + log(l) with the printed m and l
    assert abs(L[0, 0] - (g["max"][0] + math.log(g["ell"][0]))) < tol

    split = int(g["block_split"][0])
    bounds = [0, split, len(s)]
    Ob, Lb, M, Lsum, A = oracle.attention_fwd_blockwise(
        q, k, vv, bounds, scale=1.0, rows=[0], return_state=True)
    np.testing.assert_allclose(Ob[0, 0], g["o"], atol=tol, rtol=0)
    assert abs(Lsum[0, 0] - g["ell"][0]) < tol
    assert M[0, 0] == g["max"][0]
    np.testing.assert_allclose(A[0, 0], g["a2"], atol=tol, rtol=0)

    # state after block 1 alone: m_1 = 2, l_1 = 1 + e^{-1}
    _, _, M1, L1, A1 = oracle.attention_fwd_blockwise(
        q[:, :split], k[:, :split], vv[:, :split], [0, split], scale=1.0,
        rows=[0], return_state=True)
    assert M1[0, 0] == g["block1_max"][0]
    assert abs(L1[0, 0] - g["block1_ell"][0]) < tol
    # alpha = e^{m_1 - m_2} takes block 1's state to block 2's reference
    alpha = math.exp(g["block2_alpha_exp"][0])
    assert abs(alpha * L1[0, 0] + 1 + math.exp(-1) - g["ell"][0]) < tol


def test_overflow_example_stays_finite():
    """wpnews.pro section 2.2: [1000, 999] must not overflow."""
    g = read_golden("wpnews_s2_2_overflow.txt")
    s = np.array(g["scores"])
    q = np.ones((1, 2, 1))
    k = s.reshape(1, 2, 1)
    v = np.eye(2).reshape(1, 2, 2)  # O row = the softmax weights
    O, L = oracle.attention_fwd(q, k, v, scale=1.0, rows=[0])
    assert np.all(np.isfinite(O)) and np.isfinite(L).all()
    w = np.array(g["weights_printed"])
    np.testing.assert_allclose(O[0, 0], w / w.sum(), atol=g["tol_printed"][0])
    # closed form: weights [1, e^-1]/(1+e^-1), LSE = 1000 + log(1 + e^-1)
    e = math.exp(-1)
    np.testing.assert_allclose(O[0, 0], [1 / (1 + e), e / (1 + e)], atol=1e-15)
    assert abs(L[0, 0] - (1000 + math.log1p(e))) < 1e-12
    Ob, Lb = oracle.attention_fwd_blockwise(q, k, v, [0, 1, 2], scale=1.0, rows=[0])
    np.testing.assert_allclose(Ob, O, atol=1e-15)
    assert abs(Lb[0, 0] - L[0, 0]) < 1e-12


# ---------------------------------------------------------------- brute force
def _brute(q, k, v, causal, scale):
    """Direct softmax in 40-digit decimals: p_ij = exp(s_ij) / sum exp(s_ik)."""
    getcontext().prec = 40
    N, d = q.shape
    dv = v.shape[1]
    O = np.zeros((N, dv))
    L = np.zeros(N)
    sc = Decimal(repr(float(scale)))
    for i in range(N):
        keys = [j for j in range(N) if (not causal or j <= i)]
        e = {}
        for j in keys:
            s = sum(Decimal(repr(float(q[i, c]))) * Decimal(repr(float(k[j, c])))
                    for c in range(d)) * sc
            e[j] = s.exp()
        z = sum(e.values())
        for c in range(dv):
            O[i, c] = float(sum(e[j] * Decimal(repr(float(v[j, c]))) for j in keys) / z)
        L[i] = float(z.ln())
    return O, L


@pytest.mark.parametrize("N,d,dv,causal,seed", [
    (1, 1, 1, False, 0), (2, 3, 2, True, 1), (5, 4, 3, False, 2),
    (7, 2, 4, True, 3), (8, 4, 4, False, 4), (8, 4, 4, True, 5),
])
def test_brute_force_tiny(N, d, dv, causal, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((N, d)) * 1.5
    k = rng.standard_normal((N, d)) * 1.5 + 0.25  # asymmetric: q/k swap shows
    v = rng.standard_normal((N, dv))
    scale = 0.7
    Ob, Lb = _brute(q, k, v, causal, scale)
    O, L = oracle.attention_fwd(q[None], k[None], v[None], causal=causal, scale=scale)
    np.testing.assert_allclose(O[0], Ob, atol=1e-13, rtol=0)
    np.testing.assert_allclose(L[0], Lb, atol=1e-13, rtol=0)
    # rows mode gives the same rows
    rows = np.arange(N)[::-1].copy()
    Or, Lr = oracle.attention_fwd(q[None], k[None], v[None], causal=causal,
                                  scale=scale, rows=rows)
    np.testing.assert_allclose(Or[0], Ob[::-1], atol=1e-13, rtol=0)
    np.testing.assert_allclose(Lr[0], Lb[::-1], atol=1e-13, rtol=0)


def test_toy_8_tokens_d4_tiles4():
    """tokentrails.org "FlashAttention": 8 tokens, d = 4, 4 x 4 tiles,
    checked against ordinary attention."""
    rng = np.random.default_rng(8)
    q, k, v = (rng.standard_normal((1, 8, 4)) for _ in range(3))
    for causal in (False, True):
        Ob, Lb = _brute(q[0], k[0], v[0], causal, 0.5)
        Ot, Lt = oracle.attention_fwd_blockwise(q, k, v, [0, 4, 8], causal=causal)
        np.testing.assert_allclose(Ot[0], Ob, atol=1e-13)
        np.testing.assert_allclose(Lt[0], Lb, atol=1e-13)


# ------------------------------------------------------- closed forms, invariants
def _rand(rng, BH, N, d, dv=None):
    dv = dv or d
    return (rng.standard_normal((BH, N, d)), rng.standard_normal((BH, N, d)),
            rng.standard_normal((BH, N, dv)))


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(11)
    q, _, v = _rand(rng, 3, 37, 16)
    k = np.broadcast_to(rng.standard_normal((3, 1, 16)), (3, 37, 16)).copy()
    scale = 0.25
    O, L = oracle.attention_fwd(q, k, v, scale=scale)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(axis=1, keepdims=True), O.shape),
                               atol=1e-13)
    s = scale * np.einsum("bnd,bd->bn", q, k[:, 0])
    np.testing.assert_allclose(L, s + math.log(37), atol=1e-12)


def test_single_key_returns_v():
    rng = np.random.default_rng(12)
    q, k, v = _rand(rng, 4, 1, 8, 5)
    O, L = oracle.attention_fwd(q, k, v, scale=0.3)
    np.testing.assert_array_equal(O, v)
    np.testing.assert_allclose(L[:, 0], 0.3 * np.einsum("bd,bd->b", q[:, 0], k[:, 0]),
                               atol=1e-14)


def test_causal_first_row_returns_v0():
    rng = np.random.default_rng(13)
    q, k, v = _rand(rng, 2, 33, 8)
    O, L = oracle.attention_fwd(q, k, v, causal=True, scale=0.5)
    np.testing.assert_allclose(O[:, 0], v[:, 0], atol=1e-15)
    np.testing.assert_allclose(L[:, 0], 0.5 * np.einsum("bd,bd->b", q[:, 0], k[:, 0]),
                               atol=1e-14)
    # causal output of row i equals non-causal attention over keys 0..i
    for i in (1, 7, 32):
        Oi, Li = oracle.attention_fwd(q[:, :i + 1], k[:, :i + 1], v[:, :i + 1],
                                      scale=0.5, rows=[i])
        np.testing.assert_allclose(O[:, i], Oi[:, 0], atol=1e-14)
        np.testing.assert_allclose(L[:, i], Li[:, 0], atol=1e-13)


def test_rows_of_p_sum_to_one_and_value_shift():
    """sum_j P_ij = 1  <=>  adding c to every value row adds c to O."""
    rng = np.random.default_rng(14)
    q, k, v = _rand(rng, 2, 50, 8, 6)
    for causal in (False, True):
        O, _ = oracle.attention_fwd(q, k, v, causal=causal)
        ones, _ = oracle.attention_fwd(q, k, np.ones_like(v), causal=causal)
        np.testing.assert_allclose(ones, 1.0, atol=1e-14)
        c = rng.standard_normal(6)
        O2, _ = oracle.attention_fwd(q, k, v + c, causal=causal)
        np.testing.assert_allclose(O2, O + c, atol=1e-13)


def test_key_value_permutation_invariance():
    rng = np.random.default_rng(15)
    q, k, v = _rand(rng, 2, 41, 8)
    perm = rng.permutation(41)
    O, L = oracle.attention_fwd(q, k, v)
    Op, Lp = oracle.attention_fwd(q, k[:, perm], v[:, perm])
    np.testing.assert_allclose(Op, O, atol=1e-13)
    np.testing.assert_allclose(Lp, L, atol=1e-13)
    # permuting keys without values must change O (catches a K/V mix-up)
    Ox, _ = oracle.attention_fwd(q, k[:, perm], v)
    assert np.abs(Ox - O).max() > 1e-3


def test_key_shift_moves_lse_only():
    rng = np.random.default_rng(16)
    q, k, v = _rand(rng, 2, 29, 8)
    u = rng.standard_normal(8)
    scale = 0.4
    O, L = oracle.attention_fwd(q, k, v, scale=scale)
    O2, L2 = oracle.attention_fwd(q, k + u, v, scale=scale)
    np.testing.assert_allclose(O2, O, atol=1e-13)
    np.testing.assert_allclose(L2, L + scale * np.einsum("bnd,d->bn", q, u), atol=1e-12)


def test_scale_enters_as_multiplier():
    """scale * (q . k): doubling q at half the scale changes nothing."""
    rng = np.random.default_rng(17)
    q, k, v = _rand(rng, 1, 23, 8)
    O, L = oracle.attention_fwd(q, k, v, scale=0.6)
    O2, L2 = oracle.attention_fwd(2 * q, k, v, scale=0.3)
    np.testing.assert_allclose(O2, O, atol=1e-14)
    np.testing.assert_allclose(L2, L, atol=1e-13)
    # and the scale really matters
    O3, _ = oracle.attention_fwd(q, k, v, scale=1.2)
    assert np.abs(O3 - O).max() > 1e-3


# --------------------------------------------------------- blockwise == dense
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("reverse", [False, True])
def test_blockwise_equals_dense_any_split(causal, reverse):
    """Blockwise online softmax equals the dense result for any split,
    including uneven blocks (gowda.ai Exercise 26.4) and, for causal rows
    visited last block first, blocks that are entirely masked."""
    rng = np.random.default_rng(18 + 2 * causal + reverse)
    N = 61
    q, k, v = _rand(rng, 2, N, 8, 5)
    q *= 2.0  # spread the scores so the running max moves often
    O, L = oracle.attention_fwd(q, k, v, causal=causal)
    splits = [[0, N], [0, 1, N], [0, 13, 14, 40, N], list(range(0, N, 4)) + [N],
              list(range(N + 1))]
    for _ in range(5):
        cuts = sorted(set(rng.integers(1, N, size=rng.integers(1, 9)).tolist()))
        splits.append([0] + cuts + [N])
    for b in splits:
        Ob, Lb = oracle.attention_fwd_blockwise(q, k, v, b, causal=causal,
                                                reverse=reverse)
        np.testing.assert_allclose(Ob, O, atol=1e-13, rtol=0)
        np.testing.assert_allclose(Lb, L, atol=1e-12, rtol=0)


def test_blockwise_late_max_moves():
    """Scores that grow along the row make the running max move at every
    block: the rescale must be applied to both l and the accumulator."""
    N = 32
    q = np.ones((1, N, 1))
    k = np.linspace(-3, 9, N).reshape(1, N, 1)
    v = np.random.default_rng(19).standard_normal((1, N, 3))
    O, L = oracle.attention_fwd(q, k, v, scale=1.0)
    Ob, Lb = oracle.attention_fwd_blockwise(q, k, v, list(range(0, N + 1, 3)) + [N]
                                            if N % 3 else list(range(0, N + 1, 3)),
                                            scale=1.0)
    np.testing.assert_allclose(Ob, O, atol=1e-13)
    np.testing.assert_allclose(Lb, L, atol=1e-12)


# ------------------------------------------------------------ degenerate cases
def test_fully_masked_row_is_defined():
    """No key allowed: defined as O = 0, LSE = -inf, never NaN (blockwise
    guard); reachable only through the blockwise reverse order per block."""
    q = np.ones((1, 3, 2))
    k = np.ones((1, 3, 2))
    v = np.ones((1, 3, 2))
    # a block that lies entirely above the diagonal for row 0
    _, _, M, Lsum, A = oracle.attention_fwd_blockwise(
        q[:, :3], k, v, [0, 1, 3], causal=True, reverse=True, rows=[0],
        return_state=True)
    assert M[0, 0] == 2.0 / math.sqrt(2) and Lsum[0, 0] == 1.0
    np.testing.assert_array_equal(A[0, 0], [1.0, 1.0])


def test_bf16_conversion_is_exact():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F80, 0xFF80, 0x3F81, 0x0000, 0x8000,
                     0x4049], dtype=np.uint16)
    want = [1.0, -2.0, 2.0 ** -133, math.inf, -math.inf, 1.0 + 2.0 ** -7, 0.0, -0.0,
            3.140625]
    got = oracle.bf16_bits_to_f64(bits)
    np.testing.assert_array_equal(got, want)
    assert math.copysign(1.0, got[7]) == -1.0


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(20)
    q, k, v = _rand(rng, 5, 130, 16)
    a = oracle.attention_fwd(q, k, v, causal=True, nthreads=1)
    b = oracle.attention_fwd(q, k, v, causal=True, nthreads=7)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_bad_arguments_rejected():
    q = np.ones((1, 4, 2))
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, q, q, rows=[4])
    with pytest.raises(ValueError):
        oracle.attention_fwd_blockwise(q, q, q, [0, 2, 2, 4])
    with pytest.raises(ValueError):
        oracle.attention_fwd_blockwise(q, q, q, [0, 3])


# ------------------------------------------------- grouped-query attention
def test_gqa_head_mapping_closed_form():
    """Query head h reads K/V head h // (H / H_kv): with identical keys per
    K/V head, O of query head h is the mean of that K/V head's values."""
    rng = np.random.default_rng(30)
    B, H, H_kv, N, d = 2, 6, 3, 17, 4
    q = rng.standard_normal((B, H, N, d))
    k = np.broadcast_to(rng.standard_normal((B, H_kv, 1, d)), (B, H_kv, N, d)).copy()
    v = rng.standard_normal((B, H_kv, N, d)) + np.arange(H_kv).reshape(1, H_kv, 1, 1) * 10
    O, _ = oracle.attention_fwd_gqa(q, k, v, scale=0.3)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(O[b, h], np.broadcast_to(v[b, h // 2].mean(0), (N, d)),
                                       atol=1e-12)


def test_gqa_reduces_to_mha_and_mqa():
    rng = np.random.default_rng(31)
    q, k, v = (rng.standard_normal((1, 4, 23, 8)) for _ in range(3))
    O1, L1 = oracle.attention_fwd_gqa(q, k, v, causal=True)
    O2, L2 = oracle.attention_fwd(q, k, v, causal=True)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)
    # one K/V head (multi-query): every query head attends to the same K/V
    k1, v1 = k[:, :1], v[:, :1]
    Om, Lm = oracle.attention_fwd_gqa(q, k1, v1)
    for h in range(4):
        Oh, Lh = oracle.attention_fwd(q[:, h:h + 1], k1, v1)
        np.testing.assert_array_equal(Om[:, h:h + 1], Oh)
        np.testing.assert_array_equal(Lm[:, h:h + 1], Lh)
    with pytest.raises(ValueError):
        oracle.attention_fwd_gqa(q, k[:, :3], v[:, :3])


# ------------------------------------------ decoding (query rows at the end)
def test_decode_rows_are_the_last_rows_of_causal_attention():
    """The newest Nq query rows against the whole cache equal the last Nq
    rows of causal self-attention over the full sequence."""
    rng = np.random.default_rng(32)
    B, H, H_kv, N, d = 2, 4, 2, 37, 8
    q_all = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H_kv, N, d))
    v = rng.standard_normal((B, H_kv, N, d))
    O_all, L_all = oracle.attention_fwd_gqa(q_all, k, v, causal=True, scale=0.4)
    for Nq in (1, 3, N):
        O, L = oracle.attention_decode(q_all[:, :, N - Nq:], k, v, causal=True, scale=0.4)
        np.testing.assert_allclose(O, O_all[:, :, N - Nq:], atol=1e-13)
        np.testing.assert_allclose(L, L_all[:, :, N - Nq:], atol=1e-13)


def test_decode_single_row_closed_forms():
    rng = np.random.default_rng(33)
    B, H, N, d = 1, 2, 29, 6
    q = rng.standard_normal((B, H, 1, d))
    k = np.broadcast_to(rng.standard_normal((B, H, 1, d)), (B, H, N, d)).copy()
    v = rng.standard_normal((B, H, N, d))
    O, L = oracle.attention_decode(q, k, v, scale=0.5)
    np.testing.assert_allclose(O[:, :, 0], v.mean(axis=2), atol=1e-13)
    s = 0.5 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    np.testing.assert_allclose(L[:, :, 0], s + math.log(N), atol=1e-12)
    # brute force for one row (random keys) in 40-digit decimals
    kr = rng.standard_normal((N, d))
    Ob, Lb = _brute(np.concatenate([np.zeros((N - 1, d)), q[0, 0]]), kr, v[0, 0], True, 0.5)
    Od, Ld = oracle.attention_decode(q[:1, :1], kr[None, None], v[:1, :1], scale=0.5)
    np.testing.assert_allclose(Od[0, 0, 0], Ob[-1], atol=1e-13)
    assert abs(Ld[0, 0, 0] - Lb[-1]) < 1e-13


# ------------------------------------------------------------------ backward
def _loss(q, k, v, do, causal, scale):
    O, _ = oracle.attention_fwd(q, k, v, causal=causal, scale=scale)
    return float(np.sum(O * do))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    """d(sum O * dO)/dX by central differences (the definition of the
    gradient) for every element of Q, K, V on a tiny head."""
    rng = np.random.default_rng(40 + causal)
    N, d, scale = 6, 3, 0.7
    q, k, v, do = (rng.standard_normal((1, N, d)) for _ in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + eps
            fp = _loss(q, k, v, do, causal, scale)
            x[idx] = x0 - eps
            fm = _loss(q, k, v, do, causal, scale)
            x[idx] = x0
            num[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(g, num, atol=1e-7, rtol=1e-6)


def _loss_gqa(q, k, v, do, causal, scale):
    O, _ = oracle.attention_fwd_gqa(q, k, v, causal=causal, scale=scale)
    return float(np.sum(O * do))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_gqa_matches_finite_differences(causal):
    """Grouped-query gradients by central differences of sum(O * dO) with O
    from the grouped-query forward oracle: every element of Q and of the
    shared K and V heads (four query heads on two K/V heads)."""
    rng = np.random.default_rng(50 + causal)
    B, H, H_kv, N, d, scale = 1, 4, 2, 5, 3, 0.6
    q, do = (rng.standard_normal((B, H, N, d)) for _ in range(2))
    k, v = (rng.standard_normal((B, H_kv, N, d)) for _ in range(2))
    dq, dk, dv = oracle.attention_bwd_gqa(q, k, v, do, causal=causal, scale=scale)
    assert dk.shape == k.shape and dv.shape == v.shape and dq.shape == q.shape
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + eps
            fp = _loss_gqa(q, k, v, do, causal, scale)
            x[idx] = x0 - eps
            fm = _loss_gqa(q, k, v, do, causal, scale)
            x[idx] = x0
            num[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(g, num, atol=1e-7, rtol=1e-6)


def test_backward_identities():
    """Rows of dS sum to zero, so shifting every key by u leaves dQ unchanged
    and every key-gradient sum is zero; D_i = sum_r dO_ir O_ir."""
    rng = np.random.default_rng(42)
    q, k, v, do = (rng.standard_normal((2, 40, 8)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv, D = oracle.attention_bwd(q, k, v, do, causal=causal, scale=0.3,
                                             return_D=True)
        O, _ = oracle.attention_fwd(q, k, v, causal=causal, scale=0.3)
        np.testing.assert_allclose(D, np.sum(do * O, axis=-1), atol=1e-12)
        # sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0
        np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
        dq2, _, dv2 = oracle.attention_bwd(q, k + rng.standard_normal(8), v, do,
                                           causal=causal, scale=0.3)
        np.testing.assert_allclose(dq2, dq, atol=1e-11)
        np.testing.assert_allclose(dv2, dv, atol=1e-11)
        # dV = P^T dO: with dO = all ones, the column sums of P (keys' total weight)
        _, _, dv1 = oracle.attention_bwd(q, k, v, np.ones_like(do), causal=causal, scale=0.3)
        if not causal:
            np.testing.assert_allclose(dv1.sum(axis=1), 40.0 * np.ones((2, 8)), atol=1e-10)


def test_backward_with_given_D():
    """The backward's optional D input (section 3.6's D_i = sum_r dO_ir O_ir
    taken from another O): the exact D reproduces the default bit for bit,
    and a shift delta_i of D_i leaves dV unchanged and moves dQ_i by
    -scale * delta_i * sum_j P_ij K_j, which is the forward pass with K in
    place of V (dS_ij moves by -P_ij delta_i)."""
    g = np.random.default_rng(17)
    B, H, N, d = 1, 2, 9, 5
    q, k, v, do = (g.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 0.4
    for causal in (False, True):
        dq, dk, dv, D = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale,
                                             return_D=True)
        dq2, dk2, dv2 = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale, D=D)
        assert np.array_equal(dq, dq2) and np.array_equal(dk, dk2) and np.array_equal(dv, dv2)
        delta = g.standard_normal((B, H, N)) * 0.1
        dq3, dk3, dv3 = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale,
                                             D=D + delta)
        assert np.allclose(dv3, dv, rtol=0, atol=1e-13)
        wk, _ = oracle.attention_fwd(q, k, k, causal=causal, scale=scale)  # sum_j P_ij K_j
        assert np.allclose(dq3 - dq, -scale * delta[..., None] * wk, rtol=0, atol=1e-12)
