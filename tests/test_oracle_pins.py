"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

None of these re-type the oracle's formulas: each checks a closed form, an
invariant, a special case with a hand-derived answer (tests/golden/), an
independent library routine, or brute force on tiny inputs -- chosen so that a
dropped term, a wrong sign or index, or a transposed operand fails one of them.
CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from gated_deltanet_linear_gdn_gb300 import inputs as gi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf(x):
    """fp32-exact values -> bf16 bits (generator helper)."""
    return gi.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def bfv(bits):
    return gi.bf16_bits_to_f32(bits).astype(np.float64)


# --------------------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_on_fp32_values(oracle):
    """On fp32-representable values one rounding to bf16 equals torch's fp32->bf16 RNE."""
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(2000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 2000),
                        rng.standard_normal(500).astype(np.float32) * 1e-39]).astype(np.float32)
    ours = oracle.round_bf16_array(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("x,bits", [
    (1.0 + 2.0 ** -8, 0x3F80),               # tie -> even (1.0)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),           # tie -> even (1 + 2^-6)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),  # just above the tie: one rounding rounds up
    (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
    (2.0 ** -133, 0x0001),                   # smallest subnormal
    (2.0 ** -134, 0x0000),                   # tie at half the smallest subnormal -> even (0)
    (1.5 * 2.0 ** -134, 0x0001),
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),  # largest finite
    (2.0 ** 128, 0x7F80),                    # overflow -> inf
    (0.0, 0x0000),
    (-0.0, 0x8000),
])
def test_round_bf16_ieee_cases(oracle, x, bits):
    assert oracle.round_bf16(x) == bits


# --------------------------------------------------------------------------- conv

def _conv_case(D=16, W=4, B=1, num_slots=3, cache_f32=False, layout=0, seed=0):
    rng = np.random.default_rng(seed)
    x = bf(rng.standard_normal((B, D)))
    if layout == 0:
        st = rng.standard_normal((num_slots, D, W - 1)).astype(np.float32)
    else:
        st = rng.standard_normal((num_slots, W - 1, D)).astype(np.float32)
    if not cache_f32:
        st = bf(st)
    return x, st


@pytest.mark.parametrize("cache_f32", [False, True])
@pytest.mark.parametrize("layout", [0, 1])
def test_conv_one_hot_taps_pin_order(oracle, cache_f32, layout):
    """Tap W-1 multiplies the newest input, tap 0 the oldest cached one."""
    D, W = 16, 4
    x, st = _conv_case(D, W, cache_f32=cache_f32, layout=layout)
    slot = np.array([1], np.int32)
    st_before = st.copy()
    w_new = np.zeros((D, W), np.float32); w_new[:, W - 1] = 1.0
    out, _, err = oracle.conv_update(x, st, cache_f32, layout, bf(w_new), None, 0, slot, 3)
    assert err == 0
    assert np.array_equal(out, x)  # out == x bitwise
    st2 = st_before.copy()
    w_old = np.zeros((D, W), np.float32); w_old[:, 0] = 1.0
    out, _, _ = oracle.conv_update(x, st2, cache_f32, layout, bf(w_old), None, 0, slot, 3)
    oldest = st_before[1, :, 0] if layout == 0 else st_before[1, 0, :]
    oldest = oldest if not cache_f32 else bf(oldest)  # bf16 output of an fp32 cache value
    assert np.array_equal(out[0], oldest)


@pytest.mark.parametrize("cache_f32", [False, True])
@pytest.mark.parametrize("layout", [0, 1])
def test_conv_state_roll_is_a_shift(oracle, cache_f32, layout):
    D, W = 24, 4
    x, st = _conv_case(D, W, B=2, num_slots=4, cache_f32=cache_f32, layout=layout, seed=3)
    before = st.copy()
    w = bf(np.random.default_rng(1).standard_normal((D, W)) * 0.1)
    slot = np.array([3, 1], np.int32)
    oracle.conv_update(x, st, cache_f32, layout, w, None, 1, slot, 4)
    for b, s in enumerate(slot):
        if layout == 0:
            assert np.array_equal(st[s, :, :W - 2], before[s, :, 1:])
            newest = st[s, :, W - 2]
        else:
            assert np.array_equal(st[s, :W - 2, :], before[s, 1:, :])
            newest = st[s, W - 2, :]
        exp_new = bfv(x[b]).astype(np.float32) if cache_f32 else x[b]
        assert np.array_equal(newest, exp_new)
    assert np.array_equal(st[0], before[0]) and np.array_equal(st[2], before[2])


def test_conv_products_rounded_to_operand_dtype(oracle):
    """Cancellation input: (1+2^-7)^2 = 1 + 2^-6 + 2^-14 rounds to 1 + 2^-6 in bf16 and then
    cancels -(1+2^-6) * 1 exactly; with an fp32 cache the products are exact in fp32 and
    2^-14 survives. (RL-Kernel PR #469, Summary: each tap product is rounded to the operand
    dtype before the fp32 accumulation.)"""
    D, W = 8, 4
    w = np.zeros((D, W), np.float32)
    w[:, 2] = 1.0 + 2.0 ** -7
    w[:, 3] = -(1.0 + 2.0 ** -6)
    x = bf(np.ones((1, D)))
    for cache_f32, expect in [(False, 0.0), (True, 2.0 ** -14)]:
        st = np.zeros((2, D, W - 1), np.float32)
        st[1, :, 2] = 1.0 + 2.0 ** -7
        if not cache_f32:
            st = bf(st)
        out, act, _ = oracle.conv_update(x, st, cache_f32, 0, bf(w), None, 0,
                                         np.array([1], np.int32), 2)
        assert np.all(act == expect)
        assert np.all(bfv(out) == expect)


def test_conv_accumulator_is_fp32(oracle):
    """bias + 1 + 2^-30 accumulates in fp32: 2^-30 is lost next to 1 (fp32 has 24 bits)."""
    D, W = 8, 4
    w = np.zeros((D, W), np.float32); w[:, 3] = 1.0; w[:, 2] = 2.0 ** -15
    st = np.zeros((2, D, W - 1), np.float32); st[1, :, 2] = 2.0 ** -15  # product 2^-30
    x = bf(np.ones((1, D)))
    bias = bf(np.full(D, 0.0))
    out, act, _ = oracle.conv_update(x, bf(st), 0, 0, bf(w), bias, 0, np.array([1], np.int32), 2)
    assert np.all(act == 1.0)  # fp64 accumulation would give 1 + 2^-30


def test_conv_silu_odd_part_identity(oracle):
    """silu(y) - silu(-y) = y for any y: channels with negated taps give pre-activations
    y and -y exactly, so the two SiLU outputs must differ by the pre-activation."""
    D, W = 32, 4
    rng = np.random.default_rng(2)
    wh = rng.standard_normal((D // 2, W)).astype(np.float32) * 0.7
    w = np.concatenate([wh, -wh]).astype(np.float32)
    st = rng.standard_normal((2, D, W - 1)).astype(np.float32)
    st[:, D // 2:] = st[:, :D // 2]
    xh = rng.standard_normal(D // 2).astype(np.float32)
    x = bf(np.concatenate([xh, xh])[None])
    st = bf(st)
    pre_out, pre, _ = oracle.conv_update(x, st.copy(), 0, 0, bf(w), None, 0, np.array([1], np.int32), 2)
    _, act, _ = oracle.conv_update(x, st.copy(), 0, 0, bf(w), None, 1, np.array([1], np.int32), 2)
    y = pre[0, :D // 2]
    assert np.array_equal(pre[0, D // 2:], -y)
    assert np.allclose(act[0, :D // 2] - act[0, D // 2:], y, rtol=0, atol=1e-15)
    assert np.all(np.abs(y) > 0)


def test_conv_silu_limits(oracle):
    """silu(0) = 0; silu(y) -> y for large y; silu(y) -> 0 for very negative y."""
    D, W = 8, 4
    w = np.zeros((D, W), np.float32); w[:, 3] = 1.0
    xs = np.array([[0.0, 40.0, -40.0, 100.0, -100.0, 0.0, 1.0, -1.0]], np.float32)
    st = bf(np.zeros((2, D, W - 1)))
    _, act, _ = oracle.conv_update(bf(xs), st, 0, 0, bf(w), None, 1, np.array([1], np.int32), 2)
    a = act[0]
    assert a[0] == 0.0 and a[5] == 0.0
    assert abs(a[1] - 40.0) < 1e-15 and abs(a[3] - 100.0) < 1e-40
    assert -1e-15 < a[2] < 0 and -1e-40 < a[4] <= 0
    # sigmoid(1) = e / (1 + e): silu(1) - silu(-1) = 1 and silu(1) = e/(1+e)
    assert abs(a[6] - math.e / (1 + math.e)) < 1e-15


def test_conv_layouts_agree(oracle):
    D, W, B, S = 40, 4, 3, 5
    rng = np.random.default_rng(9)
    x = bf(rng.standard_normal((B, D)))
    st0 = bf(rng.standard_normal((S, D, W - 1)))
    st1 = np.ascontiguousarray(st0.transpose(0, 2, 1))
    w = bf(rng.standard_normal((D, W)) * 0.3)
    bias = bf(rng.standard_normal(D) * 0.3)
    slot = np.array([4, 2, 1], np.int32)
    o0, _, _ = oracle.conv_update(x, st0, 0, 0, w, bias, 1, slot, S)
    o1, _, _ = oracle.conv_update(x, st1, 0, 1, w, bias, 1, slot, S)
    assert np.array_equal(o0, o1)
    assert np.array_equal(st0, st1.transpose(0, 2, 1))


def test_conv_slot_contract(oracle):
    """slot <= 0: zero output, state untouched; slot >= num_slots: error bit, untouched."""
    D, W, S = 16, 4, 4
    rng = np.random.default_rng(4)
    x = bf(rng.standard_normal((4, D)))
    st = bf(rng.standard_normal((S, D, W - 1)))
    before = st.copy()
    w = bf(rng.standard_normal((D, W)))
    slot = np.array([0, -3, 4, 2], np.int32)
    out, _, err = oracle.conv_update(x, st, 0, 0, w, None, 1, slot, S)
    assert err == 1
    assert np.all(out[:3] == 0)
    assert np.array_equal(st[[0, 1, 3]], before[[0, 1, 3]])
    assert not np.array_equal(st[2], before[2])


def test_validate_slots(oracle):
    assert oracle.validate_slots([1, 2, 0, -1, 0], 3) == 0
    assert oracle.validate_slots([1, 3], 3) == 1
    assert oracle.validate_slots([2, 0, 2], 3) == 2
    assert oracle.validate_slots([0, 0, -1, -1], 1) == 0


# --------------------------------------------------------------------------- gating

def test_softplus_and_sigmoid(oracle):
    for x in [20.0000001, 25.0, 88.0, 1000.0]:
        assert oracle.softplus(x) == x  # the threshold branch returns x itself
    assert abs(oracle.softplus(0.0) - math.log(2.0)) < 1e-16
    for x in [-5.0, -0.3, 0.7, 3.0, 19.9]:
        assert abs(oracle.softplus(x) - oracle.softplus(-x) - x) < 1e-14  # sp(x) - sp(-x) = x
        assert abs(oracle.sigmoid(x) + oracle.sigmoid(-x) - 1.0) < 1e-15
    assert abs(oracle.softplus(20.0) - 20.0) < 2.1e-9  # continuous at the threshold
    assert oracle.sigmoid(0.0) == 0.5


def _identity_state_case(geo, q_vals, A_log, dt_bias, a_val, b_val, k_zero=True):
    """One decode row, conv bypassed, S0 = identity for every head, k = 0 (so k_hat = 0 and
    the update vanishes): o_h = alpha_h * S0 q_hat = alpha_h * q_hat."""
    D = geo.D
    mixed = np.zeros((1, D), np.float32)
    mixed[0, :geo.Hk * geo.dk] = q_vals
    if not k_zero:
        raise NotImplementedError
    ssm = np.zeros((2, geo.Hv, geo.dv, geo.dk))
    ssm[1] = np.eye(geo.dv, geo.dk)[None]
    a = bf(np.full((1, geo.Hv), a_val)); b = bf(np.full((1, geo.Hv), b_val))
    return bf(mixed), a, b, ssm


def test_fused_gate_and_qk_norm_closed_form(oracle):
    """With k = 0 and S0 = I: o = alpha q_hat, alpha = exp(-exp(A_log) softplus(a + dt_bias)),
    |q_hat|^2 = scale^2 sum q^2 / (sum q^2 + 1e-6) (QK norm x / sqrt(sum x^2 + 1e-6), scale on
    q after the norm; RL-Kernel PR #469, Notes, 'How the golden relates to the kernel')."""
    geo = gi.Geometry(Hk=1, Hv=2, dk=8, dv=8)
    q = np.array([1e-3, -2e-3, 0, 0, 0, 0, 5e-4, 0], np.float32)  # small: eps matters
    A_log = np.array([math.log(2.0), 0.0], np.float32)
    dt_bias = np.array([0.0, 0.5], np.float32)
    mixed, a, b, ssm = _identity_state_case(geo, q, A_log, dt_bias, a_val=0.0, b_val=0.0)
    scale = 0.37
    out, _, err = oracle.decode_step(mixed, a, b, False, A_log, dt_bias, None, None, 0, None, 0, 0,
                                     ssm, np.array([1], np.int32), geo.Hk, geo.Hv, geo.dk, geo.dv,
                                     scale=scale)
    qb = bfv(mixed[0, :8])
    ss = float(np.sum(qb ** 2))
    for h in range(2):
        alpha = math.exp(-math.exp(float(A_log[h])) * math.log1p(math.exp(float(dt_bias[h]))))
        o = out[0, h]
        assert abs(float(np.sum(o ** 2)) / alpha ** 2 - scale ** 2 * ss / (ss + 1e-6)) < 1e-12
        direction = qb / math.sqrt(ss)
        assert np.allclose(o / np.linalg.norm(o), direction, atol=1e-12)
    # head 0: exp(A_log) = 2, softplus(0) = ln 2 -> alpha = 1/4 ; head 1: alpha = exp(-sp(0.5))
    # (A_log = fp32(ln 2), so alpha_0 is 1/4 up to that rounding)
    r0 = np.linalg.norm(out[0, 0]); r1 = np.linalg.norm(out[0, 1])
    alpha0 = math.exp(-math.exp(float(A_log[0])) * math.log(2.0))
    assert abs(alpha0 - 0.25) < 1e-8
    assert abs(r0 / r1 - alpha0 / math.exp(-math.log1p(math.exp(0.5)))) < 1e-12


def test_no_qk_norm_scales_q_only(oracle):
    geo = gi.Geometry(Hk=1, Hv=1, dk=4, dv=4)
    q = np.array([0.5, -1.0, 2.0, 0.25], np.float32)
    mixed, a, b, ssm = _identity_state_case(geo, q, None, None, 0.0, 0.0)
    g = np.array([[0.0]], np.float32); beta = np.array([[0.3]], np.float32)
    out, _, _ = oracle.decode_step(mixed, g, beta, True, None, None, None, None, 0, None, 0, 0, ssm,
                                   np.array([1], np.int32), 1, 1, 4, 4, scale=0.5, qk_l2norm=False)
    assert np.array_equal(out[0, 0], 0.5 * q.astype(np.float64))


def test_gqa_head_mapping(oracle):
    """k-head of value head h is h // (Hv / Hk) (no repeat_interleave). With Hk=2, Hv=4 and
    the keys of k-head 0 zero, heads 0 and 1 see no update, heads 2 and 3 do."""
    geo = gi.Geometry(Hk=2, Hv=4, dk=8, dv=8)
    rng = np.random.default_rng(11)
    mixed = rng.standard_normal((1, geo.D)).astype(np.float32)
    mixed[0, geo.Hk * geo.dk: geo.Hk * geo.dk + geo.dk] = 0.0   # k of k-head 0
    ssm = rng.standard_normal((2, geo.Hv, geo.dv, geo.dk)) * 0.3
    S0 = ssm.copy()
    g = np.full((1, geo.Hv), -0.1, np.float32); beta = np.full((1, geo.Hv), 0.8, np.float32)
    out, _, _ = oracle.decode_step(bf(mixed), g, beta, True, None, None, None, None, 0, None, 0, 0,
                                   ssm, np.array([1], np.int32), geo.Hk, geo.Hv, geo.dk, geo.dv)
    alpha = math.exp(float(np.float32(-0.1)))  # g travels as fp32
    for h in range(4):
        decayed = alpha * S0[1, h]
        if h < 2:
            assert np.allclose(ssm[1, h], decayed, rtol=0, atol=1e-15)
        else:
            assert np.abs(ssm[1, h] - decayed).max() > 1e-3
    # heads 2 and 3 read the q of k-head 1: o_h = S_h q_hat(k-head 1)
    qb = bfv(bf(mixed)[0, geo.dk: 2 * geo.dk])
    qh = qb / math.sqrt(np.sum(qb ** 2) + 1e-6) * geo.dk ** -0.5
    for h in (2, 3):
        assert np.allclose(out[0, h], ssm[1, h] @ qh, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------- the rule

def test_hand_derived_fixture(oracle):
    with open(os.path.join(GOLDEN, "hand_rule.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        g = np.log(np.array(c["alpha"]))
        o, S = oracle.recurrent_head(c["q"], c["k"], c["v"], g, c["beta"], c["S0"])
        assert np.allclose(o, c["o"], rtol=1e-15, atol=1e-15), c["name"]
        assert np.allclose(S, c["S_final"], rtol=1e-15, atol=1e-15), c["name"]


def test_scalar_case_brute_force(oracle):
    """dk = dv = 1: s_t = a_t s_{t-1} (1 - b_t k_t^2) + b_t v_t k_t, o_t = s_t q_t (the rule
    with every product a scalar, rearranged by hand)."""
    rng = np.random.default_rng(7)
    T = 9
    q, k, v = (rng.standard_normal((T, 1)) for _ in range(3))
    g = -np.abs(rng.standard_normal(T)); beta = rng.uniform(0, 1, T)
    o, S = oracle.recurrent_head(q, k, v, g, beta, [[0.7]])
    s = 0.7
    for t in range(T):
        a = math.exp(g[t])
        s = a * s * (1 - beta[t] * k[t, 0] ** 2) + beta[t] * v[t, 0] * k[t, 0]
        assert abs(o[t, 0] - s * q[t, 0]) < 1e-14
    assert abs(S[0, 0] - s) < 1e-14


def test_beta_zero_only_decays(oracle):
    """beta = 0: S_T = exp(sum g) S0 and o_t = exp(G_t) S0 q_t."""
    rng = np.random.default_rng(1)
    T, dk, dv = 12, 16, 8
    q, k = rng.standard_normal((T, dk)), rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    g = -np.abs(rng.standard_normal(T)) * 0.3
    S0 = rng.standard_normal((dv, dk))
    o, S = oracle.recurrent_head(q, k, v, g, np.zeros(T), S0)
    G = np.cumsum(g)
    assert np.allclose(S, math.exp(G[-1]) * S0, rtol=1e-13, atol=0)
    for t in range(T):
        assert np.allclose(o[t], math.exp(G[t]) * (S0 @ q[t]), rtol=1e-12, atol=1e-14)


def test_exact_recall_orthonormal_keys(oracle):
    """Orthonormal keys, g = 0, beta = 1, zero state: S_n = sum v_i k_i^T, so S_n k_j = v_j,
    and the output at token t with q_t = k_j (j <= t) is v_j."""
    rng = np.random.default_rng(3)
    dk, dv, n = 16, 12, 10
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :n].T                        # n orthonormal rows
    v = rng.standard_normal((n, dv))
    q = keys[rng.integers(0, 1, n)]           # q_t = k_0 (stored at t = 0)
    o, S = oracle.recurrent_head(q, keys, v, np.zeros(n), np.ones(n), np.zeros((dv, dk)))
    for j in range(n):
        assert np.allclose(S @ keys[j], v[j], atol=1e-13)
    assert np.allclose(o, np.broadcast_to(v[0], o.shape), atol=1e-13)


# --------------------------------------------------------------------------- chunked form

@pytest.mark.parametrize("C,T", [(16, 16), (16, 50), (64, 64), (64, 150), (32, 77), (16, 1)])
def test_chunked_equals_recurrent(oracle, C, T):
    rng = np.random.default_rng(C * 1000 + T)
    dk, dv = 16, 12
    q = rng.standard_normal((T, dk)); k = rng.standard_normal((T, dk))
    q /= np.linalg.norm(q, axis=1, keepdims=True); k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    g = -np.abs(rng.standard_normal(T)) * 2.0
    g[::7] = -25.0  # decays whose chunk products underflow exp(G) in fp32
    beta = rng.uniform(0, 1, T)
    S0 = rng.standard_normal((dv, dk)) * 0.3
    o_r, S_r = oracle.recurrent_head(q, k, v, g, beta, S0)
    o_c, S_c = oracle.chunked_head(q, k, v, g, beta, S0, C)
    assert np.abs(o_c - o_r).max() <= 1e-12 * max(1.0, np.abs(o_r).max())
    assert np.abs(S_c - S_r).max() <= 1e-12 * max(1.0, np.abs(S_r).max())


def test_chunked_detects_a_dropped_decay(oracle):
    """Planted check of the pin itself: g != 0 and the chunked path (correct) differs from the
    recurrence run with g = 0 by far more than the pin's tolerance."""
    rng = np.random.default_rng(0)
    T, dk, dv = 20, 8, 8
    q = rng.standard_normal((T, dk)); k = rng.standard_normal((T, dk)); v = rng.standard_normal((T, dv))
    g = np.full(T, -0.5); beta = np.full(T, 0.5)
    o_c, _ = oracle.chunked_head(q, k, v, g, beta, np.zeros((dv, dk)), 8)
    o_bad, _ = oracle.recurrent_head(q, k, v, np.zeros(T), beta, np.zeros((dv, dk)))
    assert np.abs(o_c - o_bad).max() > 1e-3


def test_unit_lower_inverse(oracle):
    rng = np.random.default_rng(0)
    n = 64
    A = np.tril(rng.standard_normal((n, n)) * 0.3, -1)
    T = oracle.unit_lower_inverse(A)
    assert np.abs(T @ (np.eye(n) + A) - np.eye(n)).max() < 1e-12
    assert np.all(np.triu(T, 1) == 0) and np.all(np.diag(T) == 1)


# --------------------------------------------------------------------------- adversarial case

def _adversarial_head(seed=0, T=64, dk=128, dv=128):
    case = gi.correlated_keys(T=T, seed=seed, geo=gi.Geometry(Hk=1, Hv=1, dk=dk, dv=dv))
    y = bfv(case.mixed)
    q = y[:, :dk]; k = y[:, dk:2 * dk]; v = y[:, 2 * dk:]
    q = q / np.sqrt(np.sum(q * q, 1, keepdims=True) + 1e-6) * dk ** -0.5
    k = k / np.sqrt(np.sum(k * k, 1, keepdims=True) + 1e-6)
    return q, k, v, np.zeros(T), np.full(T, 0.9)


def test_adversarial_exact_inverse_is_accurate(oracle):
    """Correlated keys, beta = 0.9, g = 0, zero state (vLLM PR #53864, 'Numerical root cause
    and fix'): the exact chunked path is finite and equals the recurrence; the fp64 inverse
    satisfies T (I + A) = I."""
    q, k, v, g, beta = _adversarial_head()
    S0 = np.zeros((128, 128))
    o_r, S_r = oracle.recurrent_head(q, k, v, g, beta, S0)
    for C in (16, 64):
        o_c, S_c = oracle.chunked_head(q, k, v, g, beta, S0, C)
        assert np.all(np.isfinite(o_c)) and np.all(np.isfinite(S_c))
        assert np.abs(o_c - o_r).max() <= 1e-10 * np.abs(o_r).max()
        assert np.abs(S_c - S_r).max() <= 1e-10 * np.abs(S_r).max()
    A = np.tril(0.9 * (k @ k.T), -1)
    T = oracle.unit_lower_inverse(A)
    assert np.abs(T @ (np.eye(64) + A) - np.eye(64)).max() < 1e-12


def test_adversarial_three_round_bf16_newton_schulz_fails(oracle):
    """Negative control: the 3-round bf16 Newton-Schulz block inverse that vLLM PR #53864
    replaces must fail the page's output gate (max abs error < 0.1) on correlated keys."""
    q, k, v, g, beta = _adversarial_head()
    S0 = np.zeros((128, 128))
    o_r, _ = oracle.recurrent_head(q, k, v, g, beta, S0)
    o3, _ = oracle.chunked_head(q, k, v, g, beta, S0, 64, inverse_mode=3)
    assert not (np.abs(o3 - o_r).max() < 0.1)
    # the page's fix, a fourth round, passes the same gate
    o4, _ = oracle.chunked_head(q, k, v, g, beta, S0, 64, inverse_mode=4)
    assert np.abs(o4 - o_r).max() < 0.1


# --------------------------------------------------------------------------- prefill state carry

@pytest.mark.parametrize("cache_f32", [False, True])
@pytest.mark.parametrize("has_init", [0, 1])
def test_prefill_final_conv_state_is_last_inputs(oracle, cache_f32, has_init):
    """Final conv window = the last W-1 entries of (initial window ++ x)."""
    geo = gi.TINY
    case = gi.make_inputs(geo, [1, 2, 3, 5], 8, seed=2, conv_f32=cache_f32,
                          has_init=[has_init] * 4)
    st0 = case.conv_state.copy()
    ssm = case.ssm_state.astype(np.float64)
    oracle.layer(case.mixed, case.a, case.b, False, case.A_log, case.dt_bias, case.conv_w,
                 case.conv_b, 1, case.conv_state, cache_f32, 0, ssm, case.cu_seqlens, case.slot,
                 case.has_init, geo.Hk, geo.Hv, geo.dk, geo.dv)
    xf = bfv(case.mixed)
    for i, s in enumerate(case.slot):
        bos, eos = case.cu_seqlens[i], case.cu_seqlens[i + 1]
        init = st0[s].astype(np.float64) if cache_f32 else bfv(st0[s])
        if not has_init:
            init = np.zeros_like(init)
        full = np.concatenate([init, xf[bos:eos].T], axis=1)   # [D, W-1+L]
        expect = full[:, -(geo.W - 1):]
        got = case.conv_state[s].astype(np.float64) if cache_f32 else bfv(case.conv_state[s])
        assert np.array_equal(got, expect)


def test_prefill_without_initial_state_ignores_the_slot(oracle):
    """has_initial_state = 0: the sequence starts from a zero recurrent state and a zero conv
    window whatever its slot holds, and its final state is written to the slot.

    (a) Conv bypassed, direct gates, no QK norm, scale 1: every head's outputs and final state
        equal the single-head recurrence (pinned above by closed forms and hand fixtures) run
        from S0 = 0, although the slot holds a non-zero state; the sequence beside it, which
        has an initial state, equals the recurrence from its slot's state.
    (b) Conv on: the call equals one that reads slots whose state and conv window were
        zeroed beforehand, and differs from one that reads the slots as they are."""
    geo = gi.TINY
    dk, dv, Hk, Hv = geo.dk, geo.dv, geo.Hk, geo.Hv
    case = gi.make_inputs(geo, [9, 5], 6, seed=13, conv=False, gate_direct=True,
                          has_init=[0, 1], state_std=0.5)
    case.qk_l2norm = False
    ssm0 = case.ssm_state.astype(np.float64)
    ssm = ssm0.copy()
    out, _, _ = oracle.layer(case.mixed, case.a, case.b, True, case.A_log, case.dt_bias, None,
                             None, 0, None, 0, 0, ssm, case.cu_seqlens, case.slot, case.has_init,
                             Hk, Hv, dk, dv, scale=1.0, qk_l2norm=False)
    x = bfv(case.mixed)
    for i, s in enumerate(case.slot):
        assert np.abs(ssm0[s]).max() > 0.1          # the slot holds a state worth ignoring
        bos, eos = case.cu_seqlens[i], case.cu_seqlens[i + 1]
        for h in range(Hv):
            kh = h // (Hv // Hk)
            q = x[bos:eos, kh * dk:(kh + 1) * dk]
            k = x[bos:eos, (Hk + kh) * dk:(Hk + kh + 1) * dk]
            v = x[bos:eos, 2 * Hk * dk + h * dv:2 * Hk * dk + (h + 1) * dv]
            S0 = np.zeros((dv, dk)) if case.has_init[i] == 0 else ssm0[s, h]
            o_ref, S_ref = oracle.recurrent_head(q, k, v, case.a[bos:eos, h], case.b[bos:eos, h],
                                                 S0)
            assert np.allclose(out[bos:eos, h], o_ref, rtol=0, atol=1e-14)
            assert np.allclose(ssm[s, h], S_ref, rtol=0, atol=1e-14)

    case = gi.make_inputs(geo, [6, 4], 6, seed=14, has_init=[0, 0])
    runs = []
    for mode in ("no_init", "zeroed_slots", "read_slots"):
        conv = case.conv_state.copy()
        ssm = case.ssm_state.astype(np.float64)
        hi = case.has_init
        if mode != "no_init":
            hi = None
        if mode == "zeroed_slots":
            conv[case.slot] = 0
            ssm[case.slot] = 0.0
        o, _, _ = oracle.layer(case.mixed, case.a, case.b, False, case.A_log, case.dt_bias,
                               case.conv_w, case.conv_b, 1, conv, 0, 0, ssm, case.cu_seqlens,
                               case.slot, hi, Hk, Hv, dk, dv)
        runs.append((o, conv, ssm))
    (o0, c0, s0), (o1, c1, s1), (o2, _, _) = runs
    assert np.array_equal(o0, o1) and np.array_equal(c0, c1) and np.array_equal(s0, s1)
    assert not np.allclose(o0, o2)


def test_prefill_equals_decode_steps(oracle):
    """A sequence prefilled at once equals the same tokens fed as successive decode steps."""
    geo = gi.TINY
    L = 7
    case = gi.make_inputs(geo, [L], 8, seed=4)
    st_a = case.conv_state.copy(); st_b = case.conv_state.copy()
    ssm_a = case.ssm_state.astype(np.float64); ssm_b = ssm_a.copy()
    out_a, _, _ = oracle.layer(case.mixed, case.a, case.b, False, case.A_log, case.dt_bias,
                               case.conv_w, case.conv_b, 1, st_a, 0, 0, ssm_a, case.cu_seqlens,
                               case.slot, None, geo.Hk, geo.Hv, geo.dk, geo.dv)
    outs = []
    for t in range(L):
        o, _, _ = oracle.decode_step(case.mixed[t:t + 1], case.a[t:t + 1], case.b[t:t + 1], False,
                                     case.A_log, case.dt_bias, case.conv_w, case.conv_b, 1, st_b, 0,
                                     0, ssm_b, case.slot, geo.Hk, geo.Hv, geo.dk, geo.dv)
        outs.append(o[0])
    assert np.array_equal(out_a, np.stack(outs))
    assert np.array_equal(ssm_a, ssm_b) and np.array_equal(st_a, st_b)


# --------------------------------------------------------------------------- slots + invariance

def test_layer_slot_contract(oracle):
    geo = gi.TINY
    case = gi.make_inputs(geo, [1] * 4, 6, seed=8, slots=[0, 5, 6, -2])
    ssm = case.ssm_state.astype(np.float64)
    before_ssm = ssm.copy(); before_conv = case.conv_state.copy()
    out, bits, err = oracle.decode_step(case.mixed, case.a, case.b, False, case.A_log, case.dt_bias,
                                        case.conv_w, case.conv_b, 1, case.conv_state, 0, 0, ssm,
                                        case.slot, geo.Hk, geo.Hv, geo.dk, geo.dv)
    assert err == 1
    assert np.all(out[[0, 2, 3]] == 0) and np.all(bits[[0, 2, 3]] == 0)
    untouched = [0, 1, 2, 3, 4]
    assert np.array_equal(ssm[untouched], before_ssm[untouched])
    assert np.array_equal(case.conv_state[untouched], before_conv[untouched])
    assert not np.array_equal(ssm[5], before_ssm[5])


def _run_rows(oracle, case, rows, pool_perm=None):
    """Run decode for a subset of rows; optionally with the cache blocks permuted."""
    geo = case.geo
    nslot = case.num_slots
    perm = np.arange(nslot) if pool_perm is None else pool_perm
    inv = np.argsort(perm)
    conv = np.ascontiguousarray(case.conv_state[perm])
    ssm = np.ascontiguousarray(case.ssm_state[perm].astype(np.float64))
    slot = inv[case.slot[rows]].astype(np.int32)
    out, _, _ = oracle.decode_step(case.mixed[rows], case.a[rows], case.b[rows], False, case.A_log,
                                   case.dt_bias, case.conv_w, case.conv_b, 1, conv, 0, 0, ssm, slot,
                                   geo.Hk, geo.Hv, geo.dk, geo.dv)
    return out, {int(case.slot[r]): (conv[inv[case.slot[r]]], ssm[inv[case.slot[r]]]) for r in rows}


def test_oracle_batch_invariance_protocol(oracle):
    """Every row alone, sub-batches of 2 and 7 at offsets, shuffled order, contiguous and
    shuffled cache blocks: outputs and rolled state blocks bitwise equal (RL-Kernel PR #469,
    Status: the L1 conv batch-invariance protocol)."""
    case = gi.make_inputs(gi.TINY, [1] * 17, 40, seed=6)
    full_out, full_state = _run_rows(oracle, case, np.arange(17))
    rng = np.random.default_rng(0)
    runs = [[r] for r in range(17)] + [list(range(3, 5)), list(range(9, 16))]
    runs.append(list(rng.permutation(17)))
    for rows in runs:
        for perm in (None, np.concatenate([[0], 1 + rng.permutation(39)])):  # 0 stays null
            out, st = _run_rows(oracle, case, np.array(rows), perm)
            for i, r in enumerate(rows):
                assert np.array_equal(out[i], full_out[r])
                s = int(case.slot[r])
                assert np.array_equal(st[s][0], full_state[s][0])
                assert np.array_equal(st[s][1], full_state[s][1])


def test_batch_invariance_check_catches_batch_dependence(oracle):
    """Negative control: a deliberately batch-dependent head recurrence fails the same check."""
    rng = np.random.default_rng(1)
    dk = dv = 32
    rows = [(rng.standard_normal((1, dk)), rng.standard_normal((1, dk)), rng.standard_normal((1, dv)),
             -np.abs(rng.standard_normal(1)), rng.uniform(0, 1, 1), rng.standard_normal((dv, dk)))
            for _ in range(8)]

    def run(batch_rows, fn):
        return [fn(*r) for r in batch_rows]

    def invariant(fn_of_batch):
        full = run(rows, fn_of_batch(len(rows)))
        for i, r in enumerate(rows):
            alone = run([r], fn_of_batch(1))[0]
            if not (np.array_equal(alone[0], full[i][0]) and np.array_equal(alone[1], full[i][1])):
                return False
        return True

    assert invariant(lambda B: oracle.recurrent_head)
    assert not invariant(lambda B: (lambda *a: oracle.recurrent_head_batch_dependent(*a, B)))


# --------------------------------------------------------------------------- bf16 state

def test_bf16_state_is_the_fp64_state_rounded_once(oracle):
    """RL-Kernel PR #469, Summary (state ABI): the state takes its storage dtype only when it is
    written. A bf16-state call equals the full-precision call with the final state rounded
    once (RNE), and identical outputs (read out before the write)."""
    geo = gi.TINY
    case = gi.make_inputs(geo, [5, 3], 6, seed=12)
    pool16 = gi.bf16_bits_to_f32(gi.f32_to_bf16_bits(case.ssm_state)).astype(np.float64)
    conv_a, conv_b = case.conv_state.copy(), case.conv_state.copy()
    ssm_a, ssm_b = pool16.copy(), pool16.copy()
    args = (case.mixed, case.a, case.b, False, case.A_log, case.dt_bias, case.conv_w,
            case.conv_b, 1)
    out_a, _, _ = oracle.layer(*args, conv_a, 0, 0, ssm_a, case.cu_seqlens, case.slot, None,
                               geo.Hk, geo.Hv, geo.dk, geo.dv)
    out_b, _, _ = oracle.layer(*args, conv_b, 0, 0, ssm_b, case.cu_seqlens, case.slot, None,
                               geo.Hk, geo.Hv, geo.dk, geo.dv, state_bf16=True)
    assert np.array_equal(out_a, out_b)
    rounded = bfv(oracle.round_bf16_array(ssm_a.ravel())).reshape(ssm_a.shape)
    assert np.array_equal(ssm_b, rounded)
    touched = sorted(set(int(s) for s in case.slot))
    assert not np.array_equal(ssm_b[touched], pool16[touched])


def test_bf16_state_identity_step_is_exact(oracle):
    """g = 0 and beta = 0 leave S unchanged: a bf16 state round-trips bitwise."""
    geo = gi.Geometry(1, 1, 8, 8)
    rng = np.random.default_rng(4)
    pool = bfv(bf(rng.standard_normal((3, 1, 8, 8)))).copy()
    before = pool.copy()
    mixed = bf(rng.standard_normal((1, geo.D)))
    g = np.zeros((1, 1), np.float32); beta = np.zeros((1, 1), np.float32)
    oracle.decode_step(mixed, g, beta, True, None, None, None, None, 0, None, 0, 0, pool,
                       np.array([2], np.int32), 1, 1, 8, 8, state_bf16=True)
    assert np.array_equal(pool, before)


# --------------------------------------------------------------------------- output gate

def _gate_case(seed, shape=(3, 4, 128)):
    rng = np.random.default_rng(seed)
    o = rng.standard_normal(shape)
    z = gi.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(2.0))
    w = rng.standard_normal(shape[-1]).astype(np.float32)
    return o, z, w


@pytest.mark.parametrize("act", ["silu", "sigmoid"])
@pytest.mark.parametrize("offset", [0.0, 1.0])
def test_gated_rmsnorm_matches_torch_rms_norm_times_gate(oracle, act, offset):
    """RL-Kernel PR #469, Summary by CodeRabbit and Walkthrough (gated RMSNorm with SiLU or
    sigmoid gating and a weight offset): the oracle equals torch's own fp64 rms_norm with weight w + offset, times act(z)."""
    import torch
    o, z, w = _gate_case(1)
    y = oracle.gated_rmsnorm(o, z, w, offset=offset, eps=1e-6, act=act)
    zt = torch.from_numpy(gi.bf16_bits_to_f32(z).astype(np.float64))
    wt = torch.from_numpy(w.astype(np.float64)) + offset
    g = torch.nn.functional.silu(zt) if act == "silu" else torch.sigmoid(zt)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(o), [o.shape[-1]], wt, 1e-6) * g
    assert np.abs(y - ref.numpy()).max() <= 1e-13 * np.abs(ref.numpy()).max()


def test_gated_rmsnorm_closed_forms(oracle):
    """Invariants of y = o / rms(o) * (w + offset) * act(z), eps = 0."""
    o, z, w = _gate_case(2)
    y = oracle.gated_rmsnorm(o, z, w, eps=0.0)
    # scale invariance and odd symmetry in o
    assert np.abs(oracle.gated_rmsnorm(3.7 * o, z, w, eps=0.0) - y).max() <= 1e-13 * np.abs(y).max()
    assert np.array_equal(oracle.gated_rmsnorm(-o, z, w, eps=0.0), -y)
    # the normalised vector has unit rms: mean((y / ((w + off) act(z)))^2) = 1
    zf = gi.bf16_bits_to_f32(z).astype(np.float64)
    silu = zf / (1.0 + np.exp(-zf))
    n = y / (w.astype(np.float64) * silu)
    assert np.allclose(np.mean(n * n, axis=-1), 1.0, rtol=1e-12)
    # a constant head vector c*1 normalises to sign(c)*1
    c = np.full((1, 128), -0.3)
    yc = oracle.gated_rmsnorm(c, z[0, :1], w, eps=0.0)
    assert np.allclose(yc, -(w.astype(np.float64) * silu[0, :1]), rtol=1e-14, atol=0)
    # z = 0: SiLU gate is exactly 0; the sigmoid gate is exactly 1/2
    z0 = np.zeros_like(z)
    assert np.all(oracle.gated_rmsnorm(o, z0, w, act="silu") == 0.0)
    ys = oracle.gated_rmsnorm(o, z0, w, eps=0.0, act="sigmoid")
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True))
    assert np.allclose(ys, 0.5 * o / rms * w.astype(np.float64), rtol=1e-13, atol=0)
    # the weight offset: w = 0 with offset 1 equals w = 1 with offset 0
    ones = np.ones(128, np.float32)
    assert np.array_equal(oracle.gated_rmsnorm(o, z, np.zeros(128, np.float32), offset=1.0),
                          oracle.gated_rmsnorm(o, z, ones, offset=0.0))
    # eps enters under the root: a zero head stays zero, with or without eps (0/0 reads as 0)
    assert np.all(oracle.gated_rmsnorm(np.zeros((1, 128)), z[0, :1], w, eps=1e-6) == 0.0)
    assert np.all(oracle.gated_rmsnorm(np.zeros((1, 128)), z[0, :1], w, eps=0.0) == 0.0)
