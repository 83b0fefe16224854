"""Pins of the hybrid-step oracles (oracle/hybrid_oracle.c) to facts fixed outside the oracle.

Gated DeltaNet decode step (gated delta rule, Yang, Kautz and Hatamizadeh, ICLR 2025):
 - the delta rule's defining property: with no decay (alpha = 1) and a full write (beta = 1), the
   new state maps the (normalised) key to the value exactly, whatever the old state was;
 - the update is rank one along the key: directions orthogonal to k are left alone, and the k
   column becomes (1 - beta) old + beta v (closed form);
 - beta = 0 leaves alpha * S, with alpha from hand-evaluated softplus/exp cases;
 - successive writes with orthonormal keys replace the state's columns one by one;
 - the gated RMS norm on hand-made outputs;
 - the pages' state size: 36 layers x the head layout = 72 MiB.
Gated GQA decode attention:
 - one cached position returns its value; equal scores average the values over pos + 1 rows;
 - a two-position case against the logistic closed form; large scores stay finite;
 - the output gate, the cache append, and the pages' 48 KiB per token / 384 MiB at 8K.
A mutation test plants plausible mistakes in a copy of the C file and checks that these fail.
"""
import math

import numpy as np
import pytest

from int4_routed_expert_05_b300 import synth_hybrid as SH
from oracle import hybrid as H

ALPHA1 = -1000.0   # A_log with exp(A_log) = 0 exactly: alpha = 1
BETA1 = 40.0       # b with sigmoid(b) = 1 exactly in double
BETA0 = -1000.0    # b with sigmoid(b) = 0 exactly
LN3 = math.log(3.0)


def _rng(seed):
    return np.random.default_rng(seed)


def _gdn(S, q, k, v, z=None, a=None, b=None, A_log=None, dt_bias=None, norm_w=None, scale=1.0, eps=1e-6):
    Hv, dv, dk = S.shape
    z = np.zeros((Hv, dv)) if z is None else z
    a = np.zeros(Hv) if a is None else np.broadcast_to(a, (Hv,))
    b = np.full(Hv, BETA1) if b is None else np.broadcast_to(b, (Hv,))
    A_log = np.full(Hv, ALPHA1) if A_log is None else np.broadcast_to(A_log, (Hv,))
    dt_bias = np.zeros(Hv) if dt_bias is None else np.broadcast_to(dt_bias, (Hv,))
    norm_w = np.ones(dv) if norm_w is None else norm_w
    return H.gdn_step(S, q, k, v, z, a, b, A_log, dt_bias, norm_w, scale, eps_l2=0.0, eps=eps)


# ---------------------------------------------------------------- Gated DeltaNet


def test_gates_closed_form():
    # softplus(0) = ln 2, A = e^0: alpha = 1/2; softplus(ln(e - 1)) = 1, A = 2: alpha = e^-2;
    # sigmoid(+-ln 3) = 3/4, 1/4
    alpha, beta = H.gdn_gates([0.0, 0.0, 0.0], [LN3, -LN3, 0.0], [0.0, math.log(2.0), 0.0],
                              [0.0, math.log(math.e - 1.0), 50.0])
    assert alpha[0] == pytest.approx(0.5, rel=1e-15)
    assert alpha[1] == pytest.approx(math.exp(-2.0), rel=1e-14)
    assert alpha[2] == pytest.approx(math.exp(-50.0), rel=1e-13)  # softplus(50) = 50 + 2e-22
    assert beta[0] == pytest.approx(0.75, rel=1e-15)
    assert beta[1] == pytest.approx(0.25, rel=1e-15)
    assert beta[2] == 0.5


@pytest.mark.parametrize("Hk,Hv,dk,dv", [(2, 4, 8, 8), (1, 3, 16, 6), (4, 4, 5, 9)])
def test_write_then_read_returns_value(Hk, Hv, dk, dv):
    # alpha = 1, beta = 1, q = k: S_t k^ = v exactly, so o = v for any old state
    r = _rng(1)
    S = r.normal(size=(Hv, dv, dk))
    k = r.normal(size=(Hk, dk))
    v = r.normal(size=(Hv, dv))
    S1, o, _ = _gdn(S, k, k, v)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)
    # and the state differs from the old one only along k (rank-one change)
    for h in range(Hv):
        assert np.linalg.matrix_rank(S1[h] - S[h], tol=1e-10) <= 1


def test_orthogonal_directions_untouched_and_key_column_closed_form():
    # k = 2 e_0 (normalised to e_0), beta = 3/4, alpha = 1: columns 1.. stay; column 0 becomes
    # (1 - beta) S[:, 0] + beta v. Reading with q = e_1 gives scale * S[:, 1].
    r = _rng(2)
    Hk, Hv, dk, dv = 1, 2, 6, 5
    S = r.normal(size=(Hv, dv, dk))
    k = np.zeros((Hk, dk)); k[0, 0] = 2.0
    q = np.zeros((Hk, dk)); q[0, 1] = 3.0
    v = r.normal(size=(Hv, dv))
    S1, o, _ = _gdn(S, q, k, v, b=LN3, scale=0.5)
    np.testing.assert_allclose(S1[:, :, 1:], S[:, :, 1:], rtol=0, atol=1e-14)
    np.testing.assert_allclose(S1[:, :, 0], 0.25 * S[:, :, 0] + 0.75 * v, rtol=0, atol=1e-14)
    np.testing.assert_allclose(o, 0.5 * S[:, :, 1], rtol=0, atol=1e-14)


def test_decay_only_closed_form():
    # beta = 0: S_t = alpha S. Head 0: A = 1, softplus(0 + ln(e - 1)) = 1 -> alpha = 1/e.
    # Head 1: A = 2, a + dt_bias = 0 -> alpha = exp(-2 ln 2) = 1/4.
    r = _rng(3)
    S = r.normal(size=(2, 4, 4))
    q, k = r.normal(size=(1, 4)), r.normal(size=(1, 4))
    v = r.normal(size=(2, 4))
    dt = np.array([math.log(math.e - 1.0), 0.0])
    S1, _, _ = _gdn(S, q, k, v, a=np.zeros(2), b=BETA0, A_log=np.array([0.0, math.log(2.0)]), dt_bias=dt)
    np.testing.assert_allclose(S1[0], S[0] / math.e, rtol=1e-14, atol=0)
    np.testing.assert_allclose(S1[1], S[1] / 4.0, rtol=1e-14, atol=0)


def test_first_write_from_zero_state_uses_the_grouped_key_head():
    # S = 0, alpha = 1, beta = 3/4: S_t = beta v k^ k^ (value head h uses key head h // (Hv / Hk)).
    # With q = k and scale 0.5: o = 0.5 beta v.
    r = _rng(4)
    Hk, Hv, dk, dv = 2, 4, 8, 8
    k = r.normal(size=(Hk, dk))
    v = r.normal(size=(Hv, dv))
    S1, o, _ = _gdn(np.zeros((Hv, dv, dk)), k, k, v, b=LN3, scale=0.5)
    for h in range(Hv):
        kn = k[h // 2] / np.linalg.norm(k[h // 2])
        np.testing.assert_allclose(S1[h], 0.75 * np.outer(v[h], kn), rtol=0, atol=1e-14)
    np.testing.assert_allclose(o, 0.375 * v, rtol=0, atol=1e-14)


def test_successive_orthonormal_writes_replace_columns():
    # alpha = 1, beta = 1, keys e_0, e_1, e_2 in turn: column t of S becomes v_t, the rest stay
    r = _rng(5)
    dk, dv = 5, 4
    S0 = r.normal(size=(1, dv, dk))
    S = S0
    vs = r.normal(size=(3, dv))
    for t in range(3):
        k = np.zeros((1, dk)); k[0, t] = 1.0
        S, _, _ = _gdn(S, k, k, vs[t][None])
    for t in range(3):
        np.testing.assert_allclose(S[0, :, t], vs[t], rtol=0, atol=1e-14)
    np.testing.assert_allclose(S[0, :, 3:], S0[0, :, 3:], rtol=0, atol=0)


def test_gated_norm_closed_form():
    # o = 0.375 * c for every row (constant head output): RMS norm gives sign(c) (eps = 0), then
    # norm_w[r] * silu(z), silu(ln 3) = (3/4) ln 3. With eps = (0.375 c)^2 the norm is 1/sqrt 2.
    dk, dv = 4, 6
    k = np.zeros((1, dk)); k[0, 0] = 1.0
    c = -2.0
    v = np.full((1, dv), c)
    w = np.arange(1, dv + 1, dtype=np.float64)
    z = np.full((1, dv), LN3)
    silu = 0.75 * LN3
    _, o, y = _gdn(np.zeros((1, dv, dk)), k, k, v, z=z, b=LN3, norm_w=w, scale=0.5, eps=0.0)
    np.testing.assert_allclose(o, 0.375 * v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(y[0], -w * silu, rtol=1e-14)
    _, _, y = _gdn(np.zeros((1, dv, dk)), k, k, v, z=z, b=LN3, norm_w=w, scale=0.5, eps=(0.375 * c) ** 2)
    np.testing.assert_allclose(y[0], -w * silu / math.sqrt(2.0), rtol=1e-14)


def test_delta_rule_row_form_on_random_inputs():
    # the same update written the other way round, row by row:
    # S_t = alpha S + beta (v - alpha S k^) k^T, o = S_t q^ (q^ = scale q / |q|)
    r = _rng(6)
    Hk, Hv, dk, dv = 2, 4, 16, 12
    S = r.normal(size=(Hv, dv, dk))
    q, k = r.normal(size=(Hk, dk)), r.normal(size=(Hk, dk))
    v, a, b = r.normal(size=(Hv, dv)), r.normal(size=Hv), r.normal(size=Hv)
    A_log, dt = np.log(r.uniform(1, 16, Hv)), r.normal(size=Hv)
    alpha, beta = H.gdn_gates(a, b, A_log, dt)
    S1, o, _ = _gdn(S, q, k, v, a=a, b=b, A_log=A_log, dt_bias=dt, scale=0.25)
    for h in range(Hv):
        kn = k[h // 2] / np.linalg.norm(k[h // 2])
        qn = 0.25 * q[h // 2] / np.linalg.norm(q[h // 2])
        u = alpha[h] * S[h] @ kn
        want = alpha[h] * S[h] + beta[h] * np.outer(v[h] - u, kn)
        np.testing.assert_allclose(S1[h], want, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(o[h], want @ qn, rtol=1e-12, atol=1e-13)


def test_state_size_matches_the_pages():
    # 36 DeltaNet layers with a fixed state of about 72 MiB in all (fp32)
    assert SH.GDN80_LAYERS * SH.GDN80.state_floats() * 4 == 72 * 2 ** 20
    assert SH.GDN80_LAYERS + SH.GQA80_LAYERS == 48


# ---------------------------------------------------------------- gated GQA


def _gqa(Kc, Vc, pos, q, k, v, gate=None, scale=1.0):
    gate = np.full(q.shape, 40.0) if gate is None else gate   # sigmoid(40) = 1 exactly
    return H.gqa_step(Kc, Vc, pos, q, k, v, gate, scale)


def test_first_position_returns_its_value():
    r = _rng(11)
    Hq, Hkv, D, L = 4, 2, 8, 5
    Kc, Vc = r.normal(size=(Hkv, L, D)), r.normal(size=(Hkv, L, D))  # stale rows must not matter
    q, k, v = r.normal(size=(Hq, D)), r.normal(size=(Hkv, D)), r.normal(size=(Hkv, D))
    _, _, o, y = _gqa(Kc, Vc, 0, q, k, v)
    for h in range(Hq):
        np.testing.assert_allclose(o[h], v[h // 2], rtol=0, atol=1e-15)
    np.testing.assert_allclose(y, o, rtol=0, atol=0)


def test_equal_scores_average_the_values_including_the_new_one():
    r = _rng(12)
    Hq, Hkv, D, L, pos = 4, 2, 6, 9, 5
    Kc, Vc = r.normal(size=(Hkv, L, D)), r.normal(size=(Hkv, L, D))
    q = np.zeros((Hq, D))
    k, v = r.normal(size=(Hkv, D)), r.normal(size=(Hkv, D))
    _, Vn, o, _ = _gqa(Kc, Vc, pos, q, k, v)
    for h in range(Hq):
        g = h // 2
        want = (Vc[g, :pos].sum(0) + v[g]) / (pos + 1)
        np.testing.assert_allclose(o[h], want, rtol=0, atol=1e-14)


def test_two_positions_logistic_closed_form():
    # K_0 = 3 e_0 (cached), k = 2 e_1 (new); q = (1, 4, 0, 0), scale 1/2: s0 = 1.5, s1 = 4,
    # p1 = 1 / (1 + exp(s0 - s1)); o = p0 V_0 + p1 v
    D = 4
    Kc, Vc = np.zeros((1, 3, D)), np.zeros((1, 3, D))
    Kc[0, 0, 0] = 3.0
    Vc[0, 0] = [1.0, -2.0, 0.5, 4.0]
    q = np.array([[1.0, 4.0, 0.0, 0.0]])
    k = np.array([[0.0, 2.0, 0.0, 0.0]])
    v = np.array([[-1.0, 3.0, 2.0, 0.0]])
    _, _, o, _ = _gqa(Kc, Vc, 1, q, k, v, scale=0.5)
    p1 = 1.0 / (1.0 + math.exp(1.5 - 4.0))
    np.testing.assert_allclose(o[0], (1 - p1) * Vc[0, 0] + p1 * v[0], rtol=1e-15, atol=1e-15)


def test_large_scores_stay_finite():
    # scores 1000 and 1000 - ln 3: weights 3/4 and 1/4 (no overflow)
    D = 2
    Kc, Vc = np.zeros((1, 2, D)), np.zeros((1, 2, D))
    Kc[0, 0] = [1000.0, 0.0]
    Vc[0, 0] = [4.0, 0.0]
    q = np.array([[1.0, 1.0]])
    k = np.array([[0.0, 1000.0 - LN3]])
    v = np.array([[0.0, 8.0]])
    _, _, o, _ = _gqa(Kc, Vc, 1, q, k, v)
    np.testing.assert_allclose(o[0], [3.0, 2.0], rtol=1e-12)


def test_output_gate_and_cache_append():
    r = _rng(13)
    Hq, Hkv, D, L, pos = 2, 1, 4, 6, 3
    Kc, Vc = r.normal(size=(Hkv, L, D)), r.normal(size=(Hkv, L, D))
    q, k, v = r.normal(size=(Hq, D)), r.normal(size=(Hkv, D)), r.normal(size=(Hkv, D))
    gate = np.array([[LN3] * D, [-LN3] * D])
    Kn, Vn, o, y = _gqa(Kc, Vc, pos, q, k, v, gate=gate)
    np.testing.assert_allclose(y[0], 0.75 * o[0], rtol=1e-15)
    np.testing.assert_allclose(y[1], 0.25 * o[1], rtol=1e-15)
    np.testing.assert_array_equal(Kn[:, pos], k)
    np.testing.assert_array_equal(Vn[:, pos], v)
    keep = [t for t in range(L) if t != pos]
    np.testing.assert_array_equal(Kn[:, keep], Kc[:, keep])
    np.testing.assert_array_equal(Vn[:, keep], Vc[:, keep])


def test_kv_size_matches_the_pages():
    # 12 attention layers, K and V in fp32: at least 48 KiB per token, about 384 MiB at 8K
    per_token = SH.GQA80_LAYERS * 2 * SH.GQA80.n_kv_heads * SH.GQA80.head_dim * 4
    assert per_token == 48 * 1024
    assert per_token * 8192 == 384 * 2 ** 20
