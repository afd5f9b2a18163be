"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

None of these re-types the oracle's loop: each checks a closed form, an
invariant, a special case that reduces to a textbook result, or a brute-force
hand expansion.  Together they are chosen so that a plausible slip in the
oracle (decay applied after the read, read-out before the write, eps outside
the root, a transposed state, a wrong sign in the residual, a dropped decay
factor in the chunked form) fails at least one of them.

Sources: nnterp "kimi_linear" page (definition of Kimi Delta Attention: the
state decays channel by channel before each delta-rule update; L2 norm of q
and k in the kernel); Ascend model file, ``_l2_normalize`` (eps 1e-6 on the
sum of squares, inside the root) and ``_torch_chunk_kda`` (scale 1/sqrt(K) on
the normalised query, chunked form, zero padding of the tail).
"""
import numpy as np
import pytest

import oracle

EPS = 1e-6


def _rand(rng, T, H, K, V, g_lo=-0.3, g_hi=-0.01):
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    g = rng.uniform(g_lo, g_hi, (T, H, K))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, beta


def _unit(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + EPS)


# ---- L2 norm and scale ------------------------------------------------------

def test_eps_inside_root_on_sum_of_squares():
    # q = 1e-3 e_1, k = e_1, S0 = 0, one token, beta = 1, g = 0:
    #   k_hat = 1/sqrt(1 + 1e-6) e_1, q_hat = 1e-3/sqrt(1e-6 + 1e-6) e_1 = e_1/sqrt(2)
    #   o = scale * beta * (k_hat . q_hat) * v
    K, V = 4, 3
    q = np.zeros((1, 1, K)); q[0, 0, 0] = 1e-3
    k = np.zeros((1, 1, K)); k[0, 0, 0] = 1.0
    v = np.array([[[1.0, -2.0, 0.5]]])
    g = np.zeros((1, 1, K)); beta = np.ones((1, 1))
    o, S = oracle.recurrence(q, k, v, g, beta, scale=0.5)
    kq = (1 / np.sqrt(1 + 1e-6)) * (1 / np.sqrt(2.0))
    np.testing.assert_allclose(o[0, 0], 0.5 * kq * v[0, 0], rtol=1e-13)
    # eps outside the root would give ~0.999 instead of 1/sqrt(2)
    assert abs(o[0, 0, 0] / (0.5 * v[0, 0, 0]) - 0.70710643) < 1e-6


def test_default_scale_is_inverse_sqrt_K():
    rng = np.random.default_rng(1)
    q, k, v, g, b = _rand(rng, 5, 1, 16, 3)
    o1, _ = oracle.recurrence(q, k, v, g, b)
    o2, _ = oracle.recurrence(q, k, v, g, b, scale=0.25)
    np.testing.assert_allclose(o1, o2, rtol=1e-14)


# ---- closed forms -----------------------------------------------------------

def test_beta_zero_is_pure_channel_decay():
    # beta = 0: no writes. S_T = diag(exp(sum_t g_t)) S0 and
    # o_t = scale * (diag(exp(G_t)) S0)^T q_hat_t, G_t = sum_{s<=t} g_s.
    rng = np.random.default_rng(2)
    T, H, K, V = 37, 2, 5, 3
    q, k, v, g, _ = _rand(rng, T, H, K, V)
    beta = np.zeros((T, H))
    s0 = rng.standard_normal((1, H, K, V))
    o, S = oracle.recurrence(q, k, v, g, beta, initial_state=s0, scale=0.7)
    G = np.cumsum(g, axis=0)                          # [T, H, K]
    np.testing.assert_allclose(S[0], np.exp(G[-1])[:, :, None] * s0[0], rtol=1e-12)
    qh = _unit(q)
    for t in range(T):
        for h in range(H):
            expect = 0.7 * (np.exp(G[t, h])[:, None] * s0[0, h]).T @ qh[t, h]
            np.testing.assert_allclose(o[t, h], expect, rtol=1e-11, atol=1e-14)


def test_single_token_from_zero_is_one_delta_write():
    # S0 = 0, one token: the decay acts on zero, u = beta v, S = beta k_hat v^T,
    # o = scale * beta (k_hat . q_hat) v.  K != V catches a transposed state.
    rng = np.random.default_rng(3)
    K, V = 6, 4
    q, k, v, g, beta = _rand(rng, 1, 1, K, V)
    o, S = oracle.recurrence(q, k, v, g, beta, scale=0.3)
    kh, qh = _unit(k[0, 0]), _unit(q[0, 0])
    np.testing.assert_allclose(S[0, 0], beta[0, 0] * np.outer(kh, v[0, 0]), rtol=1e-13)
    np.testing.assert_allclose(o[0, 0], 0.3 * beta[0, 0] * (kh @ qh) * v[0, 0], rtol=1e-12)


def test_associative_recall_orthonormal_keys():
    # beta = 1, g = 0, S0 = 0, keys orthonormal: every write stores v_i exactly
    # under k_i.  With unit keys k_hat = c k, c^2 = 1/(1+eps); querying with
    # q_t = k_t gives o_t = scale * c^2 * v_t and S_T^T k_i = c * v_i.
    rng = np.random.default_rng(4)
    K, V, T = 16, 7, 12
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Qm[:T]                                  # T orthonormal rows
    k = keys[:, None, :]
    q = k.copy()
    v = rng.standard_normal((T, 1, V))
    g = np.zeros((T, 1, K)); beta = np.ones((T, 1))
    o, S = oracle.recurrence(q, k, v, g, beta, scale=0.2)
    c2 = 1.0 / (1.0 + EPS)
    np.testing.assert_allclose(o[:, 0], 0.2 * c2 * v[:, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(S[0, 0].T @ keys.T, np.sqrt(c2) * v[:, 0].T, rtol=1e-10, atol=1e-12)


def test_two_tokens_hand_expanded_K3_V2():
    # Brute force, T = 2, K = 3, V = 2, S0 = 0, written out by hand:
    #   S1 = b1 k1 v1^T,   o1 = s b1 (k1.q1) v1
    #   D  = diag(exp(g2)),  u2 = b2 (v2 - b1 (k1^T D k2) v1)
    #   o2 = s [ b1 (k1^T D q2) v1 + (k2.q2) u2 ]      (hats on q, k)
    q = np.array([[[0.3, -1.2, 0.8]], [[1.1, 0.4, -0.2]]])
    k = np.array([[[-0.5, 0.9, 1.3]], [[0.7, 0.7, -0.6]]])
    v = np.array([[[2.0, -1.0]], [[0.5, 3.0]]])
    g = np.array([[[-0.1, -0.2, -0.3]], [[-0.4, -0.05, -1.5]]])
    b = np.array([[0.6], [0.9]])
    s = 0.45
    o, S = oracle.recurrence(q, k, v, g, b, scale=s)
    k1, k2 = _unit(k[0, 0]), _unit(k[1, 0])
    q1, q2 = _unit(q[0, 0]), _unit(q[1, 0])
    v1, v2 = v[0, 0], v[1, 0]
    b1, b2 = b[0, 0], b[1, 0]
    d = np.exp(g[1, 0])
    o1 = s * b1 * (k1 @ q1) * v1
    u2 = b2 * (v2 - b1 * np.sum(k1 * d * k2) * v1)
    o2 = s * (b1 * np.sum(k1 * d * q2) * v1 + (k2 @ q2) * u2)
    S2 = b1 * np.outer(d * k1, v1) + np.outer(k2, u2)
    np.testing.assert_allclose(o[0, 0], o1, rtol=1e-13)
    np.testing.assert_allclose(o[1, 0], o2, rtol=1e-13)
    np.testing.assert_allclose(S[0, 0], S2, rtol=1e-13)


# ---- invariants -------------------------------------------------------------

def test_joint_linearity_in_values_and_initial_state():
    rng = np.random.default_rng(5)
    T, H, K, V = 29, 2, 8, 5
    q, k, v1, g, b = _rand(rng, T, H, K, V)
    v2 = rng.standard_normal((T, H, V))
    s1 = rng.standard_normal((1, H, K, V)); s2 = rng.standard_normal((1, H, K, V))
    a = -1.7
    o1, f1 = oracle.recurrence(q, k, v1, g, b, initial_state=s1)
    o2, f2 = oracle.recurrence(q, k, v2, g, b, initial_state=s2)
    o3, f3 = oracle.recurrence(q, k, v1 + a * v2, g, b, initial_state=s1 + a * s2)
    np.testing.assert_allclose(o3, o1 + a * o2, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(f3, f1 + a * f2, rtol=1e-10, atol=1e-12)


def test_value_columns_and_key_channels_are_equivariant():
    rng = np.random.default_rng(6)
    T, H, K, V = 23, 1, 7, 6
    q, k, v, g, b = _rand(rng, T, H, K, V)
    s0 = rng.standard_normal((1, H, K, V))
    o, S = oracle.recurrence(q, k, v, g, b, initial_state=s0)
    pv = rng.permutation(V)
    o2, S2 = oracle.recurrence(q, k, v[..., pv], g, b, initial_state=s0[..., pv])
    np.testing.assert_allclose(o2, o[..., pv], rtol=1e-12)
    np.testing.assert_allclose(S2, S[..., pv], rtol=1e-12)
    pk = rng.permutation(K)
    o3, S3 = oracle.recurrence(q[..., pk], k[..., pk], v, g[..., pk], b,
                               initial_state=s0[:, :, pk, :])
    np.testing.assert_allclose(o3, o, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(S3, S[:, :, pk, :], rtol=1e-11, atol=1e-13)


def test_heads_and_sequences_are_independent():
    rng = np.random.default_rng(7)
    lens = [5, 0, 17, 9]
    T, H, K, V = sum(lens), 3, 6, 4
    q, k, v, g, b = _rand(rng, T, H, K, V)
    s0 = rng.standard_normal((len(lens), H, K, V))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S = oracle.recurrence(q, k, v, g, b, cu_seqlens=cu, initial_state=s0)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        for h in range(H):
            oh, Sh = oracle.recurrence(q[sl, h:h + 1], k[sl, h:h + 1], v[sl, h:h + 1],
                                       g[sl, h:h + 1], b[sl, h:h + 1],
                                       initial_state=s0[n:n + 1, h:h + 1])
            np.testing.assert_allclose(o[sl, h:h + 1], oh, rtol=1e-13)
            np.testing.assert_allclose(S[n, h], Sh[0, 0], rtol=1e-13)
    # an empty sequence hands back its initial state unchanged
    np.testing.assert_array_equal(S[1], s0[1])


@pytest.mark.parametrize("split", [1, 63, 64, 65, 100])
def test_split_and_handoff(split):
    rng = np.random.default_rng(8)
    T, H, K, V = 130, 2, 8, 8
    q, k, v, g, b = _rand(rng, T, H, K, V)
    s0 = rng.standard_normal((1, H, K, V))
    o, S = oracle.recurrence(q, k, v, g, b, initial_state=s0)
    a, c = slice(0, split), slice(split, T)
    oa, Sa = oracle.recurrence(q[a], k[a], v[a], g[a], b[a], initial_state=s0)
    ob, Sb = oracle.recurrence(q[c], k[c], v[c], g[c], b[c], initial_state=Sa)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Sb, S, rtol=1e-12, atol=1e-13)


def test_contraction_without_inputs():
    # v = 0, g <= 0, beta in [0, 1], |k_hat| < 1: each step is
    # S <- (I - beta k k^T) D S, a product of contractions in Frobenius norm.
    rng = np.random.default_rng(9)
    T, K, V = 40, 8, 5
    q, k, _, g, b = _rand(rng, T, 1, K, V, g_lo=-0.2, g_hi=0.0)
    v = np.zeros((T, 1, V))
    S = rng.standard_normal((1, 1, K, V))
    prev = np.linalg.norm(S)
    for t in range(T):
        _, S = oracle.recurrence(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], b[t:t + 1],
                                 initial_state=S)
        cur = np.linalg.norm(S)
        assert cur <= prev * (1 + 1e-14)
        prev = cur


def test_query_and_key_magnitude_only_enter_through_eps():
    rng = np.random.default_rng(10)
    q, k, v, g, b = _rand(rng, 20, 2, 16, 4)
    o, S = oracle.recurrence(q, k, v, g, b)
    o2, S2 = oracle.recurrence(3.0 * q, 0.5 * k, v, g, b)
    # |q|^2, |k|^2 ~ 16 >> eps: relative change O(eps / |x|^2)
    np.testing.assert_allclose(o2, o, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(S2, S, rtol=2e-6, atol=1e-7)


# ---- the chunked form against the recurrence --------------------------------

@pytest.mark.parametrize("chunk", [1, 4, 16, 64])
def test_chunked_form_equals_recurrence(chunk):
    rng = np.random.default_rng(11 + chunk)
    T, H, K, V = 77, 2, 8, 6          # ragged tail for every chunk size
    q, k, v, g, b = _rand(rng, T, H, K, V, g_lo=-0.5, g_hi=-0.001)
    s0 = rng.standard_normal((H, K, V))
    o, S = oracle.recurrence(q, k, v, g, b, initial_state=s0[None], scale=0.35)
    oc, Sc = oracle.chunked_form(q, k, v, g, b, initial_state=s0, chunk=chunk, scale=0.35)
    np.testing.assert_allclose(oc, o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(Sc, S[0], rtol=1e-11, atol=1e-12)


def test_chunked_form_strong_decay():
    # per-token decays down to -3 (the long-prefill mix): exact pairwise exps in fp64
    rng = np.random.default_rng(12)
    T, H, K, V = 70, 1, 8, 4
    q, k, v, g, b = _rand(rng, T, H, K, V)
    strong = rng.uniform(-3, -1, g.shape)
    g = np.where(rng.uniform(size=g.shape) < 0.3, strong, g)
    o, S = oracle.recurrence(q, k, v, g, b)
    oc, Sc = oracle.chunked_form(q, k, v, g, b, chunk=64)
    np.testing.assert_allclose(oc, o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(Sc, S[0], rtol=1e-10, atol=1e-12)


# ---- the decode step --------------------------------------------------------

def test_step_advances_only_the_picked_slots():
    rng = np.random.default_rng(13)
    N, H, K, V, slots = 3, 2, 6, 5, 7
    q, k, v, g, b = _rand(rng, N, H, K, V)
    pool = rng.standard_normal((slots, H, K, V))
    idx = np.array([5, 0, 3])
    o, new = oracle.step(q, k, v, g, b, pool, state_indices=idx)
    untouched = [s for s in range(slots) if s not in idx]
    np.testing.assert_array_equal(new[untouched], pool[untouched])
    for n in range(N):
        on, Sn = oracle.recurrence(q[n:n + 1], k[n:n + 1], v[n:n + 1], g[n:n + 1], b[n:n + 1],
                                   initial_state=pool[idx[n]][None])
        np.testing.assert_allclose(o[n], on[0], rtol=1e-13)
        np.testing.assert_allclose(new[idx[n]], Sn[0], rtol=1e-13)


def test_steps_compose_to_the_sequence_recurrence():
    rng = np.random.default_rng(14)
    T, H, K, V = 9, 2, 5, 4
    q, k, v, g, b = _rand(rng, T, H, K, V)
    pool = rng.standard_normal((2, H, K, V))
    o_seq, S_seq = oracle.recurrence(q, k, v, g, b, initial_state=pool[1][None])
    p = pool
    for t in range(T):
        o_t, p = oracle.step(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], b[t:t + 1], p,
                             state_indices=[1])
        np.testing.assert_allclose(o_t[0], o_seq[t], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(p[1], S_seq[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(p[0], pool[0])


# ---------------------------------------------------------------------------
# gate activation (Ascend model file, _prefill_torch_kda / decode branch)
# ---------------------------------------------------------------------------

def _gate_params(rng, H, K):
    a_log = np.log(rng.uniform(1.0, 16.0, H))   # the model's A_log initialisation
    dt_bias = rng.standard_normal((H, K))
    return a_log, dt_bias


def test_gate_at_zero_input_is_log2_or_half_the_bound():
    """x = raw + dt_bias = 0: softplus(0) = log 2, sigmoid(0) = 1/2."""
    rng = np.random.default_rng(21)
    T, H, K = 3, 4, 5
    a_log, dt_bias = _gate_params(rng, H, K)
    raw = np.broadcast_to(-dt_bias, (T, H, K))
    g, beta = oracle.gate_activation(raw, np.zeros((T, H)), a_log, dt_bias)
    np.testing.assert_allclose(g, np.broadcast_to(-np.exp(a_log)[None, :, None] * np.log(2.0), g.shape),
                               rtol=1e-15)
    np.testing.assert_array_equal(beta, 0.5)
    g_lb, _ = oracle.gate_activation(raw, np.zeros((T, H)), a_log, dt_bias, lower_bound=-5.0)
    np.testing.assert_allclose(g_lb, -2.5, rtol=1e-15)


def test_gate_softplus_and_sigmoid_reflection_identities():
    """softplus(x) - softplus(-x) = x  and  sigmoid(x) + sigmoid(-x) = 1, through
    the full activation: g(x) - g(-x) = -exp(A_log) x ; g_lb(x) + g_lb(-x) = lb ;
    beta(r) + beta(-r) = 1."""
    rng = np.random.default_rng(22)
    T, H, K = 6, 3, 7
    a_log, dt_bias = _gate_params(rng, H, K)
    x = rng.standard_normal((T, H, K)) * 4.0
    r = rng.standard_normal((T, H)) * 6.0
    g_p, b_p = oracle.gate_activation(x - dt_bias, r, a_log, dt_bias)
    g_m, b_m = oracle.gate_activation(-x - dt_bias, -r, a_log, dt_bias)
    np.testing.assert_allclose(g_p - g_m, -np.exp(a_log)[None, :, None] * x, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b_p + b_m, 1.0, rtol=0, atol=1e-15)
    lb = -3.5
    gl_p, _ = oracle.gate_activation(x - dt_bias, r, a_log, dt_bias, lower_bound=lb)
    gl_m, _ = oracle.gate_activation(-x - dt_bias, r, a_log, dt_bias, lower_bound=lb)
    np.testing.assert_allclose(gl_p + gl_m, lb, rtol=1e-14)


def test_gate_limits_and_ranges():
    """Large positive x: softplus(x) = x to fp64 rounding; large negative x:
    softplus(x) = exp(x) (first order); the lower-bounded gate lies in (lb, 0),
    the softplus gate below 0, beta in (0, 1); per-head scale exp(A_log) and
    per-(head, channel) bias are applied where they belong."""
    H, K = 2, 3
    a_log = np.log(np.array([2.0, 8.0]))
    dt_bias = np.array([[0.0, 1.0, -1.0], [0.5, 0.0, 0.0]])
    big = np.full((1, H, K), 60.0) - dt_bias
    g, _ = oracle.gate_activation(big, np.zeros((1, H)), a_log, dt_bias)
    np.testing.assert_allclose(g[0], -np.exp(a_log)[:, None] * 60.0 * np.ones((H, K)), rtol=1e-15)
    small = np.full((1, H, K), -40.0) - dt_bias
    g, _ = oracle.gate_activation(small, np.zeros((1, H)), a_log, dt_bias)
    np.testing.assert_allclose(g[0], -np.exp(a_log)[:, None] * np.exp(-40.0) * np.ones((H, K)), rtol=1e-12)
    rng = np.random.default_rng(23)
    raw = rng.standard_normal((50, H, K)) * 5
    rb = rng.standard_normal((50, H)) * 5
    g_lb, beta = oracle.gate_activation(raw, rb, a_log, dt_bias, lower_bound=-5.0)
    assert np.all(g_lb >= -5.0) and np.all(g_lb < 0.0)  # (lb, 0); lb itself once fp64 saturates
    mid = np.abs(raw) < 0.2
    assert np.all(g_lb[mid] > -5.0)
    assert np.all(beta > 0.0) and np.all(beta < 1.0)
    g_sp, _ = oracle.gate_activation(raw, rb, a_log, dt_bias)
    assert np.all(g_sp < 0.0)
    # channel 1 of head 0 has bias +1: the same raw value gives the input x + 1
    raw1 = np.zeros((1, H, K))
    g1, _ = oracle.gate_activation(raw1, np.zeros((1, H)), a_log, dt_bias)
    np.testing.assert_allclose(g1[0, 0, 1], -np.exp(a_log[0]) * np.log1p(np.exp(1.0)), rtol=1e-15)
    np.testing.assert_allclose(g1[0, 1, 0], -np.exp(a_log[1]) * np.log1p(np.exp(0.5)), rtol=1e-15)


# ---------------------------------------------------------------------------
# output epilogue (Ascend model file, KimiDeltaAttention._project_out)
# ---------------------------------------------------------------------------

def test_output_norm_of_a_constant_row_and_gate_zero():
    """A row of equal entries c: RMS = |c| (eps = 0), so out = sign(c) w sigmoid(gate);
    gate = 0 halves it."""
    V = 8
    w = np.linspace(0.5, 2.0, V)
    o = np.full((1, 1, V), -3.0)
    out = oracle.output_gate_norm(o, np.zeros((1, 1, V)), w, 0.0)
    np.testing.assert_allclose(out[0, 0], -0.5 * w, rtol=1e-15)


def test_output_norm_scale_invariance_and_unit_rms():
    """out is unchanged when a row is scaled (eps -> 0); with weight 1 and a
    large gate the row has unit RMS; eps enters as mean(o^2) + eps."""
    rng = np.random.default_rng(31)
    T, H, V = 5, 3, 16
    o = rng.standard_normal((T, H, V))
    gate = rng.standard_normal((T, H, V))
    w = rng.uniform(0.5, 1.5, V)
    a = oracle.output_gate_norm(o, gate, w, 0.0)
    b = oracle.output_gate_norm(7.5 * o, gate, w, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-13)
    u = oracle.output_gate_norm(o, np.full((T, H, V), 60.0), np.ones(V), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(u * u, axis=-1)), 1.0, rtol=1e-13)
    # eps: a row of ones with eps = 3 has RMS factor 1 / sqrt(1 + 3) = 1/2
    e = oracle.output_gate_norm(np.ones((1, 1, V)), np.full((1, 1, V), 60.0), np.ones(V), 3.0)
    np.testing.assert_allclose(e, 0.5, rtol=1e-13)


def test_output_norm_rows_are_independent():
    """Each (token, head) row is normalised on its own: changing one row leaves
    every other output untouched."""
    rng = np.random.default_rng(32)
    o = rng.standard_normal((4, 2, 8))
    gate = rng.standard_normal((4, 2, 8))
    w = np.ones(8)
    a = oracle.output_gate_norm(o, gate, w, 1e-6)
    o2 = o.copy()
    o2[2, 1] *= -4.0
    b = oracle.output_gate_norm(o2, gate, w, 1e-6)
    mask = np.ones((4, 2), bool)
    mask[2, 1] = False
    np.testing.assert_array_equal(a[mask], b[mask])


# ---------------------------------------------------------------------------
# speculative (multi-token) decode
# ---------------------------------------------------------------------------

def _multi_inputs(rng, N, S, H, K, V):
    q = rng.standard_normal((N, S, H, K))
    k = rng.standard_normal((N, S, H, K))
    v = rng.standard_normal((N, S, H, V))
    g = -rng.uniform(0.01, 0.5, (N, S, H, K))
    b = rng.uniform(0.1, 0.9, (N, S, H))
    return q, k, v, g, b


def test_multi_step_with_one_token_is_the_step():
    rng = np.random.default_rng(41)
    N, H, K, V, slots = 3, 2, 6, 5, 6
    q, k, v, g, b = _multi_inputs(rng, N, 1, H, K, V)
    pool = rng.standard_normal((slots, H, K, V))
    idx = np.array([[4], [0], [2]])
    o, new = oracle.multi_step(q, k, v, g, b, pool, idx)
    o1, new1 = oracle.step(q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0], pool, state_indices=idx[:, 0])
    np.testing.assert_allclose(o[:, 0], o1, rtol=1e-13)
    np.testing.assert_allclose(new, new1, rtol=1e-13)


def test_multi_step_writes_every_prefix_state_and_reads_the_accepted_slot():
    """Slot idx[n, t] receives the recurrence over tokens 0..t, started from
    slot idx[n, a - 1]; outputs are the recurrence's; other slots untouched."""
    rng = np.random.default_rng(42)
    N, S, H, K, V, slots = 2, 4, 2, 5, 3, 12
    q, k, v, g, b = _multi_inputs(rng, N, S, H, K, V)
    pool = rng.standard_normal((slots, H, K, V))
    idx = np.array([[3, 7, 1, 9], [10, 2, 5, 0]])
    acc = np.array([3, 1])
    o, new = oracle.multi_step(q, k, v, g, b, pool, idx, num_accepted=acc)
    for n in range(N):
        s0 = pool[idx[n, acc[n] - 1]]
        for t in range(S):
            o_r, s_r = oracle.recurrence(q[n, :t + 1], k[n, :t + 1], v[n, :t + 1], g[n, :t + 1],
                                         b[n, :t + 1], initial_state=s0[None])
            np.testing.assert_allclose(new[idx[n, t]], s_r[0], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(o[n, t], o_r[t], rtol=1e-12, atol=1e-13)
    untouched = [s for s in range(slots) if s not in idx]
    np.testing.assert_array_equal(new[untouched], pool[untouched])


# ---------------------------------------------------------------------------
# short causal convolution (Ascend model file, KimiShortConvolution)
# ---------------------------------------------------------------------------

def test_conv_unit_tap_is_the_activation_and_shifted_taps_delay():
    """weight = e_{ks-1} gives y = act(x); weight = e_{ks-1-j} delays x by j
    (zeros before the sequence start); silu(x) = x sigmoid(x)."""
    rng = np.random.default_rng(51)
    T, D, ks = 9, 6, 4
    x = rng.standard_normal((T, D))
    w = np.zeros((ks, D))
    w[ks - 1] = 1.0
    y, _ = oracle.short_conv_prefill(x, w, [0, T], activation="silu")
    np.testing.assert_allclose(y, x / (1.0 + np.exp(-x)), rtol=1e-14)
    for j in range(ks):
        w = np.zeros((ks, D))
        w[ks - 1 - j] = 1.0
        y, _ = oracle.short_conv_prefill(x, w, [0, T], activation="none")
        ref = np.zeros_like(x)
        ref[j:] = x[:T - j]
        np.testing.assert_array_equal(y, ref)


def test_conv_matches_numpy_convolve_per_channel():
    """Without activation each channel is the causal part of a full 1-D
    convolution with the reversed taps (numpy.convolve)."""
    rng = np.random.default_rng(52)
    T, D, ks = 13, 5, 4
    x = rng.standard_normal((T, D))
    w = rng.standard_normal((ks, D))
    y, fin = oracle.short_conv_prefill(x, w, [0, T], activation="none")
    for d in range(D):
        np.testing.assert_allclose(y[:, d], np.convolve(x[:, d], w[::-1, d])[:T], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(fin[0], x[T - (ks - 1):])


def test_conv_sequences_are_independent_and_short_ones_keep_history():
    rng = np.random.default_rng(53)
    D, ks = 4, 4
    lens = [5, 2, 0, 7]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rng.standard_normal((cu[-1], D))
    w = rng.standard_normal((ks, D))
    init = rng.standard_normal((len(lens), ks - 1, D))
    y, fin = oracle.short_conv_prefill(x, w, cu, initial_states=init)
    for n, L in enumerate(lens):
        yn, fn = oracle.short_conv_prefill(x[cu[n]:cu[n + 1]], w, [0, L], initial_states=init[n:n + 1])
        np.testing.assert_array_equal(y[cu[n]:cu[n + 1]], yn)
        np.testing.assert_array_equal(fin[n], fn[0])
    np.testing.assert_array_equal(fin[2], init[2])                            # empty: unchanged
    np.testing.assert_array_equal(fin[1], np.concatenate([init[1][2:], x[cu[1]:cu[2]]]))  # 2 < ks - 1


def test_conv_prefill_then_updates_equal_the_longer_prefill():
    """Prefill T1 tokens, then one update per remaining token from the final
    state, reproduces the prefill of all T tokens (outputs and state)."""
    rng = np.random.default_rng(54)
    T, T1, D, ks = 11, 6, 3, 4
    x = rng.standard_normal((T, D))
    w = rng.standard_normal((ks, D))
    y_all, fin_all = oracle.short_conv_prefill(x, w, [0, T])
    y1, st = oracle.short_conv_prefill(x[:T1], w, [0, T1])
    np.testing.assert_array_equal(y1, y_all[:T1])
    for t in range(T1, T):
        yt, st = oracle.short_conv_update(x[t:t + 1], w, st)
        np.testing.assert_allclose(yt[0], y_all[t], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(st[0], fin_all[0], rtol=0, atol=0)


def test_conv_multi_update_is_a_prefill_from_the_accepted_slot():
    """Each sequence's S outputs are the prefill of its S tokens from the
    conv state in its accepted slot (pinned above), the state written after
    token t is that prefill's final state over tokens 0..t, and S = 1 without
    counts is the one-token update; slots of no sequence are untouched."""
    rng = np.random.default_rng(55)
    N, S, D, ks, slots = 3, 4, 5, 4, 14
    x = rng.standard_normal((N, S, D))
    w = rng.standard_normal((ks, D))
    pool = rng.standard_normal((slots, ks - 1, D))
    idx = np.array([[0, 1, 2, 3], [7, 8, 9, 10], [4, 5, 6, 13]])
    acc = np.array([1, 3, 4])
    for act in ("silu", "none"):
        y, new = oracle.short_conv_multi_update(x, w, pool, idx, acc, activation=act)
        for n in range(N):
            start = pool[idx[n, acc[n] - 1]]
            y_r, _ = oracle.short_conv_prefill(x[n], w, [0, S], activation=act, initial_states=start[None])
            np.testing.assert_allclose(y[n], y_r, rtol=1e-13, atol=1e-14)
            for t in range(S):
                _, f_t = oracle.short_conv_prefill(x[n, :t + 1], w, [0, t + 1], activation=act,
                                                   initial_states=start[None])
                np.testing.assert_array_equal(new[idx[n, t]], f_t[0])
        untouched = [s_ for s_ in range(slots) if s_ not in idx]
        np.testing.assert_array_equal(new[untouched], pool[untouched])
    y1, new1 = oracle.short_conv_multi_update(x[:, :1], w, pool, idx[:, :1])
    y_u, st_u = oracle.short_conv_update(x[:, 0], w, pool[idx[:, 0]])
    np.testing.assert_array_equal(y1[:, 0], y_u)
    np.testing.assert_array_equal(new1[idx[:, 0]], st_u)
