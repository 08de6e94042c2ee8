"""Pins for the fp64 oracle: each test checks it against something other than
itself (a closed form, an invariant of the delta rule, a hand-derived example,
an independent chunked formulation, dense-matrix brute force), chosen so that a
dropped term, a wrong sign, a transposed state or a swapped decay/update order
fails at least one of them.

The rule being pinned: KDA, the channel-wise gated delta rule (agents-report.net
"FlashKDA" article, background section), with the FlashKDA README "Kernel API"
table's argument list and [.., V, K] state layout.
"""
import os

import numpy as np
import pytest

import oracle
from tests.chunked_np import chunked_pair

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def unit(x, axis=-1):
    return x / np.linalg.norm(x, axis=axis, keepdims=True)


def activated(seed, B, T, H, K, V, decay=True, beta_range=(0.0, 1.0)):
    r = rng(seed)
    q = unit(r.standard_normal((B, T, H, K)))
    k = unit(r.standard_normal((B, T, H, K)))
    v = r.standard_normal((B, T, H, V))
    gk = -r.uniform(0.0, 1.5, (B, T, H, K)) if decay else np.zeros((B, T, H, K))
    beta = r.uniform(beta_range[0], beta_range[1], (B, T, H))
    return q, k, v, gk, beta


# ---------------------------------------------------------------- worked example
def test_hand_derived_two_token_example():
    f = {}
    with open(os.path.join(GOLDEN, "kda_k2_worked_example.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            name, *vals = line.split()
            f[name] = np.array([float(x) for x in vals])
    q = np.stack([f["q1"], f["q2"]])[None, :, None, :]
    k = np.stack([f["k1"], f["k2"]])[None, :, None, :]
    v = np.stack([f["v1"], f["v2"]])[None, :, None, :]
    gk = np.log(np.stack([f["alpha1"], f["alpha2"]]))[None, :, None, :]
    beta = np.array([f["beta1"][0], f["beta2"][0]])[None, :, None]
    out, fin = oracle.recurrence(q, k, v, gk, beta, 1.0)
    np.testing.assert_allclose(out[0, 0, 0], f["o1"], atol=1e-13)
    np.testing.assert_allclose(out[0, 1, 0], f["o2"], atol=1e-13)
    np.testing.assert_allclose(fin[0, 0].reshape(-1), f["final"], atol=1e-13)


# ---------------------------------------------------------------- closed forms
def test_single_token_closed_form_zero_state():
    # T=1, S0=0:  S1 = beta k v^T  =>  o = scale * beta (k.q) v,  final[v][c] = beta v_v k_c
    q, k, v, gk, beta = activated(1, 2, 1, 3, 16, 8)
    out, fin = oracle.recurrence(q, k, v, gk, beta, 0.37)
    kq = np.sum(k * q, -1)
    np.testing.assert_allclose(out, 0.37 * (beta * kq)[..., None] * v, rtol=1e-12, atol=1e-14)
    want = beta[:, 0, :, None, None] * v[:, 0, :, :, None] * k[:, 0, :, None, :]
    np.testing.assert_allclose(fin, want, rtol=1e-12, atol=1e-14)


def test_beta_zero_is_pure_decay_of_initial_state():
    # beta=0: S_t = Diag(exp(G_t)) S0, o_t = scale * S0^T (exp(G_t) * q_t)
    B, T, H, K, V = 1, 9, 2, 12, 7
    q, k, v, gk, _ = activated(2, B, T, H, K, V)
    beta = np.zeros((B, T, H))
    S0 = rng(3).standard_normal((B, H, V, K))           # stored layout [V][K]
    out, fin = oracle.recurrence(q, k, v, gk, beta, 0.5, initial_state=S0)
    G = np.cumsum(gk, axis=1)                           # [B,T,H,K]
    want_out = 0.5 * np.einsum("bhvc,bthc->bthv", S0, np.exp(G) * q)
    np.testing.assert_allclose(out, want_out, rtol=1e-12, atol=1e-13)
    want_fin = S0 * np.exp(G[:, -1])[:, :, None, :]
    np.testing.assert_allclose(fin, want_fin, rtol=1e-12, atol=1e-14)


def test_initial_state_layout_is_v_by_k():
    # no decay, beta=0:  o = scale * S0^T q  with  S0[c][v] = state[v][c]
    B, T, H, K, V = 1, 1, 1, 5, 3
    q, k, v, _, _ = activated(4, B, T, H, K, V, decay=False)
    state = rng(5).standard_normal((1, 1, V, K))
    out, _ = oracle.recurrence(q, k, v, np.zeros((B, T, H, K)), np.zeros((B, T, H)), 1.0,
                               initial_state=state)
    np.testing.assert_allclose(out[0, 0, 0], state[0, 0] @ q[0, 0, 0], rtol=1e-13)


# ---------------------------------------------------------------- invariants
def test_beta_one_overwrites_the_key_slot():
    # beta=1, unit k:  k^T (I - k k^T) = 0  =>  S_t^T k_t = v_t for any decay and S0.
    # Querying with q_t = k_t therefore returns scale * v_t.
    B, T, H, K, V = 2, 17, 2, 16, 16
    _, k, v, gk, _ = activated(6, B, T, H, K, V)
    beta = np.ones((B, T, H))
    S0 = rng(7).standard_normal((B, H, V, K))
    out, _ = oracle.recurrence(k, k, v, gk, beta, 0.25, initial_state=S0)
    np.testing.assert_allclose(out, 0.25 * v, rtol=1e-11, atol=1e-12)


def test_orthonormal_keys_exact_retrieval_without_decay():
    # zero decay, beta=1 writes of m orthonormal keys into S0=0, then beta=0 reads:
    # querying k_j returns scale * v_j.
    K, V, m = 32, 8, 20
    Qm, _ = np.linalg.qr(rng(8).standard_normal((K, K)))
    keys = Qm[:, :m].T                                   # m orthonormal rows
    vals = rng(9).standard_normal((m, V))
    perm = rng(10).permutation(m)
    T = 2 * m
    q = np.zeros((1, T, 1, K)); k = np.zeros((1, T, 1, K)); v = np.zeros((1, T, 1, V))
    beta = np.zeros((1, T, 1))
    k[0, :m, 0] = keys; v[0, :m, 0] = vals; beta[0, :m, 0] = 1.0; q[0, :m, 0] = keys
    q[0, m:, 0] = keys[perm]; k[0, m:, 0] = keys[perm]
    out, _ = oracle.recurrence(q, k, v, np.zeros((1, T, 1, K)), beta, 2.0)
    np.testing.assert_allclose(out[0, m:, 0], 2.0 * vals[perm], atol=1e-12)


def test_scalar_gate_reduces_to_gated_deltanet():
    # Gated DeltaNet special case: a channel-uniform decay a commutes with the
    # projection (I - b k k^T), so S_t = a (I - b k k^T) S_{t-1} + b k v^T, i.e. the
    # decay may be applied after the projection (never to the new write b k v^T).
    B, T, H, K, V = 1, 11, 1, 8, 5
    q, k, v, _, beta = activated(11, B, T, H, K, V)
    a = -rng(12).uniform(0.0, 1.0, (B, T, H, 1)) * np.ones((1, 1, 1, K))
    out, fin = oracle.recurrence(q, k, v, a, beta, 1.0)
    S = np.zeros((K, V))
    for t in range(T):
        kt, vt, bt = k[0, t, 0], v[0, t, 0], beta[0, t, 0]
        S = S - bt * np.outer(kt, kt @ S)                  # project first
        S = np.exp(a[0, t, 0, 0]) * S + bt * np.outer(kt, vt)   # then decay, then write
        np.testing.assert_allclose(out[0, t, 0], S.T @ q[0, t, 0], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(fin[0, 0], S.T, rtol=1e-11, atol=1e-13)


def test_channel_gate_order_matters():
    # With per-channel decay the projection and the decay do NOT commute: the
    # reading "decay, then project" must differ from "project, then decay".
    B, T, H, K, V = 1, 4, 1, 8, 5
    q, k, v, gk, beta = activated(27, B, T, H, K, V)
    out, _ = oracle.recurrence(q, k, v, gk, beta, 1.0)
    S = np.zeros((K, V))
    for t in range(T):
        kt, vt, bt = k[0, t, 0], v[0, t, 0], beta[0, t, 0]
        S = S - bt * np.outer(kt, kt @ S)
        S = np.exp(gk[0, t, 0])[:, None] * S + bt * np.outer(kt, vt)
    assert np.abs(out[0, -1, 0] - S.T @ q[0, -1, 0]).max() > 1e-3


def test_dense_matrix_brute_force_tiny():
    # Each step as an explicit K x K transition matrix (I - b k k^T) Diag(alpha).
    B, T, H, K, V = 1, 6, 2, 4, 4
    q, k, v, gk, beta = activated(13, B, T, H, K, V)
    S0 = rng(14).standard_normal((B, H, V, K))
    out, fin = oracle.recurrence(q, k, v, gk, beta, 0.8, initial_state=S0)
    for h in range(H):
        S = S0[0, h].T.copy()
        for t in range(T):
            kt = k[0, t, h]
            Mt = (np.eye(K) - beta[0, t, h] * np.outer(kt, kt)) @ np.diag(np.exp(gk[0, t, h]))
            S = Mt @ S + beta[0, t, h] * np.outer(kt, v[0, t, h])
            np.testing.assert_allclose(out[0, t, h], 0.8 * S.T @ q[0, t, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(fin[0, h], S.T, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("C", [1, 3, 64])
def test_chunked_formula_equals_recurrence(C):
    B, T, H, K, V = 1, 150, 2, 16, 12
    q, k, v, gk, beta = activated(15 + C, B, T, H, K, V)
    S0 = rng(16).standard_normal((B, H, V, K)) * 0.1
    out, fin = oracle.recurrence(q, k, v, gk, beta, 0.3, initial_state=S0)
    for h in range(H):
        o, S = chunked_pair(q[0, :, h], k[0, :, h], v[0, :, h], gk[0, :, h], beta[0, :, h], 0.3,
                            S0[0, h].T, C)
        np.testing.assert_allclose(out[0, :, h], o, rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(fin[0, h], S.T, rtol=1e-9, atol=1e-10)


@pytest.mark.parametrize("C", [1, 3, 64])
def test_chunked_formula_equals_recurrence_unbounded_gate(C):
    # the gate without a lower bound decays by up to ~e^-60 per token here; the chunked
    # formula (explicit exp(G_t - G_i) <= 1) must still equal the token recurrence
    r = rng(40 + C)
    B, T, H, K, V = 1, 140, 2, 16, 12
    q, k = r.standard_normal((B, T, H, K)), r.standard_normal((B, T, H, K))
    g = 2.0 * r.standard_normal((B, T, H, K))
    v = r.standard_normal((B, T, H, V)); bl = r.standard_normal((B, T, H))
    A_log = np.log(np.array([1.0, 16.0])); dt = 0.1 * r.standard_normal((H, K))
    S0 = 0.1 * r.standard_normal((B, H, V, K))
    out, fin = oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, None, initial_state=S0)
    qn, kn, gk, b = oracle.activations(q, k, g, bl, A_log, dt, None)
    assert gk.min() < -40.0
    for h in range(H):
        o, S = chunked_pair(qn[0, :, h], kn[0, :, h], v[0, :, h], gk[0, :, h], b[0, :, h], 0.3,
                            S0[0, h].T, C)
        np.testing.assert_allclose(out[0, :, h], o, rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(fin[0, h], S.T, rtol=1e-9, atol=1e-10)


# ---------------------------------------------------------------- activations
def test_gate_special_values():
    # gk = lb * sigmoid(exp(A_log) * (g + dt_bias)):
    #   g = -dt_bias -> lb/2;  lb = 0 -> 0;  exp(A_log)(g+b) = ln 3 -> sigmoid = 3/4;
    #   very large argument -> lb;  A_log -> -inf (exp -> 0) -> lb/2.
    H, K = 3, 4
    dt = rng(17).standard_normal((H, K))
    A_log = np.array([0.0, np.log(2.0), -800.0])
    g = np.empty((1, 3, H, K))
    g[0, 0] = -dt                                        # -> lb/2 on every head
    with np.errstate(divide="ignore"):
        g[0, 1] = np.log(3.0) / np.exp(A_log)[:, None] - dt  # -> 3/4 lb on heads 0, 1
    g[0, 1, 2] = 5.0                                     # head 2: finite, exp(A_log) = 0
    g[0, 2] = 1e4                                        # -> lb on heads 0, 1
    z = np.zeros((1, 3, H, K)); zb = np.zeros((1, 3, H))
    _, _, gk, _ = oracle.activations(z + 1, z + 1, g, zb, A_log, dt, -4.0)
    np.testing.assert_allclose(gk[0, 0], -2.0, rtol=1e-14)
    np.testing.assert_allclose(gk[0, 1, :2], -3.0, rtol=1e-12)
    np.testing.assert_allclose(gk[0, 2, :2], -4.0, rtol=1e-14)
    np.testing.assert_allclose(gk[0, :, 2], -2.0, rtol=1e-14)   # A_log -> -inf
    _, _, gk0, _ = oracle.activations(z + 1, z + 1, g, zb, A_log, dt, 0.0)
    assert np.all(gk0 == 0.0)


def test_unbounded_gate_special_values():
    # The gate without a lower bound (lower_bound None): gk = -exp(A_log) softplus(g + dt_bias).
    #   g + dt = 0 -> -exp(A_log) ln 2;  g + dt = ln(e - 1) -> softplus 1 -> -exp(A_log);
    #   g + dt = 1e4 -> -exp(A_log) 1e4 (no overflow);  g + dt = -800 -> 0 (to 1e-300);
    #   A_log -> -inf -> 0.
    H, K = 3, 4
    dt = rng(27).standard_normal((H, K))
    A_log = np.array([0.0, np.log(2.0), -800.0])
    g = np.empty((1, 4, H, K))
    g[0, 0] = -dt
    g[0, 1] = np.log(np.e - 1.0) - dt
    g[0, 2] = 1e4 - dt
    g[0, 3] = -800.0 - dt
    z = np.zeros((1, 4, H, K)); zb = np.zeros((1, 4, H))
    _, _, gk, _ = oracle.activations(z + 1, z + 1, g, zb, A_log, dt, None)
    np.testing.assert_allclose(gk[0, 0, :2], -np.array([1.0, 2.0])[:, None] * np.log(2.0) * np.ones(K), rtol=1e-14)
    np.testing.assert_allclose(gk[0, 1, :2], -np.array([1.0, 2.0])[:, None] * np.ones(K), rtol=1e-12)
    np.testing.assert_allclose(gk[0, 2, :2], -np.array([1.0, 2.0])[:, None] * 1e4 * np.ones(K), rtol=1e-14)
    assert np.all(np.abs(gk[0, 3]) < 1e-300) and np.all(gk[0, 3] <= 0.0)
    assert np.all(np.abs(gk[0, :, 2]) < 1e-300)          # exp(A_log) = 0
    # strictly decreasing in g, and below every bounded gate's floor for large g
    xs = np.linspace(-6.0, 6.0, 25)
    gg = (xs[:, None] - dt[0][None, :])[None, :, None, :] * np.ones((1, 25, 1, K))
    _, _, gk1, _ = oracle.activations(gg + 1, gg + 1, gg, np.zeros((1, 25, 1)), A_log[:1], dt[:1], None)
    assert np.all(np.diff(gk1[0, :, 0, 0]) < 0.0)
    assert gk1[0, -1, 0, 0] < -5.0


def test_unbounded_gate_forward_composes():
    r = rng(28)
    B, T, H, K, V = 2, 6, 2, 8, 5
    q, k = r.standard_normal((B, T, H, K)), r.standard_normal((B, T, H, K))
    g = 2.0 * r.standard_normal((B, T, H, K))
    v = r.standard_normal((B, T, H, V)); bl = r.standard_normal((B, T, H))
    A_log = np.log(r.uniform(1, 16, H)); dt = 0.1 * r.standard_normal((H, K))
    S0 = 0.02 * r.standard_normal((B, H, V, K))
    out, fin = oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, None, initial_state=S0)
    qn, kn, gk, b = oracle.activations(q, k, g, bl, A_log, dt, None)
    assert np.all(gk < 0.0)
    o2, f2 = oracle.recurrence(qn, kn, v, gk, b, 0.3, initial_state=S0)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(fin, f2)
    # and it differs from every bounded gate on these inputs (the flag is honoured)
    o3, _ = oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, -5.0, initial_state=S0)
    assert np.abs(o3 - out).max() > 1e-3


def test_beta_sigmoid_and_l2_norm():
    r = rng(18)
    B, T, H, K = 1, 5, 2, 128
    q = r.standard_normal((B, T, H, K)); k = r.standard_normal((B, T, H, K))
    k[0, 0, 0] = 0.0                                     # zero vector maps to zero
    bl = np.array([0.0, np.log(3.0), -np.log(3.0), 40.0, -40.0])[None, :, None] * np.ones((B, T, H))
    qn, kn, _, b = oracle.activations(q, k, np.zeros_like(q), bl, np.zeros(H), np.zeros((H, K)), -5.0)
    np.testing.assert_allclose(b[0, :, 0], [0.5, 0.75, 0.25, 1.0, 0.0], atol=1e-15)
    nq = np.linalg.norm(qn, axis=-1)
    np.testing.assert_allclose(nq, 1.0, atol=1e-6)      # eps=1e-6 inside the sqrt
    np.testing.assert_allclose(qn * np.linalg.norm(q, axis=-1, keepdims=True), q,
                               rtol=1e-6)               # direction kept
    assert np.all(kn[0, 0, 0] == 0.0)
    # positive rescaling of the raw q leaves the normalised q unchanged (up to eps)
    qn2, _, _, _ = oracle.activations(7.0 * q, k, np.zeros_like(q), bl, np.zeros(H), np.zeros((H, K)), -5.0)
    np.testing.assert_allclose(qn2, qn, rtol=1e-7, atol=1e-9)


def test_full_forward_equals_activations_then_recurrence():
    # kda_fwd composes the two stages; check the composition and the final-state path.
    r = rng(19)
    B, T, H, K, V = 2, 7, 3, 8, 6
    q, k, g = (r.standard_normal((B, T, H, K)) for _ in range(3))
    v = r.standard_normal((B, T, H, V)); bl = r.standard_normal((B, T, H))
    A_log = np.log(r.uniform(1, 16, H)); dt = 0.1 * r.standard_normal((H, K))
    S0 = 0.02 * r.standard_normal((B, H, V, K))
    out, fin = oracle.kda_fwd(q, k, v, g, bl, 0.4, A_log, dt, -5.0, initial_state=S0)
    qn, kn, gk, b = oracle.activations(q, k, g, bl, A_log, dt, -5.0)
    o2, f2 = oracle.recurrence(qn, kn, v, gk, b, 0.4, initial_state=S0)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(fin, f2)


# ---------------------------------------------------------------- call structure
def _raw(seed, B, T, H, K=16, V=8):
    r = rng(seed)
    q, k, g = (r.standard_normal((B, T, H, K)) for _ in range(3))
    v = r.standard_normal((B, T, H, V)); bl = r.standard_normal((B, T, H))
    A_log = np.log(r.uniform(1, 16, H)); dt = 0.1 * r.standard_normal((H, K))
    return q, k, v, g, bl, A_log, dt


def test_chained_calls_equal_one_call():
    q, k, v, g, bl, A_log, dt = _raw(20, 2, 40, 3)
    S0 = 0.02 * rng(21).standard_normal((2, 3, 8, 16))
    out, fin = oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, -5.0, initial_state=S0)
    o1, f1 = oracle.kda_fwd(q[:, :13], k[:, :13], v[:, :13], g[:, :13], bl[:, :13], 0.3, A_log, dt,
                            -5.0, initial_state=S0)
    o2, f2 = oracle.kda_fwd(q[:, 13:], k[:, 13:], v[:, 13:], g[:, 13:], bl[:, 13:], 0.3, A_log, dt,
                            -5.0, initial_state=f1)
    np.testing.assert_allclose(np.concatenate([o1, o2], 1), out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(f2, fin, rtol=1e-12, atol=1e-14)


def test_varlen_equals_separate_calls():
    lens = [5, 0, 17, 1, 9]
    T = sum(lens)
    q, k, v, g, bl, A_log, dt = _raw(22, 1, T, 2)
    S0 = 0.02 * rng(23).standard_normal((len(lens), 2, 8, 16))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    out, fin = oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, -3.0, initial_state=S0, cu_seqlens=cu)
    for n, L in enumerate(lens):
        s, e = cu[n], cu[n + 1]
        o, f = oracle.kda_fwd(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e], bl[:, s:e], 0.3, A_log,
                              dt, -3.0, initial_state=S0[n:n + 1])
        np.testing.assert_array_equal(out[:, s:e], o)
        np.testing.assert_array_equal(fin[n:n + 1], f)
    # a zero-length sequence passes its state through unchanged
    np.testing.assert_array_equal(fin[1], S0[1])


def test_head_subset_matches_full_run():
    q, k, v, g, bl, A_log, dt = _raw(24, 2, 12, 4)
    out, fin = oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, -5.0)
    o2, f2 = oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, -5.0, pairs=[(1, 2), (0, 3)])
    np.testing.assert_array_equal(o2[1, :, 2], out[1, :, 2])
    np.testing.assert_array_equal(f2[0, 3], fin[0, 3])
    assert np.isnan(o2[0, :, 0]).all()


def test_thread_count_does_not_change_results():
    q, k, v, g, bl, A_log, dt = _raw(25, 1, 30, 6)
    a = oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, -5.0, nthreads=1)
    b = oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, -5.0, nthreads=4)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_malformed_cu_seqlens_rejected():
    q, k, v, g, bl, A_log, dt = _raw(26, 1, 10, 1)
    with pytest.raises(ValueError):
        oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, -5.0, cu_seqlens=np.array([0, 4, 3, 10]))
    with pytest.raises(ValueError):
        oracle.kda_fwd(q, k, v, g, bl, 0.3, A_log, dt, -5.0, cu_seqlens=np.array([0, 4, 9]))
