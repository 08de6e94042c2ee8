"""Pins of the fp64 backward oracle (oracle.kda_bwd), CPU only.

The backward is the derivative of the forward, so it is checked against things that
the forward and the mathematics fix, not against a second copy of its formulas:
  - directional central differences of L = sum(dout * out) + sum(dfinal * final) taken
    through the (independently pinned) fp64 forward, for every input, both gates, fixed
    length and varlen with an empty sequence;
  - closed forms: one token from a zero state (out = scale beta (q_hat . k_hat) v), and
    beta = 0, where the state only decays (out_t = scale (P_t * S_0)^T q_hat_t with P_t
    the running product of the decays).
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _case(seed, B=2, T=9, H=2, K=8, V=8, varlen=None, unbounded=False):
    r = np.random.default_rng(seed)
    if varlen is not None:
        B, T = 1, int(sum(varlen))
    d = {"q": r.normal(size=(B, T, H, K)), "k": r.normal(size=(B, T, H, K)),
         "v": r.normal(size=(B, T, H, V)), "g": r.normal(size=(B, T, H, K)),
         "beta": r.normal(size=(B, T, H)), "A_log": np.log(r.uniform(1, 4, size=H)),
         "dt_bias": 0.3 * r.normal(size=(H, K)), "scale": K ** -0.5,
         "lower_bound": None if unbounded else -3.0,
         "cu_seqlens": None if varlen is None else np.concatenate([[0], np.cumsum(varlen)]).astype(np.int64)}
    N = B if varlen is None else len(varlen)
    d["initial_state"] = 0.5 * r.normal(size=(N, H, V, K))
    d["dout"] = r.normal(size=(B, T, H, V))
    d["dfinal"] = r.normal(size=(N, H, V, K))
    return d


def _loss(d, **over):
    e = dict(d, **over)
    out, fin = oracle.kda_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], e["scale"], e["A_log"],
                              e["dt_bias"], e["lower_bound"], initial_state=e["initial_state"],
                              cu_seqlens=e["cu_seqlens"], want_final=True)
    if e["cu_seqlens"] is not None:   # rows outside every sequence do not exist here
        pass
    return float(np.sum(e["dout"] * out) + np.sum(e["dfinal"] * fin))


def _grads(d):
    return oracle.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"],
                          d["dt_bias"], d["lower_bound"], d["dout"], initial_state=d["initial_state"],
                          dfinal=d["dfinal"], cu_seqlens=d["cu_seqlens"])


GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "A_log": "dA_log",
           "dt_bias": "ddt_bias", "initial_state": "dinit"}


@pytest.mark.parametrize("kind", ["bounded", "unbounded", "varlen", "varlen_unbounded"])
def test_directional_derivatives_match_central_differences(kind):
    varlen = (4, 0, 7, 1) if kind.startswith("varlen") else None
    d = _case(3 + len(kind), varlen=varlen, unbounded=kind.endswith("unbounded"))
    gr = _grads(d)
    r = np.random.default_rng(17)
    eps = 1e-6
    for name, gname in GRAD_OF.items():
        for _ in range(2):
            D = r.normal(size=np.shape(d[name]))
            fd = (_loss(d, **{name: d[name] + eps * D}) - _loss(d, **{name: d[name] - eps * D})) / (2 * eps)
            an = float(np.sum(gr[gname] * D))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (kind, name, fd, an)


def test_one_token_from_zero_state_closed_form():
    d = _case(5, B=1, T=1, H=1, K=8, V=8)
    d["initial_state"] = np.zeros_like(d["initial_state"])
    d["dfinal"] = np.zeros_like(d["dfinal"])
    gr = _grads(d)
    q, k, v, do = d["q"][0, 0, 0], d["k"][0, 0, 0], d["v"][0, 0, 0], d["dout"][0, 0, 0]
    qh, kh = q / np.sqrt(q @ q + 1e-6), k / np.sqrt(k @ k + 1e-6)
    b = 1 / (1 + np.exp(-d["beta"][0, 0, 0]))
    # out = scale * beta * (q_hat . k_hat) * v
    np.testing.assert_allclose(gr["dv"][0, 0, 0], d["scale"] * b * (qh @ kh) * do, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(gr["dbeta"][0, 0, 0], d["scale"] * (qh @ kh) * (v @ do) * b * (1 - b),
                               rtol=1e-12, atol=1e-14)
    # from a zero state the decay of this token multiplies nothing
    np.testing.assert_allclose(gr["dg"], 0.0, atol=1e-14)
    np.testing.assert_allclose(gr["dA_log"], 0.0, atol=1e-14)


def test_zero_beta_state_only_decays_closed_form():
    d = _case(6, B=1, T=6, H=1, K=8, V=8)
    d["beta"] = np.full_like(d["beta"], -1e3)   # sigmoid is exactly 0 in fp64
    gr = _grads(d)
    qn, _, gk, _ = oracle.activations(d["q"], d["k"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                                      d["lower_bound"])
    P = np.cumprod(np.exp(gk[0, :, 0]), axis=0)          # [T, K]: decay from the start through t
    # S_t[c][v] = P_t[c] S_0[c][v];  out_t = scale S_t^T q_hat_t
    dS0 = np.einsum("tc,tv->cv", d["scale"] * qn[0, :, 0] * P, d["dout"][0, :, 0])
    dS0 += P[-1][:, None] * d["dfinal"][0, 0].T
    np.testing.assert_allclose(gr["dinit"][0, 0].T, dS0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(gr["dv"], 0.0, atol=1e-14)
    np.testing.assert_allclose(gr["dk"], 0.0, atol=1e-14)


def test_zero_upstream_gives_zero_gradients():
    d = _case(7)
    d["dout"] = np.zeros_like(d["dout"])
    d["dfinal"] = np.zeros_like(d["dfinal"])
    gr = _grads(d)
    for name in GRAD_OF.values():
        assert np.all(gr[name] == 0.0), name
