"""The window in matrix form equals the token-by-token recurrence.

The verify and native kernels do not form the intermediate states.  With
the checkpoint C, gamma_t = alpha_0 ... alpha_t and rho_{t,j} = alpha_{j+1}
... alpha_t (per channel for the KDA decay), the state after token t is
  S_t = C diag(gamma_t) + sum_{j<=t} u_j (rho_{t,j} khat_j)^T,
so
  d_t = H_t khat_t = C (gamma_t khat_t) + sum_{j<t}  A_{t,j} u_j,
  o_t = S_t qhat_t = C (gamma_t qhat_t) + sum_{j<=t} B_{t,j} u_j,
  A_{t,j} = <rho_{t,j} khat_j, khat_t>,  B_{t,j} = <rho_{t,j} khat_j, qhat_t>,
and u_t = beta_t (v_t - d_t).  This file checks that algebra in fp64, in
code of its own, against the oracle's token-by-token window: a wrong
product range in gamma or rho, a dropped j = t term in B, or the decay on
the wrong side of C fails it.
"""
import math

import numpy as np
import pytest

import oracle


def matrix_form(S0, khat, qhat, alpha, beta, v):
    """u_t and o_t of one unit from the checkpoint and the window's vectors.
    alpha is [w] (one decay per token) or [w][K] (one per channel)."""
    w, K = khat.shape
    al = alpha if alpha.ndim == 2 else np.repeat(alpha[:, None], K, axis=1)
    gamma = np.cumprod(al, axis=0)
    P = S0 @ (gamma * khat).T   # [V][w]: C kt_t
    Q = S0 @ (gamma * qhat).T   # [V][w]: C qt_t

    def rho(t, j):              # alpha_{j+1} ... alpha_t, per channel
        return np.prod(al[j + 1:t + 1], axis=0) if t > j else np.ones(K)

    u = np.zeros_like(v)
    o = np.zeros_like(v)
    for t in range(w):
        d = P[:, t] + sum(np.dot(rho(t, j) * khat[j], khat[t]) * u[j] for j in range(t))
        u[t] = beta[t] * (v[t] - d)
        o[t] = Q[:, t] + sum(np.dot(rho(t, j) * khat[j], qhat[t]) * u[j] for j in range(t + 1))
    return u, o


def _unit(seed, K, V, w, extreme=False, kda=False):
    g = np.random.default_rng(seed)
    shape = (w, K) if kda else (w,)
    return dict(
        S0=g.normal(0, 0.1, (V, K)), q=g.normal(size=(w, K)), k=g.normal(size=(w, K)),
        v=g.normal(size=(w, V)),
        a=g.uniform(-20, 20, shape) if extreme else g.normal(size=shape),
        b=g.uniform(-20, 20, w) if extreme else g.normal(size=w),
        A_log=float(g.uniform(0, math.log(16))),
        dt_bias=g.uniform(-1, 1, K) if kda else float(g.uniform(-1, 1)))


def _check(d, kda):
    run = oracle.kda_window if kda else oracle.window
    ref = run(d["S0"], d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"])
    qhat = np.stack([oracle.l2norm(x) for x in d["q"]])
    beta = np.array([oracle.beta(x) for x in d["b"]])
    u, o = matrix_form(d["S0"], ref["khat"], qhat, ref["alpha"], beta, d["v"])
    scale = 1.0 + np.abs(ref["u"]).max()
    assert np.abs(u - ref["u"]).max() <= 1e-12 * scale
    scale = 1.0 + np.abs(ref["o"]).max()
    assert np.abs(o - ref["o"]).max() <= 1e-12 * scale


@pytest.mark.parametrize("w", [1, 2, 4, 6, 16])
@pytest.mark.parametrize("kda", [False, True])
def test_matrix_form_equals_recurrence(w, kda):
    for seed in range(3):
        _check(_unit(seed, K=16, V=24, w=w, kda=kda), kda)


@pytest.mark.parametrize("kda", [False, True])
def test_matrix_form_with_extreme_gates(kda):
    # decays down to exactly 0 and betas near 0 and 1
    for seed in range(4):
        _check(_unit(100 + seed, K=16, V=24, w=6, extreme=True, kda=kda), kda)


def test_matrix_form_with_a_zero_decay_mid_window():
    # alpha_2 = 0 exactly: everything before token 2 drops out of S_2 on
    d = _unit(7, K=16, V=24, w=5)
    d["a"][2] = 1e4
    assert oracle.decay(d["a"][2], d["A_log"], d["dt_bias"]) == 0.0
    _check(d, kda=False)


def test_matrix_form_catches_a_dropped_diagonal_term():
    # without the j = t term of o_t the two forms disagree: the pin has teeth
    d = _unit(11, K=16, V=24, w=4)
    ref = oracle.window(d["S0"], d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"])
    qhat = np.stack([oracle.l2norm(x) for x in d["q"]])
    beta = np.array([oracle.beta(x) for x in d["b"]])
    u, o = matrix_form(d["S0"], ref["khat"], qhat, ref["alpha"], beta, d["v"])
    o_wrong = o - np.array([np.dot(ref["khat"][t], qhat[t]) * u[t] for t in range(4)])
    assert np.abs(o_wrong - ref["o"]).max() > 1e-3
