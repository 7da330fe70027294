"""Pins of the oracle's backward (reverse-mode gradients of the recurrence).

The gradients are checked against central finite differences of the forward
oracle for the loss sum(dO * O) + sum(dS * S_final), on every input (q, k, v,
g, beta and the initial state), with and without the L2 normalisation and on a
varlen call; plus closed forms: beta = 0 and the linearity of the loss in v.
"""
import numpy as np
import pytest

import oracle


def loss(q, k, v, g, beta, s0, dO, dS, cu, scale, l2):
    o, sf = oracle.recurrent_fwd(q, k, v, g, beta, init_state=s0, cu_seqlens=cu, scale=scale, use_qk_l2norm=l2)
    return float((o * dO).sum() + (sf * dS).sum())


def finite_diff(args, name, idx, h=1e-6):
    a = {n: x.copy() for n, x in args.items() if isinstance(x, np.ndarray)}
    full = dict(args)
    plus, minus = dict(full), dict(full)
    xp, xm = a[name].copy(), a[name].copy()
    xp[idx] += h
    xm[idx] -= h
    plus[name], minus[name] = xp, xm
    return (loss(**plus) - loss(**minus)) / (2 * h)


def make(rng, B, T, H, dk, dv, N=None, cu=None):
    N = B if N is None else N
    return dict(q=rng.standard_normal((B, T, H, dk)), k=rng.standard_normal((B, T, H, dk)),
                v=rng.standard_normal((B, T, H, dv)), g=-0.3 * np.abs(rng.standard_normal((B, T, H))),
                beta=rng.uniform(0.1, 1.9, (B, T, H)), s0=rng.standard_normal((N, H, dv, dk)),
                dO=rng.standard_normal((B, T, H, dv)), dS=rng.standard_normal((N, H, dv, dk)), cu=cu)


@pytest.mark.parametrize("l2", [False, True])
def test_gradients_equal_finite_differences(l2):
    rng = np.random.default_rng(60 + l2)
    args = make(rng, B=2, T=6, H=2, dk=3, dv=2)
    args.update(scale=0.7, l2=l2)
    r = oracle.recurrent_bwd(args["q"], args["k"], args["v"], args["g"], args["beta"], args["dO"],
                             init_state=args["s0"], dfinal=args["dS"], scale=0.7, use_qk_l2norm=l2)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"), ("s0", "dinit")):
        x = args[name]
        for flat in range(0, x.size, max(1, x.size // 17)):
            idx = np.unravel_index(flat, x.shape)
            fd = finite_diff(args, name, idx)
            assert abs(r[key][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx, r[key][idx], fd)


def test_gradients_varlen_equal_finite_differences():
    rng = np.random.default_rng(62)
    lens = [3, 0, 5, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    args = make(rng, B=1, T=sum(lens), H=1, dk=3, dv=2, N=len(lens), cu=cu)
    args.update(scale=1.0, l2=True)
    r = oracle.recurrent_bwd(args["q"], args["k"], args["v"], args["g"], args["beta"], args["dO"],
                             init_state=args["s0"], dfinal=args["dS"], cu_seqlens=cu, use_qk_l2norm=True)
    for name, key in (("k", "dk"), ("g", "dg"), ("beta", "dbeta"), ("s0", "dinit")):
        x = args[name]
        for flat in range(x.size):
            idx = np.unravel_index(flat, x.shape)
            fd = finite_diff(args, name, idx)
            assert abs(r[key][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx)
    # an empty sequence passes its state gradient straight through
    np.testing.assert_array_equal(r["dinit"][1], args["dS"][1])


def test_beta_zero_and_linearity_in_v():
    """beta = 0: S_t = gamma_t S_0, so dv = 0, dk = 0, and dS0 = gamma_L dS + sum_t gamma_t dO_t q_t^T."""
    rng = np.random.default_rng(63)
    B, T, H, dk, dv = 1, 5, 1, 3, 2
    a = make(rng, B, T, H, dk, dv)
    beta = np.zeros((B, T, H))
    r = oracle.recurrent_bwd(a["q"], a["k"], a["v"], a["g"], beta, a["dO"], init_state=a["s0"], dfinal=a["dS"])
    np.testing.assert_allclose(r["dv"], 0, atol=0)
    np.testing.assert_allclose(r["dk"], 0, atol=1e-15)
    gam = np.exp(np.cumsum(a["g"][0, :, 0]))
    ds0 = gam[-1] * a["dS"][0, 0] + sum(gam[t] * np.outer(a["dO"][0, t, 0], a["q"][0, t, 0]) for t in range(T))
    np.testing.assert_allclose(r["dinit"][0, 0], ds0, atol=1e-12)
