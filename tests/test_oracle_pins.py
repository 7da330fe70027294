"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print, closed forms, a different algorithm (explicit matrix products,
a library linear solve, the dense parallel SSD form), or invariants.  A
plausible slip in the oracle (a dropped decay, decay applied after the error,
a transposed state, a wrong mask, an off-by-one in the cumulative gate) makes
at least one of them fail.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def rand_inputs(rng, B, T, H, dk, dv, decay=0.3, unit_keys=True):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    g = -decay * np.log1p(np.exp(rng.standard_normal((B, T, H))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    return q, k, v, g, beta


# --------------------------------------------------------------------------
# P-a: the worked example (deep-dive page, "手算两格记忆")
# --------------------------------------------------------------------------

def test_worked_example_golden():
    gold = json.load(open(GOLDEN))
    for case in gold["cases"]:
        S = np.array(case["S"], np.float64)[None, None]          # [1,1,dv=1,dk=2]
        k = np.array(case["k"], np.float64)[None, None]           # [1,1,2]
        v = np.array(case["v"], np.float64)[None, None]           # [1,1,1]
        q = np.array([1.0, 0.0])[None, None]
        g = np.array([[math.log(case["alpha"])]])
        b = np.array([[case["beta"]]])
        out, S1 = oracle.decode_step(S, q, k, v, g, b)
        np.testing.assert_array_equal(S1[0, 0], np.array(case["expect"]))
        # o = S_t q_t with q = e_1 reads the first cell of the updated state
        assert out[0, 0, 0] == case["expect"][0][0]
        if "must_differ_from" in case:
            assert not np.allclose(S1[0, 0], np.array(case["must_differ_from"]))
        # the same step through the sequence entry point
        o2, sf = oracle.recurrent_fwd(q[None], k[None], v[None], g[None], b[None], init_state=S)
        np.testing.assert_array_equal(sf[0, 0], np.array(case["expect"]))


def test_memory_context_figures():
    mc = json.load(open(GOLDEN))["memory_context"]
    assert mc["heads"] * mc["d"] * mc["d"] * 4 == mc["state_bytes_fp32_per_layer"] == 1 << 20
    assert mc["kv_heads"] * mc["d"] * mc["positions"] * 2 * 2 == mc["kv_bytes_bf16_per_layer"] == 64 << 20


# --------------------------------------------------------------------------
# Explicit transition-matrix form of eq. 10 (brute force)
# --------------------------------------------------------------------------

def brute_force_eq10(q, k, v, g, beta, S0):
    """S_t = S_{t-1} (alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T with
    explicit dk x dk transition matrices, o_t = S_t q_t (one sequence, one head)."""
    T, dk = k.shape
    S = S0.copy()
    outs = []
    for t in range(T):
        A = math.exp(g[t]) * (np.eye(dk) - beta[t] * np.outer(k[t], k[t]))
        S = S @ A + beta[t] * np.outer(v[t], k[t])
        outs.append(S @ q[t])
    return np.array(outs), S


@pytest.mark.parametrize("unit_keys", [True, False])
def test_recurrence_matches_explicit_transition_products(unit_keys):
    rng = np.random.default_rng(1)
    B, T, H, dk, dv = 2, 13, 3, 5, 4
    q, k, v, g, beta = rand_inputs(rng, B, T, H, dk, dv, unit_keys=unit_keys)
    S0 = rng.standard_normal((B, H, dv, dk))
    out, sf = oracle.recurrent_fwd(q, k, v, g, beta, init_state=S0)
    for b in range(B):
        for h in range(H):
            o_ref, s_ref = brute_force_eq10(q[b, :, h], k[b, :, h], v[b, :, h], g[b, :, h], beta[b, :, h], S0[b, h])
            np.testing.assert_allclose(out[b, :, h], o_ref, rtol=0, atol=1e-12)
            np.testing.assert_allclose(sf[b, h], s_ref, rtol=0, atol=1e-12)


def test_ordered_composition_two_steps():
    """S_{t+1} = S_{t-1} A_t A_{t+1} + B_t A_{t+1} + B_{t+1} (deep-dive "Decode 递归");
    the product order matters, which a state-transpose slip would break."""
    rng = np.random.default_rng(2)
    dk, dv = 4, 3
    S = rng.standard_normal((dv, dk))
    k = rng.standard_normal((2, dk))
    v = rng.standard_normal((2, dv))
    a = np.array([0.7, 0.4])
    b = np.array([0.3, 0.9])
    A = [a[i] * (np.eye(dk) - b[i] * np.outer(k[i], k[i])) for i in range(2)]
    Bm = [b[i] * np.outer(v[i], k[i]) for i in range(2)]
    expect = S @ A[0] @ A[1] + Bm[0] @ A[1] + Bm[1]
    wrong = S @ A[1] @ A[0] + Bm[1] @ A[0] + Bm[0]
    st = S[None, None]
    for i in range(2):
        _, st = oracle.decode_step(st, k[i][None, None], k[i][None, None], v[i][None, None],
                                   np.log(a[i]).reshape(1, 1), b[i].reshape(1, 1))
    np.testing.assert_allclose(st[0, 0], expect, atol=1e-13)
    assert not np.allclose(expect, wrong)


# --------------------------------------------------------------------------
# P-b / P-c: invariants of one step (deep-dive page; blog §一(二) Householder)
# --------------------------------------------------------------------------

def test_unit_key_interpolation_every_step():
    """For ||k||=1: S_t k_t = (1 - beta_t) alpha_t S_{t-1} k_t + beta_t v_t."""
    rng = np.random.default_rng(3)
    N, H, dk, dv, steps = 2, 2, 8, 6, 20
    st = rng.standard_normal((N, H, dv, dk))
    for _ in range(steps):
        q = rng.standard_normal((N, H, dk))
        k = rng.standard_normal((N, H, dk))
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        v = rng.standard_normal((N, H, dv))
        g = -np.abs(rng.standard_normal((N, H)))
        b = rng.uniform(0, 1, (N, H))
        _, new = oracle.decode_step(st, q, k, v, g, b)
        lhs = np.einsum("nhjd,nhd->nhj", new, k)
        rhs = (1 - b)[..., None] * np.exp(g)[..., None] * np.einsum("nhjd,nhd->nhj", st, k) + b[..., None] * v
        np.testing.assert_allclose(lhs, rhs, atol=1e-12)
        st = new


def test_householder_fixed_directions():
    """(I - beta k k^T) x = x for x orthogonal to k, so S_t x = alpha_t S_{t-1} x."""
    rng = np.random.default_rng(4)
    dk, dv = 7, 5
    st = rng.standard_normal((1, 1, dv, dk))
    k = rng.standard_normal(dk)
    x = rng.standard_normal(dk)
    x -= (x @ k) / (k @ k) * k
    v = rng.standard_normal(dv)
    alpha, beta = 0.8, 0.6
    _, new = oracle.decode_step(st, x[None, None], k[None, None], v[None, None],
                                np.array([[math.log(alpha)]]), np.array([[beta]]))
    np.testing.assert_allclose(new[0, 0] @ x, alpha * st[0, 0] @ x, atol=1e-12)


# --------------------------------------------------------------------------
# P-d: alpha = 1 is DeltaNet, against eqs. 6-9 written with a library solve
# --------------------------------------------------------------------------

def deltanet_chunked_eq6_9(q, k, v, beta, C):
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk))
    O = np.zeros((T, dv))
    for t0 in range(0, T, C):
        Q, K, V, b = q[t0:t0 + C], k[t0:t0 + C], v[t0:t0 + C], beta[t0:t0 + C]
        n = len(b)
        Lmat = np.eye(n) + np.tril(np.diag(b) @ (K @ K.T), -1)
        Tm = np.linalg.solve(Lmat, np.diag(b))                  # eq. 6
        W, U = Tm @ K, Tm @ V                                    # eq. 7
        Vn = U - W @ S.T
        O[t0:t0 + n] = Q @ S.T + np.tril(Q @ K.T) @ Vn           # eq. 9 (mask M)
        S = S + Vn.T @ K                                         # eq. 8
    return O, S


@pytest.mark.parametrize("C", [4, 16])
def test_alpha_one_is_deltanet(C):
    rng = np.random.default_rng(5)
    B, T, H, dk, dv = 1, 37, 2, 6, 5
    q, k, v, g, beta = rand_inputs(rng, B, T, H, dk, dv)
    g = np.zeros_like(g)
    out, sf = oracle.recurrent_fwd(q, k, v, g, beta)
    for h in range(H):
        O, S = deltanet_chunked_eq6_9(q[0, :, h], k[0, :, h], v[0, :, h], beta[0, :, h], C)
        np.testing.assert_allclose(out[0, :, h], O, atol=1e-11)
        np.testing.assert_allclose(sf[0, h], S, atol=1e-11)


# --------------------------------------------------------------------------
# P-e: beta = 0 leaves only the decay (closed form)
# --------------------------------------------------------------------------

def test_beta_zero_closed_form():
    rng = np.random.default_rng(6)
    B, T, H, dk, dv = 2, 19, 2, 5, 3
    q, k, v, g, beta = rand_inputs(rng, B, T, H, dk, dv)
    beta = np.zeros_like(beta)
    S0 = rng.standard_normal((B, H, dv, dk))
    out, sf = oracle.recurrent_fwd(q, k, v, g, beta, init_state=S0, scale=0.7)
    gam = np.exp(np.cumsum(g, axis=1))                            # gamma_t = prod alpha
    expect = gam[..., None] * np.einsum("bhjd,bthd->bthj", S0, 0.7 * q)
    np.testing.assert_allclose(out, expect, atol=1e-12)
    np.testing.assert_allclose(sf, gam[:, -1][..., None, None] * S0, atol=1e-12)


# --------------------------------------------------------------------------
# P-f: orthogonal keys reduce to the SSD parallel form (paper §2.1)
# --------------------------------------------------------------------------

def test_orthogonal_keys_ssd_parallel_form():
    rng = np.random.default_rng(7)
    T, dk, dv = 10, 12, 4
    perm = rng.permutation(dk)[:T]
    k = np.eye(dk)[perm]                                          # mutually orthogonal unit keys
    q = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    g = -0.5 * rng.uniform(0, 1, T)
    beta = rng.uniform(0.1, 1, T)
    out, _ = oracle.recurrent_fwd(q[None, :, None], k[None, :, None], v[None, :, None],
                                  g[None, :, None], beta[None, :, None])
    gam = np.exp(np.cumsum(g))
    Gamma = np.tril(gam[:, None] / gam[None, :])                  # Gamma_ij = gamma_i / gamma_j, i >= j
    O = ((q @ k.T) * Gamma) @ (beta[:, None] * v)
    np.testing.assert_allclose(out[0, :, 0], O, atol=1e-12)
    # with beta = 1 this is Mamba2 exactly
    out1, _ = oracle.recurrent_fwd(q[None, :, None], k[None, :, None], v[None, :, None],
                                   g[None, :, None], np.ones((1, T, 1)))
    np.testing.assert_allclose(out1[0, :, 0], ((q @ k.T) * Gamma) @ v, atol=1e-12)


# --------------------------------------------------------------------------
# P-g / P-h: the chunkwise form equals the recurrence; UT solve residuals
# --------------------------------------------------------------------------

@pytest.mark.parametrize("C", [1, 2, 3, 4, 8, 16, 64])
@pytest.mark.parametrize("w_form", [0, 1])
def test_chunked_equals_recurrent(C, w_form):
    rng = np.random.default_rng(8 + C)
    B, T, H, dk, dv = 2, 40, 2, 8, 6
    q, k, v, g, beta = rand_inputs(rng, B, T, H, dk, dv, decay=1.0)
    S0 = rng.standard_normal((B, H, dv, dk))
    o1, s1 = oracle.recurrent_fwd(q, k, v, g, beta, init_state=S0, scale=0.5)
    o2, s2 = oracle.chunked_fwd(q, k, v, g, beta, init_state=S0, scale=0.5, chunk_size=C, w_form=w_form)
    np.testing.assert_allclose(o2, o1, atol=1e-10)
    np.testing.assert_allclose(s2, s1, atol=1e-10)


def test_chunked_output_mask_is_decay_mask():
    """With the plain causal mask M (as one printed formula reads) instead of
    Gamma, the chunked output departs from the recurrence; Gamma matches it."""
    rng = np.random.default_rng(9)
    T, dk, dv, C = 16, 4, 3, 8
    q, k, v, g, beta = rand_inputs(rng, 1, T, 1, dk, dv, decay=1.0)
    ref, _ = oracle.recurrent_fwd(q, k, v, g, beta)
    Q, K, V, gg, bb = q[0, :C, 0], k[0, :C, 0], v[0, :C, 0], g[0, :C, 0], beta[0, :C, 0]
    W, U = oracle.ut_transform(K, V, np.exp(gg), bb)
    gam = np.exp(np.cumsum(gg))
    Gamma = np.tril(gam[:, None] / gam[None, :])
    with_gamma = (Q @ K.T * Gamma) @ U                             # S_[0] = 0
    with_mask = np.tril(Q @ K.T) @ U
    np.testing.assert_allclose(with_gamma, ref[0, :C, 0], atol=1e-12)
    assert np.abs(with_mask - ref[0, :C, 0]).max() > 1e-3


def test_ut_transform_residuals_and_w_forms():
    rng = np.random.default_rng(10)
    C, dk, dv = 16, 6, 5
    K = rng.standard_normal((C, dk))
    V = rng.standard_normal((C, dv))
    alpha = np.exp(-rng.uniform(0, 1, C))
    beta = rng.uniform(0, 1, C)
    W0, U = oracle.ut_transform(K, V, alpha, beta, w_form=0)
    W1, _ = oracle.ut_transform(K, V, alpha, beta, w_form=1)
    gam = np.cumprod(alpha)
    Gamma = np.tril(gam[:, None] / gam[None, :])
    LG = np.eye(C) + np.tril(np.diag(beta) @ (Gamma * (K @ K.T)), -1)
    L = np.eye(C) + np.tril(np.diag(beta) @ (K @ K.T), -1)
    np.testing.assert_allclose(LG @ U, beta[:, None] * V, atol=1e-12)          # Gamma-masked system
    np.testing.assert_allclose(L @ (W1 / gam[:, None]), beta[:, None] * K, atol=1e-12)  # eq. 6-7 W
    np.testing.assert_allclose(W0, W1, atol=1e-12)                              # the two W readings agree


# --------------------------------------------------------------------------
# P-i: composition, carry, varlen, decode == prefill
# --------------------------------------------------------------------------

def test_state_carry_split_equals_whole():
    rng = np.random.default_rng(11)
    B, T, H, dk, dv = 2, 30, 2, 5, 4
    q, k, v, g, beta = rand_inputs(rng, B, T, H, dk, dv)
    S0 = rng.standard_normal((B, H, dv, dk))
    o, s = oracle.recurrent_fwd(q, k, v, g, beta, init_state=S0)
    cut = 11
    oa, sa = oracle.recurrent_fwd(q[:, :cut], k[:, :cut], v[:, :cut], g[:, :cut], beta[:, :cut], init_state=S0)
    ob, sb = oracle.recurrent_fwd(q[:, cut:], k[:, cut:], v[:, cut:], g[:, cut:], beta[:, cut:], init_state=sa)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, atol=1e-13)
    np.testing.assert_allclose(sb, s, atol=1e-13)


@pytest.mark.parametrize("fn", ["recurrent", "chunked"])
def test_varlen_equals_separate_calls(fn):
    rng = np.random.default_rng(12)
    lens = [1, 9, 17, 3]
    T, H, dk, dv = sum(lens), 2, 6, 5
    q, k, v, g, beta = rand_inputs(rng, 1, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dv, dk))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    call = oracle.recurrent_fwd if fn == "recurrent" else (lambda *a, **kw: oracle.chunked_fwd(*a, chunk_size=4, **kw))
    o, s = call(q, k, v, g, beta, init_state=S0, cu_seqlens=cu)
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        on, sn = oracle.recurrent_fwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b],
                                      init_state=S0[n:n + 1])
        np.testing.assert_allclose(o[:, a:b], on, atol=1e-12)
        np.testing.assert_allclose(s[n], sn[0], atol=1e-12)


def test_decode_steps_equal_prefill():
    rng = np.random.default_rng(13)
    N, T, H, dk, dv = 3, 9, 2, 6, 4
    q, k, v, g, beta = rand_inputs(rng, N, T, H, dk, dv)
    S0 = rng.standard_normal((N, H, dv, dk))
    o, s = oracle.recurrent_fwd(q, k, v, g, beta, init_state=S0, scale=0.3)
    st = S0
    for t in range(T):
        ot, st = oracle.decode_step(st, q[:, t], k[:, t], v[:, t], g[:, t], beta[:, t], scale=0.3)
        np.testing.assert_allclose(ot, o[:, t], atol=1e-13)
    np.testing.assert_allclose(st, s, atol=1e-13)


# --------------------------------------------------------------------------
# P-j: joint linearity in (V, S_0); L2-norm flag
# --------------------------------------------------------------------------

def test_linearity_in_values_and_initial_state():
    rng = np.random.default_rng(14)
    B, T, H, dk, dv = 1, 21, 2, 5, 4
    q, k, v1, g, beta = rand_inputs(rng, B, T, H, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    S1 = rng.standard_normal((B, H, dv, dk))
    S2 = rng.standard_normal((B, H, dv, dk))
    a, b = 0.7, -1.3
    o1, s1 = oracle.recurrent_fwd(q, k, v1, g, beta, init_state=S1)
    o2, s2 = oracle.recurrent_fwd(q, k, v2, g, beta, init_state=S2)
    o, s = oracle.recurrent_fwd(q, k, a * v1 + b * v2, g, beta, init_state=a * S1 + b * S2)
    np.testing.assert_allclose(o, a * o1 + b * o2, atol=1e-12)
    np.testing.assert_allclose(s, a * s1 + b * s2, atol=1e-12)


def test_l2norm_flag_is_scale_invariant_and_unit():
    rng = np.random.default_rng(15)
    B, T, H, dk, dv = 1, 12, 2, 8, 3
    q, k, v, g, beta = rand_inputs(rng, B, T, H, dk, dv, unit_keys=False)
    o_raw, s_raw = oracle.recurrent_fwd(q, k, v, g, beta, use_qk_l2norm=True, scale=0.25)
    # per-token rescaling of q and k (by large factors, so the 1e-6 epsilon is negligible)
    f = rng.uniform(50, 100, (B, T, H, 1))
    o_s, s_s = oracle.recurrent_fwd(q * f, k * f[..., ::-1, :], v, g, beta, use_qk_l2norm=True, scale=0.25)
    np.testing.assert_allclose(o_s, o_raw, atol=1e-7)
    np.testing.assert_allclose(s_s, s_raw, atol=1e-7)
    # unit-norm inputs with the flag on change only by the epsilon
    qn = q / np.linalg.norm(q, axis=-1, keepdims=True)
    kn = k / np.linalg.norm(k, axis=-1, keepdims=True)
    o_n, _ = oracle.recurrent_fwd(qn, kn, v, g, beta, use_qk_l2norm=False, scale=0.25)
    np.testing.assert_allclose(o_n, o_raw, atol=1e-5)


def test_rejects_bad_geometry():
    rng = np.random.default_rng(16)
    q, k, v, g, beta = rand_inputs(rng, 1, 8, 1, 4, 4)
    with pytest.raises(ValueError):
        oracle.recurrent_fwd(q, k, v, g, beta, cu_seqlens=np.array([0, 5, 7], np.int32))  # does not end at T


# --------------------------------------------------------------------------
# beta in (0, 2): the negative-eigenvalue range (paper page, §2.2, translator's
# note).  No new arithmetic; these pin the sign structure and the solve.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("b", [1.3, 1.9, 2.0])
def test_beta_up_to_two_negative_eigenvalue_along_key(b):
    """Unit k, v = 0: S_t k = alpha (1 - beta) S_{t-1} k (negative for beta > 1, a reflection at 2)
    and S_t x = alpha S_{t-1} x for x orthogonal to k."""
    rng = np.random.default_rng(17)
    dk, dv = 9, 4
    st = rng.standard_normal((1, 1, dv, dk))
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    x = rng.standard_normal(dk)
    x -= (x @ k) * k
    alpha = 0.9
    _, new = oracle.decode_step(st, x[None, None], k[None, None], np.zeros((1, 1, dv)),
                                np.array([[math.log(alpha)]]), np.array([[b]]))
    np.testing.assert_allclose(new[0, 0] @ k, alpha * (1 - b) * (st[0, 0] @ k), atol=1e-12)
    np.testing.assert_allclose(new[0, 0] @ x, alpha * (st[0, 0] @ x), atol=1e-12)


def test_beta_up_to_two_is_nonexpansive_without_writes():
    """With v = 0 and unit keys, ||I - beta k k^T||_2 = max(1, |1 - beta|) = 1 for beta in [0, 2],
    so the spectral norm of S never grows faster than alpha; beyond 2 it grows by |1 - beta|."""
    rng = np.random.default_rng(18)
    dk, dv, steps = 6, 5, 40
    st = rng.standard_normal((1, 1, dv, dk))
    for _ in range(steps):
        k = rng.standard_normal(dk)
        k /= np.linalg.norm(k)
        g = -0.05 * abs(rng.standard_normal())
        b = rng.uniform(0.0, 2.0)
        _, new = oracle.decode_step(st, k[None, None], k[None, None], np.zeros((1, 1, dv)),
                                    np.array([[g]]), np.array([[b]]))
        assert np.linalg.norm(new[0, 0], 2) <= math.exp(g) * np.linalg.norm(st[0, 0], 2) * (1 + 1e-12)
        st = new
    # contrast: a rank-one state along k is scaled by exactly alpha |1 - beta| (here 1.5 at beta = 2.5)
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    s1 = np.outer(rng.standard_normal(dv), k)[None, None]
    _, new = oracle.decode_step(s1, k[None, None], k[None, None], np.zeros((1, 1, dv)),
                                np.array([[0.0]]), np.array([[2.5]]))
    np.testing.assert_allclose(new[0, 0], -1.5 * s1[0, 0], atol=1e-12)


@pytest.mark.parametrize("C", [4, 16, 64])
@pytest.mark.parametrize("w_form", [0, 1])
def test_chunked_equals_recurrent_beta_up_to_two(C, w_form):
    rng = np.random.default_rng(19)
    B, T, H, dk, dv = 1, 70, 2, 8, 5
    q, k, v, g, beta = rand_inputs(rng, B, T, H, dk, dv, decay=0.5)
    beta = 2.0 * beta
    S0 = rng.standard_normal((B, H, dv, dk))
    o1, s1 = oracle.recurrent_fwd(q, k, v, g, beta, init_state=S0, scale=0.5)
    o2, s2 = oracle.chunked_fwd(q, k, v, g, beta, init_state=S0, scale=0.5, chunk_size=C, w_form=w_form)
    np.testing.assert_allclose(o2, o1, atol=1e-9)
    np.testing.assert_allclose(s2, s1, atol=1e-9)


def test_ut_solve_with_nearly_parallel_keys_and_beta_near_two():
    """The stress case of the (I + L) solve: |L_ij| approaches beta_i |k_i . k_j| ~ 2.  The UT
    transform still satisfies its defining systems, and the chunked form still equals the recurrence."""
    rng = np.random.default_rng(20)
    C, dk, dv = 64, 16, 8
    base = rng.standard_normal(dk)
    K = base[None, :] + 0.05 * rng.standard_normal((C, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = rng.standard_normal((C, dv))
    alpha = np.exp(-0.01 * np.abs(rng.standard_normal(C)))
    beta = rng.uniform(1.8, 2.0, C)
    W, U = oracle.ut_transform(K, V, alpha, beta, w_form=0)
    b = np.cumsum(np.log(alpha))
    Gamma = np.tril(np.exp(b[:, None] - b[None, :]))
    LG = np.eye(C) + np.tril(np.diag(beta) @ (Gamma * (K @ K.T)), -1)
    assert np.abs(LG - np.eye(C)).max() > 1.7                     # the regime this test is for
    np.testing.assert_allclose(LG @ U, beta[:, None] * V, atol=1e-9 * max(1.0, np.abs(U).max()))
    np.testing.assert_allclose(LG @ W, (beta * np.exp(b))[:, None] * K, atol=1e-9 * max(1.0, np.abs(W).max()))
    q = rng.standard_normal((1, C, 1, dk))
    g = np.log(alpha)[None, :, None]
    o1, s1 = oracle.recurrent_fwd(q, K[None, :, None], V[None, :, None], g, beta[None, :, None])
    o2, s2 = oracle.chunked_fwd(q, K[None, :, None], V[None, :, None], g, beta[None, :, None], chunk_size=64)
    np.testing.assert_allclose(o2, o1, atol=1e-8)
    np.testing.assert_allclose(s2, s1, atol=1e-8)
