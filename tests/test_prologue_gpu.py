"""GPU parity of the block prologue (gdn_prologue) against the fp64 oracle.

q, k, v = SiLU(short causal convolution of the projections), alpha in Mamba2's
parameterisation, beta by a sigmoid ([paper] §3.4 "Token mixing block").

Tolerances: q, k, v are rounded once to the output dtype, so bf16 outputs may
differ from the fp64 value by one rounding (relative 2^-8) plus the fp32
arithmetic before it; fp32 outputs by the fp32 arithmetic (expf, a K-term dot
product), well under 1e-5 relative.  g and beta are fp32: 1e-5 relative.  The
carried convolution state is a copy of inputs and must match exactly.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_12_gb300 as gdn
import oracle
from gpu_helpers import assert_close, cuda, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_12_gb300 import build
    build.build()
    gdn.load_library()


def make(B, T, H, dk, dv, K, dtype, seed, N=None, with_state=True):
    """Seeded raw projections, filters and gate parameters of one prologue call."""
    gen = torch.Generator().manual_seed(seed)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    rn = lambda *s: torch.randn(s, generator=gen, dtype=torch.float32)
    N = B if N is None else N
    d = dict(xq=rn(B, T, H, dk).to(td), xk=rn(B, T, H, dk).to(td), xv=rn(B, T, H, dv).to(td),
             wq=0.5 * rn(H, dk, K), wk=0.5 * rn(H, dk, K), wv=0.5 * rn(H, dv, K),
             a=rn(B, T, H), b=rn(B, T, H), A_log=0.5 * rn(H), dt_bias=0.5 * rn(H))
    d["state"] = rn(N, K - 1, H, 2 * dk + dv).to(td) if (with_state and K > 1) else None
    return d


def reference(d, dk, cu=None):
    """The oracle's prologue on the same (rounded) inputs; returns q, k, v, g, beta, state_out."""
    st = None if d["state"] is None else d["state"].double().numpy()
    outs = []
    for name, w, lo, hi in (("xq", "wq", 0, dk), ("xk", "wk", dk, 2 * dk), ("xv", "wv", 2 * dk, None)):
        si = None if st is None else st[..., lo:hi]
        outs.append(oracle.short_conv_silu(d[name], d[w], state_in=si, cu_seqlens=cu))
    g, beta = oracle.gate_activations(d["a"], d["b"], d["A_log"], d["dt_bias"])
    so = np.concatenate([o[1] for o in outs], axis=-1)
    return outs[0][0], outs[1][0], outs[2][0], g, beta, so


def check_qkv(got, ref, dtype, what):
    got, ref = to_np(got), np.asarray(ref)
    tol = 2.0 ** -8 if dtype == "bf16" else 1e-5
    err = np.abs(got - ref) - tol * np.abs(ref) - 1e-6
    assert err.max() <= 0, f"{what}: worst excess {err.max():.3e}"


def run_gpu(d, dtype, cu=None, want_state=True):
    dd = cuda(d)
    K = d["wq"].shape[-1]
    N = (cu.numel() - 1) if cu is not None else d["xq"].shape[0]
    H, dk, dv = d["xq"].shape[2], d["xq"].shape[3], d["xv"].shape[3]
    so = None
    if want_state and K > 1:
        so = torch.full((N, K - 1, H, 2 * dk + dv), float("nan"), device="cuda").to(d["xq"].dtype)
    q, k, v, g, beta = gdn.prologue(dd["xq"], dd["xk"], dd["xv"], dd["wq"], dd["wk"], dd["wv"], dd["a"], dd["b"],
                                    dd["A_log"], dd["dt_bias"], conv_state_in=dd["state"], conv_state_out=so,
                                    cu_seqlens=None if cu is None else cu.cuda())
    torch.cuda.synchronize()
    return q, k, v, g, beta, so


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 256), (8, 16)])
def test_prologue_against_oracle(dtype, K, dk, dv):
    d = make(B=2, T=75, H=3, dk=dk, dv=dv, K=K, dtype=dtype, seed=40 + K)
    q, k, v, g, beta, so = run_gpu(d, dtype)
    rq, rk, rv, rg, rb, rso = reference(d, dk)
    check_qkv(q, rq, dtype, "q")
    check_qkv(k, rk, dtype, "k")
    check_qkv(v, rv, dtype, "v")
    np.testing.assert_allclose(to_np(g), rg, rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(to_np(beta), rb, rtol=1e-5, atol=1e-7)
    if K > 1:
        np.testing.assert_array_equal(to_np(so), rso)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prologue_varlen_short_and_empty_sequences(dtype):
    lens = [5, 0, 1, 40, 2, 17, 0, 64]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    d = make(B=1, T=sum(lens), H=2, dk=64, dv=64, K=4, dtype=dtype, seed=49, N=len(lens))
    q, k, v, g, beta, so = run_gpu(d, dtype, cu=cu)
    rq, rk, rv, rg, rb, rso = reference(d, 64, cu=cu.numpy())
    check_qkv(q, rq, dtype, "q")
    check_qkv(k, rk, dtype, "k")
    check_qkv(v, rv, dtype, "v")
    np.testing.assert_array_equal(to_np(so), rso)   # empty sequences keep their history


def test_prologue_without_state_and_two_calls_carry():
    """Zero history without a state; two calls with the state carried equal one call."""
    d = make(B=2, T=50, H=2, dk=128, dv=128, K=4, dtype="bf16", seed=50, with_state=False)
    q, k, v, g, beta, so = run_gpu(d, "bf16")
    rq, rk, rv, _, _, rso = reference(d, 128)
    check_qkv(q, rq, "bf16", "q")
    check_qkv(v, rv, "bf16", "v")
    np.testing.assert_array_equal(to_np(so), rso)
    T1 = 13
    first = {n: (t[:, :T1].contiguous() if n in ("xq", "xk", "xv", "a", "b") else t) for n, t in d.items()}
    second = {n: (t[:, T1:].contiguous() if n in ("xq", "xk", "xv", "a", "b") else t) for n, t in d.items()}
    q1, k1, v1, _, _, so1 = run_gpu(first, "bf16")
    second["state"] = so1.cpu()
    q2, k2, v2, _, _, so2 = run_gpu(second, "bf16")
    assert torch.equal(torch.cat([q1, q2], 1), q) and torch.equal(torch.cat([v1, v2], 1), v)
    assert torch.equal(so2, so)


def test_prologue_feeds_the_chunked_forward():
    """Prologue then chunked forward (tensor-core path) against the oracle chain on the same
    projections, with the oracle's q, k, v rounded to bf16 where the device stores them."""
    B, T, H, dk, dv, K = 2, 300, 4, 128, 128, 4
    d = make(B, T, H, dk, dv, K, "bf16", seed=51)
    d["a"] = d["a"] - 2.0     # slower decay, as trained models start
    dd = cuda(d)
    q, k, v, g, beta = gdn.prologue(dd["xq"], dd["xk"], dd["xv"], dd["wq"], dd["wk"], dd["wv"], dd["a"], dd["b"],
                                    dd["A_log"], dd["dt_bias"], conv_state_in=dd["state"])
    out, sf = gdn.chunk_fwd(q, k, v, g, beta, scale=dk ** -0.5)
    torch.cuda.synchronize()
    rq, rk, rv, rg, rb, _ = reference(d, dk)
    bf = lambda x: torch.from_numpy(x).to(torch.bfloat16)
    ro, rs = oracle.recurrent_fwd(bf(rq), bf(rk), bf(rv), rg, rb, scale=dk ** -0.5, use_qk_l2norm=True)
    assert_close(out, ro, "bf16", "out")
    assert_close(sf, rs, "bf16", "final_state")
