"""GPU parity of the block prologue fused into the chunked forward (gdn_prologue_chunk_fwd).

The fused call must give, bit for bit, what gdn_prologue followed by gdn_chunk_fwd gives (the short
convolution, SiLU and gate activations are the same arithmetic, and q, k, v are rounded to bf16 at
the same point), and match the fp64 oracle chain -- the oracle's short convolution + SiLU and gate
activations ([paper] §3.4 "Token mixing block", Fig. 1) feeding its token-by-token recurrence, run
on the bf16-rounded q, k, v -- at the standard bf16 tolerance.  The carried convolution state must
equal the oracle's exactly (it is a copy of inputs).  Cases: equal-length batches with a ragged last
chunk, varlen with empty, 1-token and sub-halo sequences, a carried convolution state and initial
state, every convolution width 1-4, d_v = 256.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_12_gb300 as gdn
import oracle
from gpu_helpers import assert_close, cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_12_gb300 import build
    build.build()
    gdn.load_library()


def make(B, T, H, dv, K, seed, N=None, lengths=None, with_state=True, with_init=True):
    gen = torch.Generator().manual_seed(seed)
    rn = lambda *s: torch.randn(s, generator=gen, dtype=torch.float32)
    dk = 128
    N = B if N is None else N
    d = dict(xq=rn(B, T, H, dk).to(torch.bfloat16), xk=rn(B, T, H, dk).to(torch.bfloat16),
             xv=rn(B, T, H, dv).to(torch.bfloat16), wq=0.5 * rn(H, dk, K), wk=0.5 * rn(H, dk, K),
             wv=0.5 * rn(H, dv, K), a=rn(B, T, H), b=rn(B, T, H), A_log=0.5 * rn(H) - 1.0, dt_bias=0.5 * rn(H))
    d["state"] = rn(N, K - 1, H, 2 * dk + dv).to(torch.bfloat16) if (with_state and K > 1) else None
    d["init"] = 0.02 * rn(N, H, dv, dk) if with_init else None
    d["cu"] = None
    if lengths is not None:
        cu = [0]
        for x in lengths:
            cu.append(cu[-1] + x)
        d["cu"] = torch.tensor(cu, dtype=torch.int32)
    return d


def run_fused(d):
    dd = cuda(d)
    K = d["wq"].shape[-1]
    B, T, H, dk = d["xq"].shape
    dv = d["xv"].shape[-1]
    N = (d["cu"].numel() - 1) if d["cu"] is not None else B
    so = torch.full((N, K - 1, H, 2 * dk + dv), float("nan"), device="cuda").to(torch.bfloat16) if K > 1 else None
    out, sf = gdn.prologue_chunk_fwd(dd["xq"], dd["xk"], dd["xv"], dd["wq"], dd["wk"], dd["wv"], dd["a"], dd["b"],
                                     dd["A_log"], dd["dt_bias"], conv_state_in=dd["state"], conv_state_out=so,
                                     init_state=dd["init"], cu_seqlens=dd["cu"])
    torch.cuda.synchronize()
    return out, sf, so


def run_separate(d):
    dd = cuda(d)
    q, k, v, g, beta = gdn.prologue(dd["xq"], dd["xk"], dd["xv"], dd["wq"], dd["wk"], dd["wv"], dd["a"], dd["b"],
                                    dd["A_log"], dd["dt_bias"], conv_state_in=dd["state"], cu_seqlens=dd["cu"])
    out, sf = gdn.chunk_fwd(q, k, v, g, beta, init_state=dd["init"], cu_seqlens=dd["cu"])
    torch.cuda.synchronize()
    return out, sf


def oracle_chain(d):
    dk = d["xq"].shape[-1]
    st = None if d["state"] is None else d["state"].double().numpy()
    ys, sos = [], []
    for name, w, lo, hi in (("xq", "wq", 0, dk), ("xk", "wk", dk, 2 * dk), ("xv", "wv", 2 * dk, None)):
        si = None if st is None else st[..., lo:hi]
        y, so = oracle.short_conv_silu(d[name], d[w], state_in=si, cu_seqlens=d["cu"])
        ys.append(torch.from_numpy(np.ascontiguousarray(y)).to(torch.bfloat16))   # bf16-rounded inputs of the rule
        sos.append(so)
    g, beta = oracle.gate_activations(d["a"], d["b"], d["A_log"], d["dt_bias"])
    ro, rs = oracle.recurrent_fwd(ys[0], ys[1], ys[2], g, beta, init_state=d["init"], cu_seqlens=d["cu"],
                                  scale=dk ** -0.5, use_qk_l2norm=True)
    return ro, rs, np.concatenate(sos, axis=-1)


CASES = [
    dict(B=2, T=200, H=2, dv=128, K=4, seed=51),                                        # ragged last chunk
    dict(B=1, T=sum([0, 1, 2, 70, 130, 64]), H=2, dv=128, K=4, seed=52, N=6,
         lengths=[0, 1, 2, 70, 130, 64]),                                               # varlen: empty, sub-halo
    dict(B=1, T=300, H=1, dv=256, K=3, seed=53),                                        # dv = 256
    dict(B=2, T=130, H=2, dv=128, K=2, seed=54, with_state=False, with_init=False),     # zero states
    dict(B=1, T=129, H=2, dv=128, K=1, seed=55),                                        # no history
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c['B']}T{c['T']}H{c['H']}dv{c['dv']}K{c['K']}")
def test_fused_prologue_matches_separate_calls_and_oracle(case):
    d = make(**case)
    out, sf, so = run_fused(d)
    out_s, sf_s = run_separate(d)
    # the same arithmetic as gdn_prologue + gdn_chunk_fwd: identical bits
    assert torch.equal(out.view(torch.int16), out_s.view(torch.int16)), "out differs from prologue + chunk_fwd"
    assert torch.equal(sf.view(torch.int32), sf_s.view(torch.int32)), "final state differs from prologue + chunk_fwd"
    ro, rs, ros = oracle_chain(d)
    assert_close(out, ro, "bf16", "out vs oracle chain")
    assert_close(sf, rs, "bf16", "final_state vs oracle chain")
    if so is not None:
        np.testing.assert_array_equal(so.double().cpu().numpy(), ros)


def test_fused_prologue_full_bench_shape_all_units():
    """B=4, H=16, L=2048, dk=dv=128, K=4 (the bench workload's shape)."""
    d = make(B=4, T=2048, H=16, dv=128, K=4, seed=56)
    out, sf, so = run_fused(d)
    out_s, sf_s = run_separate(d)
    assert torch.equal(out.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(sf.view(torch.int32), sf_s.view(torch.int32))
    ro, rs, ros = oracle_chain(d)
    assert_close(out, ro, "bf16", "out vs oracle chain")
    assert_close(sf, rs, "bf16", "final_state vs oracle chain")
    np.testing.assert_array_equal(so.double().cpu().numpy(), ros)
