"""GPU parity of the single-token decode step against the fp64 oracle."""
import numpy as np
import pytest
import torch

import gated_delta_rule_12_gb300 as gdn
import oracle
from gated_delta_rule_12_gb300 import inputs
from gpu_helpers import assert_close, cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_12_gb300 import build
    build.build()
    gdn.load_library()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (256, 64), (128, 256), (64, 8)])
def test_decode_steps_against_oracle(dtype, dk, dv):
    steps = 5
    d = inputs.make_decode(N=7, H=3, dk=dk, dv=dv, steps=steps, dtype=dtype, seed=21)
    dd = cuda(d)
    st = dd["state0"].clone()
    ref = d["state0"].double().numpy()
    scale = dk ** -0.5
    for t in range(steps):
        o = gdn.decode_step(st, dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], scale=scale)
        ro, ref = oracle.decode_step(ref, d["q"][t], d["k"][t], d["v"][t], d["g"][t], d["beta"][t],
                                     scale=scale, use_qk_l2norm=True)
        assert_close(o, ro, dtype, f"out step {t}")
    torch.cuda.synchronize()
    assert_close(st, ref, dtype, "state")


def test_decode_full_workload_sampled_sequences_and_chunked_agreement():
    """64 steps on N=256, H=16, d=128: sampled sequences against the oracle, and
    the whole final state against the chunked forward over the same 64 tokens."""
    w = inputs.WORKLOADS["decode_n256_h16_d128_bf16"]
    d = inputs.make(w)
    dd = cuda(d)
    st = dd["state0"].clone()
    outs = []
    for t in range(w.steps):
        outs.append(gdn.decode_step(st, dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t],
                                    scale=w.scale))
    torch.cuda.synchronize()
    O = torch.stack(outs, 0)                      # [steps, N, H, dv]
    picks = [0, 17, 128, 255]
    for n in picks:
        sel = lambda t: t[:, n:n + 1].permute(1, 0, 2, 3).contiguous()   # [1, steps, H, d]
        ro, rs = oracle.recurrent_fwd(sel(d["q"]), sel(d["k"]), sel(d["v"]),
                                      d["g"][:, n:n + 1].permute(1, 0, 2).contiguous(),
                                      d["beta"][:, n:n + 1].permute(1, 0, 2).contiguous(),
                                      init_state=d["state0"][n:n + 1], scale=w.scale, use_qk_l2norm=True)
        assert_close(O[:, n], ro[0], "bf16", f"decode out seq {n}")
        assert_close(st[n:n + 1], rs, "bf16", f"decode state seq {n}")
    # chunked forward over the same tokens, as N sequences of 64 tokens
    perm = lambda t: t.permute(1, 0, *range(2, t.dim())).contiguous()
    oc, sc = gdn.chunk_fwd(perm(dd["q"]), perm(dd["k"]), perm(dd["v"]), perm(dd["g"]), perm(dd["beta"]),
                           init_state=dd["state0"], scale=w.scale, use_qk_l2norm=True)
    torch.cuda.synchronize()
    assert_close(sc, st.double().cpu().numpy(), "bf16", "chunked vs decode state")
    assert_close(oc, perm(O).double().cpu().numpy(), "bf16", "chunked vs decode out")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_beta_up_to_two(dtype):
    """beta in (0, 2) (negative eigenvalues along k) over 16 steps."""
    steps = 16
    d = inputs.make_decode(N=5, H=2, dk=128, dv=128, steps=steps, dtype=dtype, seed=25, beta_max=2.0)
    dd = cuda(d)
    st = dd["state0"].clone()
    ref = d["state0"].double().numpy()
    for t in range(steps):
        o = gdn.decode_step(st, dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], scale=128 ** -0.5)
        ro, ref = oracle.decode_step(ref, d["q"][t], d["k"][t], d["v"][t], d["g"][t], d["beta"][t],
                                     scale=128 ** -0.5, use_qk_l2norm=True)
        assert_close(o, ro, dtype, f"out step {t}")
    torch.cuda.synchronize()
    assert_close(st, ref, dtype, "state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_degenerate_cases(dtype):
    """The step's degenerate cases ("Gated DeltaNet：先忘一点，再按误差更新记忆", "为什么再加一个遗忘门？"):
    beta = 0 writes nothing (S <- alpha S and o = alpha S q, a closed form); alpha = 1 (g = 0) is the
    plain delta rule; a zero key leaves S as alpha S; a zero query reads exactly 0."""
    steps = 6
    d = inputs.make_decode(N=3, H=2, dk=128, dv=128, steps=steps, dtype=dtype, seed=27)
    d["beta"][0] = 0          # step 0: beta = 0 everywhere
    d["g"][1] = 0             # step 1: alpha = 1
    d["k"][2, 1] = 0          # step 2: sequence 1's keys are zero
    d["q"][3, 2] = 0          # step 3: sequence 2's queries are zero
    dd = cuda(d)
    st = dd["state0"].clone()
    ref = d["state0"].double().numpy()
    for t in range(steps):
        prev = st.double().cpu().numpy()
        o = gdn.decode_step(st, dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], scale=128 ** -0.5)
        ro, ref = oracle.decode_step(ref, d["q"][t], d["k"][t], d["v"][t], d["g"][t], d["beta"][t],
                                     scale=128 ** -0.5, use_qk_l2norm=True)
        torch.cuda.synchronize()
        assert_close(o, ro, dtype, f"out step {t}")
        assert_close(st, ref, dtype, f"state step {t}")
        if t == 0:   # beta = 0: the closed form from the kernel's own previous state
            a = np.exp(d["g"][0].double().numpy())[..., None, None]
            q = d["q"][0].double().numpy()
            qh = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6) * 128 ** -0.5
            assert_close(st, a * prev, dtype, "beta=0 state vs alpha S")
            assert_close(o, np.einsum("nhvk,nhk->nhv", a * prev, qh), dtype, "beta=0 out vs alpha S q")
        if t == 3:
            assert (o[2].float() == 0).all(), "a zero query must read exactly 0"


# ---------------------------------------------------------------------------
# several tokens per call ("Decode 递归": ordered composition of steps)
# ---------------------------------------------------------------------------

def _multi_inputs(N, T, H, dk, dv, dtype, seed, beta_max=1.0):
    """Token-major [N, T, H, d] inputs of one multi-token call, from the decode generator."""
    d = inputs.make_decode(N=N, H=H, dk=dk, dv=dv, steps=T, dtype=dtype, seed=seed, beta_max=beta_max)
    tm = lambda x: x.transpose(0, 1).contiguous()     # [T, N, ...] -> [N, T, ...]
    return {"q": tm(d["q"]), "k": tm(d["k"]), "v": tm(d["v"]), "g": tm(d["g"]), "beta": tm(d["beta"]),
            "state0": d["state0"]}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 4, 7, 16])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (256, 64)])
def test_decode_multi_against_oracle_and_single_steps(dtype, T, dk, dv):
    d = _multi_inputs(N=6, T=T, H=3, dk=dk, dv=dv, dtype=dtype, seed=26, beta_max=2.0)
    dd = cuda(d)
    scale = dk ** -0.5
    st = dd["state0"].clone()
    out = gdn.decode_multi(st, dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], scale=scale)
    # the same T tokens as T single steps: identical arithmetic per token, so identical bits
    st1 = dd["state0"].clone()
    outs = [gdn.decode_step(st1, dd["q"][:, t].contiguous(), dd["k"][:, t].contiguous(),
                            dd["v"][:, t].contiguous(), dd["g"][:, t].contiguous(),
                            dd["beta"][:, t].contiguous(), scale=scale) for t in range(T)]
    torch.cuda.synchronize()
    assert torch.equal(out, torch.stack(outs, 1))
    assert torch.equal(st, st1)
    # and the fp64 recurrence over the T tokens
    ro, rs = oracle.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], init_state=d["state0"],
                                  scale=scale, use_qk_l2norm=True)
    assert_close(out, ro, dtype, "out")
    assert_close(st, rs, dtype, "state")


def test_decode_multi_full_size_matches_chunked_forward():
    """N=256, H=16, d=128, 4 tokens per call x 16 calls against the chunked forward over the same
    64 tokens, and sampled sequences against the oracle."""
    N, H, d_, T, calls = 256, 16, 128, 4, 16
    d = _multi_inputs(N=N, T=T * calls, H=H, dk=d_, dv=d_, dtype="bf16", seed=27)
    dd = cuda(d)
    st = dd["state0"].clone()
    outs = []
    for c in range(calls):
        sl = lambda x: x[:, c * T:(c + 1) * T].contiguous()
        outs.append(gdn.decode_multi(st, sl(dd["q"]), sl(dd["k"]), sl(dd["v"]), sl(dd["g"]), sl(dd["beta"])))
    O = torch.cat(outs, 1)
    co, cs = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], init_state=dd["state0"],
                           scale=d_ ** -0.5)
    torch.cuda.synchronize()
    assert_close(O, co.float().cpu().double().numpy(), "bf16", "out vs chunked")
    assert_close(st, cs.cpu().double().numpy(), "bf16", "state vs chunked")
    for n in (0, 99, 255):
        sel = lambda x: x[n:n + 1]
        ro, rs = oracle.recurrent_fwd(sel(d["q"]), sel(d["k"]), sel(d["v"]), sel(d["g"]), sel(d["beta"]),
                                      init_state=d["state0"][n:n + 1], scale=d_ ** -0.5, use_qk_l2norm=True)
        assert_close(O[n:n + 1], ro, "bf16", f"out seq {n}")
        assert_close(st[n:n + 1], rs, "bf16", f"state seq {n}")
