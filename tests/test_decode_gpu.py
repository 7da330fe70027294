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
