"""GPU parity of the chunked backward (gdn_chunk_bwd) against the fp64 oracle's
reverse-mode gradients (themselves pinned against finite differences).

Tolerances.  fp32 inputs: the gradients pass through a few more fp32 products
than the forward (the UT transform's adjoint, two scans), so they are checked
at relative L2 <= 2e-4 and max-abs <= 2e-4 of the largest reference entry.
bf16 inputs: the oracle runs on the same bf16-rounded inputs; dq, dk, dv are
returned in bf16 (one rounding, 2^-8 relative) and the arithmetic is fp32, so
relative L2 <= 5e-3 and max-abs <= 1e-2 of the largest reference entry.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_12_gb300 as gdn
import oracle
from gated_delta_rule_12_gb300 import inputs
import gpu_helpers
from gpu_helpers import cuda, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_12_gb300 import build
    build.build()
    gdn.load_library()


TOL = {"f32": (2e-4, 2e-4), "bf16": (5e-3, 1e-2)}


def check(got, ref, dtype, what):
    ref = np.asarray(ref)
    maxabs, rel = errors(got, ref)
    rl, ma = TOL[dtype]
    scale = max(float(np.abs(ref).max()), 1e-30)
    # logged with the max-abs bound in absolute terms (it is relative to the largest reference entry)
    gpu_helpers.record(what, dtype, maxabs, rel, rl, ma * scale)
    assert rel <= rl and maxabs <= ma * scale, f"{what}: rel-L2 {rel:.3e}, max-abs {maxabs:.3e} (ref max {scale:.3e})"


def grads(d, dO, dS, dk, l2=True, want_dinit=True):
    scale = dk ** -0.5
    dd = cuda(d)
    out = gdn.chunk_bwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dO.cuda(),
                        init_state=dd["init_state"], dfinal_state=None if dS is None else dS.cuda(),
                        cu_seqlens=dd["cu_seqlens"], scale=scale, use_qk_l2norm=l2, want_dinit=want_dinit)
    torch.cuda.synchronize()
    ref = oracle.recurrent_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], dO, init_state=d["init_state"],
                               dfinal=dS, cu_seqlens=d["cu_seqlens"], scale=scale, use_qk_l2norm=l2)
    return out, ref


def cotangents(d, seed, with_state=True):
    gen = torch.Generator().manual_seed(seed)
    B, T, H, dv = d["v"].shape
    dk = d["q"].shape[-1]
    N = (d["cu_seqlens"].numel() - 1) if d["cu_seqlens"] is not None else B
    dO = torch.randn((B, T, H, dv), generator=gen).to(d["q"].dtype)
    dS = torch.randn((N, H, dv, dk), generator=gen) if with_state else None
    return dO, dS


def check_all(out, ref, dtype):
    dq, dk, dv, dg, db, dinit = out
    check(dq, ref["dq"], dtype, "dq")
    check(dk, ref["dk"], dtype, "dk")
    check(dv, ref["dv"], dtype, "dv")
    check(dg, ref["dg"], dtype, "dg")
    check(db, ref["dbeta"], dtype, "dbeta")
    if dinit is not None:
        check(dinit, ref["dinit"], dtype, "dinit")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 256), (256, 64), (256, 256)])
def test_bwd_ragged_with_states(dtype, dk, dv):
    d = inputs.make_prefill(B=2, L=150, H=2, dk=dk, dv=dv, dtype=dtype, seed=70, decay=0.3, init_state=True)
    dO, dS = cotangents(d, 71)
    out, ref = grads(d, dO, dS, dk)
    check_all(out, ref, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 17, 65])
def test_bwd_short_batched_sequences(dtype, L):
    """Equal-length batches shorter than a chunk and one past it, with both state gradients."""
    d = inputs.make_prefill(B=3, L=L, H=2, dk=128, dv=64, dtype=dtype, seed=76, decay=0.3, init_state=True)
    dO, dS = cotangents(d, 77)
    out, ref = grads(d, dO, dS, 128)
    check_all(out, ref, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_varlen_beta_up_to_two(dtype):
    lens = [1, 63, 64, 65, 0, 130, 7]
    d = inputs.make_prefill(B=1, L=sum(lens), H=2, dk=128, dv=128, dtype=dtype, seed=72, decay=0.5,
                            init_state=True, num_seqs=len(lens), lengths=lens, beta_max=2.0)
    dO, dS = cotangents(d, 73)
    out, ref = grads(d, dO, dS, 128)
    check_all(out, ref, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_beta_near_two_nearly_parallel_keys(dtype):
    """The conditioning stress of the UT solve ("Gated Delta Networks", §2.2, beta in (0, 2)) for the
    gradients: keys of each head nearly parallel and beta in (1.8, 2), so the strictly-lower system
    entries approach 2 in magnitude and the chunk-local products nearly cancel; standard tolerances."""
    d = inputs.make_prefill(B=1, L=320, H=2, dk=128, dv=128, dtype=dtype, seed=24, decay=0.02, beta_max=2.0)
    k = d["k"].float()
    d["k"] = (k[:, :1] + 0.05 * k).to(d["k"].dtype)
    d["beta"] = (1.8 + 0.1 * d["beta"]).contiguous()
    dO, dS = cotangents(d, 77)
    out, ref = grads(d, dO, dS, 128)
    check_all(out, ref, dtype)


def test_bwd_without_l2norm_and_without_state_gradients():
    d = inputs.make_prefill(B=1, L=200, H=3, dk=64, dv=64, dtype="f32", seed=74, decay=0.2)
    d["q"] = d["q"] / d["q"].norm(dim=-1, keepdim=True)
    d["k"] = d["k"] / d["k"].norm(dim=-1, keepdim=True)
    dO, _ = cotangents(d, 75, with_state=False)
    out, ref = grads(d, dO, None, 64, l2=False, want_dinit=False)
    check_all(out, ref, "f32")


def test_bwd_full_size_sampled_heads():
    """B=4, H=16, L=2048, d=128 bf16 (the bench shape): every gradient of sampled
    (sequence, head) units against the oracle (units are independent)."""
    w = inputs.WORKLOADS["prefill_b4_h16_l2048_d128_bf16"]
    d = inputs.make(w)
    dO, dS = cotangents(d, 76)
    dd = cuda(d)
    out = gdn.chunk_bwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dO.cuda(), dfinal_state=dS.cuda(),
                        scale=w.scale)
    torch.cuda.synchronize()
    for n, h in ((0, 0), (1, 7), (3, 15)):
        sel = lambda t: t[n:n + 1, :, h:h + 1].contiguous()
        ref = oracle.recurrent_bwd(sel(d["q"]), sel(d["k"]), sel(d["v"]), sel(d["g"]), sel(d["beta"]), sel(dO),
                                   dfinal=dS[n:n + 1, h:h + 1], scale=w.scale, use_qk_l2norm=True)
        got = [t[n:n + 1, :, h:h + 1] for t in out[:5]] + [out[5][n:n + 1, h:h + 1]]
        check_all(got, ref, "bf16")


@pytest.mark.parametrize("L", [1, 17, 65])
def test_bwd_tensor_core_path_short_sequences(L):
    """bf16 with dk = dv = 128 runs the tensor-core prep, reverse scan and local kernels: one-token
    chunks, a ragged single chunk and a ragged second chunk, with initial and final state gradients."""
    d = inputs.make_prefill(B=3, L=L, H=2, dk=128, dv=128, dtype="bf16", seed=77, decay=0.3, init_state=True)
    dO, dS = cotangents(d, 78)
    out, ref = grads(d, dO, dS, 128)
    check_all(out, ref, "bf16")


def test_bwd_tensor_core_path_without_l2norm_and_without_state_gradients():
    """The tensor-core kernels without the L2 normalisation (pre-normalised inputs), no final-state
    cotangent and no initial-state gradient requested."""
    d = inputs.make_prefill(B=2, L=130, H=2, dk=128, dv=128, dtype="f32", seed=79, decay=0.2)
    d["q"] = (d["q"] / d["q"].norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    d["k"] = (d["k"] / d["k"].norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    d["v"] = d["v"].to(torch.bfloat16)
    dO, _ = cotangents(d, 80, with_state=False)
    out, ref = grads(d, dO, None, 128, l2=False, want_dinit=False)
    check_all(out, ref, "bf16")
