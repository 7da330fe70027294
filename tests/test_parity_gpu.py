"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases span several chunks, ragged tails, varlen boundaries (including
length-0 and length-1 sequences), d_v > d_k, state carry and both dtypes.
Full-size workloads are checked on all units where the oracle is quick and on
sampled (sequence, head) units otherwise (units are independent).
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_12_gb300 as gdn
import oracle
from gated_delta_rule_12_gb300 import inputs
from gpu_helpers import assert_close, cuda, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_12_gb300 import build
    build.build()
    gdn.load_library()


def run_both(d, dk, scale=None, l2=True):
    scale = dk ** -0.5 if scale is None else scale
    dd = cuda(d)
    out, sf = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], init_state=dd["init_state"],
                            cu_seqlens=dd["cu_seqlens"], scale=scale, use_qk_l2norm=l2)
    torch.cuda.synchronize()
    ro, rs = oracle.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], init_state=d["init_state"],
                                  cu_seqlens=d["cu_seqlens"], scale=scale, use_qk_l2norm=l2)
    return out, sf, ro, rs


def test_headline_small_fp32_case_exact_config():
    """B=1, H=2, L=256, d=64, fp32, zero initial state, seed 0."""
    w = inputs.WORKLOADS["prefill_b1_h2_l256_d64_f32"]
    d = inputs.make(w)
    out, sf, ro, rs = run_both(d, w.dk)
    assert out.shape == (1, 256, 2, 64) and sf.shape == (1, 2, 64, 64)
    assert_close(out, ro, "f32", "out")
    assert_close(sf, rs, "f32", "final_state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 256), (128, 32), (256, 128), (256, 64)])
def test_prefill_ragged_with_initial_state(dtype, dk, dv):
    d = inputs.make_prefill(B=2, L=200, H=3, dk=dk, dv=dv, dtype=dtype, seed=11, decay=0.3, init_state=True)
    out, sf, ro, rs = run_both(d, dk)
    assert_close(out, ro, dtype, "out")
    assert_close(sf, rs, dtype, "final_state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 17, 64, 65])
def test_short_batched_sequences(dtype, L):
    """Equal-length batches shorter than, equal to and one past a chunk, on both chunk paths."""
    d = inputs.make_prefill(B=3, L=L, H=2, dk=128, dv=128, dtype=dtype, seed=19, decay=0.3, init_state=True)
    out, sf, ro, rs = run_both(d, 128)
    assert_close(out, ro, dtype, "out")
    assert_close(sf, rs, dtype, "final_state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_varlen_boundaries(dtype):
    lens = [1, 63, 64, 65, 0, 130, 7, 128]
    d = inputs.make_prefill(B=1, L=sum(lens), H=2, dk=128, dv=128, dtype=dtype, seed=12, decay=0.5,
                            init_state=True, num_seqs=len(lens), lengths=lens)
    out, sf, ro, rs = run_both(d, 128)
    assert_close(out, ro, dtype, "out")
    assert_close(sf, rs, dtype, "final_state")
    # a length-0 sequence keeps its initial state
    np.testing.assert_allclose(sf[4].cpu().numpy(), d["init_state"][4].numpy(), atol=0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_dk256_varlen_and_agreement_with_decode(dtype):
    """dk = 256 on the chunked forward (CUDA-core path): varlen with empty and 1-token sequences against
    the oracle, and the same tokens through the multi-token decode (which takes dk = 256 too) give the
    same outputs and final states."""
    lens = [1, 0, 70, 129]
    d = inputs.make_prefill(B=1, L=sum(lens), H=2, dk=256, dv=64, dtype=dtype, seed=57, decay=0.3,
                            init_state=True, num_seqs=len(lens), lengths=lens)
    out, sf, ro, rs = run_both(d, 256)
    assert_close(out, ro, dtype, "out")
    assert_close(sf, rs, dtype, "final_state")
    # equal-length batch through the decode path: 3 sequences of 20 tokens
    e = inputs.make_prefill(B=3, L=20, H=2, dk=256, dv=64, dtype=dtype, seed=58, decay=0.3, init_state=True)
    ee = cuda(e)
    o_c, s_c = gdn.chunk_fwd(ee["q"], ee["k"], ee["v"], ee["g"], ee["beta"], init_state=ee["init_state"])
    st = ee["init_state"].clone()
    o_d = gdn.decode_multi(st, ee["q"], ee["k"], ee["v"], ee["g"], ee["beta"])
    torch.cuda.synchronize()
    ro2, rs2 = oracle.recurrent_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], init_state=e["init_state"],
                                    scale=256 ** -0.5, use_qk_l2norm=True)
    assert_close(o_c, ro2, dtype, "chunked out")
    assert_close(o_d, ro2, dtype, "decode out")
    assert_close(s_c, rs2, dtype, "chunked state")
    assert_close(st, rs2, dtype, "decode state")


def test_heavy_decay_no_overflow():
    d = inputs.make_prefill(B=1, L=256, H=2, dk=128, dv=128, dtype="bf16", seed=13, decay=4.0)
    out, sf, ro, rs = run_both(d, 128)
    assert torch.isfinite(out.float()).all() and torch.isfinite(sf).all()
    assert_close(out, ro, "bf16", "out")
    assert_close(sf, rs, "bf16", "final_state")


def test_without_l2norm_on_prenormalised_inputs():
    d = inputs.make_prefill(B=1, L=150, H=2, dk=64, dv=64, dtype="f32", seed=14)
    d["q"] = d["q"] / d["q"].norm(dim=-1, keepdim=True)
    d["k"] = d["k"] / d["k"].norm(dim=-1, keepdim=True)
    out, sf, ro, rs = run_both(d, 64, l2=False)
    assert_close(out, ro, "f32", "out")
    assert_close(sf, rs, "f32", "final_state")


def test_empty_sequence_axis():
    d = inputs.make_prefill(B=2, L=0, H=2, dk=64, dv=64, dtype="f32", seed=15, init_state=True)
    dd = cuda(d)
    out, sf = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], init_state=dd["init_state"])
    torch.cuda.synchronize()
    assert out.numel() == 0
    np.testing.assert_array_equal(sf.cpu().numpy(), d["init_state"].numpy())


def test_state_carry_two_calls_equal_one():
    d = inputs.make_prefill(B=2, L=300, H=2, dk=128, dv=128, dtype="bf16", seed=16, init_state=True)
    dd = cuda(d)
    o, s = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], init_state=dd["init_state"])
    cut = 130
    sl = lambda t, a, b: t[:, a:b].contiguous()
    o1, s1 = gdn.chunk_fwd(*(sl(dd[n], 0, cut) for n in ("q", "k", "v", "g", "beta")), init_state=dd["init_state"])
    o2, s2 = gdn.chunk_fwd(*(sl(dd[n], cut, 300) for n in ("q", "k", "v", "g", "beta")), init_state=s1)
    torch.cuda.synchronize()
    ro, rs = oracle.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], init_state=d["init_state"],
                                  scale=128 ** -0.5, use_qk_l2norm=True)
    assert_close(torch.cat([o1, o2], 1), ro, "bf16", "split out")
    assert_close(s2, rs, "bf16", "split state")


def test_device_error_word_clear_after_call():
    d = cuda(inputs.make_prefill(B=1, L=128, H=1, dk=64, dv=64, dtype="f32", seed=17))
    ws = torch.full((gdn.chunk_fwd_workspace_size(1, 128, 1, 64, 64, 0, torch.float32),), 0xFF,
                    dtype=torch.uint8, device="cuda")
    gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], workspace=ws)
    gdn.check_device_error(ws)   # raises if the word is not clear


def test_bounded_wait_gives_up_and_reports_timeout():
    """The failure path without a fault: a kernel whose bounded wait (the one every mbarrier wait of
    the tensor-core kernels uses) sees a phase that nothing completes gives up after its limit, the
    error word reads back as GDN_ERR_DEVICE_TIMEOUT, and a chunked-forward call on the same workspace
    afterwards runs and matches the oracle: the context stays usable."""
    import time
    ws = torch.zeros((gdn.chunk_fwd_workspace_size(1, 128, 2, 128, 128, 0, torch.bfloat16),),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    gdn.selftest_wait_timeout(ws, limit_us=20000)
    with pytest.raises(gdn.GDNError) as err:
        gdn.check_device_error(ws)
    assert err.value.code == 5, err.value            # GDN_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 >= 0.02          # it waited out its limit
    gdn.check_device_error(ws)                        # reading the word cleared it
    d = inputs.make_prefill(B=1, L=128, H=2, dk=128, dv=128, dtype="bf16", seed=31, init_state=True)
    dd = cuda(d)
    out, sf = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], init_state=dd["init_state"],
                            workspace=ws)
    gdn.check_device_error(ws)
    ro, rs = oracle.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], init_state=d["init_state"],
                                  scale=128 ** -0.5, use_qk_l2norm=True)
    assert_close(out, ro, "bf16", "out after the timeout")
    assert_close(sf, rs, "bf16", "final_state after the timeout")


# ---------------------------------------------------------------------------
# full-size workloads
# ---------------------------------------------------------------------------

def test_full_prefill_b4_h16_l2048_all_units():
    w = inputs.WORKLOADS["prefill_b4_h16_l2048_d128_bf16"]
    d = inputs.make(w)
    out, sf, ro, rs = run_both(d, w.dk)
    assert_close(out, ro, "bf16", "out")
    assert_close(sf, rs, "bf16", "final_state")


def test_full_varlen_t32768_all_units():
    w = inputs.WORKLOADS["varlen_t32768_h16_d128_bf16"]
    d = inputs.make(w)
    out, sf, ro, rs = run_both(d, w.dk)
    assert_close(out, ro, "bf16", "out")
    assert_close(sf, rs, "bf16", "final_state")


def test_full_large_heavy_decay_sampled_units():
    """Every sequence of the large workload, 3 heads of each (24 of its 256 units, drawn without
    replacement; units are independent), through one oracle call over all 24."""
    w = inputs.WORKLOADS["prefill_b8_h32_l8192_dk128_dv256_bf16"]
    d = inputs.make(w)
    dd = cuda(d)
    out, sf = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], scale=w.scale, use_qk_l2norm=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(sf).all()
    rng = np.random.default_rng(4)
    picks = [(b, int(h)) for b in range(w.B) for h in rng.choice(w.H, size=3, replace=False)]
    # the picked units as 24 sequences of one head each
    sel = lambda t: torch.stack([t[b, :, h:h + 1] for b, h in picks]).contiguous()
    ro, rs = oracle.recurrent_fwd(sel(d["q"]), sel(d["k"]), sel(d["v"]), sel(d["g"]), sel(d["beta"]),
                                  scale=w.scale, use_qk_l2norm=True)
    out_h = out.cpu()
    sf_h = sf.cpu()
    got_o = torch.stack([out_h[b, :, h:h + 1] for b, h in picks])
    got_s = torch.stack([sf_h[b, h:h + 1] for b, h in picks])
    assert_close(got_o, ro, "bf16", "out (24 sampled units)")
    assert_close(got_s, rs, "bf16", "final_state (24 sampled units)")
    for i, (b, h) in enumerate(picks):   # and unit by unit
        assert_close(got_o[i], ro[i], "bf16", f"out[{b},{h}]")
        assert_close(got_s[i], rs[i], "bf16", f"state[{b},{h}]")


# ---------------------------------------------------------------------------
# beta in (0, 2): the negative-eigenvalue range (paper page, §2.2, translator's note)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("bf16", 128, 256), ("f32", 64, 64),
                                         ("f32", 128, 128), ("bf16", 64, 96)])
def test_beta_up_to_two(dtype, dk, dv):
    d = inputs.make_prefill(B=2, L=200, H=3, dk=dk, dv=dv, dtype=dtype, seed=23, decay=0.3,
                            init_state=True, beta_max=2.0)
    assert float(d["beta"].max()) > 1.5
    out, sf, ro, rs = run_both(d, dk)
    assert_close(out, ro, dtype, "out")
    assert_close(sf, rs, dtype, "final_state")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_beta_near_two_nearly_parallel_keys(dtype):
    """Stress of the UT solve: keys of each head nearly parallel and beta in (1.8, 2), so the
    strictly-lower system entries approach 2 in magnitude; several chunks, light decay.  Every
    intra-chunk product nearly cancels here (the output rms is ~0.03, an order of magnitude below the
    terms it is the difference of); the standard tolerances still apply."""
    d = inputs.make_prefill(B=1, L=320, H=2, dk=128, dv=128, dtype=dtype, seed=24, decay=0.02, beta_max=2.0)
    k = d["k"].float()
    k = k[:, :1] + 0.05 * k                      # every key close to the head's first key
    d["k"] = k.to(d["k"].dtype)
    d["beta"] = (1.8 + 0.1 * d["beta"]).contiguous()
    out, sf, ro, rs = run_both(d, 128)
    assert torch.isfinite(out.float()).all() and torch.isfinite(sf).all()
    assert_close(out, ro, dtype, "out")
    assert_close(sf, rs, dtype, "final_state")


def test_fp16_operand_range_is_reported():
    """Values far outside the fp16 range on the tensor-core path are reported as GDN_ERR_RANGE through
    the device error word (no fault, no hang), and the next ordinary call on the same workspace is
    clean and correct."""
    d = inputs.make_prefill(B=1, L=128, H=2, dk=128, dv=128, dtype="bf16", seed=37)
    big = dict(d, v=(d["v"].float() * 1e6).to(torch.bfloat16))
    ws = torch.zeros((gdn.chunk_fwd_workspace_size(1, 128, 2, 128, 128, 0, torch.bfloat16),),
                     dtype=torch.uint8, device="cuda")
    dd = cuda(big)
    gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], workspace=ws)
    with pytest.raises(gdn.GDNError) as err:
        gdn.check_device_error(ws)
    assert err.value.code == 6, err.value            # GDN_ERR_RANGE
    dd = cuda(d)
    out, sf = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], workspace=ws)
    gdn.check_device_error(ws)
    ro, rs = oracle.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=128 ** -0.5, use_qk_l2norm=True)
    assert_close(out, ro, "bf16", "out after the range error")
    assert_close(sf, rs, "bf16", "final_state after the range error")


@pytest.mark.parametrize("dtype,dk", [("bf16", 128), ("f32", 64)])
def test_degenerate_gates_and_vectors(dtype, dk):
    """The degenerate cases of eq. 10 ("Gated Delta Networks", §3.1), on the tensor-core path (bf16,
    dk = 128) and the CUDA-core path (fp32, dk = 64):
      * beta = 0 everywhere: nothing is written, the state only decays, so
        o_t = (prod_{s<=t} alpha_s) S_0 q^_t and the final state is (prod alpha) S_0 (closed form);
      * g = 0 everywhere (alpha = 1): the plain delta rule over several chunks;
      * zero keys and zero queries at some tokens: a zero key writes and erases nothing, a zero
        query reads exactly 0."""
    # beta = 0: the closed form, independently of the oracle
    d = inputs.make_prefill(B=2, L=150, H=2, dk=dk, dv=dk, dtype=dtype, seed=81, decay=0.05, init_state=True)
    d["beta"] = torch.zeros_like(d["beta"])
    out, sf, ro, rs = run_both(d, dk)
    assert_close(out, ro, dtype, "beta=0 out")
    assert_close(sf, rs, dtype, "beta=0 final_state")
    g = d["g"].double().numpy()                                    # [B, T, H]
    q = d["q"].double().numpy()
    qh = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6) * dk ** -0.5
    S0 = d["init_state"].double().numpy()                          # [B, H, dv, dk]
    decay = np.exp(np.cumsum(g, axis=1))                           # prod_{s<=t} alpha_s
    closed = np.einsum("bth,bhvk,bthk->bthv", decay, S0, qh)
    assert_close(out, closed, dtype, "beta=0 out vs closed form")
    assert_close(sf, S0 * decay[:, -1][..., None, None], dtype, "beta=0 final_state vs closed form")
    # alpha = 1
    d = inputs.make_prefill(B=1, L=320, H=2, dk=dk, dv=dk, dtype=dtype, seed=82, init_state=True)
    d["g"] = torch.zeros_like(d["g"])
    out, sf, ro, rs = run_both(d, dk)
    assert_close(out, ro, dtype, "g=0 out")
    assert_close(sf, rs, dtype, "g=0 final_state")
    # zero keys and queries
    d = inputs.make_prefill(B=2, L=200, H=2, dk=dk, dv=dk, dtype=dtype, seed=83, decay=0.2, init_state=True)
    zk, zq = [3, 64, 65, 127, 199], [0, 5, 63, 64, 130]
    d["k"][:, zk] = 0
    d["q"][:, zq] = 0
    out, sf, ro, rs = run_both(d, dk)
    assert_close(out, ro, dtype, "zero k/q out")
    assert_close(sf, rs, dtype, "zero k/q final_state")
    assert (out[:, zq].float() == 0).all(), "a zero query must read exactly 0"
