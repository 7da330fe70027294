"""Host-side checks of the seeded input recipe (no GPU): the workload table against the stated
configurations, and the generators' shapes, ranges, structure and determinism; and the profiling
driver's refusal to run without a GPU."""
import math

import pytest
import torch

from gated_delta_rule_12_gb300 import inputs

W = inputs.WORKLOADS


def test_workload_table_matches_the_configurations():
    w0 = W["prefill_b1_h2_l256_d64_f32"]
    assert (w0.B, w0.L, w0.H, w0.dk, w0.dv, w0.dtype, w0.seed, w0.init_state) == (1, 256, 2, 64, 64, "f32", 0, False)
    w1 = W["prefill_b4_h16_l2048_d128_bf16"]
    assert (w1.B, w1.L, w1.H, w1.dk, w1.dv, w1.dtype, w1.init_state) == (4, 2048, 16, 128, 128, "bf16", False)
    w2 = W["varlen_t32768_h16_d128_bf16"]
    assert (w2.kind, w2.L, w2.num_seqs, w2.H, w2.dk, w2.dv, w2.init_state) == ("varlen", 32768, 8, 16, 128, 128, True)
    w3 = W["decode_n256_h16_d128_bf16"]
    assert (w3.kind, w3.num_seqs, w3.steps, w3.H, w3.dk, w3.dv) == ("decode", 256, 64, 16, 128, 128)
    w4 = W["prefill_b8_h32_l8192_dk128_dv256_bf16"]
    assert (w4.B, w4.L, w4.H, w4.dk, w4.dv, w4.decay) == (8, 8192, 32, 128, 256, 1.0)
    assert all(w.chunk_size == 64 for w in W.values())
    assert all(w.decay == 0.1 for n, w in W.items() if n != w4.name)
    assert w1.scale == 1.0 / math.sqrt(128)


def test_prefill_generator_shapes_ranges_and_rounding():
    d = inputs.make_prefill(B=2, L=100, H=3, dk=64, dv=32, dtype="bf16", seed=5, init_state=True)
    assert d["q"].shape == (2, 100, 3, 64) and d["v"].shape == (2, 100, 3, 32)
    assert d["q"].dtype == d["k"].dtype == d["v"].dtype == torch.bfloat16
    assert d["g"].dtype == d["beta"].dtype == torch.float32 and d["g"].shape == (2, 100, 3)
    assert bool((d["g"] <= 0).all()) and bool(((d["beta"] > 0) & (d["beta"] < 1)).all())
    assert d["init_state"].shape == (2, 3, 32, 64) and d["cu_seqlens"] is None
    assert abs(float(d["init_state"].std()) - 0.02) < 0.002
    # g = -0.1 softplus(z): the mean of softplus(N(0,1)) is about 0.806
    assert abs(float(-d["g"].mean()) / 0.1 - 0.806) < 0.05
    f = inputs.make_prefill(B=1, L=10, H=1, dk=8, dv=8, dtype="f32", seed=5)
    assert f["q"].dtype == torch.float32 and f["init_state"] is None


def test_generators_are_deterministic_per_seed():
    a = inputs.make_prefill(B=1, L=70, H=2, dk=16, dv=16, dtype="bf16", seed=9, init_state=True)
    b = inputs.make_prefill(B=1, L=70, H=2, dk=16, dv=16, dtype="bf16", seed=9, init_state=True)
    c = inputs.make_prefill(B=1, L=70, H=2, dk=16, dv=16, dtype="bf16", seed=10, init_state=True)
    for n in ("q", "k", "v", "g", "beta", "init_state"):
        assert torch.equal(a[n], b[n])
    assert not torch.equal(a["q"], c["q"])


def test_varlen_lengths_sum_exactly_and_stay_in_range():
    d = inputs.make_prefill(B=1, L=32768, H=1, dk=8, dv=8, dtype="bf16", seed=2, num_seqs=8, init_state=True)
    cu = d["cu_seqlens"]
    assert cu.dtype == torch.int32 and cu.numel() == 9 and int(cu[0]) == 0 and int(cu[-1]) == 32768
    lens = (cu[1:] - cu[:-1]).tolist()
    assert all(x >= 1 for x in lens)
    # drawn in [512, 8192] and rescaled by 32768 / sum (a factor between 0.5 and 8)
    assert all(256 <= x <= 65536 for x in lens)
    assert d["init_state"].shape == (8, 1, 8, 8)


def test_beta_up_to_two_and_decode_generator():
    g, beta = inputs.draw_gates((1000,), 0.5, torch.Generator().manual_seed(1), beta_max=2.0)
    assert bool(((beta > 0) & (beta < 2)).all()) and float(beta.max()) > 1.0
    d = inputs.make_decode(N=4, H=2, dk=16, dv=8, steps=3, dtype="bf16", seed=3)
    assert d["q"].shape == (3, 4, 2, 16) and d["v"].shape == (3, 4, 2, 8) and d["g"].shape == (3, 4, 2)
    assert d["state0"].shape == (4, 2, 8, 16) and d["state0"].dtype == torch.float32


def test_profile_case_refuses_to_run_without_a_gpu(monkeypatch):
    """The profiling driver runs entry points on a GPU only; without one it stops with a message
    instead of falling back to anything on the host."""
    import torch
    from gated_delta_rule_12_gb300 import profile_case
    monkeypatch.setattr(torch.cuda, "is_available", lambda: False)
    with pytest.raises(SystemExit) as e:
        profile_case.main(["--op", "bwd", "--B", "1", "--L", "64"])
    assert "CUDA device" in str(e.value)


def test_profile_case_rejects_unknown_ops():
    from gated_delta_rule_12_gb300 import profile_case
    with pytest.raises(SystemExit):
        profile_case.main(["--op", "prefill"])
