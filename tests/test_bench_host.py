"""Host-side checks of bench.py's per-unit work formulas (no GPU).

The algorithmic bytes and FLOP that the roofline divides by are recomputed here from the
workload shapes, term by term, and compared with bench.py's functions:
- q, k, v and out once at the element size;
- g and beta as fp32;
- the fp32 state read once when an initial state is given, and written once.
The FLOP figure counts the dense tiles of one chunk per token-head: the Gram and QK products,
the W and U products, the state products, and the output product.
"""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from gated_delta_rule_12_gb300 import inputs  # noqa: E402

W = inputs.WORKLOADS


def test_prefill_bytes_of_the_bench_workload():
    # B4 H16 L2048 d128 bf16, zero initial state: 8192 x 16 token-heads of
    # (2*128 + 2*128) bf16 values and two fp32 gates, plus 4 x 16 fp32 128x128 final states
    token_heads = 4 * 2048 * 16
    io = token_heads * ((128 + 128 + 128 + 128) * 2 + 4 + 4)
    states = 4 * 16 * 128 * 128 * 4
    assert bench.prefill_algorithmic_bytes(W["prefill_b4_h16_l2048_d128_bf16"]) == io + states == 139_460_608


def test_prefill_bytes_count_the_initial_state_when_given():
    # varlen: 32768 tokens, 8 sequences with nonzero initial states (read once and written once)
    io = 32768 * 16 * (4 * 128 * 2 + 8)
    states = 8 * 16 * 128 * 128 * 4 * 2
    assert bench.prefill_algorithmic_bytes(W["varlen_t32768_h16_d128_bf16"]) == io + states


def test_prefill_bytes_with_distinct_head_sizes_and_fp32():
    w = W["prefill_b8_h32_l8192_dk128_dv256_bf16"]
    assert bench.prefill_algorithmic_bytes(w) == 8 * 8192 * 32 * ((2 * 128 + 2 * 256) * 2 + 8) + 8 * 32 * 256 * 128 * 4
    w0 = W["prefill_b1_h2_l256_d64_f32"]
    assert bench.prefill_algorithmic_bytes(w0) == 256 * 2 * (4 * 64 * 4 + 8) + 2 * 64 * 64 * 4


def test_decode_bytes_single_and_multi_token():
    w = W["decode_n256_h16_d128_bf16"]
    state_rw = 2 * 128 * 128 * 4
    tok = 4 * 128 * 2 + 8
    assert bench.decode_algorithmic_bytes(w) == 256 * 16 * (state_rw + tok) == 541_097_984
    for T in (1, 4, 16):
        assert bench.decode_multi_algorithmic_bytes(w, T) == 256 * 16 * (state_rw + T * tok)
    assert bench.decode_multi_algorithmic_bytes(w, 1) == bench.decode_algorithmic_bytes(w)


def test_prefill_flops_of_the_bench_workload():
    # per token-head with chunk C: K K^T and Q K^T (2 C dk each), W (2 C dk), U (2 C dv),
    # the intra-chunk output (2 C dv), and S W^T, S q, V_new^T K (2 dk dv each)
    w = W["prefill_b4_h16_l2048_d128_bf16"]
    C, dk, dv = 64, 128, 128
    per_th = 2 * C * dk * 3 + 2 * C * dv * 2 + 2 * dk * dv * 3
    assert bench.prefill_algorithmic_flops(w) == 4 * 2048 * 16 * per_th
    assert abs(bench.prefill_algorithmic_flops(w) / 1e9 - 23.62) < 0.01


@pytest.mark.parametrize("units,world,ms,expect", [(8192, 1, 0.1, 8.192e7), (8192, 4, 0.2, 1.6384e8)])
def test_job_throughput(units, world, ms, expect):
    assert bench.job_throughput(units, world, ms) == pytest.approx(expect)
