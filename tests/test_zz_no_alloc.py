"""gdn_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate.

Some callers may not call cudaMalloc (or anything that allocates) where they
run the operator -- plugin hosts and serving runtimes that plan all device
memory up front, bindings without a device allocator -- so they cannot pass a
workspace.  The no-alloc entry point uses a fixed scratch array inside the
library's device image instead.  These tests check it through the C ABI
against the regular entry point, on two calls in a row (the array keeps the
previous call's contents, so the second call shows nothing stale leaks), and
that a problem too large for the array is refused before any work.

This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import gated_delta_rule_12_gb300 as gdn
from gated_delta_rule_12_gb300 import inputs
from gpu_helpers import assert_close, cuda


def _lib():
    from gated_delta_rule_12_gb300 import build
    build.build()
    return gdn.load_library()


def _call_noalloc(lib, d, out, sf, dt, scale):
    q = d["q"]
    B, T, H, dk = q.shape
    dv = d["v"].shape[-1]
    cu = d["cu_seqlens"]
    p = lambda t: None if t is None else t.data_ptr()
    return lib.gdn_chunk_fwd_noalloc(p(q), p(d["k"]), p(d["v"]), p(d["g"]), p(d["beta"]), p(d["init_state"]),
                                     p(cu), (cu.numel() - 1) if cu is not None else 0, p(out), p(sf),
                                     B, T, H, dk, dv, dt, ctypes.c_float(scale), 1, 64,
                                     torch.cuda.current_stream().cuda_stream)


def test_noalloc_rejects_problems_beyond_the_fixed_scratch():
    lib = _lib()
    fake = 1 << 20   # never dereferenced: the size check comes first
    rc = lib.gdn_chunk_fwd_noalloc(fake, fake, fake, fake, fake, None, None, 0, fake, None,
                                   8, 8192, 32, 128, 256, gdn.GDN_BF16, ctypes.c_float(0.1), 1, 64, None)
    assert rc == 3   # GDN_ERR_WORKSPACE
    # the header's scratch formula: 256 B + 64 * (12 + 4 * (dk + dv)) B per chunk slot and head
    need = lambda B, T, H, dk, dv: 256 + B * -(-T // 64) * H * 64 * (12 + 4 * (dk + dv))
    assert need(8, 8192, 32, 128, 256) > gdn.NOALLOC_SCRATCH_BYTES
    assert need(1, 2048, 8, 128, 128) < gdn.NOALLOC_SCRATCH_BYTES < need(1, 2048, 16, 128, 128)


@pytest.mark.gpu
def test_noalloc_matches_chunk_fwd_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib()
    cases = [
        ("bf16", inputs.make_prefill(B=2, L=200, H=3, dk=128, dv=128, dtype="bf16", seed=31, init_state=True)),
        ("f32", inputs.make_prefill(B=1, L=sum([5, 64, 131]), H=2, dk=64, dv=64, dtype="f32", seed=32,
                                    init_state=True, num_seqs=3, lengths=[5, 64, 131])),
    ]
    for dtype, host in cases:
        d = cuda(host)
        dk = d["q"].shape[-1]
        scale = dk ** -0.5
        ref_out, ref_sf = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], init_state=d["init_state"],
                                        cu_seqlens=d["cu_seqlens"], scale=scale, use_qk_l2norm=True)
        out = torch.full_like(ref_out, float("nan"))
        sf = torch.full_like(ref_sf, float("nan"))
        rc = _call_noalloc(lib, d, out, sf, gdn.GDN_BF16 if dtype == "bf16" else gdn.GDN_F32, scale)
        assert rc == 0, gdn.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        assert_close(out, ref_out.double().cpu().numpy(), dtype, f"noalloc out ({dtype})")
        assert_close(sf, ref_sf.double().cpu().numpy(), dtype, f"noalloc state ({dtype})")
