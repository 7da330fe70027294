"""gdn_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate.

Some callers may not call cudaMalloc (or anything that allocates) where they
run the operator -- plugin hosts and serving runtimes that plan all device
memory up front, bindings without a device allocator -- so they cannot pass a
workspace.  The no-alloc entry point uses a fixed scratch array inside the
library's device image instead.  That array is shared by every call and keeps
the previous call's contents, so these tests call it several times in a row
through the C ABI and compare every result with the fp64 oracle (and with the
regular entry point):

  * A, then B (another size and dtype), then A again: the second A must match
    the first bit for bit, so nothing B left in the array leaks into A;
  * a problem whose last chunk is short right after one whose last chunk was
    nearly full, so the padded rows of the short chunk sit over non-zero
    leftovers.

A problem too large for the array is refused before any work.  This file is
collected last on purpose, so a run that stops at the first failure has run
every other test before it.
"""
import ctypes

import numpy as np
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


def test_noalloc_wrapper_checks_dtypes_before_any_launch():
    """The Python wrapper refuses an int64 cu_seqlens, non-fp32 gates or states and mis-shaped
    outputs before it passes pointers on (the kernels would misread them); no GPU is needed."""
    _lib()
    d = inputs.make_prefill(B=1, L=70, H=2, dk=64, dv=64, dtype="f32", seed=41, init_state=True,
                            num_seqs=2, lengths=[30, 40])
    out = torch.empty((1, 70, 2, 64))
    sf = torch.empty((2, 2, 64, 64))
    args = lambda **kw: dict(dict(q=d["q"], k=d["k"], v=d["v"], g=d["g"], beta=d["beta"], out=out,
                                  final_state=sf, init_state=d["init_state"], cu_seqlens=d["cu_seqlens"]), **kw)
    with pytest.raises(TypeError, match="cu_seqlens"):
        gdn.chunk_fwd_noalloc(**args(cu_seqlens=d["cu_seqlens"].to(torch.int64)))
    with pytest.raises(TypeError, match="g must be float32"):
        gdn.chunk_fwd_noalloc(**args(g=d["g"].to(torch.bfloat16)))
    with pytest.raises(TypeError, match="init_state"):
        gdn.chunk_fwd_noalloc(**args(init_state=d["init_state"].double()))
    with pytest.raises(ValueError, match="final_state"):
        gdn.chunk_fwd_noalloc(**args(final_state=torch.empty((1, 2, 64, 64))))
    with pytest.raises(ValueError, match="out"):
        gdn.chunk_fwd_noalloc(**args(out=torch.empty((1, 69, 2, 64))))
    with pytest.raises(ValueError, match="pass out"):
        gdn.chunk_fwd_noalloc(**args(out=None))
    with pytest.raises(TypeError, match="cu_seqlens"):
        gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"].to(torch.int64))


def _oracle(host, scale):
    import oracle
    return oracle.recurrent_fwd(host["q"], host["k"], host["v"], host["g"], host["beta"],
                                init_state=host["init_state"], cu_seqlens=host["cu_seqlens"], scale=scale,
                                use_qk_l2norm=True)


def _run(lib, host, dtype):
    """One no-alloc call through the C ABI into NaN-filled outputs; checked against the oracle and the
    regular entry point.  Returns the outputs."""
    d = cuda(host)
    dk = d["q"].shape[-1]
    scale = dk ** -0.5
    B, T, H, _ = d["q"].shape
    N = (d["cu_seqlens"].numel() - 1) if d["cu_seqlens"] is not None else B
    out = torch.full((B, T, H, d["v"].shape[-1]), float("nan"), dtype=d["q"].dtype, device="cuda")
    sf = torch.full((N, H, d["v"].shape[-1], dk), float("nan"), dtype=torch.float32, device="cuda")
    rc = _call_noalloc(lib, d, out, sf, gdn.GDN_BF16 if dtype == "bf16" else gdn.GDN_F32, scale)
    assert rc == 0, gdn.STATUS.get(rc, rc)
    torch.cuda.synchronize()
    ro, rs = _oracle(host, scale)
    assert_close(out, ro, dtype, f"noalloc out vs oracle ({dtype})")
    assert_close(sf, rs, dtype, f"noalloc state vs oracle ({dtype})")
    ref_out, ref_sf = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], init_state=d["init_state"],
                                    cu_seqlens=d["cu_seqlens"], scale=scale, use_qk_l2norm=True)
    torch.cuda.synchronize()
    assert_close(out, ref_out.double().cpu().numpy(), dtype, f"noalloc out vs gdn_chunk_fwd ({dtype})")
    assert_close(sf, ref_sf.double().cpu().numpy(), dtype, f"noalloc state vs gdn_chunk_fwd ({dtype})")
    return out, sf


@pytest.mark.gpu
def test_noalloc_calls_in_a_row_match_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib()
    a = inputs.make_prefill(B=2, L=200, H=3, dk=128, dv=128, dtype="bf16", seed=31, init_state=True)
    b = inputs.make_prefill(B=1, L=sum([5, 64, 131]), H=2, dk=64, dv=64, dtype="f32", seed=32,
                            init_state=True, num_seqs=3, lengths=[5, 64, 131])
    out_a1, sf_a1 = _run(lib, a, "bf16")
    _run(lib, b, "f32")
    out_a2, sf_a2 = _run(lib, a, "bf16")
    # the same problem again, after another one used the array: bit for bit the same result
    assert torch.equal(out_a1.view(torch.int16), out_a2.view(torch.int16))
    assert torch.equal(sf_a1.view(torch.int32), sf_a2.view(torch.int32))


@pytest.mark.gpu
def test_noalloc_short_tail_after_a_long_one():
    """A last chunk of 62 tokens, then one of 2 tokens in the same slots: the short chunk's padded
    rows lie over the previous call's data, which must not reach the result."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib()
    long_tail = inputs.make_prefill(B=2, L=190, H=2, dk=128, dv=128, dtype="f32", seed=33, decay=0.3,
                                    init_state=True)
    short_tail = inputs.make_prefill(B=2, L=130, H=2, dk=128, dv=128, dtype="f32", seed=34, decay=0.3,
                                     init_state=True)
    _run(lib, long_tail, "f32")
    out, sf = _run(lib, short_tail, "f32")
    assert np.isfinite(out.cpu().numpy()).all() and np.isfinite(sf.cpu().numpy()).all()
