"""GB300 (sm_103a) gated delta rule: Python binding of libgdn.so.

This module only marshals arguments: it checks tensor placement, dtype and
contiguity, allocates outputs/workspace with PyTorch when the caller does not
pass them, and calls the C ABI declared in ``include/gdn.h`` through ctypes on
the current PyTorch CUDA stream.  Every step of the computation runs in the
library's CUDA kernels; there is no other code path.  If ``libgdn.so`` cannot
be loaded the calls raise: there is no fallback.

Entry points (same names as the C ABI, without the ``gdn_`` prefix):
    chunk_fwd(q, k, v, g, beta, ...)      -> (out, final_state)
    decode_step(state, q, k, v, g, beta)  -> out            (state updated in place)
    decode_multi(state, q, k, v, g, beta) -> out [N,T,H,dv] (T tokens per call, state in place)
    prologue(xq, xk, xv, wq, wk, wv, a, b, A_log, dt_bias, ...) -> (q, k, v, g, beta)
    prologue_chunk_fwd(xq, xk, xv, wq, wk, wv, a, b, A_log, dt_bias, ...) -> (out, final_state)
                                          (prologue fused into the chunked forward)
    chunk_fwd_workspace_size(...)         -> bytes
    chunk_fwd_kernel_count(...)           -> kernels one chunk_fwd call launches
    chunk_bwd(q, k, v, g, beta, dout, ...) -> (dq, dk, dv, dg, dbeta, dinit_state)
    check_device_error(workspace)         -> None or raises
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgdn.so")

GDN_OK = 0
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_WORKSPACE",
          4: "GDN_ERR_CUDA", 5: "GDN_ERR_DEVICE_TIMEOUT", 6: "GDN_ERR_RANGE"}
GDN_F32, GDN_BF16 = 0, 1
CHUNK = 64

EXPORTS = ["gdn_status_string", "gdn_chunk_fwd_workspace_size", "gdn_chunk_fwd_kernel_count", "gdn_chunk_fwd",
           "gdn_chunk_bwd_workspace_size", "gdn_chunk_bwd", "gdn_decode_step", "gdn_decode_multi", "gdn_prologue",
           "gdn_check_device_error", "gdn_chunk_fwd_noalloc", "gdn_prologue_chunk_fwd_workspace_size",
           "gdn_prologue_chunk_fwd"]
NOALLOC_SCRATCH_BYTES = 32 << 20


class GDNError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what} failed: {STATUS.get(code, code)}")


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_f32 = ctypes.c_float
_sz = ctypes.c_size_t


def load_library(path: str = LIB_PATH, build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libgdn.so (optionally building it first) and declare the ABI."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            if build_if_missing:
                from . import build as _b
                path = _b.build()
            else:
                raise RuntimeError(f"libgdn.so not found at {path}; run gated_delta_rule_12_gb300.build.build()")
        lib = ctypes.CDLL(path)
        lib.gdn_status_string.argtypes = [ctypes.c_int]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_chunk_fwd_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int]
        lib.gdn_chunk_fwd_workspace_size.restype = _sz
        lib.gdn_chunk_fwd_kernel_count.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int]
        lib.gdn_chunk_fwd_kernel_count.restype = _i32
        lib.gdn_chunk_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
                                      _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _f32, _i32, _i32,
                                      _vp, _sz, _vp]
        lib.gdn_chunk_fwd.restype = ctypes.c_int
        lib.gdn_chunk_bwd_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int]
        lib.gdn_chunk_bwd_workspace_size.restype = _sz
        lib.gdn_chunk_bwd.argtypes = [_vp] * 6 + [_vp, _i32] + [_vp] * 8 + [_i32] * 5 + [ctypes.c_int, _f32, _i32, _i32,
                                                                                         _vp, _sz, _vp]
        lib.gdn_chunk_bwd.restype = ctypes.c_int
        lib.gdn_decode_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _i32, _i32, _i32, _i32, ctypes.c_int, _f32, _i32, _vp]
        lib.gdn_decode_step.restype = ctypes.c_int
        lib.gdn_decode_multi.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                         _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _f32, _i32, _vp]
        lib.gdn_decode_multi.restype = ctypes.c_int
        lib.gdn_prologue.argtypes = [_vp] * 12 + [_vp, _i32] + [_vp] * 5 + [_i32] * 6 + [ctypes.c_int, _vp]
        lib.gdn_prologue.restype = ctypes.c_int
        lib.gdn_check_device_error.argtypes = [_vp, _vp]
        lib.gdn_check_device_error.restype = ctypes.c_int
        lib.gdn_selftest_wait_timeout.argtypes = [_vp, ctypes.c_uint32, _vp]
        lib.gdn_selftest_wait_timeout.restype = ctypes.c_int
        lib.gdn_chunk_fwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
                                              _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _f32, _i32, _i32,
                                              _vp]
        lib.gdn_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.gdn_prologue_chunk_fwd_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int]
        lib.gdn_prologue_chunk_fwd_workspace_size.restype = _sz
        lib.gdn_prologue_chunk_fwd.argtypes = [_vp] * 13 + [_vp, _i32, _vp, _vp] + [_i32] * 6 + \
            [ctypes.c_int, _f32, _i32, _i32, _vp, _sz, _vp]
        lib.gdn_prologue_chunk_fwd.restype = ctypes.c_int
        _lib = lib
        return lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GDN_F32
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)



def _check_chunk_args(q, k, v, g, beta, init_state, cu_seqlens, out, final_state):
    """The checks every chunked-forward wrapper makes before it hands raw pointers to the C ABI:
    dtypes (the kernels read cu_seqlens as int32 and g, beta and the states as fp32, so any other
    dtype would be misread on the device), shapes, placement and contiguity."""
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k must be [B,T,H,dk] and v [B,T,H,dv]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    _dt(q)
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be [N+1] with N >= 1")
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    for t, what in ((g, "g"), (beta, "beta")):
        if t.dtype != torch.float32:
            raise TypeError(f"{what} must be float32")
        if tuple(t.shape) != (B, T, H):
            raise ValueError(f"{what} must be [B,T,H]")
    for t, what in ((init_state, "init_state"), (final_state, "final_state")):
        if t is None:
            continue
        if t.dtype != torch.float32:
            raise TypeError(f"{what} must be float32")
        if tuple(t.shape) != (N, H, dv, dk):
            raise ValueError(f"{what} must be [N,H,dv,dk] = {(N, H, dv, dk)}")
    if out is not None:
        if out.dtype != q.dtype:
            raise TypeError("out must have the dtype of q")
        if tuple(out.shape) != (B, T, H, dv):
            raise ValueError(f"out must be [B,T,H,dv] = {(B, T, H, dv)}")
    _need_cuda(q, k, v, g, beta, init_state, cu_seqlens, out, final_state)

def chunk_fwd_workspace_size(B, T, H, dk, dv, num_seqs=0, dtype=torch.bfloat16) -> int:
    dt = GDN_BF16 if dtype == torch.bfloat16 else GDN_F32
    return int(load_library().gdn_chunk_fwd_workspace_size(B, T, H, dk, dv, num_seqs, dt))


def chunk_fwd_kernel_count(B, T, H, dk, dv, num_seqs=0, dtype=torch.bfloat16) -> int:
    """Kernels one ``chunk_fwd`` call of this size launches (0 if unsupported)."""
    dt = GDN_BF16 if dtype == torch.bfloat16 else GDN_F32
    return int(load_library().gdn_chunk_fwd_kernel_count(B, T, H, dk, dv, num_seqs, dt))


def chunk_fwd(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale=None, use_qk_l2norm=True,
              out=None, final_state=None, output_final_state=True, workspace=None, chunk_size=CHUNK,
              stream=None):
    """Chunked forward of the gated delta rule (see ``gdn_chunk_fwd`` in include/gdn.h).

    q, k [B,T,H,dk], v [B,T,H,dv] (fp32 or bf16); g, beta [B,T,H] fp32;
    init_state [N,H,dv,dk] fp32 or None; cu_seqlens int32 [N+1] (device) or None.
    Returns ``(out, final_state)``; final_state is None if not requested.
    """
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if scale is None:
        scale = dk ** -0.5
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device)
    _check_chunk_args(q, k, v, g, beta, init_state, cu_seqlens, out, final_state)
    dt = _dt(q)
    num_seqs = N if cu_seqlens is not None else 0
    need = int(lib.gdn_chunk_fwd_workspace_size(B, T, H, dk, dv, num_seqs, dt))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib.gdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                           _ptr(cu_seqlens), num_seqs, _ptr(out), _ptr(final_state),
                           B, T, H, dk, dv, dt, float(scale), int(bool(use_qk_l2norm)), int(chunk_size),
                           _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_chunk_fwd")
    return out, final_state


def chunk_bwd(q, k, v, g, beta, dout, init_state=None, dfinal_state=None, cu_seqlens=None, scale=None,
              use_qk_l2norm=True, want_dinit=True, workspace=None, chunk_size=CHUNK, stream=None):
    """Backward of ``chunk_fwd`` (``gdn_chunk_bwd``): returns ``(dq, dk, dv, dg, dbeta, dinit_state)``
    for the loss gradients ``dout`` [B,T,H,dv] and ``dfinal_state`` [N,H,dv,dk] (or None)."""
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if scale is None:
        scale = dk ** -0.5
    dq, dkk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    db = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    dinit = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device) if want_dinit else None
    for t in (g, beta, init_state, dfinal_state):
        if t is not None and t.dtype != torch.float32:
            raise TypeError("g, beta and states must be float32")
    if dout.dtype != q.dtype:
        raise TypeError("dout must have the dtype of q")
    _need_cuda(q, k, v, g, beta, dout, init_state, dfinal_state, cu_seqlens)
    dt = _dt(q)
    num_seqs = N if cu_seqlens is not None else 0
    need = int(lib.gdn_chunk_bwd_workspace_size(B, T, H, dk, dv, num_seqs, dt))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib.gdn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state), _ptr(cu_seqlens),
                           num_seqs, _ptr(dout), _ptr(dfinal_state), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dg),
                           _ptr(db), _ptr(dinit), B, T, H, dk, dv, dt, float(scale), int(bool(use_qk_l2norm)),
                           int(chunk_size), _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_chunk_bwd")
    return dq, dkk, dvv, dg, db, dinit


def decode_step(state, q, k, v, g, beta, scale=None, use_qk_l2norm=True, out=None, stream=None):
    """One decode token per (sequence, head); ``state`` [N,H,dv,dk] fp32 is updated in place.

    q, k [N,H,dk], v [N,H,dv] (fp32 or bf16); g, beta [N,H] fp32.  Returns out [N,H,dv].
    """
    lib = load_library()
    N, H, dv, dk = state.shape
    if scale is None:
        scale = dk ** -0.5
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    if state.dtype != torch.float32 or g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("state, g and beta must be float32")
    _need_cuda(state, q, k, v, g, beta, out)
    rc = lib.gdn_decode_step(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(out),
                             N, H, dk, dv, _dt(q), float(scale), int(bool(use_qk_l2norm)), _stream(stream))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_decode_step")
    return out


def decode_multi(state, q, k, v, g, beta, scale=None, use_qk_l2norm=True, out=None, stream=None):
    """T decode tokens per (sequence, head) in one call; ``state`` [N,H,dv,dk] fp32 is updated in place.

    q, k [N,T,H,dk], v [N,T,H,dv] (fp32 or bf16); g, beta [N,T,H] fp32.  Returns out [N,T,H,dv],
    the same as T successive ``decode_step`` calls.
    """
    lib = load_library()
    N, H, dv, dk = state.shape
    T = q.shape[1]
    if scale is None:
        scale = dk ** -0.5
    if out is None:
        out = torch.empty((N, T, H, dv), dtype=q.dtype, device=q.device)
    if state.dtype != torch.float32 or g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("state, g and beta must be float32")
    if q.shape != (N, T, H, dk) or k.shape != (N, T, H, dk) or v.shape != (N, T, H, dv) or g.shape != (N, T, H) \
            or beta.shape != (N, T, H) or out.shape != (N, T, H, dv):
        raise ValueError("decode_multi: inconsistent shapes")
    _need_cuda(state, q, k, v, g, beta, out)
    rc = lib.gdn_decode_multi(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(out),
                              N, T, H, dk, dv, _dt(q), float(scale), int(bool(use_qk_l2norm)), _stream(stream))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_decode_multi")
    return out


def prologue(xq, xk, xv, wq, wk, wv, a, b, A_log, dt_bias, conv_state_in=None, conv_state_out=None,
             cu_seqlens=None, out=None, stream=None):
    """Block prologue (``gdn_prologue``): q, k, v = SiLU(short causal conv of the projections),
    g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b), in one pass.

    xq, xk [B,T,H,dk], xv [B,T,H,dv] (fp32 or bf16); wq, wk [H,dk,K], wv [H,dv,K] fp32;
    a, b [B,T,H] fp32; A_log, dt_bias [H] fp32; conv states [N,K-1,H,2dk+dv] (dtype of x) or None.
    Returns ``(q, k, v, g, beta)``; ``out`` may pass those five tensors preallocated.
    """
    lib = load_library()
    B, T, H, dk = xq.shape
    dv = xv.shape[-1]
    K = wq.shape[-1]
    if out is None:
        out = (torch.empty_like(xq), torch.empty_like(xk), torch.empty_like(xv),
               torch.empty((B, T, H), dtype=torch.float32, device=xq.device),
               torch.empty((B, T, H), dtype=torch.float32, device=xq.device))
    q, k, v, g, beta = out
    for t in (wq, wk, wv, a, b, A_log, dt_bias, g, beta):
        if t.dtype != torch.float32:
            raise TypeError("filters, gate projections, gate parameters and g, beta must be float32")
    if wq.shape != (H, dk, K) or wk.shape != (H, dk, K) or wv.shape != (H, dv, K):
        raise ValueError("prologue: filters must be [H, d, K]")
    _need_cuda(xq, xk, xv, wq, wk, wv, a, b, A_log, dt_bias, conv_state_in, conv_state_out, cu_seqlens,
               q, k, v, g, beta)
    num_seqs = (cu_seqlens.numel() - 1) if cu_seqlens is not None else 0
    rc = lib.gdn_prologue(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(a), _ptr(b),
                          _ptr(A_log), _ptr(dt_bias), _ptr(conv_state_in), _ptr(conv_state_out),
                          _ptr(cu_seqlens), num_seqs, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                          B, T, H, dk, dv, K, _dt(xq), _stream(stream))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_prologue")
    return q, k, v, g, beta


def prologue_chunk_fwd(xq, xk, xv, wq, wk, wv, a, b, A_log, dt_bias, conv_state_in=None, conv_state_out=None,
                       init_state=None, cu_seqlens=None, scale=None, use_qk_l2norm=True, out=None, final_state=None,
                       output_final_state=True, workspace=None, chunk_size=CHUNK, stream=None):
    """Block prologue and chunked forward in one call (``gdn_prologue_chunk_fwd``): the result of
    ``prologue`` followed by ``chunk_fwd``, without q, k, v, g, beta ever being written out.

    xq, xk [B,T,H,dk], xv [B,T,H,dv] bf16 (dk = 128, dv a multiple of 128); wq, wk [H,dk,K], wv [H,dv,K]
    fp32; a, b [B,T,H] fp32; A_log, dt_bias [H] fp32; conv states [N,K-1,H,2dk+dv] bf16 or None;
    init_state [N,H,dv,dk] fp32 or None; cu_seqlens int32 [N+1] or None.  Returns ``(out, final_state)``.
    """
    lib = load_library()
    B, T, H, dk = xq.shape
    dv = xv.shape[-1]
    K = wq.shape[-1]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if scale is None:
        scale = dk ** -0.5
    if xq.dtype != torch.bfloat16 or xk.dtype != torch.bfloat16 or xv.dtype != torch.bfloat16:
        raise TypeError("prologue_chunk_fwd: projections must be bfloat16")
    for t in (wq, wk, wv, a, b, A_log, dt_bias, init_state, final_state):
        if t is not None and t.dtype != torch.float32:
            raise TypeError("filters, gate projections, gate parameters and states must be float32")
    if wq.shape != (H, dk, K) or wk.shape != (H, dk, K) or wv.shape != (H, dv, K):
        raise ValueError("prologue_chunk_fwd: filters must be [H, d, K]")
    if a.shape != (B, T, H) or b.shape != (B, T, H) or A_log.shape != (H,) or dt_bias.shape != (H,):
        raise ValueError("prologue_chunk_fwd: gate shapes")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    for t in (conv_state_in, conv_state_out):
        if t is not None and (t.dtype != torch.bfloat16 or tuple(t.shape) != (N, K - 1, H, 2 * dk + dv)):
            raise ValueError("conv states must be bfloat16 [N, K-1, H, 2dk+dv]")
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=xq.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dv, dk), dtype=torch.float32, device=xq.device)
    _need_cuda(xq, xk, xv, wq, wk, wv, a, b, A_log, dt_bias, conv_state_in, conv_state_out, init_state, cu_seqlens,
               out, final_state)
    num_seqs = N if cu_seqlens is not None else 0
    need = int(lib.gdn_prologue_chunk_fwd_workspace_size(B, T, H, dk, dv, num_seqs, GDN_BF16))
    if need == 0:
        raise GDNError(2, "gdn_prologue_chunk_fwd (unsupported size)")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=xq.device)
    rc = lib.gdn_prologue_chunk_fwd(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(a), _ptr(b),
                                    _ptr(A_log), _ptr(dt_bias), _ptr(conv_state_in), _ptr(conv_state_out),
                                    _ptr(init_state), _ptr(cu_seqlens), num_seqs, _ptr(out), _ptr(final_state),
                                    B, T, H, dk, dv, K, GDN_BF16, float(scale), int(bool(use_qk_l2norm)),
                                    int(chunk_size), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_prologue_chunk_fwd")
    return out, final_state


def check_device_error(workspace, stream=None):
    rc = load_library().gdn_check_device_error(_ptr(workspace), _stream(stream))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_check_device_error")


def selftest_wait_timeout(workspace, limit_us=20000, stream=None):
    """``gdn_selftest_wait_timeout``: enqueue a kernel whose bounded wait on a phase that nothing
    completes gives up after ``limit_us`` and records the timeout in ``workspace``'s error word
    (read back by ``check_device_error``, which then raises GDN_ERR_DEVICE_TIMEOUT)."""
    _need_cuda(workspace)
    rc = load_library().gdn_selftest_wait_timeout(_ptr(workspace), int(limit_us), _stream(stream))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_selftest_wait_timeout")


def chunk_fwd_noalloc(q, k, v, g, beta, out, final_state=None, init_state=None, cu_seqlens=None, scale=None,
                      use_qk_l2norm=True, chunk_size=CHUNK, stream=None):
    """``gdn_chunk_fwd_noalloc``: the chunked forward with the library's fixed
    device scratch array instead of a workspace, for callers that cannot
    allocate.  The caller passes every output buffer; nothing is allocated.
    Problems needing more than ``NOALLOC_SCRATCH_BYTES`` of scratch are
    rejected (GDN_ERR_WORKSPACE).  Calls that overlap on the GPU race."""
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = dk ** -0.5
    if out is None:
        raise ValueError("chunk_fwd_noalloc allocates nothing: pass out")
    _check_chunk_args(q, k, v, g, beta, init_state, cu_seqlens, out, final_state)
    num_seqs = (cu_seqlens.numel() - 1) if cu_seqlens is not None else 0
    rc = lib.gdn_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                                   _ptr(cu_seqlens), num_seqs, _ptr(out), _ptr(final_state),
                                   B, T, H, dk, dv, _dt(q), float(scale), int(bool(use_qk_l2norm)),
                                   int(chunk_size), _stream(stream))
    if rc != GDN_OK:
        what = "gdn_chunk_fwd_noalloc"
        if rc == 3:
            what += f" (problem needs more than the {NOALLOC_SCRATCH_BYTES >> 20} MiB fixed scratch)"
        raise GDNError(rc, what)
    return out, final_state
