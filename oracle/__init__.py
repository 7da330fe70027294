"""fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
reference leg of ``bench.py`` may import this package.  The product path (the
CUDA library under ``gated_delta_rule_12_gb300/`` and its binding) never does,
and the two share no code: the oracle is plain C compiled with gcc
(``gdn_oracle.c``) plus the ctypes marshalling below.

What it computes, and where each step comes from, is documented at the top of
``gdn_oracle.c``.  Every array argument is converted to a C-contiguous float64
numpy array before the call, so callers may pass torch tensors (CPU), numpy
arrays of any float dtype, or bf16-rounded values (the rounding is kept: the
oracle then runs on exactly the values the device sees).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I32P = ctypes.POINTER(ctypes.c_int32)
_i32 = ctypes.c_int32


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``oracle/_build/liboracle.so`` (gcc, -O2)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lpthread", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_recurrent_fwd.argtypes = [_D, _D, _D, _D, _D, _D, _I32P, _i32, _D, _D,
                                                 _i32, _i32, _i32, _i32, _i32,
                                                 ctypes.c_double, _i32, _i32]
            lib.oracle_recurrent_fwd.restype = ctypes.c_int
            lib.oracle_chunked_fwd.argtypes = [_D, _D, _D, _D, _D, _D, _I32P, _i32, _D, _D,
                                               _i32, _i32, _i32, _i32, _i32,
                                               ctypes.c_double, _i32, _i32, _i32, _i32]
            lib.oracle_chunked_fwd.restype = ctypes.c_int
            lib.oracle_recurrent_bwd.argtypes = [_D, _D, _D, _D, _D, _D, _I32P, _i32, _D, _D,
                                                 _D, _D, _D, _D, _D, _D,
                                                 _i32, _i32, _i32, _i32, _i32, ctypes.c_double, _i32, _i32]
            lib.oracle_recurrent_bwd.restype = ctypes.c_int
            lib.oracle_short_conv_silu.argtypes = [_D, _D, _D, _I32P, _i32, _i32, _i32, _i32, _i32, _i32, _D, _D]
            lib.oracle_short_conv_silu.restype = ctypes.c_int
            lib.oracle_gate_activations.argtypes = [_D, _D, _D, _D, ctypes.c_int64, _i32, _D, _D]
            lib.oracle_gate_activations.restype = ctypes.c_int
            lib.oracle_decode_step.argtypes = [_D, _D, _D, _D, _D, _D, _D,
                                               _i32, _i32, _i32, _i32,
                                               ctypes.c_double, _i32, _i32]
            lib.oracle_decode_step.restype = ctypes.c_int
            lib.oracle_ut_transform.argtypes = [_D, _D, _D, _D, _i32, _i32, _i32, _i32, _D, _D]
            lib.oracle_ut_transform.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_D)


def _cu(cu):
    if cu is None:
        return None, None
    if hasattr(cu, "detach"):
        cu = cu.detach().cpu().numpy()
    cu = np.ascontiguousarray(np.asarray(cu, dtype=np.int32))
    return cu, cu.ctypes.data_as(_I32P)


def num_threads() -> int:
    """Host threads the oracle uses by default (all online cores)."""
    return int(_load().oracle_num_threads())


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def _prep(q, k, v, g, beta, init_state, cu_seqlens):
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    s0 = _f64(init_state)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, T, H) or g.shape != (B, T, H) or beta.shape != (B, T, H):
        raise ValueError("oracle: inconsistent shapes")
    cu, cup = _cu(cu_seqlens)
    N = (len(cu) - 1) if cu is not None else B
    if s0 is not None and s0.shape != (N, H, dv, dk):
        raise ValueError("oracle: init_state must be [N, H, dv, dk]")
    return q, k, v, g, beta, s0, cu, cup, B, T, H, dk, dv, N


def recurrent_fwd(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale=1.0,
                  use_qk_l2norm=False, nthreads=0):
    """Token-by-token gated delta rule (the definition).

    Returns ``(out [B,T,H,dv], final_state [N,H,dv,dk])`` as float64 arrays.
    """
    q, k, v, g, beta, s0, cu, cup, B, T, H, dk, dv, N = _prep(q, k, v, g, beta, init_state, cu_seqlens)
    out = np.zeros((B, T, H, dv), np.float64)
    sf = np.zeros((N, H, dv, dk), np.float64)
    rc = _load().oracle_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0),
                                      cup, N, _ptr(out), _ptr(sf), B, T, H, dk, dv,
                                      float(scale), int(bool(use_qk_l2norm)), int(nthreads))
    _check(rc, "recurrent_fwd")
    return out, sf


def chunked_fwd(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale=1.0,
                use_qk_l2norm=False, chunk_size=64, w_form=0, nthreads=0):
    """Chunkwise (WY/UT) gated delta rule in fp64, any chunk size.

    ``w_form=0`` builds W<- from the single Gamma-masked system;
    ``w_form=1`` builds the ungated W of eq. 6-7 and decays it by diag(gamma).
    """
    q, k, v, g, beta, s0, cu, cup, B, T, H, dk, dv, N = _prep(q, k, v, g, beta, init_state, cu_seqlens)
    out = np.zeros((B, T, H, dv), np.float64)
    sf = np.zeros((N, H, dv, dk), np.float64)
    rc = _load().oracle_chunked_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0),
                                    cup, N, _ptr(out), _ptr(sf), B, T, H, dk, dv,
                                    float(scale), int(bool(use_qk_l2norm)), int(chunk_size),
                                    int(w_form), int(nthreads))
    _check(rc, "chunked_fwd")
    return out, sf


def decode_step(state, q, k, v, g, beta, scale=1.0, use_qk_l2norm=False, nthreads=0):
    """One gated-delta-rule token per (sequence, head).

    ``state`` [N,H,dv,dk] is copied (float64) and the updated copy returned
    together with ``out`` [N,H,dv].
    """
    st = _f64(state).copy()
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    N, H, dv, dk = st.shape
    if q.shape != (N, H, dk) or k.shape != (N, H, dk) or v.shape != (N, H, dv) \
            or g.shape != (N, H) or beta.shape != (N, H):
        raise ValueError("oracle: inconsistent decode shapes")
    out = np.zeros((N, H, dv), np.float64)
    rc = _load().oracle_decode_step(_ptr(st), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    _ptr(out), N, H, dk, dv, float(scale),
                                    int(bool(use_qk_l2norm)), int(nthreads))
    _check(rc, "decode_step")
    return out, st


def ut_transform(K, V, alpha, beta, w_form=0):
    """UT transform of one chunk: returns ``(W<- [C,dk], U~ [C,dv])``."""
    K, V, alpha, beta = (_f64(t) for t in (K, V, alpha, beta))
    C, dk = K.shape
    dv = V.shape[1]
    W = np.zeros((C, dk), np.float64)
    U = np.zeros((C, dv), np.float64)
    rc = _load().oracle_ut_transform(_ptr(K), _ptr(V), _ptr(alpha), _ptr(beta), C, dk, dv,
                                     int(w_form), _ptr(W), _ptr(U))
    _check(rc, "ut_transform")
    return W, U


def recurrent_bwd(q, k, v, g, beta, dout, init_state=None, dfinal=None, cu_seqlens=None, scale=1.0,
                  use_qk_l2norm=False, nthreads=0):
    """Gradients of the token recurrence (reverse mode) for the loss
    sum(dout * out) + sum(dfinal * final_state).

    Returns a dict with dq, dk [B,T,H,dk], dv [B,T,H,dv], dg, dbeta [B,T,H] and dinit [N,H,dv,dk].
    """
    q, k, v, g, beta, s0, cu, cup, B, T, H, dk, dv, N = _prep(q, k, v, g, beta, init_state, cu_seqlens)
    dout = _f64(dout)
    dsf = _f64(dfinal)
    if dout.shape != (B, T, H, dv) or (dsf is not None and dsf.shape != (N, H, dv, dk)):
        raise ValueError("oracle: dout must be [B,T,H,dv] and dfinal [N,H,dv,dk]")
    r = {n: np.zeros(shape, np.float64) for n, shape in (("dq", (B, T, H, dk)), ("dk", (B, T, H, dk)),
                                                          ("dv", (B, T, H, dv)), ("dg", (B, T, H)),
                                                          ("dbeta", (B, T, H)), ("dinit", (N, H, dv, dk)))}
    rc = _load().oracle_recurrent_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0), cup, N,
                                      _ptr(dout), _ptr(dsf), _ptr(r["dq"]), _ptr(r["dk"]), _ptr(r["dv"]),
                                      _ptr(r["dg"]), _ptr(r["dbeta"]), _ptr(r["dinit"]), B, T, H, dk, dv,
                                      float(scale), int(bool(use_qk_l2norm)), int(nthreads))
    _check(rc, "recurrent_bwd")
    return r


def short_conv_silu(x, w, state_in=None, cu_seqlens=None):
    """Block prologue of one of q, k, v: short causal depthwise convolution, then SiLU.

    x [B,T,H,d]; w [H,d,K] (tap K-1 multiplies the current token); state_in
    [N,K-1,H,d] (the K-1 inputs before each sequence, oldest first) or None for
    zeros.  Returns ``(y [B,T,H,d], state_out [N,K-1,H,d])``.
    """
    x, w = _f64(x), _f64(w)
    B, T, H, d = x.shape
    K = w.shape[-1]
    if w.shape != (H, d, K):
        raise ValueError("oracle: w must be [H, d, K]")
    cu, cup = _cu(cu_seqlens)
    N = (len(cu) - 1) if cu is not None else B
    si = _f64(state_in)
    if si is not None and si.shape != (N, K - 1, H, d):
        raise ValueError("oracle: state_in must be [N, K-1, H, d]")
    y = np.zeros_like(x)
    so = np.zeros((N, K - 1, H, d), np.float64)
    rc = _load().oracle_short_conv_silu(_ptr(x), _ptr(w), _ptr(si), cup, N, B, T, H, d, K, _ptr(y), _ptr(so))
    _check(rc, "short_conv_silu")
    return y, so


def gate_activations(a, b, A_log, dt_bias):
    """alpha (as g = log alpha) in Mamba2's parameterisation and beta = sigmoid(b).

    a, b [..., H]; A_log, dt_bias [H].  Returns ``(g, beta)`` shaped like a.
    """
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    H = a.shape[-1]
    if b.shape != a.shape or A_log.shape != (H,) or dt_bias.shape != (H,):
        raise ValueError("oracle: gate shapes")
    g = np.zeros_like(a)
    beta = np.zeros_like(a)
    rc = _load().oracle_gate_activations(_ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), a.size // H, H,
                                         _ptr(g), _ptr(beta))
    _check(rc, "gate_activations")
    return g, beta
