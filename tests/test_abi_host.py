"""Host-side checks of the C ABI (no GPU needed).

The library must build for sm_103a, load, and export every function the
public header declares.  Argument validation runs on the host before any
CUDA call, so the error paths are exercised here with pointers that are
never dereferenced.
"""
import ctypes
import os
import re

import pytest

import gated_delta_rule_12_gb300 as gdn
from gated_delta_rule_12_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.load_library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(gdn_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(gdn.EXPORTS) <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libgdn.so does not export {n}"
    # and the symbol is a real dynamic export (not only resolvable by ctypes magic)
    out = os.popen(f"nm -D --defined-only {gdn.LIB_PATH}").read()
    for n in names:
        assert re.search(rf"\bT {n}\b", out), f"{n} missing from the dynamic symbol table"


def test_header_compiles_as_plain_c(tmp_path):
    """include/gdn.h is a C header: a C99 translation unit that takes the address of every
    declared entry point compiles warning-free with gcc."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    inc = os.path.join(ROOT, "include")
    with open(os.path.join(inc, "gdn.h")) as f:
        names = sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", f.read())))
    assert names, "no entry points found in the header"
    src = tmp_path / "use_gdn.c"
    src.write_text('#include "gdn.h"\n'
                   "void *const gdn_entry_points[] = {\n" + "".join(f"    (void *)&{n},\n" for n in names) + "};\n"
                   "int gdn_ok(gdn_status s) { return s == GDN_OK; }\n")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", inc, "-c", str(src), "-o",
                        str(tmp_path / "use_gdn.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(lib):
    for code, name in gdn.STATUS.items():
        assert lib.gdn_status_string(code).decode() == name
    assert lib.gdn_status_string(99).decode() == "GDN_UNKNOWN_STATUS"


def test_workspace_size_rules(lib):
    ws = lib.gdn_chunk_fwd_workspace_size
    assert ws(4, 2048, 16, 128, 128, 0, gdn.GDN_BF16) > 0
    assert ws(1, 32768, 16, 128, 128, 8, gdn.GDN_BF16) > 0
    assert ws(1, 256, 2, 64, 64, 0, gdn.GDN_F32) > 0
    assert ws(4, 100, 2, 128, 128, 8, gdn.GDN_BF16) == 0     # varlen needs B == 1
    assert ws(1, 64, 1, 96, 64, 0, gdn.GDN_F32) == 0         # unsupported dk
    assert ws(0, 64, 1, 64, 64, 0, gdn.GDN_F32) == 0
    # dk = 256 (CUDA-core path): the fp32 layout, 256 B + 64 * (12 + 4 * (dk + dv)) B per chunk and head
    assert ws(1, 128, 2, 256, 128, 0, gdn.GDN_BF16) == 256 + 2 * 2 * 64 * (12 + 4 * (256 + 128))
    assert lib.gdn_chunk_fwd_kernel_count(1, 128, 2, 256, 128, 0, gdn.GDN_BF16) == 3
    assert lib.gdn_chunk_bwd_workspace_size(1, 128, 2, 256, 128, 0, gdn.GDN_BF16) > 0    # the backward takes dk = 256 too
    assert lib.gdn_chunk_bwd_workspace_size(1, 128, 2, 96, 128, 0, gdn.GDN_BF16) == 0
    # grows with the problem
    assert ws(1, 4096, 2, 64, 64, 0, 0) > ws(1, 2048, 2, 64, 64, 0, 0)
    assert ws(1, 0, 2, 64, 64, 0, 0) >= 256


def test_backward_workspace_size_rules(lib):
    ws = lib.gdn_chunk_bwd_workspace_size

    def per_block(dk, dv):
        # fp32 per (chunk, head): q^, k^, Qd, Kd, W~ and three dk-wide scratch rows (8 x 64 dk),
        # b (64), T, A and the raw K^K^T, Q^K^T (4 x 64 x 64), U, V_new, dV_new and A^T dO
        # (4 x 64 dv), and three dv x dk matrices (S, dS', dO^T Qd)
        return 4 * (8 * 64 * dk + 64 + 4 * 64 * 64 + 4 * 64 * dv + 3 * dv * dk)

    assert ws(4, 2048, 16, 128, 128, 0, gdn.GDN_BF16) == 256 + 4 * 32 * 16 * per_block(128, 128)
    assert ws(1, 100, 2, 64, 32, 0, gdn.GDN_F32) == 256 + 2 * 2 * per_block(64, 32)   # ragged: 2 chunks
    assert ws(1, 32768, 16, 128, 128, 8, gdn.GDN_BF16) == 256 + (32768 // 64 + 8 + 1) * 16 * per_block(128, 128)
    assert ws(4, 100, 2, 128, 128, 8, gdn.GDN_BF16) == 0     # varlen needs B == 1
    assert ws(1, 64, 1, 96, 64, 0, gdn.GDN_F32) == 0         # unsupported dk


def test_kernel_count_rules(lib):
    kc = lib.gdn_chunk_fwd_kernel_count
    assert kc(4, 2048, 16, 128, 128, 0, gdn.GDN_BF16) == 2      # tensor-core path: UT + recurrence
    assert kc(8, 8192, 32, 128, 256, 0, gdn.GDN_BF16) == 2
    assert kc(1, 256, 2, 64, 64, 0, gdn.GDN_F32) == 3           # CUDA-core path
    assert kc(4, 2048, 16, 128, 128, 0, gdn.GDN_F32) == 3
    assert kc(2, 0, 2, 64, 64, 0, gdn.GDN_F32) == 1             # no tokens: the state copy alone
    assert kc(1, 64, 1, 96, 64, 0, gdn.GDN_F32) == 0            # unsupported
    assert kc(4, 100, 2, 128, 128, 8, gdn.GDN_BF16) == 0


def _call_chunk(lib, **over):
    fake = 1 << 20  # 256-aligned, never dereferenced: validation fails first
    args = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, s0=None, cu=None, nseq=0, out=fake, sf=None,
                B=1, T=64, H=1, dk=64, dv=64, dt=gdn.GDN_F32, scale=0.125, l2=1, C=64,
                ws=fake, wsb=1 << 30, stream=None)
    args.update(over)
    a = args
    return lib.gdn_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["s0"], a["cu"], a["nseq"], a["out"],
                             a["sf"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["dt"], a["scale"], a["l2"],
                             a["C"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(C=32), 2),                       # chunk size other than 64
    (dict(dk=96), 2),                      # unsupported head dim
    (dict(dv=48), 2),
    (dict(B=0), 1),
    (dict(H=0), 1),
    (dict(dt=7), 1),
    (dict(q=None), 1),                     # NULL input with tokens present
    (dict(out=None), 1),
    (dict(k=(1 << 20) + 4), 1),            # misaligned
    (dict(g=(1 << 20) + 2), 1),
    (dict(ws=None), 3),                    # no workspace
    (dict(ws=(1 << 20) + 16), 3),          # workspace not 256-aligned
    (dict(wsb=64), 3),                     # workspace too small
    (dict(cu=1 << 20, nseq=0), 1),         # varlen without a sequence count
    (dict(cu=1 << 20, nseq=2, B=2), 1),    # varlen needs B == 1
    (dict(nseq=3), 1),                     # num_seqs inconsistent with B
])
def test_chunk_fwd_validation(lib, over, code):
    assert _call_chunk(lib, **over) == code


def _call_bwd(lib, **over):
    fake = 1 << 20  # 256-aligned, never dereferenced: validation fails first
    args = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, s0=None, cu=None, nseq=0, dout=fake, dsf=None,
                dq=fake, dk_=fake, dv_=fake, dg=fake, db=fake, dinit=None,
                B=1, T=64, H=1, dk=64, dv=64, dt=gdn.GDN_F32, scale=0.125, l2=1, C=64,
                ws=fake, wsb=1 << 30, stream=None)
    args.update(over)
    a = args
    return lib.gdn_chunk_bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["s0"], a["cu"], a["nseq"], a["dout"],
                             a["dsf"], a["dq"], a["dk_"], a["dv_"], a["dg"], a["db"], a["dinit"],
                             a["B"], a["T"], a["H"], a["dk"], a["dv"], a["dt"], a["scale"], a["l2"], a["C"],
                             a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(C=32), 2),                       # chunk size other than 64
    (dict(dk=96), 2),                      # unsupported head dim
    (dict(dv=48), 2),
    (dict(B=0), 1),
    (dict(H=0), 1),
    (dict(dt=7), 1),
    (dict(dout=None), 1),                  # NULL output gradient with tokens present
    (dict(dg=None), 1),                    # NULL gradient buffer
    (dict(dq=(1 << 20) + 4), 1),           # misaligned
    (dict(db=(1 << 20) + 2), 1),
    (dict(dinit=(1 << 20) + 8), 1),
    (dict(ws=None), 3),                    # no workspace
    (dict(ws=(1 << 20) + 16), 3),          # workspace not 256-aligned
    (dict(wsb=64), 3),                     # workspace too small
    (dict(cu=1 << 20, nseq=0), 1),         # varlen without a sequence count
    (dict(cu=1 << 20, nseq=2, B=2), 1),    # varlen needs B == 1
    (dict(nseq=3), 1),                     # num_seqs inconsistent with B
])
def test_chunk_bwd_validation(lib, over, code):
    assert _call_bwd(lib, **over) == code


def test_decode_validation(lib):
    fake = 1 << 20
    d = lib.gdn_decode_step
    assert d(fake, fake, fake, fake, fake, fake, fake, 4, 2, 96, 64, 0, 1.0, 1, None) == 2   # dk
    assert d(fake, fake, fake, fake, fake, fake, fake, 4, 2, 128, 12, 0, 1.0, 1, None) == 2  # dv % 8
    assert d(None, fake, fake, fake, fake, fake, fake, 4, 2, 128, 64, 0, 1.0, 1, None) == 1
    assert d(fake + 8, fake, fake, fake, fake, fake, fake, 4, 2, 128, 64, 0, 1.0, 1, None) == 1   # state
    assert d(fake, fake + 2, fake, fake, fake, fake, fake, 4, 2, 128, 64, 0, 1.0, 1, None) == 1   # fp32 q
    assert d(fake, fake, fake, fake, fake + 2, fake, fake, 4, 2, 128, 64, 0, 1.0, 1, None) == 1   # g
    assert d(fake, fake, fake, fake, fake, fake, fake, 4, 0, 128, 64, 0, 1.0, 1, None) == 1
    assert d(fake, fake, fake, fake, fake, fake, fake, 0, 2, 128, 64, 0, 1.0, 1, None) == 0  # nothing to do


def test_decode_multi_validation(lib):
    fake = 1 << 20
    d = lib.gdn_decode_multi
    #            state q     k     v     g     beta  out   N  T  H  dk   dv  dt scale l2 stream
    assert d(fake, fake, fake, fake, fake, fake, fake, 4, 3, 2, 96, 64, 0, 1.0, 1, None) == 2    # dk
    assert d(fake, fake, fake, fake, fake, fake, fake, 4, 3, 2, 128, 12, 0, 1.0, 1, None) == 2   # dv % 8
    assert d(fake, fake, fake, fake, fake, fake, fake, 4, -1, 2, 128, 64, 0, 1.0, 1, None) == 1  # T < 0
    assert d(fake, fake, fake, fake, None, fake, fake, 4, 3, 2, 128, 64, 0, 1.0, 1, None) == 1   # g
    assert d(fake + 8, fake, fake, fake, fake, fake, fake, 4, 3, 2, 128, 64, 0, 1.0, 1, None) == 1   # state
    assert d(fake, fake, fake, fake + 1, fake, fake, fake, 4, 3, 2, 128, 64, 1, 1.0, 1, None) == 1   # bf16 v
    assert d(fake, fake, fake, fake, fake, fake, fake, 4, 0, 2, 128, 64, 0, 1.0, 1, None) == 0   # T = 0
    assert d(None, None, None, None, None, None, None, 0, 3, 2, 128, 64, 0, 1.0, 1, None) == 0   # N = 0


def test_prologue_validation(lib):
    fake = 1 << 20
    P = lib.gdn_prologue

    def call(**o):
        a = dict(xq=fake, xk=fake, xv=fake, wq=fake, wk=fake, wv=fake, ga=fake, gb=fake, al=fake, dtb=fake,
                 si=None, so=None, cu=None, nseq=0, q=fake, k=fake, v=fake, g=fake, beta=fake,
                 B=2, T=64, H=2, dk=64, dv=64, K=4, dt=gdn.GDN_BF16)
        a.update(o)
        return P(a["xq"], a["xk"], a["xv"], a["wq"], a["wk"], a["wv"], a["ga"], a["gb"], a["al"], a["dtb"],
                 a["si"], a["so"], a["cu"], a["nseq"], a["q"], a["k"], a["v"], a["g"], a["beta"],
                 a["B"], a["T"], a["H"], a["dk"], a["dv"], a["K"], a["dt"], None)

    assert call(K=5) == 2 and call(K=0) == 2          # filter width 1..4
    assert call(dk=12) == 2 and call(dv=264) == 2    # multiples of 8 up to 256
    assert call(xq=fake + 8) == 1                    # 16-byte aligned projections
    assert call(g=fake + 2) == 1                     # 4-byte aligned fp32 arrays
    assert call(wq=None) == 1
    assert call(cu=fake, nseq=2) == 1                # varlen needs B == 1
    bytes_ = 2 * 3 * 2 * (2 * 64 + 64) * 2
    assert call(si=fake, so=fake + bytes_ - 16) == 1   # overlapping convolution states
    assert call(T=0, so=None) == 0                   # nothing to do


def test_check_device_error_validation(lib):
    assert lib.gdn_check_device_error(None, None) == 1
    assert lib.gdn_check_device_error((1 << 20) + 8, None) == 1


def test_selftest_wait_timeout_validation(lib):
    fake = 1 << 20
    st = lib.gdn_selftest_wait_timeout
    assert st(None, 1000, None) == 1              # no workspace
    assert st(fake + 8, 1000, None) == 1          # not 256-aligned
    assert st(fake, 0, None) == 1                 # limit below 1 us
    assert st(fake, 1000001, None) == 1           # limit above 1 s


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 64, 1, 64)
    with pytest.raises(ValueError):
        gdn.chunk_fwd(q, q, q, torch.zeros(1, 64, 1), torch.zeros(1, 64, 1), out=q.clone(),
                      final_state=torch.zeros(1, 1, 64, 64), workspace=torch.zeros(1 << 20, dtype=torch.uint8))


def test_product_path_does_not_reference_the_oracle():
    pkg = os.path.join(ROOT, "gated_delta_rule_12_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "gdn_oracle" not in text and "liboracle" not in text, f
