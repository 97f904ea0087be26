"""The C-ABI library builds for sm_103a, loads and exports every entry point
that include/fp8kv.h declares, and the Python binding mirrors them (no compute
call is made here: this runs on hosts without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8kv.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fpk_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from fp8_paged_kv_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_path():
    syms = declared_symbols()
    for name in ("fpk_kv_append_fp8", "fpk_kv_append_bf16", "fpk_page_tags_bump",
                 "fpk_page_tags_validate", "fpk_paged_decode_attn_fp8",
                 "fpk_paged_decode_attn_bf16", "fpk_decode_workspace_bytes", "fpk_status_str"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, f"not exported: {missing}"


def test_binding_mirrors_the_header():
    import fp8_paged_kv_gb300 as fpk
    assert set(fpk.SIGNATURES) == set(declared_symbols())
    for name in declared_symbols():
        if name not in ("fpk_version", "fpk_status_str"):
            assert callable(getattr(fpk, name)), name


def test_host_only_entry_points(lib):
    lib.fpk_version.restype = ctypes.c_int
    lib.fpk_status_str.restype = ctypes.c_char_p
    assert lib.fpk_version() >= 100
    for s in range(5):
        assert lib.fpk_status_str(s)
    assert b"unknown" in lib.fpk_status_str(99)


def test_argument_errors_are_synchronous_without_a_device(lib):
    """Invalid arguments are rejected before anything touches a device."""
    f = lib.fpk_page_tags_bump
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
    assert f(None, None, -1, 4, None) == 1          # FPK_EINVAL
    assert f(None, None, 0, 4, None) == 0           # nothing to do
    g = lib.fpk_decode_workspace_bytes
    g.restype = ctypes.c_size_t
    g.argtypes = [ctypes.c_int32] * 5
    assert g(4, 64, 7, 128, 16) == 0                 # Hq % Hkv != 0
    assert g(4, 64, 8, 64, 16) == 0                  # unsupported D
    assert g(4, 64, 8, 128, 16) > 0                  # fixed split count needs no device


def test_no_oracle_in_the_product():
    """The product package never imports or links the oracle."""
    pkg = os.path.join(ROOT, "fp8_paged_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "fp8kv_oracle" not in text, f


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """Without the built library the binding raises; it has no fallback."""
    import fp8_paged_kv_gb300 as fpk
    monkeypatch.setattr(fpk, "_lib", None)
    with pytest.raises(fpk.FpkError, match="no fallback"):
        fpk.load_library(str(tmp_path / "absent.so"))


def test_cpu_tensors_are_refused(lib):
    """Every compute entry point refuses host tensors before calling the
    library: there is no CPU path to fall back to."""
    import torch

    import fp8_paged_kv_gb300 as fpk
    B, Hq, Hkv, D, ps, P = 2, 8, 2, 128, 16, 4
    pool8 = torch.zeros(2 * P * Hkv * ps * D, dtype=torch.uint8)
    pool16 = torch.zeros(2 * P * Hkv * ps * D, dtype=torch.bfloat16)
    kv = torch.zeros(B, Hkv, D, dtype=torch.bfloat16)
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16)
    pt = torch.zeros(B, 2, dtype=torch.int32)
    lens = torch.ones(B, dtype=torch.int32)
    sc = torch.ones(1)
    out, lse = torch.zeros(B, Hq, D), torch.zeros(B, Hq)
    ws = torch.zeros(4096, dtype=torch.uint8)
    tags, exp = torch.zeros(P, dtype=torch.int32), torch.zeros(B, 2, dtype=torch.int32)
    mask = torch.zeros(B, dtype=torch.uint8)
    geo = dict(Hkv=Hkv, page_size=ps, num_pages=P)
    calls = {
        "append_fp8": lambda: fpk.fpk_kv_append_fp8(kv, kv, pool8, sc, sc, pt, lens, D=D, **geo),
        "append_bf16": lambda: fpk.fpk_kv_append_bf16(kv, kv, pool16, pt, lens, D=D, **geo),
        "bump": lambda: fpk.fpk_page_tags_bump(tags, torch.zeros(1, dtype=torch.int32), num_pages=P),
        "validate": lambda: fpk.fpk_page_tags_validate(pt, exp, lens, tags, mask, num_pages=P,
                                                       page_size=ps),
        "attn_fp8": lambda: fpk.fpk_paged_decode_attn_fp8(q, pool8, sc, sc, pt, lens, None, out, lse,
                                                          ws, sm_scale=0.1, **geo),
        "attn_fp8_tc": lambda: fpk.fpk_paged_decode_attn_fp8_tc(q, pool8, sc, sc, pt, lens, None, out,
                                                                lse, ws, sm_scale=0.1, **geo),
        "attn_bf16": lambda: fpk.fpk_paged_decode_attn_bf16(q, pool16, pt, lens, None, out, lse, ws,
                                                            sm_scale=0.1, **geo),
        "step_fp8": lambda: fpk.fpk_decode_step_fp8(kv, kv, pool8, sc, sc, pt, lens, tags, exp, mask,
                                                    q, out, lse, ws, sm_scale=0.1, **geo),
        "w4_gemv": lambda: fpk.fpk_w4_gemv(torch.zeros(1, 128, dtype=torch.bfloat16),
                                           torch.zeros(64, dtype=torch.uint8),
                                           torch.zeros(1, dtype=torch.bfloat16), torch.zeros(1, 1)),
    }
    for name, call in calls.items():
        with pytest.raises(fpk.FpkError, match="CUDA"):
            call()


def test_attention_argument_errors_before_any_device_call():
    """The attention entry points reject bad shapes, missing pointers and
    misaligned buffers synchronously, before they ask for a device.  Every call
    here returns at one of those checks (the pointers are never dereferenced);
    the test is skipped where a device exists, so that a regression in the
    order of the checks can never launch on the fake pointers."""
    import torch

    import fp8_paged_kv_gb300 as fpk
    if torch.cuda.is_available():
        pytest.skip("host-side checks only; run where no device is visible")
    lib = fpk.load_library()
    A = 1 << 20  # a 256-byte aligned fake address
    OK, EINVAL, EUNSUP = fpk.FPK_OK, fpk.FPK_EINVAL, fpk.FPK_EUNSUPPORTED

    def fp8(q=A, kv=A, ks=A, vs=A, pt=A, lens=A, out=A, ws=A, B=2, Hq=16, Hkv=2, D=128, ps=16,
            num_pages=8, max_pages=4, splits=0):
        return lib.fpk_paged_decode_attn_fp8(q, kv, ks, vs, pt, max_pages, lens, None, out, None, ws,
                                             1 << 20, splits, 0.1, B, Hq, Hkv, D, ps, num_pages, None)

    def bf16(q=A, kv=A, pt=A, lens=A, out=A, ws=A, B=2, Hq=16, Hkv=2, D=128, ps=16):
        return lib.fpk_paged_decode_attn_bf16(q, kv, pt, 4, lens, None, out, None, ws, 1 << 20, 0, 0.1,
                                              B, Hq, Hkv, D, ps, 8, None)

    assert fp8(B=0, q=None, kv=None, out=None, ws=None) == OK        # nothing to do
    assert fp8(Hq=15) == EINVAL                                     # Hq % Hkv != 0
    assert fp8(Hkv=0) == EINVAL
    assert fp8(B=-1) == EINVAL
    assert fp8(splits=-1) == EINVAL
    assert fp8(max_pages=-1) == EINVAL
    assert fp8(D=64) == EUNSUP
    assert fp8(Hq=32, Hkv=2) == EUNSUP                              # G = 16 > 8
    assert fp8(ps=24) == EUNSUP and fp8(ps=512) == EUNSUP
    for name in ("q", "kv", "ks", "vs", "pt", "lens", "out", "ws"):
        assert fp8(**{name: None}) == EINVAL, name                   # required pointers
    assert fp8(q=A + 2) == EINVAL                                   # q 16-byte aligned
    assert fp8(kv=A + 8) == EINVAL
    assert fp8(out=A + 4) == EINVAL                                 # out 16-byte aligned
    assert fp8(ws=A + 16) == EINVAL                                 # workspace 256-byte aligned
    assert bf16(Hq=15) == EINVAL and bf16(D=256) == EUNSUP
    assert bf16(out=A + 4) == EINVAL and bf16(ws=None) == EINVAL
    assert bf16(B=0, q=None) == OK

    # the tensor-core variant checks the same arguments, and rejects pools
    # whose 128-byte rows exceed 32-bit tensor-map coordinates
    def tc(q=A, kv=A, ks=A, vs=A, pt=A, lens=A, out=A, ws=A, B=2, Hq=16, Hkv=2, D=128, ps=16,
           num_pages=8, splits=0):
        return lib.fpk_paged_decode_attn_fp8_tc(q, kv, ks, vs, pt, 4, lens, None, out, None, ws,
                                                1 << 20, splits, 0.1, B, Hq, Hkv, D, ps, num_pages,
                                                None)

    assert tc(B=0, q=None, kv=None, out=None, ws=None) == OK
    assert tc(Hq=15) == EINVAL and tc(B=-1) == EINVAL and tc(splits=-1) == EINVAL
    assert tc(D=64) == EUNSUP and tc(ps=24) == EUNSUP and tc(Hq=32, Hkv=2) == EUNSUP
    assert tc(num_pages=1 << 23, Hkv=8, Hq=64, ps=16) == EUNSUP     # 2^31 rows of 128 bytes
    for name in ("q", "kv", "ks", "vs", "pt", "lens", "out", "ws"):
        assert tc(**{name: None}) == EINVAL, name
    assert tc(q=A + 2) == EINVAL and tc(kv=A + 8) == EINVAL and tc(out=A + 4) == EINVAL
    assert tc(ws=A + 16) == EINVAL

    # the allocation-free entry point checks the same arguments (it has no
    # workspace) before it looks up its scratch or clears it
    def noalloc(q=A, kv=A, ks=A, vs=A, pt=A, lens=A, out=A, B=2, Hq=16, Hkv=2, D=128, ps=16,
                splits=0):
        return lib.fpk_paged_decode_attn_fp8_noalloc(q, kv, ks, vs, pt, 4, lens, None, out, None,
                                                     splits, 0.1, B, Hq, Hkv, D, ps, 8, None)

    assert noalloc(B=0, q=None, kv=None, out=None) == OK
    assert noalloc(Hq=15) == EINVAL and noalloc(B=-1) == EINVAL and noalloc(splits=-1) == EINVAL
    assert noalloc(D=64) == EUNSUP and noalloc(ps=24) == EUNSUP
    for name in ("q", "kv", "ks", "vs", "pt", "lens", "out"):
        assert noalloc(**{name: None}) == EINVAL, name
    assert noalloc(q=A + 2) == EINVAL and noalloc(kv=A + 8) == EINVAL and noalloc(out=A + 4) == EINVAL

    # the tag check rejects missing tables before it clears the abort count
    def validate(pt=A, ex=A, lens=A, live=A, mask=A, count=A, B=2):
        return lib.fpk_page_tags_validate(pt, ex, lens, 4, live, 8, B, 16, mask, count, None)

    for name in ("pt", "ex", "lens", "live", "mask"):
        assert validate(**{name: None}) == EINVAL, name
    assert validate(B=-1) == EINVAL


def test_write_and_gemv_argument_errors_before_any_device_call():
    """The same for the cache writes and the weight GEMV: every call below
    returns at a host-side check (skipped where a device exists)."""
    import torch

    import fp8_paged_kv_gb300 as fpk
    if torch.cuda.is_available():
        pytest.skip("host-side checks only; run where no device is visible")
    lib = fpk.load_library()
    A = 1 << 20
    OK, EINVAL, EUNSUP = fpk.FPK_OK, fpk.FPK_EINVAL, fpk.FPK_EUNSUPPORTED

    def append(k=A, v=A, pool=A, ks=A, vs=A, pt=A, lens=A, B=2, Hkv=2, D=128, ps=16, num_pages=8,
               max_pages=4):
        return lib.fpk_kv_append_fp8(k, v, pool, ks, vs, pt, max_pages, lens, None, None, None,
                                     B, Hkv, D, ps, num_pages, None)

    def prefill(cu=A, n=32, B=2):
        return lib.fpk_kv_prefill_fp8(A, A, cu, n, A, A, A, A, 4, None, None, None, B, 2, 128, 16, 8,
                                      None)

    assert append(B=0, k=None) == OK
    assert append(Hkv=0) == EINVAL and append(B=-1) == EINVAL and append(num_pages=-1) == EINVAL
    assert append(D=64) == EUNSUP and append(ps=8) == EUNSUP and append(ps=272) == EUNSUP
    for name in ("k", "v", "pool", "ks", "vs", "pt", "lens"):
        assert append(**{name: None}) == EINVAL, name
    assert append(k=A + 2) == EINVAL and append(v=A + 8) == EINVAL and append(pool=A + 1) == EINVAL
    assert prefill(n=0) == OK and prefill(n=-1) == EINVAL and prefill(cu=None) == EINVAL

    def w4(x=A, codes=A, scales=A, y=A, B=1, N=64, K=256):
        return lib.fpk_w4_gemv(x, codes, scales, y, B, N, K, None)

    assert w4(B=0) == OK and w4(N=0) == OK
    assert w4(B=17) == EUNSUP and w4(N=24) == EUNSUP and w4(K=200) == EUNSUP
    assert w4(B=-1) == EINVAL and w4(N=-16) == EINVAL
    for name in ("x", "codes", "scales", "y"):
        assert w4(**{name: None}) == EINVAL, name
    assert w4(x=A + 4) == EINVAL and w4(codes=A + 8) == EINVAL
    assert lib.fpk_w8_gemv(A, A, None, A, 1, 64, 256, None) == EINVAL   # row scales required


def test_header_is_plain_c(tmp_path, lib):
    """include/fp8kv.h compiles as strict C99 and a C program links against
    the library and calls its host-only entry points."""
    import shutil
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from fp8_paged_kv_gb300 import LIB_PATH
    src = tmp_path / "abi.c"
    src.write_text('#include "fp8kv.h"\n#include <stdio.h>\n'
                   'int main(void) { printf("%d %s\\n", fpk_version(), fpk_status_str(FPK_ENOSPC));\n'
                   '  return 0; }\n')
    exe = tmp_path / "abi"
    libdir = os.path.dirname(LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                    os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lfp8kv",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split(" ", 1)
    assert int(out[0]) >= 100 and out[1].strip()


def test_library_exports_nothing_undeclared(lib):
    """Every fpk_ symbol the library exports is declared in the header."""
    import shutil
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("no nm")
    from fp8_paged_kv_gb300 import LIB_PATH
    out = subprocess.run([nm, "-D", "--defined-only", LIB_PATH], check=True, capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.split() and ln.split()[-1].startswith("fpk_")}
    assert exported == set(declared_symbols())
