"""The kernel-source digest that ties a committed ncu record to the code it was
taken on: comments and layout do not change it, code does."""
import os

import bench


def _files():
    csrc = os.path.join(bench.ROOT, "fp8_paged_kv_gb300", "csrc")
    out = {}
    for n in bench.KERNEL_SOURCES:
        with open(os.path.join(csrc, n), encoding="utf-8") as f:
            out[n] = f.read()
    return out


def test_strip_comments_keeps_literals():
    src = 'int a = 1; // tail\n/* block\n spans */ const char* s = "x//y /*z*/"; char c = \'"\';\n\tb  =  2;'
    assert bench._strip_comments(src) == 'int a = 1; const char* s = "x//y /*z*/"; char c = \'"\'; b = 2;'


def test_digest_ignores_comments_and_layout():
    f = _files()
    base = bench.kernel_source_digest(lambda n: f[n])
    assert base == bench.kernel_source_digest()
    g = dict(f)
    g["decode_attn.cu"] = "// a new first line\n" + f["decode_attn.cu"].replace("\n", "\n\n", 3) + "\n/* end */\n"
    assert bench.kernel_source_digest(lambda n: g[n]) == base


def test_digest_follows_code():
    f = _files()
    base = bench.kernel_source_digest(lambda n: f[n])
    for name in bench.KERNEL_SOURCES:
        g = dict(f)
        g[name] = f[name] + "\nstatic int extra_symbol;\n"
        assert bench.kernel_source_digest(lambda n: g[n]) != base, name


def test_committed_records_carry_a_digest():
    # every attention record under profiles/ names the digest of the code it
    # measured; bench.py reports its traffic only while that digest is current
    import glob
    import json
    recs = glob.glob(os.path.join(bench.ROOT, "profiles", "paged_decode_attn_*.json"))
    assert recs
    for p in recs:
        with open(p) as fh:
            d = json.load(fh)
        h = d["source_sha256_16"]
        assert len(h) == 16 and int(h, 16) >= 0, os.path.basename(p)
        assert d["dram_bytes_per_launch"] > 0
