"""CPU oracle of the FP8 paged-KV decode path (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg and reference arm (``bench.py --impl reference``) import this
package.  The product library never does, and this
package imports nothing from it: the two share no code.

The arithmetic lives in ``fp8kv_oracle.c`` (plain C, fp64); this module only
compiles it with gcc and marshals numpy arrays to it.  Every function states
what the method computes and which page passage it follows; the C file's
header lists the readings taken where the pages are silent.

Parity status: the e4m3 codec, append, bump and validation are pinned by the
closed-form and brute-force tests under ``tests/test_oracle_*.py``; attention
is pinned by closed forms, a separate dense brute force and library softmax
attention (no worked numeric example exists in the pages).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8kv_oracle.c")
_LIB = os.path.join(_HERE, "libfp8kv_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_D = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off) into a shared object."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.orc_e4m3_decode.restype = _D
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode.argtypes = [_F]
            lib.orc_e4m3_encode_array.argtypes = [_P, _I64, _P]
            lib.orc_e4m3_decode_array.argtypes = [_P, _I64, _P]
            lib.orc_quantize_bf16.restype = ctypes.c_uint8
            lib.orc_quantize_bf16.argtypes = [ctypes.c_uint16, _F]
            lib.orc_quantize_bf16_array.argtypes = [_P, _I64, _F, _P]
            lib.orc_amax_scale_bf16.restype = _F
            lib.orc_amax_scale_bf16.argtypes = [_P, _I64]
            lib.orc_w4_quantize.argtypes = [_P, _I, _I, _P, _P]
            lib.orc_w8_quantize.argtypes = [_P, _I, _I, _P, _P]
            lib.orc_w4_pack.argtypes = [_P, _I, _I, _P]
            lib.orc_w8_pack.argtypes = [_P, _I, _I, _P]
            lib.orc_w4_gemv.argtypes = [_P, _I, _P, _P, _I, _I, _P]
            lib.orc_w8_gemv.argtypes = [_P, _I, _P, _P, _I, _I, _P]
            lib.orc_kv_append.argtypes = [_P, _P, _I, _P, _F, _F, _P, _I, _P,
                                          _P, _P, _P, _I, _I, _I, _I, _I]
            lib.orc_kv_prefill.argtypes = [_P, _P, _P, _I, _P, _F, _F, _P, _I,
                                           _P, _P, _P, _I, _I, _I, _I, _I]
            lib.orc_page_tags_bump.argtypes = [_P, _P, _I, _I]
            lib.orc_page_tags_validate.restype = _I
            lib.orc_page_tags_validate.argtypes = [_P, _P, _P, _I, _P, _I, _I, _I, _P]
            lib.orc_paged_attention.argtypes = [_P, _P, _I, _D, _D, _P, _I, _P, _P, _D,
                                                _I, _I, _I, _I, _I, _I, _P, _P, _P]
            lib.orc_dense_attention.argtypes = [_P, _P, _P, _I, _I, _D, _P, _P, _P]
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "need a C-contiguous numpy array"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# e4m3 codec
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """OCP E4M3 decode of uint8 codes to float64 (NaN for S.1111.111)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().orc_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    """E4M3 encode of float32 values: nearest, ties to even, saturate at 448."""
    a = _c(x, np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().orc_e4m3_encode_array(_ptr(a), a.size, _ptr(out))
    return out


def quantize_bf16(xbits, scale: float) -> np.ndarray:
    """Code of float(bf16 x) / scale (one IEEE fp32 division, then encode)."""
    xb = _c(xbits, np.uint16)
    out = np.empty(xb.shape, np.uint8)
    _load().orc_quantize_bf16_array(_ptr(xb), xb.size, float(np.float32(scale)), _ptr(out))
    return out


def amax_scale_bf16(xbits) -> np.float32:
    """Per-tensor scale amax / 448 over the finite bf16 elements (1 if amax = 0)."""
    xb = _c(xbits, np.uint16)
    return np.float32(_load().orc_amax_scale_bf16(_ptr(xb), xb.size))


# --------------------------------------------------------------------------
# cache writes, tags
# --------------------------------------------------------------------------

def kv_append(k_new, v_new, kv_pool, k_scale, v_scale, page_table, seq_lens,
              live_tags=None, expected_tags=None, abort_mask=None, *, fp8: bool,
              Hkv: int, D: int, page_size: int, num_pages: int):
    """One decode-step append per request at position seq_lens[r]-1 (in place)."""
    B, max_pages = page_table.shape
    _load().orc_kv_append(_ptr(_c(k_new, np.uint16)), _ptr(_c(v_new, np.uint16)), int(fp8),
                          _ptr(kv_pool), float(k_scale), float(v_scale),
                          _ptr(_c(page_table, np.int32)), max_pages, _ptr(_c(seq_lens, np.int32)),
                          _ptr(live_tags), _ptr(expected_tags), _ptr(abort_mask),
                          B, Hkv, D, page_size, num_pages)


def kv_prefill(k, v, cu_seqlens, kv_pool, k_scale, v_scale, page_table,
               live_tags=None, expected_tags=None, abort_mask=None, *, fp8: bool,
               Hkv: int, D: int, page_size: int, num_pages: int):
    """Write whole prompts: rows cu[r]..cu[r+1]-1 go to positions 0.. of request r."""
    B, max_pages = page_table.shape
    _load().orc_kv_prefill(_ptr(_c(k, np.uint16)), _ptr(_c(v, np.uint16)),
                           _ptr(_c(cu_seqlens, np.int32)), int(fp8),
                           _ptr(kv_pool), float(k_scale), float(v_scale),
                           _ptr(_c(page_table, np.int32)), max_pages,
                           _ptr(live_tags), _ptr(expected_tags), _ptr(abort_mask),
                           B, Hkv, D, page_size, num_pages)


def page_tags_bump(live_tags: np.ndarray, pages, num_pages: int) -> None:
    """+1 (mod 2^32) on every listed page's live tag, in place."""
    p = _c(pages, np.int32)
    _load().orc_page_tags_bump(_ptr(live_tags), _ptr(p), p.size, num_pages)


def page_tags_validate(page_table, expected_tags, seq_lens, live_tags, num_pages: int,
                       page_size: int):
    """Returns (abort_mask uint8 [B], abort_count)."""
    pt = _c(page_table, np.int32)
    B, max_pages = pt.shape
    mask = np.empty(B, np.uint8)
    n = _load().orc_page_tags_validate(_ptr(pt), _ptr(_c(expected_tags, np.uint32)),
                                       _ptr(_c(seq_lens, np.int32)), max_pages,
                                       _ptr(_c(live_tags, np.uint32)), num_pages, B,
                                       page_size, _ptr(mask))
    return mask, n


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def paged_attention(q, kv_pool, page_table, seq_lens, *, fp8: bool, k_scale=1.0,
                    v_scale=1.0, abort_mask=None, sm_scale: float, Hkv: int, page_size: int,
                    num_pages: int):
    """fp64 decode attention over the page table; returns (out [B][Hq][D], lse [B][Hq])."""
    qb = _c(q, np.uint16)
    B, Hq, D = qb.shape
    pt = _c(page_table, np.int32)
    max_pages = pt.shape[1]
    out = np.empty((B, Hq, D), np.float64)
    lse = np.empty((B, Hq), np.float64)
    scores = np.empty(max(1, max_pages * page_size), np.float64)
    am = None if abort_mask is None else _c(abort_mask, np.uint8)
    _load().orc_paged_attention(_ptr(qb), _ptr(kv_pool), int(fp8),
                                float(k_scale), float(v_scale), _ptr(pt), max_pages,
                                _ptr(_c(seq_lens, np.int32)), _ptr(am), float(sm_scale),
                                B, Hq, Hkv, D, page_size, num_pages,
                                _ptr(scores), _ptr(out), _ptr(lse))
    return out, lse


def dense_attention(q, K, V, sm_scale: float):
    """Textbook softmax(q K^T sm_scale) V for one query; q [D], K,V [L][D] float64."""
    qd = _c(q, np.float64)
    Kd = _c(K, np.float64)
    Vd = _c(V, np.float64)
    L, D = Kd.shape
    out = np.empty(D, np.float64)
    lse = ctypes.c_double()
    scores = np.empty(max(1, L), np.float64)
    _load().orc_dense_attention(_ptr(qd), _ptr(Kd), _ptr(Vd), L, D, float(sm_scale),
                                _ptr(scores), _ptr(out), ctypes.byref(lse))
    return out, lse.value


# --------------------------------------------------------------------------
# weight-only quantised GEMV
# --------------------------------------------------------------------------

def w4_quantize(w_bits):
    """INT4 codes q [N][K] (int8 in [-8, 7]) and bf16 scales [N][K/128], natural layout."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    q = np.empty((N, K), np.int8)
    sc = np.empty((N, K // 128), np.uint16)
    _load().orc_w4_quantize(_ptr(w), N, K, _ptr(q), _ptr(sc))
    return q, sc


def w8_quantize(w_bits):
    """e4m3 codes [N][K] and fp32 row scales [N], natural layout."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    c = np.empty((N, K), np.uint8)
    r = np.empty(N, np.float32)
    _load().orc_w8_quantize(_ptr(w), N, K, _ptr(c), _ptr(r))
    return c, r


def w4_pack(q):
    """INT4 codes in the slice layout (the library's weight format)."""
    q = _c(q, np.int8)
    N, K = q.shape
    out = np.zeros(N * K // 2, np.uint8)
    _load().orc_w4_pack(_ptr(q), N, K, _ptr(out))
    return out


def w8_pack(codes):
    """e4m3 codes in the slice layout."""
    c = _c(codes, np.uint8)
    N, K = c.shape
    out = np.zeros(N * K, np.uint8)
    _load().orc_w8_pack(_ptr(c), N, K, _ptr(out))
    return out


def w4_gemv(x_bits, q, scales):
    """y [B][N] = x . (q * s)^T in fp64."""
    x = _c(x_bits, np.uint16)
    q = _c(q, np.int8)
    sc = _c(scales, np.uint16)
    B, K = x.shape
    N = q.shape[0]
    y = np.empty((B, N), np.float64)
    _load().orc_w4_gemv(_ptr(x), B, _ptr(q), _ptr(sc), N, K, _ptr(y))
    return y


def w8_gemv(x_bits, codes, row_scales):
    """y [B][N] = x . (decode(codes) * r)^T in fp64."""
    x = _c(x_bits, np.uint16)
    c = _c(codes, np.uint8)
    r = _c(row_scales, np.float32)
    B, K = x.shape
    N = c.shape[0]
    y = np.empty((B, N), np.float64)
    _load().orc_w8_gemv(_ptr(x), B, _ptr(c), _ptr(r), N, K, _ptr(y))
    return y
