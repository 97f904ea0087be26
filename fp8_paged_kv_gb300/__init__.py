"""fp8_paged_kv_gb300 -- Python binding of libfp8kv (the C ABI in include/fp8kv.h).

Argument marshalling only: every function takes torch CUDA tensors, checks
dtype / device / contiguity, and passes raw pointers, sizes and the current
CUDA stream to the C entry point of the same name.  All computation happens in
the library's CUDA kernels; there is no CPU or PyTorch fallback.  If the
library is missing or cannot be loaded the first call raises.

The decode-pool path (Cloudflare Kimi/GLM serving write-up): quantise-on-append
of each new token's K/V into e4m3 pages, page-tag bump on reallocation, the
separate batched tag check that aborts stale requests, and split-KV decode
attention over the FP8 (or BF16) cache with a cross-split combine.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8kv.so")

FPK_OK, FPK_EINVAL, FPK_EUNSUPPORTED, FPK_ENOSPC, FPK_ECUDA = 0, 1, 2, 3, 4

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/fp8kv.h
SIGNATURES = {
    "fpk_version": (ctypes.c_int, []),
    "fpk_selftest_bounded_wait": (ctypes.c_int, [_P, _P, _P]),
    "fpk_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "fpk_kv_append_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P,
                                         _I32, _I32, _I32, _I32, _I32, _P]),
    "fpk_kv_append_bf16": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _P, _P,
                                          _I32, _I32, _I32, _I32, _I32, _P]),
    "fpk_kv_prefill_fp8": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _P, _P, _I32, _P, _P, _P,
                                          _I32, _I32, _I32, _I32, _I32, _P]),
    "fpk_kv_prefill_bf16": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _I32, _P, _P, _P,
                                           _I32, _I32, _I32, _I32, _I32, _P]),
    "fpk_quantize_e4m3": (ctypes.c_int, [_P, _P, _P, _I64, _P]),
    "fpk_amax_scale_bf16": (ctypes.c_int, [_P, _I64, _P, _P, _P]),
    "fpk_page_tags_bump": (ctypes.c_int, [_P, _P, _I32, _I32, _P]),
    "fpk_page_tags_validate": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _I32, _I32, _P, _P, _P]),
    "fpk_decode_append_check_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P,
                                                   _I32, _I32, _I32, _I32, _I32, _P]),
    "fpk_decode_append_check_bf16": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _P, _P,
                                                    _I32, _I32, _I32, _I32, _I32, _P]),
    "fpk_decode_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "fpk_paged_decode_attn_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _P,
                                                 _SZ, _I32, _F, _I32, _I32, _I32, _I32, _I32, _I32,
                                                 _P]),
    "fpk_paged_decode_attn_fp8_tc": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _P,
                                                    _SZ, _I32, _F, _I32, _I32, _I32, _I32, _I32,
                                                    _I32, _P]),
    "fpk_paged_decode_attn_bf16": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _P, _P, _P, _SZ,
                                                  _I32, _F, _I32, _I32, _I32, _I32, _I32, _I32, _P]),
    "fpk_paged_decode_attn_fp8_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P, _P, _P,
                                                         _P, _I32, _F, _I32, _I32, _I32, _I32, _I32,
                                                         _I32, _P]),
    "fpk_decode_step_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P,
                                           _P, _P, _SZ, _I32, _F, _I32, _I32, _I32, _I32, _I32,
                                           _I32, _P]),
    "fpk_decode_step_bf16": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                            _SZ, _I32, _F, _I32, _I32, _I32, _I32, _I32, _I32, _P]),
    "fpk_decode_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "fpk_w4_quantize": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _P]),
    "fpk_w4_gemv": (ctypes.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _P]),
    "fpk_w8_quantize": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _P]),
    "fpk_w8_gemv": (ctypes.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _P]),
}

_lock = threading.Lock()
_lib = None


class FpkError(RuntimeError):
    pass


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfp8kv.so (built by fp8_paged_kv_gb300.build); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise FpkError(f"{path} not found: build it first "
                               "(python -m fp8_paged_kv_gb300.build); there is no fallback")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int, what: str) -> None:
    if status != FPK_OK:
        msg = load_library().fpk_status_str(status).decode()
        raise FpkError(f"{what}: status {status} ({msg})")


def _ptr(t, dtype=None, name="tensor", allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise FpkError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise FpkError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise FpkError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise FpkError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise FpkError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_U8 = torch.uint8
_I32T = torch.int32
_F32 = torch.float32
_BF16 = torch.bfloat16
_TAGS = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
_BF16_LIKE = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)


def version() -> int:
    return load_library().fpk_version()


def fpk_kv_append_fp8(k_new, v_new, kv_pool, k_scale, v_scale, page_table, seq_lens,
                      live_tags=None, expected_tags=None, abort_mask=None, *, Hkv, D, page_size,
                      num_pages, stream=None):
    B, max_pages = page_table.shape
    _check(load_library().fpk_kv_append_fp8(
        _ptr(k_new, _BF16_LIKE, "k_new"), _ptr(v_new, _BF16_LIKE, "v_new"),
        _ptr(kv_pool, _U8, "kv_pool"),
        _ptr(k_scale, _F32, "k_scale"), _ptr(v_scale, _F32, "v_scale"),
        _ptr(page_table, _I32T, "page_table"), max_pages, _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(live_tags, _TAGS, "live_tags", True), _ptr(expected_tags, _TAGS, "expected_tags", True),
        _ptr(abort_mask, _U8, "abort_mask", True), B, Hkv, D, page_size, num_pages,
        _stream(stream)), "fpk_kv_append_fp8")


def fpk_kv_append_bf16(k_new, v_new, kv_pool, page_table, seq_lens, live_tags=None,
                       expected_tags=None, abort_mask=None, *, Hkv, D, page_size, num_pages,
                       stream=None):
    B, max_pages = page_table.shape
    _check(load_library().fpk_kv_append_bf16(
        _ptr(k_new, _BF16_LIKE, "k_new"), _ptr(v_new, _BF16_LIKE, "v_new"),
        _ptr(kv_pool, _BF16_LIKE, "kv_pool"),
        _ptr(page_table, _I32T, "page_table"), max_pages, _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(live_tags, _TAGS, "live_tags", True), _ptr(expected_tags, _TAGS, "expected_tags", True),
        _ptr(abort_mask, _U8, "abort_mask", True), B, Hkv, D, page_size, num_pages,
        _stream(stream)), "fpk_kv_append_bf16")


def fpk_kv_prefill_fp8(k, v, cu_seqlens, kv_pool, k_scale, v_scale, page_table,
                       live_tags=None, expected_tags=None, abort_mask=None, *, Hkv, D, page_size,
                       num_pages, stream=None):
    B, max_pages = page_table.shape
    _check(load_library().fpk_kv_prefill_fp8(
        _ptr(k, _BF16_LIKE, "k"), _ptr(v, _BF16_LIKE, "v"), _ptr(cu_seqlens, _I32T, "cu_seqlens"),
        k.shape[0], _ptr(kv_pool, _U8, "kv_pool"),
        _ptr(k_scale, _F32, "k_scale"), _ptr(v_scale, _F32, "v_scale"),
        _ptr(page_table, _I32T, "page_table"), max_pages,
        _ptr(live_tags, _TAGS, "live_tags", True), _ptr(expected_tags, _TAGS, "expected_tags", True),
        _ptr(abort_mask, _U8, "abort_mask", True), B, Hkv, D, page_size, num_pages,
        _stream(stream)), "fpk_kv_prefill_fp8")


def fpk_kv_prefill_bf16(k, v, cu_seqlens, kv_pool, page_table, live_tags=None,
                        expected_tags=None, abort_mask=None, *, Hkv, D, page_size, num_pages,
                        stream=None):
    B, max_pages = page_table.shape
    _check(load_library().fpk_kv_prefill_bf16(
        _ptr(k, _BF16_LIKE, "k"), _ptr(v, _BF16_LIKE, "v"), _ptr(cu_seqlens, _I32T, "cu_seqlens"),
        k.shape[0], _ptr(kv_pool, _BF16_LIKE, "kv_pool"),
        _ptr(page_table, _I32T, "page_table"), max_pages,
        _ptr(live_tags, _TAGS, "live_tags", True), _ptr(expected_tags, _TAGS, "expected_tags", True),
        _ptr(abort_mask, _U8, "abort_mask", True), B, Hkv, D, page_size, num_pages,
        _stream(stream)), "fpk_kv_prefill_bf16")


def fpk_decode_append_check_fp8(k_new, v_new, kv_pool, k_scale, v_scale, page_table, seq_lens,
                                live_tags, expected_tags, abort_mask, *, Hkv, D, page_size,
                                num_pages, stream=None):
    B, max_pages = page_table.shape
    _check(load_library().fpk_decode_append_check_fp8(
        _ptr(k_new, _BF16_LIKE, "k_new"), _ptr(v_new, _BF16_LIKE, "v_new"),
        _ptr(kv_pool, _U8, "kv_pool"), _ptr(k_scale, _F32, "k_scale"), _ptr(v_scale, _F32, "v_scale"),
        _ptr(page_table, _I32T, "page_table"), max_pages, _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(live_tags, _TAGS, "live_tags"), _ptr(expected_tags, _TAGS, "expected_tags"),
        _ptr(abort_mask, _U8, "abort_mask"), B, Hkv, D, page_size, num_pages, _stream(stream)),
        "fpk_decode_append_check_fp8")


def fpk_decode_append_check_bf16(k_new, v_new, kv_pool, page_table, seq_lens, live_tags,
                                 expected_tags, abort_mask, *, Hkv, D, page_size, num_pages,
                                 stream=None):
    B, max_pages = page_table.shape
    _check(load_library().fpk_decode_append_check_bf16(
        _ptr(k_new, _BF16_LIKE, "k_new"), _ptr(v_new, _BF16_LIKE, "v_new"),
        _ptr(kv_pool, _BF16_LIKE, "kv_pool"),
        _ptr(page_table, _I32T, "page_table"), max_pages, _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(live_tags, _TAGS, "live_tags"), _ptr(expected_tags, _TAGS, "expected_tags"),
        _ptr(abort_mask, _U8, "abort_mask"), B, Hkv, D, page_size, num_pages, _stream(stream)),
        "fpk_decode_append_check_bf16")


def fpk_quantize_e4m3(x, scale, out, stream=None):
    _check(load_library().fpk_quantize_e4m3(_ptr(x, _F32, "x"), _ptr(scale, _F32, "scale"),
                                            _ptr(out, _U8, "out"), x.numel(), _stream(stream)),
           "fpk_quantize_e4m3")


def fpk_amax_scale_bf16(x, scale, scratch, stream=None):
    _check(load_library().fpk_amax_scale_bf16(_ptr(x, _BF16_LIKE, "x"), x.numel(),
                                              _ptr(scale, _F32, "scale"), _ptr(scratch, _TAGS, "scratch"),
                                              _stream(stream)), "fpk_amax_scale_bf16")


def fpk_page_tags_bump(live_tags, pages, *, num_pages, stream=None):
    _check(load_library().fpk_page_tags_bump(_ptr(live_tags, _TAGS, "live_tags"),
                                             _ptr(pages, _I32T, "pages"), pages.numel(), num_pages,
                                             _stream(stream)), "fpk_page_tags_bump")


def fpk_page_tags_validate(page_table, expected_tags, seq_lens, live_tags, abort_mask,
                           abort_count=None, *, num_pages, page_size, stream=None):
    B, max_pages = page_table.shape
    _check(load_library().fpk_page_tags_validate(
        _ptr(page_table, _I32T, "page_table"), _ptr(expected_tags, _TAGS, "expected_tags"),
        _ptr(seq_lens, _I32T, "seq_lens"), max_pages, _ptr(live_tags, _TAGS, "live_tags"),
        num_pages, B, page_size, _ptr(abort_mask, _U8, "abort_mask"),
        _ptr(abort_count, _I32T, "abort_count", True), _stream(stream)), "fpk_page_tags_validate")


def fpk_decode_workspace_bytes(B, Hq, Hkv, D=128, num_splits=0) -> int:
    n = load_library().fpk_decode_workspace_bytes(B, Hq, Hkv, D, num_splits)
    if n == 0 and B > 0:
        raise FpkError("fpk_decode_workspace_bytes: invalid shape or no CUDA device")
    return int(n)


def fpk_paged_decode_attn_fp8(q, kv_pool, k_scale, v_scale, page_table, seq_lens,
                              abort_mask, out, lse, workspace, *, Hkv, page_size, num_pages,
                              sm_scale, num_splits=0, stream=None):
    B, Hq, D = q.shape
    _check(load_library().fpk_paged_decode_attn_fp8(
        _ptr(q, _BF16_LIKE, "q"), _ptr(kv_pool, _U8, "kv_pool"),
        _ptr(k_scale, _F32, "k_scale"), _ptr(v_scale, _F32, "v_scale"),
        _ptr(page_table, _I32T, "page_table"), page_table.shape[1], _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(abort_mask, _U8, "abort_mask", True), _ptr(out, _F32, "out"),
        _ptr(lse, _F32, "lse", True), _ptr(workspace, _U8, "workspace"),
        workspace.numel(), num_splits, sm_scale, B, Hq, Hkv, D, page_size, num_pages,
        _stream(stream)), "fpk_paged_decode_attn_fp8")


def fpk_paged_decode_attn_fp8_tc(q, kv_pool, k_scale, v_scale, page_table, seq_lens,
                                 abort_mask, out, lse, workspace, *, Hkv, page_size, num_pages,
                                 sm_scale, num_splits=0, stream=None):
    """fpk_paged_decode_attn_fp8 on the tcgen05 tensor cores (same arguments)."""
    B, Hq, D = q.shape
    _check(load_library().fpk_paged_decode_attn_fp8_tc(
        _ptr(q, _BF16_LIKE, "q"), _ptr(kv_pool, _U8, "kv_pool"),
        _ptr(k_scale, _F32, "k_scale"), _ptr(v_scale, _F32, "v_scale"),
        _ptr(page_table, _I32T, "page_table"), page_table.shape[1], _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(abort_mask, _U8, "abort_mask", True), _ptr(out, _F32, "out"),
        _ptr(lse, _F32, "lse", True), _ptr(workspace, _U8, "workspace"),
        workspace.numel(), num_splits, sm_scale, B, Hq, Hkv, D, page_size, num_pages,
        _stream(stream)), "fpk_paged_decode_attn_fp8_tc")


def fpk_decode_step_fp8(k_new, v_new, kv_pool, k_scale, v_scale, page_table, seq_lens, live_tags,
                        expected_tags, abort_mask, q, out, lse, workspace, *, Hkv, page_size,
                        num_pages, sm_scale, num_splits=0, stream=None):
    B, Hq, D = q.shape
    _check(load_library().fpk_decode_step_fp8(
        _ptr(k_new, _BF16_LIKE, "k_new"), _ptr(v_new, _BF16_LIKE, "v_new"), _ptr(kv_pool, _U8, "kv_pool"),
        _ptr(k_scale, _F32, "k_scale"), _ptr(v_scale, _F32, "v_scale"),
        _ptr(page_table, _I32T, "page_table"), page_table.shape[1], _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(live_tags, _TAGS, "live_tags", True), _ptr(expected_tags, _TAGS, "expected_tags", True),
        _ptr(abort_mask, _U8, "abort_mask", True), _ptr(q, _BF16_LIKE, "q"), _ptr(out, _F32, "out"),
        _ptr(lse, _F32, "lse", True), _ptr(workspace, _U8, "workspace"), workspace.numel(),
        num_splits, sm_scale, B, Hq, Hkv, D, page_size, num_pages, _stream(stream)),
        "fpk_decode_step_fp8")


def fpk_decode_step_bf16(k_new, v_new, kv_pool, page_table, seq_lens, live_tags, expected_tags,
                         abort_mask, q, out, lse, workspace, *, Hkv, page_size, num_pages, sm_scale,
                         num_splits=0, stream=None):
    B, Hq, D = q.shape
    _check(load_library().fpk_decode_step_bf16(
        _ptr(k_new, _BF16_LIKE, "k_new"), _ptr(v_new, _BF16_LIKE, "v_new"),
        _ptr(kv_pool, _BF16_LIKE, "kv_pool"), _ptr(page_table, _I32T, "page_table"),
        page_table.shape[1], _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(live_tags, _TAGS, "live_tags", True), _ptr(expected_tags, _TAGS, "expected_tags", True),
        _ptr(abort_mask, _U8, "abort_mask", True), _ptr(q, _BF16_LIKE, "q"), _ptr(out, _F32, "out"),
        _ptr(lse, _F32, "lse", True),
        _ptr(workspace, _U8, "workspace"), workspace.numel(), num_splits, sm_scale, B, Hq, Hkv, D,
        page_size, num_pages, _stream(stream)), "fpk_decode_step_bf16")


def fpk_paged_decode_attn_bf16(q, kv_pool, page_table, seq_lens, abort_mask, out, lse,
                               workspace, *, Hkv, page_size, num_pages, sm_scale, num_splits=0,
                               stream=None):
    B, Hq, D = q.shape
    _check(load_library().fpk_paged_decode_attn_bf16(
        _ptr(q, _BF16_LIKE, "q"), _ptr(kv_pool, _BF16_LIKE, "kv_pool"),
        _ptr(page_table, _I32T, "page_table"),
        page_table.shape[1], _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(abort_mask, _U8, "abort_mask", True), _ptr(out, _F32, "out"),
        _ptr(lse, _F32, "lse", True), _ptr(workspace, _U8, "workspace"),
        workspace.numel(), num_splits, sm_scale, B, Hq, Hkv, D, page_size, num_pages,
        _stream(stream)), "fpk_paged_decode_attn_bf16")


def fpk_paged_decode_attn_fp8_noalloc(q, kv_pool, k_scale, v_scale, page_table, seq_lens,
                                      abort_mask, out, lse, *, Hkv, page_size, num_pages, sm_scale,
                                      num_splits=0, stream=None):
    """FP8 decode attention without a caller workspace, for callers that cannot
    allocate device memory; the scratch is a fixed array inside the library
    (batches needing more than 16 MiB of it are rejected).  Calls that overlap
    on the GPU share that scratch and race."""
    B, Hq, D = q.shape
    _check(load_library().fpk_paged_decode_attn_fp8_noalloc(
        _ptr(q, _BF16_LIKE, "q"), _ptr(kv_pool, _U8, "kv_pool"),
        _ptr(k_scale, _F32, "k_scale"), _ptr(v_scale, _F32, "v_scale"),
        _ptr(page_table, _I32T, "page_table"), page_table.shape[1], _ptr(seq_lens, _I32T, "seq_lens"),
        _ptr(abort_mask, _U8, "abort_mask", True), _ptr(out, _F32, "out"),
        _ptr(lse, _F32, "lse", True), num_splits, sm_scale, B, Hq, Hkv, D, page_size, num_pages,
        _stream(stream)), "fpk_paged_decode_attn_fp8_noalloc")


def fpk_decode_status(workspace, stream=None) -> int:
    """Status word of an attention workspace; workspace=None reads the one of the
    last allocation-free call on the current device."""
    v = ctypes.c_int32(0)
    _check(load_library().fpk_decode_status(_ptr(workspace, _U8, "workspace", allow_none=True),
                                            ctypes.byref(v), _stream(stream)), "fpk_decode_status")
    return int(v.value)


def fpk_selftest_bounded_wait(status, elapsed_ns, stream=None):
    """One CTA waits on an mbarrier nothing arrives on; the bounded wait gives up
    after its limit and reports it in status[0] (elapsed time in elapsed_ns[0])."""
    _check(load_library().fpk_selftest_bounded_wait(_ptr(status, torch.int32, "status"),
                                                    _ptr(elapsed_ns, torch.int64, "elapsed_ns"),
                                                    _stream(stream)), "fpk_selftest_bounded_wait")


# ---------------------------------------------------------------- weight GEMV
def fpk_w4_quantize(w, codes, scales, stream=None):
    N, K = w.shape
    _check(load_library().fpk_w4_quantize(_ptr(w, _BF16_LIKE, "w"), _ptr(codes, _U8, "codes"),
                                          _ptr(scales, _BF16_LIKE, "scales"), N, K, _stream(stream)),
           "fpk_w4_quantize")


def fpk_w4_gemv(x, codes, scales, y, stream=None):
    B, K = x.shape
    N = y.shape[1]
    _check(load_library().fpk_w4_gemv(_ptr(x, _BF16_LIKE, "x"), _ptr(codes, _U8, "codes"),
                                      _ptr(scales, _BF16_LIKE, "scales"), _ptr(y, _F32, "y"), B, N, K,
                                      _stream(stream)), "fpk_w4_gemv")


def fpk_w8_quantize(w, codes, row_scales, stream=None):
    N, K = w.shape
    _check(load_library().fpk_w8_quantize(_ptr(w, _BF16_LIKE, "w"), _ptr(codes, _U8, "codes"),
                                          _ptr(row_scales, _F32, "row_scales"), N, K, _stream(stream)),
           "fpk_w8_quantize")


def fpk_w8_gemv(x, codes, row_scales, y, stream=None):
    B, K = x.shape
    N = y.shape[1]
    _check(load_library().fpk_w8_gemv(_ptr(x, _BF16_LIKE, "x"), _ptr(codes, _U8, "codes"),
                                      _ptr(row_scales, _F32, "row_scales"), _ptr(y, _F32, "y"), B, N, K,
                                      _stream(stream)), "fpk_w8_gemv")
