"""Device-resident decode pool: torch allocates, libfp8kv computes.

A DecodePool holds one layer's paged KV pool (e4m3 or bf16), the page table,
the live and expected page tags, the per-tensor scales and the output and
workspace buffers of a decode batch, and runs the decode step in the order
the pages describe: write the new token's K/V into its page, check every
request's (page, tag) mapping in a separate batched operation, then attend
over the pages of the requests that passed.  All arithmetic runs in the
library's kernels (see fp8_paged_kv_gb300.__init__); this module only moves
arrays between numpy and the device.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (fpk_decode_append_check_bf16, fpk_decode_append_check_fp8, fpk_decode_step_bf16,
               fpk_decode_step_fp8, fpk_decode_workspace_bytes, fpk_kv_append_bf16, fpk_kv_append_fp8,
               fpk_kv_prefill_bf16, fpk_kv_prefill_fp8, fpk_page_tags_bump,
               fpk_page_tags_validate, fpk_paged_decode_attn_bf16, fpk_paged_decode_attn_fp8,
               fpk_paged_decode_attn_fp8_tc)

NAN_E4M3 = 0x7F          # e4m3 NaN code: fills slots no token was written to
NAN_BF16 = 0x7FC0


def to_device(a: np.ndarray, device) -> torch.Tensor:
    """numpy -> CUDA tensor; uint32 tags travel as int32, bf16 bits as bfloat16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def _arena(device, specs):
    """One device buffer holding several tensors, each at a 256-byte aligned
    offset, so that a step's inputs (or results) move between host and device
    in one copy.  Returns (buffer, {name: view})."""
    offs, total = [], 0
    for _, shape, dtype in specs:
        total = (total + 255) // 256 * 256
        offs.append(total)
        total += int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.zeros(max(total, 1), dtype=torch.uint8, device=device)
    views = {}
    for (name, shape, dtype), off in zip(specs, offs):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        views[name] = buf[off:off + n].view(dtype).view(shape)
    return buf, views


class DecodePool:
    def __init__(self, wl, fp8: bool = True, device="cuda", num_splits: int | None = None,
                 tensor_cores: bool = False):
        self.wl = wl
        self.fp8 = fp8
        # FP8 attention on the tcgen05 tensor cores (fpk_paged_decode_attn_fp8_tc)
        # instead of the warp-level kernel; attend() only
        self.tensor_cores = tensor_cores
        self.device = torch.device(device)
        dev = self.device
        n = 2 * wl.num_pages * wl.Hkv * wl.page_size * wl.D      # K and V of every slot
        if fp8:
            self.kv_pool = torch.full((n,), NAN_E4M3, dtype=torch.uint8, device=dev)
        else:
            self.kv_pool = torch.full((n,), NAN_BF16, dtype=torch.int16, device=dev).view(torch.bfloat16)
        self.page_table = to_device(wl.page_table, dev)
        self.live_tags = to_device(wl.live_tags, dev)
        self.expected_tags = to_device(wl.expected_tags, dev)
        self.k_scale = torch.tensor([float(wl.k_scale)], dtype=torch.float32, device=dev)
        self.v_scale = torch.tensor([float(wl.v_scale)], dtype=torch.float32, device=dev)
        # a step's inputs and results, each in one buffer (io_in, io_out); a
        # second pair is made on demand for pipelined host steps (io_slot)
        self._io = [self._new_io()]
        self.io_slot(0)
        self.seq_lens.copy_(to_device(wl.prompt_lens.astype(np.int32), dev))
        self.q.copy_(to_device(wl.q, dev))
        self.abort_count = torch.zeros(1, dtype=torch.int32, device=dev)
        self.num_splits = wl.num_splits if num_splits is None else num_splits
        ws = fpk_decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.D, self.num_splits)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev)
        self.count_aborts = True

    def _new_io(self):
        wl, dev = self.wl, self.device
        io_in, v_in = _arena(dev, [("q", (wl.B, wl.Hq, wl.D), torch.bfloat16),
                                   ("k_new", (wl.B, wl.Hkv, wl.D), torch.bfloat16),
                                   ("v_new", (wl.B, wl.Hkv, wl.D), torch.bfloat16),
                                   ("seq_lens", (wl.B,), torch.int32)])
        io_out, v_out = _arena(dev, [("out", (wl.B, wl.Hq, wl.D), torch.float32),
                                     ("lse", (wl.B, wl.Hq), torch.float32),
                                     ("abort_mask", (wl.B,), torch.uint8)])
        return io_in, v_in, io_out, v_out

    def io_slot(self, i: int):
        """Point the step's inputs and results at I/O buffer pair i (0 or 1)."""
        while len(self._io) <= i:
            self._io.append(self._new_io())
        self.io_in, v_in, self.io_out, v_out = self._io[i]
        self.q, self.k_new, self.v_new, self.seq_lens = (v_in[k] for k in ("q", "k_new", "v_new", "seq_lens"))
        self.out, self.lse, self.abort_mask = (v_out[k] for k in ("out", "lse", "abort_mask"))

    @property
    def kw(self):
        w = self.wl
        return dict(Hkv=w.Hkv, D=w.D, page_size=w.page_size, num_pages=w.num_pages)

    # ---------------------------------------------------------------- writes
    def prefill(self, chunk_tokens: int = 1 << 22):
        """Bulk-write every request's prompt (positions 0..prompt_len-1)."""
        wl = self.wl
        B = wl.B
        cu = wl.cu_prompt.astype(np.int64)
        r0 = 0
        while r0 < B:
            r1 = r0 + 1
            while r1 < B and cu[r1 + 1] - cu[r0] <= chunk_tokens:
                r1 += 1
            # requests [r0, r1) in one call: a page table with only their rows
            k = to_device(wl.k_prompt[cu[r0]:cu[r1]], self.device)
            v = to_device(wl.v_prompt[cu[r0]:cu[r1]], self.device)
            cu_sub = to_device((cu[r0:r1 + 1] - cu[r0]).astype(np.int32), self.device)
            pt = self.page_table[r0:r1]
            ex = self.expected_tags[r0:r1]
            if self.fp8:
                fpk_kv_prefill_fp8(k, v, cu_sub, self.kv_pool, self.k_scale, self.v_scale,
                                   pt, self.live_tags, ex, None, **self.kw)
            else:
                fpk_kv_prefill_bf16(k, v, cu_sub, self.kv_pool, pt, self.live_tags, ex,
                                    None, **self.kw)
            del k, v
            r0 = r1
        torch.cuda.synchronize(self.device)

    def set_step(self, step: int):
        """Upload decode step `step`'s new K/V rows, query and context lengths.
        Existing buffers are overwritten in place (captured CUDA graphs keep
        pointing at them)."""
        kn, vn = self.wl.step_tokens(step)
        new = dict(k_new=to_device(kn, self.device), v_new=to_device(vn, self.device),
                   q=to_device(self.wl.step_query(step), self.device),
                   seq_lens=to_device(self.wl.seq_lens_after(step), self.device))
        for name, t in new.items():
            cur = getattr(self, name)
            if cur is not None and cur.shape == t.shape and cur.dtype == t.dtype:
                cur.copy_(t)
            else:
                setattr(self, name, t)

    def append(self, stream=None, guard: bool = True):
        tags = (self.live_tags, self.expected_tags, self.abort_mask) if guard else (None, None, None)
        if self.fp8:
            fpk_kv_append_fp8(self.k_new, self.v_new, self.kv_pool, self.k_scale,
                              self.v_scale, self.page_table, self.seq_lens, *tags, stream=stream,
                              **self.kw)
        else:
            fpk_kv_append_bf16(self.k_new, self.v_new, self.kv_pool, self.page_table,
                               self.seq_lens, *tags, stream=stream, **self.kw)

    # ----------------------------------------------------------------- tags
    def bump(self, pages: torch.Tensor, stream=None):
        fpk_page_tags_bump(self.live_tags, pages, num_pages=self.wl.num_pages, stream=stream)

    def validate(self, stream=None):
        # count_aborts=False skips the device-side count (and its zeroing); the
        # abort mask alone carries the same information to the host
        fpk_page_tags_validate(self.page_table, self.expected_tags, self.seq_lens, self.live_tags,
                               self.abort_mask, self.abort_count if self.count_aborts else None,
                               num_pages=self.wl.num_pages, page_size=self.wl.page_size,
                               stream=stream)

    # ------------------------------------------------------------ attention
    def attend(self, use_mask: bool = True, stream=None, num_splits: int | None = None):
        wl = self.wl
        ns = self.num_splits if num_splits is None else num_splits
        mask = self.abort_mask if use_mask else None
        kw = dict(Hkv=wl.Hkv, page_size=wl.page_size, num_pages=wl.num_pages,
                  sm_scale=wl.sm_scale, num_splits=ns, stream=stream)
        if self.fp8:
            attn = fpk_paged_decode_attn_fp8_tc if self.tensor_cores else fpk_paged_decode_attn_fp8
            attn(self.q, self.kv_pool, self.k_scale, self.v_scale, self.page_table, self.seq_lens,
                 mask, self.out, self.lse, self.workspace, **kw)
        else:
            fpk_paged_decode_attn_bf16(self.q, self.kv_pool, self.page_table,
                                       self.seq_lens, mask, self.out, self.lse, self.workspace, **kw)

    def append_check(self, stream=None):
        """The step's cache write and batched tag check in one launch."""
        if self.fp8:
            fpk_decode_append_check_fp8(self.k_new, self.v_new, self.kv_pool, self.k_scale,
                                        self.v_scale, self.page_table, self.seq_lens,
                                        self.live_tags, self.expected_tags, self.abort_mask,
                                        stream=stream, **self.kw)
        else:
            fpk_decode_append_check_bf16(self.k_new, self.v_new, self.kv_pool, self.page_table,
                                         self.seq_lens, self.live_tags, self.expected_tags,
                                         self.abort_mask, stream=stream, **self.kw)

    def step(self, validate: bool = True, stream=None):
        """One decode step.  With validation: the cache write and the batched tag
        check (one launch; a separate operation from attention), then attention
        over the requests that passed, launched as a programmatic dependent of
        the check (fpk_decode_step_*).  Without it (the no-op tracker): the same
        two launches with no tag check -- the write unguarded, attention over
        every request.  With count_aborts the check runs as its own launch so
        that it also produces the device-side count."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        if validate and self.count_aborts:
            self.append(stream=main)
            self.validate(stream=main)
            self.attend(use_mask=True, stream=main)
            return
        wl = self.wl
        kw = dict(Hkv=wl.Hkv, page_size=wl.page_size, num_pages=wl.num_pages,
                  sm_scale=wl.sm_scale, num_splits=self.num_splits, stream=main)
        tags = (self.live_tags, self.expected_tags, self.abort_mask) if validate else (None, None, None)
        if self.fp8:
            fpk_decode_step_fp8(self.k_new, self.v_new, self.kv_pool, self.k_scale, self.v_scale,
                                self.page_table, self.seq_lens, *tags, self.q, self.out, self.lse,
                                self.workspace, **kw)
        else:
            fpk_decode_step_bf16(self.k_new, self.v_new, self.kv_pool, self.page_table,
                                 self.seq_lens, *tags, self.q, self.out, self.lse, self.workspace,
                                 **kw)

    # ------------------------------------------------------------- readback
    def pool_bytes(self):
        """Host copy of the KV pool as raw uint8 (e4m3) / uint16 (bf16) elements."""
        if self.fp8:
            return self.kv_pool.cpu().numpy()
        return self.kv_pool.view(torch.int16).cpu().numpy().view(np.uint16)


class HostPipeline:
    """Decode steps fed from pinned host memory and drained back to it, with
    the copies of neighbouring steps under each step's kernels.

    Step i reads its inputs (q, new K/V rows, context lengths: one buffer)
    from host_in[i % len(host_in)] and leaves its results (out, lse, abort
    mask: one buffer) in host_out[i % len(host_out)].  The pool's two I/O
    buffer pairs alternate between steps.  On a copy stream, step i+1's
    inputs go in and step i-1's results come out while step i runs on the
    compute stream; every step still copies its own inputs in and its own
    results out.  Ordering, per buffer pair b = i % 2:
      - copy-in of step i waits until step i-2 (the last user of pair b) ends;
      - step i waits for its copy-in and for the copy-out of step i-2;
      - copy-out of step i waits until step i ends.
    run() only enqueues work (it can be captured in a CUDA graph); the host
    buffers must be pinned and stay alive until the copies complete.
    """

    def __init__(self, pool: "DecodePool", host_in, host_out, validate: bool = True):
        self.pool = pool
        self.host_in = list(host_in)
        self.host_out = list(host_out)
        self.validate = validate
        for h in self.host_in + self.host_out:
            if h.is_cuda or not h.is_pinned():
                raise ValueError("host buffers must be pinned host tensors")
        pool.io_slot(1)
        pool.io_slot(0)
        if any(h.numel() * h.element_size() != pool.io_in.numel() for h in self.host_in) or \
           any(h.numel() * h.element_size() != pool.io_out.numel() for h in self.host_out):
            raise ValueError("host buffers must match the pool's I/O buffers in size")
        self.copy_stream = torch.cuda.Stream(device=pool.device)

    def bytes_per_step(self):
        return self.pool.io_in.numel(), self.pool.io_out.numel()

    def run(self, n: int):
        """Enqueue n pipelined decode steps on the current stream (and the copy stream)."""
        pool, x = self.pool, self.copy_stream
        comp = torch.cuda.current_stream(pool.device)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        done, copied_in, copied_out = [None] * n, [None] * n, [None] * n
        x.wait_stream(comp)

        def copy_in(i):
            with torch.cuda.stream(x):
                if i >= 2:
                    x.wait_event(done[i - 2])
                pool._io[i % 2][0].copy_(self.host_in[i % len(self.host_in)].view(torch.uint8).view(-1),
                                         non_blocking=True)
                copied_in[i] = ev()
                copied_in[i].record(x)

        def copy_out(i):
            with torch.cuda.stream(x):
                x.wait_event(done[i])
                self.host_out[i % len(self.host_out)].view(torch.uint8).view(-1).copy_(
                    pool._io[i % 2][2], non_blocking=True)
                copied_out[i] = ev()
                copied_out[i].record(x)

        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            comp.wait_event(copied_in[i])
            if i >= 2:
                comp.wait_event(copied_out[i - 2])
            pool.io_slot(i % 2)
            pool.step(validate=self.validate, stream=comp)
            done[i] = ev()
            done[i].record(comp)
            if i >= 1:
                copy_out(i - 1)
        copy_out(n - 1)
        comp.wait_stream(x)
        pool.io_slot(0)


def admission_cap(budget_bytes: int, context: int, *, Hkv: int, D: int, page_size: int,
                  fp8: bool):
    """Requests of `context` tokens a one-layer KV pool of `budget_bytes` admits.

    A page holds K and V of page_size tokens for every kv head: 2*Hkv*page_size*D
    elements of 1 byte (e4m3) or 2 (bf16).  The pool has floor(budget / page
    bytes) pages and a request needs ceil(context / page_size) of them.
    Returns (pages in the pool, pages per request, requests admitted).
    """
    page_bytes = 2 * Hkv * page_size * D * (1 if fp8 else 2)
    pages = budget_bytes // page_bytes
    per_request = -(-context // page_size)
    return pages, per_request, (pages // per_request if per_request else 0)
