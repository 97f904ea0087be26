"""Seeded synthetic inputs for the FP8 paged-KV decode path.

Shared by the oracle tests, the GPU parity tests and the benchmark.  This
module draws random numbers, rounds them to bf16 bit patterns and lays out
page tables and tags; it holds none of the method's arithmetic (no e4m3
coding, no attention, no tag check).  Every array is numpy and every draw
comes from a PCG64 stream keyed by (seed, purpose, index), so a request's
values can be regenerated alone and the results are the same on any host.

Workloads (shapes of the decode-pool serving described in the Cloudflare
Kimi/GLM write-up pages; the pages' own production traffic and eval suites
are not available, these stand in for them by shape only):

  tiny      B=2, Hq=8/Hkv=2, ps=16, 64-page pool, contexts 100 and 257,
            request 1 carries one stale expected tag, 1 decode step.
  b32_8k    B=32, Hq=64/Hkv=8, ps=16, every context 8192, pool exactly
            16384 pages; K,V ~ N(0, 0.5^2) with 1% of the Hkv*D channels x20.
  b64_var   B=64, Hq=64/Hkv=8, ps=16, contexts U[1024, 16384], pool 1.2x the
            pages needed after 256 decode steps, pages scattered.
  long128k  B=4, Hq=64/Hkv=8, ps=64, every context 131072.
  churn     256 requests, Hq=32/Hkv=8, ps=16, prompts of 8192 tokens
            (decode steps and reallocation are driven by the host ledger).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

D_HEAD = 128


def rng_for(seed: int, *key) -> np.random.Generator:
    """Independent PCG64 stream for (seed, key...) -- platform independent."""
    words = [int(seed) & 0xFFFFFFFF]
    for k in key:
        if isinstance(k, str):
            words.extend(k.encode())
        else:
            words.append(int(k) & 0xFFFFFFFF)
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(words)))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns uint16 bits.

    Input preparation only: workloads are defined as bf16 tensors.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) >> 16).astype(np.uint16)
    if nan.any():
        r[nan] = ((u[nan] >> 16) | np.uint32(0x40)).astype(np.uint16)
    return r


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    """One decode-pool batch: prompts already in the cache plus decode steps.

    Attributes (numpy):
      q            uint16 bf16 bits [B][Hq][D] (the query of decode step 0)
      prompt_lens  int32 [B]  tokens written before the first decode step
      k_prompt     uint16 [N][Hkv][D], v_prompt likewise, cu_prompt int32 [B+1]
      page_table   int32 [B][max_pages], -1 beyond the pages a request owns
      live_tags    uint32 [num_pages]
      expected_tags uint32 [B][max_pages]
      k_scale, v_scale  float32 per-tensor scales (amax / 448 of the values)
    """
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    num_pages: int
    max_pages: int
    steps: int
    prompt_lens: np.ndarray
    cu_prompt: np.ndarray
    k_prompt: np.ndarray
    v_prompt: np.ndarray
    q: np.ndarray
    page_table: np.ndarray
    live_tags: np.ndarray
    expected_tags: np.ndarray
    k_scale: np.float32
    v_scale: np.float32
    sigma: float = 1.0
    outlier_channels: Optional[np.ndarray] = None
    num_splits: int = 0
    stale: list = dataclasses.field(default_factory=list)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def sm_scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.D)))

    def seq_lens_after(self, step: int) -> np.ndarray:
        """Context length of every request once decode step `step` (0-based) appended."""
        return (self.prompt_lens + step + 1).astype(np.int32)

    def step_tokens(self, step: int):
        """bf16 bits (k_new, v_new), each [B][Hkv][D], for decode step `step`."""
        g = rng_for(self.seed, "step", step)
        k = self._draw(g, (self.B, self.Hkv, self.D))
        v = self._draw(g, (self.B, self.Hkv, self.D))
        return bf16_bits(k), bf16_bits(v)

    def step_query(self, step: int) -> np.ndarray:
        if step == 0:
            return self.q
        g = rng_for(self.seed, "q", step)
        return bf16_bits(g.standard_normal((self.B, self.Hq, self.D), dtype=np.float32))

    def _draw(self, g, shape):
        x = g.standard_normal(shape, dtype=np.float32) * np.float32(self.sigma)
        if self.outlier_channels is not None and self.outlier_channels.size:
            flat = x.reshape(shape[:-2] + (self.Hkv * self.D,))
            flat[..., self.outlier_channels] *= np.float32(20.0)
        return x

    def kv_bytes(self, fp8: bool = True, step: int = 0) -> int:
        """KV bytes one attention pass over the contexts after `step` reads."""
        tokens = int(self.seq_lens_after(step).sum())
        return tokens * 2 * self.Hkv * self.D * (1 if fp8 else 2)


def _scale_of(amax: float) -> np.float32:
    a = np.float32(amax)
    return np.float32(1.0) if a == 0 else np.float32(a / np.float32(448.0))


def _build(name, seed, B, Hq, Hkv, ps, prompt_lens, steps, num_pages, *, sigma=1.0,
           outlier_frac=0.0, scatter=True, max_pages=None, D=D_HEAD, num_splits=0):
    prompt_lens = np.asarray(prompt_lens, np.int32)
    final_lens = prompt_lens + steps
    need = -(-final_lens // ps)
    if max_pages is None:
        max_pages = int(need.max()) if B else 0
    total = int(need.sum())
    assert total <= num_pages, "pool too small for the workload"
    # page assignment: a seeded permutation of the pool, handed out in order
    perm = rng_for(seed, "perm").permutation(num_pages).astype(np.int32) if scatter \
        else np.arange(num_pages, dtype=np.int32)
    page_table = np.full((B, max(max_pages, 1)), -1, np.int32)
    o = 0
    for r in range(B):
        page_table[r, :need[r]] = perm[o:o + need[r]]
        o += need[r]
    live = rng_for(seed, "tags").integers(0, 2**32, size=num_pages, dtype=np.uint64).astype(np.uint32)
    expected = np.zeros_like(page_table, dtype=np.uint32)
    mapped = page_table >= 0
    expected[mapped] = live[page_table[mapped]]

    n_ch = int(round(outlier_frac * Hkv * D))
    outl = np.sort(rng_for(seed, "outliers").choice(Hkv * D, size=n_ch, replace=False)) \
        if n_ch else None
    wl = Workload(name=name, seed=seed, B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                  num_pages=num_pages, max_pages=page_table.shape[1], steps=steps,
                  prompt_lens=prompt_lens, cu_prompt=np.zeros(B + 1, np.int32),
                  k_prompt=np.zeros((0, Hkv, D), np.uint16), v_prompt=np.zeros((0, Hkv, D), np.uint16),
                  q=bf16_bits(rng_for(seed, "q", 0).standard_normal((B, Hq, D), dtype=np.float32)),
                  page_table=page_table, live_tags=live, expected_tags=expected,
                  k_scale=np.float32(1), v_scale=np.float32(1), sigma=sigma,
                  outlier_channels=outl, num_splits=num_splits)
    cu = np.zeros(B + 1, np.int64)
    cu[1:] = np.cumsum(prompt_lens)
    assert cu[-1] < 2**31
    wl.cu_prompt = cu.astype(np.int32)
    N = int(cu[-1])
    kp = np.empty((N, Hkv, D), np.uint16)
    vp = np.empty((N, Hkv, D), np.uint16)

    def fill(job):
        # one chunk of one prompt from its own stream: K rows, then V rows
        r, c = job
        n0 = c * PROMPT_CHUNK
        n1 = min(int(prompt_lens[r]), n0 + PROMPT_CHUNK)
        g = rng_for(seed, "prompt", r, c)
        amax = []
        for dst in (kp, vp):
            x = wl._draw(g, (n1 - n0, Hkv, D))
            dst[cu[r] + n0:cu[r] + n1] = bf16_bits(x)
            amax.append(_amax_bf16(x))
        return amax

    jobs = [(r, c) for r in range(B) for c in range(-(-int(prompt_lens[r]) // PROMPT_CHUNK))]
    kmax = vmax = 0.0
    with _draw_pool() as ex:
        for km, vm in ex.map(fill, jobs):
            kmax, vmax = max(kmax, km), max(vmax, vm)
    for s in range(steps):
        k, v = wl.step_tokens(s)
        kmax = max(kmax, float(np.abs(bf16_to_f32(k)).max()))
        vmax = max(vmax, float(np.abs(bf16_to_f32(v)).max()))
    wl.k_prompt, wl.v_prompt = kp, vp
    wl.k_scale, wl.v_scale = _scale_of(kmax), _scale_of(vmax)
    return wl


# tokens of a prompt drawn from one stream; chunks are drawn in parallel
PROMPT_CHUNK = 4096


def _amax_bf16(x: np.ndarray) -> float:
    """max |bf16(x)| over a float32 array: rounding to nearest is monotonic in
    |x|, so it is the rounding of max |x|."""
    if x.size == 0:
        return 0.0
    m = np.float32(max(float(x.max()), -float(x.min())))
    return float(bf16_to_f32(bf16_bits(np.array([m], np.float32)))[0])


def _draw_pool():
    """Threads for drawing prompt chunks (numpy's generators and ufuncs release
    the interpreter lock on large arrays)."""
    import concurrent.futures as cf
    import os
    return cf.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))


def tiny(seed: int = 1) -> Workload:
    """B=2, contexts 100 and 257 after one decode step; request 1 has one stale tag."""
    wl = _build("tiny", seed, B=2, Hq=8, Hkv=2, ps=16, prompt_lens=[99, 256], steps=1,
                num_pages=64)
    # one stale expected entry in request 1: the page was reallocated once since
    P1 = -(-257 // 16)
    i = int(rng_for(seed, "stale").integers(0, P1))
    wl.expected_tags[1, i] = wl.expected_tags[1, i] - np.uint32(1)
    wl.stale = [(1, i)]
    return wl


def b32_8k(seed: int = 2) -> Workload:
    """B=32, every context 8192 (8191 prompt + 1 decode), pool exactly 16384 pages."""
    return _build("b32_8k", seed, B=32, Hq=64, Hkv=8, ps=16, prompt_lens=[8191] * 32, steps=1,
                  num_pages=16384, sigma=0.5, outlier_frac=0.01)


def b64_var(seed: int = 3, steps: int = 256) -> Workload:
    """B=64, prompts U[1024, 16384], `steps` decode steps, pool 1.2x the pages needed."""
    lens = rng_for(seed, "lens").integers(1024, 16384, size=64, endpoint=True).astype(np.int32)
    need = int((-(-(lens + steps) // 16)).sum())
    return _build("b64_var", seed, B=64, Hq=64, Hkv=8, ps=16, prompt_lens=lens, steps=steps,
                  num_pages=int(math.ceil(1.2 * need)))


def long128k(seed: int = 4) -> Workload:
    """B=4, every context 131072 (131071 prompt + 1 decode), ps=64, 64 splits per (r, kv head)."""
    return _build("long128k", seed, B=4, Hq=64, Hkv=8, ps=64, prompt_lens=[131071] * 4, steps=1,
                  num_pages=8192, num_splits=64 * 4 * 8)


def custom(seed: int, B: int, Hq: int, Hkv: int, ps: int, prompt_lens, steps: int = 1,
           pool_factor: float = 1.5, sigma: float = 1.0, outlier_frac: float = 0.0,
           extra_pages: int = 0, max_pages=None) -> Workload:
    """Small parity cases: any lengths (zeros and ragged tails allowed)."""
    lens = np.asarray(prompt_lens, np.int32)
    need = int((-(-(lens + steps) // ps)).sum())
    pool = max(1, int(math.ceil(pool_factor * need)) + extra_pages)
    return _build(f"custom{seed}", seed, B=B, Hq=Hq, Hkv=Hkv, ps=ps, prompt_lens=lens,
                  steps=steps, num_pages=pool, sigma=sigma, outlier_frac=outlier_frac,
                  max_pages=max_pages)


WORKLOADS = {"tiny": tiny, "b32_8k": b32_8k, "b64_var": b64_var, "long128k": long128k}
