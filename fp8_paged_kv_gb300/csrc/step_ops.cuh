// step_ops.cuh -- the per-token cache write and the per-request tag check as
// device functions, shared by the stand-alone kernels (kv_write.cu,
// page_tags.cu) and the one-launch append-and-check kernel (decode_step.cu).
#pragma once

#include "common.cuh"
#include "quant.cuh"

namespace fpk {

struct WriteArgs {
  const uint16_t* k_src;     // bf16 [rows][Hkv][D]
  const uint16_t* v_src;
  const int32_t* seq_lens;   // decode mode: position = seq_lens[r] - 1, row r
  const int32_t* cu_seqlens; // prefill mode: row i of request r at position i - cu[r]
  uint8_t* kv_pool;
  const float* k_scale;
  const float* v_scale;
  const int32_t* page_table;
  const uint32_t* live_tags;
  const uint32_t* expected_tags;
  uint8_t* abort_mask;
  int64_t rows;
  int B, Hkv, D, page_size, num_pages, max_pages;
};

__device__ __forceinline__ int request_of_row(const int32_t* cu, int B, int64_t row) {
  // largest r with cu[r] <= row (cu non-decreasing, cu[0] = 0)
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(__ldg(cu + mid)) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One unit of token writing: 8 consecutive dims of one (token row, kv head).
// Returns without writing (and marks the request aborted) when the
// destination slot fails the guard.
template <bool kFp8, bool kPrefill>
__device__ __forceinline__ void write_unit(const WriteArgs& a, int64_t u, const Divisor& ks,
                                           const Divisor& vs) {
  const int chunks = a.D >> 3;
  {
    const int c = static_cast<int>(u % chunks);
    const int h = static_cast<int>((u / chunks) % a.Hkv);
    const int64_t row = u / (static_cast<int64_t>(chunks) * a.Hkv);
    int r, pos;
    if (kPrefill) {
      r = request_of_row(a.cu_seqlens, a.B, row);
      pos = static_cast<int>(row - __ldg(a.cu_seqlens + r));
    } else {
      r = static_cast<int>(row);
      pos = __ldg(a.seq_lens + r) - 1;
      if (pos < 0) return;
    }
    const int pi = pos / a.page_size;
    const int off = pos - pi * a.page_size;
    bool ok = pi < a.max_pages;
    int page = -1;
    if (ok) {
      page = __ldg(a.page_table + static_cast<int64_t>(r) * a.max_pages + pi);
      ok = page >= 0 && page < a.num_pages;
    }
    if (ok && a.live_tags != nullptr && a.expected_tags != nullptr)
      ok = __ldg(a.live_tags + page) ==
           __ldg(a.expected_tags + static_cast<int64_t>(r) * a.max_pages + pi);
    if (!ok) {
      if (a.abort_mask != nullptr) a.abort_mask[r] = 1;
      return;
    }
    const int64_t src = (row * a.Hkv + h) * a.D + 8 * c;
    const uint4 kraw = __ldg(reinterpret_cast<const uint4*>(a.k_src + src));
    const uint4 vraw = __ldg(reinterpret_cast<const uint4*>(a.v_src + src));
    // the token's 16-token tile: K block [16][D], then V block [D][16]
    const int64_t tile = ((static_cast<int64_t>(page) * a.Hkv + h) * (a.page_size >> 4) + (off >> 4)) *
                         2 * 16 * a.D;
    const int64_t kdst = tile + (off & 15) * a.D + 8 * c;
    const int64_t vblk = tile + 16 * a.D;
    const int vcol = off & 15;
    const uint16_t* kb = reinterpret_cast<const uint16_t*>(&kraw);
    const uint16_t* vb = reinterpret_cast<const uint16_t*>(&vraw);
    if (kFp8) {
      uint32_t kw[2];
      uint8_t vq[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float k0 = div_by(bf16_bits_to_float(kb[2 * i]), ks);
        const float k1 = div_by(bf16_bits_to_float(kb[2 * i + 1]), ks);
        const float v0 = div_by(bf16_bits_to_float(vb[2 * i]), vs);
        const float v1 = div_by(bf16_bits_to_float(vb[2 * i + 1]), vs);
        const uint16_t kp = __nv_cvt_float2_to_fp8x2(make_float2(k0, k1), __NV_SATFINITE, __NV_E4M3);
        const uint16_t vp = __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
        if (i & 1) kw[i >> 1] |= static_cast<uint32_t>(kp) << 16; else kw[i >> 1] = kp;
        vq[2 * i] = static_cast<uint8_t>(vp & 0xFF);
        vq[2 * i + 1] = static_cast<uint8_t>(vp >> 8);
      }
      *reinterpret_cast<uint2*>(a.kv_pool + kdst) = make_uint2(kw[0], kw[1]);
#pragma unroll
      for (int i = 0; i < 8; ++i) a.kv_pool[vblk + static_cast<int64_t>(8 * c + i) * 16 + vcol] = vq[i];
    } else {
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.kv_pool) + kdst) = kraw;
      uint16_t* vpool = reinterpret_cast<uint16_t*>(a.kv_pool);
#pragma unroll
      for (int i = 0; i < 8; ++i) vpool[vblk + static_cast<int64_t>(8 * c + i) * 16 + vcol] = vb[i];
    }
  }
}

// One CTA per request.  Each thread checks up to kCheckPerThread table
// entries per round: all table loads of the round, then all live-tag gathers
// (at a clamped, always valid index, so none waits behind a compare), then
// the compares -- two dependent memory round trips per round.
constexpr int kValidateThreads = 256;
constexpr int kCheckPerThread = 8;

// The check of request r by one whole CTA of kValidateThreads threads: writes
// abort_mask[r] and returns whether the request aborts (to every thread).
__device__ __forceinline__ int check_request(const int32_t* __restrict__ page_table,
                                             const uint32_t* __restrict__ expected_tags,
                                             const int32_t* __restrict__ seq_lens, int max_pages,
                                             const uint32_t* __restrict__ live_tags, int num_pages,
                                             int page_size, uint8_t* __restrict__ abort_mask, int r) {
  const int32_t* pt = page_table + static_cast<int64_t>(r) * max_pages;
  const uint32_t* ex = expected_tags + static_cast<int64_t>(r) * max_pages;
  // The first round's table loads do not wait for the context length: they
  // cover the row's first entries (up to its width), and only entries below
  // the request's page count are compared.
  const int L = __ldg(seq_lens + r);
  int P = -1;  // known once L has arrived
  int bad = 0;
  for (int base = 0; base < max_pages && (P < 0 || (base < P && !bad));
       base += kCheckPerThread * kValidateThreads) {
    int page[kCheckPerThread];
    uint32_t want[kCheckPerThread], live[kCheckPerThread];
#pragma unroll
    for (int k = 0; k < kCheckPerThread; ++k) {
      const int i = base + k * kValidateThreads + threadIdx.x;
      page[k] = i < max_pages ? __ldg(pt + i) : 0;
      want[k] = i < max_pages ? __ldg(ex + i) : 0u;
    }
    if (P < 0) {
      P = L > 0 ? (L + page_size - 1) / page_size : 0;
      bad = P > max_pages || (P > 0 && num_pages <= 0);
      if (bad || P == 0) break;  // from here on num_pages > 0: every gather index is valid
    }
#pragma unroll
    for (int k = 0; k < kCheckPerThread; ++k) {
      const bool in_range = page[k] >= 0 && page[k] < num_pages;
      live[k] = __ldg(live_tags + (in_range ? page[k] : 0));
    }
#pragma unroll
    for (int k = 0; k < kCheckPerThread; ++k) {
      const int i = base + k * kValidateThreads + threadIdx.x;
      const bool in_range = page[k] >= 0 && page[k] < num_pages;
      if (i < P && (!in_range || live[k] != want[k])) bad = 1;
    }
  }
  if (P < 0) {  // an empty table (max_pages == 0): only the length can abort
    P = L > 0 ? (L + page_size - 1) / page_size : 0;
    bad = P > max_pages;
  }
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) abort_mask[r] = static_cast<uint8_t>(bad != 0);
  return bad;
}


// Grid for a grid-stride kernel: min(want, CTAs resident at once on the
// current device), so that no CTA waits for another to finish its whole loop
// (api.cu).
int resident_grid(const void* kernel, int threads, size_t dyn_smem, int64_t want);

// The cache write and tag check of one decode step as one launch
// (decode_step.cu); argument checks as fpk_decode_append_check_fp8.
int append_check_entry(bool fp8, const void* k_new, const void* v_new, void* kv_pool,
                       const float* k_scale, const float* v_scale, const int32_t* page_table,
                       int32_t max_pages, const int32_t* seq_lens, const uint32_t* live_tags,
                       const uint32_t* expected_tags, uint8_t* abort_mask, int32_t B, int32_t Hkv,
                       int32_t D, int32_t page_size, int32_t num_pages, void* stream);

}  // namespace fpk
