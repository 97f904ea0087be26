// kv_write.cu -- quantise-on-append and bulk prompt writes into the paged cache.
//
// The decode pool of the Cloudflare Kimi deployment keeps its KV cache as FP8
// e4m3 in place of BF16 ("Cosa ha cambiato Cloudflare per Kimi e GLM",
// remio.ai); requests write pages of the shared physical cache as well as
// read them (iitog.ru summary, third technique).  Every token write is
// guarded by its destination page's tag so that a stale mapping can never
// overwrite a page another request now owns: the write is skipped and the
// request is marked aborted.
//
// Decode appends (one token per request): one thread handles 8 consecutive
// dims of one (token, kv head): a 16-byte bf16 load per tensor, an 8-byte
// (fp8) or 16-byte (bf16) store into the token-major K block of the token's
// 16-token tile, and 8 strided element stores into the tile's dim-major V
// block.
//
// Prompt writes fill whole tiles, so they go tile by tile: one CTA writes the
// 16 tokens of one (request, tile, kv head), reading 2 x 4 KiB of bf16 and
// writing the K block as 128-byte token rows and the V block as 4-token words
// of each dim row; the page guard is taken once per tile (a tile never spans
// two pages).  The per-scale amax reduction that feeds the quantiser's scale
// is here too.
#include "step_ops.cuh"

namespace fpk {
namespace {

template <bool kFp8, bool kPrefill>
__global__ void __launch_bounds__(256) write_tokens_kernel(WriteArgs a) {
  const int64_t units = a.rows * a.Hkv * (a.D >> 3);
  const Divisor ks = make_divisor(kFp8 ? __ldg(a.k_scale) : 1.f);
  const Divisor vs = make_divisor(kFp8 ? __ldg(a.v_scale) : 1.f);
  for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x)
    write_unit<kFp8, kPrefill>(a, u, ks, vs);
}

__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ x,
                                                       const float* __restrict__ scale,
                                                       uint8_t* __restrict__ out, int64_t n) {
  const float s = __ldg(scale);
  const int64_t pairs = n >> 1;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < pairs;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float a = __fdiv_rn(__ldg(x + 2 * i), s);
    const float b = __fdiv_rn(__ldg(x + 2 * i + 1), s);
    const uint16_t p = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    out[2 * i] = static_cast<uint8_t>(p & 0xFF);
    out[2 * i + 1] = static_cast<uint8_t>(p >> 8);
  }
  if ((n & 1) && blockIdx.x == 0 && threadIdx.x == 0) {
    const float a = __fdiv_rn(__ldg(x + n - 1), s);
    const uint16_t p = __nv_cvt_float2_to_fp8x2(make_float2(a, 0.f), __NV_SATFINITE, __NV_E4M3);
    out[n - 1] = static_cast<uint8_t>(p & 0xFF);
  }
}

constexpr int kDimW = 128;          // head dimension (the only one supported)
constexpr int kTileThreads = 256;   // 16 tokens x 16 groups of 8 dims
constexpr int kTileMaxB = 4096;     // requests whose offsets fit in shared memory

// e4m3 codes of the two bf16 values of a word (low half first); kFast takes
// the corrected-product division (divisor with a normal reciprocal).
template <bool kFast = false>
__device__ __forceinline__ uint32_t quant_pair(uint32_t bf16x2, const Divisor& s) {
  const float x0 = __uint_as_float(bf16x2 << 16), x1 = __uint_as_float(bf16x2 & 0xFFFF0000u);
  const float a = kFast ? div_fast(x0, s) : div_by(x0, s);
  const float b = kFast ? div_fast(x1, s) : div_by(x1, s);
  return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

template <bool kFp8, bool kFast>
__device__ __forceinline__ void prefill_units(const WriteArgs& a, const int* s_tile0, const int* s_row0,
                                              int units, const Divisor& ks, const Divisor& vs,
                                              int lane, int warp) {
  const int tpp = a.page_size >> 4;
  const int warps = kTileThreads / 32;
  const int tk = lane >> 1, hk = (lane & 1) * 64;  // K: token, first dim
  const int dv = 4 * lane;                          // V: first dim
  // units < 2^31 (checked on the host): 32-bit index arithmetic
  for (int u = static_cast<int>(blockIdx.x) * warps + warp; u < units; u += static_cast<int>(gridDim.x) * warps) {
    const bool is_v = (u & 1) != 0;
    const int th = u >> 1;
    const int tile = th / a.Hkv;
    const int h = th - tile * a.Hkv;
    int lo = 0, hi = a.B - 1;  // the request: largest r with s_tile0[r] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tile0[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int j = tile - s_tile0[r];
    const int row0 = s_row0[r] + 16 * j;                // first source row of the tile
    const int n = min(16, s_row0[r + 1] - row0);        // tokens in this tile
    // guard loads (page id, then the two tags) ...
    const int pi = (16 * j) / a.page_size;
    const bool in_table = pi < a.max_pages;
    const int page = in_table ? __ldg(a.page_table + static_cast<int64_t>(r) * a.max_pages + pi) : -1;
    // ... while the source rows load: K as 8 x 16 bytes of one token, or V as
    // 16 tokens x 8 bytes, in the same 32 registers
    uint4 src[8];
    if (!is_v) {
      const uint16_t* ksrc = a.k_src + (static_cast<int64_t>(row0 + tk) * a.Hkv + h) * kDimW + hk;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        src[i] = tk < n ? __ldg(reinterpret_cast<const uint4*>(ksrc) + i) : make_uint4(0, 0, 0, 0);
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const uint2 v = q < n ? __ldg(reinterpret_cast<const uint2*>(
                                    a.v_src + (static_cast<int64_t>(row0 + q) * a.Hkv + h) * kDimW + dv))
                              : make_uint2(0, 0);
        if (q & 1) {
          src[q >> 1].z = v.x;
          src[q >> 1].w = v.y;
        } else {
          src[q >> 1].x = v.x;
          src[q >> 1].y = v.y;
        }
      }
    }
    bool ok = in_table && page >= 0 && page < a.num_pages;
    if (ok && a.live_tags != nullptr && a.expected_tags != nullptr)
      ok = __ldg(a.live_tags + page) == __ldg(a.expected_tags + static_cast<int64_t>(r) * a.max_pages + pi);
    if (!ok) {
      if (lane == 0 && a.abort_mask != nullptr) a.abort_mask[r] = 1;
      continue;
    }
    const uint4* kr = src;  // K part
    // V part: token q's dims dv..dv+3 are (src[q/2].x, .y) for even q, (.z, .w) for odd q
    auto vx = [&](int q) { return (q & 1) ? src[q >> 1].z : src[q >> 1].x; };
    auto vy = [&](int q) { return (q & 1) ? src[q >> 1].w : src[q >> 1].y; };
    const int64_t tb = ((static_cast<int64_t>(page) * a.Hkv + h) * tpp + (j % tpp)) * 2 * 16 * kDimW;
    const int64_t vb = tb + 16 * kDimW;
    if (kFp8) {
      // K: 64 codes of token tk
      if (!is_v && tk < n) {
        uint4 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          w[i].x = quant_pair<kFast>(kr[2 * i].x, ks) | (quant_pair<kFast>(kr[2 * i].y, ks) << 16);
          w[i].y = quant_pair<kFast>(kr[2 * i].z, ks) | (quant_pair<kFast>(kr[2 * i].w, ks) << 16);
          w[i].z = quant_pair<kFast>(kr[2 * i + 1].x, ks) | (quant_pair<kFast>(kr[2 * i + 1].y, ks) << 16);
          w[i].w = quant_pair<kFast>(kr[2 * i + 1].z, ks) | (quant_pair<kFast>(kr[2 * i + 1].w, ks) << 16);
        }
        uint4* dst = reinterpret_cast<uint4*>(a.kv_pool + tb + tk * kDimW + hk);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = w[i];
      }
      // V: dims dv .. dv+3, tokens 0..15 -> four 16-byte dim rows
      if (!is_v) continue;
      uint32_t rows[4][4];
#pragma unroll
      for (int q = 0; q < 16; q += 2) {
        // codes of tokens q, q+1 for dims dv, dv+1 (from x) and dv+2, dv+3 (from y)
        const uint32_t lo0 = (vx(q) & 0xFFFFu) | (vx(q + 1) << 16);
        const uint32_t hi0 = (vx(q) >> 16) | (vx(q + 1) & 0xFFFF0000u);
        const uint32_t lo1 = (vy(q) & 0xFFFFu) | (vy(q + 1) << 16);
        const uint32_t hi1 = (vy(q) >> 16) | (vy(q + 1) & 0xFFFF0000u);
        const uint32_t c[4] = {quant_pair<kFast>(lo0, vs), quant_pair<kFast>(hi0, vs), quant_pair<kFast>(lo1, vs),
                               quant_pair<kFast>(hi1, vs)};
        const int wi = q >> 2, sh = (q & 2) * 8;  // word of the row, byte offset of token q
#pragma unroll
        for (int d = 0; d < 4; ++d) {
          if (sh == 0) rows[d][wi] = c[d];
          else rows[d][wi] |= c[d] << 16;
        }
      }
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        uint8_t* row = a.kv_pool + vb + (dv + d) * 16;
        if (n == 16) {
          *reinterpret_cast<uint4*>(row) = make_uint4(rows[d][0], rows[d][1], rows[d][2], rows[d][3]);
        } else {
          for (int q = 0; q < n; ++q) row[q] = static_cast<uint8_t>(rows[d][q >> 2] >> (8 * (q & 3)));
        }
      }
    } else {
      uint16_t* pool = reinterpret_cast<uint16_t*>(a.kv_pool);
      if (!is_v && tk < n) {
        uint4* dst = reinterpret_cast<uint4*>(pool + tb + tk * kDimW + hk);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = kr[i];
      }
      // V rows of 16 bf16: element (dim dv+d, token q)
      if (!is_v) continue;
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        uint32_t w[8];
#pragma unroll
        for (int q = 0; q < 16; q += 2) {
          const uint32_t e0 = d < 2 ? vx(q) : vy(q);
          const uint32_t e1 = d < 2 ? vx(q + 1) : vy(q + 1);
          const uint32_t b0 = (d & 1) ? (e0 >> 16) : (e0 & 0xFFFFu);
          const uint32_t b1 = (d & 1) ? (e1 >> 16) : (e1 & 0xFFFFu);
          w[q >> 1] = b0 | (b1 << 16);
        }
        uint16_t* row = pool + vb + (dv + d) * 16;
        if (n == 16) {
          reinterpret_cast<uint4*>(row)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(row)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
          for (int q = 0; q < n; ++q) row[q] = static_cast<uint16_t>(w[q >> 1] >> (16 * (q & 1)));
        }
      }
    }
  }
}

// Prompt write: one warp per (request, 16-token tile, kv head, K or V) unit,
// in a grid-stride loop over the units (K/V, then kv head, fastest).  The requests' first
// tile numbers and first source rows are scanned into shared memory once per
// CTA; a unit's source loads are issued before its page guard resolves, and
// only the stores wait for the guard.
//   K: lane l writes token l/2, dims 64*(l&1) .. +63 (64 bytes of a 128-byte
//      token row in e4m3, 128 bytes in bf16).
//   V: lane l writes dims 4l .. 4l+3 over the 16 tokens (four dim rows of
//      16 codes, or 16 bf16).
template <bool kFp8>
__global__ void __launch_bounds__(kTileThreads) prefill_tiles_kernel(WriteArgs a) {
  extern __shared__ int s_meta[];  // [0, B]: first tile of request r; [B+1, 2B+2): first source row
  int* s_tile0 = s_meta;
  int* s_row0 = s_meta + a.B + 1;
  __shared__ int s_warp[kTileThreads / 32];
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  // ---- scan of ceil(len_r / 16) over the requests
  const int chunk = (a.B + kTileThreads - 1) / kTileThreads;
  const int rb = min(a.B, t * chunk), re = min(a.B, rb + chunk);
  int mine = 0;
  for (int r = rb; r < re; ++r) mine += (__ldg(a.cu_seqlens + r + 1) - __ldg(a.cu_seqlens + r) + 15) >> 4;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int i = 0; i < warp; ++i) before += s_warp[i];
  int run = before + incl - mine;
  for (int r = rb; r < re; ++r) {
    const int c0 = __ldg(a.cu_seqlens + r);
    s_tile0[r] = run;
    s_row0[r] = c0;
    run += (__ldg(a.cu_seqlens + r + 1) - c0 + 15) >> 4;
  }
  if (t == kTileThreads - 1) {
    s_tile0[a.B] = before + incl;
    s_row0[a.B] = __ldg(a.cu_seqlens + a.B);
  }
  __syncthreads();
  const int units = s_tile0[a.B] * a.Hkv * 2;
  const Divisor ks = make_divisor(kFp8 ? __ldg(a.k_scale) : 1.f);
  const Divisor vs = make_divisor(kFp8 ? __ldg(a.v_scale) : 1.f);
  // one division path for the whole kernel (uniform), so the unrolled body
  // carries no per-element fallback
  if (!kFp8 || (ks.recip_ok && vs.recip_ok))
    prefill_units<kFp8, true>(a, s_tile0, s_row0, units, ks, vs, lane, warp);
  else
    prefill_units<kFp8, false>(a, s_tile0, s_row0, units, ks, vs, lane, warp);
}

// amax over the finite values of a bf16 tensor, as the largest |x| bit
// pattern (an integer max: exact and independent of the reduction order);
// the CTA that arrives last turns it into scale = amax / 448 (1 if amax = 0).
// scratch[0] is the running maximum, scratch[1] the arrival count; both start
// at zero.
__global__ void __launch_bounds__(256) amax_scale_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                         float* __restrict__ scale, uint32_t* scratch) {
  __shared__ uint32_t s_max[8];
  const int64_t nv = n >> 3;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  uint32_t m2 = 0;  // two 16-bit running maxima
  auto fold = [&](uint32_t w) {
    w &= 0x7FFF7FFFu;
    w &= __vcmpltu2(w, 0x7F807F80u);  // inf and NaN count as 0
    m2 = __vmaxu2(m2, w);
  };
  int64_t i = g;
  for (; i + 3 * stride < nv; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __ldcs(xv + i + k * stride);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      fold(v[k].x);
      fold(v[k].y);
      fold(v[k].z);
      fold(v[k].w);
    }
  }
  for (; i < nv; i += stride) {
    const uint4 v = __ldcs(xv + i);
    fold(v.x);
    fold(v.y);
    fold(v.z);
    fold(v.w);
  }
  for (int64_t e = (nv << 3) + g; e < n; e += stride) fold(x[e]);
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < (blockDim.x >> 5); ++k) m = max(m, s_max[k]);
    atomicMax(scratch, m);
    __threadfence();
    if (atomicAdd(scratch + 1, 1u) == gridDim.x - 1) {
      __threadfence();
      const uint32_t am = atomicMax(scratch, 0u);
      const float amax = __uint_as_float(am << 16);
      *scale = am == 0 ? 1.f : __fdiv_rn(amax, 448.f);
    }
  }
}

int check_shapes(int B, int Hkv, int D, int page_size, int num_pages, int max_pages) {
  if (B < 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0 || max_pages < 0)
    return FPK_EINVAL;
  if (D != 128 || page_size % 16 != 0 || page_size > 256) return FPK_EUNSUPPORTED;
  return FPK_OK;
}

int launch_write(const WriteArgs& a, bool fp8, bool prefill, cudaStream_t s) {
  const int64_t units = a.rows * a.Hkv * (a.D >> 3);
  if (units == 0) return FPK_OK;
  const int64_t want = (units + 255) / 256;
  auto kern = fp8 ? (prefill ? write_tokens_kernel<true, true> : write_tokens_kernel<true, false>)
                  : (prefill ? write_tokens_kernel<false, true> : write_tokens_kernel<false, false>);
  const int grid = resident_grid(reinterpret_cast<const void*>(kern), 256, 0, want);
  kern<<<grid, 256, 0, s>>>(a);
  return checked_launch_status();
}

int write_entry(bool fp8, bool prefill, const void* k, const void* v, const int32_t* seq_lens,
                const int32_t* cu, int64_t rows, void* kv_pool, const float* k_scale,
                const float* v_scale, const int32_t* page_table, int32_t max_pages,
                const uint32_t* live_tags, const uint32_t* expected_tags, uint8_t* abort_mask,
                int32_t B, int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
                void* stream) {
  int st = check_shapes(B, Hkv, D, page_size, num_pages, max_pages);
  if (st != FPK_OK) return st;
  if (rows < 0) return FPK_EINVAL;
  if (rows == 0 || B == 0) return FPK_OK;
  if (!k || !v || !kv_pool || !page_table || (prefill ? !cu : !seq_lens)) return FPK_EINVAL;
  if (fp8 && (!k_scale || !v_scale)) return FPK_EINVAL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(kv_pool)) return FPK_EINVAL;
  WriteArgs a;
  a.k_src = static_cast<const uint16_t*>(k);
  a.v_src = static_cast<const uint16_t*>(v);
  a.seq_lens = seq_lens;
  a.cu_seqlens = cu;
  a.kv_pool = static_cast<uint8_t*>(kv_pool);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.page_table = page_table;
  a.live_tags = live_tags;
  a.expected_tags = expected_tags;
  a.abort_mask = abort_mask;
  a.rows = rows;
  a.B = B;
  a.Hkv = Hkv;
  a.D = D;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.max_pages = max_pages;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the tile-wise path indexes its units in 32 bits
  const bool tile_path = prefill && B <= kTileMaxB &&
                         ((rows + 15) / 16 + B) * static_cast<int64_t>(Hkv) * 2 < (int64_t(1) << 31);
  if (tile_path) {
    // tile-wise prompt write (the per-token kernel below covers larger batches)
    const int64_t want = (((rows + 15) / 16 + B) * Hkv * 2 + 7) / 8;  // units, 8 warps per CTA
    const size_t smem = static_cast<size_t>(2 * (B + 1)) * sizeof(int);
    auto kern = fp8 ? prefill_tiles_kernel<true> : prefill_tiles_kernel<false>;
    const int grid = resident_grid(reinterpret_cast<const void*>(kern), kTileThreads, smem, want);
    kern<<<grid, kTileThreads, smem, s>>>(a);
    return checked_launch_status();
  }
  return launch_write(a, fp8, prefill, s);
}

}  // namespace
}  // namespace fpk

extern "C" int fpk_kv_append_fp8(const void* k_new, const void* v_new, uint8_t* kv_pool,
                                 const float* k_scale, const float* v_scale,
                                 const int32_t* page_table, int32_t max_pages,
                                 const int32_t* seq_lens, const uint32_t* live_tags,
                                 const uint32_t* expected_tags, uint8_t* abort_mask, int32_t B,
                                 int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
                                 void* stream) {
  return fpk::write_entry(true, false, k_new, v_new, seq_lens, nullptr, B, kv_pool, k_scale,
                          v_scale, page_table, max_pages, live_tags, expected_tags, abort_mask, B,
                          Hkv, D, page_size, num_pages, stream);
}

extern "C" int fpk_kv_append_bf16(const void* k_new, const void* v_new, void* kv_pool,
                                  const int32_t* page_table, int32_t max_pages,
                                  const int32_t* seq_lens, const uint32_t* live_tags,
                                  const uint32_t* expected_tags, uint8_t* abort_mask, int32_t B,
                                  int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
                                  void* stream) {
  return fpk::write_entry(false, false, k_new, v_new, seq_lens, nullptr, B, kv_pool, nullptr,
                          nullptr, page_table, max_pages, live_tags, expected_tags, abort_mask, B,
                          Hkv, D, page_size, num_pages, stream);
}

extern "C" int fpk_kv_prefill_fp8(const void* k, const void* v, const int32_t* cu_seqlens,
                                  int32_t n_tokens, uint8_t* kv_pool,
                                  const float* k_scale, const float* v_scale,
                                  const int32_t* page_table, int32_t max_pages,
                                  const uint32_t* live_tags, const uint32_t* expected_tags,
                                  uint8_t* abort_mask, int32_t B, int32_t Hkv, int32_t D,
                                  int32_t page_size, int32_t num_pages, void* stream) {
  return fpk::write_entry(true, true, k, v, nullptr, cu_seqlens, n_tokens, kv_pool, k_scale,
                          v_scale, page_table, max_pages, live_tags, expected_tags, abort_mask, B,
                          Hkv, D, page_size, num_pages, stream);
}

extern "C" int fpk_kv_prefill_bf16(const void* k, const void* v, const int32_t* cu_seqlens,
                                   int32_t n_tokens, void* kv_pool,
                                   const int32_t* page_table, int32_t max_pages,
                                   const uint32_t* live_tags, const uint32_t* expected_tags,
                                   uint8_t* abort_mask, int32_t B, int32_t Hkv, int32_t D,
                                   int32_t page_size, int32_t num_pages, void* stream) {
  return fpk::write_entry(false, true, k, v, nullptr, cu_seqlens, n_tokens, kv_pool, nullptr,
                          nullptr, page_table, max_pages, live_tags, expected_tags, abort_mask, B,
                          Hkv, D, page_size, num_pages, stream);
}

extern "C" int fpk_quantize_e4m3(const float* x, const float* scale, uint8_t* out, int64_t n,
                                 void* stream) {
  if (n < 0) return FPK_EINVAL;
  if (n == 0) return FPK_OK;
  if (!x || !scale || !out) return FPK_EINVAL;
  const int64_t want = ((n >> 1) + 255) / 256 + 1;
  const int grid = fpk::resident_grid(reinterpret_cast<const void*>(fpk::quantize_kernel), 256, 0, want);
  fpk::quantize_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, scale, out, n);
  return fpk::checked_launch_status();
}

extern "C" int fpk_amax_scale_bf16(const void* x, int64_t n, float* scale, uint32_t* scratch,
                                   void* stream) {
  if (n < 0 || !scale || !scratch || (n > 0 && !x)) return FPK_EINVAL;
  if (n > 0 && !fpk::aligned16(x)) return FPK_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 2 * sizeof(uint32_t), s) != cudaSuccess) return FPK_ECUDA;
  const int64_t want = ((n >> 3) + 1023) / 1024;  // four 16-byte loads per thread
  const int grid = fpk::resident_grid(reinterpret_cast<const void*>(fpk::amax_scale_kernel), 256, 0,
                                      want < 1 ? 1 : want);
  fpk::amax_scale_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x), n, scale, scratch);
  return fpk::checked_launch_status();
}
