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
  const float ks = kFp8 ? __ldg(a.k_scale) : 1.f;
  const float vs = kFp8 ? __ldg(a.v_scale) : 1.f;
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
constexpr int kTileMaxB = 8192;     // requests whose tile offsets fit in shared memory

__device__ __forceinline__ uint32_t quant_pair(uint32_t bf16x2, float s) {
  const float a = __fdiv_rn(bf16_bits_to_float(static_cast<uint16_t>(bf16x2 & 0xFFFF)), s);
  const float b = __fdiv_rn(bf16_bits_to_float(static_cast<uint16_t>(bf16x2 >> 16)), s);
  return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Prompt write, one CTA per (request, 16-token tile, kv head) unit in a
// grid-stride loop.  The requests' first tile numbers are scanned into
// shared memory once per CTA (s_tile0[r], r = 0..B).
template <bool kFp8>
__global__ void __launch_bounds__(kTileThreads) prefill_tiles_kernel(WriteArgs a) {
  extern __shared__ int s_tile0[];
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
    s_tile0[r] = run;
    run += (__ldg(a.cu_seqlens + r + 1) - __ldg(a.cu_seqlens + r) + 15) >> 4;
  }
  if (t == kTileThreads - 1) s_tile0[a.B] = before + incl;
  __syncthreads();
  const int64_t units = static_cast<int64_t>(s_tile0[a.B]) * a.Hkv;
  const float ks = kFp8 ? __ldg(a.k_scale) : 1.f;
  const float vs = kFp8 ? __ldg(a.v_scale) : 1.f;
  const int tpp = a.page_size >> 4;
  // K: token tk, dims ck..ck+7.  V: tokens 4*qv..4*qv+3, dims 2*dv, 2*dv+1.
  const int tk = t >> 4, ck = (t & 15) * 8;
  const int qv = t & 3, dv = t >> 2;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int tile = static_cast<int>(u / a.Hkv);
    const int h = static_cast<int>(u - static_cast<int64_t>(tile) * a.Hkv);
    int lo = 0, hi = a.B - 1;  // the request: largest r with s_tile0[r] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tile0[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int j = tile - s_tile0[r];
    const int row0 = __ldg(a.cu_seqlens + r) + 16 * j;  // first source row of the tile
    const int n = min(16, __ldg(a.cu_seqlens + r + 1) - row0);  // tokens in this tile
    const int pi = (16 * j) / a.page_size;
    bool ok = pi < a.max_pages;
    int page = -1;
    if (ok) {
      page = __ldg(a.page_table + static_cast<int64_t>(r) * a.max_pages + pi);
      ok = page >= 0 && page < a.num_pages;
    }
    if (ok && a.live_tags != nullptr && a.expected_tags != nullptr)
      ok = __ldg(a.live_tags + page) == __ldg(a.expected_tags + static_cast<int64_t>(r) * a.max_pages + pi);
    if (!ok) {
      if (t == 0 && a.abort_mask != nullptr) a.abort_mask[r] = 1;
      continue;
    }
    const int64_t tb = ((static_cast<int64_t>(page) * a.Hkv + h) * tpp + (j % tpp)) * 2 * 16 * kDimW;
    const int64_t vb = tb + 16 * kDimW;
    // K rows
    if (tk < n) {
      const int64_t src = (static_cast<int64_t>(row0 + tk) * a.Hkv + h) * kDimW + ck;
      const uint4 kr = __ldg(reinterpret_cast<const uint4*>(a.k_src + src));
      if (kFp8) {
        const uint32_t w0 = quant_pair(kr.x, ks) | (quant_pair(kr.y, ks) << 16);
        const uint32_t w1 = quant_pair(kr.z, ks) | (quant_pair(kr.w, ks) << 16);
        *reinterpret_cast<uint2*>(a.kv_pool + tb + tk * kDimW + ck) = make_uint2(w0, w1);
      } else {
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.kv_pool) + tb + tk * kDimW + ck) = kr;
      }
    }
    // V columns: four tokens of two dims
    uint32_t vw[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int tok = 4 * qv + q;
      vw[q] = 0;
      if (tok < n)
        vw[q] = __ldg(reinterpret_cast<const uint32_t*>(
            a.v_src + (static_cast<int64_t>(row0 + tok) * a.Hkv + h) * kDimW + 2 * dv));
    }
    const bool full = 4 * qv + 3 < n;
    if (kFp8) {
      // quant_pair(x) gives the codes of (dim 2dv, dim 2dv+1) of one token
      const uint32_t c0 = quant_pair(vw[0], vs), c1 = quant_pair(vw[1], vs);
      const uint32_t c2 = quant_pair(vw[2], vs), c3 = quant_pair(vw[3], vs);
      const uint32_t row_a = (c0 & 0xFF) | ((c1 & 0xFF) << 8) | ((c2 & 0xFF) << 16) | ((c3 & 0xFF) << 24);
      const uint32_t row_b = (c0 >> 8) | (c1 & 0xFF00) | ((c2 & 0xFF00) << 8) | ((c3 & 0xFF00) << 16);
      uint8_t* pa = a.kv_pool + vb + (2 * dv) * 16 + 4 * qv;
      uint8_t* pb = pa + 16;
      if (full) {
        *reinterpret_cast<uint32_t*>(pa) = row_a;
        *reinterpret_cast<uint32_t*>(pb) = row_b;
      } else {
        for (int q = 0; q < 4 && 4 * qv + q < n; ++q) {
          pa[q] = static_cast<uint8_t>(row_a >> (8 * q));
          pb[q] = static_cast<uint8_t>(row_b >> (8 * q));
        }
      }
    } else {
      uint16_t* pa = reinterpret_cast<uint16_t*>(a.kv_pool) + vb + (2 * dv) * 16 + 4 * qv;
      uint16_t* pb = pa + 16;
      if (full) {
        *reinterpret_cast<uint2*>(pa) = make_uint2((vw[0] & 0xFFFF) | (vw[1] << 16), (vw[2] & 0xFFFF) | (vw[3] << 16));
        *reinterpret_cast<uint2*>(pb) = make_uint2((vw[0] >> 16) | (vw[1] & 0xFFFF0000u),
                                                   (vw[2] >> 16) | (vw[3] & 0xFFFF0000u));
      } else {
        for (int q = 0; q < 4 && 4 * qv + q < n; ++q) {
          pa[q] = static_cast<uint16_t>(vw[q] & 0xFFFF);
          pb[q] = static_cast<uint16_t>(vw[q] >> 16);
        }
      }
    }
  }
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
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t want = (units + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count(dev) > 0 ? device_sm_count(dev) : 132) * 16;
  const int grid = static_cast<int>(want < cap ? want : cap);
  if (fp8) {
    if (prefill) write_tokens_kernel<true, true><<<grid, 256, 0, s>>>(a);
    else write_tokens_kernel<true, false><<<grid, 256, 0, s>>>(a);
  } else {
    if (prefill) write_tokens_kernel<false, true><<<grid, 256, 0, s>>>(a);
    else write_tokens_kernel<false, false><<<grid, 256, 0, s>>>(a);
  }
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
  if (prefill && B <= kTileMaxB) {
    // tile-wise prompt write (the per-token kernel below covers larger batches)
    int dev = 0;
    cudaGetDevice(&dev);
    const int sms = device_sm_count(dev) > 0 ? device_sm_count(dev) : 132;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const int64_t want = (rows + 15) / 16 * Hkv + B * Hkv;  // an upper bound of the units
    const int grid = static_cast<int>(want < cap ? want : cap);
    const size_t smem = static_cast<size_t>(B + 1) * sizeof(int);
    if (fp8) prefill_tiles_kernel<true><<<grid, kTileThreads, smem, s>>>(a);
    else prefill_tiles_kernel<false><<<grid, kTileThreads, smem, s>>>(a);
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
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t want = ((n >> 1) + 255) / 256 + 1;
  const int64_t cap = static_cast<int64_t>(fpk::device_sm_count(dev) > 0 ? fpk::device_sm_count(dev) : 132) * 32;
  const int grid = static_cast<int>(want < cap ? want : cap);
  fpk::quantize_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, scale, out, n);
  return fpk::checked_launch_status();
}

extern "C" int fpk_amax_scale_bf16(const void* x, int64_t n, float* scale, uint32_t* scratch,
                                   void* stream) {
  if (n < 0 || !scale || !scratch || (n > 0 && !x)) return FPK_EINVAL;
  if (n > 0 && !fpk::aligned16(x)) return FPK_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 2 * sizeof(uint32_t), s) != cudaSuccess) return FPK_ECUDA;
  int dev = 0;
  cudaGetDevice(&dev);
  const int sms = fpk::device_sm_count(dev) > 0 ? fpk::device_sm_count(dev) : 132;
  const int64_t want = ((n >> 3) + 1023) / 1024;  // four 16-byte loads per thread
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
  fpk::amax_scale_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x), n, scale, scratch);
  return fpk::checked_launch_status();
}
