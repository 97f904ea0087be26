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
// One thread handles 8 consecutive dims of one (token, kv head): a 16-byte
// bf16 load per tensor, an 8-byte (fp8) or 16-byte (bf16) store into the
// token-major K block of the token's 16-token tile, and 8 strided element
// stores into the tile's dim-major V block.
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
  return launch_write(a, fp8, prefill, static_cast<cudaStream_t>(stream));
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
