// decode_step.cu -- the cache write and the batched tag check of a decode step
// in one launch.
//
// Per decode step the pages' path writes the new token's K/V into its page
// ("Cosa ha cambiato Cloudflare per Kimi e GLM", remio.ai: the cache is held
// as e4m3) and checks every request's recorded (page, tag) mapping before the
// decode operations read the pages (same section, and "La sicurezza della
// cache KV condivisa diventa una questione di produzione": a separate batched
// check, kept out of attention).  The two touch disjoint data -- the check
// reads tables and tags, the write stores one slot per request -- and where
// the write refuses a stale slot, the check marks the same request for the
// same table entry.  So one launch carries both: CTAs [0, B) check one request
// each, the remaining CTAs write tokens.  Attention, launched after this
// kernel, reads the written slots and the abort mask.
#include "step_ops.cuh"

namespace fpk {
namespace {

constexpr int kWriteCtas = 64;  // CTAs that share the token writes (grid-stride)

// CTAs [0, B * nparts) check one request per cluster of nparts CTAs; the
// rest (a multiple of nparts, in clusters that hold no barrier) write tokens.
template <bool kFp8>
__global__ void __launch_bounds__(kValidateThreads, kCheckCtasPerSm) append_check_kernel(WriteArgs w,
                                                                        const uint32_t* live_tags,
                                                                        const uint32_t* expected_tags,
                                                                        uint8_t* abort_mask,
                                                                        int nparts) {
  // a programmatically dependent attention launch may start its set-up now;
  // it reads nothing this kernel writes before this grid has completed
  griddep_launch_dependents();
  // no tags: the no-op tracker -- no check CTAs, unguarded writes
  const int nchk = (live_tags != nullptr && expected_tags != nullptr) ? w.B * nparts : 0;
  if (static_cast<int>(blockIdx.x) < nchk) {
    check_request(w.page_table, expected_tags, w.seq_lens, w.max_pages, live_tags, w.num_pages,
                  w.page_size, abort_mask, nullptr, nparts);
    return;
  }
  const int64_t units = w.rows * w.Hkv * (w.D >> 3);
  const Divisor ks = make_divisor(kFp8 ? __ldg(w.k_scale) : 1.f);
  const Divisor vs = make_divisor(kFp8 ? __ldg(w.v_scale) : 1.f);
  const int64_t stride = static_cast<int64_t>(gridDim.x - nchk) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x - nchk) * blockDim.x + threadIdx.x; u < units;
       u += stride)
    write_unit<kFp8, false>(w, u, ks, vs);
}

}  // namespace

int append_check_entry(bool fp8, const void* k_new, const void* v_new, void* kv_pool,
                       const float* k_scale, const float* v_scale, const int32_t* page_table,
                       int32_t max_pages, const int32_t* seq_lens, const uint32_t* live_tags,
                       const uint32_t* expected_tags, uint8_t* abort_mask, int32_t B, int32_t Hkv,
                       int32_t D, int32_t page_size, int32_t num_pages, void* stream) {
  if (B < 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0 || max_pages < 0)
    return FPK_EINVAL;
  if (D != 128 || page_size % 16 != 0 || page_size > 256) return FPK_EUNSUPPORTED;
  if (B == 0) return FPK_OK;
  if (!k_new || !v_new || !kv_pool || !page_table || !seq_lens) return FPK_EINVAL;
  // the check needs both tag arrays and the mask; with neither tag array it is
  // the no-op tracker
  const bool check = live_tags != nullptr || expected_tags != nullptr;
  if (check && (!live_tags || !expected_tags || !abort_mask)) return FPK_EINVAL;
  if (fp8 && (!k_scale || !v_scale)) return FPK_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kv_pool)) return FPK_EINVAL;
  WriteArgs w;
  w.k_src = static_cast<const uint16_t*>(k_new);
  w.v_src = static_cast<const uint16_t*>(v_new);
  w.seq_lens = seq_lens;
  w.cu_seqlens = nullptr;
  w.kv_pool = static_cast<uint8_t*>(kv_pool);
  w.k_scale = k_scale;
  w.v_scale = v_scale;
  w.page_table = page_table;
  w.live_tags = check ? live_tags : nullptr;
  w.expected_tags = check ? expected_tags : nullptr;
  w.abort_mask = check ? abort_mask : nullptr;
  w.rows = B;
  w.B = B;
  w.Hkv = Hkv;
  w.D = D;
  w.page_size = page_size;
  w.num_pages = num_pages;
  w.max_pages = max_pages;
  const int64_t units = static_cast<int64_t>(B) * Hkv * (D >> 3);
  const int64_t want = (units + kValidateThreads - 1) / kValidateThreads;
  const int nparts = check ? check_parts(max_pages, B) : 1;
  // write CTAs rounded up to whole clusters
  const int64_t nwrite = ((want < kWriteCtas ? want : kWriteCtas) + nparts - 1) / nparts * nparts;
  const int64_t grid = (check ? static_cast<int64_t>(B) * nparts : 0) + nwrite;
  if (grid > 0x7fffffff) return FPK_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fp8)
    return launch_check_grid(append_check_kernel<true>, static_cast<int>(grid), nparts, s, w, w.live_tags,
                             w.expected_tags, w.abort_mask, nparts);
  return launch_check_grid(append_check_kernel<false>, static_cast<int>(grid), nparts, s, w, w.live_tags,
                           w.expected_tags, w.abort_mask, nparts);
}

}  // namespace fpk

extern "C" int fpk_decode_append_check_fp8(const void* k_new, const void* v_new, uint8_t* kv_pool,
                                           const float* k_scale, const float* v_scale,
                                           const int32_t* page_table, int32_t max_pages,
                                           const int32_t* seq_lens, const uint32_t* live_tags,
                                           const uint32_t* expected_tags, uint8_t* abort_mask,
                                           int32_t B, int32_t Hkv, int32_t D, int32_t page_size,
                                           int32_t num_pages, void* stream) {
  return fpk::append_check_entry(true, k_new, v_new, kv_pool, k_scale, v_scale, page_table, max_pages,
                                 seq_lens, live_tags, expected_tags, abort_mask, B, Hkv, D, page_size,
                                 num_pages, stream);
}

extern "C" int fpk_decode_append_check_bf16(const void* k_new, const void* v_new, void* kv_pool,
                                            const int32_t* page_table, int32_t max_pages,
                                            const int32_t* seq_lens, const uint32_t* live_tags,
                                            const uint32_t* expected_tags, uint8_t* abort_mask,
                                            int32_t B, int32_t Hkv, int32_t D, int32_t page_size,
                                            int32_t num_pages, void* stream) {
  return fpk::append_check_entry(false, k_new, v_new, kv_pool, nullptr, nullptr, page_table, max_pages,
                                 seq_lens, live_tags, expected_tags, abort_mask, B, Hkv, D, page_size,
                                 num_pages, stream);
}
