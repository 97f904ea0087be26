// page_tags.cu -- per-page generation tags: bump on reallocation and the
// separate batched validation that runs before attention.
//
// Every physical page carries a tag that changes whenever the page is
// reallocated; the server records the (page, tag) pairs each request expects;
// supported decode operations check them before reading and a mismatch aborts
// the request ("Cosa ha cambiato Cloudflare per Kimi e GLM" and "La sicurezza
// della cache KV condivisa diventa una questione di produzione", remio.ai).
// The check is its own batched kernel -- a pure gather-compare -- and is not
// fused into attention ("La sicurezza della cache KV condivisa...": fused, the
// check could race between GPU thread groups).
#include "step_ops.cuh"

namespace fpk {
namespace {

__global__ void __launch_bounds__(256) bump_kernel(uint32_t* __restrict__ live_tags,
                                                   const int32_t* __restrict__ pages, int n,
                                                   int num_pages) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int p = __ldg(pages + i);
  if (p >= 0 && p < num_pages) atomicAdd(live_tags + p, 1u);
}

// One request per cluster of `nparts` CTAs (one CTA for short tables).
__global__ void __launch_bounds__(kValidateThreads, kCheckCtasPerSm) validate_kernel(
    const int32_t* __restrict__ page_table, const uint32_t* __restrict__ expected_tags,
    const int32_t* __restrict__ seq_lens, int max_pages, const uint32_t* __restrict__ live_tags,
    int num_pages, int page_size, uint8_t* __restrict__ abort_mask, int32_t* __restrict__ abort_count,
    int nparts) {
  check_request(page_table, expected_tags, seq_lens, max_pages, live_tags, num_pages, page_size,
                abort_mask, abort_count, nparts);
}

}  // namespace
}  // namespace fpk

extern "C" int fpk_page_tags_bump(uint32_t* live_tags, const int32_t* pages, int32_t n,
                                  int32_t num_pages, void* stream) {
  if (n < 0 || num_pages < 0) return FPK_EINVAL;
  if (n == 0) return FPK_OK;
  if (!live_tags || !pages) return FPK_EINVAL;
  fpk::bump_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(live_tags, pages,
                                                                                  n, num_pages);
  return fpk::checked_launch_status();
}

extern "C" int fpk_page_tags_validate(const int32_t* page_table, const uint32_t* expected_tags,
                                      const int32_t* seq_lens, int32_t max_pages,
                                      const uint32_t* live_tags, int32_t num_pages, int32_t B,
                                      int32_t page_size, uint8_t* abort_mask, int32_t* abort_count,
                                      void* stream) {
  if (B < 0 || max_pages < 0 || num_pages < 0 || page_size <= 0) return FPK_EINVAL;
  // a rejected call queues nothing; with B == 0 the count is still zeroed
  if (B > 0 && (!page_table || !expected_tags || !seq_lens || !live_tags || !abort_mask))
    return FPK_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (abort_count != nullptr && cudaMemsetAsync(abort_count, 0, sizeof(int32_t), s) != cudaSuccess)
    return FPK_ECUDA;
  if (B == 0) return FPK_OK;
  const int nparts = fpk::check_parts(max_pages, B);
  if (static_cast<int64_t>(B) * nparts > 0x7fffffff) return FPK_EINVAL;
  return fpk::launch_check_grid(fpk::validate_kernel, B * nparts, nparts, s, page_table, expected_tags,
                                seq_lens, max_pages, live_tags, num_pages, page_size, abort_mask,
                                abort_count, nparts);
}
