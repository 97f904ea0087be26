/*
 * fp8kv.h -- C ABI of libfp8kv, the GB300 (sm_103a) decode-pool hot path over
 * a paged FP8 e4m3 KV cache with page-tag integrity checks.
 *
 * What it implements is described by the Cloudflare Workers AI write-up on
 * serving Kimi K2.6 and GLM 5.2 (reported by "Il serving di modelli piu
 * piccoli di Cloudflare riduce la memoria, ma la sicurezza diventa la prova
 * decisiva", remio.ai, and its Portuguese and Korean editions; and by the
 * iitog.ru and manulx.blog summaries):
 *   - the KV cache of the decode pool is stored as FP8 e4m3 in place of BF16,
 *     halving its bytes (section "Cosa ha cambiato Cloudflare per Kimi e GLM");
 *   - the attention kernel converts the FP8 values as it reads them (section
 *     "Perche le cache piu piccole di Cloudflare battono la velocita pura");
 *   - every physical page carries a tag that changes on each reallocation, the
 *     server records the (page, tag) pairs each request expects, and a separate
 *     batched check compares them before supported decode operations read the
 *     pages; a mismatch aborts that request (sections "Cosa ha cambiato..." and
 *     "La sicurezza della cache KV condivisa diventa una questione di
 *     produzione"); with the check off, a no-op tracker costs nothing.
 * The pages give no kernel design and no layouts: every layout and schedule
 * below is this library's own.
 *
 * ---------------------------------------------------------------------------
 * Conventions for every entry point
 * ---------------------------------------------------------------------------
 * Pointers: every array argument is a DEVICE pointer unless stated otherwise.
 * The caller owns all memory; the library allocates nothing, keeps no
 * per-call state and launches only on the given stream (`stream` is a
 * cudaStream_t passed as void*; NULL means the legacy default stream).  All
 * calls are asynchronous with respect to the host; synchronise the stream
 * before reading results.
 *
 * Shapes: B requests, Hq query heads, Hkv kv heads (G = Hq/Hkv query heads
 * share one kv head: query head h reads kv head h / G), head dimension D,
 * page_size tokens per physical page, num_pages pages in the pool, max_pages
 * columns in each request's page table.
 *
 * Supported sizes: D == 128; page_size a multiple of 16 in [16, 256];
 * 1 <= G <= 8.  Others return FPK_EUNSUPPORTED.  B == 0 is a no-op (FPK_OK);
 * Hq or Hkv below 1 is FPK_EINVAL.
 *
 * KV pool layout (one pool per layer holding K and V; bytes per element: 1
 * for the e4m3 pool, 2 for the bf16 pool):
 *   kv_pool [num_pages][Hkv][page_size/16][2][16*D]
 *   i.e. every page holds, per kv head, page_size/16 tiles of 16 tokens, and
 *   each tile is its K block [16 tokens][D] (token-major) immediately
 *   followed by its V block [D][16 tokens] (dim-major).  A tile's K and V are
 *   therefore one contiguous 2*16*D-element run.
 *   Token t of a request lives in page page_table[r][t / page_size] at slot
 *   s = t % page_size: K element d at tile (s/16), row s%16, column d; V
 *   element d at tile (s/16), row d, column s%16.  The pool pointer must be
 *   16-byte aligned.
 * Page table:     int32  [B][max_pages]   (row-major; entries past a request's
 *                                          ceil(L/page_size) pages are ignored)
 * Expected tags:  uint32 [B][max_pages]   (same shape as the page table)
 * Live tags:      uint32 [num_pages]
 * seq_lens:       int32  [B]              context length L_r of each request
 * Scales:         float  [1] each         per-tensor dequantisation scale:
 *                 value = decode_e4m3(code) * scale; positive and finite.
 *
 * E4M3 is the OCP OFP8 E4M3 format (bias 7, no infinities, NaN = S.1111.111,
 * largest finite 448).  Quantisation computes float(x)/scale with one IEEE
 * fp32 division and rounds to nearest-even with saturation to +-448; NaN
 * encodes as 0x7F.
 *
 * Errors: the return value is synchronous.  FPK_OK on success;
 * FPK_EINVAL for a NULL required pointer, a negative size or Hq % Hkv != 0;
 * FPK_EUNSUPPORTED for sizes outside the supported set; FPK_ENOSPC when a
 * workspace is too small; FPK_ECUDA when a launch fails (the CUDA error is
 * left pending for the caller to read).  Data faults -- a stale tag, a page id
 * outside [0, num_pages), a context longer than the page table -- are never API
 * errors: they fail closed per request (no page of that request is read or
 * written, its attention output is 0 and its lse is -inf) and are reported in
 * abort_mask / abort_count where those are given.
 */
#ifndef FP8KV_H_
#define FP8KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FPK_OK 0
#define FPK_EINVAL 1
#define FPK_EUNSUPPORTED 2
#define FPK_ENOSPC 3
#define FPK_ECUDA 4

/* ------------------------------------------------------------------------
 * Weight-only quantised decode GEMV (the pages' second technique: "La
 * compressione dei pesi GLM modifica il compromesso tra le fasi", remio.ai --
 * GLM 5.2's weights went from FP8 to INT4 because decode streams every weight
 * from HBM at each step; INT4 weights are expanded before the multiply).  The
 * pages give no format; this one is the library's own:
 *
 *   W [N][K] bf16 (N % 16 == 0, K % 128 == 0) is cut into slices of 16 rows x
 *   128 k, stored slice-row-block major: slice (n / 16, k / 128).
 *   INT4: per row and group of 128 k, scale s = bf16(amax / 7) over the
 *     group's finite values; code q = clamp(rint(w / s), -8, 7) (fp32 IEEE
 *     division, ties to even), 0 for a non-finite w or s == 0; stored as the
 *     nibble q + 8.  Dequantised weight q * s.  A slice is 1024 bytes: byte
 *     512*h + 16*l + 4*u + (0..3) holds word u of row 8*h + l/4 (l = 0..31);
 *     nibble p (bits 4p..4p+3) of word u is k = 16*v + 4*(l % 4) + i with
 *     v = 2u + ((p >> 1) & 1), i = 2*(p & 1) + (p >> 2).
 *     codes: N*K/2 bytes; scales: bf16 [N][K/128] (row-major).
 *   e4m3: per row, scale r = amax / 448 over the row's finite values (1 if
 *     that amax is 0); codes e4m3(w / r) as the cache quantiser.  A slice is
 *     2048 bytes: byte 1024*h + 512*c + 16*l + b holds row 8*h + l/4,
 *     k = 16*(4c + b/4) + 4*(l % 4) + b % 4.  codes: N*K bytes; row_scales:
 *     float [N].
 *
 * y[b][n] = sum_k x[b][k] * Wq[n][k] for b < B, 1 <= B <= 16 (decode tokens);
 * x bf16 [B][K] (16-byte aligned), y float [B][N].  Accumulation is fp32 on
 * the tensor cores; for K > 2048 the K chunks are added into y with atomics
 * (y is zeroed by the call first), so the last bits of y may vary between
 * calls.  B > 16 returns FPK_EUNSUPPORTED.
 * ------------------------------------------------------------------------ */
int fpk_w4_quantize(const void* w, uint8_t* codes, void* scales, int32_t N, int32_t K, void* stream);
int fpk_w4_gemv(const void* x, const uint8_t* codes, const void* scales, float* y, int32_t B,
                int32_t N, int32_t K, void* stream);
int fpk_w8_quantize(const void* w, uint8_t* codes, float* row_scales, int32_t N, int32_t K,
                    void* stream);
int fpk_w8_gemv(const void* x, const uint8_t* codes, const float* row_scales, float* y, int32_t B,
                int32_t N, int32_t K, void* stream);

/* Library ABI version (major * 100 + minor). */
int fpk_version(void);

/* Human-readable text for a status code (static storage; never NULL). */
const char* fpk_status_str(int status);

/*
 * Quantise-on-append for one decode step (FP8 cache).
 * Source: "Cosa ha cambiato Cloudflare per Kimi e GLM" (the cache is held as
 * e4m3) and the iitog.ru summary's third technique (requests write the pages
 * of the shared cache).
 *
 * For every request r with L = seq_lens[r] >= 1 (seq_lens already counts the
 * new token) and every kv head h and dim d, writes the K element of slot
 * pos % page_size of page page_table[r][pos / page_size] (pos = L - 1) as
 *   e4m3(float(k_new[r][h][d]) / *k_scale)
 * and the V element likewise with *v_scale, at their places in kv_pool.
 * Guard (fail closed): when pos / page_size >= max_pages, the page id is
 * outside [0, num_pages), or live_tags and expected_tags are both given and
 * live_tags[page] != expected_tags[r][pos / page_size], nothing of request r
 * is written and abort_mask[r] is set to 1 (if abort_mask is non-NULL; other
 * entries are left as they are).
 *   k_new, v_new : bf16 [B][Hkv][D] (device)
 *   live_tags, expected_tags, abort_mask : nullable (NULL = no tag guard)
 */
int fpk_kv_append_fp8(const void* k_new, const void* v_new, uint8_t* kv_pool,
                      const float* k_scale, const float* v_scale,
                      const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                      const uint32_t* live_tags, const uint32_t* expected_tags,
                      uint8_t* abort_mask, int32_t B, int32_t Hkv, int32_t D,
                      int32_t page_size, int32_t num_pages, void* stream);

/* Same as fpk_kv_append_fp8 for the BF16 comparison cache: the bf16 bit
 * patterns are copied unchanged (pools hold uint16 elements).  The pages keep
 * BF16 caches where compute dominates ("Cosa ha cambiato...", last paragraphs). */
int fpk_kv_append_bf16(const void* k_new, const void* v_new, void* kv_pool,
                       const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                       const uint32_t* live_tags, const uint32_t* expected_tags,
                       uint8_t* abort_mask, int32_t B, int32_t Hkv, int32_t D,
                       int32_t page_size, int32_t num_pages, void* stream);

/*
 * Bulk write of whole prompts into the pages (the cache a decode pool receives
 * from prefill).  Rows cu_seqlens[r] .. cu_seqlens[r+1]-1 of k, v (bf16
 * [n_tokens][Hkv][D]) are request r's tokens at positions 0, 1, ...; each token
 * is written exactly as fpk_kv_append_fp8 writes one, with the same guard.
 *   cu_seqlens : int32 [B+1] (device), cu_seqlens[0] == 0, non-decreasing,
 *                cu_seqlens[B] == n_tokens.
 */
int fpk_kv_prefill_fp8(const void* k, const void* v, const int32_t* cu_seqlens, int32_t n_tokens,
                       uint8_t* kv_pool, const float* k_scale, const float* v_scale,
                       const int32_t* page_table, int32_t max_pages,
                       const uint32_t* live_tags, const uint32_t* expected_tags,
                       uint8_t* abort_mask, int32_t B, int32_t Hkv, int32_t D,
                       int32_t page_size, int32_t num_pages, void* stream);

/* BF16-cache variant of fpk_kv_prefill_fp8 (bit copy). */
int fpk_kv_prefill_bf16(const void* k, const void* v, const int32_t* cu_seqlens, int32_t n_tokens,
                        void* kv_pool, const int32_t* page_table, int32_t max_pages,
                        const uint32_t* live_tags, const uint32_t* expected_tags,
                        uint8_t* abort_mask, int32_t B, int32_t Hkv, int32_t D,
                        int32_t page_size, int32_t num_pages, void* stream);

/*
 * Element-wise quantiser: out[i] = e4m3(x[i] / *scale) for i < n, with the
 * same division and rounding as the append.  x: float [n], out: uint8 [n].
 */
int fpk_quantize_e4m3(const float* x, const float* scale, uint8_t* out, int64_t n, void* stream);

/*
 * Per-tensor scale of a bf16 tensor for the e4m3 cache: *scale = amax / 448,
 * amax = max |x[i]| over the finite elements (infinities and NaNs are
 * skipped); *scale = 1 when amax == 0 or n == 0.  The division is one IEEE
 * fp32 division.  The pages state only that the cache holds e4m3 values
 * ("Cosa ha cambiato Cloudflare per Kimi e GLM", remio.ai); one fp32 scale per
 * tensor equal to amax / 448 is this library's reading.  Use it on a prompt's
 * K (resp. V) before fpk_kv_prefill_fp8, which reads the scale on the device.
 *   x       : bf16 [n] (device, 16-byte aligned)
 *   scale   : float [1] (device, written)
 *   scratch : uint32 [2] (device), caller-owned; the call zeroes it first.
 *             Calls that share scratch must not overlap on the GPU.
 * Result is bit-exact (the max is an integer max of bit patterns).
 */
int fpk_amax_scale_bf16(const void* x, int64_t n, float* scale, uint32_t* scratch, void* stream);

/*
 * Page reallocation: live_tags[pages[i]] += 1 (mod 2^32) for i < n.
 * Source: "Cosa ha cambiato..." -- a page's tag changes every time the page is
 * reallocated; "La sicurezza della cache KV condivisa..." -- the tags behave
 * like generation counters.  Ids outside [0, num_pages) are ignored; an id
 * listed k times advances by k.  n == 0 launches nothing.
 *   pages : int32 [n] (device)
 */
int fpk_page_tags_bump(uint32_t* live_tags, const int32_t* pages, int32_t n, int32_t num_pages,
                       void* stream);

/*
 * Batched page-tag validation, a separate pure gather-compare that runs before
 * attention (never fused into it: "La sicurezza della cache KV condivisa..."
 * says the check was kept out of the attention kernel because GPU thread
 * groups could have raced there).
 * For every request r, with P = ceil(seq_lens[r] / page_size) (0 if L <= 0):
 *   abort_mask[r] = 1 iff P > max_pages, or some i < P has page_table[r][i]
 *   outside [0, num_pages) or live_tags[page_table[r][i]] != expected_tags[r][i];
 *   otherwise abort_mask[r] = 0 (the mask is overwritten).
 *   abort_count (nullable, int32 [1]) receives the number of aborted requests
 *   (the mismatch-rate signal the pages ask operators to watch).
 */
int fpk_page_tags_validate(const int32_t* page_table, const uint32_t* expected_tags,
                           const int32_t* seq_lens, int32_t max_pages,
                           const uint32_t* live_tags, int32_t num_pages, int32_t B,
                           int32_t page_size, uint8_t* abort_mask, int32_t* abort_count,
                           void* stream);

/*
 * One launch carrying a decode step's cache write and its batched tag check:
 * exactly fpk_kv_append_fp8 (with the tag guard) followed by
 * fpk_page_tags_validate (without abort_count), for the same arguments.  The
 * check remains a separate batched operation, kept out of attention ("La
 * sicurezza della cache KV condivisa..."); sharing a launch with the write is
 * safe because the two touch disjoint data, and wherever the write refuses a
 * stale slot the check marks the same request for the same table entry.
 * abort_mask (uint8 [B]) is overwritten with the check's result.  With
 * live_tags and expected_tags both NULL (the no-op tracker) the launch only
 * writes, unguarded, and abort_mask is not touched; one of them NULL is
 * FPK_EINVAL.
 */
int fpk_decode_append_check_fp8(const void* k_new, const void* v_new, uint8_t* kv_pool,
                                const float* k_scale, const float* v_scale,
                                const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                                const uint32_t* live_tags, const uint32_t* expected_tags,
                                uint8_t* abort_mask, int32_t B, int32_t Hkv, int32_t D,
                                int32_t page_size, int32_t num_pages, void* stream);

/* BF16-cache variant of fpk_decode_append_check_fp8 (bit copy, no scales). */
int fpk_decode_append_check_bf16(const void* k_new, const void* v_new, void* kv_pool,
                                 const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                                 const uint32_t* live_tags, const uint32_t* expected_tags,
                                 uint8_t* abort_mask, int32_t B, int32_t Hkv, int32_t D,
                                 int32_t page_size, int32_t num_pages, void* stream);

/*
 * Workspace (device bytes) that fpk_paged_decode_attn_* needs for this batch
 * shape and split count.  num_splits == 0 means the automatic count the
 * attention call would choose on the CURRENT device.
 */
size_t fpk_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t num_splits);

/*
 * Split-KV decode attention over the FP8 e4m3 cache, dequantising on read,
 * with the cross-split log-sum-exp combine.
 * Sources: "Perche le cache piu piccole..." (the kernel converts FP8 on read),
 * "La sicurezza della cache KV condivisa..." (paged attention over physical
 * pages; aborted requests read nothing).
 *
 * For request r, query head h, kv head hk = h / G, tokens j < L = seq_lens[r]:
 *   s_j   = sm_scale * sum_d q[r][h][d] * decode(K code) * *k_scale
 *   out[r][h][:] = sum_j exp(s_j - m) * decode(V code) * *v_scale / sum_j exp(s_j - m)
 *   lse[r][h]    = m + ln(sum_j exp(s_j - m)),   m = max_j s_j
 * A request with L <= 0, abort_mask[r] != 0, L > max_pages * page_size, or a
 * page id outside [0, num_pages) among its first ceil(L/page_size) entries
 * gets out = 0 and lse = -inf, and (except for the last case, found while
 * streaming) none of its pages is read.
 *   q         : bf16 [B][Hq][D]
 *   abort_mask: uint8 [B] from fpk_page_tags_validate, or NULL (no-op tracker:
 *               no tag check)
 *   out       : float [B][Hq][D], 16-byte aligned;  lse: float [B][Hq], nullable
 *   workspace : >= fpk_decode_workspace_bytes(...) bytes, 256-byte aligned,
 *               owned by the caller.  Zero it ONCE after allocating: it holds
 *               arrival counters that every call leaves at zero
 *               again, split partials, and in its first 4 bytes a status word
 *               the kernel sets to nonzero (and never clears) if a bounded
 *               internal wait gave up; read it with fpk_decode_status and
 *               re-zero the whole workspace after a nonzero status.  Calls
 *               that share a workspace must not overlap on the GPU.
 *   num_splits: number of split-KV work units the batch's KV tiles are
 *               divided into (balanced by tile count across all requests and
 *               kv heads); each split's partial enters the log-sum-exp
 *               combine.  0 = automatic: one wave of CTAs, at most 16 per
 *               (request, kv head); when every non-empty request has the
 *               same length, one whole (request, kv head) per CTA if they
 *               fill 3/4 of a wave or more, else an equal number of splits
 *               per (request, kv head) (at most 16); when lengths
 *               differ and the non-empty (request, kv head) pairs number at
 *               most a third of a wave, each is cut into splits of one
 *               common tile count c (its last split shorter): the smallest c
 *               for which the splits number no more than a wave, one split
 *               per CTA.  With equal context lengths, num_splits = S * B * Hkv
 *               gives exactly S splits per (request, kv head).  At most one
 *               wave of CTAs is launched; with more splits than that, each
 *               CTA runs several consecutive splits in turn.  Every split's
 *               partial and every combine order are fixed, so repeated calls
 *               on the same inputs give identical bits.
 *   sm_scale  : softmax scale (1/sqrt(D) for standard attention).
 */
int fpk_paged_decode_attn_fp8(const void* q, const uint8_t* kv_pool,
                              const float* k_scale, const float* v_scale,
                              const int32_t* page_table, int32_t max_pages,
                              const int32_t* seq_lens, const uint8_t* abort_mask,
                              float* out, float* lse, void* workspace, size_t workspace_bytes,
                              int32_t num_splits, float sm_scale, int32_t B, int32_t Hq,
                              int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
                              void* stream);

/*
 * Variant of fpk_paged_decode_attn_fp8 on the fifth-generation tensor cores
 * (tcgen05.mma of kind f8f6f4, accumulators in tensor memory): same
 * arguments, same results within the same tolerance, same workspace
 * (fpk_decode_workspace_bytes covers it), same fail-closed rules.
 * Source: "Perche le cache piu piccole di Cloudflare battono la velocita pura"
 * (the decode kernel reads the FP8 cache and converts it as it reads): here
 * the e4m3 codes of K and V enter the MMAs as they lie in shared memory, and
 * the query and the softmax weights enter as four e4m3 parts each
 * (x = c0 + c1/16 + c2/256 + c3/4096, 16 significant bits), recombined in
 * fp32 from the accumulators.
 * Differences from fpk_paged_decode_attn_fp8:
 *   - num_splits == 0 picks one wave of CTAs (at most 16 splits per
 *     (request, kv head)), or, when every non-empty request has the same
 *     length, the uniform rule of fpk_paged_decode_attn_fp8; mixed-length
 *     small batches keep equal-size splits (no segment-aligned partition);
 *   - a split count above the batch's 16-token tile count is lowered to it;
 *   - every split of a segment is merged in one level (no groups above 16);
 *   - the pool may hold at most 2^31 rows of 128 bytes (256 GiB), else
 *     FPK_EUNSUPPORTED.
 * Bit-identical on repeated calls with the same inputs and split count.
 */
int fpk_paged_decode_attn_fp8_tc(const void* q, const uint8_t* kv_pool,
                                 const float* k_scale, const float* v_scale,
                                 const int32_t* page_table, int32_t max_pages,
                                 const int32_t* seq_lens, const uint8_t* abort_mask,
                                 float* out, float* lse, void* workspace, size_t workspace_bytes,
                                 int32_t num_splits, float sm_scale, int32_t B, int32_t Hq,
                                 int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
                                 void* stream);

/* BF16-cache variant of fpk_paged_decode_attn_fp8: same semantics with
 * kv_pool holding bf16 values (no scales). */
int fpk_paged_decode_attn_bf16(const void* q, const void* kv_pool,
                               const int32_t* page_table, int32_t max_pages,
                               const int32_t* seq_lens, const uint8_t* abort_mask,
                               float* out, float* lse, void* workspace, size_t workspace_bytes,
                               int32_t num_splits, float sm_scale, int32_t B, int32_t Hq,
                               int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
                               void* stream);

/*
 * One whole decode step: fpk_decode_append_check_fp8 (the new token's write
 * and the batched tag check, one launch) followed by
 * fpk_paged_decode_attn_fp8 over the requests that passed, in the order the
 * pages give (write, check before the decode operation reads, attend:
 * "Cosa ha cambiato Cloudflare per Kimi e GLM" and "La sicurezza della cache
 * KV condivisa...").  The check stays its own kernel; the attention kernel is
 * launched as a programmatic dependent of it, so its set-up (work split,
 * barriers) overlaps the check, and it reads the abort mask and the cache only
 * once the check kernel has completed.  Arguments as in the two calls.  With
 * live_tags and expected_tags both NULL (the no-op tracker) the step writes
 * unguarded and attends every request, ignoring abort_mask.  All arguments
 * are checked before anything is launched.
 */
int fpk_decode_step_fp8(const void* k_new, const void* v_new, uint8_t* kv_pool,
                        const float* k_scale, const float* v_scale,
                        const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                        const uint32_t* live_tags, const uint32_t* expected_tags,
                        uint8_t* abort_mask, const void* q, float* out, float* lse,
                        void* workspace, size_t workspace_bytes, int32_t num_splits,
                        float sm_scale, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                        int32_t page_size, int32_t num_pages, void* stream);

/* BF16-cache variant of fpk_decode_step_fp8 (no scales). */
int fpk_decode_step_bf16(const void* k_new, const void* v_new, void* kv_pool,
                         const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                         const uint32_t* live_tags, const uint32_t* expected_tags,
                         uint8_t* abort_mask, const void* q, float* out, float* lse,
                         void* workspace, size_t workspace_bytes, int32_t num_splits,
                         float sm_scale, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t page_size, int32_t num_pages, void* stream);

/*
 * Allocation-free variant of fpk_paged_decode_attn_fp8 (same arguments and
 * results, minus the workspace).  The write-up has no counterpart of this
 * entry point; it exists for callers that cannot allocate device memory --
 * operator hosts and plugin interfaces that hand an operator only its inputs
 * and outputs, processes held to a fixed device-memory budget, and
 * latency-critical loops that cannot afford cudaMalloc's implicit device
 * synchronisation.  The caller still passes q, the pool, tables, out and lse.
 *
 * Scratch: a fixed 16 MiB array inside the library, which every GPU that
 * loads the library holds until the process exits.  A batch whose workspace
 * (fpk_decode_workspace_bytes) would exceed 16 MiB is rejected with
 * FPK_ENOSPC before anything is launched.  The call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 * Set-up: the first call on a device looks up the array's device address on
 * that device (the device current at the call); make that first call before
 * any stream capture.  The address is kept per device and context: after a
 * device reset the next call looks it up again (set-up again, so again
 * outside any capture).
 * Sharing: every call on a device uses the same array and clears its status
 * word and counters first; calls that overlap on the GPU (other streams or
 * other host threads) race on it and must be serialised by the caller.
 * Errors: arguments are checked before any CUDA call, so a rejected call
 * queues nothing.  The kernel's status word (a bounded wait that gave up
 * leaves some out/lse rows unwritten) stays in the scratch until the next
 * call: read it with fpk_decode_status(NULL, ...) on the same device.
 */
int fpk_paged_decode_attn_fp8_noalloc(const void* q, const uint8_t* kv_pool,
                                      const float* k_scale, const float* v_scale,
                                      const int32_t* page_table, int32_t max_pages,
                                      const int32_t* seq_lens, const uint8_t* abort_mask,
                                      float* out, float* lse, int32_t num_splits, float sm_scale,
                                      int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                      int32_t page_size, int32_t num_pages, void* stream);

/*
 * Copies the workspace status word to *status (HOST pointer) and synchronises
 * the stream.  0 means no bounded wait inside the attention kernels gave up.
 * workspace == NULL reads the status word of the last
 * fpk_paged_decode_attn_fp8_noalloc call on the current device instead.
 */
int fpk_decode_status(const void* workspace, int32_t* status, void* stream);

/*
 * Self-test of the bounded waits (the failure report every kernel relies on,
 * not a step of the path).  Launches one CTA that waits on an mbarrier nothing
 * arrives on: the wait gives up after its time limit (2 s), ORs 1 into *status
 * (the same bit the attention kernel sets in its workspace status word) and
 * the kernel exits; *elapsed_ns receives the time the wait took.  The context
 * stays usable.
 *   status    : uint32 [1], device; elapsed_ns: uint64 [1], device
 */
int fpk_selftest_bounded_wait(uint32_t* status, unsigned long long* elapsed_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8KV_H_ */
