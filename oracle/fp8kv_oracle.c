/*
 * fp8kv_oracle.c -- plain, slow CPU oracle of the FP8 paged-KV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the package entry's smoke check and
 * the benchmark's CPU-baseline leg and reference arm load it.  It shares no header, helper,
 * table or constant with the CUDA path.
 *
 * What the method computes (sources are the five web pages reporting the
 * Cloudflare Workers AI write-up on serving Kimi K2.6 / GLM 5.2):
 *
 *  - "Il serving di modelli piu piccoli di Cloudflare riduce la memoria, ma la
 *    sicurezza diventa la prova decisiva" (remio.ai, Italian edition),
 *    section "Cosa ha cambiato Cloudflare per Kimi e GLM": the Kimi KV cache is
 *    held as FP8 e4m3 instead of BF16 (half the bytes); every physical cache
 *    page carries a tag that changes whenever the page is reallocated; the
 *    server records which pages and tags each request expects; the mappings
 *    are checked before supported decode operations read the pages, and a
 *    mismatch aborts the affected request.
 *  - same page, section "Perche le cache piu piccole di Cloudflare battono la
 *    velocita pura": the attention kernel converts the cached values when it
 *    reads them.
 *  - same page, section "La sicurezza della cache KV condivisa diventa una
 *    questione di produzione": paged attention splits the cache into reusable
 *    blocks with a logical-to-physical mapping per sequence; the check runs as
 *    a separate batched operation, not fused into attention; tags behave like
 *    generation counters.
 *  - "Cloudflare uskorila Kimi na 41% szhatiem KV-kesha" (iitog.ru), the
 *    paragraph on the third technique: many requests both read and write the
 *    pages of one physical cache.
 *
 * The pages fix neither formulas nor layouts.  Readings taken here (each one
 * is listed in the design notes of the repository):
 *   e4m3 = OCP OFP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
 *   bits, no infinities, NaN = S.1111.111, largest finite 448); encoding is
 *   round-to-nearest-even with saturation to +-448; NaN encodes as 0x7F;
 *   quantisation divides by a per-tensor fp32 scale in IEEE fp32 first;
 *   the softmax scale is an explicit argument (1/sqrt(D) in the workloads);
 *   query head h reads kv head h / (Hq/Hkv); tags are uint32 compared for
 *   equality and bumped by +1 modulo 2^32; a page id outside [0, num_pages)
 *   aborts; only the first ceil(L/page_size) entries of a page table are
 *   checked; an aborted or empty request yields out = 0, lse = -inf.
 *
 * Pool layout (the library's documented storage format, restated here from
 * its definition, not shared with it): one KV pool per layer,
 *   kv_pool[num_pages][Hkv][page_size/16][2][16*D]
 * i.e. for every page, kv head and 16-token tile of the page, the tile's K
 * block [16 tokens][D] (token-major) followed by its V block [D][16 tokens]
 * (dim-major); element = 1 byte (e4m3 code) or 2 bytes (bf16 bit pattern).
 *
 * All floating point is fp64 except the single fp32 division x/scale that the
 * quantiser is defined on.  Build with -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* bf16 and e4m3 codecs                                                       */
/* ------------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32 bit pattern. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* E4M3 decode: e == 0 -> (-1)^s * m * 2^-9 (subnormal),
 * else (-1)^s * (1 + m/8) * 2^(e-7); S.1111.111 is NaN. */
double orc_e4m3_decode(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* E4M3 encode of an fp32 value: round to nearest, ties to even, saturate
 * finite and infinite overflow to +-448, NaN -> 0x7F, -0 -> 0x80. */
uint8_t orc_e4m3_encode(float xf)
{
    double x = (double)xf;
    uint8_t sign;
    double a;
    int code;

    if (isnan(x))
        return 0x7F;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs(x);
    if (isinf(a))
        return (uint8_t)(sign | 0x7E);

    if (a < ldexp(1.0, -6)) {
        /* subnormal binade: multiples of 2^-9; q == 8 is the smallest normal */
        double q = nearbyint(a * 512.0);
        code = (int)q;
    } else {
        int e2;
        double f = frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
        int E = e2 - 1;                    /* a = (2f) * 2^E, 2f in [1, 2) */
        double mant = nearbyint((2.0 * f - 1.0) * 8.0);
        int field;
        if (mant >= 8.0) {                 /* rounding carried into the exponent */
            mant = 0.0;
            E += 1;
        }
        field = E + 7;
        if (field > 15 || (field == 15 && mant > 6.0))
            code = 0x7E;                   /* saturate to 448 */
        else
            code = (field << 3) | (int)mant;
    }
    return (uint8_t)(sign | code);
}

void orc_e4m3_encode_array(const float *x, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(x[i]);
}

void orc_e4m3_decode_array(const uint8_t *c, int64_t n, double *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = orc_e4m3_decode(c[i]);
}

/* The quantiser input: float(bf16 x) / scale as one IEEE fp32 division. */
uint8_t orc_quantize_bf16(uint16_t xbits, float scale)
{
    volatile float num = bf16_bits_to_float(xbits);
    volatile float q = num / scale;
    return orc_e4m3_encode(q);
}

void orc_quantize_bf16_array(const uint16_t *xbits, int64_t n, float scale, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = orc_quantize_bf16(xbits[i], scale);
}

/*
 * Per-tensor scale of the e4m3 cache: amax / 448 over the finite elements of a
 * bf16 tensor, 1 when there is no nonzero finite element.  The pages name the
 * e4m3 format only ("Cosa ha cambiato Cloudflare per Kimi e GLM"); one fp32
 * scale per tensor with the tensor's largest magnitude mapped to the largest
 * finite code (448) is the reading taken.  amax is exact in double; the scale
 * is one IEEE fp32 division.
 */
float orc_amax_scale_bf16(const uint16_t *xbits, int64_t n)
{
    int64_t i;
    double amax = 0.0;
    volatile float a, q;
    for (i = 0; i < n; ++i) {
        double x = (double)bf16_bits_to_float(xbits[i]);
        if (isfinite(x) && fabs(x) > amax)
            amax = fabs(x);
    }
    if (amax == 0.0)
        return 1.0f;
    a = (float)amax;
    q = a / 448.0f;
    return q;
}

/* ------------------------------------------------------------------------- */
/* pool indexing (the documented layout)                                      */
/* ------------------------------------------------------------------------- */

/* first element of the (K, V) block pair of the tile holding slot `off` */
static int64_t tile_base(int64_t page, int h, int off, int Hkv, int ps, int D)
{
    return (((page * Hkv + h) * (int64_t)(ps / 16) + off / 16) * 2) * 16 * (int64_t)D;
}

static int64_t k_index(int64_t page, int h, int off, int d, int Hkv, int ps, int D)
{
    return tile_base(page, h, off, Hkv, ps, D) + (int64_t)(off % 16) * D + d;
}

static int64_t v_index(int64_t page, int h, int off, int d, int Hkv, int ps, int D)
{
    return tile_base(page, h, off, Hkv, ps, D) + 16 * (int64_t)D + (int64_t)d * 16 + off % 16;
}

/* ------------------------------------------------------------------------- */
/* writing tokens into pages                                                  */
/* ------------------------------------------------------------------------- */

/*
 * Write one token's K and V rows (all Hkv heads) of request r at position pos.
 * The destination page's tag is compared first; a page id out of range, a
 * position beyond the page table or a stale tag skips the write and marks the
 * request in abort_mask (when given).  Returns 1 if written, 0 if skipped.
 */
static int write_token(const uint16_t *krow, const uint16_t *vrow, int is_fp8,
                       void *kv_pool, float k_scale, float v_scale,
                       const int32_t *page_table, int max_pages, int r, int pos,
                       const uint32_t *live_tags, const uint32_t *expected_tags,
                       uint8_t *abort_mask, int Hkv, int D, int ps, int num_pages)
{
    int pi = pos / ps, off = pos % ps, h, d;
    int32_t page;
    if (pos < 0 || pi >= max_pages) {
        if (abort_mask) abort_mask[r] = 1;
        return 0;
    }
    page = page_table[(int64_t)r * max_pages + pi];
    if (page < 0 || page >= num_pages) {
        if (abort_mask) abort_mask[r] = 1;
        return 0;
    }
    if (live_tags && expected_tags &&
        live_tags[page] != expected_tags[(int64_t)r * max_pages + pi]) {
        if (abort_mask) abort_mask[r] = 1;
        return 0;
    }
    for (h = 0; h < Hkv; ++h) {
        for (d = 0; d < D; ++d) {
            uint16_t kb = krow[(int64_t)h * D + d], vb = vrow[(int64_t)h * D + d];
            int64_t ki = k_index(page, h, off, d, Hkv, ps, D);
            int64_t vi = v_index(page, h, off, d, Hkv, ps, D);
            if (is_fp8) {
                ((uint8_t *)kv_pool)[ki] = orc_quantize_bf16(kb, k_scale);
                ((uint8_t *)kv_pool)[vi] = orc_quantize_bf16(vb, v_scale);
            } else {
                ((uint16_t *)kv_pool)[ki] = kb;
                ((uint16_t *)kv_pool)[vi] = vb;
            }
        }
    }
    return 1;
}

/*
 * Decode-step append: one new token per request, written at position
 * seq_lens[r] - 1 (seq_lens already counts the new token).  Requests with
 * seq_lens[r] <= 0 append nothing.  k_new, v_new: bf16 [B][Hkv][D].
 */
void orc_kv_append(const uint16_t *k_new, const uint16_t *v_new, int is_fp8,
                   void *kv_pool, float k_scale, float v_scale,
                   const int32_t *page_table, int max_pages, const int32_t *seq_lens,
                   const uint32_t *live_tags, const uint32_t *expected_tags,
                   uint8_t *abort_mask, int B, int Hkv, int D, int ps, int num_pages)
{
    int r;
    for (r = 0; r < B; ++r) {
        int L = seq_lens[r];
        if (L <= 0)
            continue;
        write_token(k_new + (int64_t)r * Hkv * D, v_new + (int64_t)r * Hkv * D, is_fp8,
                    kv_pool, k_scale, v_scale, page_table, max_pages, r, L - 1,
                    live_tags, expected_tags, abort_mask, Hkv, D, ps, num_pages);
    }
}

/*
 * Bulk write of whole prompts: rows cu_seqlens[r] .. cu_seqlens[r+1]-1 of
 * k, v (bf16 [N][Hkv][D]) are request r's tokens at positions 0, 1, ...
 */
void orc_kv_prefill(const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens, int is_fp8,
                    void *kv_pool, float k_scale, float v_scale,
                    const int32_t *page_table, int max_pages,
                    const uint32_t *live_tags, const uint32_t *expected_tags,
                    uint8_t *abort_mask, int B, int Hkv, int D, int ps, int num_pages)
{
    int r, i;
    for (r = 0; r < B; ++r) {
        for (i = cu_seqlens[r]; i < cu_seqlens[r + 1]; ++i) {
            write_token(k + (int64_t)i * Hkv * D, v + (int64_t)i * Hkv * D, is_fp8,
                        kv_pool, k_scale, v_scale, page_table, max_pages, r,
                        i - cu_seqlens[r], live_tags, expected_tags, abort_mask,
                        Hkv, D, ps, num_pages);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* page tags                                                                  */
/* ------------------------------------------------------------------------- */

/* Reallocation: each listed page's tag advances by one, modulo 2^32.  Ids
 * outside [0, num_pages) are ignored; a repeated id advances once per entry. */
void orc_page_tags_bump(uint32_t *live_tags, const int32_t *pages, int n, int num_pages)
{
    int i;
    for (i = 0; i < n; ++i) {
        int32_t p = pages[i];
        if (p >= 0 && p < num_pages)
            live_tags[p] = live_tags[p] + 1u;
    }
}

/*
 * Batched check before the pages are read: request r is aborted iff one of
 * its first P_r = ceil(seq_lens[r] / ps) table entries names a page outside
 * [0, num_pages) or a page whose live tag differs from the expected tag, or
 * P_r exceeds the table width.  abort_mask is overwritten; returns the count.
 */
int orc_page_tags_validate(const int32_t *page_table, const uint32_t *expected_tags,
                           const int32_t *seq_lens, int max_pages,
                           const uint32_t *live_tags, int num_pages, int B, int ps,
                           uint8_t *abort_mask)
{
    int r, i, count = 0;
    for (r = 0; r < B; ++r) {
        int L = seq_lens[r];
        int P = L > 0 ? (L + ps - 1) / ps : 0;
        int bad = 0;
        if (P > max_pages)
            bad = 1;
        for (i = 0; i < P && !bad; ++i) {
            int32_t page = page_table[(int64_t)r * max_pages + i];
            if (page < 0 || page >= num_pages)
                bad = 1;
            else if (live_tags[page] != expected_tags[(int64_t)r * max_pages + i])
                bad = 1;
        }
        abort_mask[r] = (uint8_t)bad;
        count += bad;
    }
    return count;
}

/* ------------------------------------------------------------------------- */
/* attention                                                                  */
/* ------------------------------------------------------------------------- */

static double load_k(const void *pool, int is_fp8, int64_t idx, double scale)
{
    if (is_fp8)
        return orc_e4m3_decode(((const uint8_t *)pool)[idx]) * scale;
    return (double)bf16_bits_to_float(((const uint16_t *)pool)[idx]);
}

/*
 * Decode attention over the paged cache, fp64, no splitting.
 * For request r and query head h (kv head h / G):
 *   s_j = sm_scale * sum_d q[d] * khat_j[d],      j < L_r
 *   out = sum_j exp(s_j - m) vhat_j / sum_j exp(s_j - m),  m = max_j s_j
 *   lse = m + log(sum_j exp(s_j - m))
 * khat = decode(code) * k_scale for the FP8 cache, the bf16 value otherwise.
 * Aborted (abort_mask[r] != 0), empty, over-long or out-of-range-page requests
 * give out = 0, lse = -inf.  scores: caller scratch of >= max_pages*ps doubles.
 */
void orc_paged_attention(const uint16_t *q, const void *kv_pool, int is_fp8,
                         double k_scale, double v_scale, const int32_t *page_table, int max_pages,
                         const int32_t *seq_lens, const uint8_t *abort_mask, double sm_scale,
                         int B, int Hq, int Hkv, int D, int ps, int num_pages,
                         double *scores, double *out, double *lse)
{
    int r, h, j, d;
    int G = Hq / Hkv;
    for (r = 0; r < B; ++r) {
        int L = seq_lens[r];
        int P = L > 0 ? (L + ps - 1) / ps : 0;
        int dead = (L <= 0) || (abort_mask && abort_mask[r]) || (P > max_pages);
        int i;
        for (i = 0; i < P && !dead; ++i) {
            int32_t page = page_table[(int64_t)r * max_pages + i];
            if (page < 0 || page >= num_pages)
                dead = 1;
        }
        for (h = 0; h < Hq; ++h) {
            int hk = h / G;
            double *o = out + ((int64_t)r * Hq + h) * D;
            const uint16_t *qr = q + ((int64_t)r * Hq + h) * D;
            double m = -INFINITY, l = 0.0;
            if (dead) {
                for (d = 0; d < D; ++d) o[d] = 0.0;
                lse[(int64_t)r * Hq + h] = -INFINITY;
                continue;
            }
            for (j = 0; j < L; ++j) {
                int64_t page = page_table[(int64_t)r * max_pages + j / ps];
                double acc = 0.0;
                for (d = 0; d < D; ++d) {
                    double kv = load_k(kv_pool, is_fp8, k_index(page, hk, j % ps, d, Hkv, ps, D), k_scale);
                    acc += (double)bf16_bits_to_float(qr[d]) * kv;
                }
                scores[j] = acc * sm_scale;
                if (scores[j] > m) m = scores[j];
            }
            for (d = 0; d < D; ++d) o[d] = 0.0;
            for (j = 0; j < L; ++j) {
                int64_t page = page_table[(int64_t)r * max_pages + j / ps];
                double p = exp(scores[j] - m);
                l += p;
                for (d = 0; d < D; ++d)
                    o[d] += p * load_k(kv_pool, is_fp8, v_index(page, hk, j % ps, d, Hkv, ps, D), v_scale);
            }
            for (d = 0; d < D; ++d) o[d] /= l;
            lse[(int64_t)r * Hq + h] = m + log(l);
        }
    }
}

/*
 * Textbook dense attention for one query vector, written without paging:
 * softmax(q K^T * sm_scale) V with K, V given densely as [L][D] doubles.
 */
void orc_dense_attention(const double *q, const double *K, const double *V, int L, int D,
                         double sm_scale, double *scores, double *out, double *lse)
{
    int j, d;
    double m = -INFINITY, z = 0.0;
    for (j = 0; j < L; ++j) {
        double s = 0.0;
        for (d = 0; d < D; ++d) s += q[d] * K[(int64_t)j * D + d];
        scores[j] = s * sm_scale;
        m = fmax(m, scores[j]);
    }
    for (j = 0; j < L; ++j) {
        scores[j] = exp(scores[j] - m);
        z += scores[j];
    }
    for (d = 0; d < D; ++d) {
        double acc = 0.0;
        for (j = 0; j < L; ++j) acc += scores[j] / z * V[(int64_t)j * D + d];
        out[d] = acc;
    }
    *lse = m + log(z);
}

/* ------------------------------------------------------------------------- */
/* weight-only quantised GEMV (the pages' second technique)                   */
/* ------------------------------------------------------------------------- */
/*
 * "La compressione dei pesi GLM modifica il compromesso tra le fasi"
 * (remio.ai): GLM 5.2's weights went from FP8 to INT4 for decode, where every
 * weight is read from memory at each step.  The pages give no format; the
 * readings taken (groups of 128 along K with a bf16 scale amax / 7 and codes
 * rint(w / s) clamped to [-8, 7]; e4m3 weights with an fp32 scale
 * amax / 448 per row) are restated here from their definitions.
 */

/* float -> bf16 bits, round to nearest even (NaN -> quiet NaN). */
static uint16_t bf16_round(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x40u);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

/* INT4: q [N][K] in [-8, 7] and bf16 scales [N][K/128], natural layout. */
void orc_w4_quantize(const uint16_t *w, int N, int K, int8_t *q, uint16_t *scales)
{
    int n, g, k, G = K / 128;
    for (n = 0; n < N; ++n) {
        for (g = 0; g < G; ++g) {
            double amax = 0.0;
            volatile float af, sq;
            float sf;
            uint16_t sb;
            for (k = 128 * g; k < 128 * (g + 1); ++k) {
                double x = (double)bf16_bits_to_float(w[(int64_t)n * K + k]);
                if (isfinite(x) && fabs(x) > amax) amax = fabs(x);
            }
            af = (float)amax;
            sq = af / 7.0f;
            sb = bf16_round(sq);
            scales[(int64_t)n * G + g] = sb;
            sf = bf16_bits_to_float(sb);
            for (k = 128 * g; k < 128 * (g + 1); ++k) {
                float x = bf16_bits_to_float(w[(int64_t)n * K + k]);
                int code = 0;
                if (sf != 0.0f && isfinite(x)) {
                    volatile float r = x / sf;
                    float v = nearbyintf(r);
                    code = v > 7.0f ? 7 : v < -8.0f ? -8 : (int)v;
                }
                q[(int64_t)n * K + k] = (int8_t)code;
            }
        }
    }
}

/* e4m3 weights: codes [N][K] and fp32 row scales [N], natural layout. */
void orc_w8_quantize(const uint16_t *w, int N, int K, uint8_t *codes, float *row_scales)
{
    int n, k;
    for (n = 0; n < N; ++n) {
        double amax = 0.0;
        volatile float af, r;
        for (k = 0; k < K; ++k) {
            double x = (double)bf16_bits_to_float(w[(int64_t)n * K + k]);
            if (isfinite(x) && fabs(x) > amax) amax = fabs(x);
        }
        af = (float)amax;
        r = amax == 0.0 ? 1.0f : af / 448.0f;
        row_scales[n] = r;
        for (k = 0; k < K; ++k)
            codes[(int64_t)n * K + k] = orc_quantize_bf16(w[(int64_t)n * K + k], r);
    }
}

/* The INT4 slice layout, written from its definition: byte
 * 512h + 16l + 4u + p/2 of slice (s, g) holds, in its low (p even) or high
 * nibble, element (16s + 8h + l/4, 128g + 16(2u + ((p>>1)&1)) + 4(l%4) + 2(p&1) + (p>>2)). */
void orc_w4_pack(const int8_t *q, int N, int K, uint8_t *out)
{
    int s, g, h, l, u, p, G = K / 128;
    for (s = 0; s < N / 16; ++s)
        for (g = 0; g < G; ++g)
            for (h = 0; h < 2; ++h)
                for (l = 0; l < 32; ++l)
                    for (u = 0; u < 4; ++u)
                        for (p = 0; p < 8; ++p) {
                            int row = 16 * s + 8 * h + l / 4;
                            int k = 128 * g + 16 * (2 * u + ((p >> 1) & 1)) + 4 * (l % 4) + 2 * (p & 1) + (p >> 2);
                            uint8_t nib = (uint8_t)(q[(int64_t)row * K + k] + 8);
                            int64_t byte = ((int64_t)s * G + g) * 1024 + 512 * h + 16 * l + 4 * u + p / 2;
                            if ((p & 1) == 0) out[byte] = (uint8_t)((out[byte] & 0xF0) | nib);
                            else out[byte] = (uint8_t)((out[byte] & 0x0F) | (nib << 4));
                        }
}

/* The e4m3 slice layout: byte 1024h + 512c + 16l + b of slice (s, g) holds
 * element (16s + 8h + l/4, 128g + 16(4c + b/4) + 4(l%4) + b%4). */
void orc_w8_pack(const uint8_t *codes, int N, int K, uint8_t *out)
{
    int s, g, h, c, l, b, G = K / 128;
    for (s = 0; s < N / 16; ++s)
        for (g = 0; g < G; ++g)
            for (h = 0; h < 2; ++h)
                for (c = 0; c < 2; ++c)
                    for (l = 0; l < 32; ++l)
                        for (b = 0; b < 16; ++b) {
                            int row = 16 * s + 8 * h + l / 4;
                            int k = 128 * g + 16 * (4 * c + b / 4) + 4 * (l % 4) + b % 4;
                            out[((int64_t)s * G + g) * 2048 + 1024 * h + 512 * c + 16 * l + b] =
                                codes[(int64_t)row * K + k];
                        }
}

/* y[b][n] = sum_k x[b][k] * q[n][k] * s[n][k/128], in fp64. */
void orc_w4_gemv(const uint16_t *x, int B, const int8_t *q, const uint16_t *scales, int N, int K,
                 double *y)
{
    int b, n, k, G = K / 128;
    for (b = 0; b < B; ++b)
        for (n = 0; n < N; ++n) {
            double acc = 0.0;
            for (k = 0; k < K; ++k)
                acc += (double)bf16_bits_to_float(x[(int64_t)b * K + k]) * (double)q[(int64_t)n * K + k] *
                       (double)bf16_bits_to_float(scales[(int64_t)n * G + k / 128]);
            y[(int64_t)b * N + n] = acc;
        }
}

/* y[b][n] = sum_k x[b][k] * decode(code[n][k]) * r[n], in fp64. */
void orc_w8_gemv(const uint16_t *x, int B, const uint8_t *codes, const float *row_scales, int N, int K,
                 double *y)
{
    int b, n, k;
    for (b = 0; b < B; ++b)
        for (n = 0; n < N; ++n) {
            double acc = 0.0;
            for (k = 0; k < K; ++k)
                acc += (double)bf16_bits_to_float(x[(int64_t)b * K + k]) *
                       orc_e4m3_decode(codes[(int64_t)n * K + k]);
            y[(int64_t)b * N + n] = acc * (double)row_scales[n];
        }
}
