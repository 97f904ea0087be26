// wgemv.cu -- weight-only quantised decode GEMV, y[b] = W x[b] for a decode
// batch of up to 16 tokens: INT4 weights in groups of 128 along K with one
// bf16 scale per group, or e4m3 weights with one fp32 scale per row (the
// comparison); bf16 activations, fp32 output.
//
// The Cloudflare write-up's second technique ("La compressione dei pesi GLM
// modifica il compromesso tra le fasi", remio.ai): GLM 5.2's weights went from
// FP8 to INT4 because decode streams every weight from HBM at each step, so
// fewer bytes per weight make each token faster; INT4 weights are expanded
// before the multiplication.  The pages give no format: the groups of 128, the
// amax/7 scale, the excess-8 nibbles and the slice layout are this library's.
//
// Layout (both formats): W [N][K] is cut into slices of 16 rows x 128 k, each
// stored in the order one warp's m16n8k16 fragments consume it, so every lane
// reads its operand words as 16-byte vectors straight from HBM.  Within a
// 16-k step the four k of a lane (t = lane % 4) are 4t .. 4t+3 -- a fixed
// permutation of the fragment's k order applied to both operands, so each
// lane's activation operand is one 8-byte load of 4 consecutive k.
//   INT4 slice, 1024 bytes: byte 512*half + 16*lane + 4*w + (0..3) holds
//     word w (steps 2w, 2w+1) of row 8*half + lane/4; nibble p of the word
//     (bits 4p..4p+3) is element k = 16*s + 4*(lane%4) + j with
//     s = 2w + ((p >> 1) & 1), j = 2*(p & 1) + (p >> 2); value = nibble - 8.
//   e4m3 slice, 2048 bytes: byte 1024*half + 512*part + 16*lane + b holds row
//     8*half + lane/4, k = 16*(4*part + b/4) + 4*(lane%4) + b%4.
// Slices are stored [N/16][K/128] (slice row-block major).
#include "step_ops.cuh"

namespace fpk {
namespace {

constexpr int kGroupK = 128;
constexpr int kW4SliceBytes = 16 * kGroupK / 2;
constexpr int kW8SliceBytes = 16 * kGroupK;
constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kKChunk = 2048;  // k per CTA (split-K)
// INT4 weights at one token: the largest K one CTA takes whole (its 64 rows'
// group scales fill the same table as 128 rows of a kKChunk chunk, twice over)
constexpr int kWholeKMax = 8192;
constexpr int kGscaleEntries = (kGemvWarps / 2) * 16 * (kWholeKMax / kGroupK);
static_assert(kGemvWarps * 16 * (2 * kKChunk / kGroupK) <= kGscaleEntries, "the scale table holds a chunk's too");
constexpr int kXPad = 16;      // bf16 of padding per staged activation row

__device__ __forceinline__ int w4_nibble_index(int s, int j) {
  return 2 * (s & 1) + ((j & 1) ? 4 : 0) + (j >> 1);
}

// Fifteen magnitudes of bf16 finite values: the largest |x| of the 32 values
// of a lane over the 4 lanes that share a row (lanes 4r .. 4r+3).
__device__ __forceinline__ float row_amax4(float m) {
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  return m;
}

// Lane's 32 values of one row of a slice: k = 16 s + 4 t + j -> v[4 s + j].
__device__ __forceinline__ void load_row32(const uint16_t* __restrict__ rowp, int t, float (&v)[32]) {
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(rowp + 16 * s + 4 * t));
    v[4 * s + 0] = __uint_as_float(raw.x << 16);
    v[4 * s + 1] = __uint_as_float(raw.x & 0xFFFF0000u);
    v[4 * s + 2] = __uint_as_float(raw.y << 16);
    v[4 * s + 3] = __uint_as_float(raw.y & 0xFFFF0000u);
  }
}

// INT4 quantiser: one warp per (slice, group).  Per row and group:
// s = bf16(amax / 7) over the finite values, q = clamp(rint(w / s), -8, 7)
// (0 for a non-finite w or s == 0), stored as q + 8.
__global__ void __launch_bounds__(256) w4_quantize_kernel(const uint16_t* __restrict__ w,
                                                          uint8_t* __restrict__ codes,
                                                          uint16_t* __restrict__ scales, int N, int K) {
  const int G = K / kGroupK;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (unit >= static_cast<int64_t>(N / 16) * G) return;
  const int lane = threadIdx.x & 31, rr = lane >> 2, t = lane & 3;
  const int slice = static_cast<int>(unit / G), g = static_cast<int>(unit % G);
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    const int row = 16 * slice + 8 * half + rr;
    float v[32];
    load_row32(w + static_cast<int64_t>(row) * K + kGroupK * g, t, v);
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (isfinite(v[i])) m = fmaxf(m, fabsf(v[i]));
    m = row_amax4(m);
    const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(m, 7.f));
    const float sf = __bfloat162float(sb);
    uint32_t word[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x = v[4 * s + j];
        int q = 0;
        if (sf != 0.f && isfinite(x)) q = max(-8, min(7, static_cast<int>(rintf(__fdiv_rn(x, sf)))));
        word[s >> 1] |= static_cast<uint32_t>(q + 8) << (4 * w4_nibble_index(s, j));
      }
    }
    *reinterpret_cast<uint4*>(codes + static_cast<int64_t>(unit) * kW4SliceBytes + 512 * half + 16 * lane) =
        make_uint4(word[0], word[1], word[2], word[3]);
    if (t == 0) scales[static_cast<int64_t>(row) * G + g] = *reinterpret_cast<const uint16_t*>(&sb);
  }
}

// e4m3 weights, step 1: the per-row scale amax / 448 over the finite values
// (1 if there are none but zeros); one warp per row.
__global__ void __launch_bounds__(256) w8_row_scale_kernel(const uint16_t* __restrict__ w,
                                                           float* __restrict__ row_scales, int N, int K) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= N) return;
  const int lane = threadIdx.x & 31;
  const uint16_t* p = w + static_cast<int64_t>(row) * K;
  uint32_t m2 = 0;  // two 16-bit maxima of |x| bit patterns, non-finite as 0
  for (int k = 8 * lane; k < K; k += 256) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p + k));
    const uint32_t ws[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t a = ws[i] & 0x7FFF7FFFu;
      a &= __vcmpltu2(a, 0x7F807F80u);
      m2 = __vmaxu2(m2, a);
    }
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = __reduce_max_sync(0xffffffffu, m);
  if (lane == 0) row_scales[row] = m == 0 ? 1.f : __fdiv_rn(__uint_as_float(m << 16), 448.f);
}

// e4m3 weights, step 2: codes e4m3(w / row_scale) in slice order; one warp per
// (slice, group).
__global__ void __launch_bounds__(256) w8_quantize_kernel(const uint16_t* __restrict__ w,
                                                          const float* __restrict__ row_scales,
                                                          uint8_t* __restrict__ codes, int N, int K) {
  const int G = K / kGroupK;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (unit >= static_cast<int64_t>(N / 16) * G) return;
  const int lane = threadIdx.x & 31, rr = lane >> 2, t = lane & 3;
  const int slice = static_cast<int>(unit / G), g = static_cast<int>(unit % G);
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    const int row = 16 * slice + 8 * half + rr;
    const Divisor d = make_divisor(__ldg(row_scales + row));
    float v[32];
    load_row32(w + static_cast<int64_t>(row) * K + kGroupK * g, t, v);
    uint32_t word[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(div_by(v[4 * i], d), div_by(v[4 * i + 1], d)),
                                                   __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(div_by(v[4 * i + 2], d), div_by(v[4 * i + 3], d)),
                                                   __NV_SATFINITE, __NV_E4M3);
      word[i] = lo | (hi << 16);  // step i, j = 0..3
    }
    uint8_t* dst = codes + static_cast<int64_t>(unit) * kW8SliceBytes + 1024 * half + 16 * lane;
    *reinterpret_cast<uint4*>(dst) = make_uint4(word[0], word[1], word[2], word[3]);
    *reinterpret_cast<uint4*>(dst + 512) = make_uint4(word[4], word[5], word[6], word[7]);
  }
}

struct GemvArgs {
  const uint16_t* x;        // bf16 [B][K]
  const uint8_t* codes;     // slices [N/16][K/128]
  const uint16_t* gscales;  // INT4: bf16 [N][K/128]
  const float* rscales;     // e4m3: fp32 [N]
  float* y;                 // fp32 [B][N]
  int B, N, K;
  int kc;                   // k per CTA (a multiple of 128, at most kKChunk)
  int atomic;               // several K chunks add into y
};

// Asynchronous 16-byte global -> shared copy (Ampere-style cp.async, L2 only).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// f16x2 of two nibbles of v (bits 0..3 and 16..19 when kHigh is false, bits
// 4..7 and 20..23 when true) by placing them in the mantissa of 1024.0
// (0x6400: the unit in the last place is 1), then subtracting the bias:
// 1024 + 8 gives n - 8; for the upper nibbles, 1024 + 16 n - (1024 + 128)
// gives 16 (n - 8) -- every step exact in f16.
// mask and magic are passed in registers so that the and-or is one LOP3.
__device__ __forceinline__ uint32_t w4_pair_to_f16x2(uint32_t v, uint32_t mask, uint32_t magic, uint32_t bias) {
  uint32_t b;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(b) : "r"(v), "r"(mask), "r"(magic));  // (v & mask) | magic
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&b), *reinterpret_cast<const __half2*>(&bias));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// One CTA: 8 warps x one 16-row slice each, over one K chunk of up to 2048.
// Each lane streams its own 16-byte words of the warp's slice groups into a
// shared-memory ring with cp.async (in the slice layout a lane reads back only
// the bytes it copied itself, so no cross-lane barrier is needed), keeping
// kRing - 1 groups in flight without holding them in registers.  The chunk's
// activations are staged once per CTA as f16: row b scaled by a power of two
// 2^e_b that takes its largest |x| into [2^14, 2^15), which is exact for every
// value not below 2^-14 after scaling (f16 has more mantissa bits than bf16);
// for INT4 the activations at k = 2, 3 (mod 4) are staged divided by 16,
// because the weights there come out of the nibble trick multiplied by 16.
// kNT n8 tiles of batch columns (B <= 8 kNT); only the B real rows are staged.
// kRing groups of ring per warp (kRing - 1 in flight).  kSplit == 2: the CTA
// takes the whole K for 4 slices, warps w and w + 4 one half of K each, and
// the halves are summed in shared memory -- y is written once, without
// atomics or a zeroing pass.
template <bool kW4, int kNT, int kRing, int kSplit = 1>
__global__ void __launch_bounds__(kGemvThreads) wgemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) uint8_t gsm[];
  constexpr int kSliceBytes = kW4 ? kW4SliceBytes : kW8SliceBytes;
  constexpr int kRingBytesPerWarp = kRing * kSliceBytes;
  constexpr int kVec = kSliceBytes / 512;                 // 16-byte words per lane per group
  constexpr int kSlicesPerCta = kGemvWarps / kSplit;
  static_assert(kRingBytesPerWarp >= 32 * 16 * kNT, "a warp's ring holds its lanes' partial sums");
  __shared__ float s_unscale[8 * kNT];                    // 2^-e_b per staged row
  // INT4 group scales of the CTA's rows, [row][group of the CTA's chunk]
  __shared__ __align__(16) uint16_t s_gscale[kW4 ? kGscaleEntries : 1];
  const int G = a.K / kGroupK;
  const int k0 = blockIdx.y * a.kc;
  const int kc = min(a.kc, a.K - k0);
  const int ng = kc / kGroupK;
  const int g0 = k0 / kGroupK;
  const int xstride = kc + kXPad;
  const int rows = min(a.B, 8 * kNT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wslot = warp % kSlicesPerCta;  // slice of the CTA
  const int khalf = warp / kSlicesPerCta;  // part of the CTA's K this warp takes
  const int slice = blockIdx.x * kSlicesPerCta + wslot;
  const bool has_slice = slice < a.N / 16;
  const int wng = ng / kSplit;             // this warp's groups
  const int wg0 = khalf * wng;             // its first group within the CTA's chunk
  uint16_t* xs = reinterpret_cast<uint16_t*>(gsm + kGemvWarps * kRingBytesPerWarp);
  // ---- this warp's weight stream starts first
  const uint8_t* wp =
      a.codes + (static_cast<int64_t>(has_slice ? slice : 0) * G + g0 + wg0) * kSliceBytes + 16 * lane;
  const uint32_t ring = smem_addr(gsm + warp * kRingBytesPerWarp) + 16 * lane;
  auto issue = [&](int gi) {
    if (has_slice && gi < wng) {
#pragma unroll
      for (int i = 0; i < kVec; ++i)
        cp_async16(ring + (gi % kRing) * kSliceBytes + 512 * i, wp + static_cast<int64_t>(gi) * kSliceBytes + 512 * i);
    }
    cp_async_commit();  // one group per step, empty or not: the wait counts stay uniform
  };
#pragma unroll
  for (int gi = 0; gi < kRing - 1; ++gi) issue(gi);
  // ---- the CTA's INT4 group scales for this chunk (ng per row).  A row's
  // run of scales starts on a 16-byte boundary when G, g0 and ng are
  // multiples of 8: then 8 at a time, every thread's loads issued before any
  // of its stores (one round trip); otherwise element by element.
  if (kW4) {
    const int total = kSlicesPerCta * 16 * ng;
    const int row_base = blockIdx.x * kSlicesPerCta * 16;
    if (G % 8 == 0 && g0 % 8 == 0 && ng % 8 == 0 && (reinterpret_cast<uintptr_t>(a.gscales) & 15u) == 0) {
      constexpr int kMaxV = kGscaleEntries / 8 / kGemvThreads;
      const int per_row = ng / 8;
      uint4 v[kMaxV];
#pragma unroll
      for (int u = 0; u < kMaxV; ++u) {
        const int i = threadIdx.x + u * kGemvThreads;
        const int rrow = i / per_row, q = i - rrow * per_row;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (i < total / 8 && row_base + rrow < a.N)
          v[u] = __ldg(reinterpret_cast<const uint4*>(a.gscales + static_cast<int64_t>(row_base + rrow) * G + g0) + q);
      }
#pragma unroll
      for (int u = 0; u < kMaxV; ++u) {
        const int i = threadIdx.x + u * kGemvThreads;
        if (i < total / 8) reinterpret_cast<uint4*>(s_gscale)[i] = v[u];
      }
    } else {
      for (int i = threadIdx.x; i < total; i += kGemvThreads) {
        const int rrow = i / ng, gi = i - rrow * ng;
        const int row = row_base + rrow;
        s_gscale[i] = row < a.N ? __ldg(a.gscales + static_cast<int64_t>(row) * G + g0 + gi) : 0;
      }
    }
  }
  // ---- stage the chunk's activations: items of 8 values, thread tid takes
  // items tid, tid + kGemvThreads, ... of each row.  A row's loads all go out
  // before any of them is used (one round trip); the raw bf16 go to their
  // place in shared memory while the row's largest |x| (bit patterns,
  // non-finite as 0) is taken per warp; after the block maximum every thread
  // turns its own items into the scaled f16 copy in place.
  __shared__ uint32_t s_wmax[8 * kNT][kGemvWarps];
  constexpr int kMaxItems = kWholeKMax / 8 / kGemvThreads;  // items per thread and row
  {
    uint32_t m2[8 * kNT];
#pragma unroll
    for (int b = 0; b < 8 * kNT; ++b) {
      m2[b] = 0u;
      if (b < rows) {
        const uint4* xrow = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(b) * a.K + k0);
        uint4 v[kMaxItems];
#pragma unroll
        for (int u = 0; u < kMaxItems; ++u) {
          const int item = threadIdx.x + u * kGemvThreads;
          v[u] = item < kc / 8 ? __ldg(xrow + item) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kMaxItems; ++u) {
          const int item = threadIdx.x + u * kGemvThreads;
          if (item < kc / 8) {
            *reinterpret_cast<uint4*>(xs + b * xstride + 8 * item) = v[u];
            const uint32_t ws[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t w2 = ws[q] & 0x7FFF7FFFu;
              w2 &= __vcmpltu2(w2, 0x7F807F80u);
              m2[b] = __vmaxu2(m2[b], w2);
            }
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < 8 * kNT; ++b) {
      if (b < rows) {
        const uint32_t mb = __reduce_max_sync(0xffffffffu, max(m2[b] & 0xFFFFu, m2[b] >> 16));
        if (lane == 0) s_wmax[b][warp] = mb;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int b = 0; b < 8 * kNT; ++b) {
    if (b < rows) {
      uint32_t mb = 0u;
#pragma unroll
      for (int w2 = 0; w2 < kGemvWarps; ++w2) mb = max(mb, s_wmax[b][w2]);
      const int e = mb == 0 ? 0 : min(max(14 - ilogbf(__uint_as_float(mb << 16)), -126), 126);
      const float sc = __int_as_float((127 + e) << 23);
      if (threadIdx.x == 0) s_unscale[b] = __int_as_float((127 - e) << 23);
#pragma unroll
      for (int u = 0; u < kMaxItems; ++u) {
        const int item = threadIdx.x + u * kGemvThreads;
        if (item < kc / 8) {
          const uint4 v = *reinterpret_cast<const uint4*>(xs + b * xstride + 8 * item);
          const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            // elements 8 item + 2q, + 1: k mod 4 = 2q mod 4, 2q mod 4 + 1
            const float f = (kW4 && (q & 1)) ? sc * 0.0625f : sc;
            o[q] = pack_f16x2(__uint_as_float(ws[q] << 16) * f, __uint_as_float(ws[q] & 0xFFFF0000u) * f);
          }
          *reinterpret_cast<uint4*>(xs + b * xstride + 8 * item) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
  __syncthreads();
  if (kSplit == 1 && !has_slice) {
    cp_async_wait<0>();
    return;
  }
  const int rr = lane >> 2, t = lane & 3;
  const int row0 = 16 * slice + rr, row1 = row0 + 8;
  const int lrow0 = 16 * wslot + rr, lrow1 = lrow0 + 8;  // rows within the CTA's scale table

  float acc[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  // batch column 8 nt + rr of the B operand; columns past B repeat the last
  // staged row: every output column of the MMA depends on its own B column
  // only, and the columns past B are never written out
  const uint16_t* xcol[kNT];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) xcol[nt] = xs + min(8 * nt + rr, rows - 1) * xstride + kGroupK * wg0 + 4 * t;
  // nibble masks, the f16 magic 1024 and the biases, in registers
  const uint32_t mlo = 0x000F000Fu, mhi = 0x00F000F0u, magic = 0x64006400u;
  const uint32_t blo = 0x64086408u, bhi = 0x64806480u;  // 1032, 1152
  const uint16_t* gsc0 = &s_gscale[kW4 ? lrow0 * ng + wg0 : 0];
  const uint16_t* gsc1 = &s_gscale[kW4 ? lrow1 * ng + wg0 : 0];

  // ring bookkeeping by running offsets: group gi is read from slot rd; the
  // group kRing - 1 ahead is written into the slot the previous group left
  // (whose words are in registers by now)
  const uint8_t* ring_ld = gsm + warp * kRingBytesPerWarp + 16 * lane;
  const uint8_t* gsrc = wp + static_cast<int64_t>(kRing - 1) * kSliceBytes;
  uint32_t rd = 0, wr = (kRing - 1) * kSliceBytes;
  for (int gi = 0; gi < (has_slice ? wng : 0); ++gi) {
    cp_async_wait<kRing - 2>();  // group gi has landed (this lane's words)
    uint4 cur[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) cur[i] = *reinterpret_cast<const uint4*>(ring_ld + rd + 512 * i);
    if (gi + kRing - 1 < wng) {
#pragma unroll
      for (int i = 0; i < kVec; ++i) cp_async16(ring + wr + 512 * i, gsrc + 512 * i);
    }
    cp_async_commit();
    gsrc += kSliceBytes;
    wr = rd;
    rd = rd + kSliceBytes == kRingBytesPerWarp ? 0u : rd + kSliceBytes;
    // two accumulator chains per group (even and odd steps)
    float ae[kNT][4], ao[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      ae[nt][0] = ae[nt][1] = ae[nt][2] = ae[nt][3] = 0.f;
      ao[nt][0] = ao[nt][1] = ao[nt][2] = ao[nt][3] = 0.f;
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t af[4];
      if (kW4) {
        // cur[0]: row0's words, cur[1]: row1's; word s/2; odd steps use the
        // nibbles 8 bits up
        const uint32_t v0 = s < 2 ? cur[0].x : s < 4 ? cur[0].y : s < 6 ? cur[0].z : cur[0].w;
        const uint32_t v1 = s < 2 ? cur[1].x : s < 4 ? cur[1].y : s < 6 ? cur[1].z : cur[1].w;
        const uint32_t u0 = (s & 1) ? v0 >> 8 : v0;
        const uint32_t u1 = (s & 1) ? v1 >> 8 : v1;
        af[0] = w4_pair_to_f16x2(u0, mlo, magic, blo);  // row0, j0 j1: n - 8
        af[1] = w4_pair_to_f16x2(u1, mlo, magic, blo);  // row1, j0 j1
        af[2] = w4_pair_to_f16x2(u0, mhi, magic, bhi);  // row0, j2 j3: 16 (n - 8)
        af[3] = w4_pair_to_f16x2(u1, mhi, magic, bhi);  // row1, j2 j3
      } else {
        // cur[0], cur[1]: row0 steps 0-3, 4-7; cur[2], cur[3]: row1; word = step
        const uint4& r0 = cur[s >> 2];
        const uint4& r1 = cur[2 + (s >> 2)];
        const uint32_t c0 = (s & 3) == 0 ? r0.x : (s & 3) == 1 ? r0.y : (s & 3) == 2 ? r0.z : r0.w;
        const uint32_t c1 = (s & 3) == 0 ? r1.x : (s & 3) == 1 ? r1.y : (s & 3) == 2 ? r1.z : r1.w;
        af[0] = e4m3x2_to_f16x2(static_cast<uint16_t>(c0 & 0xFFFFu));
        af[1] = e4m3x2_to_f16x2(static_cast<uint16_t>(c1 & 0xFFFFu));
        af[2] = e4m3x2_to_f16x2(static_cast<uint16_t>(c0 >> 16));
        af[3] = e4m3x2_to_f16x2(static_cast<uint16_t>(c1 >> 16));
      }
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const uint2 bv = *reinterpret_cast<const uint2*>(xcol[nt] + kGroupK * gi + 16 * s);
        if (s & 1) mma_f16(ao[nt], af, bv.x, bv.y);
        else mma_f16(ae[nt], af, bv.x, bv.y);
      }
    }
    if (kW4) {
      const float s0 = bf16_bits_to_float(gsc0[gi]);
      const float s1 = bf16_bits_to_float(gsc1[gi]);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        acc[nt][0] = fmaf(ae[nt][0] + ao[nt][0], s0, acc[nt][0]);
        acc[nt][1] = fmaf(ae[nt][1] + ao[nt][1], s0, acc[nt][1]);
        acc[nt][2] = fmaf(ae[nt][2] + ao[nt][2], s1, acc[nt][2]);
        acc[nt][3] = fmaf(ae[nt][3] + ao[nt][3], s1, acc[nt][3]);
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] += ae[nt][e] + ao[nt][e];
    }
  }
  cp_async_wait<0>();
  if (kSplit == 2) {
    // the second half's sums go through its warp's ring (every copy of it
    // has landed and been read); the first half adds them
    float* part = reinterpret_cast<float*>(gsm + (wslot + kSlicesPerCta) * kRingBytesPerWarp) + 4 * kNT * lane;
    if (khalf == 1) {
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
        *reinterpret_cast<float4*>(part + 4 * nt) = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    }
    __syncthreads();
    if (khalf == 1 || !has_slice) return;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const float4 o = *reinterpret_cast<const float4*>(part + 4 * nt);
      acc[nt][0] += o.x;
      acc[nt][1] += o.y;
      acc[nt][2] += o.z;
      acc[nt][3] += o.w;
    }
  }
  float r0s = 1.f, r1s = 1.f;
  if (!kW4) {
    r0s = __ldg(a.rscales + row0);
    r1s = __ldg(a.rscales + row1);
  }
  // accumulator (row, column): c0 (row0, 2t), c1 (row0, 2t+1), c2 (row1, 2t), c3 (row1, 2t+1)
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int b = 8 * nt + 2 * t + (e & 1);
      const int row = e < 2 ? row0 : row1;
      if (b < a.B) {
        float* yp = a.y + static_cast<int64_t>(b) * a.N + row;
        const float v = acc[nt][e] * (e < 2 ? r0s : r1s) * s_unscale[b];
        if (a.atomic) atomicAdd(yp, v);
        else *yp = v;
      }
    }
  }
}

// bf16x2 of two excess-8 nibbles (bits 0..3 and 16..19 of v): 128 + nibble is
// exact in bf16 (one unit in the last place at 128), so subtracting 136 gives
// the signed code exactly.
__device__ __forceinline__ uint32_t w4_pair_to_bf16x2(uint32_t v) {
  const uint32_t b = (v & 0x000F000Fu) | 0x43004300u;
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&b),
                                   __floats2bfloat162_rn(136.f, 136.f));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// bf16x2 of two e4m3 codes (bits 0..7 and 8..15), exactly: e4m3 -> f16 -> f32 -> bf16.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t c) {
  const uint32_t h = e4m3x2_to_f16x2(static_cast<uint16_t>(c & 0xFFFFu));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  return pack_bf16x2(f.x, f.y);
}

// Register-streaming variant for batches of 5..16 tokens, where the staged
// activations leave too little shared memory for the landing rings: one CTA
// of 8 warps x one 16-row slice each over one K chunk of kKChunk, kPF groups
// of weights in flight per lane in registers, activations staged as the bf16
// values they are (8 kNT rows, zeros past B), bf16 weights from the nibbles.
// kNT n8 tiles of batch columns (B <= 8 * kNT).
template <bool kW4, int kNT>
__global__ void __launch_bounds__(kGemvThreads) wgemv_regs_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) uint16_t xs[];  // [8 * kNT][kc + kXPad]
  constexpr int kSliceBytes = kW4 ? kW4SliceBytes : kW8SliceBytes;
  constexpr int kVec = kW4 ? 2 : 4;  // 16-byte words per lane per group
  constexpr int kPF = kW4 ? 4 : 2;
  const int G = a.K / kGroupK;
  const int k0 = blockIdx.y * a.kc;
  const int kc = min(a.kc, a.K - k0);
  const int ng = kc / kGroupK;
  const int xstride = kc + kXPad;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = blockIdx.x * kGemvWarps + warp;
  const bool has_slice = slice < a.N / 16;
  const int rr = lane >> 2, t = lane & 3;
  const int g0 = k0 / kGroupK;
  const uint8_t* wp = a.codes + (static_cast<int64_t>(has_slice ? slice : 0) * G + g0) * kSliceBytes + 16 * lane;
  const int row0 = 16 * slice + rr, row1 = row0 + 8;
  auto load_group = [&](int gi, uint4 (&v)[kVec]) {
#pragma unroll
    for (int i = 0; i < kVec; ++i)
      v[i] = has_slice && gi < ng
                 ? __ldcs(reinterpret_cast<const uint4*>(wp + static_cast<int64_t>(gi) * kSliceBytes + 512 * i))
                 : make_uint4(0u, 0u, 0u, 0u);
  };
  // ---- INT4: the first weight groups start streaming, then the activations
  // of this chunk are staged (rows past B are zero), 4 of a thread's items at
  // a time with their loads all issued before any store (the host uses this
  // kernel with chunks of at most kKChunk, which the batches cover; a loop
  // takes any rest).  e4m3 stages first and then starts its weights: the
  // order measured faster for each (INT4 at 5-8 tokens 42 against 44 us;
  // e4m3 52 against 54 us).
  uint4 buf[kPF][kVec];
  auto item_src = [&](int i, int items, uint4& v) {
    const int b = i / (kc / 8), c = i - b * (kc / 8);
    v = make_uint4(0u, 0u, 0u, 0u);
    if (i < items && b < a.B) v = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(b) * a.K + k0) + c);
  };
  auto item_dst = [&](int i, int items, const uint4& v) {
    const int b = i / (kc / 8), c = i - b * (kc / 8);
    if (i < items) *reinterpret_cast<uint4*>(xs + b * xstride + 8 * c) = v;
  };
  const int items = 8 * kNT * (kc / 8);
  if constexpr (kW4) {
#pragma unroll
    for (int u = 0; u < kPF; ++u) load_group(u, buf[u]);
    constexpr int kBatchItems = 4;
    constexpr int kCovered = 8 * kNT * (kKChunk / 8);
#pragma unroll 1
    for (int i0 = threadIdx.x; i0 < kCovered; i0 += kBatchItems * kGemvThreads) {
      uint4 v[kBatchItems];
#pragma unroll
      for (int u = 0; u < kBatchItems; ++u) item_src(i0 + u * kGemvThreads, items, v[u]);
#pragma unroll
      for (int u = 0; u < kBatchItems; ++u) item_dst(i0 + u * kGemvThreads, items, v[u]);
    }
    for (int i = kCovered + threadIdx.x; i < items; i += kGemvThreads) {
      uint4 v;
      item_src(i, items, v);
      item_dst(i, items, v);
    }
  } else {
    for (int i = threadIdx.x; i < items; i += kGemvThreads) {
      uint4 v;
      item_src(i, items, v);
      item_dst(i, items, v);
    }
  }
  __syncthreads();
  if (!has_slice) return;
  if constexpr (!kW4) {
#pragma unroll
    for (int u = 0; u < kPF; ++u) load_group(u, buf[u]);
  }

  float acc[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  for (int gb = 0; gb < ng; gb += kPF) {
#pragma unroll
    for (int u = 0; u < kPF; ++u) {
      const int gi = gb + u;
      if (gi >= ng) break;
      uint4 cur[kVec];
#pragma unroll
      for (int i = 0; i < kVec; ++i) cur[i] = buf[u][i];
      load_group(gi + kPF, buf[u]);  // the group kPF ahead, into the slot just freed
      const uint16_t* xg = xs + kGroupK * gi + 4 * t;
      float accg[kNT][4];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) accg[nt][0] = accg[nt][1] = accg[nt][2] = accg[nt][3] = 0.f;
      float (&dst)[kNT][4] = kW4 ? accg : acc;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        uint32_t af[4];
        if (kW4) {
          // cur[0]: row0's words, cur[1]: row1's; word s/2, nibble pairs at shift 8*(s&1) (+4)
          const uint32_t w0 = s < 2 ? cur[0].x : s < 4 ? cur[0].y : s < 6 ? cur[0].z : cur[0].w;
          const uint32_t w1 = s < 2 ? cur[1].x : s < 4 ? cur[1].y : s < 6 ? cur[1].z : cur[1].w;
          const int sh = 8 * (s & 1);
          af[0] = w4_pair_to_bf16x2(w0 >> sh);        // row0, j0 j1
          af[1] = w4_pair_to_bf16x2(w1 >> sh);        // row1, j0 j1
          af[2] = w4_pair_to_bf16x2(w0 >> (sh + 4));  // row0, j2 j3
          af[3] = w4_pair_to_bf16x2(w1 >> (sh + 4));  // row1, j2 j3
        } else {
          // cur[0], cur[1]: row0 steps 0-3, 4-7; cur[2], cur[3]: row1; word = step
          const uint4& r0 = cur[s >> 2];
          const uint4& r1 = cur[2 + (s >> 2)];
          const uint32_t c0 = (s & 3) == 0 ? r0.x : (s & 3) == 1 ? r0.y : (s & 3) == 2 ? r0.z : r0.w;
          const uint32_t c1 = (s & 3) == 0 ? r1.x : (s & 3) == 1 ? r1.y : (s & 3) == 2 ? r1.z : r1.w;
          af[0] = e4m3x2_to_bf16x2(c0);
          af[1] = e4m3x2_to_bf16x2(c1);
          af[2] = e4m3x2_to_bf16x2(c0 >> 16);
          af[3] = e4m3x2_to_bf16x2(c1 >> 16);
        }
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const uint2 bv = *reinterpret_cast<const uint2*>(xg + (8 * nt + rr) * xstride + 16 * s);
          mma_bf16(dst[nt], af, bv.x, bv.y);
        }
      }
      if (kW4) {
        const float s0 = bf16_bits_to_float(__ldg(a.gscales + static_cast<int64_t>(row0) * G + g0 + gi));
        const float s1 = bf16_bits_to_float(__ldg(a.gscales + static_cast<int64_t>(row1) * G + g0 + gi));
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          acc[nt][0] = fmaf(accg[nt][0], s0, acc[nt][0]);
          acc[nt][1] = fmaf(accg[nt][1], s0, acc[nt][1]);
          acc[nt][2] = fmaf(accg[nt][2], s1, acc[nt][2]);
          acc[nt][3] = fmaf(accg[nt][3], s1, acc[nt][3]);
        }
      }
    }
  }
  float r0s = 1.f, r1s = 1.f;
  if (!kW4) {
    r0s = __ldg(a.rscales + row0);
    r1s = __ldg(a.rscales + row1);
  }
  // accumulator (row, column): c0 (row0, 2t), c1 (row0, 2t+1), c2 (row1, 2t), c3 (row1, 2t+1)
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int b = 8 * nt + 2 * t + (e & 1);
      const int row = e < 2 ? row0 : row1;
      if (b < a.B) {
        float* yp = a.y + static_cast<int64_t>(b) * a.N + row;
        const float v = acc[nt][e] * (e < 2 ? r0s : r1s);
        if (a.atomic) atomicAdd(yp, v);
        else *yp = v;
      }
    }
  }
}

int check_w_shapes(int N, int K) {
  if (N < 0 || K < 0) return FPK_EINVAL;
  if (N % 16 != 0 || K % kGroupK != 0) return FPK_EUNSUPPORTED;
  return FPK_OK;
}

template <bool kW4>
int gemv_entry(const void* x, const uint8_t* codes, const void* gscales, const float* rscales, float* y,
               int32_t B, int32_t N, int32_t K, void* stream) {
  int st = check_w_shapes(N, K);
  if (st != FPK_OK) return st;
  if (B < 0) return FPK_EINVAL;
  if (B > 16) return FPK_EUNSUPPORTED;
  if (B == 0 || N == 0) return FPK_OK;
  if (!x || !codes || !y || (kW4 ? !gscales : !rscales)) return FPK_EINVAL;
  if (!aligned16(x) || !aligned16(codes)) return FPK_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return cudaMemsetAsync(y, 0, sizeof(float) * B * static_cast<size_t>(N), s) == cudaSuccess ? FPK_OK : FPK_ECUDA;
  GemvArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.codes = codes;
  a.gscales = static_cast<const uint16_t*>(gscales);
  a.rscales = rscales;
  a.y = y;
  a.B = B;
  a.N = N;
  a.K = K;
  // Kernel and ring depth by batch: in the landing-ring kernel the staged
  // activations (B rows of f16) and the rings share the shared memory,
  // three CTAs (24 warps) per SM at 1 and 3-4 tokens, two at 2; beyond 4
  // tokens too little is left for the rings, and the register-streaming
  // kernel is faster.  (Smaller K chunks to keep three CTAs were measured
  // slower: each CTA's staging and ring fill then cover too few groups; so
  // was summing the K chunks of a row block in a thread-block cluster instead
  // of atomics into a zeroed y: 41.0 against 36.8 us at one token.)
  // INT4 at one token with K up to 8192: one CTA per 4 slices over the
  // whole K, the two halves of K summed in the CTA -- no split-K atomics,
  // hence no zeroing of y before the kernel (a second launch per call)
  const bool whole_k = kW4 && B == 1 && K % (2 * kGroupK) == 0 && K <= kWholeKMax;
  // INT4 at two tokens: chunks of 2 kKChunk, one wave of CTAs at three per SM
  // (measured at 28672 x 8192: 34.8 us against 44.0 with kKChunk)
  const int chunk = whole_k ? K : kW4 && B == 2 ? 2 * kKChunk : kKChunk;
  const int kc = K < chunk ? K : chunk;
  a.kc = kc;
  const int chunks = (K + kc - 1) / kc;
  a.atomic = chunks > 1;
  if (a.atomic && cudaMemsetAsync(y, 0, sizeof(float) * B * static_cast<size_t>(N), s) != cudaSuccess)
    return FPK_ECUDA;
  const int nt = B <= 8 ? 1 : 2;
  const int slices_per_cta = whole_k ? kGemvWarps / 2 : kGemvWarps;
  const dim3 grid((N / 16 + slices_per_cta - 1) / slices_per_cta, chunks);
  if (B > 4) {
    // 5..16 tokens: the register-streaming kernel (measured faster there:
    // INT4 at 28672 x 8192, 8 tokens 43 against 50 us, 16 tokens 53 against 72 us)
    const size_t rsm = static_cast<size_t>(8 * nt) * (kc + kXPad) * sizeof(uint16_t);
    void (*rk)(GemvArgs) = nt == 1 ? wgemv_regs_kernel<kW4, 1> : wgemv_regs_kernel<kW4, 2>;
    if (rsm > 48 * 1024 &&
        cudaFuncSetAttribute(rk, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(rsm)) != cudaSuccess)
      return FPK_ECUDA;
    rk<<<grid, kGemvThreads, rsm, s>>>(a);
    return checked_launch_status();
  }
  // 1..4 tokens: the landing-ring kernel; ring groups per warp -- INT4 6
  // (three CTAs per SM), e4m3 4 or 3
  const int ring = kW4 ? 6 : (B <= 2 ? 4 : 3);
  const size_t smem = static_cast<size_t>(kGemvWarps) * ring * (kW4 ? kW4SliceBytes : kW8SliceBytes) +
                      static_cast<size_t>(B) * (kc + kXPad) * sizeof(uint16_t);
  void (*kern)(GemvArgs);
  if constexpr (kW4) kern = whole_k ? wgemv_kernel<true, 1, 6, 2> : wgemv_kernel<true, 1, 6>;
  else kern = B <= 2 ? wgemv_kernel<false, 1, 4> : wgemv_kernel<false, 1, 3>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return FPK_ECUDA;
  kern<<<grid, kGemvThreads, smem, s>>>(a);
  return checked_launch_status();
}

}  // namespace
}  // namespace fpk

extern "C" int fpk_w4_quantize(const void* w, uint8_t* codes, void* scales, int32_t N, int32_t K,
                               void* stream) {
  int st = fpk::check_w_shapes(N, K);
  if (st != FPK_OK) return st;
  if (N == 0 || K == 0) return FPK_OK;
  if (!w || !codes || !scales) return FPK_EINVAL;
  if (!fpk::aligned16(codes) || (reinterpret_cast<uintptr_t>(w) & 7u) != 0) return FPK_EINVAL;
  const int64_t units = static_cast<int64_t>(N / 16) * (K / fpk::kGroupK);
  fpk::w4_quantize_kernel<<<static_cast<unsigned>((units + 7) / 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(w), codes, static_cast<uint16_t*>(scales), N, K);
  return fpk::checked_launch_status();
}

extern "C" int fpk_w8_quantize(const void* w, uint8_t* codes, float* row_scales, int32_t N, int32_t K,
                               void* stream) {
  int st = fpk::check_w_shapes(N, K);
  if (st != FPK_OK) return st;
  if (N == 0 || K == 0) return FPK_OK;
  if (!w || !codes || !row_scales) return FPK_EINVAL;
  if (!fpk::aligned16(codes) || !fpk::aligned16(w)) return FPK_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fpk::w8_row_scale_kernel<<<(N + 7) / 8, 256, 0, s>>>(static_cast<const uint16_t*>(w), row_scales, N, K);
  const int64_t units = static_cast<int64_t>(N / 16) * (K / fpk::kGroupK);
  fpk::w8_quantize_kernel<<<static_cast<unsigned>((units + 7) / 8), 256, 0, s>>>(
      static_cast<const uint16_t*>(w), row_scales, codes, N, K);
  return fpk::checked_launch_status();
}

extern "C" int fpk_w4_gemv(const void* x, const uint8_t* codes, const void* scales, float* y, int32_t B,
                           int32_t N, int32_t K, void* stream) {
  return fpk::gemv_entry<true>(x, codes, scales, nullptr, y, B, N, K, stream);
}

extern "C" int fpk_w8_gemv(const void* x, const uint8_t* codes, const float* row_scales, float* y, int32_t B,
                           int32_t N, int32_t K, void* stream) {
  return fpk::gemv_entry<false>(x, codes, nullptr, row_scales, y, B, N, K, stream);
}
