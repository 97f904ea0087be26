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
  int atomic;               // several K chunks add into y
};

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

// One CTA: 8 warps x one 16-row slice each, over one K chunk.  kNT n8 tiles of
// batch columns (B <= 8 * kNT).  kPF groups of weights are in flight per lane.
template <bool kW4, int kNT>
__global__ void __launch_bounds__(kGemvThreads) wgemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) uint16_t xs[];  // [8 * kNT][kc + kXPad]
  constexpr int kSliceBytes = kW4 ? kW4SliceBytes : kW8SliceBytes;
  constexpr int kVec = kW4 ? 2 : 4;  // 16-byte words per lane per group
  constexpr int kPF = kW4 ? 4 : 2;
  const int G = a.K / kGroupK;
  const int k0 = blockIdx.y * kKChunk;
  const int kc = min(kKChunk, a.K - k0);
  const int ng = kc / kGroupK;
  const int xstride = kc + kXPad;
  // ---- stage the activations of this chunk (rows past B are zero)
  for (int i = threadIdx.x; i < 8 * kNT * (kc / 8); i += kGemvThreads) {
    const int b = i / (kc / 8), c = i - b * (kc / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (b < a.B) v = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(b) * a.K + k0) + c);
    *reinterpret_cast<uint4*>(xs + b * xstride + 8 * c) = v;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = blockIdx.x * kGemvWarps + warp;
  if (slice >= a.N / 16) return;
  const int rr = lane >> 2, t = lane & 3;
  const int g0 = k0 / kGroupK;
  const uint8_t* wp = a.codes + (static_cast<int64_t>(slice) * G + g0) * kSliceBytes + 16 * lane;
  const int row0 = 16 * slice + rr, row1 = row0 + 8;

  float acc[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  auto load_group = [&](int gi, uint4 (&v)[kVec]) {
#pragma unroll
    for (int i = 0; i < kVec; ++i)
      v[i] = gi < ng ? __ldcs(reinterpret_cast<const uint4*>(wp + static_cast<int64_t>(gi) * kSliceBytes + 512 * i))
                     : make_uint4(0u, 0u, 0u, 0u);
  };
  uint4 buf[kPF][kVec];
#pragma unroll
  for (int u = 0; u < kPF; ++u) load_group(u, buf[u]);

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
  const int chunks = (K + kKChunk - 1) / kKChunk;
  a.atomic = chunks > 1;
  if (a.atomic && cudaMemsetAsync(y, 0, sizeof(float) * B * static_cast<size_t>(N), s) != cudaSuccess)
    return FPK_ECUDA;
  const int nt = B <= 8 ? 1 : 2;
  const int kc = K < kKChunk ? K : kKChunk;
  const size_t smem = static_cast<size_t>(8 * nt) * (kc + kXPad) * sizeof(uint16_t);
  const dim3 grid((N / 16 + kGemvWarps - 1) / kGemvWarps, chunks);
  auto kern = nt == 1 ? wgemv_kernel<kW4, 1> : wgemv_kernel<kW4, 2>;
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
