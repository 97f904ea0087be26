// decode_attn_tc.cu -- split-KV paged decode attention over the FP8 e4m3 cache
// on the fifth-generation tensor cores: tcgen05.mma of kind f8f6f4 reading the
// e4m3 K and V tiles straight from shared memory, with its accumulators in
// tensor memory (TMEM).
//
// What it computes is the same as fpk_paged_decode_attn_fp8 (decode_attn.cu):
// the decode pool's attention reads the FP8 e4m3 cache and converts it as it
// reads ("Perche le cache piu piccole di Cloudflare battono la velocita pura",
// remio.ai), pages are reached through each request's page table, requests
// that failed the tag check read nothing ("La sicurezza della cache KV
// condivisa...").  The pages give no kernel design; this variant is built for
// the sm_103a tensor cores:
//
// * Operands.  A block of 8 tiles (128 tokens) of one (request, kv head) is one
//   MMA tile: S^T = K Q^T with M = 128 tokens, and O^T = V^T P^T with M = 128
//   dims.  K rows land through a tensor-map copy (cp.async.bulk.tensor) with
//   the 128-byte swizzle, which is the canonical K-major layout of an e4m3
//   operand with 128-byte rows; the V block of a tile ([128 dims][16 tokens])
//   is already the canonical K-major core-matrix layout and lands by a plain
//   bulk copy.  No e4m3 code of the cache is converted or rewritten by a
//   thread.
// * Precision.  The tensor cores take both operands of one MMA in the same
//   format, so the query and the softmax weights enter as e4m3 too, each split
//   into four e4m3 parts x = c0 + c1/16 + c2/256 + c3/4096 (every part rounds
//   the remainder of the ones before it): the four parts of the 8 heads of a
//   GQA group are the N = 32 columns of both MMAs, and the part sums are
//   recombined in fp32 when the accumulators are read.  Four parts carry 16
//   significant bits, more than the f16 the warp-level kernel uses.
// * Pipeline (one CTA per SM).  Producer warps 0 and 1 take alternate blocks
//   and land each block's K rows in a 4-slot K ring (tensor-map copies) and
//   its V blocks in an 8-slot V ring (bulk copies), one mbarrier per slot: a
//   K slot is free once the block's S^T has been computed, a V slot once its
//   O^T has.  Warp 2 owns the tensor memory (S double-buffered, O in four
//   buffers, 256 columns) and one of its threads issues the MMAs and commits
//   them to mbarriers.  Warps 3-18 are two groups of 8 that take alternate
//   blocks, each with its own running (m, l, O) merged at the end of every
//   piece; within a group two warps share each TMEM lane quarter, one for
//   heads 0-3 and one for heads 4-7: a thread per (token, four heads) runs the
//   online softmax in the log2 domain and writes the e4m3 parts of P, a thread
//   per (dim, four heads) folds each block's O into registers with the
//   running rescale.
// * Work split and combine: the partition of attn_plan.cuh (equal tile-count
//   splits over the segment list; with the automatic count, a uniform batch
//   takes one whole segment per CTA or equal splits per segment).  A split
//   piece writes its partial and takes an arrival ticket; the arrival that
//   completes a segment merges its partials by log-sum-exp.  Nothing waits on
//   another CTA.
// * Safety.  Every mbarrier wait is bounded (status word); TMEM is freed on
//   every path once the MMAs in flight have completed.
#include <atomic>
#include <mutex>

#include <cuda.h>  // CUtensorMap and the tensor-map encoder's types (entry point fetched at run time)

#include "attn_plan.cuh"
#include "common.cuh"

namespace fpk {
namespace {

constexpr int kBlkTiles = 8;                         // tiles per MMA block
constexpr int kParts = 4;                            // e4m3 parts of q and p
constexpr int kTcN = kParts * kGroupMax;             // MMA N: 32 columns
constexpr int kHalfHeads = kGroupMax / 2;            // heads of one consumer warpgroup
// The K rows and the V blocks of a block land in two rings: a K slot is free
// again once the block's S^T = K Q^T has run, a V slot only once O^T = V^T P^T
// has (after the softmax), so the V ring is the deeper one.
constexpr int kStagesK = 4;
constexpr int kStagesV = 8;
constexpr int kSlotBytes = kBlkTiles * kTile * kDim;  // K rows (or V blocks) of a block: 16 KiB
constexpr int kOBufs = 4;                             // O accumulators in TMEM
constexpr int kTcQBytes = kTcN * kDim;               // [32 rows][128 B], 128-byte swizzle
constexpr int kTcPBytes = kTcN * kBlkTiles * kTile;  // [128 tokens] x [32 columns]
constexpr int kConsWarps = 16;  // two groups of 8, alternate blocks
constexpr int kProdWarps = 2;             // copy issue, alternate blocks
constexpr int kMmaWarp = kProdWarps;      // TMEM owner and MMA issue
constexpr int kTcWarps = kProdWarps + 1 + kConsWarps;
constexpr int kTcThreads = 32 * kTcWarps;
constexpr int kTmemCols = 256;  // S[0..1], O[0..3]: 32 columns each
constexpr float kTcLn2 = 0.6931471805599453f;
constexpr float kTcLog2e = 1.4426950408889634f;

// MMA column of part k of head h: the 16 columns of heads 0-3 first, then
// those of heads 4-7, so that each consumer warpgroup reads one contiguous run
__host__ __device__ constexpr int col_of(int k, int h) { return 16 * (h >> 2) + 4 * k + (h & 3); }

// barriers (8 bytes each)
constexpr int kBarFullK = 0;                        // [kStagesK] K slot landed (TMA)
constexpr int kBarEmptyK = kBarFullK + kStagesK;    // [kStagesK] K slot read (MMA commit)
constexpr int kBarFullV = kBarEmptyK + kStagesK;    // [kStagesV] V slot landed (TMA)
constexpr int kBarEmptyV = kBarFullV + kStagesV;    // [kStagesV] V slot read (MMA commit)
constexpr int kBarSFull = kBarEmptyV + kStagesV;    // [2] S ready (MMA commit)
constexpr int kBarSFree = kBarSFull + 2;          // [2] S read (consumer warps)
constexpr int kBarPFull = kBarSFree + 2;          // [2] P written (consumer warps)
constexpr int kBarOFull = kBarPFull + 2;          // [kOBufs] O block ready (MMA commit)
constexpr int kBarOFree = kBarOFull + kOBufs;     // [kOBufs] O block read (consumer warps)
constexpr int kBarQFull = kBarOFree + kOBufs;     // query parts written (consumer warps)
constexpr int kBarCons = kBarQFull + 1;           // [2] barrier of one consumer group
constexpr int kBarConsAll = kBarCons + 2;         // barrier of both consumer groups
constexpr int kBarDone = kBarConsAll + 1;         // every MMA of the CTA completed
constexpr int kNumBars = kBarDone + 1;

// shared-memory map, from a 1024-byte aligned base
constexpr int kOffV = kStagesK * kSlotBytes;
constexpr int kOffQ = kOffV + kStagesV * kSlotBytes;
constexpr int kOffP = kOffQ + kTcQBytes;
constexpr int kOffX = kOffP + 2 * kTcPBytes;                // group 1's (O, m, l) at the end of a piece
// block maxima [group][block pair parity][lane quarter][head], then the
// sums of l [group][lane quarter][head]
constexpr int kOffRed = kOffX + (kGroupMax * kDim + 2 * kGroupMax) * 4;
constexpr int kRedSums = 2 * 2 * 4 * kGroupMax;
constexpr int kOffMult = kOffRed + (kRedSums + 2 * 4 * kGroupMax) * 4;  // float [8] score multipliers
// uint32 [kStagesV] bad tiles of each block in a V slot; [2][16] warp faults by piece parity
constexpr int kOffFault = kOffMult + kGroupMax * 4;
constexpr int kOffBars = (kOffFault + (kStagesV + 2 * kConsWarps) * 4 + 7) / 8 * 8;
constexpr int kOffMisc = kOffBars + kNumBars * 8;  // TMEM base, s_last, start
constexpr int kOffScan = kOffMisc + 32;            // int64 [warps] sums, int [warps][3] nz/min/max
constexpr int kTcSmemUsed = kOffScan + kTcWarps * 8 + kTcWarps * 3 * 4;
constexpr int kTcSmemBytes = kTcSmemUsed + 1024;  // room to align the base
static_assert(kOffQ % 1024 == 0, "swizzled operands need 1024-byte alignment");

struct TcArgs {
  const uint16_t* q;
  const uint8_t* kv_pool;
  const float* k_scale;
  const float* v_scale;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const uint8_t* abort_mask;
  float* out;
  float* lse;
  uint32_t* status;
  int* seg_count;  // per-segment arrival tickets, zero between calls
  float2* part_ml;
  float* part_o;
  int B, Hq, Hkv, G, page_size, num_pages, max_pages, W;
  int auto_split;
  float sm_scale_log2;
};

// ---------------------------------------------------------------------------
// tcgen05 / tensor-map PTX
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Shared-memory matrix descriptor: start, leading- and stride-dimension byte
// offsets (16-byte units), descriptor version 1, layout (0: no swizzle, 2:
// 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(layout) << 61);
}

// Instruction descriptor of kind::f8f6f4: E4M3 x E4M3 -> F32, both operands
// K-major, M = 128, N = 32.
constexpr uint32_t kIdesc = (1u << 4)                // D format F32
                            | (0u << 7) | (0u << 10)  // A, B format E4M3
                            | (static_cast<uint32_t>(kTcN >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(acc)
      : "memory");
}

// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane (the warp's lane
// quarter), waited for inside the same asm block.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two fp32 to two e4m3 codes (lo in the low byte), nearest-even, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The values of two e4m3 codes (low byte first).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t codes) {
  const uint32_t h = e4m3x2_to_f16x2(static_cast<uint16_t>(codes));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Reductions of four per-lane values over the 32 lanes of a warp: lane l
// ends with the result for value (l >> 3) & 3 (6 shuffles instead of 20).
template <bool kMax>
__device__ __forceinline__ float warp_reduce4(const float (&v)[4], int lane) {
  const unsigned kFull = 0xffffffffu;
  auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : x + y; };
  const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1;
  float w[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b4 ? v[i] : v[i + 2], keep = b4 ? v[i + 2] : v[i];
    w[i] = op(keep, __shfl_xor_sync(kFull, send, 16));
  }
  const float send = b3 ? w[0] : w[1], keep = b3 ? w[1] : w[0];
  float y = op(keep, __shfl_xor_sync(kFull, send, 8));
  y = op(y, __shfl_xor_sync(kFull, y, 4));
  y = op(y, __shfl_xor_sync(kFull, y, 2));
  return op(y, __shfl_xor_sync(kFull, y, 1));
}

// Part sums of head i of a warpgroup from its 16 accumulator columns
// (column 4 k + i holds part k): 4096 (c0 + c1/16 + c2/256 + c3/4096) by
// Horner's rule.
__device__ __forceinline__ float part_sum(const float (&v)[16], int i) {
  return fmaf(fmaf(fmaf(v[i], 16.f, v[4 + i]), 16.f, v[8 + i]), 16.f, v[12 + i]);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    paged_decode_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap kmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* const sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_addr(sm);
  float* const s_red = reinterpret_cast<float*>(sm + kOffRed);  // block maxima, then sums of l
  float* const s_mult = reinterpret_cast<float*>(sm + kOffMult);
  uint32_t* const s_fault = reinterpret_cast<uint32_t*>(sm + kOffFault);
  uint32_t* const s_wfault = s_fault + kStagesV;
  uint32_t* const s_tmem = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  int* const s_last = reinterpret_cast<int*>(sm + kOffMisc + 4);
  int* const s_start = reinterpret_cast<int*>(sm + kOffMisc + 8);  // r, h, t, n
  int64_t* const s_wsum = reinterpret_cast<int64_t*>(sm + kOffScan);
  int* const s_wstat = reinterpret_cast<int*>(sm + kOffScan + kTcWarps * 8);  // [warps][3] nz, min, max
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBars + 8 * i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int w = blockIdx.x;
  const int nctas = static_cast<int>(gridDim.x);
  const unsigned kFull = 0xffffffffu;

  // ---- prologue: total tiles and this CTA's start (block scan over requests)
  const int chunk = (a.B + kTcThreads - 1) / kTcThreads;
  const int rb = tid * chunk;
  const int re = min(a.B, rb + chunk);
  int64_t mine = 0;
  int nz = 0, tmin = 0x7fffffff, tmax = 0;
  for (int r = rb; r < re; ++r) {
    const int n = tiles_of(a, r);
    mine += n;
    if (n > 0) {
      ++nz;
      tmin = min(tmin, n);
      tmax = max(tmax, n);
    }
  }
  int64_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  nz = __reduce_add_sync(kFull, nz);
  tmin = __reduce_min_sync(kFull, tmin);
  tmax = __reduce_max_sync(kFull, tmax);
  if (lane == 31) s_wsum[warp] = incl;
  if (lane == 0) {
    s_wstat[3 * warp] = nz;
    s_wstat[3 * warp + 1] = tmin;
    s_wstat[3 * warp + 2] = tmax;
  }
  if (tid == 0) s_start[0] = -1;
  __syncthreads();
  int64_t before = 0, total = 0;
  int nz_all = 0, tmin_all = 0x7fffffff, tmax_all = 0;
#pragma unroll
  for (int i = 0; i < kTcWarps; ++i) {
    if (i < warp) before += s_wsum[i];
    total += s_wsum[i];
    nz_all += s_wstat[3 * i];
    tmin_all = min(tmin_all, s_wstat[3 * i + 1]);
    tmax_all = max(tmax_all, s_wstat[3 * i + 2]);
  }
  const int64_t excl = before + incl - mine;
  const int64_t T = total * a.Hkv;
  // split count: the caller's (or the automatic) count, one whole segment per
  // CTA or equal splits per segment for a uniform batch with the automatic
  // count, and never more splits than tiles (every split owns tiles)
  int64_t W64 = a.W;
  if (a.auto_split && nz_all > 0 && tmin_all == tmax_all) {
    const int64_t u = uniform_auto_splits(static_cast<int64_t>(nz_all) * a.Hkv, nctas);
    if (u > 0) W64 = u;
  }
  if (W64 > T) W64 = T;
  const int W = static_cast<int>(W64);
  const int64_t s0 = W > 0 ? static_cast<int64_t>(w) * W / nctas : 0;
  const int64_t s1 = W > 0 ? static_cast<int64_t>(w + 1) * W / nctas : 0;
  const int64_t b0 = W > 0 ? s0 * T / W : 0;
  const int64_t b1 = W > 0 ? s1 * T / W : 0;
  const bool has_work = b0 < b1;  // uniform over the CTA
  if (has_work && mine > 0 && b0 >= excl * a.Hkv && b0 < (excl + mine) * a.Hkv) {
    int64_t base = excl * a.Hkv;
    for (int r = rb; r < re; ++r) {
      const int n = tiles_of(a, r);
      const int64_t span = static_cast<int64_t>(n) * a.Hkv;
      if (b0 < base + span) {
        const int64_t off = b0 - base;
        s_start[0] = r;
        s_start[1] = static_cast<int>(off / n);
        s_start[2] = static_cast<int>(off % n);
        s_start[3] = n;
        break;
      }
      base += span;
    }
  }
  if (has_work) {
    if (tid == 0) {
      // arrivals per phase: the consumer-warp barriers take one per consumer
      // warp, the others one (an arm with its transaction bytes, or a commit)
      for (int i = 0; i < kNumBars; ++i) {
        const bool by_group = (i >= kBarSFree && i < kBarSFree + 2) || (i >= kBarPFull && i < kBarPFull + 2) ||
                              (i >= kBarOFree && i < kBarOFree + kOBufs) || i == kBarQFull ||
                              (i >= kBarCons && i < kBarCons + 2);
        mbar_init(bar(i), i == kBarConsAll ? kConsWarps : by_group ? kConsWarps / 2 : 1);
      }
      fence_barrier_init();
    }
    if (warp == kMmaWarp) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(s_tmem)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Everything above reads only inputs supplied before the previous kernel on
  // the stream began; from here on the abort mask and the cache may be read.
  griddep_wait();
  auto zero_dead_rows = [&](int t0, int nt) {
    for (int r = w; r < a.B; r += nctas) {
      if (tiles_of(a, r) == 0 || is_aborted(a, r)) {
        float* orow = a.out + static_cast<int64_t>(r) * a.Hq * kDim;
        for (int i = t0; i < a.Hq * kDim; i += nt) orow[i] = 0.f;
        if (a.lse != nullptr)
          for (int i = t0; i < a.Hq; i += nt) a.lse[static_cast<int64_t>(r) * a.Hq + i] = -INFINITY;
      }
    }
  };
  if (!has_work) {
    zero_dead_rows(tid, kTcThreads);
    return;
  }
  const uint32_t tmem = *s_tmem;
  Cursor start;
  start.r = s_start[0];
  start.h = s_start[1];
  start.t = s_start[2];
  start.n = s_start[3];
  start.x = b0;
  start.remaining = b1 - b0;
  start.split = -1;
  const bool bad_start = start.r < 0;  // inconsistent inputs (cannot happen)
  if (bad_start && tid == 0) atomicOr(a.status, kStatusBadStart);
  const int tpp = a.page_size >> 4;  // tiles per page

  if (warp < kProdWarps && !bad_start) {
    // ======================= producer warps =======================
    // Producer warp w takes the blocks j with j % 2 == w (the copy requests of
    // one warp issue at a limited rate, so two warps keep more in flight).
    // Lane i (mod 16) < 8 copies the K rows of tile i of a block (tensor map,
    // 128-byte swizzle) and lane 8 + i (mod 16) its V block (plain bulk
    // copy), the two half-warps on alternate blocks; lane 0 arms the stage's
    // barrier with the bytes of the tiles that exist and are in range.
    const uint64_t pol = l2_policy_evict_first();
    const int pw = warp;
    Cursor cur = start;
    Piece p;
    uint32_t j = 0;
    uint32_t last = 0;  // blocks this warp armed, as 1 + the last one's index
    bool ok = true;
    int ab_r = -1;
    bool ab = false;
    const int ti = lane & 7;
    while (ok && next_piece(cur, a, T, W, p)) {
      if (p.r != ab_r) {
        ab_r = p.r;
        ab = is_aborted(a, p.r);
      }
      if (ab) continue;
      const int32_t* ptrow = a.page_table + static_cast<int64_t>(p.r) * a.max_pages;
      const int nblk = (p.t1 - p.t0 + kBlkTiles - 1) / kBlkTiles;
      // this warp's blocks of the piece: blk0, blk0 + 2, ...; page ids are
      // loaded two of them ahead, so that copies never wait for the table
      const int blk0 = static_cast<int>((static_cast<uint32_t>(pw) - j) & 1u);
      auto load_id = [&](int b) -> int {
        const int t = p.t0 + b * kBlkTiles + ti;
        return b < nblk && t < p.t1 ? __ldg(ptrow + t / tpp) : -1;
      };
      int pg0 = load_id(blk0), pg1 = load_id(blk0 + 2);
      for (int blk = blk0; blk < nblk; blk += 2) {
        const uint32_t jb = j + static_cast<uint32_t>(blk);
        const uint32_t ks = jb % kStagesK, kround = jb / kStagesK;
        const uint32_t vs = jb % kStagesV, vround = jb / kStagesV;
        const int t = p.t0 + blk * kBlkTiles + ti;
        const bool present = t < p.t1;
        const int pg = pg0;
        pg0 = pg1;
        pg1 = load_id(blk + 4);
        {
          bool got = true;
          if (lane == 0 && kround > 0) got = mbar_wait(bar(kBarEmptyK + ks), (kround - 1) & 1, a.status);
          if (lane == 0 && got && vround > 0) got = mbar_wait(bar(kBarEmptyV + vs), (vround - 1) & 1, a.status);
          if (!__shfl_sync(kFull, got, 0)) {
            ok = false;
            break;
          }
        }
        const bool good = present && pg >= 0 && pg < a.num_pages;
        const uint32_t bad = __ballot_sync(kFull, present && !good) & 0xffu;
        const uint32_t goodm = __ballot_sync(kFull, good) & 0xffu;
        const uint32_t fk = bar(kBarFullK + ks), fv = bar(kBarFullV + vs);
        if (lane == 0) {
          s_fault[vs] = bad;
          const uint32_t bytes = static_cast<uint32_t>(__popc(goodm)) * kTile * kDim;
          if (bytes == 0) {
            mbar_arrive(fk);
            mbar_arrive(fv);
          } else {
            mbar_arrive_expect_tx(fk, bytes);
            mbar_arrive_expect_tx(fv, bytes);
          }
        }
        last = jb + 1;
        __syncwarp();
        if (good && (lane >> 4) == static_cast<int>((jb >> 1) & 1)) {
          const int64_t blkid = (static_cast<int64_t>(pg) * a.Hkv + p.h) * tpp + t % tpp;
          if ((lane & 15) < kBlkTiles)
            tma_load_2d(sbase + ks * kSlotBytes + ti * kTile * kDim, &kmap, 0, static_cast<int>(blkid * 2 * kTile),
                        fk, pol);
          else
            bulk_g2s(sbase + kOffV + vs * kSlotBytes + ti * kTile * kDim,
                     a.kv_pool + blkid * 2 * kTile * kDim + kTile * kDim, kTile * kDim, fv, pol);
        }
      }
      j += static_cast<uint32_t>(nblk);
    }
    if (lane == 0) {
      // every copy this warp issued has landed before the CTA exits (at once
      // unless a wait gave up): the last use of each of its slots
      for (uint32_t b = last > kStagesV ? last - kStagesV : 0; b < last; ++b) {
        if ((b & 1) != static_cast<uint32_t>(pw)) continue;
        mbar_wait(bar(kBarFullV + b % kStagesV), (b / kStagesV) & 1, a.status);
        if (b + kStagesK >= last) mbar_wait(bar(kBarFullK + b % kStagesK), (b / kStagesK) & 1, a.status);
      }
    }
  } else if (warp == kMmaWarp && !bad_start) {
    // ======================= MMA warp (one issuing thread) =======================
    // Two queues, issued as they become ready: S^T = K Q^T of the next block
    // (its K rows landed, its S buffer read by the consumers, and for the
    // first block of a new segment the query parts written), and O^T = V^T P^T
    // of the oldest block whose P is written (and whose O buffer is free).  A
    // group's next S is then computed while the group is still on its
    // current block.  One thread polls the barriers, bounded like every wait.
    if (lane == 0) {
      Cursor cur = start;
      Piece p;
      bool ok = true, more = true, have_piece = false, need_q = false;
      int ab_r = -1, q_seg = -1;
      bool ab = false;
      uint32_t qn = 0, jq = 0, jp = 0, piece_end = 0;
      const uint32_t tS = tmem, tO = tmem + 2 * kTcN;
      const uint32_t qaddr = sbase + kOffQ;
      auto advance = [&]() {
        while (more) {
          if (!next_piece(cur, a, T, W, p)) {
            more = false;
            return;
          }
          if (p.r != ab_r) {
            ab_r = p.r;
            ab = is_aborted(a, p.r);
          }
          if (ab) continue;
          const int seg = p.r * a.Hkv + p.h;
          need_q = seg != q_seg;
          q_seg = seg;
          piece_end = jq + static_cast<uint32_t>((p.t1 - p.t0 + kBlkTiles - 1) / kBlkTiles);
          have_piece = true;
          return;
        }
      };
      advance();
      uint64_t t0 = global_timer_ns();
      uint32_t spins = 0;
      while (ok && (have_piece || jp < jq)) {
        bool progress = false;
        if (jp < jq) {
          // O^T = V^T P^T of block jp: V blocks K-major without swizzle (core
          // matrices of 8 dims x 16 tokens; 128 B apart along the dims, 2 KiB
          // apart along the tokens), P K-major without swizzle (core matrices
          // of 8 columns x 16 tokens; 128 B along the columns, 512 B along
          // the tokens)
          const uint32_t sb = jp & 1, u = jp >> 1, ob = jp % kOBufs, ou = jp / kOBufs;
          if (mbar_test(bar(kBarPFull + sb), u & 1) && (ou == 0 || mbar_test(bar(kBarOFree + ob), (ou - 1) & 1))) {
            tc_fence_after();
            const uint32_t vaddr = sbase + kOffV + (jp % kStagesV) * kSlotBytes;
            const uint32_t paddr = sbase + kOffP + sb * kTcPBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc(vaddr + kk * 2 * kTile * kDim, kTile * kDim, 128, 0);
              const uint64_t bd = smem_desc(paddr + kk * 2 * 512, 512, 128, 0);
              mma_e4m3(tO + ob * kTcN, ad, bd, kk > 0);
            }
            mma_commit(bar(kBarOFull + ob));
            mma_commit(bar(kBarEmptyV + jp % kStagesV));
            ++jp;
            progress = true;
          }
        }
        if (have_piece) {
          if (need_q && mbar_test(bar(kBarQFull), qn & 1)) {
            ++qn;
            need_q = false;
          }
          const uint32_t ks = jq % kStagesK, kround = jq / kStagesK, sb = jq & 1, u = jq >> 1;
          if (!need_q && mbar_test(bar(kBarFullK + ks), kround & 1) &&
              (u == 0 || mbar_test(bar(kBarSFree + sb), (u - 1) & 1))) {
            tc_fence_after();
            // S^T = K Q^T: K rows and query parts K-major, 128-byte swizzle
            // (8-row groups 1024 B apart); each K step of 32 advances 32 B
            const uint32_t kaddr = sbase + ks * kSlotBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc(kaddr + 32 * kk, 16, 1024, 2);
              const uint64_t bd = smem_desc(qaddr + 32 * kk, 16, 1024, 2);
              mma_e4m3(tS + sb * kTcN, ad, bd, kk > 0);
            }
            mma_commit(bar(kBarSFull + sb));
            mma_commit(bar(kBarEmptyK + ks));
            if (++jq == piece_end) {
              have_piece = false;
              advance();
            }
            progress = true;
          }
        }
        if (progress) {
          t0 = global_timer_ns();
          spins = 0;
        } else if ((++spins & 255u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) {
          atomicOr(a.status, kStatusWaitTimeout);
          ok = false;
        }
      }
      // every MMA issued has completed before the tensor memory is freed
      mma_commit(bar(kBarDone));
      mbar_wait(bar(kBarDone), 0, a.status);
    }
    __syncwarp();
  } else if (warp > kMmaWarp && !bad_start) {
    // ======================= consumer warps =======================
    // Two groups of 8 warps take alternate blocks (group g the blocks with
    // j % 2 == g, in S, P and O buffer g), each with its own running (m, l, O)
    // over its blocks; at the end of a piece group 1 hands its state to
    // group 0, which merges the two and writes the result.  Within a group,
    // warp c takes TMEM lane quarter c % 4 and heads 4 (c / 4) .. + 3.
    const int cw = warp - kMmaWarp - 1;  // consumer warp 0..15
    const int grp = cw >> 3;             // block parity of this group
    const int c8 = cw & 7;
    const int wq = warp & 3;             // TMEM lane quarter of this warp
    const int hh = c8 >> 2;              // heads 4 hh .. 4 hh + 3 of the GQA group
    const int row = 32 * wq + lane;      // token of S / dim of O this thread reads
    const uint32_t lane_off = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t col0 = static_cast<uint32_t>(16 * hh);
    const int gt = c8 * 32 + lane;       // thread of the group 0..255
    const float kscale = __ldg(a.k_scale), vscale = __ldg(a.v_scale);
    const float kNegInf = -INFINITY;
    uint8_t* const s_q = sm + kOffQ;
    float* const s_xo = reinterpret_cast<float*>(sm + kOffX);  // group 1's O [8 heads][128 dims]
    float* const s_xml = s_xo + kGroupMax * kDim;                  // and its (m, l) per head
    Cursor cur = start;
    Piece p;
    uint32_t j = 0, gph = 0, aph = 0, npieces = 0;
    bool ok = true;
    int ab_r = -1, q_seg = -1;
    bool ab = false;
    float mult[kHalfHeads];
    // barrier of this group's 8 warps, and of all 16 consumer warps (bounded waits)
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarCons + grp));
      const bool got = mbar_wait(bar(kBarCons + grp), gph & 1, a.status);
      ++gph;
      return __all_sync(kFull, got);
    };
    auto all_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarConsAll));
      const bool got = mbar_wait(bar(kBarConsAll), aph & 1, a.status);
      ++aph;
      return __all_sync(kFull, got);
    };
    zero_dead_rows(cw * 32 + lane, 32 * kConsWarps);
    while (ok && next_piece(cur, a, T, W, p)) {
      if (p.r != ab_r) {
        ab_r = p.r;
        ab = is_aborted(a, p.r);
      }
      if (ab) continue;
      const int seg = p.r * a.Hkv + p.h;
      const int L = __ldg(a.seq_lens + p.r);
      if (seg != q_seg) {
        // ---- query parts of the GQA group's heads (B operand of S^T = K Q^T),
        // written by group 0: warp c takes head c, each lane 4 dims; a
        // power-of-two prescale takes the head's largest |q| into [128, 256)
        q_seg = seg;
        if (grp == 0) {
          const int hd = c8, d0 = lane * 4;
          float v[4];
          uint2 raw = make_uint2(0, 0);
          if (hd < a.G)
            raw = __ldg(reinterpret_cast<const uint2*>(a.q + (static_cast<int64_t>(p.r) * a.Hq + p.h * a.G + hd) * kDim + d0));
          const uint16_t* e = reinterpret_cast<const uint16_t*>(&raw);
          float amax = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[k] = bf16_bits_to_float(e[k]);
            amax = fmaxf(amax, fabsf(v[k]));
          }
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
          int e2 = 0;
          if (amax > 0.f && isfinite(amax)) e2 = min(max(7 - ilogbf(amax), -126), 126);
          const float sc = __int_as_float((127 + e2) << 23);
          const float isc = __int_as_float((127 - e2) << 23);
#pragma unroll
          for (int k = 0; k < 4; ++k) v[k] *= sc;
#pragma unroll
          for (int part = 0; part < kParts; ++part) {
            const uint32_t c01 = f32x2_to_e4m3x2(v[0], v[1]);
            const uint32_t c23 = f32x2_to_e4m3x2(v[2], v[3]);
            if (part + 1 < kParts) {
              const float2 d01 = e4m3x2_to_float2(c01), d23 = e4m3x2_to_float2(c23);
              v[0] = (v[0] - d01.x) * 16.f;
              v[1] = (v[1] - d01.y) * 16.f;
              v[2] = (v[2] - d23.x) * 16.f;
              v[3] = (v[3] - d23.y) * 16.f;
            }
            const int n = col_of(part, hd);
            const int off = n * 128 + ((((d0 >> 4) ^ (n & 7)) << 4) | (d0 & 15));
            *reinterpret_cast<uint32_t*>(s_q + off) = c01 | (c23 << 16);
          }
          if (lane == 0) s_mult[hd] = hd < a.G ? kscale * a.sm_scale_log2 * isc * (1.f / 4096.f) : 0.f;
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarQFull));
        }
        if (!all_sync()) {
          ok = false;
          break;
        }
#pragma unroll
        for (int i = 0; i < kHalfHeads; ++i) mult[i] = s_mult[4 * hh + i];
      }
      float m[kHalfHeads], lpart[kHalfHeads], o[kHalfHeads], alpha_prev[kHalfHeads];
#pragma unroll
      for (int i = 0; i < kHalfHeads; ++i) {
        m[i] = kNegInf;
        lpart[i] = 0.f;
        o[i] = 0.f;
        alpha_prev[i] = 0.f;
      }
      uint32_t fault = 0;
      // fold block i's O^T (this thread's dim, its four heads) into o with the
      // block's rescale
      auto accumulate = [&](uint32_t i, const float (&al)[kHalfHeads]) -> bool {
        const uint32_t ob = i % kOBufs, ou = i / kOBufs;
        if (!__all_sync(kFull, mbar_wait(bar(kBarOFull + ob), ou & 1, a.status))) return false;
        tc_fence_after();
        float pv[16];
        tmem_ld16(tmem + (2 + ob) * kTcN + col0 + lane_off, pv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarOFree + ob));
#pragma unroll
        for (int h = 0; h < kHalfHeads; ++h) o[h] = fmaf(o[h], al[h], part_sum(pv, h));
        return true;
      };
      const int nblk = (p.t1 - p.t0 + kBlkTiles - 1) / kBlkTiles;
      bool have_prev = false;  // this group has a block of this piece in O
      for (int blk = 0; blk < nblk; ++blk, ++j) {
        if (static_cast<int>(j & 1) != grp) continue;
        const uint32_t vs = j % kStagesV, vround = j / kStagesV, u = j >> 1;
        // ---- scores of this thread's token
        if (!__all_sync(kFull, mbar_wait(bar(kBarSFull + grp), u & 1, a.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[16];
        tmem_ld16(tmem + grp * kTcN + col0 + lane_off, sv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSFree + grp));
        // the stage's fault bits (the copies have landed: S is computed)
        if (!__all_sync(kFull, mbar_wait(bar(kBarFullV + vs), vround & 1, a.status))) {
          ok = false;
          break;
        }
        const uint32_t fb = s_fault[vs];
        fault |= fb;
        const int tile0 = p.t0 + blk * kBlkTiles;
        const int tt = tile0 + (row >> 4);
        const bool valid = tt < p.t1 && !((fb >> (row >> 4)) & 1u) && tt * kTile + (row & 15) < L;
        float s[kHalfHeads];
#pragma unroll
        for (int h = 0; h < kHalfHeads; ++h) s[h] = valid ? part_sum(sv, h) * mult[h] : kNegInf;
        // ---- block maximum per head over the 128 tokens
        {
          const float wm = warp_reduce4<true>(s, lane);
          if ((lane & 7) == 0) s_red[((grp * 2 + (u & 1)) * 4 + wq) * kGroupMax + 4 * hh + (lane >> 3)] = wm;
        }
        if (!group_sync()) {
          ok = false;
          break;
        }
        float alpha[kHalfHeads], pr[kHalfHeads];
        {
          const float4* rq = reinterpret_cast<const float4*>(s_red + (grp * 2 + (u & 1)) * 4 * kGroupMax + 4 * hh);
          const float4 r0 = rq[0], r1 = rq[2], r2 = rq[4], r3 = rq[6];
          const float bmax[4] = {fmaxf(fmaxf(r0.x, r1.x), fmaxf(r2.x, r3.x)), fmaxf(fmaxf(r0.y, r1.y), fmaxf(r2.y, r3.y)),
                                 fmaxf(fmaxf(r0.z, r1.z), fmaxf(r2.z, r3.z)), fmaxf(fmaxf(r0.w, r1.w), fmaxf(r2.w, r3.w))};
#pragma unroll
          for (int h = 0; h < kHalfHeads; ++h) {
            const float mn = fmaxf(m[h], bmax[h]);
            alpha[h] = m[h] == kNegInf ? 0.f : fast_exp2(m[h] - mn);
            pr[h] = valid ? fast_exp2(s[h] - mn) : 0.f;
            lpart[h] = fmaf(lpart[h], alpha[h], pr[h]);
            m[h] = mn;
          }
        }
        // ---- this group's previous block's O, before its P buffer is
        // rewritten: the wait for that O is the wait for the PV MMA that read
        // the buffer (the MMA thread may compute this block's S before it)
        if (have_prev && !accumulate(j - 2, alpha_prev)) {
          ok = false;
          break;
        }
        have_prev = true;
#pragma unroll
        for (int h = 0; h < kHalfHeads; ++h) alpha_prev[h] = alpha[h];
        // ---- P = e4m3 parts of 256 p into this group's P buffer (K-major,
        // core matrices of 8 columns x 16 tokens)
        {
          uint8_t* const pb = sm + kOffP + grp * kTcPBytes + (row >> 4) * 512 + (row & 15);
          float x0 = pr[0] * 256.f, x1 = pr[1] * 256.f, x2 = pr[2] * 256.f, x3 = pr[3] * 256.f;
#pragma unroll
          for (int part = 0; part < kParts; ++part) {
            const uint32_t c01 = f32x2_to_e4m3x2(x0, x1);
            const uint32_t c23 = f32x2_to_e4m3x2(x2, x3);
            // columns 16 hh + 4 part + i: core matrix 2 hh + part / 2, row 4 (part % 2) + i
            uint8_t* const pc = pb + (2 * hh + (part >> 1)) * 128 + (part & 1) * 64;
            pc[0] = static_cast<uint8_t>(c01 & 0xffu);
            pc[16] = static_cast<uint8_t>(c01 >> 8);
            pc[32] = static_cast<uint8_t>(c23 & 0xffu);
            pc[48] = static_cast<uint8_t>(c23 >> 8);
            if (part + 1 < kParts) {
              const float2 d01 = e4m3x2_to_float2(c01), d23 = e4m3x2_to_float2(c23);
              x0 = (x0 - d01.x) * 16.f;
              x1 = (x1 - d01.y) * 16.f;
              x2 = (x2 - d23.x) * 16.f;
              x3 = (x3 - d23.y) * 16.f;
            }
          }
        }
        // ---- V columns of tokens that take no part are zeroed (a stale or
        // unwritten slot may hold NaN codes, and 0 x NaN is NaN); group thread
        // gt takes dim row gt % 128 of the block's even or odd tiles
        if (tile0 + kBlkTiles > p.t1 || fb != 0u || (tile0 + kBlkTiles) * kTile > L) {
#pragma unroll 1
          for (int i = gt >> 7; i < kBlkTiles; i += 2) {
            const int ti = tile0 + i;
            const bool gone = ti >= p.t1 || ((fb >> i) & 1u);
            const int nv = gone ? 0 : min(kTile, L - ti * kTile);
            if (nv < kTile) {
              uint4* vrow = reinterpret_cast<uint4*>(sm + kOffV + vs * kSlotBytes + i * kTile * kDim +
                                                     (gt & 127) * 16);
              uint4 x = nv <= 0 ? make_uint4(0, 0, 0, 0) : *vrow;
              if (nv > 0) {
                uint32_t* wds = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const int keep = nv - 4 * q4;  // bytes of this word that stay
                  wds[q4] = keep >= 4 ? wds[q4] : keep <= 0 ? 0u : (wds[q4] & (0xffffffffu >> (8 * (4 - keep))));
                }
              }
              *vrow = x;
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + grp));
      }
      if (!ok) break;
      // this group's last block of the piece (j - 1 or j - 2 by parity)
      const uint32_t jlast = ((j - 1) & 1) == static_cast<uint32_t>(grp) ? j - 1 : j - 2;
      if (have_prev && !accumulate(jlast, alpha_prev)) {
        ok = false;
        break;
      }
      // ---- the group's (m, l, O): l summed over its 128 token threads
      float* const s_lsum = s_red + kRedSums + grp * 4 * kGroupMax;
      {
        const float ws = warp_reduce4<false>(lpart, lane);
        if ((lane & 7) == 0) s_lsum[wq * kGroupMax + 4 * hh + (lane >> 3)] = ws;
        const uint32_t wf = __any_sync(kFull, fault != 0);
        if (lane == 0) s_wfault[(npieces & 1) * kConsWarps + cw] = wf;
      }
      if (!all_sync()) {
        ok = false;
        break;
      }
      float l[kHalfHeads];
#pragma unroll
      for (int h = 0; h < kHalfHeads; ++h)
        l[h] = s_lsum[4 * hh + h] + s_lsum[kGroupMax + 4 * hh + h] + s_lsum[2 * kGroupMax + 4 * hh + h] +
               s_lsum[3 * kGroupMax + 4 * hh + h];
      // group 1 hands its state over (every thread its dim's O; (m, l) once)
      if (grp == 1) {
#pragma unroll
        for (int h = 0; h < kHalfHeads; ++h) {
          s_xo[(4 * hh + h) * kDim + row] = o[h];
          if (row == 0) {
            s_xml[2 * (4 * hh + h)] = m[h];
            s_xml[2 * (4 * hh + h) + 1] = l[h];
          }
        }
      }
      if (!all_sync()) {
        ok = false;
        break;
      }
      if (grp == 0) {
        uint32_t anyf = 0;
#pragma unroll
        for (int i = 0; i < kConsWarps; ++i) anyf |= s_wfault[(npieces & 1) * kConsWarps + i];
        const bool dead = anyf != 0;
#pragma unroll
        for (int h = 0; h < kHalfHeads; ++h) {
          const float m1 = s_xml[2 * (4 * hh + h)], l1 = s_xml[2 * (4 * hh + h) + 1];
          const float mm = fmaxf(m[h], m1);
          const float f0 = m[h] == kNegInf ? 0.f : fast_exp2(m[h] - mm);
          const float f1 = m1 == kNegInf ? 0.f : fast_exp2(m1 - mm);
          o[h] = o[h] * f0 + s_xo[(4 * hh + h) * kDim + row] * f1;
          l[h] = l[h] * f0 + l1 * f1;
          m[h] = mm;
        }
        const float oscale = vscale * (1.f / 1048576.f);  // p entered as 256 p, parts as 4096 x
        const bool whole = p.t0 == 0 && p.t1 == p.n;
        if (whole) {
#pragma unroll
          for (int h = 0; h < kHalfHeads; ++h) {
            const int hd = 4 * hh + h;
            if (hd < a.G) {
              const int64_t orow = static_cast<int64_t>(p.r) * a.Hq + p.h * a.G + hd;
              const bool dh = dead || l[h] == 0.f;
              a.out[orow * kDim + row] = dh ? 0.f : o[h] * oscale / l[h];
              if (row == 0 && a.lse != nullptr) a.lse[orow] = dh ? kNegInf : (m[h] + __log2f(l[h])) * kTcLn2;
            }
          }
        } else {
          const int64_t slot = static_cast<int64_t>(seg) + p.s;
#pragma unroll
          for (int h = 0; h < kHalfHeads; ++h) {
            const int hd = 4 * hh + h;
            if (hd < a.G) {
              a.part_o[(slot * a.G + hd) * kDim + row] = o[h] * oscale;
              if (row == 0)
                a.part_ml[slot * a.G + hd] = dead ? make_float2(kNegInf, -1.f) : make_float2(m[h], l[h]);
            }
          }
          // arrival ticket; the arrival that completes the segment merges its
          // partials (splits w0..w1, slots seg + w)
          const int64_t xseg = p.x0 - p.t0;
          const int sw0 = worker_of(xseg, T, W), sw1 = worker_of(xseg + p.n - 1, T, W);
          const int cnt = sw1 - sw0 + 1;
          __threadfence();
          if (!group_sync()) {
            ok = false;
            break;
          }
          if (gt == 0) {
            *s_last = atomicAdd(a.seg_count + seg, 1) + 1 == cnt;
            __threadfence();
          }
          if (!group_sync()) {
            ok = false;
            break;
          }
          if (*s_last) {
            __threadfence();
            float M[kHalfHeads], Wt[kHalfHeads], acc[kHalfHeads];
            bool any_dead = false;
#pragma unroll
            for (int h = 0; h < kHalfHeads; ++h) {
              M[h] = kNegInf;
              Wt[h] = 0.f;
              acc[h] = 0.f;
            }
            for (int i = 0; i < cnt; ++i) {
              const int64_t sl = static_cast<int64_t>(seg) + sw0 + i;
#pragma unroll
              for (int h = 0; h < kHalfHeads; ++h) {
                const float2 ml = __ldcg(a.part_ml + sl * a.G + min(4 * hh + h, a.G - 1));
                M[h] = fmaxf(M[h], ml.x);
                any_dead |= ml.y < 0.f;
              }
            }
#pragma unroll 2
            for (int i = 0; i < cnt; ++i) {
              const int64_t sl = static_cast<int64_t>(seg) + sw0 + i;
              float po[kHalfHeads];
              float2 ml[kHalfHeads];
#pragma unroll
              for (int h = 0; h < kHalfHeads; ++h) {
                const int hx = min(4 * hh + h, a.G - 1);
                ml[h] = __ldcg(a.part_ml + sl * a.G + hx);
                po[h] = __ldcg(a.part_o + (sl * a.G + hx) * kDim + row);
              }
#pragma unroll
              for (int h = 0; h < kHalfHeads; ++h) {
                const float f = ml[h].x == kNegInf ? 0.f : fast_exp2(ml[h].x - M[h]);
                Wt[h] = fmaf(ml[h].y, f, Wt[h]);
                acc[h] = fmaf(po[h], f, acc[h]);
              }
            }
#pragma unroll
            for (int h = 0; h < kHalfHeads; ++h) {
              const int hd = 4 * hh + h;
              if (hd < a.G) {
                const int64_t orow = static_cast<int64_t>(p.r) * a.Hq + p.h * a.G + hd;
                const bool dh = any_dead || Wt[h] == 0.f;
                a.out[orow * kDim + row] = dh ? 0.f : acc[h] / Wt[h];
                if (row == 0 && a.lse != nullptr) a.lse[orow] = dh ? kNegInf : (M[h] + __log2f(Wt[h])) * kTcLn2;
              }
            }
            if (gt == 0) a.seg_count[seg] = 0;  // ready for the next call
          }
        }
      }
      ++npieces;
    }
  }
  // ---- every role is done; the tensor memory is freed by the warp that took it
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr int kTcMaxDevices = 64;
std::atomic<int> g_tc_per_sm[kTcMaxDevices];

int prepare_tc_kernel(int dev) {
  std::atomic<int>& slot = g_tc_per_sm[dev];
  int v = slot.load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaFuncSetAttribute(paged_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes) !=
      cudaSuccess)
    return -1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, paged_decode_tc_kernel, kTcThreads, kTcSmemBytes) !=
          cudaSuccess ||
      per_sm <= 0)
    return -1;
  slot.store(per_sm, std::memory_order_relaxed);
  return per_sm;
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled tensor_map_encoder() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
  });
  return fn;
}

// The pool as rows of 128 bytes (a tile is 32 rows: 16 K rows, then the V
// block); boxes of 16 rows land with the 128-byte swizzle.
int encode_pool_map(CUtensorMap* m, const void* kv_pool, int64_t rows) {
  EncodeTiled enc = tensor_map_encoder();
  if (enc == nullptr) return FPK_ECUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDim)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kDim), static_cast<cuuint32_t>(kTile)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv_pool), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FPK_OK : FPK_ECUDA;
}

}  // namespace
}  // namespace fpk

extern "C" int fpk_paged_decode_attn_fp8_tc(const void* q, const uint8_t* kv_pool, const float* k_scale,
                                            const float* v_scale, const int32_t* page_table,
                                            int32_t max_pages, const int32_t* seq_lens,
                                            const uint8_t* abort_mask, float* out, float* lse,
                                            void* workspace, size_t workspace_bytes, int32_t num_splits,
                                            float sm_scale, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                            int32_t page_size, int32_t num_pages, void* stream) {
  using namespace fpk;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0 || max_pages < 0 ||
      num_splits < 0 || Hq % Hkv != 0)
    return FPK_EINVAL;
  const int G = Hq / Hkv;
  if (D != kDim || G > kGroupMax || page_size % kTile != 0 || page_size > 256) return FPK_EUNSUPPORTED;
  // the pool's 128-byte rows are addressed with 32-bit tensor-map coordinates
  const int64_t rows = static_cast<int64_t>(num_pages) * Hkv * (page_size / kTile) * 2 * kTile;
  if (rows > 0x7fffffffll) return FPK_EUNSUPPORTED;
  if (B == 0) return FPK_OK;
  if (!q || !kv_pool || !k_scale || !v_scale || !page_table || !seq_lens || !out || !workspace)
    return FPK_EINVAL;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FPK_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kTcMaxDevices) return FPK_ECUDA;
  const int per_sm = prepare_tc_kernel(dev);
  const int wave = device_sm_count(dev) * per_sm;
  if (per_sm <= 0 || wave <= 0) return FPK_ECUDA;
  int W = num_splits;
  if (W == 0) {
    const int64_t cap = static_cast<int64_t>(kAutoSplitsPerSegment) * B * Hkv;
    W = cap < wave ? static_cast<int>(cap) : wave;
  }
  const int per_cta = (W + wave - 1) / wave;
  const int ctas = W <= wave ? W : (W + per_cta - 1) / per_cta;
  const WsLayout l = layout(B, Hkv, G, W);
  if (workspace_bytes < l.total) return FPK_ENOSPC;
  CUtensorMap kmap;
  if (encode_pool_map(&kmap, kv_pool, rows > 0 ? rows : 2 * kTile) != FPK_OK) return FPK_ECUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  TcArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.kv_pool = kv_pool;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.abort_mask = abort_mask;
  a.out = out;
  a.lse = lse;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.seg_count = reinterpret_cast<int*>(ws + l.seg_count);
  a.part_ml = reinterpret_cast<float2*>(ws + l.part_ml);
  a.part_o = reinterpret_cast<float*>(ws + l.part_o);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.max_pages = max_pages;
  a.W = W;
  a.auto_split = num_splits == 0;
  a.sm_scale_log2 = sm_scale * kTcLog2e;
  paged_decode_tc_kernel<<<ctas, kTcThreads, kTcSmemBytes, static_cast<cudaStream_t>(stream)>>>(a, kmap);
  return checked_launch_status();
}
