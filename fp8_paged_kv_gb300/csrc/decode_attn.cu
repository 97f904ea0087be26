// decode_attn.cu -- split-KV paged decode attention over the FP8 e4m3 (or the
// BF16 comparison) cache, dequantising on read, plus the cross-split combine.
//
// The Cloudflare Kimi decode pool reads an FP8 e4m3 KV cache and the attention
// kernel converts the values as it reads them ("Perche le cache piu piccole di
// Cloudflare battono la velocita pura", remio.ai); pages are reusable physical
// blocks reached through a per-sequence table and requests that failed the tag
// check read nothing ("La sicurezza della cache KV condivisa...").  The pages
// give no kernel design; this one is built for GB300:
//
// * Work split.  All (request, kv head) segments are laid end to end as a
//   list of 16-token tiles cut into W splits of equal tile count (W = one
//   wave of CTAs by default), so variable context lengths cost no tail.  At
//   most one wave of CTAs runs; with more splits than that a CTA takes
//   consecutive splits in turn without draining its copy pipeline between
//   them, keeping its query fragments while the segment stays the same.  A
//   CTA finds its start with a block scan over seq_lens.  With the automatic
//   count, batches with few segments get split boundaries on segment
//   boundaries instead: equal lengths give every segment the same number of
//   splits (one whole segment per CTA once they fill 3/4 of a wave), unequal
//   ones cut every segment into splits of one common size, one per CTA.
// * Data movement.  Warp 0 is a producer: each of its lanes issues one
//   cp.async.bulk (TMA) copy of one tile's K block [16 tok][128] and V block
//   [128][16 tok] -- adjacent in the pool layout, so one copy of 4 KiB (FP8),
//   or 8 KiB for two adjacent tiles of one page -- into a ring of shared-memory
//   stages completing on mbarriers, with an L2 evict-first hint.  The FP8
//   kernel comes with an 8-stage and a 12-stage ring; the deeper one is used
//   while the grid's copies in flight stay within a budget.  Page ids
//   outside the pool are never dereferenced.
// * Math.  Consumer warps take ring stages round-robin.  With the GQA group on
//   the N side of the tensor-core tile, S^T = K Q^T and O^T = V^T P^T are
//   m16n8k16 MMAs; e4m3 codes convert exactly to f16 in registers (the query
//   gets a per-head power-of-two prescale into f16 range), P = hi + lo is
//   transposed from accumulator to operand layout with movmatrix, softmax is
//   online in the log2 domain with warp-shuffle reductions.  The dims of each 16-wide
//   k-step and the tokens of each tile are visited in a fixed permuted order
//   (the same on both operands), so every operand fragment is a contiguous
//   4-byte run of shared memory.
// * Merge.  At the end of each segment piece the consumer warps merge their
//   (m, l, O) in shared memory; a CTA that owns a whole segment writes the
//   final output, otherwise it writes a partial and counts an arrival (its
//   consecutive arrivals on one counter in one ticket); the CTA whose
//   arrivals complete a segment's count merges its partials by log-sum-exp,
//   in two levels above 16 partials (one launch per call; nothing ever waits
//   on another CTA).
// * Safety.  Every wait is bounded (status word in the workspace); no barrier
//   without a timeout is used after the prologue.
#include <atomic>

#include "attn_plan.cuh"
#include "common.cuh"
#include "step_ops.cuh"

namespace fpk {
namespace {

constexpr int kMergeStride = 132;  // floats per head row of the merge buffer
constexpr int kMergeBars = 7;      // merge_free, cbar, the three rounds of the two-slot merge, the four-slot one,
                                   // the staged combine's copies
constexpr int64_t kInflightBudget = 26ll << 20;  // bytes of ring stages over the grid (see Cfg)
constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
static_assert(kConsumerWarps * 32 == 128, "the split-segment combine gives each consumer thread one of the 128 dims");
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <bool kFp8, bool kDeep = false>
struct Cfg {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kBlockBytes = kTile * kDim * kElem;  // one K (or V) tile
  // a stage holds two consecutive tiles, each as it lies in the pool:
  // [K tile 0][V tile 0][K tile 1][V tile 1]
  static constexpr int kStageBytes = 4 * kBlockBytes;
  // Ring depth: kStages stages in shared memory, of which a launch uses all or
  // kStagesShallow.  Deeper rings keep more copies in flight per CTA, which
  // pays while the whole grid's copies in flight stay under kInflightBudget;
  // beyond it (measured on GB300: about 26 MiB over the GPU) the memory
  // system serves the copies more slowly than with the shallower ring.  The
  // deep FP8 variant holds 12 stages; the others hold only the shallow ring
  // (a larger shared-memory footprint costs a little even when unused).
  static constexpr int kStages = kFp8 ? (kDeep ? 12 : 8) : 4;
  static constexpr int kStagesShallow = kFp8 ? 8 : 4;
  // Within a segment piece consumer warp c takes stages c, c+4, ...; with
  // the depth a multiple of the warp count, the previous round of a stage was
  // consumed by the same warp, so no warp ever waits on a stage's mbarrier
  // while its previous phase is still pending (the parity test would alias
  // two phases back).  Across pieces the merge barrier gives the same order.
  static_assert(kStages % kConsumerWarps == 0 && kStagesShallow % kConsumerWarps == 0,
                "ring depths must be multiples of the consumer warps");
  static_assert(kStages <= 16, "a producer batch gives each stage two lanes");
  static constexpr int kRingBytes = kStages * kStageBytes;
  // (m, l, O) slots of the merge of the consumer warps' results: four (one
  // round), or two (two rounds) in the deep variant, whose ring leaves no
  // room for four at two CTAs per SM.
  static constexpr int kMergeSlots = kDeep ? 2 : 4;
  static constexpr int kMergeBytes = kMergeSlots * kGroupMax * kMergeStride * 4;
  // (m, l) per warp and head, then one fault flag per warp; rounded to 16 bytes
  // so that the mbarriers that follow stay 8-byte aligned for any warp count
  static constexpr int kMlBytes = (kConsumerWarps * kGroupMax * 4 * 2 + kConsumerWarps * 4 + 15) / 16 * 16;
  static constexpr int kBarBytes = (2 * kStages + kMergeBars) * 8;
  static constexpr int kSmemBytes = kRingBytes + kMergeBytes + kMlBytes + kBarBytes + kStages * 4 + 64;
};

struct AttnArgs {
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
  int* seg_count;    // per-segment arrival tickets, zero between calls
  int* group_count;  // per-group arrival tickets (indexed by slot), zero between calls
  float2* part_ml;
  float* part_o;
  int B, Hq, Hkv, G, page_size, num_pages, max_pages, W;
  int auto_split;  // W is the automatic count: the kernel may pick one split per segment
  float sm_scale_log2;
};

// Slots of the members i0, i0 + stride, ... of one segment's partials: member
// i is split w0 + i when every split owns tiles, else the owner of tile i.
struct Members {
  int64_t seg, xseg;
  int w0, i0, stride;
  bool dense;
};

// Atomic add with acquire-release semantics at GPU scope (returns the old
// value): the writes that happen before it are visible to the thread whose
// atomic reads its result, and the caller sees the writes released by the
// atomics it reads.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Four 8 x 8 matrices of 16-bit elements from shared memory (ldmatrix).
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Token (row of the tile) that fragment row i stands for: rows 2t, 2t+1,
// 2t+8, 2t+9 map to tokens 4t..4t+3, so each lane's V operand is one
// contiguous 4-token run.
__device__ __forceinline__ int token_of_row(int i) {
  return 4 * ((i & 7) >> 1) + (i & 1) + 2 * (i >> 3);
}

// The smallest common split size (in tiles) whose split count over the
// batch's non-empty (request, kv head) segments fits the CTAs: every thread
// counts the splits for one candidate between ceil(T / CTAs) and
// ceil(T / (CTAs - segments)) (the last always fits: each segment's rounding
// adds at most one split); a block min picks the smallest that fits.  A
// segment's tile count fits in 32 bits, and so do the candidates that matter
// (larger ones are clamped: they give one split per segment).  Called by
// every thread of the CTA; kept out of line so that launches that never take
// this partition do not carry its code in their prologue (measured on GB300:
// inlined, it slowed small single launches by about 2 us).
__device__ __noinline__ int64_t tightest_split_size(const AttnArgs& a, int64_t T, int nctas, int64_t segs,
                                                    int64_t* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t hi = (T + (nctas - segs) - 1) / (nctas - segs);
  const int64_t lo = T > nctas ? (T + nctas - 1) / nctas : 1;
  const int64_t cand = lo + (hi - lo) * tid / (kThreads - 1);
  const uint32_t c32 = static_cast<uint32_t>(min(cand, static_cast<int64_t>(0x7fffffff)));
  int64_t cnt = 0;
  for (int r = 0; r < a.B; ++r) {
    const uint32_t n = static_cast<uint32_t>(tiles_of(a, r));
    cnt += (n + c32 - 1u) / c32;
  }
  cnt *= a.Hkv;
  int64_t best = cnt <= nctas ? cand : hi;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, o));
  if (lane == 0) s_warp[warp] = best;
  __syncthreads();
  int64_t c = s_warp[0];
#pragma unroll
  for (int i = 1; i < kThreads / 32; ++i) c = min(c, s_warp[i]);
  __syncthreads();  // s_warp is reused by the caller
  return c;
}

template <bool kFp8, bool kDeep>
__global__ void __launch_bounds__(kThreads, 2) paged_decode_split_kernel(const AttnArgs a) {
  using C = Cfg<kFp8, kDeep>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  float* s_o = reinterpret_cast<float*>(smem + C::kRingBytes);
  float* s_m = s_o + C::kMergeSlots * kGroupMax * kMergeStride;
  float* s_l = s_m + kConsumerWarps * kGroupMax;
  int* s_wfault = reinterpret_cast<int*>(s_l + kConsumerWarps * kGroupMax);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kRingBytes + C::kMergeBytes + C::kMlBytes);
  int* s_stage_fault = reinterpret_cast<int*>(bars + 2 * C::kStages + kMergeBars);

  __shared__ int64_t s_warp_sum[kThreads / 32], s_warp_splits[kThreads / 32];
  __shared__ int s_warp_nz[kThreads / 32], s_warp_min[kThreads / 32], s_warp_max[kThreads / 32];
  __shared__ int s_start[7];  // r, h, t0, n; segment-aligned partition: t1, first split of the segment, splits
  __shared__ int64_t s_start_x;
  __shared__ int s_last;
  __shared__ Piece s_pend_piece;  // the pending arrivals of split pieces (see publish_partial)
  __shared__ int s_pend_seg, s_pend_k;
  __shared__ int* s_pend_ctr;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int w = blockIdx.x;
  const unsigned kFull = 0xffffffffu;

  // barriers: stage s is full0 + 8 s (filled) and empty0 + 8 s (consumed),
  // then the merge barriers
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = full0 + 8 * C::kStages;
  const uint32_t merge_free = full0 + 16 * C::kStages;
  const uint32_t cbar = merge_free + 8;  // consumer-warp barrier of the split-segment combine
  // the two-slot merge of a piece: warps 2, 3 have filled slots 0, 1 (mrg0);
  // warps 0, 1 have read them (mrg1); warps 0, 1 have filled them (mrg2).
  // The four-slot merge: every warp has filled its slot (mrg4).
  const uint32_t mrg0 = cbar + 8, mrg1 = cbar + 16, mrg2 = cbar + 24, mrg4 = cbar + 32;
  const uint32_t comb_bar = cbar + 40;  // the staged combine's bulk copies have landed
  // ---- prologue: total tiles and this CTA's start (block scan over requests)
  const int chunk = (a.B + kThreads - 1) / kThreads;
  const int rb = tid * chunk;
  const int re = min(a.B, rb + chunk);
  int64_t mine = 0;
  int nz = 0, tmin = 0x7fffffff, tmax = 0;  // requests with tiles; their fewest and most
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
  if (lane == 31) s_warp_sum[warp] = incl;
  if (lane == 0) {
    s_warp_nz[warp] = nz;
    s_warp_min[warp] = tmin;
    s_warp_max[warp] = tmax;
  }
  if (tid == 0) {
    s_start[0] = -1;
    s_pend_k = 0;
  }
  __syncthreads();
  int64_t before = 0, total = 0;
  int nz_all = 0, tmin_all = 0x7fffffff, tmax_all = 0;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) {
    if (i < warp) before += s_warp_sum[i];
    total += s_warp_sum[i];
    nz_all += s_warp_nz[i];
    tmin_all = min(tmin_all, s_warp_min[i]);
    tmax_all = max(tmax_all, s_warp_max[i]);
  }
  const int64_t excl = before + incl - mine;
  const int64_t T = total * a.Hkv;
  const int nctas = static_cast<int>(gridDim.x);
  // Split count.  With the automatic count, a batch whose (request, kv head)
  // segments all have the same length takes uniform_auto_splits: a batch of
  // between 3/4 of the CTAs and all of them runs one whole segment per CTA
  // (no split partials, no cross-CTA combine: that costs less than the idle
  // quarter of the CTAs); a smaller one gets an equal number of splits per
  // segment, aligned to the segments.
  int W = a.W;
  if (a.auto_split && nz_all > 0 && tmin_all == tmax_all) {
    const int64_t u = uniform_auto_splits(static_cast<int64_t>(nz_all) * a.Hkv, nctas);
    if (u > 0) W = static_cast<int>(u);
  }
  // Segment-aligned partition (automatic count, lengths not all equal, at
  // most a third as many segments as CTAs): every non-empty segment is cut
  // into splits of csz tiles (its last one shorter), csz the smallest size
  // whose split count fits the CTAs (at most ceil(T / (CTAs - segments))):
  // one split per CTA, none straddling two segments, none more than half
  // above T / CTAs.  (Measured on GB300 with 8192-token-scale mixed lengths:
  // up to a third of the CTAs it gains 2-22 %; at half of them, with
  // ceil(T / (CTAs - segments)), the larger splits lost up to 27 %.)
  const int64_t segs_nz = static_cast<int64_t>(nz_all) * a.Hkv;
  const bool aligned = a.auto_split && nz_all > 0 && tmin_all != tmax_all && 3 * segs_nz <= nctas;
  int64_t csz = 1, excl_splits = 0, mine_splits = 0;
  if (aligned) {
    csz = tightest_split_size(a, T, nctas, segs_nz, s_warp_splits);
    for (int r = rb; r < re; ++r) {
      const int n = tiles_of(a, r);
      mine_splits += static_cast<int64_t>(a.Hkv) * ((n + csz - 1) / csz);
    }
    int64_t inc = mine_splits;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) s_warp_splits[warp] = inc;
    __syncthreads();
    int64_t bef = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) {
      if (i < warp) bef += s_warp_splits[i];
      tot += s_warp_splits[i];
    }
    excl_splits = bef + inc - mine_splits;
    W = static_cast<int>(tot);  // < CTAs
  }
  // this CTA runs splits [s0, s1) one after another: tiles [b0, b1)
  // (aligned: split w alone, its tiles found below)
  const int64_t s0 = static_cast<int64_t>(w) * W / nctas;
  const int64_t s1 = static_cast<int64_t>(w + 1) * W / nctas;
  const int64_t b0 = aligned ? 0 : s0 * T / W;
  const int64_t b1 = aligned ? (w < W ? 1 : 0) : s1 * T / W;
  const bool has_work = b0 < b1;  // uniform over the CTA
  // ring depth of this launch, from the CTAs that have work
  int64_t active = W < nctas ? W : nctas;
  if (T < active) active = T;
  const uint32_t depth =
      active * C::kStages * C::kStageBytes <= kInflightBudget ? C::kStages : C::kStagesShallow;
  if (aligned) {
    if (has_work && mine_splits > 0 && w >= excl_splits && w < excl_splits + mine_splits) {
      int64_t base = excl_splits, xbase = excl * a.Hkv;
      for (int r = rb; r < re; ++r) {
        const int n = tiles_of(a, r);
        const int m = static_cast<int>((n + csz - 1) / csz);  // splits of each of its segments
        const int64_t span = static_cast<int64_t>(m) * a.Hkv;
        if (w < base + span) {
          const int off = static_cast<int>(w - base);
          const int h = off / m, j = off - h * m;
          const int t0 = static_cast<int>(j * csz);
          s_start[0] = r;
          s_start[1] = h;
          s_start[2] = t0;
          s_start[3] = n;
          s_start[4] = static_cast<int>(min(static_cast<int64_t>(n), t0 + csz));
          s_start[5] = static_cast<int>(base) + h * m;
          s_start[6] = m;
          s_start_x = xbase + static_cast<int64_t>(h) * n + t0;
          break;
        }
        base += span;
        xbase += static_cast<int64_t>(n) * a.Hkv;
      }
    }
  } else if (has_work && mine > 0 && b0 >= excl * a.Hkv && b0 < (excl + mine) * a.Hkv) {
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
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(merge_free, kConsumerWarps);
    mbar_init(cbar, kConsumerWarps);
    mbar_init(mrg0, 2);
    mbar_init(mrg1, 2);
    mbar_init(mrg2, 2);
    mbar_init(mrg4, kConsumerWarps);
    mbar_init(comb_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Everything above reads only inputs the caller supplied before the
  // previous kernel on the stream began; from here on the abort mask and the
  // cache may be read (a no-op unless launched as a programmatic dependent).
  griddep_wait();
  // requests that read nothing (empty, aborted, over-long) get out = 0 and
  // lse = -inf; the CTAs share this round-robin (in a working CTA the
  // consumer warps do it while the producer starts its copies)
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
    zero_dead_rows(tid, kThreads);
    return;
  }
  if (s_start[0] < 0) {  // inconsistent inputs (cannot happen): nothing to do
    if (tid == 0) atomicOr(a.status, kStatusBadStart);
    return;
  }
  Cursor start;
  start.r = s_start[0];
  start.h = s_start[1];
  start.t = s_start[2];
  start.n = s_start[3];
  start.x = aligned ? s_start_x : b0;
  start.remaining = aligned ? s_start[4] - s_start[2] : b1 - b0;
  start.split = aligned ? w : -1;
  const int tpp = a.page_size >> 4;  // tiles per page

  if (warp == 0) {
    // ======================= producer warp =======================
    // Bulk copies issued by one thread complete one after another, so every
    // copy gets its own lane: lanes 2s and 2s+1 serve stage s of a batch of
    // up to 16 stages, one tile each (a tile's K and V blocks are adjacent in
    // the pool: one copy); two adjacent tiles of one page go as one copy.  The
    // even lane polls the stage's "empty" barrier and, once it is free, sets
    // the stage's transaction count; after a warp sync both lanes issue.
    // Stages are issued the moment they are free, so the ring never drains at
    // a batch boundary, and a batch only waits on stages that an earlier batch
    // filled.  Page ids of the next batch of a piece load while this one polls.
    const int batch = static_cast<int>(depth);  // a batch never wraps around the ring
    const uint64_t pol = l2_policy_evict_first();
    const int si = lane >> 1;  // stage slot of this lane within a batch
    const int ci = lane & 1;   // tile of the stage this lane copies
    Cursor cur = start;
    Piece p;
    uint32_t j = 0;  // stages issued so far
    bool ok = true;
    int ab_r = -1;      // request whose abort flag is cached
    bool ab = false;
    while (ok && next_piece(cur, a, T, W, p)) {
      const int32_t* ptrow = a.page_table + static_cast<int64_t>(p.r) * a.max_pages;
      const int nst = (p.t1 - p.t0 + 1) >> 1;
      auto load_id = [&](int k0) {
        int pg = -1;
        if (si < batch && k0 + si < nst) {
          const int t = p.t0 + 2 * (k0 + si) + ci;
          if (t < p.t1) pg = __ldg(ptrow + t / tpp);
        }
        return pg;
      };
      int pg = load_id(0);  // table reads only: harmless for an aborted request
      if (p.r != ab_r) {
        ab_r = p.r;
        ab = is_aborted(a, p.r);
      }
      if (ab) continue;  // the consumers skip it too
      for (int k0 = 0; k0 < nst && ok; k0 += batch) {
        const int cnt = min(batch, nst - k0);
        const int nxt = load_id(k0 + batch);  // prefetch (unused past the piece)
        const bool member = si < cnt;
        const int tA = p.t0 + 2 * (k0 + si);
        const bool hasB = tA + 1 < p.t1;
        const int pgA = __shfl_sync(kFull, pg, lane & ~1);
        const int pgB = __shfl_sync(kFull, pg, lane | 1);
        const bool okA = pgA >= 0 && pgA < a.num_pages;
        const bool okB = hasB && pgB >= 0 && pgB < a.num_pages;
        const bool pair = okA && okB && tA / tpp == (tA + 1) / tpp;  // adjacent tiles of one page
        const uint32_t jj = j + si;
        const uint32_t stage = jj % depth;
        const uint32_t round = jj / depth;
        const uint32_t fb = full0 + 8 * stage;
        bool todo = member;
        bool ready = false;
        bool issued = false;
        const uint64_t t0 = global_timer_ns();
        uint32_t spins = 0;
        while (__any_sync(kFull, todo)) {
          if (todo && ci == 0 && !ready &&
              (round == 0 || mbar_test(empty0 + 8 * stage, (round - 1) & 1))) {
            ready = true;
            s_stage_fault[stage] = (okA ? 0 : 1) | ((hasB && !okB) ? 2 : 0);
            const uint32_t bytes = (okA ? 2u * C::kBlockBytes : 0u) + (okB ? 2u * C::kBlockBytes : 0u);
            if (bytes == 0) mbar_arrive(fb);
            else mbar_arrive_expect_tx(fb, bytes);
          }
          __syncwarp();
          const bool go = __shfl_sync(kFull, ready, lane & ~1) && todo;
          if (go) {
            todo = false;
            issued = true;
            const uint32_t dst = smem_addr(ring + stage * C::kStageBytes) + ci * 2 * C::kBlockBytes;
            const int t = tA + ci;
            const int64_t blk = (static_cast<int64_t>(ci == 0 ? pgA : pgB) * a.Hkv + p.h) * tpp + t % tpp;
            const uint8_t* src = a.kv_pool + blk * 2 * C::kBlockBytes;
            if (pair) {
              if (ci == 0) bulk_g2s(dst, src, 4 * C::kBlockBytes, fb, pol);
            } else if (ci == 0 ? okA : okB) {
              bulk_g2s(dst, src, 2 * C::kBlockBytes, fb, pol);
            }
          }
          // the give-up decision is taken by lane 0 for the whole warp
          const bool late = (++spins & 255u) == 0u && global_timer_ns() - t0 > kWaitLimitNs;
          if (__shfl_sync(kFull, late, 0)) {
            if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
            ok = false;
            break;
          }
        }
        if (!ok) {
          // this batch's copies that did go out must land before the CTA exits
          if (issued && ci == 0) mbar_wait(fb, round & 1, a.status);
          break;
        }
        j += cnt;
        pg = nxt;
      }
    }
    if (!ok && lane == 0) {
      // give in-flight copies (bounded) time to land before the CTA exits
      for (uint32_t s = 0; s < depth && s < j; ++s) {
        const uint32_t issued = (j - 1 - s) / depth + 1;
        mbar_wait(full0 + 8 * s, (issued - 1) & 1, a.status);
      }
    }
    return;
  }

  // ======================= consumer warps =======================
  const int c = warp - 1;
  constexpr int nslots = C::kMergeSlots;
  static_assert(nslots == kConsumerWarps || nslots == 2, "the merge takes four slots or two");
  float* const s_mo = s_o;
  const int g = lane >> 2;   // MMA group id: A row / B column
  const int t4 = lane & 3;   // thread in group
  const int rowA = token_of_row(g);  // token of fragment row g (row g+8 is rowA + 2)
  const float kscale = kFp8 ? __ldg(a.k_scale) : 1.f;
  const float vscale = kFp8 ? __ldg(a.v_scale) : 1.f;
  const float vmul = kFp8 ? vscale : 1.f;
  Cursor cur = start;
  Piece p;
  uint32_t jbase = 0;
  uint32_t piece_idx = 0;
  uint32_t cphase = 0;  // completed phases of cbar
  const int ct_all = c * 32 + lane;  // consumer thread 0..127
  bool ok = true;
  const float kNegInf = -INFINITY;
  // barrier of the four consumer warps (bounded wait); false if it gave up
  auto consumer_sync = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive(cbar);
    const bool got = mbar_wait(cbar, cphase & 1, a.status);
    ++cphase;
    return __all_sync(kFull, got);
  };
  // Arrival ticket on a counter in global memory: one acquire-release atomic
  // by consumer thread 0 after a barrier of the consumer warps, so every
  // partial this CTA wrote before the barrier is visible to the CTA whose
  // atomic completes `count`, and that CTA, after its own barrier, sees every
  // other CTA's partials (no thread-wide fences); returns 1 for the arrival
  // that completes `count`, 0 for the others, -1 if a barrier gave up.
  // Nothing ever waits on another CTA.
  auto ticket = [&](int* ctr, int count, int arrivals) -> int {
    if (!consumer_sync()) return -1;
    if (ct_all == 0) s_last = atom_add_acq_rel_gpu(ctr, arrivals) + arrivals == count;
    if (!consumer_sync()) return -1;
    return s_last;
  };
  // Log-sum-exp of n partials (unnormalised sums with their (M, l) pairs in
  // the log2 domain), taken from slots slot_of(k) for k < n, a chunk of slots
  // at a time: the chunk's (m, l) pairs are staged in shared memory, one
  // thread per head turns them into weights e^(m - M) against the running
  // maximum M (rescaling the running sums when M grows), then every thread
  // accumulates weight x partial for one float4 of dims of two heads.  Head
  // indices past the group are clamped rather than branched on, so the loads
  // of several slots are in flight together.  The result goes to the final
  // output rows of (r, h) when dst < 0, else, as a partial, to slot dst.
  // Staged: once the CTA has no piece left its ring is idle, and when the n
  // partials fit there they arrive by bulk copies (one per partial, issued
  // from separate lanes) while the (m, l) pairs load; the sums are then taken
  // from shared memory.  Measured on 16 partials (64 KiB) in a one-request
  // launch: 8.4 us for the combine by batches of register loads, 10.2 us with
  // cp.async into shared memory, 6.5-7 us by bulk copies.
  uint32_t comb_phase = 0;  // staged combines so far (the parity of comb_bar)
  auto combine = [&](const Members& mb, int n, int r, int h, int64_t dst, bool ring_idle) -> bool {
    auto slot_of = [&](int k) -> int64_t {
      const int i = mb.i0 + k * mb.stride;
      return mb.seg + (mb.dense ? mb.w0 + i : worker_of(mb.xseg + i, T, W));
    };
    float2* s_w = reinterpret_cast<float2*>(s_o);
    constexpr int kChunk = C::kMergeSlots * kGroupMax * kMergeStride / (2 * kGroupMax);
    float* s_M = s_m;              // running maximum per head
    float* s_r = s_m + kGroupMax;  // rescale of the running sums by this chunk
    float* s_W = s_l;              // running sum of weights per head
    int* s_dead = s_wfault;        // some split faulted
    const int ct = ct_all;
    const int d4 = ct & 31;
    const int hq0 = ct >> 5;  // heads hq0 and hq0 + 4
    const int hh0 = min(hq0, a.G - 1);
    const int hh1 = min(hq0 + 4, a.G - 1);
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
    if (ct < kGroupMax) {
      s_M[ct] = kNegInf;
      s_W[ct] = 0.f;
    }
    if (ct == 0) *s_dead = 0;
    const uint32_t pbytes = static_cast<uint32_t>(a.G) * kDim * 4;  // one partial
    const bool staged = ring_idle && n <= kChunk && n * pbytes <= static_cast<uint32_t>(C::kRingBytes);
    if (staged) {
      if (c == 0) {
        if (lane == 0) mbar_arrive_expect_tx(comb_bar, n * pbytes);
        __syncwarp();
        // the partials were written through the generic proxy; the copies read them through the async one
        asm volatile("fence.proxy.async.global;" ::: "memory");
        const uint64_t pol = l2_policy_evict_first();
        for (int i = lane; i < n; i += 32)
          bulk_g2s(smem_addr(ring) + i * pbytes, a.part_o + slot_of(i) * a.G * kDim, pbytes, comb_bar, pol);
      }
      for (int e = ct; e < n * a.G; e += kConsumerWarps * 32) {
        const int i = e / a.G;
        const int hd = e - i * a.G;
        s_w[i * kGroupMax + hd] = __ldcg(a.part_ml + slot_of(i) * a.G + hd);
      }
      const bool got = mbar_wait(comb_bar, comb_phase & 1, a.status);
      ++comb_phase;
      if (!__all_sync(kFull, got)) {
        // the copies must land (bounded) before the CTA exits
        if (c == 0 && lane == 0) mbar_wait(comb_bar, (comb_phase - 1) & 1, a.status);
        return false;
      }
      if (!consumer_sync()) return false;
      if (ct < a.G) {
        float mn = kNegInf;
        bool dd = false;
        for (int i = 0; i < n; ++i) {
          const float2 ml = s_w[i * kGroupMax + ct];
          mn = fmaxf(mn, ml.x);
          dd |= ml.y < 0.f;
        }
        float wsum = 0.f;
        for (int i = 0; i < n; ++i) {
          const float2 ml = s_w[i * kGroupMax + ct];
          const float f = ml.x == kNegInf ? 0.f : fast_exp2(ml.x - mn);
          wsum = fmaf(ml.y, f, wsum);
          s_w[i * kGroupMax + ct].x = f;
        }
        s_M[ct] = mn;
        s_W[ct] = wsum;
        if (dd) *s_dead = 1;
      }
      if (!consumer_sync()) return false;
      const float4* po = reinterpret_cast<const float4*>(ring);
      for (int i = 0; i < n; ++i) {
        const float f0 = s_w[i * kGroupMax + hh0].x;
        const float f1 = s_w[i * kGroupMax + hh1].x;
        const float4 v0 = po[(i * a.G + hh0) * (kDim / 4) + d4];
        const float4 v1 = po[(i * a.G + hh1) * (kDim / 4) + d4];
        acc0 = make_float4(fmaf(v0.x, f0, acc0.x), fmaf(v0.y, f0, acc0.y), fmaf(v0.z, f0, acc0.z),
                           fmaf(v0.w, f0, acc0.w));
        acc1 = make_float4(fmaf(v1.x, f1, acc1.x), fmaf(v1.y, f1, acc1.y), fmaf(v1.z, f1, acc1.z),
                           fmaf(v1.w, f1, acc1.w));
      }
      // every thread has read the ring before a later combine of this CTA refills it
      if (!consumer_sync()) return false;
    }
    for (int c0 = 0; !staged && c0 < n; c0 += kChunk) {
      const int nc = min(kChunk, n - c0);
      for (int e = ct; e < nc * a.G; e += kConsumerWarps * 32) {
        const int i = e / a.G;
        const int hd = e - i * a.G;
        s_w[i * kGroupMax + hd] = __ldcg(a.part_ml + slot_of(c0 + i) * a.G + hd);
      }
      if (!consumer_sync()) return false;
      if (ct < a.G) {
        float mc = kNegInf;
        bool dd = false;
        for (int i = 0; i < nc; ++i) {
          const float2 ml = s_w[i * kGroupMax + ct];
          mc = fmaxf(mc, ml.x);
          dd |= ml.y < 0.f;
        }
        const float mo = s_M[ct];
        const float mn = fmaxf(mo, mc);
        const float rs = mo == kNegInf ? 0.f : fast_exp2(mo - mn);
        float wsum = s_W[ct] * rs;
        for (int i = 0; i < nc; ++i) {
          const float2 ml = s_w[i * kGroupMax + ct];
          const float f = ml.x == kNegInf ? 0.f : fast_exp2(ml.x - mn);
          wsum = fmaf(ml.y, f, wsum);
          s_w[i * kGroupMax + ct].x = f;
        }
        s_M[ct] = mn;
        s_r[ct] = rs;
        s_W[ct] = wsum;
        if (dd) *s_dead = 1;
      }
      if (!consumer_sync()) return false;
      {
        const float r0 = s_r[hh0], r1 = s_r[hh1];
        acc0 = make_float4(acc0.x * r0, acc0.y * r0, acc0.z * r0, acc0.w * r0);
        acc1 = make_float4(acc1.x * r1, acc1.y * r1, acc1.z * r1, acc1.w * r1);
      }
      // the slots' loads are issued four at a time, all before their FMAs:
      // the partials sit in L2, and one slot per round trip made the combine
      // of 16 partials eight dependent L2 round trips
      for (int i0 = 0; i0 < nc; i0 += 4) {
        float4 v0[4], v1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = min(i0 + j, nc - 1);  // past the end: a repeated load, not used
          const float4* po = reinterpret_cast<const float4*>(a.part_o + slot_of(c0 + i) * a.G * kDim);
          v0[j] = __ldcg(po + hh0 * (kDim / 4) + d4);
          v1[j] = __ldcg(po + hh1 * (kDim / 4) + d4);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (i0 + j < nc) {
            const float f0 = s_w[(i0 + j) * kGroupMax + hh0].x;
            const float f1 = s_w[(i0 + j) * kGroupMax + hh1].x;
            acc0 = make_float4(fmaf(v0[j].x, f0, acc0.x), fmaf(v0[j].y, f0, acc0.y),
                               fmaf(v0[j].z, f0, acc0.z), fmaf(v0[j].w, f0, acc0.w));
            acc1 = make_float4(fmaf(v1[j].x, f1, acc1.x), fmaf(v1[j].y, f1, acc1.y),
                               fmaf(v1[j].z, f1, acc1.z), fmaf(v1[j].w, f1, acc1.w));
          }
        }
      }
      // every thread is done with this chunk's weights before the next overwrites them
      if (c0 + kChunk < n && !consumer_sync()) return false;
    }
    const bool dead = *s_dead != 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int hd = hq0 + 4 * j;
      if (hd < a.G) {
        const float W = s_W[hd];
        const float4 av = j == 0 ? acc0 : acc1;
        if (dst < 0) {
          const bool dh = dead || W == 0.f;
          const float iw = dh ? 0.f : 1.f / W;
          const int64_t row = static_cast<int64_t>(r) * a.Hq + h * a.G + hd;
          reinterpret_cast<float4*>(a.out + row * kDim)[d4] =
              make_float4(av.x * iw, av.y * iw, av.z * iw, av.w * iw);
          if (d4 == 0 && a.lse != nullptr) a.lse[row] = dh ? kNegInf : (s_M[hd] + __log2f(W)) * kLn2;
        } else {
          // each thread overwrites only the dims it read itself; the (m, l)
          // pairs were all read before the last barrier
          reinterpret_cast<float4*>(a.part_o + (dst * a.G + hd) * kDim)[d4] = av;
          if (d4 == 0)
            a.part_ml[dst * a.G + hd] = dead ? make_float2(kNegInf, -1.f)
                                             : make_float2(W == 0.f ? kNegInf : s_M[hd], W);
        }
      }
    }
    return true;
  };
  // A piece that is not a whole segment has written its partial to its slot.
  // Members of the segment are numbered i = 0..nsl-1 in tile order.  Up to
  // kDirect members, the arrival that completes the segment's count combines
  // them all.  Beyond that the members form groups of K ~ sqrt(nsl): the
  // arrival completing a group folds it into the slot of its first member,
  // and the group completing the segment's count combines the group results,
  // so no CTA reads more than about max(K, nsl / K) partials.
  // A CTA's consecutive pieces that count on the same counter (consecutive
  // splits of one segment or group) arrive together: one fenced atomic adds
  // them all, when the next piece counts elsewhere or the CTA is done.
  struct Pending {
    int* ctr;
    int n, k, K, ng, r, h, seg;
    int64_t dst;
    Members mb;
  };
  auto pending_of = [&](const Piece& p, int seg) -> Pending {
    constexpr int kDirect = 16;
    const int64_t xseg = p.x0 - p.t0;  // global index of the segment's first tile
    // splits holding a piece of this segment: all of w0..w1 when every split
    // owns tiles (T >= W), else one per tile (the i-th is the owner of tile i);
    // in the segment-aligned partition, its own run of splits
    const int w0 = aligned ? s_start[5] : worker_of(xseg, T, W);
    const int w1 = aligned ? s_start[5] + s_start[6] - 1 : worker_of(xseg + p.n - 1, T, W);
    const bool dense = aligned || T >= W;
    const int nsl = dense ? w1 - w0 + 1 : p.n;
    const int me = dense ? p.s - w0 : p.t0;
    Pending q;
    q.mb.seg = seg;
    q.mb.xseg = xseg;
    q.mb.w0 = w0;
    q.mb.dense = dense;
    q.mb.i0 = 0;
    q.mb.stride = 1;
    q.ctr = a.seg_count + seg;
    q.n = nsl;
    q.dst = -1;
    q.K = 1;
    q.ng = 1;
    q.k = 1;
    q.r = p.r;
    q.h = p.h;
    q.seg = seg;
    if (nsl > kDirect) {
      int K = static_cast<int>(sqrtf(static_cast<float>(nsl)));
      while (K * K < nsl) ++K;
      q.K = K;
      q.ng = (nsl + K - 1) / K;
      const int gi = me / K;
      q.mb.i0 = gi * K;
      q.n = min(K, nsl - q.mb.i0);
      q.dst = seg + (dense ? w0 + q.mb.i0 : worker_of(xseg + q.mb.i0, T, W));
      q.ctr = a.group_count + q.dst;
    }
    return q;
  };
  // the pending arrivals: ticket, and the combines they complete
  // (ring_idle: the CTA has no piece left, see combine)
  auto flush = [&](Pending q, bool ring_idle) -> bool {
    int arrivals = q.k;
    for (;;) {
      const int last = ticket(q.ctr, q.n, arrivals);
      if (last < 0) return false;
      if (last == 0) return true;
      if (!combine(q.mb, q.n, q.r, q.h, q.dst, ring_idle)) return false;
      if (ct_all == 0) *q.ctr = 0;  // ready for the next call
      if (q.dst < 0) return true;
      // the group is folded into the slot of its first member: on to the
      // segment's count of groups
      q.ctr = a.seg_count + q.seg;
      q.n = q.ng;
      q.dst = -1;
      q.mb.i0 = 0;
      q.mb.stride = q.K;
      arrivals = 1;
    }
  };
  // The pending arrivals live in shared memory (the same for every consumer
  // thread): the piece that opened them and their count.  Consumer thread 0
  // updates them only after a barrier that every reader has passed.
  auto publish_partial = [&](const Piece& p, int seg) -> bool {
    int* const ctr = pending_of(p, seg).ctr;
    const int pk = s_pend_k;
    const bool same = pk > 0 && s_pend_ctr == ctr;
    if (pk > 0 && !same) {
      Pending q = pending_of(s_pend_piece, s_pend_seg);
      q.k = pk;
      if (!flush(q, false)) return false;  // its barriers follow every thread's reads above
    } else if (!consumer_sync()) {
      return false;
    }
    if (ct_all == 0) {
      if (same) {
        s_pend_k = pk + 1;
      } else {
        s_pend_piece = p;
        s_pend_seg = seg;
        s_pend_ctr = ctr;
        s_pend_k = 1;
      }
    }
    return true;
  };

  zero_dead_rows(ct_all, kConsumerWarps * 32);
  int ab_r = -1;  // request whose abort flag is cached
  bool ab = false;
  int q_r = -1, q_h = -1;  // segment whose query fragments qf hold
  uint32_t qf[8][2];
  float mult_own = 0.f;
  while (ok && next_piece(cur, a, T, W, p)) {
    if (p.r != ab_r) {
      ab_r = p.r;
      ab = is_aborted(a, p.r);  // used after the query loads below are issued
    }
    const int ntiles = p.t1 - p.t0;
    const int L = __ldg(a.seq_lens + p.r);
    // ---- query fragments (B operand of S^T = K Q^T), heads of this kv group;
    // kept from the previous piece when it was of the same segment
    if (p.r != q_r || p.h != q_h) {
      q_r = p.r;
      q_h = p.h;
      const bool has = g < a.G;
      const uint16_t* qrow = a.q + (static_cast<int64_t>(p.r) * a.Hq + p.h * a.G + (has ? g : 0)) * kDim;
      if (kFp8) {
        float v[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (has) raw = __ldg(reinterpret_cast<const uint4*>(qrow + 64 * cc + 16 * t4 + 8 * hh));
            const uint16_t* e = reinterpret_cast<const uint16_t*>(&raw);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[16 * cc + 8 * hh + k] = bf16_bits_to_float(e[k]);
          }
        }
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
        // power-of-two prescale taking the head's largest |q| into [2^14, 2^15)
        int e2 = 0;
        if (amax > 0.f && isfinite(amax)) e2 = min(max(14 - ilogbf(amax), -126), 126);
        const float sc = __int_as_float((127 + e2) << 23);
        const float isc = __int_as_float((127 - e2) << 23);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int o = 16 * (kk >> 2) + 4 * (kk & 3);
          qf[kk][0] = pack_f16x2(v[o] * sc, v[o + 1] * sc);
          qf[kk][1] = pack_f16x2(v[o + 2] * sc, v[o + 3] * sc);
        }
        mult_own = has ? kscale * a.sm_scale_log2 * isc : 0.f;
      } else {
        uint4 raw[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          raw[cc] = make_uint4(0, 0, 0, 0);
          if (has) raw[cc] = __ldg(reinterpret_cast<const uint4*>(qrow + 32 * cc + 8 * t4));
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qf[kk][0] = word_of(raw[kk >> 1], 2 * (kk & 1));
          qf[kk][1] = word_of(raw[kk >> 1], 2 * (kk & 1) + 1);
        }
        mult_own = has ? a.sm_scale_log2 : 0.f;
      }
    }
    if (ab) continue;  // output zeroed above; nothing read
    // score multipliers of the two heads (2*t4, 2*t4+1) whose columns this lane holds
    const float mult0 = __shfl_sync(kFull, mult_own, 8 * t4);
    const float mult1 = __shfl_sync(kFull, mult_own, 8 * t4 + 4);

    float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    int fault = 0;
    const int nst = (ntiles + 1) >> 1;  // stages of this piece, two tiles each

    // ring position of stage k of this piece, advanced by the warp count
    uint32_t stage = (jbase + c) % depth;
    uint32_t round = (jbase + c) / depth;
    for (int k = c; k < nst; k += kConsumerWarps) {
      if (k != c) {
        stage += kConsumerWarps;
        if (stage >= depth) {
          stage -= depth;
          ++round;
        }
      }
      const bool got = mbar_wait(full0 + 8 * stage, round & 1, a.status);
      if (!__all_sync(kFull, got)) {
        ok = false;
        break;
      }
      const int fbits = s_stage_fault[stage];
      fault |= fbits;
      const uint8_t* Sb = ring + stage * C::kStageBytes;  // [K0][V0][K1][V1]
      const int tA = p.t0 + 2 * k;
      // tokens of each tile that take part: 0 for a tile past the piece or on a bad page
      int nv[2];
      nv[0] = (fbits & 1) ? 0 : min(kTile, L - tA * kTile);
      nv[1] = (tA + 1 >= p.t1 || (fbits & 2)) ? 0 : min(kTile, L - (tA + 1) * kTile);
      // ---- FP8: copy this lane's K and V operands of both tiles to registers
      // and hand the stage back at once, so the producer refills it while the
      // math below runs (the bf16 operands are twice as large and stay in
      // shared memory until the stage's math is done)
      uint4 kr[2][4];
      uint32_t vr[2][8][2];
      if (kFp8) {
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          const uint8_t* Ks = Sb + 2 * tt * C::kBlockBytes;
          const uint8_t* Vs = Ks + C::kBlockBytes;
          kr[tt][0] = lds128(Ks + rowA * kDim + 16 * t4);
          kr[tt][1] = lds128(Ks + rowA * kDim + 64 + 16 * t4);
          kr[tt][2] = lds128(Ks + (rowA + 2) * kDim + 16 * t4);
          kr[tt][3] = lds128(Ks + (rowA + 2) * kDim + 64 + 16 * t4);
          // V operand words by ldmatrix: four 8 x 8 b16 blocks of dim rows
          // (16 bytes each) per load; lane 8i + r gives the address of row r
          // of block i, and lane 4g + t receives bytes 4t .. 4t+3 of row g of
          // every block, i.e. tokens 4t .. 4t+3 of one dim
#pragma unroll
          for (int mt = 0; mt < 8; mt += 2) {
            const int dim = 16 * mt + 8 * (lane >> 3) + (lane & 7);
            ldmatrix_x4(smem_addr(Vs + dim * 16), vr[tt][mt][0], vr[tt][mt][1], vr[tt][mt + 1][0],
                        vr[tt][mt + 1][1]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);
      }
      // ---- S^T = K Q^T for both tiles (rows: tokens, cols: heads); four independent chains
      float sc[2][4];
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t af[4];
          if (kFp8) {
            const uint32_t wa = word_of(kr[tt][kk >> 2], kk & 3);
            const uint32_t wb = word_of(kr[tt][2 + (kk >> 2)], kk & 3);
            e4m3x4_to_f16x4(wa, af[0], af[2]);
            e4m3x4_to_f16x4(wb, af[1], af[3]);
            if (kk & 1) mma_f16(acc1, af, qf[kk][0], qf[kk][1]);
            else mma_f16(acc0, af, qf[kk][0], qf[kk][1]);
          } else {
            const uint8_t* Ks = Sb + 2 * tt * C::kBlockBytes;
            const int wi = 2 * (kk & 1);
            const uint4 ka = lds128(Ks + rowA * 2 * kDim + 64 * (kk >> 1) + 16 * t4);
            const uint4 kb = lds128(Ks + (rowA + 2) * 2 * kDim + 64 * (kk >> 1) + 16 * t4);
            af[0] = word_of(ka, wi);
            af[1] = word_of(kb, wi);
            af[2] = word_of(ka, wi + 1);
            af[3] = word_of(kb, wi + 1);
            if (kk & 1) mma_bf16(acc1, af, qf[kk][0], qf[kk][1]);
            else mma_bf16(acc0, af, qf[kk][0], qf[kk][1]);
          }
        }
        sc[tt][0] = (acc0[0] + acc1[0]) * mult0;
        sc[tt][1] = (acc0[1] + acc1[1]) * mult1;
        sc[tt][2] = (acc0[2] + acc1[2]) * mult0;
        sc[tt][3] = (acc0[3] + acc1[3]) * mult1;
        if (nv[tt] < kTile) {
          // select, never multiply: a stale slot may hold NaN codes
          if (rowA >= nv[tt]) sc[tt][0] = sc[tt][1] = kNegInf;
          if (rowA + 2 >= nv[tt]) sc[tt][2] = sc[tt][3] = kNegInf;
        }
      }
      // ---- online softmax (log2 domain), per head over the stage's 32 tokens
      float tm0 = fmaxf(fmaxf(sc[0][0], sc[0][2]), fmaxf(sc[1][0], sc[1][2]));
      float tm1 = fmaxf(fmaxf(sc[0][1], sc[0][3]), fmaxf(sc[1][1], sc[1][3]));
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        tm0 = fmaxf(tm0, __shfl_xor_sync(kFull, tm0, off));
        tm1 = fmaxf(tm1, __shfl_xor_sync(kFull, tm1, off));
      }
      const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);
      if (__any_sync(kFull, mn0 > m0 || mn1 > m1)) {
        const float al0 = mn0 == m0 ? 1.f : fast_exp2(m0 - mn0);
        const float al1 = mn1 == m1 ? 1.f : fast_exp2(m1 - mn1);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
        l0 *= al0;
        l1 *= al1;
        m0 = mn0;
        m1 = mn1;
      }
      const float base0 = m0 == kNegInf ? 0.f : m0, base1 = m1 == kNegInf ? 0.f : m1;
      // ---- P^T as the B operand of O^T = V^T P^T, per tile, as P = hi + lo:
      // two f16 (FP8 cache) or bf16 (BF16 cache) parts.  One f16 P alone
      // errs by up to 2^-12 of each p, which reaches the 2e-3 absolute
      // tolerance on outlier channels where the output is small against |V|.
      uint32_t pb[2][2], pl[2][2];
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const float p0 = fast_exp2(sc[tt][0] - base0), p1 = fast_exp2(sc[tt][1] - base1);
        const float p2 = fast_exp2(sc[tt][2] - base0), p3 = fast_exp2(sc[tt][3] - base1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        const uint32_t pr0 = kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
        const uint32_t pr1 = kFp8 ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3);
        pb[tt][0] = movmatrix_trans(pr0);
        pb[tt][1] = movmatrix_trans(pr1);
        if (kFp8) {
          const float2 h0 = __half22float2(*reinterpret_cast<const __half2*>(&pr0));
          const float2 h1 = __half22float2(*reinterpret_cast<const __half2*>(&pr1));
          pl[tt][0] = movmatrix_trans(pack_f16x2(p0 - h0.x, p1 - h0.y));
          pl[tt][1] = movmatrix_trans(pack_f16x2(p2 - h1.x, p3 - h1.y));
        } else {
          pl[tt][0] = movmatrix_trans(pack_bf16x2(p0 - __uint_as_float(pr0 << 16),
                                                  p1 - __uint_as_float(pr0 & 0xffff0000u)));
          pl[tt][1] = movmatrix_trans(pack_bf16x2(p2 - __uint_as_float(pr1 << 16),
                                                  p3 - __uint_as_float(pr1 & 0xffff0000u)));
        }
      }
      // ---- O^T += V^T P^T (V columns past the context are zeroed: stale slots may hold NaN codes)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const int nvt = nv[tt] - 4 * t4;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          if (kFp8) {
            uint32_t va = vr[tt][mt][0], vb = vr[tt][mt][1];
            if (nvt < 4) {
              const uint32_t keep = nvt <= 0 ? 0u : (0xffffffffu >> (8 * (4 - nvt)));
              va &= keep;
              vb &= keep;
            }
            uint32_t af[4];
            e4m3x4_to_f16x4(va, af[0], af[2]);
            e4m3x4_to_f16x4(vb, af[1], af[3]);
            mma_f16(o[mt], af, pb[tt][0], pb[tt][1]);
            mma_f16(o[mt], af, pl[tt][0], pl[tt][1]);
          } else {
            const uint8_t* Vs = Sb + (2 * tt + 1) * C::kBlockBytes;
            const uint2 va = *reinterpret_cast<const uint2*>(Vs + (16 * mt + g) * 32 + 8 * t4);
            const uint2 vb = *reinterpret_cast<const uint2*>(Vs + (16 * mt + g + 8) * 32 + 8 * t4);
            uint32_t af[4] = {va.x, vb.x, va.y, vb.y};
            if (nvt < 4) {
              const uint32_t k0 = nvt <= 0 ? 0u : nvt == 1 ? 0x0000ffffu : 0xffffffffu;
              const uint32_t k1 = nvt <= 2 ? 0u : nvt == 3 ? 0x0000ffffu : 0xffffffffu;
              af[0] &= k0;
              af[1] &= k0;
              af[2] &= k1;
              af[3] &= k1;
            }
            mma_bf16(o[mt], af, pb[tt][0], pb[tt][1]);
            mma_bf16(o[mt], af, pl[tt][0], pl[tt][1]);
          }
        }
      }
      if (!kFp8) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);
      }
    }
    jbase += nst;
    if (!ok) break;

    // ---- merge the consumer warps' (m, l, O) of this piece.  Four slots:
    // every warp fills its own and the output loop below combines them.  Two
    // slots: warps 2, 3 are folded into warps 0, 1, whose results go back
    // into the two slots for the output loop.
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, off);
      l1 += __shfl_xor_sync(kFull, l1, off);
    }
    fault = __any_sync(kFull, fault);
    if (piece_idx > 0) {
      const bool got = mbar_wait(merge_free, (piece_idx - 1) & 1, a.status);
      if (!__all_sync(kFull, got)) break;
    }
    // this lane's (m, l, O) into slot sl
    auto put = [&](int sl) {
      float* mo = s_mo + sl * kGroupMax * kMergeStride;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        mo[(2 * t4) * kMergeStride + 16 * mt + g] = o[mt][0];
        mo[(2 * t4 + 1) * kMergeStride + 16 * mt + g] = o[mt][1];
        mo[(2 * t4) * kMergeStride + 16 * mt + g + 8] = o[mt][2];
        mo[(2 * t4 + 1) * kMergeStride + 16 * mt + g + 8] = o[mt][3];
      }
      if (g == 0) {
        s_m[sl * kGroupMax + 2 * t4] = m0;
        s_m[sl * kGroupMax + 2 * t4 + 1] = m1;
        s_l[sl * kGroupMax + 2 * t4] = l0;
        s_l[sl * kGroupMax + 2 * t4 + 1] = l1;
      }
      if (lane == 0) s_wfault[sl] = fault;
      __syncwarp();
    };
    // log-sum-exp of slot sl's (m, l, O) into this lane's
    auto take = [&](int sl) {
      const float* mo = s_mo + sl * kGroupMax * kMergeStride;
      const float n0 = s_m[sl * kGroupMax + 2 * t4], n1 = s_m[sl * kGroupMax + 2 * t4 + 1];
      const float M0 = fmaxf(m0, n0), M1 = fmaxf(m1, n1);
      const float a0 = m0 == kNegInf ? 0.f : fast_exp2(m0 - M0), a1 = m1 == kNegInf ? 0.f : fast_exp2(m1 - M1);
      const float b0 = n0 == kNegInf ? 0.f : fast_exp2(n0 - M0), b1 = n1 == kNegInf ? 0.f : fast_exp2(n1 - M1);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] = fmaf(mo[(2 * t4) * kMergeStride + 16 * mt + g], b0, o[mt][0] * a0);
        o[mt][1] = fmaf(mo[(2 * t4 + 1) * kMergeStride + 16 * mt + g], b1, o[mt][1] * a1);
        o[mt][2] = fmaf(mo[(2 * t4) * kMergeStride + 16 * mt + g + 8], b0, o[mt][2] * a0);
        o[mt][3] = fmaf(mo[(2 * t4 + 1) * kMergeStride + 16 * mt + g + 8], b1, o[mt][3] * a1);
      }
      l0 = fmaf(s_l[sl * kGroupMax + 2 * t4], b0, l0 * a0);
      l1 = fmaf(s_l[sl * kGroupMax + 2 * t4 + 1], b1, l1 * a1);
      m0 = M0;
      m1 = M1;
      fault |= s_wfault[sl];
      __syncwarp();  // every lane has read the slot before any lane writes it
    };
    auto arrive_wait = [&](uint32_t arrive_bar, uint32_t wait_bar) -> bool {
      if (arrive_bar != 0u && lane == 0) mbar_arrive(arrive_bar);
      if (wait_bar == 0u) return true;
      return __all_sync(kFull, mbar_wait(wait_bar, piece_idx & 1, a.status));
    };
    {
      bool got = true;
      if constexpr (nslots == kConsumerWarps) {
        put(c);
        got = arrive_wait(mrg4, mrg4);
      } else if (c >= 2) {
        put(c - 2);
        got = arrive_wait(mrg0, mrg2);
      } else {
        got = arrive_wait(0u, mrg0);
        if (got) {
          take(c);
          got = arrive_wait(mrg1, mrg1);  // both slots read before either is rewritten
          if (got) {
            put(c);
            got = arrive_wait(mrg2, mrg2);
          }
        }
      }
      if (!got) break;
    }
    const int seg = p.r * a.Hkv + p.h;
    const bool whole = p.t0 == 0 && p.t1 == p.n;
    int anyfault = 0;
#pragma unroll
    for (int k = 0; k < nslots; ++k) anyfault |= s_wfault[k];
    {
      // 16 threads per head, 8 consecutive dims each: the slots' weights for
      // the head, then two float4 of each slot
      const int hd = ct_all >> 4;
      const int d0 = (ct_all & 15) * 8;
      if (hd < a.G) {
        float mk[nslots];
        float M = kNegInf;
#pragma unroll
        for (int k = 0; k < nslots; ++k) {
          mk[k] = s_m[k * kGroupMax + hd];
          M = fmaxf(M, mk[k]);
        }
        const bool dead = anyfault || M == kNegInf;
        float wsum = 0.f;
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
#pragma unroll
        for (int k = 0; k < nslots; ++k) {
          const float f = mk[k] == kNegInf ? 0.f : fast_exp2(mk[k] - M);
          wsum = fmaf(s_l[k * kGroupMax + hd], f, wsum);
          const float4* src = reinterpret_cast<const float4*>(s_mo + (k * kGroupMax + hd) * kMergeStride + d0);
          const float4 x0 = src[0], x1 = src[1];
          v0 = make_float4(fmaf(x0.x, f, v0.x), fmaf(x0.y, f, v0.y), fmaf(x0.z, f, v0.z), fmaf(x0.w, f, v0.w));
          v1 = make_float4(fmaf(x1.x, f, v1.x), fmaf(x1.y, f, v1.y), fmaf(x1.z, f, v1.z), fmaf(x1.w, f, v1.w));
        }
        float4* dst;
        float sc;
        if (whole) {
          const int64_t row = static_cast<int64_t>(p.r) * a.Hq + p.h * a.G + hd;
          dst = reinterpret_cast<float4*>(a.out + row * kDim + d0);
          sc = dead ? 0.f : vmul / wsum;
          if (d0 == 0 && a.lse != nullptr) a.lse[row] = dead ? kNegInf : (M + __log2f(wsum)) * kLn2;
        } else {
          const int64_t slot = static_cast<int64_t>(seg) + p.s;
          dst = reinterpret_cast<float4*>(a.part_o + (slot * a.G + hd) * kDim + d0);
          sc = vmul;
          if (d0 == 0) a.part_ml[slot * a.G + hd] = dead ? make_float2(kNegInf, -1.f) : make_float2(M, wsum);
        }
        dst[0] = make_float4(v0.x * sc, v0.y * sc, v0.z * sc, v0.w * sc);
        dst[1] = make_float4(v1.x * sc, v1.y * sc, v1.z * sc, v1.w * sc);
      }
    }
    if (!whole && !publish_partial(p, seg)) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(merge_free);
    ++piece_idx;
  }
  // the last arrivals of this CTA (its shared-memory merge buffers are free:
  // no piece follows)
  if (ok && consumer_sync() && s_pend_k > 0) {
    Pending q = pending_of(s_pend_piece, s_pend_seg);
    q.k = s_pend_k;
    flush(q, true);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
std::atomic<int> g_auto_ctas[3][kMaxDevices];  // resident CTAs per SM: BF16, FP8, deep FP8

template <bool kFp8, bool kDeep = false>
int prepare_kernel(int dev) {
  std::atomic<int>& slot = g_auto_ctas[kDeep ? 2 : kFp8 ? 1 : 0][dev];
  int v = slot.load(std::memory_order_relaxed);
  if (v > 0) return v;
  auto kern = paged_decode_split_kernel<kFp8, kDeep>;
  constexpr int smem = Cfg<kFp8, kDeep>::kSmemBytes;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) !=
          cudaSuccess ||
      per_sm <= 0)
    return -1;
  slot.store(per_sm, std::memory_order_relaxed);
  return per_sm;
}

int auto_splits(int wave, int B, int Hkv) {
  const int64_t cap = static_cast<int64_t>(kAutoSplitsPerSegment) * B * Hkv;
  return cap < wave ? static_cast<int>(cap) : wave;
}

int auto_workers(int dev) {
  const int sms = device_sm_count(dev);
  const int a8 = prepare_kernel<true>(dev);
  const int a16 = prepare_kernel<false>(dev);
  if (sms <= 0 || a8 <= 0 || a16 <= 0) return -1;
  return sms * (a8 > a16 ? a8 : a16);
}

int check_attn_shapes(int B, int Hq, int Hkv, int D, int page_size, int num_pages, int max_pages,
                      int num_splits) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0 || max_pages < 0 ||
      num_splits < 0)
    return FPK_EINVAL;
  if (Hq % Hkv != 0) return FPK_EINVAL;
  const int G = Hq / Hkv;
  if (D != kDim || G > kGroupMax || page_size % kTile != 0 || page_size > 256) return FPK_EUNSUPPORTED;
  return FPK_OK;
}

enum class AttnLaunch { kPlain, kCheckOnly, kAfterStepWrite };

// The deep-ring FP8 variant pays when the CTAs that will have work keep no
// more than kInflightBudget of stages in flight: a grid of at most W CTAs, or
// the split count the kernel takes for a uniform batch (uniform_auto_splits;
// the host cannot see the context lengths and assumes every request holds
// tokens -- if they turn out uneven, the deep variant runs with its shallow
// ring).  It must also fit as many CTAs per SM as the shallow one.
bool deep_ring(int dev, int W, int ctas, int B, int Hkv, bool auto_split) {
  using D = Cfg<true, true>;
  int64_t active = W < ctas ? W : ctas;
  if (auto_split) {
    const int64_t u = uniform_auto_splits(static_cast<int64_t>(B) * Hkv, ctas);
    if (u > 0) active = u;
  }
  if (active * D::kStages * D::kStageBytes > kInflightBudget) return false;
  const int deep = prepare_kernel<true, true>(dev);
  return deep > 0 && deep >= prepare_kernel<true, false>(dev);
}

template <bool kFp8, bool kDeep>
int launch_split_kernel(const AttnArgs& a, int dev, int ctas, cudaStream_t s, bool after_step_write) {
  constexpr int smem = Cfg<kFp8, kDeep>::kSmemBytes;
  if (prepare_kernel<kFp8, kDeep>(dev) <= 0) return FPK_ECUDA;  // sets the kernel's shared-memory size
  if (!after_step_write) {
    paged_decode_split_kernel<kFp8, kDeep><<<ctas, kThreads, smem, s>>>(a);
    return checked_launch_status();
  }
  // launched as a programmatic dependent of the step's write + check kernel:
  // its set-up overlaps that kernel; it reads the mask and the cache only
  // after griddep_wait()
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, paged_decode_split_kernel<kFp8, kDeep>, a) != cudaSuccess) return FPK_ECUDA;
  return checked_launch_status();
}

// Shapes, required pointers and alignment of an attention call; no CUDA call
// is made, so a rejected call has queued nothing.  need_workspace: the caller
// supplies the workspace (the allocation-free entry point does not).
template <bool kFp8>
int check_attn_args(const void* q, const void* kv_pool, const float* k_scale, const float* v_scale,
                    const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                    const float* out, const void* workspace, bool need_workspace, int32_t num_splits,
                    int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                    int32_t num_pages) {
  int st = check_attn_shapes(B, Hq, Hkv, D, page_size, num_pages, max_pages, num_splits);
  if (st != FPK_OK) return st;
  if (B == 0) return FPK_OK;
  if (!q || !kv_pool || !page_table || !seq_lens || !out || (need_workspace && !workspace))
    return FPK_EINVAL;
  if (kFp8 && (!k_scale || !v_scale)) return FPK_EINVAL;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FPK_EINVAL;
  return FPK_OK;
}

template <bool kFp8>
int attn_entry(const void* q, const void* kv_pool, const float* k_scale,
               const float* v_scale, const int32_t* page_table, int32_t max_pages,
               const int32_t* seq_lens, const uint8_t* abort_mask, float* out, float* lse,
               void* workspace, size_t workspace_bytes, int32_t num_splits, float sm_scale,
               int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
               int32_t num_pages, void* stream, AttnLaunch mode = AttnLaunch::kPlain) {
  int st = check_attn_args<kFp8>(q, kv_pool, k_scale, v_scale, page_table, max_pages, seq_lens, out,
                                 workspace, true, num_splits, B, Hq, Hkv, D, page_size, num_pages);
  if (st != FPK_OK || B == 0) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FPK_ECUDA;
  const int per_sm = prepare_kernel<kFp8>(dev);
  const int wave = device_sm_count(dev) * per_sm;  // CTAs resident at once
  if (per_sm <= 0 || wave <= 0) return FPK_ECUDA;
  const int W = num_splits == 0 ? auto_splits(wave, B, Hkv) : num_splits;
  // more splits than a wave: a CTA runs several in turn, as few as the wave
  // allows (k = ceil(W / wave)), and no more CTAs are launched than that
  // count needs -- an equal number of splits per CTA, each CTA with a larger
  // share of the memory system
  const int per_cta = (W + wave - 1) / wave;
  const int ctas = W <= wave ? W : (W + per_cta - 1) / per_cta;
  const int G = Hq / Hkv;
  const WsLayout l = layout(B, Hkv, G, W);
  if (workspace_bytes < l.total) return FPK_ENOSPC;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AttnArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.kv_pool = static_cast<const uint8_t*>(kv_pool);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.abort_mask = abort_mask;
  a.out = out;
  a.lse = lse;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.seg_count = reinterpret_cast<int*>(ws + l.seg_count);
  a.group_count = reinterpret_cast<int*>(ws + l.group_count);
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
  a.sm_scale_log2 = sm_scale * kLog2e;
  if (mode == AttnLaunch::kCheckOnly) return FPK_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kFp8 && deep_ring(dev, W, ctas, B, Hkv, num_splits == 0))
    return launch_split_kernel<true, true>(a, dev, ctas, s, mode == AttnLaunch::kAfterStepWrite);
  return launch_split_kernel<kFp8, false>(a, dev, ctas, s, mode == AttnLaunch::kAfterStepWrite);
}

}  // namespace
}  // namespace fpk

extern "C" size_t fpk_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                             int32_t num_splits) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_splits < 0 || D != fpk::kDim) return 0;
  int W = num_splits;
  if (W == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= fpk::kMaxDevices) return 0;
    W = fpk::auto_workers(dev);
    if (W <= 0) return 0;
  }
  return fpk::layout(B, Hkv, Hq / Hkv, W).total;
}

extern "C" int fpk_paged_decode_attn_fp8(const void* q, const uint8_t* kv_pool,
                                         const float* k_scale, const float* v_scale,
                                         const int32_t* page_table, int32_t max_pages,
                                         const int32_t* seq_lens, const uint8_t* abort_mask,
                                         float* out, float* lse, void* workspace,
                                         size_t workspace_bytes, int32_t num_splits,
                                         float sm_scale, int32_t B, int32_t Hq, int32_t Hkv,
                                         int32_t D, int32_t page_size, int32_t num_pages,
                                         void* stream) {
  return fpk::attn_entry<true>(q, kv_pool, k_scale, v_scale, page_table, max_pages, seq_lens,
                               abort_mask, out, lse, workspace, workspace_bytes, num_splits,
                               sm_scale, B, Hq, Hkv, D, page_size, num_pages, stream);
}

extern "C" int fpk_paged_decode_attn_bf16(const void* q, const void* kv_pool,
                                          const int32_t* page_table, int32_t max_pages,
                                          const int32_t* seq_lens, const uint8_t* abort_mask,
                                          float* out, float* lse, void* workspace,
                                          size_t workspace_bytes, int32_t num_splits,
                                          float sm_scale, int32_t B, int32_t Hq, int32_t Hkv,
                                          int32_t D, int32_t page_size, int32_t num_pages,
                                          void* stream) {
  return fpk::attn_entry<false>(q, kv_pool, nullptr, nullptr, page_table, max_pages, seq_lens,
                                abort_mask, out, lse, workspace, workspace_bytes, num_splits,
                                sm_scale, B, Hq, Hkv, D, page_size, num_pages, stream);
}

extern "C" int fpk_decode_step_fp8(const void* k_new, const void* v_new, uint8_t* kv_pool,
                                   const float* k_scale, const float* v_scale,
                                   const int32_t* page_table, int32_t max_pages,
                                   const int32_t* seq_lens, const uint32_t* live_tags,
                                   const uint32_t* expected_tags, uint8_t* abort_mask, const void* q,
                                   float* out, float* lse, void* workspace, size_t workspace_bytes,
                                   int32_t num_splits, float sm_scale, int32_t B, int32_t Hq,
                                   int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
                                   void* stream) {
  // every argument of both launches is checked before either is issued
  int st = fpk::attn_entry<true>(q, kv_pool, k_scale, v_scale, page_table, max_pages, seq_lens,
                                 abort_mask, out, lse, workspace, workspace_bytes, num_splits,
                                 sm_scale, B, Hq, Hkv, D, page_size, num_pages, stream,
                                 fpk::AttnLaunch::kCheckOnly);
  if (st != FPK_OK) return st;
  if ((live_tags != nullptr || expected_tags != nullptr) && (!live_tags || !expected_tags || !abort_mask))
    return FPK_EINVAL;
  if (live_tags == nullptr) abort_mask = nullptr;  // the no-op tracker: no check, no mask
  st = fpk::append_check_entry(true, k_new, v_new, kv_pool, k_scale, v_scale, page_table, max_pages,
                               seq_lens, live_tags, expected_tags, abort_mask, B, Hkv, D, page_size,
                               num_pages, stream);
  if (st != FPK_OK) return st;
  return fpk::attn_entry<true>(q, kv_pool, k_scale, v_scale, page_table, max_pages, seq_lens,
                               abort_mask, out, lse, workspace, workspace_bytes, num_splits,
                               sm_scale, B, Hq, Hkv, D, page_size, num_pages, stream,
                               fpk::AttnLaunch::kAfterStepWrite);
}

extern "C" int fpk_decode_step_bf16(const void* k_new, const void* v_new, void* kv_pool,
                                    const int32_t* page_table, int32_t max_pages,
                                    const int32_t* seq_lens, const uint32_t* live_tags,
                                    const uint32_t* expected_tags, uint8_t* abort_mask, const void* q,
                                    float* out, float* lse, void* workspace, size_t workspace_bytes,
                                    int32_t num_splits, float sm_scale, int32_t B, int32_t Hq,
                                    int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
                                    void* stream) {
  int st = fpk::attn_entry<false>(q, kv_pool, nullptr, nullptr, page_table, max_pages, seq_lens,
                                  abort_mask, out, lse, workspace, workspace_bytes, num_splits,
                                  sm_scale, B, Hq, Hkv, D, page_size, num_pages, stream,
                                  fpk::AttnLaunch::kCheckOnly);
  if (st != FPK_OK) return st;
  if ((live_tags != nullptr || expected_tags != nullptr) && (!live_tags || !expected_tags || !abort_mask))
    return FPK_EINVAL;
  if (live_tags == nullptr) abort_mask = nullptr;  // the no-op tracker: no check, no mask
  st = fpk::append_check_entry(false, k_new, v_new, kv_pool, nullptr, nullptr, page_table, max_pages,
                               seq_lens, live_tags, expected_tags, abort_mask, B, Hkv, D, page_size,
                               num_pages, stream);
  if (st != FPK_OK) return st;
  return fpk::attn_entry<false>(q, kv_pool, nullptr, nullptr, page_table, max_pages, seq_lens,
                                abort_mask, out, lse, workspace, workspace_bytes, num_splits,
                                sm_scale, B, Hq, Hkv, D, page_size, num_pages, stream,
                               fpk::AttnLaunch::kAfterStepWrite);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the FP8 attention entry point.
//
// Some callers cannot allocate device memory for a workspace: operator hosts
// and plugin interfaces that hand an operator only its inputs and outputs,
// processes held to a fixed device-memory budget, and latency-critical loops
// that cannot afford cudaMalloc's implicit device synchronisation.  For them
// the scratch lives in the file-scope array below, a fixed 16 MiB that every
// GPU loading this library keeps until the process exits.  In host code the
// array's name is only a host-side stand-in, so its device address is looked
// up once per device (with that device current) and passed to the kernel.
// ---------------------------------------------------------------------------
#include <mutex>

namespace fpk {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address, looked up once per device and context: a device
// reset (or a primary context released and retained again) gives the device a
// new context, in which the module and its array are loaded afresh.
struct NoAllocSlot {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_noalloc_mu;
NoAllocSlot g_noalloc_slot[kMaxDevices];

// Identity of the calling thread's current context (0 if it cannot be had):
// the driver's context id, which no later context reuses.
unsigned long long current_context_id() {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != 0 || ctx == nullptr ||
      get_id(ctx, &id) != 0)
    return 0;
  return id;
}

// Set-up, once per device (and context): the scratch array's device address
// on `dev`, which must be the current device.  Without a context id the
// address is looked up on every call.
int noalloc_scratch_address(int dev, void** addr) {
  // before the runtime's first call on this device there may be no current
  // context (id 0); the symbol lookup creates it, so the id kept is read after
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocSlot& slot = g_noalloc_slot[dev];
  const unsigned long long id = current_context_id();
  if (slot.addr == nullptr || id == 0 || slot.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FPK_ECUDA;
    slot.addr = p;
    slot.ctx_id = current_context_id();
  }
  *addr = slot.addr;
  return FPK_OK;
}

}  // namespace
}  // namespace fpk

extern "C" int fpk_paged_decode_attn_fp8_noalloc(const void* q, const uint8_t* kv_pool,
                                                 const float* k_scale,
                                                 const float* v_scale, const int32_t* page_table,
                                                 int32_t max_pages, const int32_t* seq_lens,
                                                 const uint8_t* abort_mask, float* out, float* lse,
                                                 int32_t num_splits, float sm_scale, int32_t B,
                                                 int32_t Hq, int32_t Hkv, int32_t D,
                                                 int32_t page_size, int32_t num_pages,
                                                 void* stream) {
  // every argument is checked before any CUDA call: a rejected call queues nothing
  int st = fpk::check_attn_args<true>(q, kv_pool, k_scale, v_scale, page_table, max_pages, seq_lens,
                                      out, nullptr, false, num_splits, B, Hq, Hkv, D, page_size,
                                      num_pages);
  if (st != FPK_OK || B == 0) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= fpk::kMaxDevices) return FPK_ECUDA;
  void* scratch = nullptr;
  st = fpk::noalloc_scratch_address(dev, &scratch);
  if (st != FPK_OK) return st;
  int W = num_splits;
  if (W == 0) {
    const int per_sm = fpk::prepare_kernel<true>(dev);
    if (per_sm <= 0) return FPK_ECUDA;
    W = fpk::auto_splits(fpk::device_sm_count(dev) * per_sm, B, Hkv);
    if (W <= 0) return FPK_ECUDA;
  }
  const fpk::WsLayout l = fpk::layout(B, Hkv, Hq / Hkv, W);
  if (l.total > fpk::kNoAllocScratchBytes) return FPK_ENOSPC;  // batch too large for the fixed scratch
  // the status word and the arrival counters must start at zero
  if (cudaMemsetAsync(scratch, 0, l.part_ml, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FPK_ECUDA;
  return fpk::attn_entry<true>(q, kv_pool, k_scale, v_scale, page_table, max_pages, seq_lens,
                               abort_mask, out, lse, scratch, fpk::kNoAllocScratchBytes, num_splits, sm_scale,
                               B, Hq, Hkv, D, page_size, num_pages, stream);
}

extern "C" int fpk_decode_status(const void* workspace, int32_t* status, void* stream) {
  if (!status) return FPK_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* src = workspace;
  if (src == nullptr) {
    // the allocation-free entry point's scratch on the current device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= fpk::kMaxDevices) return FPK_ECUDA;
    void* addr = nullptr;
    const int st = fpk::noalloc_scratch_address(dev, &addr);
    if (st != FPK_OK) return st;
    src = addr;
  }
  if (cudaMemcpyAsync(status, src, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FPK_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FPK_ECUDA;
  return FPK_OK;
}
