// attn_plan.cuh -- the work partition and workspace layout shared by the two
// split-KV attention kernels (decode_attn.cu: warp-level MMA; decode_attn_tc.cu:
// tcgen05 MMA with tensor-memory accumulators).
//
// All (request, kv head) segments of a batch are laid end to end as a list of
// 16-token tiles, T tiles in all; the list is cut into W splits of equal tile
// count, split w owning tiles [floor(w T / W), floor((w+1) T / W)).  A CTA
// walks its tile range piece by piece, a piece being the longest run that
// stays inside one segment and one split.  A piece that covers a whole
// segment writes the final output; any other piece writes the partial
// (m, l, O) of its split into slot `segment + split` of the workspace, and the
// segment's partials are merged by log-sum-exp.  The pages (the Cloudflare
// write-up on serving Kimi K2.6 and GLM 5.2) give no kernel design: the split
// scheme is this library's own.
#pragma once

#include <stdint.h>
#include <stddef.h>

#include "common.cuh"

namespace fpk {
namespace {

constexpr int kTile = 16;     // tokens per tile
constexpr int kDim = 128;     // head dimension
constexpr int kGroupMax = 8;  // query heads per kv head (N of the MMA tile)

// The automatic split count: one wave of CTAs, but no more than 16 splits per
// (request, kv head) segment -- small batches then keep the one-level combine
// and CTAs with enough tiles to cover their start-up.
constexpr int kAutoSplitsPerSegment = 16;

// The automatic split count of a batch whose segments all have one length
// (seen on the device, from the context lengths): one whole segment per CTA
// when the segments fill between 3/4 of the CTAs and all of them; with fewer
// segments, the same number of splits for each (as many as the CTAs allow,
// at most kAutoSplitsPerSegment), which puts every split boundary on a
// segment boundary -- no split straddles two segments.  0: keep the count.
__host__ __device__ __forceinline__ int64_t uniform_auto_splits(int64_t segs, int64_t nctas) {
  if (segs <= 0 || segs > nctas) return 0;
  if (4 * segs >= 3 * nctas) return segs;
  int64_t m = nctas / segs;
  if (m > kAutoSplitsPerSegment) m = kAutoSplitsPerSegment;
  return segs * m;
}

struct Piece {
  int r, h, t0, t1, n;
  int s;       // split whose partial this piece produces
  int64_t x0;  // global tile index of tile t0
};

struct Cursor {
  int r, h, t, n;
  int64_t x, remaining;
  int split;  // >= 0: the CTA's one split of a segment-aligned partition
};

// Tiles of request r in the work list: its context length only.  The work
// list is built before the abort mask may be read (the mask can come from the
// kernel launched just before this one); pieces of aborted requests are
// skipped after the dependency wait.
template <class Args>
__device__ __forceinline__ int tiles_of(const Args& a, int r) {
  return tiles_of_request(a.seq_lens, nullptr, r, a.max_pages, a.page_size);
}

template <class Args>
__device__ __forceinline__ bool is_aborted(const Args& a, int r) {
  return a.abort_mask != nullptr && __ldcg(a.abort_mask + r) != 0;
}

// Worker w owns global tiles [floor(w T / W), floor((w+1) T / W)); the owner
// of tile x is floor(((x + 1) W - 1) / T).  With W > T some workers own none.
__device__ __forceinline__ int worker_of(int64_t x, int64_t T, int W) {
  return static_cast<int>(((x + 1) * W - 1) / T);
}

// The next piece of a CTA's tile range: the longest run that stays inside one
// (request, kv head) segment and one split.
template <class Args>
__device__ __forceinline__ bool next_piece(Cursor& c, const Args& a, int64_t T, int W, Piece& p) {
  if (c.remaining <= 0) return false;
  const int s = c.split >= 0 ? c.split : worker_of(c.x, T, W);
  const int64_t split_end = c.split >= 0 ? c.x + c.remaining : (static_cast<int64_t>(s) + 1) * T / W;
  int64_t take64 = c.n - c.t;
  if (c.remaining < take64) take64 = c.remaining;
  if (split_end - c.x < take64) take64 = split_end - c.x;
  const int take = static_cast<int>(take64);
  p.s = s;
  p.r = c.r;
  p.h = c.h;
  p.t0 = c.t;
  p.t1 = c.t + take;
  p.n = c.n;
  p.x0 = c.x;
  c.remaining -= take;
  c.x += take;
  c.t += take;
  if (c.remaining > 0 && c.t == c.n) {
    c.t = 0;
    if (++c.h == a.Hkv) {
      c.h = 0;
      do {
        ++c.r;
        c.n = c.r < a.B ? tiles_of(a, c.r) : 1;
      } while (c.n == 0);
      if (c.r >= a.B) c.remaining = 0;  // unreachable with consistent inputs
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// workspace (caller-owned, zeroed once after allocation)
// ---------------------------------------------------------------------------
// [0, 256): the status word (offset 0) and small per-call scalars
// seg_count:   int [B * Hkv]          per-segment arrival tickets, zero between calls
// group_count: int [B * Hkv + W]      per-group arrival tickets, zero between calls
// part_ml:     float2 [slots][G]      (m, l) of each split partial (log2 domain)
// part_o:      float [slots][G][128]  unnormalised O of each split partial
// with slots = B * Hkv + W.
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t seg_count, group_count, part_ml, part_o, total;
};

inline WsLayout layout(int64_t B, int64_t Hkv, int64_t G, int64_t W) {
  WsLayout l;
  const int64_t segs = B * Hkv;
  const int64_t slots = segs + W;
  l.seg_count = 256;
  l.group_count = l.seg_count + align256(static_cast<size_t>(segs) * sizeof(int));
  l.part_ml = l.group_count + align256(static_cast<size_t>(slots) * sizeof(int));
  l.part_o = l.part_ml + align256(static_cast<size_t>(slots * G) * sizeof(float2));
  l.total = l.part_o + align256(static_cast<size_t>(slots * G * kDim) * sizeof(float));
  return l;
}

}  // namespace
}  // namespace fpk
