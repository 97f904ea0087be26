// step_ops.cuh -- the per-token cache write and the per-request tag check as
// device functions, shared by the stand-alone kernels (kv_write.cu,
// page_tags.cu) and the one-launch append-and-check kernel (decode_step.cu).
#pragma once

#include "common.cuh"
#include "quant.cuh"

namespace fpk {

struct WriteArgs {
  const uint16_t* k_src;     // bf16 [rows][Hkv][D]
  const uint16_t* v_src;
  const int32_t* seq_lens;   // decode mode: position = seq_lens[r] - 1, row r
  const int32_t* cu_seqlens; // prefill mode: row i of request r at position i - cu[r]
  uint8_t* kv_pool;
  const float* k_scale;
  const float* v_scale;
  const int32_t* page_table;
  const uint32_t* live_tags;
  const uint32_t* expected_tags;
  uint8_t* abort_mask;
  int64_t rows;
  int B, Hkv, D, page_size, num_pages, max_pages;
};

__device__ __forceinline__ int request_of_row(const int32_t* cu, int B, int64_t row) {
  // largest r with cu[r] <= row (cu non-decreasing, cu[0] = 0)
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(__ldg(cu + mid)) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One unit of token writing: 8 consecutive dims of one (token row, kv head).
// Returns without writing (and marks the request aborted) when the
// destination slot fails the guard.
template <bool kFp8, bool kPrefill>
__device__ __forceinline__ void write_unit(const WriteArgs& a, int64_t u, const Divisor& ks,
                                           const Divisor& vs) {
  const int chunks = a.D >> 3;
  {
    const int c = static_cast<int>(u % chunks);
    const int h = static_cast<int>((u / chunks) % a.Hkv);
    const int64_t row = u / (static_cast<int64_t>(chunks) * a.Hkv);
    // the source rows do not depend on the slot: their loads go out first, so
    // only the stores wait for the slot and its guard
    const int64_t src = (row * a.Hkv + h) * a.D + 8 * c;
    const uint4 kraw = __ldg(reinterpret_cast<const uint4*>(a.k_src + src));
    const uint4 vraw = __ldg(reinterpret_cast<const uint4*>(a.v_src + src));
    int r, pos;
    if (kPrefill) {
      r = request_of_row(a.cu_seqlens, a.B, row);
      pos = static_cast<int>(row - __ldg(a.cu_seqlens + r));
    } else {
      r = static_cast<int>(row);
      pos = __ldg(a.seq_lens + r) - 1;
      if (pos < 0) return;
    }
    const int pi = pos / a.page_size;
    const int off = pos - pi * a.page_size;
    bool ok = pi < a.max_pages;
    int page = -1;
    const bool guarded = a.live_tags != nullptr && a.expected_tags != nullptr;
    if (ok) {
      // the table entry and its expected tag load together; the live tag after
      const int64_t e = static_cast<int64_t>(r) * a.max_pages + pi;
      page = __ldg(a.page_table + e);
      const uint32_t want = guarded ? __ldg(a.expected_tags + e) : 0u;
      ok = page >= 0 && page < a.num_pages;
      if (ok && guarded) ok = __ldg(a.live_tags + page) == want;
    }
    if (!ok) {
      if (a.abort_mask != nullptr) a.abort_mask[r] = 1;
      return;
    }
    // the token's 16-token tile: K block [16][D], then V block [D][16]
    const int64_t tile = ((static_cast<int64_t>(page) * a.Hkv + h) * (a.page_size >> 4) + (off >> 4)) *
                         2 * 16 * a.D;
    const int64_t kdst = tile + (off & 15) * a.D + 8 * c;
    const int64_t vblk = tile + 16 * a.D;
    const int vcol = off & 15;
    const uint16_t* kb = reinterpret_cast<const uint16_t*>(&kraw);
    const uint16_t* vb = reinterpret_cast<const uint16_t*>(&vraw);
    if (kFp8) {
      uint32_t kw[2];
      uint8_t vq[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float k0 = div_by(bf16_bits_to_float(kb[2 * i]), ks);
        const float k1 = div_by(bf16_bits_to_float(kb[2 * i + 1]), ks);
        const float v0 = div_by(bf16_bits_to_float(vb[2 * i]), vs);
        const float v1 = div_by(bf16_bits_to_float(vb[2 * i + 1]), vs);
        const uint16_t kp = __nv_cvt_float2_to_fp8x2(make_float2(k0, k1), __NV_SATFINITE, __NV_E4M3);
        const uint16_t vp = __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
        if (i & 1) kw[i >> 1] |= static_cast<uint32_t>(kp) << 16; else kw[i >> 1] = kp;
        vq[2 * i] = static_cast<uint8_t>(vp & 0xFF);
        vq[2 * i + 1] = static_cast<uint8_t>(vp >> 8);
      }
      *reinterpret_cast<uint2*>(a.kv_pool + kdst) = make_uint2(kw[0], kw[1]);
#pragma unroll
      for (int i = 0; i < 8; ++i) a.kv_pool[vblk + static_cast<int64_t>(8 * c + i) * 16 + vcol] = vq[i];
    } else {
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.kv_pool) + kdst) = kraw;
      uint16_t* vpool = reinterpret_cast<uint16_t*>(a.kv_pool);
#pragma unroll
      for (int i = 0; i < 8; ++i) vpool[vblk + static_cast<int64_t>(8 * c + i) * 16 + vcol] = vb[i];
    }
  }
}

// The tag check of one request runs on one CTA, or, for a very long table,
// on a thread-block cluster of `nparts` CTAs (2..kCheckClusterMax; the
// hardware runs a cluster's CTAs at the same time, on different SMs where it
// can), so the rounds of table loads and live-tag gathers a long table needs
// are shared out.  Thread t of part k takes entries k*256 + t + j*nparts*256.
// Each thread checks up to kCheckPerThread entries per round: all table loads
// of the round, then all live-tag gathers (at a clamped, always valid index,
// so none waits behind a compare), then the compares.  The parts' results
// meet in the leader CTA's shared memory and the leader alone writes
// abort_mask[r]: no scratch memory and no clearing pass are needed.
// Measured on GB300 (decode step with and without the check, attention as
// the check's programmatic dependent): with one CTA per request the check
// adds 0.0-0.1 % at 32 x 8k, 64 x 1k-16k and 4 x 128k tokens (up to 2048
// table entries); clusters of 2-8 CTAs cost 0.2-0.5 % there.
constexpr int kValidateThreads = 256;
constexpr int kCheckPerThread = 4;
// Register bound of the check and write kernels (__launch_bounds__ minimum
// CTAs per SM): 6 CTAs of 256 threads cap them at 40 registers, so one of
// their CTAs (10 240 registers) still fits beside two attention CTAs (2 x 160
// threads x 168 registers) and the attention launched as their programmatic
// dependent starts on every SM while they run.
constexpr int kCheckCtasPerSm = 6;
constexpr int kCheckClusterMax = 8;
// Table entries one CTA checks before the request gets another: 4096, four
// rounds of one entry per thread and kCheckPerThread per round.
constexpr int kCheckEntriesPerCta = 4096;
// Check CTAs of a launch beyond which requests get no more parts (parts pay
// only while the requests leave most SMs without a check CTA).
constexpr int kCheckGridCap = 128;

// Parts of the check cluster of each of B requests with tables of max_pages
// columns: a power of two.
__host__ __device__ __forceinline__ int check_parts(int max_pages, int B) {
  int n = 1;
  while (n < kCheckClusterMax && static_cast<int64_t>(n) * kCheckEntriesPerCta < max_pages &&
         2 * static_cast<int64_t>(n) * B <= kCheckGridCap)
    n <<= 1;
  return n;
}

// Thread-block cluster barrier halves and a store into another CTA's shared
// memory (PTX barrier.cluster, mapa, st.shared::cluster).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void st_cluster_u32(const void* local, uint32_t rank, uint32_t v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// The entries of request r's table that part `part` of `nparts` checks; the
// OR over the CTA's threads, returned to every thread.
__device__ __forceinline__ int check_entries(const int32_t* __restrict__ page_table,
                                             const uint32_t* __restrict__ expected_tags,
                                             const int32_t* __restrict__ seq_lens, int max_pages,
                                             const uint32_t* __restrict__ live_tags, int num_pages,
                                             int page_size, int r, int part, int nparts) {
  const int32_t* pt = page_table + static_cast<int64_t>(r) * max_pages;
  const uint32_t* ex = expected_tags + static_cast<int64_t>(r) * max_pages;
  const int gt = part * kValidateThreads + static_cast<int>(threadIdx.x);
  const int stride = nparts * kValidateThreads;
  // The first round's table loads do not wait for the context length: they
  // cover the row's first entries (up to its width), and only entries below
  // the request's page count are compared.
  const int L = __ldg(seq_lens + r);
  int P = -1;  // known once L has arrived
  int bad = 0;
  for (int base = 0; base < max_pages && (P < 0 || (base < P && !bad)); base += kCheckPerThread * stride) {
    int page[kCheckPerThread];
    uint32_t want[kCheckPerThread], live[kCheckPerThread];
#pragma unroll
    for (int k = 0; k < kCheckPerThread; ++k) {
      const int i = base + k * stride + gt;
      page[k] = i < max_pages ? __ldg(pt + i) : 0;
      want[k] = i < max_pages ? __ldg(ex + i) : 0u;
    }
    if (P < 0) {
      P = L > 0 ? (L + page_size - 1) / page_size : 0;
      bad = P > max_pages || (P > 0 && num_pages <= 0);
      if (bad || P == 0) break;  // from here on num_pages > 0: every gather index is valid
    }
#pragma unroll
    for (int k = 0; k < kCheckPerThread; ++k) {
      const bool in_range = page[k] >= 0 && page[k] < num_pages;
      live[k] = __ldg(live_tags + (in_range ? page[k] : 0));
    }
#pragma unroll
    for (int k = 0; k < kCheckPerThread; ++k) {
      const int i = base + k * stride + gt;
      const bool in_range = page[k] >= 0 && page[k] < num_pages;
      if (i < P && (!in_range || live[k] != want[k])) bad = 1;
    }
  }
  if (P < 0) {  // an empty table (max_pages == 0): only the length can abort
    P = L > 0 ? (L + page_size - 1) / page_size : 0;
    bad = P > max_pages;
  }
  return __syncthreads_or(bad);
}

// The check of request blockIdx.x / nparts by part blockIdx.x % nparts (the
// CTA's rank in its cluster of nparts CTAs; nparts == 1: no cluster).  Every
// thread of every CTA of the cluster must call it (it holds cluster
// barriers).  The leader writes abort_mask[r] and, for an abort, adds one to
// *abort_count (nullable); returns whether the request aborts, to the
// leader's threads (the other parts' own share only).
__device__ __forceinline__ int check_request(const int32_t* __restrict__ page_table,
                                             const uint32_t* __restrict__ expected_tags,
                                             const int32_t* __restrict__ seq_lens, int max_pages,
                                             const uint32_t* __restrict__ live_tags, int num_pages,
                                             int page_size, uint8_t* __restrict__ abort_mask,
                                             int32_t* __restrict__ abort_count, int nparts) {
  __shared__ uint32_t s_part_bad[kCheckClusterMax];
  const int r = static_cast<int>(blockIdx.x) / nparts;
  const int part = static_cast<int>(blockIdx.x) - r * nparts;
  // this CTA has started: after the matching wait below, every CTA of the
  // cluster is running and its shared memory may be written
  if (nparts > 1) cluster_arrive_relaxed();
  int bad = check_entries(page_table, expected_tags, seq_lens, max_pages, live_tags, num_pages,
                          page_size, r, part, nparts);
  if (nparts > 1) {
    cluster_wait_acquire();
    if (threadIdx.x == 0) st_cluster_u32(&s_part_bad[part], 0, static_cast<uint32_t>(bad));
    // every part's flag is in the leader's shared memory after this barrier
    // (and no CTA exits while another may still write its shared memory)
    cluster_arrive_release();
    cluster_wait_acquire();
    if (part == 0) {
      bad = 0;
      for (int k = 0; k < nparts; ++k) bad |= static_cast<int>(s_part_bad[k]);
    }
  }
  if (part == 0 && threadIdx.x == 0) {
    abort_mask[r] = static_cast<uint8_t>(bad != 0);
    if (bad && abort_count != nullptr) atomicAdd(abort_count, 1);
  }
  return bad;
}

// Launches `kernel` over `grid` CTAs of kValidateThreads threads whose first
// check_ctas CTAs form clusters of `nparts` (grid a multiple of nparts); a
// plain launch when nparts == 1 (page_tags.cu).
template <typename... Exp, typename... Act>
int launch_check_grid(void (*kernel)(Exp...), int grid, int nparts, cudaStream_t s, Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kValidateThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nparts;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = nparts > 1 ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<Act&&>(args)...) != cudaSuccess) return FPK_ECUDA;
  return checked_launch_status();
}


// Grid for a grid-stride kernel: min(want, CTAs resident at once on the
// current device), so that no CTA waits for another to finish its whole loop
// (api.cu).
int resident_grid(const void* kernel, int threads, size_t dyn_smem, int64_t want);

// The cache write and tag check of one decode step as one launch
// (decode_step.cu); argument checks as fpk_decode_append_check_fp8.
int append_check_entry(bool fp8, const void* k_new, const void* v_new, void* kv_pool,
                       const float* k_scale, const float* v_scale, const int32_t* page_table,
                       int32_t max_pages, const int32_t* seq_lens, const uint32_t* live_tags,
                       const uint32_t* expected_tags, uint8_t* abort_mask, int32_t B, int32_t Hkv,
                       int32_t D, int32_t page_size, int32_t num_pages, void* stream);

}  // namespace fpk
