// api.cu -- library-wide entry points and host helpers of libfp8kv.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "step_ops.cuh"

namespace fpk {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
}  // namespace

int device_sm_count(int device) {
  if (device < 0 || device >= kMaxDevices) return 0;
  int v = g_sm_count[device].load(std::memory_order_relaxed);
  if (v > 0) return v;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  g_sm_count[device].store(n, std::memory_order_relaxed);
  return n;
}

// Status after a launch: FPK_ECUDA if the launch reported an error.  The error
// is peeked, not cleared, so that the caller's own checks still see it.
int checked_launch_status() {
  return cudaPeekAtLastError() == cudaSuccess ? FPK_OK : FPK_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int resident_grid(const void* kernel, int threads, size_t dyn_smem, int64_t want) {
  if (want <= 0) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const int sms = device_sm_count(dev);
  if (want <= sms) return static_cast<int>(want);  // resident whatever the occupancy
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, dyn_smem) != cudaSuccess ||
      per_sm <= 0 || sms <= 0)
    return static_cast<int>(want < 1024 ? want : 1024);
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  return static_cast<int>(want < cap ? want : cap);
}

namespace {
// Self-test of the bounded wait every kernel uses: one CTA waits on an
// mbarrier that nothing arrives on.  The wait gives up after kWaitLimitNs,
// sets kStatusWaitTimeout in *status and returns; the kernel records how long
// the wait took.
__global__ void bounded_wait_selftest_kernel(uint32_t* status, unsigned long long* elapsed_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  const uint64_t t0 = global_timer_ns();
  const bool got = mbar_wait(smem_addr(&bar), 0, status);
  if (threadIdx.x == 0) *elapsed_ns = got ? 0ull : global_timer_ns() - t0;
}
}  // namespace

}  // namespace fpk

extern "C" int fpk_selftest_bounded_wait(uint32_t* status, unsigned long long* elapsed_ns, void* stream) {
  if (!status || !elapsed_ns) return FPK_EINVAL;
  fpk::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, elapsed_ns);
  return fpk::checked_launch_status();
}

extern "C" int fpk_version(void) { return 100; }

extern "C" const char* fpk_status_str(int status) {
  switch (status) {
    case FPK_OK: return "ok";
    case FPK_EINVAL: return "invalid argument (null pointer, negative size or Hq % Hkv != 0)";
    case FPK_EUNSUPPORTED: return "unsupported size (D, page_size or group size)";
    case FPK_ENOSPC: return "workspace too small";
    case FPK_ECUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}
