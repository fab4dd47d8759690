// Hardware-aware prefix scheduler in one CTA.
//
// billytse.dev DSpark page, section 6: with l_r positions verified for request r, the
// target processes B = sum_r (1 + l_r) tokens and commits tau = sum_r (1 + sum_{j<=l_r}
// a_{r,j}) in expectation; the goal is max Theta = tau * SPS(B).  Positions are taken in
// descending expected return and added one at a time while Theta rises; section 7: the
// first drop stops the scan (early stopping), which keeps admission non-anticipating.
//
// In one CTA: keys (A desc, r asc, j asc) with A = floor(clamp(a, 0, 1) 2^32 + 1/2) are
// sorted by a bitonic network in shared memory; a block-wide prefix sum gives the exact
// integer S_n; every n evaluates Theta_n = double(R 2^32 + S_n) * double(sps[R + n])
// against Theta_{n-1} (plain double products, no fused multiply-add) and the smallest
// failing n is found with a shared-memory atomicMin.
//
// Two-step capacity (weigao.cc DSpark-vs-MTP page, "4. hardware-aware prefix scheduler";
// billytse.dev section 7): when a capacity K decided two steps earlier is given, the
// first K items of this step's order are admitted instead of the first n* (n* = the early-
// stop count), and n* is written out as the capacity of the step after next.
//
// Fixed-threshold truncation (billytse.dev section 8; xhh.club page on load-dependent
// thresholds): one warp per request, lane j - 1 tests a[r, j] > threshold and a ballot
// gives the leading run.
#include "schedule_block.cuh"

namespace dspark {

namespace {

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(
    const float* __restrict__ a, int R, int gamma, int Npad, const float* __restrict__ sps,
    const int32_t* K_in, int32_t* K_out, int32_t* __restrict__ ell,
    int32_t* __restrict__ B_total, double* __restrict__ theta, size_t scratch_bytes) {
  extern __shared__ unsigned long long keys[];
  pdl_wait();                 // the expected returns come from the previous kernel
  pdl_launch_dependents();
  schedule_block<true>(a, R, gamma, Npad, sps, K_in, K_out, ell, B_total, theta, keys, scratch_bytes);
}

constexpr int kThreshThreads = 1024;

__global__ void __launch_bounds__(kThreshThreads) schedule_threshold_kernel(
    const float* __restrict__ a, int R, int gamma, float threshold, int32_t* __restrict__ ell,
    int32_t* __restrict__ B_total) {
  __shared__ int warp_tot[kThreshThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int total = 0;
  for (int r = warp; r < R; r += kThreshThreads / 32) {
    // lanes past gamma count as failures, so the leading run stops at gamma at most
    const bool pass = lane < gamma && a[(size_t)r * gamma + lane] > threshold;
    const unsigned fail = ~__ballot_sync(0xffffffffu, pass);
    const int l = fail ? __ffs(fail) - 1 : 32;    // all 32 pass only when gamma == 32
    if (lane == 0) ell[r] = l;
    total += 1 + l;
  }
  if (lane == 0) warp_tot[warp] = total;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long t = 0;
    for (int w = 0; w < kThreshThreads / 32; ++w) t += warp_tot[w];
    *B_total = (int32_t)t;
  }
}

}  // namespace

cudaError_t launch_schedule_threshold(const float* a, int R, int gamma, float threshold,
                                      int32_t* ell, int32_t* B_total, cudaStream_t stream) {
  return launch_pdl(schedule_threshold_kernel, dim3(1), dim3(kThreshThreads), 0, stream, a, R,
                    gamma, threshold, ell, B_total);
}

cudaError_t launch_schedule(const float* a, int R, int gamma, const float* sps,
                            const int32_t* K_in, int32_t* K_out, int32_t* ell, int32_t* B_total,
                            double* theta, int* err, cudaStream_t stream) {
  (void)err;
  const int N = R * gamma;
  int Npad = 2;
  while (Npad < N) Npad <<= 1;
  // the keys of the ranking or the network (Npad words), or the radix sort's arrays
  size_t smem = (size_t)Npad * sizeof(unsigned long long);
  if (N > kSchedThreads && schedule_radix_bytes(N) > smem) smem = schedule_radix_bytes(N);
  // the shared-memory attribute is set once per device
  static std::atomic<int> cache[kMaxCachedDevices];
  const int ok = per_device_grid(cache, [] {
    size_t most = (size_t)kMaxScheduleItems * sizeof(unsigned long long);
    if (schedule_radix_bytes(kMaxScheduleItems) > most) most = schedule_radix_bytes(kMaxScheduleItems);
    return cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)most) == cudaSuccess
               ? 1 : -1;
  });
  if (ok <= 0) return cudaErrorInvalidConfiguration;
  return launch_pdl(schedule_kernel, dim3(1), dim3(kSchedThreads), smem, stream, a, R, gamma, Npad,
                    sps, K_in, K_out, ell, B_total, theta, smem);
}

}  // namespace dspark
