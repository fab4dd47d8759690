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
#include "internal.h"

namespace dspark {
namespace {

constexpr int kSchedThreads = 1024;

__device__ __forceinline__ long long fixed_point_a(float a) {
  double x = (double)a;
  if (!(x > 0.0)) return 0;
  if (x > 1.0) x = 1.0;
  return (long long)floor(__dadd_rn(__dmul_rn(x, 4294967296.0), 0.5));
}

__device__ __forceinline__ double theta_at(long long R, long long S, float sps) {
  return __dmul_rn((double)(R * 4294967296LL + S), (double)sps);
}

// K_in (may be null, may alias K_out): the capacity decided two steps earlier; a negative
// value or null admits this step's own early-stop count.  K_out (may be null) receives
// that count.
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(
    const float* __restrict__ a, int R, int gamma, int Npad, const float* __restrict__ sps,
    const int32_t* K_in, int32_t* K_out, int32_t* __restrict__ ell,
    int32_t* __restrict__ B_total, double* __restrict__ theta) {
  extern __shared__ unsigned long long keys[];
  __shared__ long long warp_tot[32];
  __shared__ int first_fail, k_in_s;
  __shared__ float sps_s[kSchedThreads + 1];   // sps[R .. R + N] when N <= kSchedThreads
  __shared__ int cnt_s[kSchedThreads];         // admitted items per request when R <= kSchedThreads
  pdl_wait();                 // the expected returns come from the previous kernel
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int N = R * gamma;
  const bool small = N <= kSchedThreads;
  // the SPS table entries the scan reads, fetched together with the expected returns
  if (small && tid <= N) sps_s[tid] = sps[R + tid];
  if (R <= kSchedThreads && tid < R) cnt_s[tid] = 0;

  for (int i = tid; i < Npad; i += kSchedThreads) {
    unsigned long long key = ~0ull;
    if (i < N) {
      const int r = i / gamma, j = i - r * gamma;
      const long long A = fixed_point_a(a[i]);
      key = ((unsigned long long)(4294967296LL - A) << 21) | ((unsigned long long)r << 5) |
            (unsigned long long)j;
    }
    keys[i] = key;
  }
  if (R > kSchedThreads)
    for (int r = tid; r < R; r += kSchedThreads) ell[r] = 0;
  if (tid == 0) {
    first_fail = N + 1;
    k_in_s = K_in ? *K_in : -1;     // read before K_out (which may alias it) is written
  }
  __syncthreads();

  if (small) {
    // small batches: every key is distinct, so its rank is the number of smaller keys;
    // one pass of broadcast shared-memory reads, no sorting network
    const unsigned long long mine = tid < N ? keys[tid] : ~0ull;
    int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
    if (tid < N) {            // only the threads that own a key rank it
      int j = 0;
      for (; j + 4 <= N; j += 4) {
        r0 += keys[j] < mine ? 1 : 0;
        r1 += keys[j + 1] < mine ? 1 : 0;
        r2 += keys[j + 2] < mine ? 1 : 0;
        r3 += keys[j + 3] < mine ? 1 : 0;
      }
      for (; j < N; ++j) r0 += keys[j] < mine ? 1 : 0;
    }
    const int rank = r0 + r1 + r2 + r3;
    __syncthreads();
    if (tid < N) keys[rank] = mine;
    __syncthreads();
  } else
  // bitonic sort, ascending key = (A desc, r asc, j asc)
  for (int size = 2; size <= Npad; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < (Npad >> 1); i += kSchedThreads) {
        const int lo = 2 * stride * (i / stride) + (i % stride);
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long x = keys[lo], y = keys[hi];
        if ((x > y) == up) {
          keys[lo] = y;
          keys[hi] = x;
        }
      }
      __syncthreads();
    }
  }

  // exact prefix sums S_n over the sorted A values: contiguous chunks per thread
  const int per = (N + kSchedThreads - 1) / kSchedThreads;
  const int c0 = min(N, tid * per), c1 = min(N, c0 + per);
  long long local = 0;
  for (int i = c0; i < c1; ++i) local += 4294967296LL - (long long)(keys[i] >> 21);
  // block exclusive scan of the chunk totals
  const int lane = tid & 31, warp = tid >> 5;
  long long incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long t = warp_tot[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long u = __shfl_up_sync(0xffffffffu, t, d);
      if (lane >= d) t += u;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  long long S = incl - local + (warp > 0 ? warp_tot[warp - 1] : 0);  // exclusive prefix
  int fail = N + 1;
  for (int i = c0; i < c1; ++i) {
    const long long A = 4294967296LL - (long long)(keys[i] >> 21);
    const int n = i + 1;
    const double th_prev = theta_at(R, S, small ? sps_s[n - 1] : sps[R + n - 1]);
    S += A;
    const double th = theta_at(R, S, small ? sps_s[n] : sps[R + n]);
    if (!(th > th_prev)) {
      fail = n;
      break;
    }
  }
  if (fail <= N) atomicMin(&first_fail, fail);
  __syncthreads();
  const int n_star = first_fail - 1;
  const int admitted = k_in_s < 0 ? n_star : min(k_in_s, N);
  if (K_out && tid == 0) *K_out = n_star;
  if (R <= kSchedThreads) {
    // per-request counts in shared memory, then one coalesced store of ell
    for (int i = tid; i < admitted; i += kSchedThreads)
      atomicAdd(&cnt_s[(int)((keys[i] >> 5) & 0xFFFFull)], 1);
    __syncthreads();
    if (tid < R) ell[tid] = cnt_s[tid];
  } else {
    for (int i = tid; i < admitted; i += kSchedThreads) {
      const int r = (int)((keys[i] >> 5) & 0xFFFFull);
      atomicAdd(&ell[r], 1);
    }
  }
  // Theta at the stop: S_admitted lies in the chunk holding item `admitted`
  if (admitted == 0) {
    if (tid == 0) {
      *B_total = R;
      *theta = theta_at(R, 0, small ? sps_s[0] : sps[R]) / 4294967296.0;
    }
  } else if (admitted - 1 >= c0 && admitted - 1 < c1) {
    long long Sa = incl - local + (warp > 0 ? warp_tot[warp - 1] : 0);
    for (int i = c0; i < admitted; ++i) Sa += 4294967296LL - (long long)(keys[i] >> 21);
    *B_total = R + admitted;
    *theta = theta_at(R, Sa, small ? sps_s[admitted] : sps[R + admitted]) / 4294967296.0;
  }
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
  const size_t smem = (size_t)Npad * sizeof(unsigned long long);
  // the shared-memory attribute is set once per device
  static std::atomic<int> cache[kMaxCachedDevices];
  const int ok = per_device_grid(cache, [] {
    return cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(kMaxScheduleItems * sizeof(unsigned long long))) == cudaSuccess
               ? 1 : -1;
  });
  if (ok <= 0) return cudaErrorInvalidConfiguration;
  return launch_pdl(schedule_kernel, dim3(1), dim3(kSchedThreads), smem, stream, a, R, gamma, Npad,
                    sps, K_in, K_out, ell, B_total, theta);
}

}  // namespace dspark
