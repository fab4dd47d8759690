// The hardware-aware prefix scheduler as a block-level device function, shared by the
// scheduler kernel and the confidence kernel (which runs it in its last CTA).  See
// schedule.cu for the method and its citations.
#pragma once

#include "internal.h"

namespace dspark {

static constexpr int kSchedThreads = 1024;

static __device__ __forceinline__ long long fixed_point_a(float a) {
  double x = (double)a;
  if (!(x > 0.0)) return 0;
  if (x > 1.0) x = 1.0;
  return (long long)floor(__dadd_rn(__dmul_rn(x, 4294967296.0), 0.5));
}

static __device__ __forceinline__ double theta_at(long long R, long long S, float sps) {
  return __dmul_rn((double)(R * 4294967296LL + S), (double)sps);
}


// The scheduler run by one whole CTA of nthr = blockDim.x threads (a multiple of 32, at
// most kSchedThreads).  keys: Npad 64-bit words of shared memory.  K_in (may be null, may
// alias K_out): the capacity decided two steps earlier; a negative value or null admits
// this step's own early-stop count.  K_out (may be null) receives that count.
static __device__ void schedule_block(const float* __restrict__ a, int R, int gamma, int Npad,
                               const float* __restrict__ sps, const int32_t* K_in,
                               int32_t* K_out, int32_t* __restrict__ ell,
                               int32_t* __restrict__ B_total, double* __restrict__ theta,
                               unsigned long long* keys) {
  __shared__ long long warp_tot[32];
  __shared__ int first_fail, k_in_s;
  __shared__ float sps_s[kSchedThreads + 1];   // sps[R .. R + N] when N <= nthr
  __shared__ int cnt_s[kSchedThreads];         // admitted items per request when R <= nthr
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int N = R * gamma;
  const bool small = N <= nthr;
  // the SPS table entries the scan reads, fetched together with the expected returns
  if (small)
    for (int i = tid; i <= N; i += nthr) sps_s[i] = sps[R + i];
  if (R <= nthr && tid < R) cnt_s[tid] = 0;
  if (tid < 32) warp_tot[tid] = 0;

  for (int i = tid; i < Npad; i += nthr) {
    unsigned long long key = ~0ull;
    if (i < N) {
      const int r = i / gamma, j = i - r * gamma;
      const long long A = fixed_point_a(a[i]);
      key = ((unsigned long long)(4294967296LL - A) << 21) | ((unsigned long long)r << 5) |
            (unsigned long long)j;
    }
    keys[i] = key;
  }
  if (R > nthr)
    for (int r = tid; r < R; r += nthr) ell[r] = 0;
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
      for (int i = tid; i < (Npad >> 1); i += nthr) {
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
  const int per = (N + nthr - 1) / nthr;
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
  if (R <= nthr) {
    // per-request counts in shared memory, then one coalesced store of ell
    for (int i = tid; i < admitted; i += nthr)
      atomicAdd(&cnt_s[(int)((keys[i] >> 5) & 0xFFFFull)], 1);
    __syncthreads();
    if (tid < R) ell[tid] = cnt_s[tid];
  } else {
    for (int i = tid; i < admitted; i += nthr) {
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
  __syncthreads();          // the block's shared state is free again when this returns
}

}  // namespace dspark
