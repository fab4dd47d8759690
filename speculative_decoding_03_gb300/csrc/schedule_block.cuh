// The hardware-aware prefix scheduler as a block-level device function, shared by the
// scheduler kernel and the confidence kernel (which runs it in its last CTA).  See
// schedule.cu for the method and its citations.
#pragma once

#include "internal.h"

namespace dspark {

static constexpr int kSchedThreads = 1024;

// A = floor(clamp(a, 0, 1) 2^32 + 1/2) (NaN -> 0), exactly, in integer arithmetic: a is
// m 2^(sh - 32) with an integer mantissa m < 2^24, so a 2^32 = m 2^sh, rounded half up.
static __device__ __forceinline__ long long fixed_point_a(float a) {
  if (!(a > 0.f)) return 0;
  if (a >= 1.f) return 4294967296LL;
  const uint32_t u = __float_as_uint(a);
  const int ex = (int)(u >> 23);                          // 0 for subnormal a
  const unsigned long long m = ex ? ((u & 0x7FFFFFu) | 0x800000u) : (u & 0x7FFFFFu);
  const int sh = (ex ? ex : 1) - 118;                     // 32 - 127 - 23 + exponent
  if (sh >= 0) return (long long)(m << sh);               // sh <= 8 below 1
  if (sh < -40) return 0;                                 // below 2^-16
  return (long long)((m + (1ull << (-sh - 1))) >> (-sh));
}

// The sort key of item i = r gamma + j: (A desc, r asc, j asc) as one 64-bit integer.
static __device__ __forceinline__ unsigned long long schedule_key(float a, int r, int j) {
  return ((unsigned long long)(4294967296LL - fixed_point_a(a)) << 21) |
         ((unsigned long long)r << 5) | (unsigned long long)j;
}

static __device__ __forceinline__ double theta_at(long long R, long long S, float sps) {
  return __dmul_rn((double)(R * 4294967296LL + S), (double)sps);
}


// Shared memory the radix path of schedule_block needs for N items: two 32-bit key arrays,
// two 16-bit index arrays and the per-warp digit counters.
static constexpr int kRadixBits = 7;
static constexpr int kRadixBins = 1 << kRadixBits;
static constexpr int kRadixStride = 33;   // counters of one digit, one per warp, padded
__host__ __device__ constexpr size_t schedule_radix_bytes(int N) {
  return (size_t)N * 12 + (size_t)kRadixBins * kRadixStride * sizeof(int);
}

// LSD radix sort of the N items by the key K = 2^32 - A (A as in fixed_point_a, so K has
// 33 bits: bit 32 set only for A = 0), 7 bits a pass, 5 passes; every pass is a stable
// counting sort and the items enter in index order i = r * gamma + j, so equal keys keep
// (r, j) order: the order (A desc, r asc, j asc) of the sorting network below.  Warp w owns
// the items w * 32 PER .. in rounds of 32 (item = base + 32 q + lane, index order within the
// warp); a round ranks its lanes per digit with one ballot per digit bit, per-warp counters carry the
// ranks across rounds, and one block scan over (digit, warp) gives every bucket's base.
// The K bit 32 rides in bit 15 of the 16-bit index (i < 2^15).  One CTA of kSchedThreads
// threads; returns the arrays holding the sorted keys and indices.
static __device__ void schedule_radix_sort(const float* __restrict__ a, int N, uint8_t* scratch,
                                           uint32_t** K_out, uint16_t** I_out) {
  constexpr int kPer = kMaxScheduleItems / kSchedThreads;   // rounds per warp, at most
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* const K0 = reinterpret_cast<uint32_t*>(scratch);
  uint32_t* const K1 = K0 + N;
  uint16_t* const I0 = reinterpret_cast<uint16_t*>(scratch + (size_t)N * 8);
  uint16_t* const I1 = I0 + N;
  // [digit][warp], a digit's row padded to 33 words so that the lanes of a warp, which
  // read the counters of different digits, hit different banks
  int* cnt = reinterpret_cast<int*>(scratch + (size_t)N * 12);
  __shared__ int scan_tot[32];
  for (int i = tid; i < N; i += kSchedThreads) {
    const long long A = fixed_point_a(a[i]);
    K0[i] = (uint32_t)(4294967296LL - A);         // low 32 bits
    I0[i] = (uint16_t)(i | (A == 0 ? 0x8000 : 0));
  }
  const int per = (N + kSchedThreads - 1) / kSchedThreads;
  const int wbase = warp * 32 * per;
  const unsigned lt = (1u << lane) - 1u;
  int src = 0;
  for (int pass = 0; pass < 5; ++pass, src ^= 1) {
    const uint32_t* Ks = src ? K1 : K0;
    const uint16_t* Is = src ? I1 : I0;
    uint32_t* Kd = src ? K0 : K1;
    uint16_t* Id = src ? I0 : I1;
    for (int i = tid; i < kRadixBins * kRadixStride; i += kSchedThreads) cnt[i] = 0;
    __syncthreads();
    int off[kPer];
    auto digit = [&](int item) -> int {
      const uint32_t k = Ks[item];
      const uint32_t top = (Is[item] >> 15) & 1u;
      return pass < 4 ? (int)((k >> (kRadixBits * pass)) & (kRadixBins - 1))
                      : (int)((k >> 28) | (top << 4));
    };
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      off[q] = 0;
      if (q < per) {
        const int item = wbase + 32 * q + lane;
        const bool valid = item < N;
        const int d = valid ? digit(item) : kRadixBins;
        // the lanes with the same digit (bit 7: past the end): one ballot per bit
        unsigned peers = 0xffffffffu;
#pragma unroll
        for (int bit = 0; bit <= kRadixBits; ++bit) {
          const bool on = (d >> bit) & 1;
          const unsigned bb = __ballot_sync(0xffffffffu, on);
          peers &= on ? bb : ~bb;
        }
        const int cur = valid ? cnt[d * kRadixStride + warp] : 0;
        off[q] = cur + __popc(peers & lt);
        __syncwarp();
        if (valid && (peers & lt) == 0) cnt[d * kRadixStride + warp] = cur + __popc(peers);
        __syncwarp();
      }
    }
    __syncthreads();
    // exclusive scan of the counters in (digit, warp) order: four per thread
    {
      int c4[4], sum = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = 4 * tid + u;                 // entry (digit e / 32, warp e % 32)
        c4[u] = cnt[(e >> 5) * kRadixStride + (e & 31)];
        sum += c4[u];
      }
      int incl = sum;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += t;
      }
      if (lane == 31) scan_tot[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        int t = scan_tot[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, t, d);
          if (lane >= d) t += u;
        }
        scan_tot[lane] = t;
      }
      __syncthreads();
      int run = incl - sum + (warp > 0 ? scan_tot[warp - 1] : 0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = 4 * tid + u;
        cnt[(e >> 5) * kRadixStride + (e & 31)] = run;
        run += c4[u];
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      if (q < per) {
        const int item = wbase + 32 * q + lane;
        if (item < N) {
          const int d = digit(item);
          const int dst = cnt[d * kRadixStride + warp] + off[q];
          Kd[dst] = Ks[item];
          Id[dst] = Is[item];
        }
      }
    }
    __syncthreads();
  }
  *K_out = src ? K1 : K0;
  *I_out = src ? I1 : I0;
}

// The scheduler run by one whole CTA of nthr = blockDim.x threads (a multiple of 32, at
// most kSchedThreads).  keys: scratch shared memory of scratch_bytes bytes, at least Npad
// 64-bit words; with kSchedThreads threads, more than nthr items and
// schedule_radix_bytes(N) bytes the items are sorted by the radix path, else by ranking
// (N <= nthr) or a sorting network.  K_in (may be null, may alias K_out): the capacity
// decided two steps earlier; a negative value or null admits this step's own early-stop
// count.  K_out (may be null) receives that count.  kRadix: whether the radix path is
// compiled in (the scheduler kernel; the blocks that run the scheduler inside another
// kernel keep their registers for it).
// presorted: keys[0 .. N) already hold the N items' keys in ascending order (a is then
// not read).
template <bool kRadix>
static __device__ void schedule_block(const float* __restrict__ a, int R, int gamma, int Npad,
                               const float* __restrict__ sps, const int32_t* K_in,
                               int32_t* K_out, int32_t* __restrict__ ell,
                               int32_t* __restrict__ B_total, double* __restrict__ theta,
                               unsigned long long* keys, size_t scratch_bytes,
                               bool presorted = false) {
  __shared__ long long warp_tot[32];
  __shared__ long long a_top_s;
  __shared__ int first_fail, k_in_s;
  __shared__ float sps_s[kSchedThreads + 1];   // sps[R .. R + N] when N <= nthr
  __shared__ int cnt_s[kSchedThreads];         // admitted items per request when R <= nthr
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int N = R * gamma;
  const bool small = N <= nthr;
  const bool radix = kRadix && !presorted && !small && nthr == kSchedThreads &&
                     N <= kMaxScheduleItems && scratch_bytes >= schedule_radix_bytes(N);
  // the SPS table entries the scan reads, fetched together with the expected returns
  if (small)
    for (int i = tid; i <= N; i += nthr) sps_s[i] = sps[R + i];
  if (R <= nthr && tid < R) cnt_s[tid] = 0;
  if (tid < 32) warp_tot[tid] = 0;

  for (int i = tid; i < (radix || presorted ? 0 : Npad); i += nthr) {
    unsigned long long key = ~0ull;
    if (i < N) {
      const int r = i / gamma, j = i - r * gamma;
      key = schedule_key(a[i], r, j);
    }
    keys[i] = key;
  }
  if (R > nthr)
    for (int r = tid; r < R; r += nthr) ell[r] = 0;
  if (tid == 0) {
    first_fail = N + 1;
    k_in_s = K_in ? *K_in : -1;     // read before K_out (which may alias it) is written
    a_top_s = 0;
  }
  __syncthreads();

  if (kRadix && radix && k_in_s < 0) {
    // The scan stops at the first item when even the largest expected return does not raise
    // Theta; then nothing is admitted and no order is needed (without a capacity): the
    // outputs are those of the full scan, from one block-wide maximum of A.
    long long top = 0;
    for (int i = tid; i < N; i += nthr) top = max(top, fixed_point_a(a[i]));
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) top = max(top, __shfl_xor_sync(0xffffffffu, top, d));
    if ((tid & 31) == 0) atomicMax(reinterpret_cast<unsigned long long*>(&a_top_s), (unsigned long long)top);
    __syncthreads();
    const double th0 = theta_at(R, 0, sps[R]);
    if (!(theta_at(R, a_top_s, sps[R + 1]) > th0)) {
      if (R <= nthr && tid < R) ell[tid] = 0;       // (more requests were zeroed above)
      if (tid == 0) {
        if (K_out) *K_out = 0;
        *B_total = R;
        *theta = th0 / 4294967296.0;
      }
      __syncthreads();
      return;
    }
  }

  uint32_t* rK = nullptr;
  uint16_t* rI = nullptr;
  if (presorted) {
  } else if (kRadix && radix) {
    schedule_radix_sort(a, N, reinterpret_cast<uint8_t*>(keys), &rK, &rI);
  } else if (small) {
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

  // the sorted items' A and request
  auto A_at = [&](int i) -> long long {
    if (kRadix && radix) return (rI[i] & 0x8000) ? 0LL : 4294967296LL - (long long)rK[i];
    return 4294967296LL - (long long)(keys[i] >> 21);
  };
  auto r_at = [&](int i) -> int {
    if (kRadix && radix) return (int)(rI[i] & 0x7FFF) / gamma;
    return (int)((keys[i] >> 5) & 0xFFFFull);
  };
  // exact prefix sums S_n over the sorted A values: contiguous chunks per thread
  const int per = (N + nthr - 1) / nthr;
  const int c0 = min(N, tid * per), c1 = min(N, c0 + per);
  long long local = 0;
  for (int i = c0; i < c1; ++i) local += A_at(i);
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
  if (c0 < c1) {
    // Theta_n against Theta_{n-1}; each Theta is computed once (it is the next item's
    // previous value)
    double th_prev = theta_at(R, S, small ? sps_s[c0] : sps[R + c0]);
    for (int i = c0; i < c1; ++i) {
      S += A_at(i);
      const double th = theta_at(R, S, small ? sps_s[i + 1] : sps[R + i + 1]);
      if (!(th > th_prev)) {
        fail = i + 1;
        break;
      }
      th_prev = th;
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
      atomicAdd(&cnt_s[r_at(i)], 1);
    __syncthreads();
    if (tid < R) ell[tid] = cnt_s[tid];
  } else {
    for (int i = tid; i < admitted; i += nthr) {
      const int r = r_at(i);
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
    for (int i = c0; i < admitted; ++i) Sa += A_at(i);
    *B_total = R + admitted;
    *theta = theta_at(R, Sa, small ? sps_s[admitted] : sps[R + admitted]) / 4294967296.0;
  }
  __syncthreads();          // the block's shared state is free again when this returns
}

}  // namespace dspark
