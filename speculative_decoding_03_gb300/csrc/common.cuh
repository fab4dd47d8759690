// Device helpers shared by the DSpark kernels: status word, counter-based random
// numbers, the uniform / Gumbel transforms and small math helpers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

// ----------------------------------------------------------------------------------------
// Device status word: kernels never trap; a failed device-side check records its code
// here (first writer wins) and the kernel skips the offending access.
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ void set_device_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ----------------------------------------------------------------------------------------
// Philox4x32 with kPhiloxRounds = 7 rounds (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11: the Philox4x32 round function; 7 is the fewest rounds
// that paper reports passing TestU01 BigCrush, its default being 10): per round two
// 32x32->64 multiplies with the round constants, the high halves mixed into the other
// counter words and the key; the key advances by the two Weyl constants between rounds.
// Key = (seed low word, seed high word).  The draw for
// vocabulary index v of (request b, position k, stream s) is word v % 4 of the block with
// counter (v / 4, k, b, s): one 128-bit block feeds one 128-bit logit load.
// ----------------------------------------------------------------------------------------
constexpr int kPhiloxRounds = 7;
__device__ __forceinline__ uint4 philox4x32(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < kPhiloxRounds; ++round) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ uint4 draw_block(uint64_t seed, uint32_t v4, uint32_t k, uint32_t b,
                                            uint32_t stream) {
  return philox4x32(make_uint4(v4, k, b, stream), (uint32_t)seed, (uint32_t)(seed >> 32));
}

// The key of every round of the same generator, k[2 i] = seed low + i 0x9E3779B9 and
// k[2 i + 1] = seed high + i 0xBB67AE85, evaluated once on the host: passed to a kernel as
// a parameter, the rounds read it from the constant bank instead of advancing the key.
struct PhiloxKeys {
  uint32_t k[2 * kPhiloxRounds];
};
inline PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys r;
  for (int i = 0; i < kPhiloxRounds; ++i) {
    r.k[2 * i] = (uint32_t)seed + (uint32_t)i * 0x9E3779B9u;
    r.k[2 * i + 1] = (uint32_t)(seed >> 32) + (uint32_t)i * 0xBB67AE85u;
  }
  return r;
}
__device__ __forceinline__ uint4 philox4x32(uint4 c, const PhiloxKeys& rk) {
#pragma unroll
  for (int round = 0; round < kPhiloxRounds; ++round) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ rk.k[2 * round], lo1, hi0 ^ c.w ^ rk.k[2 * round + 1], lo0);
  }
  return c;
}
__device__ __forceinline__ uint4 draw_block(const PhiloxKeys& rk, uint32_t v4, uint32_t k,
                                            uint32_t b, uint32_t stream) {
  return philox4x32(make_uint4(v4, k, b, stream), rk);
}
// The same block with one 32x32->64 multiply per product (the draft samplers' form).
__device__ __forceinline__ uint4 philox_wide(uint4 c, const PhiloxKeys& rk) {
#pragma unroll
  for (int round = 0; round < kPhiloxRounds; ++round) {
    const unsigned long long p0 = (unsigned long long)0xD2511F53u * c.x;
    const unsigned long long p1 = (unsigned long long)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ rk.k[2 * round], (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ rk.k[2 * round + 1], (uint32_t)p0);
  }
  return c;
}

// U01(x) = ((x >> 9) + 1/2) 2^-23 and its exact complement 1 - U01(x); both are exact in
// fp32 (24 significant bits at most).  Built without an integer conversion: the float with
// bits 0x4B000000 | n is 2^23 + n, and one fused multiply-add removes 2^23 - 1/2.
__device__ __forceinline__ float u01(uint32_t x) {
  return fmaf(__uint_as_float(0x4B000000u | (x >> 9)), 0x1.0p-23f, -(1.f - 0x1.0p-24f));
}
__device__ __forceinline__ float one_minus_u01(uint32_t x) {
  return fmaf(__uint_as_float(0x4B000000u | ((~x) >> 9)), 0x1.0p-23f, -(1.f - 0x1.0p-24f));
}

// The Exp(1) variate E = -log(u) = -log1p(-w), accurate near u -> 1 (small w), which is
// where the largest Gumbel values g = -log(E) come from.
__device__ __forceinline__ float exp1_from_w(float w) { return -log1pf(-w); }

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32); exp(x) = 2^(x log2 e).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// Orderable 64-bit argmax key: larger score first, then smaller index.
__device__ __forceinline__ unsigned long long argmax_key(float score, int idx) {
  uint32_t u = __float_as_uint(score);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

// ----------------------------------------------------------------------------------------
// Row-softmax + Gumbel-argmax partial state, merged across threads, warps and CTAs.
//   m     running max of the logits seen
//   s     sum of exp(z - m) over the logits seen
//   score best Gumbel score z + g seen (-inf if none), idx its index (-1 if none)
//   z     logit of the best element (for q = exp(z - m) / s)
// ----------------------------------------------------------------------------------------
struct RowState {
  float m, s, score, z;
  int idx;
};

__device__ __forceinline__ RowState row_state_empty() {
  RowState r;
  r.m = -INFINITY;
  r.s = 0.f;
  r.score = -INFINITY;
  r.z = -INFINITY;
  r.idx = -1;
  return r;
}

__device__ __forceinline__ bool better(float sa, int ia, float sb, int ib) {
  // is (sa, ia) better than (sb, ib)?  larger score, then smaller valid index
  if (ia < 0) return false;
  if (ib < 0) return true;
  return sa > sb || (sa == sb && ia < ib);
}

__device__ __forceinline__ RowState row_state_merge(const RowState& a, const RowState& b) {
  RowState o;
  o.m = fmaxf(a.m, b.m);
  const float sa = (a.m == -INFINITY) ? 0.f : a.s * expf(a.m - o.m);
  const float sb = (b.m == -INFINITY) ? 0.f : b.s * expf(b.m - o.m);
  o.s = sa + sb;
  if (better(b.score, b.idx, a.score, a.idx)) {
    o.score = b.score; o.idx = b.idx; o.z = b.z;
  } else {
    o.score = a.score; o.idx = a.idx; o.z = a.z;
  }
  return o;
}

__device__ __forceinline__ RowState row_state_shfl_xor(const RowState& a, int mask) {
  RowState o;
  o.m = __shfl_xor_sync(0xffffffffu, a.m, mask);
  o.s = __shfl_xor_sync(0xffffffffu, a.s, mask);
  o.score = __shfl_xor_sync(0xffffffffu, a.score, mask);
  o.z = __shfl_xor_sync(0xffffffffu, a.z, mask);
  o.idx = __shfl_xor_sync(0xffffffffu, a.idx, mask);
  return o;
}

__device__ __forceinline__ RowState row_state_warp_reduce(RowState a) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) a = row_state_merge(a, row_state_shfl_xor(a, m));
  return a;
}

// Block-wide reduction; every thread gets the result.  smem holds 32 RowStates.
__device__ __forceinline__ RowState row_state_block_reduce(RowState a, RowState* smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  a = row_state_warp_reduce(a);
  if (lane == 0) smem[warp] = a;
  __syncthreads();
  RowState r = (lane < nwarps) ? smem[lane] : row_state_empty();
  r = row_state_warp_reduce(r);
  __syncthreads();
  return r;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream serialization
// may be scheduled while the previous kernel on the stream is still draining: pdl_wait()
// (griddepcontrol.wait) blocks until that kernel has completed and its writes are visible,
// and every such kernel calls it before reading anything an earlier kernel wrote and before
// it can exit.  pdl_launch_dependents() lets the next kernel be scheduled once every CTA of
// this grid has issued it.  Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 128-bit streaming load: read once, cache-streaming (evict-first) hint.
__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}

}  // namespace dspark
