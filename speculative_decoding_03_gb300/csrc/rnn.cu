// The RNN head's weight preparation and its hidden-state projection.
//
// weigao.cc DSpark-vs-MTP page, "2. Markov head and RNN head": each step of the head
// concatenates the previous state, the previous token's embedding and the position's
// hidden state, and one linear layer splits the result into gate, candidate and output
// (state_k = gate * state_{k-1} + (1 - gate) * candidate; bias_k = W2 tanh(output)).
// W_rnn [2r + H, 3r] bf16 holds that layer: rows [0, r) take the state, rows [r, 2r) the
// token embedding (the head's W1 row), rows [2r, 2r + H) the hidden state; column blocks
// [0, r), [r, 2r), [2r, 3r) are gate, candidate and output.
//
//   rnn_pack_kernel     Wrec[c][j] = W_rnn[j][c] for j < 2r: the recurrent rows transposed,
//                       so that the draft's recurrence reads each output column's 2r
//                       weights contiguously (done once per weights)
//   rnn_project_kernel  hp[m][c] = b_rnn[c] + sum_j h[m][j] W_rnn[2r + j][c]: the part of
//                       the layer that does not depend on the drafted tokens, for every
//                       (request, position) row m at once, before the draft, on the tensor
//                       cores (see the kernel).
#include <cooperative_groups.h>
#include <string.h>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace cg = cooperative_groups;

namespace dspark {
namespace {

constexpr int kPackTile = 32;

__global__ void __launch_bounds__(kPackTile * 8) rnn_pack_kernel(const uint16_t* __restrict__ W,
                                                                 int r, uint16_t* __restrict__ Wrec) {
  __shared__ uint16_t tile[kPackTile][kPackTile + 2];
  const int C = 3 * r, J = 2 * r;
  const int c0 = blockIdx.x * kPackTile, j0 = blockIdx.y * kPackTile;
  const int tx = threadIdx.x % kPackTile, ty = threadIdx.x / kPackTile;
  for (int y = ty; y < kPackTile; y += 8) {
    const int j = j0 + y, c = c0 + tx;
    tile[y][tx] = (j < J && c < C) ? W[(size_t)j * C + c] : (uint16_t)0;
  }
  __syncthreads();
  for (int y = ty; y < kPackTile; y += 8) {
    const int c = c0 + y, j = j0 + tx;
    if (c < C && j < J) Wrec[(size_t)c * J + j] = tile[tx][y];
  }
}

// The projection on the tensor cores.  h is fp32 and W_rnn bf16: h is split exactly into
// three bf16 terms, h = h0 + h1 + h2 (h0 = bf16(h), h1 = bf16(h - h0), h2 = h - h0 - h1,
// which has at most 8 significant bits, so it is a bf16 value), every product of a bf16
// term and a bf16 weight is exact in fp32, and the MMAs accumulate the three products in
// fp32: the result has fp32 accuracy.
//
// D (128 output columns c = TMEM lanes, 128 rows m = TMEM columns) = W_h^T h^T: A is the
// weight tile, MN-major (W_rnn's hidden rows are [H][3r], c contiguous), loaded by TMA in
// two 64-column boxes with the 128-byte swizzle; B is the three planes of h, K-major,
// written by eight converter warps in the 128-byte-swizzled layout (16-byte chunk q of row
// n at chunk q ^ (n % 8) of line n).  K is cut into 64-wide chunks and the chunks are split
// eight ways over a thread-block cluster; a 3-stage ring (A tile + three planes, 64 KB a
// stage) overlaps the TMA loads, the conversion of the next chunk (its h values loaded
// into registers one chunk ahead) and the MMAs.  Each CTA then writes its partial tile to
// shared memory and sums one eighth of the rows over the eight partial tiles, read from
// the cluster's shared memory in rank order (a fixed order: the result does not depend on
// scheduling), adds the bias and stores hp.  The waits are bounded; the call has no status
// word, so a CTA whose wait ran out writes NaN to its rows of the tile instead.
constexpr int kPrjM = 128, kPrjN = 128, kPrjK = 64, kPrjStages = 3, kPrjSplit = 8;
constexpr int kPrjConvWarps = 8, kPrjThreads = (kPrjConvWarps + 1) * 32;
constexpr int kPrjABytes = kPrjM * kPrjK * 2;               // 16 KB
constexpr int kPrjPlaneBytes = kPrjN * kPrjK * 2;           // 16 KB
constexpr int kPrjStageBytes = kPrjABytes + 3 * kPrjPlaneBytes;
constexpr int kPrjSmemBytes = kPrjStages * kPrjStageBytes + 1024;
constexpr int kPrjGroups = kPrjN * kPrjK / 8 / (kPrjConvWarps * 32);   // 8-element groups a thread
constexpr unsigned long long kPrjTimeoutNs = 2000000000ull;
static_assert(kPrjM * kPrjN * 4 <= kPrjStages * kPrjStageBytes, "partial tile fits the ring");

__device__ __forceinline__ uint32_t prj_bf16(float x) {    // round to nearest even (finite x)
  const uint32_t u = __float_as_uint(x);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__global__ void __cluster_dims__(1, 1, kPrjSplit) __launch_bounds__(kPrjThreads, 1)
rnn_project_kernel(const __grid_constant__ CUtensorMap wmap, const float* __restrict__ h,
                   const float* __restrict__ bias, int M, int H, int C, float* __restrict__ hp) {
  using namespace sm100;
  extern __shared__ uint8_t prj_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(prj_smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t full[kPrjStages], empty[kPrjStages], conv[kPrjStages], done;
  __shared__ uint32_t tmem_s;
  __shared__ int fail_s;
  cg::cluster_group cluster = cg::this_cluster();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * kPrjM, m0 = blockIdx.y * kPrjN;
  const int split = (int)cluster.block_rank();
  const int n_chunks = (H + kPrjK - 1) / kPrjK;
  const int ch_lo = split * n_chunks / kPrjSplit;
  const int nc = (split + 1) * n_chunks / kPrjSplit - ch_lo;      // may be 0 for a small H
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPrjStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&conv[i], kPrjConvWarps);
    }
    mbar_init(&done, 1);
    fail_s = 0;
    fence_mbar_init();
  }
  if (warp == kPrjConvWarps) {
    tmem_alloc(&tmem_s, kPrjN);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_s;
  pdl_wait();
  pdl_launch_dependents();

  if (warp == kPrjConvWarps) {
    // ------------------------------------------------- TMA producer and MMA issuer (lane 0)
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      const uint64_t keep = policy_evict_last();
      auto load_a = [&](int i) {
        const int s = i % kPrjStages, k0 = (ch_lo + i) * kPrjK;
        uint8_t* a = smem + s * kPrjStageBytes;
        mbar_arrive_expect_tx(&full[s], (uint32_t)kPrjABytes);
        tma_load_2d(a, &wmap, &full[s], c0, k0, keep);
        tma_load_2d(a + kPrjK * 128, &wmap, &full[s], c0 + 64, k0, keep);
      };
      for (int i = 0; i < nc && i < kPrjStages; ++i) load_a(i);
      const uint32_t idesc = idesc_bf16_f32(kPrjM, kPrjN, 1, 0);
      bool ok = true;
      int issued = nc < kPrjStages ? nc : kPrjStages;   // chunks whose A tile was requested
      for (int i = 0; i < nc && ok; ++i) {
        const int s = i % kPrjStages;
        const uint32_t par = (uint32_t)(i / kPrjStages) & 1u;
        ok = mbar_wait(&full[s], par, kPrjTimeoutNs) && mbar_wait(&conv[s], par, kPrjTimeoutNs);
        if (!ok) break;
        tc_fence_after_sync();
        uint8_t* st = smem + s * kPrjStageBytes;
        // A: 16 K rows of the MN-major tile are 2048 bytes apart, the second 64-column box
        // kPrjK * 128 bytes after the first; B: 32 bytes per 16-element K step in a plane
        const uint64_t a_base = smem_desc(smem_u32(st), kPrjK * 128, 1024, kSwizzle128B);
#pragma unroll
        for (int kk = 0; kk < kPrjK / 16; ++kk) {
#pragma unroll
          for (int pl = 0; pl < 3; ++pl) {
            const uint64_t b_base = smem_desc(smem_u32(st + kPrjABytes + pl * kPrjPlaneBytes), 16,
                                              1024, kSwizzle128B);
            umma_bf16_f32(tmem, a_base + (uint64_t)(kk * (2048 >> 4)), b_base + (uint64_t)(kk * 2),
                          idesc, (i > 0 || kk > 0 || pl > 0) ? 1u : 0u);
          }
        }
        umma_commit(&empty[s]);
        if (i + kPrjStages < nc) {
          // the stage is reloaded once its MMAs have completed
          if (!(ok = mbar_wait(&empty[s], par, kPrjTimeoutNs))) break;
          load_a(i + kPrjStages);
          ++issued;
        }
      }
      if (!ok) atomicExch(&fail_s, 1);
      // done arrives once every issued MMA has completed (a CTA without K chunks issues
      // none and does not wait for it); every issued copy lands before the CTA goes on
      if (nc > 0) umma_commit(&done);
      for (int i = 0; i < issued; ++i) {
        const int s = i % kPrjStages;
        if (i + kPrjStages >= issued)
          mbar_wait(&full[s], (uint32_t)(i / kPrjStages) & 1u, kPrjTimeoutNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ converters
    // a thread's group g: row n = idx / 8 and 8-element K chunk q = idx % 8 of the stage,
    // idx = thread + 256 g
    float4 nxt[kPrjGroups][2];
    auto load_h = [&](int i) {
      const int k0 = (ch_lo + i) * kPrjK;
#pragma unroll
      for (int g = 0; g < kPrjGroups; ++g) {
        const int idx = threadIdx.x + g * kPrjConvWarps * 32, n = idx >> 3, q = idx & 7;
        const int m = m0 + n, k = k0 + q * 8;
        const float* src = h + (size_t)m * H + k;
        nxt[g][0] = (m < M && k < H) ? __ldg(reinterpret_cast<const float4*>(src))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        nxt[g][1] = (m < M && k + 4 < H) ? __ldg(reinterpret_cast<const float4*>(src + 4))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    if (nc > 0) load_h(0);
    for (int i = 0; i < nc; ++i) {
      const int s = i % kPrjStages;
      float x[kPrjGroups][8];
#pragma unroll
      for (int g = 0; g < kPrjGroups; ++g) {
        x[g][0] = nxt[g][0].x; x[g][1] = nxt[g][0].y; x[g][2] = nxt[g][0].z; x[g][3] = nxt[g][0].w;
        x[g][4] = nxt[g][1].x; x[g][5] = nxt[g][1].y; x[g][6] = nxt[g][1].z; x[g][7] = nxt[g][1].w;
      }
      if (i + 1 < nc) load_h(i + 1);
      // the stage's planes are free once the MMAs of chunk i - kPrjStages have completed
      if (i >= kPrjStages &&
          !mbar_wait(&empty[s], (uint32_t)(i / kPrjStages - 1) & 1u, kPrjTimeoutNs))
        atomicExch(&fail_s, 1);
      uint8_t* pl0 = smem + s * kPrjStageBytes + kPrjABytes;
#pragma unroll
      for (int g = 0; g < kPrjGroups; ++g) {
        const int idx = threadIdx.x + g * kPrjConvWarps * 32, n = idx >> 3, q = idx & 7;
        uint32_t w0[4], w1[4], w2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t t0[2], t1[2], t2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float v = x[g][2 * e + u];
            t0[u] = prj_bf16(v);
            const float r1 = v - __uint_as_float(t0[u] << 16);
            t1[u] = prj_bf16(r1);
            t2[u] = prj_bf16(r1 - __uint_as_float(t1[u] << 16));
          }
          w0[e] = t0[0] | (t0[1] << 16);
          w1[e] = t1[0] | (t1[1] << 16);
          w2[e] = t2[0] | (t2[1] << 16);
        }
        const size_t off = (size_t)n * 128 + (size_t)((q ^ (n & 7)) << 4);
        *reinterpret_cast<uint4*>(pl0 + off) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
        *reinterpret_cast<uint4*>(pl0 + kPrjPlaneBytes + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
        *reinterpret_cast<uint4*>(pl0 + 2 * kPrjPlaneBytes + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv[s]);
    }
  }

  // ---------------------------------------------------------------------- epilogue
  if (nc > 0 && !mbar_wait(&done, 0, kPrjTimeoutNs)) atomicExch(&fail_s, 1);
  tc_fence_after_sync();
  __syncthreads();                      // every MMA and conversion done: the ring is free
  float* part = reinterpret_cast<float*>(smem);   // [128 rows n][128 columns c]
  if (warp < kPrjConvWarps) {
    const int qd = warp & 3, half = warp >> 2;    // TMEM lane quarter, column half
    const int c = qd * 32 + lane;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int n0 = half * 64 + cc * 16;
      float v[16];
      if (nc > 0) {
        tmem_ld_32x32b_x16(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)n0, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) part[(n0 + j) * kPrjM + c] = v[j];
    }
  }
  tc_fence_before_sync();
  cluster.sync();
  {
    // rows [split * 16, split * 16 + 16) of the tile, summed over the ranks in order
    constexpr int kRows = kPrjN / kPrjSplit, kQuads = kRows * kPrjM / 4;
    int failed = 0;
    for (int rk = 0; rk < kPrjSplit; ++rk) failed |= *cluster.map_shared_rank(&fail_s, rk);
    for (int t = threadIdx.x; t < kQuads; t += kPrjThreads) {
      const int n = split * kRows + t / (kPrjM / 4), c4 = (t % (kPrjM / 4)) * 4;
      const int m = m0 + n, c = c0 + c4;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int rk = 0; rk < kPrjSplit; ++rk) {
        const float4 v = *reinterpret_cast<const float4*>(cluster.map_shared_rank(part, rk) + n * kPrjM + c4);
        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
      }
      if (m < M && c < C) {
        const float4 b4 = *reinterpret_cast<const float4*>(bias + c);
        float4 o = make_float4(sum.x + b4.x, sum.y + b4.y, sum.z + b4.z, sum.w + b4.w);
        if (failed) o = make_float4(__int_as_float(0x7FC00000), __int_as_float(0x7FC00000),
                                    __int_as_float(0x7FC00000), __int_as_float(0x7FC00000));
        *reinterpret_cast<float4*>(hp + (size_t)m * C + c) = o;
      }
    }
  }
  cluster.sync();                       // the other CTAs' tiles stay until every read is done
  if (warp == kPrjConvWarps) tmem_dealloc(tmem, kPrjN);
}

}  // namespace

cudaError_t launch_rnn_pack(const uint16_t* W_rnn, int r, uint16_t* Wrec, cudaStream_t stream) {
  const dim3 grid(cdiv(3 * r, kPackTile), cdiv(2 * r, kPackTile));
  rnn_pack_kernel<<<grid, kPackTile * 8, 0, stream>>>(W_rnn, r, Wrec);
  return cudaGetLastError();
}

cudaError_t launch_rnn_project(const float* h, const uint16_t* W_rnn, const float* b_rnn, int M,
                               int H, int r, float* hp, cudaStream_t stream) {
  static std::atomic<int> attr_set[kMaxCachedDevices];
  if (per_device_grid(attr_set, [] {
        return cudaFuncSetAttribute(rnn_project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kPrjSmemBytes) == cudaSuccess ? 1 : -1;
      }) <= 0)
    return cudaErrorInvalidValue;
  const int C = 3 * r;
  // the hidden-state rows W_rnn[2r:] as a {C, H} tensor: 64-column boxes of 64 K rows
  CUtensorMap wmap;
  memset(&wmap, 0, sizeof(wmap));
  if (!encode_w2_map(&wmap, W_rnn + (size_t)2 * r * C, C, H, kPrjK)) return cudaErrorInvalidValue;
  const dim3 grid(cdiv(C, kPrjM), cdiv(M, kPrjN), kPrjSplit);
  return launch_pdl(rnn_project_kernel, grid, dim3(kPrjThreads), (size_t)kPrjSmemBytes, stream, wmap,
                    h, b_rnn, M, H, C, hp);
}

}  // namespace dspark
