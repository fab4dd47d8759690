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
//                       (request, position) row m at once, before the draft.  A CUDA-core
//                       fp32 contraction (bf16 weights are exact in fp32): 64 x 64 output
//                       tiles split four ways along K over a thread-block cluster, reduced
//                       through distributed shared memory.
#include <cooperative_groups.h>

#include "internal.h"

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

constexpr int kProjM = 64, kProjN = 64, kProjK = 32, kProjThreads = 256;
constexpr int kProjSplit = 4;           // CTAs of a cluster, each a quarter of K

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

struct ProjSmem {
  float hsT[2][kProjK][kProjM + 4];     // h slices, transposed: [j][m]
  float ws[2][kProjK][kProjN];          // W slices: [j][c]
};

// M = rows of h (B * gamma), H = hidden size (multiple of 4), r = rank.  Grid (3r / 64,
// ceil(M / 64), 4) in clusters of (1, 1, 4): the four CTAs of a cluster compute the same
// 64 x 64 output tile over a quarter of K each (4 x 4 outputs per thread, the next K slice
// loaded into registers while the current one is used), then each sums one quarter of the
// tile's rows over the four partial tiles, read from the cluster's shared memory in rank
// order (a fixed order: the result does not depend on scheduling).
__global__ void __cluster_dims__(1, 1, kProjSplit) __launch_bounds__(kProjThreads)
rnn_project_kernel(const float* __restrict__ h, const uint16_t* __restrict__ W,
                   const float* __restrict__ bias, int M, int H, int r, float* __restrict__ hp) {
  __shared__ __align__(16) unsigned char raw[sizeof(ProjSmem) > kProjM * kProjN * 4
                                             ? sizeof(ProjSmem) : kProjM * kProjN * 4];
  ProjSmem& sm = *reinterpret_cast<ProjSmem*>(raw);
  float* part = reinterpret_cast<float*>(raw);     // [64][64] partial tile, after the loop
  cg::cluster_group cluster = cg::this_cluster();
  pdl_wait();
  pdl_launch_dependents();
  const int C = 3 * r;
  const int m0 = blockIdx.y * kProjM, c0 = blockIdx.x * kProjN;
  const int split = (int)cluster.block_rank();
  const int n_slices = (H + kProjK - 1) / kProjK;
  const int s_lo = split * n_slices / kProjSplit, s_hi = (split + 1) * n_slices / kProjSplit;
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;          // 4 columns, 4 rows per thread
  const uint16_t* Wh = W + (size_t)2 * r * C;      // the hidden-state rows
  // loader roles: h 64 x 32 floats = two float4 per thread; W 32 x 64 bf16 = one uint4
  const int hm = tid / 8, hj = (tid % 8) * 4;
  const int wj = tid / 8, wc = (tid % 8) * 8;
  float4 hv[2];
  uint4 wv;
  auto load = [&](int sl) {
    const int k0 = sl * kProjK;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int m = m0 + hm + 32 * u;
      hv[u] = (m < M && k0 + hj < H) ? __ldg(reinterpret_cast<const float4*>(h + (size_t)m * H + k0 + hj))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    wv = (k0 + wj < H && c0 + wc < C) ? __ldg(reinterpret_cast<const uint4*>(Wh + (size_t)(k0 + wj) * C + c0 + wc))
                                      : make_uint4(0u, 0u, 0u, 0u);
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      sm.hsT[buf][hj + 0][hm + 32 * u] = hv[u].x;
      sm.hsT[buf][hj + 1][hm + 32 * u] = hv[u].y;
      sm.hsT[buf][hj + 2][hm + 32 * u] = hv[u].z;
      sm.hsT[buf][hj + 3][hm + 32 * u] = hv[u].w;
    }
    float* d = &sm.ws[buf][wj][wc];
    d[0] = bf16_lo(wv.x); d[1] = bf16_hi(wv.x); d[2] = bf16_lo(wv.y); d[3] = bf16_hi(wv.y);
    d[4] = bf16_lo(wv.z); d[5] = bf16_hi(wv.z); d[6] = bf16_lo(wv.w); d[7] = bf16_hi(wv.w);
  };
  float acc[4][4] = {};
  if (s_lo < s_hi) {
    load(s_lo);
    store(0);
  }
  __syncthreads();
  for (int sl = s_lo; sl < s_hi; ++sl) {
    const int buf = (sl - s_lo) & 1;
    if (sl + 1 < s_hi) load(sl + 1);
#pragma unroll 8
    for (int jj = 0; jj < kProjK; ++jj) {
      const float4 a = *reinterpret_cast<const float4*>(&sm.hsT[buf][jj][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&sm.ws[buf][jj][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (sl + 1 < s_hi) store(buf ^ 1);
    __syncthreads();
  }
  // this CTA's partial tile into its shared memory (the slices are no longer read)
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(part + (ty * 4 + i) * kProjN + tx * 4) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  cluster.sync();
  // rows [16 split, 16 split + 16) of the tile: one float4 per thread, summed in rank order
  {
    const int row = split * (kProjM / kProjSplit) + tid / 16, col = (tid % 16) * 4;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kProjSplit; ++q) {
      const float* rp = cluster.map_shared_rank(part, q);
      const float4 v = *reinterpret_cast<const float4*>(rp + row * kProjN + col);
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    const int m = m0 + row, c = c0 + col;
    if (m < M && c < C) {
      const float4 b4 = *reinterpret_cast<const float4*>(bias + c);
      *reinterpret_cast<float4*>(hp + (size_t)m * C + c) =
          make_float4(sum.x + b4.x, sum.y + b4.y, sum.z + b4.z, sum.w + b4.w);
    }
  }
  cluster.sync();            // the other CTAs' tiles stay in place until every read is done
}

}  // namespace

cudaError_t launch_rnn_pack(const uint16_t* W_rnn, int r, uint16_t* Wrec, cudaStream_t stream) {
  const dim3 grid(cdiv(3 * r, kPackTile), cdiv(2 * r, kPackTile));
  rnn_pack_kernel<<<grid, kPackTile * 8, 0, stream>>>(W_rnn, r, Wrec);
  return cudaGetLastError();
}

cudaError_t launch_rnn_project(const float* h, const uint16_t* W_rnn, const float* b_rnn, int M,
                               int H, int r, float* hp, cudaStream_t stream) {
  const dim3 grid(cdiv(3 * r, kProjN), cdiv(M, kProjM), kProjSplit);
  return launch_pdl(rnn_project_kernel, grid, dim3(kProjThreads), 0, stream, h, W_rnn, b_rnn, M, H,
                    r, hp);
}

}  // namespace dspark
