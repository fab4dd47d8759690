// Confidence head and survival product.
//
// weigao.cc DSpark-vs-MTP page, "3. confidence head": c_k = P(position k survives |
// positions < k accepted) from one linear layer on [output_hidden_k ;
// markov_embedding(prev_token)] (AcceptRatePredictor with confidence_head_with_markov),
// here followed by a sigmoid; the Markov embedding is the W1 row of the predecessor.
// billytse.dev DSpark page, section 5: a_j = prod_{i<=j} c_i.
//
// One CTA per request, one warp per draft position: each lane accumulates its share of
// the two dot products (batches of eight independent 128-bit loads of h and w_c in flight
// per lane, one 16-byte load of the bf16 Markov row), the warp reduces, and thread 0
// applies the sigmoid and multiplies the survival left to right.
#include "internal.h"

namespace dspark {
namespace {

__global__ void confidence_kernel(const float* __restrict__ h, const int32_t* __restrict__ anchor,
                                  const int32_t* __restrict__ tokens,
                                  const uint16_t* __restrict__ W1, const float* __restrict__ w_c,
                                  float b_c, int gamma, int H, int r, int V,
                                  float* __restrict__ c_out, float* __restrict__ a_out, int* err) {
  __shared__ float logit[32];
  pdl_wait();                 // the drafted tokens come from the previous kernel
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int k = threadIdx.x >> 5;  // 0-based position handled by this warp
  const int lane = threadIdx.x & 31;
  if (k < gamma) {
    const size_t o = (size_t)b * gamma + k;
    int prev = (k == 0) ? anchor[b] : tokens[o - 1];
    bool ok = prev >= 0 && prev < V;
    if (!ok) {
      if (lane == 0) set_device_error(err, DSPARK_ERR_DEVICE_CHECK);
      prev = 0;
    }
    constexpr int kBatch = 8;
    float acc[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) acc[u] = 0.f;
    const float4* hv = reinterpret_cast<const float4*>(h + o * H);
    const float4* wv = reinterpret_cast<const float4*>(w_c);
    const int H4 = H >> 2;
    for (int i0 = lane; i0 < H4; i0 += 32 * kBatch) {
      float4 x[kBatch], w[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + 32 * u;
        if (i < H4) {
          x[u] = __ldcs(hv + i);
          w[u] = __ldg(wv + i);
        } else {
          x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          w[u] = x[u];
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        acc[u] = fmaf(x[u].x, w[u].x, acc[u]);
        acc[u] = fmaf(x[u].y, w[u].y, acc[u]);
        acc[u] = fmaf(x[u].z, w[u].z, acc[u]);
        acc[u] = fmaf(x[u].w, w[u].w, acc[u]);
      }
    }
    // the Markov row: 8 bf16 (16 bytes) per lane and step (r % 16 == 0)
    const uint16_t* e = W1 + (size_t)prev * r;
    for (int i = 8 * lane; i < r; i += 256) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(e + i));
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w_c + H + i));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w_c + H + i + 4));
      acc[0] = fmaf(__uint_as_float(q.x << 16), w0.x, acc[0]);
      acc[1] = fmaf(__uint_as_float(q.x & 0xFFFF0000u), w0.y, acc[1]);
      acc[2] = fmaf(__uint_as_float(q.y << 16), w0.z, acc[2]);
      acc[3] = fmaf(__uint_as_float(q.y & 0xFFFF0000u), w0.w, acc[3]);
      acc[4] = fmaf(__uint_as_float(q.z << 16), w1.x, acc[4]);
      acc[5] = fmaf(__uint_as_float(q.z & 0xFFFF0000u), w1.y, acc[5]);
      acc[6] = fmaf(__uint_as_float(q.w << 16), w1.z, acc[6]);
      acc[7] = fmaf(__uint_as_float(q.w & 0xFFFF0000u), w1.w, acc[7]);
    }
    float accs = 0.f;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) accs += acc[u];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) accs += __shfl_xor_sync(0xffffffffu, accs, m);
    if (lane == 0) logit[k] = accs;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float surv = 1.f;
    for (int j = 0; j < gamma; ++j) {
      const float c = 1.f / (1.f + expf(-(logit[j] + b_c)));
      surv *= c;
      c_out[(size_t)b * gamma + j] = c;
      a_out[(size_t)b * gamma + j] = surv;
    }
  }
}

}  // namespace

cudaError_t launch_confidence(const float* h, const int32_t* anchor, const int32_t* tokens,
                              const uint16_t* W1, const float* w_c, float b_c, int B, int gamma,
                              int H, int r, int V, float* c, float* a, int* err,
                              cudaStream_t stream) {
  return launch_pdl(confidence_kernel, dim3(B), dim3(32 * gamma), 0, stream, h, anchor, tokens, W1,
                    w_c, b_c, gamma, H, r, V, c, a, err);
}

}  // namespace dspark
