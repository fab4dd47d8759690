// Confidence head and survival product.
//
// weigao.cc DSpark-vs-MTP page, "3. confidence head": c_k = P(position k survives |
// positions < k accepted) from one linear layer on [output_hidden_k ;
// markov_embedding(prev_token)] (AcceptRatePredictor with confidence_head_with_markov),
// here followed by a sigmoid; the Markov embedding is the W1 row of the predecessor.
// billytse.dev DSpark page, section 5: a_j = prod_{i<=j} c_i.
//
// One CTA per request, one warp per draft position: each lane accumulates its share of
// the two dot products with 128-bit loads (fp32 fused multiply-add chains), the warp
// reduces, and thread 0 applies the sigmoid and multiplies the survival left to right.
#include "internal.h"

namespace dspark {
namespace {

__global__ void confidence_kernel(const float* __restrict__ h, const int32_t* __restrict__ anchor,
                                  const int32_t* __restrict__ tokens,
                                  const uint16_t* __restrict__ W1, const float* __restrict__ w_c,
                                  float b_c, int gamma, int H, int r, int V,
                                  float* __restrict__ c_out, float* __restrict__ a_out, int* err) {
  __shared__ float logit[32];
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
    float acc = 0.f;
    const float4* hv = reinterpret_cast<const float4*>(h + o * H);
    const float4* wv = reinterpret_cast<const float4*>(w_c);
    for (int i = lane; i < (H >> 2); i += 32) {
      const float4 x = __ldcs(hv + i);
      const float4 w = __ldg(wv + i);
      acc = fmaf(x.x, w.x, acc);
      acc = fmaf(x.y, w.y, acc);
      acc = fmaf(x.z, w.z, acc);
      acc = fmaf(x.w, w.w, acc);
    }
    const uint16_t* e = W1 + (size_t)prev * r;
    for (int i = lane; i < r; i += 32) acc = fmaf(bf16_bits_to_float(__ldg(e + i)), __ldg(w_c + H + i), acc);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) logit[k] = acc;
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
  confidence_kernel<<<B, 32 * gamma, 0, stream>>>(h, anchor, tokens, W1, w_c, b_c, gamma, H, r, V,
                                                  c, a, err);
  return cudaGetLastError();
}

}  // namespace dspark
