// Confidence head and survival product.
//
// weigao.cc DSpark-vs-MTP page, "3. confidence head": c_k = P(position k survives |
// positions < k accepted) from one linear layer on [output_hidden_k ;
// markov_embedding(prev_token)] (AcceptRatePredictor with confidence_head_with_markov),
// here followed by a sigmoid; the Markov embedding is the W1 row of the predecessor.
// billytse.dev DSpark page, section 5: a_j = prod_{i<=j} c_i.
//
// One CTA per request, wpp warps per draft position (wpp = min(4, 32 / gamma)): each
// warp accumulates its share of the h dot product with up to eight independent 128-bit
// loads per lane in flight (h is an input, so the first of them are issued before the
// kernel waits for the draft), the position's first warp adds the bf16 Markov row, and
// thread 0 applies the sigmoid and multiplies the survival left to right.
//
// With the scheduler fused in (dspark_confidence_schedule), every CTA counts itself in a
// workspace counter after its survivals are written (a fence, then an atomic add); the CTA
// that counts last runs the prefix scheduler of schedule.cu over all of them and resets
// the counter.  Nothing waits: the last CTA simply finds every other one done.
#include "schedule_block.cuh"

namespace dspark {
namespace {

struct SchedArgs {
  const float* sps;
  int32_t* ell;
  int32_t* B_total;
  double* theta;
  unsigned int* done;        // zero between calls
  int Npad;
};

template <bool Sched>
__global__ void __launch_bounds__(1024) confidence_kernel(
    const float* __restrict__ h, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, const uint16_t* __restrict__ W1,
    const float* __restrict__ w_c, float b_c, int gamma, int H, int r, int V, int wpp,
    float* __restrict__ c_out, float* __restrict__ a_out, int* err, SchedArgs sa) {
  __shared__ float part_s[32];
  __shared__ int last_s;
  constexpr int kBatch = 8;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = warp / wpp, part = warp - k * wpp;    // 0-based position, share of H
  const size_t o = (size_t)b * gamma + k;
  const int H4 = H >> 2, stride = 32 * wpp;
  const float4* hv = reinterpret_cast<const float4*>(h + o * H);
  const float4* wv = reinterpret_cast<const float4*>(w_c);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  auto load_batch = [&](int base, float4 (&x)[kBatch]) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + stride * u;
      x[u] = i < H4 ? __ldcs(hv + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto use_batch = [&](int base, const float4 (&x)[kBatch]) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + stride * u;
      if (i < H4) {
        const float4 w = __ldg(wv + i);
        acc[u & 3] = fmaf(x[u].x, w.x, acc[u & 3]);
        acc[u & 3] = fmaf(x[u].y, w.y, acc[u & 3]);
        acc[u & 3] = fmaf(x[u].z, w.z, acc[u & 3]);
        acc[u & 3] = fmaf(x[u].w, w.w, acc[u & 3]);
      }
    }
  };
  // h does not depend on the previous kernel: the first batch is in flight while it drains
  const int base0 = part * 32 + lane;
  float4 x[kBatch];
  load_batch(base0, x);
  pdl_wait();                 // the drafted tokens come from the previous kernel
  pdl_launch_dependents();
  use_batch(base0, x);
  for (int base = base0 + stride * kBatch; base < H4; base += stride * kBatch) {
    load_batch(base, x);
    use_batch(base, x);
  }
  if (part == 0) {
    // the Markov row: 8 bf16 (16 bytes) per lane and step (r % 16 == 0)
    int prev = (k == 0) ? anchor[b] : tokens[o - 1];
    if (!(prev >= 0 && prev < V)) {
      if (lane == 0) set_device_error(err, DSPARK_ERR_DEVICE_CHECK);
      prev = 0;
    }
    const uint16_t* e = W1 + (size_t)prev * r;
    for (int i = 8 * lane; i < r; i += 256) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(e + i));
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w_c + H + i));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w_c + H + i + 4));
      acc[0] = fmaf(__uint_as_float(q.x << 16), w0.x, acc[0]);
      acc[1] = fmaf(__uint_as_float(q.x & 0xFFFF0000u), w0.y, acc[1]);
      acc[2] = fmaf(__uint_as_float(q.y << 16), w0.z, acc[2]);
      acc[3] = fmaf(__uint_as_float(q.y & 0xFFFF0000u), w0.w, acc[3]);
      acc[0] = fmaf(__uint_as_float(q.z << 16), w1.x, acc[0]);
      acc[1] = fmaf(__uint_as_float(q.z & 0xFFFF0000u), w1.y, acc[1]);
      acc[2] = fmaf(__uint_as_float(q.w << 16), w1.z, acc[2]);
      acc[3] = fmaf(__uint_as_float(q.w & 0xFFFF0000u), w1.w, acc[3]);
    }
  }
  float accs = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) accs += __shfl_xor_sync(0xffffffffu, accs, m);
  if (lane == 0) part_s[warp] = accs;
  __syncthreads();
  if (threadIdx.x == 0) {
    float surv = 1.f;
    for (int j = 0; j < gamma; ++j) {
      float logit = 0.f;
      for (int q = 0; q < wpp; ++q) logit += part_s[j * wpp + q];
      const float c = 1.f / (1.f + expf(-(logit + b_c)));
      surv *= c;
      c_out[(size_t)b * gamma + j] = c;
      a_out[(size_t)b * gamma + j] = surv;
    }
  }
  if constexpr (Sched) {
    if (threadIdx.x == 0) {
      __threadfence();            // this CTA's survivals before its count
      last_s = atomicAdd(sa.done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (last_s) {
      __threadfence();            // every other CTA's survivals after their counts
      extern __shared__ unsigned long long keys[];
      schedule_block<false>(a_out, (int)gridDim.x, gamma, sa.Npad, sa.sps, nullptr, nullptr, sa.ell,
                     sa.B_total, sa.theta, keys, (size_t)sa.Npad * sizeof(unsigned long long));
      if (threadIdx.x == 0) *sa.done = 0u;
    }
  }
}

}  // namespace

cudaError_t launch_confidence(const float* h, const int32_t* anchor, const int32_t* tokens,
                              const uint16_t* W1, const float* w_c, float b_c, int B, int gamma,
                              int H, int r, int V, float* c, float* a, int* err,
                              cudaStream_t stream) {
  int wpp = 32 / gamma;
  if (wpp > 4) wpp = 4;
  if (wpp < 1) wpp = 1;
  SchedArgs sa = {};
  return launch_pdl(confidence_kernel<false>, dim3(B), dim3(32 * wpp * gamma), 0, stream, h,
                    anchor, tokens, W1, w_c, b_c, gamma, H, r, V, wpp, c, a, err, sa);
}

cudaError_t launch_confidence_schedule(const float* h, const int32_t* anchor,
                                       const int32_t* tokens, const uint16_t* W1,
                                       const float* w_c, float b_c, int B, int gamma, int H,
                                       int r, int V, const float* sps, float* c, float* a,
                                       int32_t* ell, int32_t* B_total, double* theta,
                                       unsigned int* done, int* err, cudaStream_t stream) {
  int wpp = 32 / gamma;
  if (wpp > 4) wpp = 4;
  if (wpp < 1) wpp = 1;
  const int N = B * gamma;
  int Npad = 2;
  while (Npad < N) Npad <<= 1;
  static std::atomic<int> cache[kMaxCachedDevices];
  const int ok = per_device_grid(cache, [] {
    return cudaFuncSetAttribute(confidence_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(kMaxScheduleItems * sizeof(unsigned long long))) == cudaSuccess
               ? 1 : -1;
  });
  if (ok <= 0) return cudaErrorInvalidConfiguration;
  SchedArgs sa;
  sa.sps = sps;
  sa.ell = ell;
  sa.B_total = B_total;
  sa.theta = theta;
  sa.done = done;
  sa.Npad = Npad;
  return launch_pdl(confidence_kernel<true>, dim3(B), dim3(32 * wpp * gamma),
                    (size_t)Npad * sizeof(unsigned long long), stream, h, anchor, tokens, W1, w_c,
                    b_c, gamma, H, r, V, wpp, c, a, err, sa);
}

}  // namespace dspark
