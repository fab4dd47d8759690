// Draft sampling for one position k: softmax statistics and the Gumbel-max draw over
// z = U_k + bias in one streaming pass.
//
// billytse.dev DSpark page, section 3.2: p_k(v | x_<k) = softmax(U_k(v) + B_k(x_<k, v));
// the sample is drawn by Gumbel-max, x_k = argmax_v (z_v + g_v), g_v = -log(E_v),
// E_v = -log(u_v) ~ Exp(1).  Equivalently x_k = argmax_v exp(z_v - m) / E_v for any
// reference m (the "exponential race" form), which needs no log for most elements:
//
//   each thread streams float4 pieces of its row segment, keeps the running max m, the
//   running sum s = sum exp(z - m) and the best ratio br = exp(z_best - m) / E_best,
//   rescaling s and br when m grows.  Since E = -log(1 - w) >= w with w = 1 - u, an
//   element can only beat br if exp(z - m) > br * w; only those elements evaluate the
//   accurate E = -log1p(-w) and the exact ratio.
//
// Segments are merged as (m, s, score = m + log br, index) with ties to the smaller
// index; the last CTA of a row merges all segments and writes x_k, q_k(x_k), m and s.
#include "internal.h"

namespace dspark {
namespace {

__global__ void __launch_bounds__(kSampleThreads) draft_sample_kernel(
    const float* __restrict__ U, const float* __restrict__ bias, int gamma, int V, int k,
    uint64_t seed, int splits, int seg, RowState* __restrict__ partials,
    uint32_t* __restrict__ counters, int32_t* __restrict__ tokens, float* __restrict__ q_tok,
    float* __restrict__ row_max, float* __restrict__ row_sumexp) {
  __shared__ RowState red[32];
  __shared__ int is_last;
  const int split = blockIdx.x, b = blockIdx.y;
  const int v_begin = split * seg;
  const int v_end = min(V, v_begin + seg);
  const float* Urow = U + ((size_t)b * gamma + (k - 1)) * V;
  const float* Brow = bias + (size_t)b * V;

  float m = -INFINITY, s = 0.f, br = 0.f, bz = -INFINITY;
  int bi = -1;
  for (int v = v_begin + 4 * threadIdx.x; v < v_end; v += 4 * kSampleThreads) {
    const float4 u4 = ld_stream_f4(Urow + v);
    const float4 b4 = __ldcg(reinterpret_cast<const float4*>(Brow + v));
    const float z[4] = {u4.x + b4.x, u4.y + b4.y, u4.z + b4.z, u4.w + b4.w};
    const float mn = fmaxf(fmaxf(m, fmaxf(z[0], z[1])), fmaxf(z[2], z[3]));
    const float f = ex2_approx((m - mn) * kLog2e);   // 0 on the first piece (m = -inf)
    s *= f;
    br *= f;
    m = mn;
    const uint4 d = draw_block(seed, (uint32_t)(v >> 2), (uint32_t)k, (uint32_t)b, 0u);
    const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float e = ex2_approx((z[i] - m) * kLog2e);
      s += e;
      const float w = one_minus_u01(dw[i]);
      if (e > br * w) {                 // only candidates pay for the accurate log
        const float ratio = e / exp1_from_w(w);
        if (ratio > br) {
          br = ratio;
          bi = v + i;
          bz = z[i];
        }
      }
    }
  }
  RowState st;
  st.m = m;
  st.s = s;
  st.idx = bi;
  st.z = bz;
  st.score = (bi >= 0) ? m + logf(br) : -INFINITY;
  st = row_state_block_reduce(st, red);

  if (threadIdx.x == 0) {
    partials[(size_t)b * splits + split] = st;
    __threadfence();
    const uint32_t done = atomicAdd(&counters[b], 1u);
    is_last = (done == (uint32_t)splits - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (threadIdx.x < 32) {
    RowState acc = row_state_empty();
    for (int i = threadIdx.x; i < splits; i += 32) {
      const RowState* src = partials + (size_t)b * splits + i;
      RowState q;
      q.m = __ldcg(&src->m);
      q.s = __ldcg(&src->s);
      q.score = __ldcg(&src->score);
      q.z = __ldcg(&src->z);
      q.idx = __ldcg(&src->idx);
      acc = row_state_merge(acc, q);
    }
    acc = row_state_warp_reduce(acc);
    if (threadIdx.x == 0) {
      const size_t o = (size_t)b * gamma + (k - 1);
      tokens[o] = acc.idx;
      q_tok[o] = expf(acc.z - acc.m) / acc.s;
      row_max[o] = acc.m;
      row_sumexp[o] = acc.s;
      counters[b] = 0u;
    }
  }
}

}  // namespace

cudaError_t launch_draft_sample(const Plan& p, const float* U, const float* bias, int k,
                                uint64_t seed, RowState* partials, uint32_t* counters,
                                int32_t* tokens, float* q_tok, float* row_max, float* row_sumexp,
                                int* err, cudaStream_t stream) {
  (void)err;
  dim3 grid(p.draft.splits, p.B);
  draft_sample_kernel<<<grid, kSampleThreads, 0, stream>>>(U, bias, p.gamma, p.V, k, seed,
                                                           p.draft.splits, p.draft.seg, partials,
                                                           counters, tokens, q_tok, row_max,
                                                           row_sumexp);
  return cudaGetLastError();
}

}  // namespace dspark
