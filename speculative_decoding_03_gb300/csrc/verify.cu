// Lossless verification of the scheduled draft prefixes.
//
// billytse.dev DSpark page, section 1: accept x_k with probability min(1, p_k(x_k) /
// q_k(x_k)), keep the longest accepted prefix and fix the first rejected position with a
// token drawn from the residual; xhh.club DSpark page (Q&A on the acceptance rule): the
// residual is norm(max(0, p - q)), which makes the output follow p exactly.  When every
// verified position is accepted the target contributes its own bonus token (the tau of
// billytse.dev section 1 counts it), drawn from target row l + 1.
//
// Kernels, in order on the stream:
//   target_stats   for every verified row (b, k <= l_b): max M and log-sum-exp of T[b, k]
//                  and p_k(x_k) (rows are split over CTAs, the last CTA merges)
//   decide         one thread per request: the acceptance tests in order, the first
//                  reject, the accepted prefix, and which row the final token comes from
//   bias_gemm      (shared with the draft) W1[x_{j-1}] W2 for the rows with a reject at j
//   final_sample   Gumbel-max over log(P_j - Q_j) on {P_j > Q_j} (residual), or over
//                  T[b, l+1] (bonus); the last CTA of a row writes the token
//   fallback       only for rows whose residual support came out empty in fp32: Gumbel-
//                  max over T[b, j] with the residual's random stream
#include "internal.h"

namespace dspark {
namespace {

enum : int { kModeNone = 0, kModeResidual = 1, kModeBonus = 2 };

__device__ __forceinline__ int clamp_ell(const int32_t* ell, int b, int gamma, int* err) {
  int L = ell[b];
  if (L < 0 || L > gamma) {
    set_device_error(err, DSPARK_ERR_DEVICE_CHECK);
    L = L < 0 ? 0 : gamma;
  }
  return L;
}

__device__ __forceinline__ RowState load_partial(const RowState* src) {
  RowState q;
  q.m = __ldcg(&src->m);
  q.s = __ldcg(&src->s);
  q.score = __ldcg(&src->score);
  q.z = __ldcg(&src->z);
  q.idx = __ldcg(&src->idx);
  return q;
}

// Gumbel value of the 32-bit draw x: g = -log(-log1p(-w)), w = 1 - U01(x).
__device__ __forceinline__ float gumbel_of(uint32_t x) {
  return -logf(exp1_from_w(one_minus_u01(x)));
}

// Writes this CTA's partial and returns true in the CTA that completes the row.
__device__ __forceinline__ bool publish_partial(RowState st, RowState* slot, uint32_t* counter,
                                                int splits, int* is_last_s) {
  if (threadIdx.x == 0) {
    *slot = st;
    __threadfence();
    const uint32_t done = atomicAdd(counter, 1u);
    *is_last_s = (done == (uint32_t)splits - 1);
  }
  __syncthreads();
  const bool last = *is_last_s != 0;
  if (last) __threadfence();
  return last;
}

__device__ __forceinline__ RowState merge_partials(const RowState* base, int splits) {
  RowState acc = row_state_empty();
  for (int i = threadIdx.x; i < splits; i += 32) acc = row_state_merge(acc, load_partial(base + i));
  return row_state_warp_reduce(acc);
}

// ---------------------------------------------------------------------- target stats
__global__ void __launch_bounds__(kSampleThreads) target_stats_kernel(
    const float* __restrict__ T, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ ell, int gamma, int V, int splits, int seg,
    RowState* __restrict__ partials, uint32_t* __restrict__ counters, float* __restrict__ M_out,
    float* __restrict__ lnS_out, float* __restrict__ p_out, int* err) {
  __shared__ RowState red[32];
  __shared__ int is_last;
  const int row = blockIdx.y;                 // b * gamma + (k - 1)
  const int b = row / gamma, k = row - b * gamma + 1;
  if (k > clamp_ell(ell, b, gamma, nullptr)) return;
  const float* Trow = T + ((size_t)b * (gamma + 1) + (k - 1)) * V;
  const int v_begin = blockIdx.x * seg, v_end = min(V, v_begin + seg);
  float m = -INFINITY, s = 0.f;
  for (int v = v_begin + 4 * threadIdx.x; v < v_end; v += 4 * kSampleThreads) {
    const float4 t = ld_stream_f4(Trow + v);
    const float mn = fmaxf(fmaxf(m, fmaxf(t.x, t.y)), fmaxf(t.z, t.w));
    s *= ex2_approx((m - mn) * kLog2e);
    m = mn;
    s += ex2_approx((t.x - m) * kLog2e) + ex2_approx((t.y - m) * kLog2e) +
         ex2_approx((t.z - m) * kLog2e) + ex2_approx((t.w - m) * kLog2e);
  }
  RowState st = row_state_empty();
  st.m = m;
  st.s = s;
  st = row_state_block_reduce(st, red);
  if (!publish_partial(st, partials + (size_t)row * splits + blockIdx.x, &counters[row], splits,
                       &is_last))
    return;
  if (threadIdx.x < 32) {
    const RowState acc = merge_partials(partials + (size_t)row * splits, splits);
    if (threadIdx.x == 0) {
      const int x = tokens[(size_t)b * gamma + (k - 1)];
      float p = 0.f;
      if (x >= 0 && x < V) {
        p = expf(__ldg(Trow + x) - acc.m) / acc.s;
      } else {
        set_device_error(err, DSPARK_ERR_DEVICE_CHECK);
      }
      M_out[row] = acc.m;
      lnS_out[row] = logf(acc.s);
      p_out[row] = p;
      counters[row] = 0u;
    }
  }
}

// ----------------------------------------------------------------------------- decide
__global__ void decide_kernel(const int32_t* __restrict__ anchor,
                              const int32_t* __restrict__ tokens,
                              const float* __restrict__ q_tok, const float* __restrict__ p_t,
                              const int32_t* __restrict__ ell, int B, int gamma, uint64_t seed,
                              int32_t* __restrict__ accept_len, int32_t* __restrict__ out_tokens,
                              int32_t* __restrict__ n_out, int32_t* __restrict__ mode,
                              int32_t* __restrict__ pos, int32_t* __restrict__ prev_tok,
                              int32_t* __restrict__ fallback, int* err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int L = clamp_ell(ell, b, gamma, err);
  int j = 0;  // first rejected position, 0 if none
  for (int k = 1; k <= L; ++k) {
    const size_t o = (size_t)b * gamma + (k - 1);
    const float u = u01(draw_block(seed, 0u, (uint32_t)k, (uint32_t)b, 1u).x);
    if (!(u < p_t[o] / q_tok[o])) {
      j = k;
      break;
    }
  }
  const int acc = j ? j - 1 : L;
  for (int i = 0; i <= gamma; ++i)
    out_tokens[(size_t)b * (gamma + 1) + i] = i < acc ? tokens[(size_t)b * gamma + i] : -1;
  accept_len[b] = acc;
  n_out[b] = acc + 1;
  fallback[b] = 0;
  if (j) {
    mode[b] = kModeResidual;
    pos[b] = j;
    prev_tok[b] = (j == 1) ? anchor[b] : tokens[(size_t)b * gamma + (j - 2)];
  } else {
    mode[b] = kModeBonus;
    pos[b] = L + 1;
    prev_tok[b] = -1;
  }
}

// ----------------------------------------------------------------------- final sample
__global__ void __launch_bounds__(kSampleThreads) final_sample_kernel(
    const float* __restrict__ T, const float* __restrict__ U, const float* __restrict__ bias,
    const float* __restrict__ row_max, const float* __restrict__ row_sumexp,
    const float* __restrict__ M_t, const float* __restrict__ lnS_t,
    const int32_t* __restrict__ mode, const int32_t* __restrict__ pos,
    const int32_t* __restrict__ accept_len, int gamma, int V, uint64_t seed, int splits, int seg,
    RowState* __restrict__ partials, uint32_t* __restrict__ counters,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ fallback) {
  __shared__ RowState red[32];
  __shared__ int is_last;
  const int b = blockIdx.y;
  const int md = mode[b], k = pos[b];
  const int v_begin = blockIdx.x * seg, v_end = min(V, v_begin + seg);
  RowState st = row_state_empty();
  if (md == kModeResidual) {
    const size_t o = (size_t)b * gamma + (k - 1);
    const float* Trow = T + ((size_t)b * (gamma + 1) + (k - 1)) * V;
    const float* Urow = U + o * V;
    const float* Brow = bias + (size_t)b * V;
    const float q_off = row_max[o] + logf(row_sumexp[o]);   // log Q = z - q_off
    const float p_off = M_t[o] + lnS_t[o];                   // log P = T - p_off
    for (int v = v_begin + 4 * threadIdx.x; v < v_end; v += 4 * kSampleThreads) {
      const float4 t4 = ld_stream_f4(Trow + v);
      const float4 u4 = ld_stream_f4(Urow + v);
      const float4 b4 = __ldcg(reinterpret_cast<const float4*>(Brow + v));
      const float t[4] = {t4.x, t4.y, t4.z, t4.w};
      const float z[4] = {u4.x + b4.x, u4.y + b4.y, u4.z + b4.z, u4.w + b4.w};
      const uint4 dr = draw_block(seed, (uint32_t)(v >> 2), (uint32_t)k, (uint32_t)b, 2u);
      const uint32_t dw[4] = {dr.x, dr.y, dr.z, dr.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lq = z[i] - q_off;
        const float d = (t[i] - p_off) - lq;     // log(P / Q)
        if (d > 0.f) {
          // log(P - Q) = log Q + log(expm1(log P - log Q)), accurate when P ~ Q; for
          // d > 20 it is log P to within 2e-9
          const float lres = d > 20.f ? lq + d : lq + logf(expm1f(d));
          const float score = lres + gumbel_of(dw[i]);
          if (better(score, v + i, st.score, st.idx)) {
            st.score = score;
            st.idx = v + i;
          }
        }
      }
    }
  } else if (md == kModeBonus) {
    const float* Trow = T + ((size_t)b * (gamma + 1) + (k - 1)) * V;
    for (int v = v_begin + 4 * threadIdx.x; v < v_end; v += 4 * kSampleThreads) {
      const float4 t4 = ld_stream_f4(Trow + v);
      const float t[4] = {t4.x, t4.y, t4.z, t4.w};
      const uint4 dr = draw_block(seed, (uint32_t)(v >> 2), (uint32_t)k, (uint32_t)b, 3u);
      const uint32_t dw[4] = {dr.x, dr.y, dr.z, dr.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float score = t[i] + gumbel_of(dw[i]);
        if (better(score, v + i, st.score, st.idx)) {
          st.score = score;
          st.idx = v + i;
        }
      }
    }
  } else {
    return;
  }
  st = row_state_block_reduce(st, red);
  if (!publish_partial(st, partials + (size_t)b * splits + blockIdx.x, &counters[b], splits,
                       &is_last))
    return;
  if (threadIdx.x < 32) {
    const RowState acc = merge_partials(partials + (size_t)b * splits, splits);
    if (threadIdx.x == 0) {
      if (acc.idx >= 0) {
        out_tokens[(size_t)b * (gamma + 1) + accept_len[b]] = acc.idx;
      } else {
        fallback[b] = 1;
      }
      counters[b] = 0u;
    }
  }
}

// --------------------------------------------------------------------------- fallback
__global__ void __launch_bounds__(kSampleThreads) fallback_kernel(
    const float* __restrict__ T, const int32_t* __restrict__ pos,
    const int32_t* __restrict__ accept_len, const int32_t* __restrict__ fallback, int gamma,
    int V, uint64_t seed, int splits, int seg, RowState* __restrict__ partials,
    uint32_t* __restrict__ counters, int32_t* __restrict__ out_tokens) {
  __shared__ RowState red[32];
  __shared__ int is_last;
  const int b = blockIdx.y;
  if (!fallback[b]) return;
  const int k = pos[b];
  const float* Trow = T + ((size_t)b * (gamma + 1) + (k - 1)) * V;
  const int v_begin = blockIdx.x * seg, v_end = min(V, v_begin + seg);
  RowState st = row_state_empty();
  for (int v = v_begin + 4 * threadIdx.x; v < v_end; v += 4 * kSampleThreads) {
    const float4 t4 = ld_stream_f4(Trow + v);
    const float t[4] = {t4.x, t4.y, t4.z, t4.w};
    const uint4 dr = draw_block(seed, (uint32_t)(v >> 2), (uint32_t)k, (uint32_t)b, 2u);
    const uint32_t dw[4] = {dr.x, dr.y, dr.z, dr.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float score = t[i] + gumbel_of(dw[i]);
      if (better(score, v + i, st.score, st.idx)) {
        st.score = score;
        st.idx = v + i;
      }
    }
  }
  st = row_state_block_reduce(st, red);
  if (!publish_partial(st, partials + (size_t)b * splits + blockIdx.x, &counters[b], splits,
                       &is_last))
    return;
  if (threadIdx.x < 32) {
    const RowState acc = merge_partials(partials + (size_t)b * splits, splits);
    if (threadIdx.x == 0) {
      out_tokens[(size_t)b * (gamma + 1) + accept_len[b]] = acc.idx;
      counters[b] = 0u;
    }
  }
}

}  // namespace

cudaError_t launch_verify(const Plan& p, const float* T, const float* U, const uint16_t* W1,
                          const CUtensorMap* w2_map, const int32_t* anchor,
                          const int32_t* tokens, const float* q_tok, const float* row_max,
                          const float* row_sumexp, const int32_t* ell, uint64_t seed,
                          int32_t* accept_len, int32_t* out_tokens, int32_t* n_out, void* ws,
                          cudaStream_t stream) {
  const int B = p.B, gamma = p.gamma, V = p.V;
  int* err = ws_at<int>(ws, p.off_err);
  float* bias = ws_at<float>(ws, p.off_bias);
  RowState* part = ws_at<RowState>(ws, p.off_part);
  RowState* part_stats = part;
  RowState* part_ver = part + (size_t)B * gamma * p.stats.splits;
  uint32_t* cnt_stats = ws_at<uint32_t>(ws, p.off_cnt);
  uint32_t* cnt_ver = cnt_stats + (size_t)B * gamma;
  uint32_t* cnt_fb = cnt_ver + B;
  float* M_t = ws_at<float>(ws, p.off_M);
  float* lnS_t = ws_at<float>(ws, p.off_lnS);
  float* p_t = ws_at<float>(ws, p.off_p);
  int32_t* mode = ws_at<int32_t>(ws, p.off_mode);
  int32_t* pos = ws_at<int32_t>(ws, p.off_pos);
  int32_t* prev = ws_at<int32_t>(ws, p.off_prev);
  int32_t* fb = ws_at<int32_t>(ws, p.off_fallback);

  cudaError_t e = cudaMemsetAsync(cnt_stats, 0, ((size_t)B * gamma + 2 * (size_t)B) * sizeof(uint32_t),
                                  stream);
  if (e != cudaSuccess) return e;
  target_stats_kernel<<<dim3(p.stats.splits, B * gamma), kSampleThreads, 0, stream>>>(
      T, tokens, ell, gamma, V, p.stats.splits, p.stats.seg, part_stats, cnt_stats, M_t, lnS_t, p_t,
      err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  decide_kernel<<<cdiv(B, 128), 128, 0, stream>>>(anchor, tokens, q_tok, p_t, ell, B, gamma, seed,
                                                  accept_len, out_tokens, n_out, mode, pos, prev,
                                                  fb, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_bias_gemm(w2_map, W1, prev, 1, B, V, p.r, bias, err, stream)) != cudaSuccess)
    return e;
  final_sample_kernel<<<dim3(p.ver.splits, B), kSampleThreads, 0, stream>>>(
      T, U, bias, row_max, row_sumexp, M_t, lnS_t, mode, pos, accept_len, gamma, V, seed,
      p.ver.splits, p.ver.seg, part_ver, cnt_ver, out_tokens, fb);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fallback_kernel<<<dim3(p.ver.splits, B), kSampleThreads, 0, stream>>>(
      T, pos, accept_len, fb, gamma, V, seed, p.ver.splits, p.ver.seg, part_ver, cnt_fb, out_tokens);
  return cudaGetLastError();
}

}  // namespace dspark
