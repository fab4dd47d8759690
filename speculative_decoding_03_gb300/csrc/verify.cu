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
//   target_stats   for every verified row (b, k <= l_b) and segment of it: the max and the
//                  sum of exp of T[b, k] over the segment (a partial, no cross-CTA merge)
//   decide         one warp per request, one lane per position: merges the row partials
//                  into M, log S and p_k(x_k), runs the acceptance tests, finds the first
//                  reject, the accepted prefix, and which row the final token comes from,
//                  and writes the final draw's record (row, mode, log normalisers)
//   bias_gemm      (shared with the draft) W1[x_{j-1}] W2 for the rows with a reject at j
//   final_sample   Gumbel-max over log(P_j - Q_j) on {P_j > Q_j} (residual), or over
//                  T[b, l+1] (bonus): one partial (best score, index) per segment
//   finalize       one CTA per request merges the partials and writes the token; only
//                  for a row whose residual support came out empty in fp32 it draws the
//                  fallback: Gumbel-max over T[b, j] with the residual's random stream
//
// Greedy drafts (billytse.dev section 11) propose the point mass at x_k: q_k(x_k) = 1, so
// the test is u < p_k(x_k), and the residual max(0, P_j - Q_j) is P_j without x_j.  Then
// no bias is needed (no bias_gemm launch) and final_sample runs the bonus race over T[b, j]
// with the residual's stream and x_j excluded.
#include "internal.h"

namespace dspark {
namespace {

enum : int { kModeNone = 0, kModeResidual = 1, kModeBonus = 2, kModePointResidual = 3 };

// What the final draw of request b needs besides the rows it reads, written by the
// decision kernel: the mode, the position k of the row drawn from (T[b, k - 1]), the
// excluded token (greedy drafts' point residual, else -1), the residual's compact bias
// slot, and its log normalisers (log P = T - off_a, log Q = z - off_b).  32 bytes, so the
// final-sample kernel fetches it with two independent 16-byte loads.
struct __align__(16) ItemRec {
  int md, k, excl, slot;
  float off_a, off_b, pad0, pad1;
};

__device__ __forceinline__ int clamp_ell(const int32_t* ell, int b, int gamma, int* err) {
  int L = ell[b];
  if (L < 0 || L > gamma) {
    set_device_error(err, DSPARK_ERR_DEVICE_CHECK);
    L = L < 0 ? 0 : gamma;
  }
  return L;
}

// mbarrier and 1-D bulk copy (global -> shared, completing on an mbarrier)
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init_cta(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init_cta() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_cta() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx_cta(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// bounded wait (about 2 s of SM cycles); false on timeout
__device__ __forceinline__ bool mbar_wait_cta(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(10000000u)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > 4000000000ll) return false;
  }
}

// 1/x on the special-function unit (PTX rcp.approx.ftz.f32, relative error below 2^-22)
__device__ __forceinline__ float rcp_approx_ftz(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Gumbel value of the 32-bit draw x: g = -log(-log1p(-w)), w = 1 - U01(x).
__device__ __forceinline__ float gumbel_of(uint32_t x) {
  return -logf(exp1_from_w(one_minus_u01(x)));
}

// ---------------------------------------------------------------------- target stats
// Grid (splits, B * gamma) with blockIdx.y = (k - 1) * B + b: rows ordered by position,
// so the CTAs of verified rows (k <= l_b) come first and the rest exit at once.  Every
// thread issues all kStatsVec of its 128-bit loads before using any of them; the CTA
// reduces only (max, sum of exp) and publishes them as a partial.
__device__ __forceinline__ void max_sum_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  s = s * ex2_approx((m - mn) * kLog2e) + s2 * ex2_approx((m2 - mn) * kLog2e);
  m = mn;
}

__global__ void __launch_bounds__(kSampleThreads) target_stats_kernel(
    const float* __restrict__ T, const int32_t* __restrict__ ell, int B, int gamma, int V,
    int splits, float2* __restrict__ partials, int* __restrict__ n_res) {
  __shared__ float red_m[kSampleThreads / 32], red_s[kSampleThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  // the decision kernel that follows counts the residual rows from zero
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *n_res = 0;
  // rows (k, b) in position order; the grid's y extent is capped at 65535, so a CTA takes
  // every gridDim.y-th row
  for (int y = blockIdx.y; y < B * gamma; y += gridDim.y) {
    const int k = y / B + 1, b = y - (k - 1) * B;
    if (k > clamp_ell(ell, b, gamma, nullptr)) continue;
    const int row = b * gamma + (k - 1);
    const float* Trow = T + ((size_t)b * (gamma + 1) + (k - 1)) * V;
    const int v0 = blockIdx.x * kStatsSeg + 4 * threadIdx.x;
    float4 t[kStatsVec];
#pragma unroll
    for (int j = 0; j < kStatsVec; ++j) {
      const int v = v0 + j * 4 * kSampleThreads;
      t[j] = v < V ? ld_stream_f4(Trow + v) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kStatsVec; ++j) m = fmaxf(m, fmaxf(fmaxf(t[j].x, t[j].y), fmaxf(t[j].z, t[j].w)));
    float s = 0.f;
    if (m != -INFINITY) {
      const float mL = m * kLog2e;
#pragma unroll
      for (int j = 0; j < kStatsVec; ++j)
        s += ex2_approx(fmaf(t[j].x, kLog2e, -mL)) + ex2_approx(fmaf(t[j].y, kLog2e, -mL)) +
             ex2_approx(fmaf(t[j].z, kLog2e, -mL)) + ex2_approx(fmaf(t[j].w, kLog2e, -mL));
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
      max_sum_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    if (lane == 0) { red_m[warp] = m; red_s[warp] = s; }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kSampleThreads / 32; ++w) max_sum_merge(m, s, red_m[w], red_s[w]);
      partials[(size_t)row * splits + blockIdx.x] = make_float2(m, s);
    }
    __syncthreads();   // red_m / red_s are rewritten by the next row
  }
}

// ----------------------------------------------------------------------------- decide
// One warp per request; lane k - 1 owns position k.  Verified lanes merge their row's
// target partials (M, S), compute p_k(x_k) and test u_k < p_k(x_k) / q_k(x_k); a ballot
// gives the first reject.  q_tok == null: greedy drafts, q_k(x_k) = 1.  rnn_rows: the
// residual's bias rows are the RNN head's output rows instead of W1 rows.
__global__ void __launch_bounds__(128) decide_kernel(
    const float* __restrict__ T, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, const float* __restrict__ q_tok,
    const float2* __restrict__ stats, int splits, const int32_t* __restrict__ ell, int B,
    int gamma, int V, uint64_t seed, int32_t* __restrict__ accept_len,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ n_out, int32_t* __restrict__ mode,
    int32_t* __restrict__ pos,
    int32_t* __restrict__ res_prev, int32_t* __restrict__ slot_of, int* __restrict__ n_res,
    int32_t* __restrict__ fallback, int* err, int rnn_rows, const float* __restrict__ row_max,
    const float* __restrict__ row_sumexp, ItemRec* __restrict__ rec) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  const int L = clamp_ell(ell, b, gamma, lane == 0 ? err : nullptr);
  const int k = lane + 1;
  bool reject = false;
  float m_own = 0.f, lns_own = 0.f;      // this lane's row: M and log S
  if (k <= L) {
    const int row = b * gamma + (k - 1);
    // the token, its target logit and the row partials are independent loads: issue them
    // together (partials in batches of 16), then merge
    const int x = tokens[(size_t)b * gamma + (k - 1)];
    const bool x_ok = x >= 0 && x < V;
    const float tx = x_ok ? __ldg(T + ((size_t)b * (gamma + 1) + (k - 1)) * V + x) : 0.f;
    float m = -INFINITY, s = 0.f;
    for (int i0 = 0; i0 < splits; i0 += 16) {
      float2 q[16];
#pragma unroll
      for (int u = 0; u < 16; ++u)
        q[u] = i0 + u < splits ? __ldcg(stats + (size_t)row * splits + i0 + u)
                               : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int u = 0; u < 16; ++u) max_sum_merge(m, s, q[u].x, q[u].y);
    }
    float p = 0.f;
    if (x_ok) {
      p = expf(tx - m) / s;
    } else {
      set_device_error(err, DSPARK_ERR_DEVICE_CHECK);
    }
    m_own = m;
    lns_own = logf(s);
    const float u = u01(draw_block(seed, 0u, (uint32_t)k, (uint32_t)b, 1u).x);
    reject = q_tok ? !(u < p / q_tok[row]) : !(u < p);
  }
  const unsigned rej = __ballot_sync(0xffffffffu, reject);
  const int j = rej ? __ffs(rej) : 0;    // first rejected position, 0 if none
  const int acc = j ? j - 1 : L;
  // the rejected row's target normalisers, from the lane that owns it
  const float m_j = __shfl_sync(0xffffffffu, m_own, j ? j - 1 : 0);
  const float lns_j = __shfl_sync(0xffffffffu, lns_own, j ? j - 1 : 0);
  for (int i = lane; i <= gamma; i += 32)
    out_tokens[(size_t)b * (gamma + 1) + i] = i < acc ? tokens[(size_t)b * gamma + i] : -1;
  if (lane == 0) {
    accept_len[b] = acc;
    n_out[b] = acc + 1;
    fallback[b] = 0;
    ItemRec r;
    r.excl = -1;
    r.slot = 0;
    r.off_a = r.off_b = r.pad0 = r.pad1 = 0.f;
    if (j && !q_tok) {
      mode[b] = kModePointResidual;
      pos[b] = j;
      slot_of[b] = -1;
      r.md = kModePointResidual;
      r.k = j;
      r.excl = tokens[(size_t)b * gamma + (j - 1)];
    } else if (j) {
      mode[b] = kModeResidual;
      pos[b] = j;
      // a slot of the compact residual rows, and the bias operand of the rejected row: the
      // Markov head's predecessor token, or the RNN head's output row (b, j) of the draft
      const int slot = atomicAdd(n_res, 1);
      slot_of[b] = slot;
      res_prev[slot] = rnn_rows ? b * gamma + (j - 1)
                                : ((j == 1) ? anchor[b] : tokens[(size_t)b * gamma + (j - 2)]);
      const size_t o = (size_t)b * gamma + (j - 1);
      r.md = kModeResidual;
      r.k = j;
      r.slot = slot;
      r.off_a = m_j + lns_j;                          // log P = T - off_a
      r.off_b = row_max[o] + logf(row_sumexp[o]);     // log Q = z - off_b
    } else {
      mode[b] = kModeBonus;
      pos[b] = L + 1;
      slot_of[b] = -1;
      r.md = kModeBonus;
      r.k = L + 1;
    }
    rec[b] = r;
  }
}

// ----------------------------------------------------------------------- final sample
// Gumbel-max in exponential-race form with a conservative two-phase filter.  Residual:
// score_v = log(P_v - Q_v) - log E_v with E_v = -log1p(-w_v), and w <= E <= w / (1 - w),
// so with r_v = P_v - Q_v
//     r_v (1 - w_v) / w_v  <=  exp(score_v)  <=  r_v / w_v.
// Phase 1 computes both bounds for every logit of the CTA's segment (two exp2 per logit,
// no logarithms) and the CTA-wide best lower bound L; phase 2 scores exactly, with the same
// fp32 formulas as an unfiltered scan, only the logits whose upper bound reaches L (a few
// per CTA).  Bounds and L carry a 2^-12 relative slack, far above the fp32 errors of
// either side, so the argmax is that of the unfiltered scan.  The bonus row (all drafts
// accepted) is the same race over exp(T_v - m), m the CTA's largest logit.
constexpr float kRaceSlack = 0x1.0p-12f;

__device__ __forceinline__ float block_max_f(float x, float* red) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  x = red[0];
#pragma unroll
  for (int w = 1; w < kSampleThreads / 32; ++w) x = fmaxf(x, red[w]);
  __syncthreads();
  return x;
}

// A logit of a segment that the exponential race keeps (its upper bound reaches the
// segment's best lower bound): index, target logit, draft logit z (residual rows) and the
// draw's w = 1 - u.  A segment hands up to kCandMax of them to the finalize kernel, which
// scores them exactly; a segment with more scores them itself.
struct __align__(16) Cand {
  int idx;
  float t, z, w;
};
constexpr int kCandMax = 64;

// The exact race score of one logit, the unfiltered scan's fp32 formula: residual rows
// log(P - Q) - log E = log Q + log(expm1(log P - log Q)) - log E (for log P - log Q > 20 it
// is log P to within 2e-9), else T - log E; E = -log1p(-w) from the draw's w.
__device__ __forceinline__ float exact_score(bool residual, float t, float z, float w, float off_a,
                                             float off_b) {
  if (residual) {
    const float lq = z - off_b;
    const float d = (t - off_a) - lq;          // log(P / Q) > 0
    const float lres = d > 20.f ? lq + d : lq + logf(expm1f(d));
    return lres - logf(exp1_from_w(w));
  }
  return t - logf(exp1_from_w(w));
}

// One CTA scores one segment of kVerSeg logits of one row: t / zz hold this thread's
// kVerVec float4 of T and of z = U + bias (residual rows only), v0 the first vocabulary
// index of the thread's first float4.  Not residual: the race over T alone with random
// stream `stream`, skipping index `excl` (-1: none).  Every thread of the CTA calls it.
// The segment's candidates go to cand_s (their count to *cnt_s, zero on entry); returns
// their count, or, when they do not fit, -1 with the CTA's best (score, index), which the
// CTA then scored itself, in `best` (every thread).
__device__ __forceinline__ int race_segment(const float4 (&t)[kVerVec],
                                            const float4 (&zz)[kVerVec], int v0, int V,
                                            bool residual, float off_a, float off_b,
                                            uint32_t stream, int excl, const PhiloxKeys& keys, int k,
                                            int b, RowState* red, float* redf, Cand* cand_s,
                                            int* cnt_s, RowState& best) {
  if (!residual) {
    // bonus: reference = the CTA's largest logit (exp(T - m) <= 1)
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kVerVec; ++j) m = fmaxf(m, fmaxf(fmaxf(t[j].x, t[j].y), fmaxf(t[j].z, t[j].w)));
    off_a = block_max_f(m, redf);
  }
  // phase 1: per logit the upper bound numerator r_hi (compared against L w) and the
  // thread's best lower bound
  float r_hi[kVerVec][4], w[kVerVec][4];
  float Lt = 0.f;
#pragma unroll
  for (int j = 0; j < kVerVec; ++j) {
    const int v = v0 + j * 4 * kSampleThreads;
    const uint4 dr = draw_block(keys, (uint32_t)(v >> 2), (uint32_t)k, (uint32_t)b, stream);
    const uint32_t dw[4] = {dr.x, dr.y, dr.z, dr.w};
    const float tv[4] = {t[j].x, t[j].y, t[j].z, t[j].w};
    const float zv[4] = {zz[j].x, zz[j].y, zz[j].z, zz[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[j][i] = one_minus_u01(dw[i]);
      float r, e;
      bool in = v < V;
      if (residual) {
        const float lp = tv[i] - off_a, lq = zv[i] - off_b;
        in = in && (lp - lq > 0.f);                    // the residual's support
        const float P = ex2_approx(lp * kLog2e), Q = ex2_approx(lq * kLog2e);
        r = P - Q;
        e = (P + Q) * kRaceSlack;
        // both flushed to zero: the bounds say nothing, keep it for exact scoring
        if (in && P + Q == 0.f) { r = INFINITY; e = 0.f; }
      } else {
        in = in && v + i != excl;
        r = ex2_approx(fmaf(tv[i], kLog2e, -off_a * kLog2e));
        e = r * kRaceSlack;
      }
      r_hi[j][i] = in ? r + e : -1.f;
      if (in && r - e > 0.f && r != INFINITY)
        Lt = fmaxf(Lt, (r - e) * (1.f - w[j][i]) * rcp_approx_ftz(w[j][i]) * (1.f - kRaceSlack));
    }
  }
  const float L = block_max_f(Lt, redf);
  // phase 2: the logits whose upper bound reaches L into the shared candidate list
  unsigned cms[kVerVec];
#pragma unroll
  for (int j = 0; j < kVerVec; ++j) {
    unsigned cm = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) cm |= (r_hi[j][i] >= 0.f && r_hi[j][i] >= L * w[j][i] ? 1u : 0u) << i;
    cms[j] = cm;
    if (cm == 0u) continue;
    const int v = v0 + j * 4 * kSampleThreads;
    const float tv[4] = {t[j].x, t[j].y, t[j].z, t[j].w};
    const float zv[4] = {zz[j].x, zz[j].y, zz[j].z, zz[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (!((cm >> i) & 1u)) continue;
      const int slot = atomicAdd(cnt_s, 1);
      if (slot < kCandMax) {
        Cand c;
        c.idx = v + i;
        c.t = tv[i];
        c.z = zv[i];
        c.w = w[j][i];
        cand_s[slot] = c;
      }
    }
  }
  __syncthreads();
  const int n = *(volatile int*)cnt_s;
  if (n <= kCandMax) return n;
  // more candidates than the list holds (rare): score them here
  RowState st = row_state_empty();
#pragma unroll
  for (int j = 0; j < kVerVec; ++j) {
    const unsigned cm = cms[j];
    if (cm == 0u) continue;
    const int v = v0 + j * 4 * kSampleThreads;
    const float tv[4] = {t[j].x, t[j].y, t[j].z, t[j].w};
    const float zv[4] = {zz[j].x, zz[j].y, zz[j].z, zz[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (!((cm >> i) & 1u)) continue;
      const float score = exact_score(residual, tv[i], zv[i], w[j][i], off_a, off_b);
      if (better(score, v + i, st.score, st.idx)) {
        st.score = score;
        st.idx = v + i;
      }
    }
  }
  // the CTA's best (score, index): two shuffles per level, one word pair per warp
  float sc = st.score;
  int ix = st.idx;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float osc = __shfl_xor_sync(0xffffffffu, sc, o);
    const int oix = __shfl_xor_sync(0xffffffffu, ix, o);
    if (better(osc, oix, sc, ix)) { sc = osc; ix = oix; }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { red[warp].score = sc; red[warp].idx = ix; }
  __syncthreads();
  sc = red[0].score;
  ix = red[0].idx;
#pragma unroll
  for (int wi = 1; wi < kSampleThreads / 32; ++wi)
    if (better(red[wi].score, red[wi].idx, sc, ix)) { sc = red[wi].score; ix = red[wi].idx; }
  __syncthreads();
  best = row_state_empty();
  best.score = sc;
  best.idx = ix;
  return -1;
}

// Persistent: CTA g scores the segments (b, seg) = items g, g + G, ... (item = b * splits +
// seg).  Thread 0 brings the next item's rows into the other half of a double buffer with
// 1-D bulk copies (T, and U and bias for residual rows) while the CTA scores the current
// one, so HBM latency overlaps the scoring.  An item's output is its candidates
// (cand[item * kCandMax ..], count in cand_n[item]), or, count -1, the (index, score) of
// its best in cand[item * kCandMax] when it scored them itself.
__global__ void __launch_bounds__(kSampleThreads) final_sample_kernel(
    const float* __restrict__ T, const float* __restrict__ U, const float* __restrict__ bias,
    const ItemRec* __restrict__ rec, int B, int gamma, int V, const PhiloxKeys keys, int splits,
    int* __restrict__ cand_n, Cand* __restrict__ cand, int* err) {
  extern __shared__ float4 fs_buf[];            // [2][3][kVerSeg / 4]
  __shared__ uint64_t full[2];
  __shared__ Cand cand_s[kCandMax];
  __shared__ int cnt_s;
  __shared__ RowState red[32];
  __shared__ float redf[kSampleThreads / 32];
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init_cta(&full[0], 1);
    mbar_init_cta(&full[1], 1);
    fence_mbar_init_cta();
  }
  __syncthreads();
  pdl_wait();                   // the records come from the decision kernel
  pdl_launch_dependents();
  const int n_items = B * splits, G = gridDim.x;
  constexpr int kSlot = kVerSeg / 4;            // float4 per array slot
  // An item's record (its request's, from the decision kernel) is loaded by thread 0 one
  // item ahead of its copies, two independent loads used only at the next item, and
  // published with the copies (the expect-tx arrival releases it).
  struct ItemMeta {
    int md, k, excl, slot;
    float off_a, off_b;
  };
  __shared__ ItemMeta meta_s[2];
  auto load_meta = [&](int item) -> ItemMeta {  // thread 0
    const int4* src = reinterpret_cast<const int4*>(rec + item / splits);
    const int4 a = __ldcg(src), c = __ldcg(src + 1);
    ItemMeta m;
    m.md = a.x;
    m.k = a.y;
    m.excl = a.z;
    m.slot = a.w;
    m.off_a = __int_as_float(c.x);
    m.off_b = __int_as_float(c.y);
    return m;
  };
  auto issue = [&](int item, int buf, const ItemMeta& m) {   // thread 0
    const int b = item / splits, seg = item - b * splits;
    const int md = m.md, k = m.k;
    const int v0 = seg * kVerSeg;
    const uint32_t bytes = (uint32_t)(min(kVerSeg, V - v0)) * 4u;
    float4* dst = fs_buf + (size_t)buf * 3 * kSlot;
    meta_s[buf] = m;
    fence_proxy_async_cta();    // the buffer's previous generic reads come first
    if (md == kModeResidual) {
      const size_t o = (size_t)b * gamma + (k - 1);
      mbar_expect_tx_cta(&full[buf], 3u * bytes);
      bulk_g2s(dst, T + ((size_t)b * (gamma + 1) + (k - 1)) * V + v0, bytes, &full[buf]);
      bulk_g2s(dst + kSlot, U + o * V + v0, bytes, &full[buf]);
      bulk_g2s(dst + 2 * kSlot, bias + (size_t)m.slot * V + v0, bytes, &full[buf]);
    } else if (md == kModeBonus || md == kModePointResidual) {
      mbar_expect_tx_cta(&full[buf], bytes);
      bulk_g2s(dst, T + ((size_t)b * (gamma + 1) + (k - 1)) * V + v0, bytes, &full[buf]);
    } else {
      mbar_arrive_cta(&full[buf]);
    }
  };
  ItemMeta next;                                // thread 0: the record of item + G
  if (tid == 0 && blockIdx.x < n_items) {
    issue(blockIdx.x, 0, load_meta(blockIdx.x));
    if (blockIdx.x + G < n_items) next = load_meta(blockIdx.x + G);
  }
  int it = 0;
  for (int item = blockIdx.x; item < n_items; item += G, ++it) {
    const int buf = it & 1;
    if (tid == 0 && item + G < n_items) {
      issue(item + G, buf ^ 1, next);
      if (item + 2 * G < n_items) next = load_meta(item + 2 * G);
    }
    const bool ok = mbar_wait_cta(&full[buf], (uint32_t)(it >> 1) & 1u);
    if (!ok && tid == 0) set_device_error(err, DSPARK_ERR_TIMEOUT);
    const int b = item / splits, seg = item - b * splits;
    const ItemMeta m = meta_s[buf];
    const int md = m.md, k = m.k;
    const bool residual = md == kModeResidual;
    if (tid == 0) cnt_s = 0;                    // (ordered by the barrier below)
    if (md != kModeNone && !__syncthreads_and(ok)) {
      if (tid == 0) cand_n[item] = 0;
    } else if (md != kModeNone) {
      const int v0 = seg * kVerSeg + 4 * tid;
      const int n4 = (min(kVerSeg, V - seg * kVerSeg) + 3) / 4;
      const float4* src = fs_buf + (size_t)buf * 3 * kSlot;
      float4 t[kVerVec], zz[kVerVec];
#pragma unroll
      for (int j = 0; j < kVerVec; ++j) {
        const int q = tid + j * kSampleThreads;
        t[j] = q < n4 ? src[q] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        zz[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (residual && q < n4) {
          const float4 u4 = src[kSlot + q], b4 = src[2 * kSlot + q];
          zz[j] = make_float4(u4.x + b4.x, u4.y + b4.y, u4.z + b4.z, u4.w + b4.w);
        }
      }
      const float off_a = m.off_a, off_b = m.off_b;   // residual: log P = T - off_a, log Q = z - off_b
      const uint32_t stream = md == kModeBonus ? 3u : 2u;
      const int excl = m.excl;
      RowState best;
      const int n = race_segment(t, zz, v0, V, residual, off_a, off_b, stream, excl, keys, k, b,
                                 red, redf, cand_s, &cnt_s, best);
      Cand* dst = cand + (size_t)item * kCandMax;
      if (n >= 0) {
        if (tid < n) dst[tid] = cand_s[tid];
        if (tid == 0) cand_n[item] = n;
      } else if (tid == 0) {
        Cand c;
        c.idx = best.idx;
        c.t = best.score;
        c.z = c.w = 0.f;
        dst[0] = c;
        cand_n[item] = -1;
      }
    }
    __syncthreads();            // every thread is done with this buffer before it is refilled
  }
}

// One CTA per request: thread t scores the candidates of segments t, t + 256, .. exactly
// and the block's best (score, index) is the token.  If the residual's
// support came out empty in fp32 (no segment has a candidate), the whole CTA draws the
// fallback instead: Gumbel-max over T[b, j] with the residual's random stream (a path the
// acceptance rule practically never takes, so it is not split further).
__global__ void __launch_bounds__(kSampleThreads) finalize_kernel(
    const float* __restrict__ T, const ItemRec* __restrict__ rec, const int* __restrict__ cand_n,
    const Cand* __restrict__ cand, int splits, int gamma, int V, const PhiloxKeys keys,
    const int32_t* __restrict__ mode, const int32_t* __restrict__ pos,
    const int32_t* __restrict__ accept_len, int32_t* __restrict__ out_tokens,
    int32_t* __restrict__ fallback) {
  __shared__ RowState red[32];
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int md = mode[b];
  if (md == kModeNone) return;
  const bool residual = md == kModeResidual;
  const float off_a = __ldcg(&rec[b].off_a), off_b = __ldcg(&rec[b].off_b);
  // thread t takes segments t, t + 256, ..: every segment's few candidates in one round
  RowState acc = row_state_empty();
  for (int seg = threadIdx.x; seg < splits; seg += kSampleThreads) {
    const size_t item = (size_t)b * splits + seg;
    const int n = __ldcg(cand_n + item);
    const Cand* src = cand + item * kCandMax;
    if (n < 0) {
      const Cand c = src[0];
      if (better(c.t, c.idx, acc.score, acc.idx)) { acc.score = c.t; acc.idx = c.idx; }
      continue;
    }
    for (int i = 0; i < (n < kCandMax ? n : kCandMax); ++i) {
      const Cand c = src[i];
      const float score = exact_score(residual, c.t, c.z, c.w, off_a, off_b);
      if (better(score, c.idx, acc.score, acc.idx)) { acc.score = score; acc.idx = c.idx; }
    }
  }
  acc = row_state_block_reduce(acc, red);
  if (acc.idx >= 0) {
    if (threadIdx.x == 0) out_tokens[(size_t)b * (gamma + 1) + accept_len[b]] = acc.idx;
    return;
  }
  // fallback
  const int k = pos[b];
  const float* Trow = T + ((size_t)b * (gamma + 1) + (k - 1)) * V;
  RowState st = row_state_empty();
  for (int v = 4 * threadIdx.x; v < V; v += 4 * kSampleThreads) {
    const float4 t4 = ld_stream_f4(Trow + v);
    const float t[4] = {t4.x, t4.y, t4.z, t4.w};
    const uint4 dr = draw_block(keys, (uint32_t)(v >> 2), (uint32_t)k, (uint32_t)b, 2u);
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
  if (threadIdx.x == 0) {
    fallback[b] = 1;
    out_tokens[(size_t)b * (gamma + 1) + accept_len[b]] = st.idx;
  }
}

}  // namespace

namespace {
constexpr size_t kFinalSmem = 2 * 3 * kVerSeg * sizeof(float);
int final_sample_grid(int n_items) {
  static std::atomic<int> cache[kMaxCachedDevices];
  int g = per_device_grid(cache, [] {
    int per = 0;
    if (cudaFuncSetAttribute(final_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kFinalSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, final_sample_kernel, kSampleThreads,
                                                      kFinalSmem) != cudaSuccess ||
        per < 1)
      return -1;
    return per;
  });
  if (g < 1) g = 1;
  return g < n_items ? g : n_items;
}
}  // namespace

cudaError_t launch_verify(const Plan& p, const float* T, const float* U, const uint16_t* W1,
                          const uint16_t* W2, const uint16_t* W2p, const float* E_all,
                          const int32_t* anchor,
                          const int32_t* tokens, const float* q_tok, const float* row_max,
                          const float* row_sumexp, const int32_t* ell, uint64_t seed,
                          int32_t* accept_len, int32_t* out_tokens, int32_t* n_out, void* ws,
                          cudaStream_t stream) {
  // q_tok == null: greedy drafts (point-mass proposals; U, W1, W2 and the row statistics
  // are not read)
  const bool point_mass = q_tok == nullptr;
  const int B = p.B, gamma = p.gamma, V = p.V;
  int* err = ws_at<int>(ws, p.off_err);
  float* bias = ws_at<float>(ws, p.off_bias);
  RowState* part = ws_at<RowState>(ws, p.off_part);
  float2* part_stats = reinterpret_cast<float2*>(part);
  int* cand_n = ws_at<int>(ws, p.off_cand_n);
  Cand* cand = ws_at<Cand>(ws, p.off_cand);
  int32_t* mode = ws_at<int32_t>(ws, p.off_mode);
  int32_t* pos = ws_at<int32_t>(ws, p.off_pos);
  int32_t* res_prev = ws_at<int32_t>(ws, p.off_prev);
  int32_t* slot_of = ws_at<int32_t>(ws, p.off_slot);
  int* n_res = ws_at<int>(ws, p.off_nres);
  int32_t* fb = ws_at<int32_t>(ws, p.off_fallback);
  const PhiloxKeys keys = philox_keys(seed);
  ItemRec* rec = ws_at<ItemRec>(ws, p.off_rec);

  cudaError_t e = launch_pdl(target_stats_kernel, dim3(p.stats.splits, B * gamma < 65535 ? B * gamma : 65535),
                             dim3(kSampleThreads), 0, stream, T, ell, B, gamma, V,
                             p.stats.splits, part_stats, n_res);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decide_kernel, dim3(cdiv(B, 4)), dim3(128), 0, stream, T, anchor, tokens, q_tok,
                 (const float2*)part_stats, p.stats.splits, ell, B, gamma, V, seed, accept_len,
                 out_tokens, n_out, mode, pos, res_prev, slot_of, n_res, fb,
                 err, E_all ? 1 : 0, row_max, row_sumexp, rec);
  if (e != cudaSuccess) return e;
  if (!point_mass) {
    // only the rejected requests' rows, in the slots the decision kernel gave them
    e = E_all ? launch_bias_gemm_rows(W2, W2p, E_all, B * gamma, res_prev, B, n_res, V, p.r, bias,
                                      err, stream)
              : launch_bias_gemm(W2, W2p, W1, res_prev, 1, B, n_res, V, p.r, bias, err, stream);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(final_sample_kernel, dim3(final_sample_grid(B * p.ver.splits)),
                 dim3(kSampleThreads), kFinalSmem, stream, T, U, (const float*)bias,
                 (const ItemRec*)rec, B, gamma, V, keys, p.ver.splits, cand_n, cand, err);
  if (e != cudaSuccess) return e;
  e = launch_pdl(finalize_kernel, dim3(B), dim3(kSampleThreads), 0, stream, T,
                 (const ItemRec*)rec, (const int*)cand_n, (const Cand*)cand, p.ver.splits, gamma,
                 V, keys, (const int32_t*)mode, (const int32_t*)pos, (const int32_t*)accept_len,
                 out_tokens, fb);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dspark
