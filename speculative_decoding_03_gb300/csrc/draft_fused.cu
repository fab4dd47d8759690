// The whole draft of one step in one persistent, warp-specialised kernel.
//
// billytse.dev DSpark page, sections 3.2 and 3.3: for k = 1..gamma, in order,
//   bias = W1[x_{k-1}] W2;  z = U_k + bias;  x_k ~ softmax(z)   (x_0 = the anchor)
// for every request at once.  x_k is drawn by Gumbel-max: argmax_v z_v - log E_v with
// E_v = -log u_v, i.e. argmax_v exp(z_v - M) / E_v for any reference M.
//
// The greedy variant (billytse.dev section 11: the serving example drafts greedily) is the
// same kernel with x_k = argmax_v z_v (ties to the smallest v): the samplers keep the
// softmax sums and the warp's first largest logit instead of the race, and q_k(x_k) = 1
// because the proposal is the point mass at x_k.
//
// Layout of the work: the vocabulary is cut into 128-row tiles; each CTA (one per SM,
// cooperative launch) owns a contiguous run of tiles for the whole call.  For every
// position k and every chunk of NB requests ("job") the CTA:
//   producer warps  one streams the W2^T tiles (K-chunks of up to 64 rank rows, MN-major,
//                   128-byte swizzle), another the U tiles [NB requests x 128 v], into
//                   shared-memory rings with TMA; neither depends on the drafted tokens,
//                   so the rings run ahead across positions while the CTA waits for x_k;
//   MMA warp        issues tcgen05.mma (M = 128 vocabulary rows, N = NB requests, K = r)
//                   into one of four tensor-memory accumulators;
//   4 transposers   read the accumulator (lane = vocabulary row) and add it to the U
//                   tile in place, so the U stage holds the z rows [b][v] (four
//                   accumulators and four U / z tiles in flight, so the MMA, transposer
//                   and sampler stages overlap; without a separate z ring the W2 ring
//                   gets the shared memory for eight stages);
//   16 samplers     read the z rows (row-contiguous, 128-bit shared loads); each warp owns
//                   NB/16
//                   requests and keeps, per request, a lazy softmax reference M, per-lane
//                   sums of exp(z - M) and maxima, and the best exact Gumbel score
//                   z* - log E*.  Since w <= E = -log(1 - w) <= w / (1 - w) (w = 1 - u),
//                   exp(z - M) / w bounds an element's ratio exp(z - M) / E from above and
//                   exp(z - M)(1 - w) / w from below: an element is a candidate only if
//                   its upper bound beats exp(best - M) and the best lower bound of the
//                   warp's candidates; only the survivors (about one per warp) evaluate
//                   the exact score with log1p and log, like the oracle.
// After its last tile of position k a CTA publishes per-request partials (M, sum, best
// score, index, logit) and folds its best (score, index) into a 64-bit atomicMax key;
// one grid barrier per position (bounded spin) makes every x_k known to every CTA, which
// then gathers W1[x_k] for the next position.  The CTA with index b mod G merges the
// partials of request b into x_k, q_k(x_k), max and sum, while it waits at the next
// barrier.
//
// Failure handling: every wait is bounded (2 s).  A wait that runs out records
// DSPARK_ERR_TIMEOUT and sets a CTA-wide abort flag; from then on the sampler threads
// run their fixed loop counts without waiting or working (so their named barriers and
// the grid barrier still line up), the other roles stop, and the producer and the MMA
// issuer drain their in-flight copies and MMAs before the CTA releases tensor memory.
#include <string.h>

#include <type_traits>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace dspark {
namespace {

using namespace sm100;

constexpr int kWarps = 23;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerWarp = 0;      // W2 stages
constexpr int kMmaWarp = 1;
constexpr int kFirstSampler = 6;      // warps 2..5 transpose, 6..21 sample
constexpr int kUProducerWarp = 22;    // U tiles
constexpr int kSamplers = 16;
constexpr int kSamplerThreads = kSamplers * 32;
constexpr int kWStagesMarkov = 8;     // W2 K-chunk ring (16 KB each at K-chunk 64)
constexpr int kRnnRecBytes = 16384;   // shared memory for a recurrence CTA's rows of Wrec
// The state and the E rows are read by every CTA right after the recurrence CTAs write
// them: 152 CTAs reading the same lines at once queue on the few L2 slices that hold them
// (measured: 4.2 us for a 32 KB gather against 2.2 us when each CTA reads other lines), so
// the writers keep kRnnCopies copies and CTA c reads copy c % kRnnCopies.  Every copy
// costs the writers stores before their release; two copies measured best (RNN draft
// 209.7 / 203.3 / 204.6 / 208.5 us with 1 / 2 / 4 / 8 copies).
constexpr int kRnnCopies = kRnnStateCopies;
static_assert(kRnnCopies <= 16, "one copy per lane of a half-warp");
constexpr int kDepthMarkov = 4;       // accumulators in TMEM, z tiles and U tiles in flight
constexpr int kKChunkMax = 64;
constexpr int kNamedBarSamplers = 1;
constexpr int kGatherWarps = 4;       // sampler warps 0..3 also gather E
constexpr int kNamedBarGather = 2;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLazy = 32.f;             // reference raise margin (exp(32) fits fp32 sums)
constexpr float kShrink = 1.f - 0x1.0p-16f;  // filter slack, well above fp32 rounding

// 1 - U01(x) = ((~x >> 9) + 1/2) 2^-23 built exactly: the float with bits
// 0x4B000000 | n is 2^23 + n, and one fused multiply-add removes 2^23 - 1/2.
__device__ __forceinline__ float w_of_draw(uint32_t x) {
  const float f = __uint_as_float(0x4B000000u | ((~x) >> 9));
  return fmaf(f, 0x1.0p-23f, -(1.f - 0x1.0p-24f));
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct DraftParams {
  const uint16_t* W1;
  const uint16_t* W2p;             // packed W2 tile images (null: tiles come by TMA from W2)
  const int32_t* anchor;
  int B, gamma, V, r;
  int n_tiles, n_chunks, kc;       // kc = K rows per W2 stage (<= 64)
  uint64_t seed;
  PhiloxKeys philox;               // the generator's round keys for this seed
  RowState* partials;              // [3][B][G], position k in slot k % 3
  unsigned long long* keys;        // [gamma][B], zeroed before launch
  unsigned int* grid_count;        // zeroed before launch
  int32_t* tokens;
  float* q_tok;
  float* row_max;
  float* row_sumexp;
  int* err;
  long long wait_cycles;           // bound of every wait
  unsigned int grid_extra;         // added to every barrier target (0; tests: unreachable)
  // RNN head (unused by the Markov head)
  const uint16_t* Wrec;            // [3r][2r] the recurrent rows of W_rnn, transposed
  const float* hp;                 // [B][gamma][3r] hidden-state block of the layer, with bias
  float* E_all;                    // [B][gamma][r] tanh(output) of every position (written)
  uint16_t* E_hl;                  // [kRnnCopies][B][2][r] the current position's rows as bf16 hi, lo
  float* state;                    // [kRnnCopies][2][B][r] s_{k-1} / s_k
  unsigned int* rec_count;         // arrivals of the recurrence CTAs
  int n_rec, dpc;                  // recurrence CTAs, state entries per recurrence CTA
};

// Shared-memory layout: the W2 ring, the U ring (whose stages the transposers turn into
// z tiles in place), two E operand buffers, and for the RNN head the recurrence's scratch
// and its Wrec rows.  The RNN head's E operand has 2 NB rows (the hi and the lo bf16 image
// of each request's row, see the MMA issue loop), so it takes one accumulator and U tile
// less in flight and a 3-stage W2 ring.
template <int NB, bool Rnn>
struct Smem {
  static constexpr int kWStages = Rnn ? 3 : kWStagesMarkov;
  static constexpr int kDepth = Rnn ? 3 : kDepthMarkov;
  static constexpr int kUStages = kDepth;
  static constexpr int kWStageBytes = 2 * kKChunkMax * 128;  // two 64-column boxes
  static constexpr int kUStageBytes = NB * 128 * 4;
  static constexpr int kNE = Rnn ? 2 * NB : NB;               // rows of the E operand (MMA N)
  static constexpr int kEBytes = kNE * 256 * 2;               // up to r = 256
  static constexpr int kZBytes = NB * 128 * 4;             // RNN: the recurrence's scratch
  static constexpr int kOffW = 0;
  static constexpr int kOffU = kOffW + kWStages * kWStageBytes;
  static constexpr int kOffE = kOffU + kUStages * kUStageBytes;
  static constexpr int kOffZ = kOffE + 2 * kEBytes;
  static constexpr int kOffRec = kOffZ + (Rnn ? kDepth * kZBytes : 0);
  static constexpr int kRecBytes = Rnn ? kRnnRecBytes : 0;     // a recurrence CTA's Wrec rows
  static constexpr int kBytes = kOffRec + kRecBytes;
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Order-preserving map of a (non-NaN) float to a 32-bit unsigned key and back: larger
// float <-> larger key, so the warp's integer max reduction (redux.sync) gives the exact
// float maximum in one instruction.
__device__ __forceinline__ uint32_t float_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ float warp_max(float x) {
  return key_float(__reduce_max_sync(0xffffffffu, float_key(x)));
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ int token_of_key(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

// bf16 bits of a finite float, rounded to nearest even
__device__ __forceinline__ uint32_t bf16_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}
__device__ __forceinline__ float bf16_val(uint32_t b) { return __uint_as_float(b << 16); }

// One step k of the RNN head for state entries [d0, d0 + dpc) of every request, by the 16
// sampler warps of a recurrence CTA, after the grid barrier of position k-1 (x_{k-1} known)
// and before E_k exists.  The operands go to a scratch region of shared memory (the size
// of three z tiles) with cp.async, which holds no registers: the previous state rows
// s_{k-1}[b] (none at k = 1, where the state is zero) and, once the argmax keys give
// x_{k-1}, the embedding rows W1[x_{k-1}] -- all of a round's copies in flight together,
// about two L2 round trips in all.  Requests go in rounds of as many as fit.  An item is
// one (entry e, request b of the round); half-warp h (warp h / 2, lanes 16 (h % 2) ..)
// takes items h, h + 32, ...  Lane l of a half-warp forms the sums over the 8-entry chunks
// l, l + 16, ... of both halves of the 2r-long operand [s_{k-1}[b] ; W1[x_{k-1}]] against
// the three rows of Wrec (shared memory when a recurrence CTA's 3 dpc rows were staged
// there, row (g, e) at (g dpc + e) 2r, else global memory), and four shuffles reduce them,
// leaving the same sums in every lane.  Then s_k[b][i] = gate s_{k-1}[b][i] +
// (1 - gate) tanh(cand), E_k[b][i] = tanh(output) and E_k's two bf16 terms hi = bf16(E),
// lo = bf16(E - hi) for the tensor-core operand are written: lane c of the half-warp
// writes copy c of the state and of the bf16 terms, lane 0 the fp32 row.  Everything other
// CTAs wrote in this call (the state, the argmax keys) is read through L2.
constexpr int kRnnHalves = 2 * kSamplers;

// row (g, e) of this CTA's recurrent weights: shared memory when staged, else global
__device__ __forceinline__ const uint16_t* rnn_row(const DraftParams& p, const uint16_t* wsm,
                                                   int g, int e, int d0) {
  const int R2 = 2 * p.r;
  return wsm ? wsm + (size_t)(g * p.dpc + e) * R2 : p.Wrec + (size_t)(g * p.r + d0 + e) * R2;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ float half_warp_sum(float a) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
  return a;
}

// a += sum over 8 entries of x (8 floats at xf, or 8 bf16 at xb) times the 8 bf16 at w
__device__ __forceinline__ float dot8_f32(const float* xf, uint4 w, float a) {
  const float4 x0 = reinterpret_cast<const float4*>(xf)[0];
  const float4 x1 = reinterpret_cast<const float4*>(xf)[1];
  a = fmaf(x0.x, bf16_val(w.x & 0xFFFFu), a); a = fmaf(x0.y, bf16_val(w.x >> 16), a);
  a = fmaf(x0.z, bf16_val(w.y & 0xFFFFu), a); a = fmaf(x0.w, bf16_val(w.y >> 16), a);
  a = fmaf(x1.x, bf16_val(w.z & 0xFFFFu), a); a = fmaf(x1.y, bf16_val(w.z >> 16), a);
  a = fmaf(x1.z, bf16_val(w.w & 0xFFFFu), a); a = fmaf(x1.w, bf16_val(w.w >> 16), a);
  return a;
}
__device__ __forceinline__ float dot8_bf16(uint4 x, uint4 w, float a) {
  a = fmaf(bf16_val(x.x & 0xFFFFu), bf16_val(w.x & 0xFFFFu), a);
  a = fmaf(bf16_val(x.x >> 16), bf16_val(w.x >> 16), a);
  a = fmaf(bf16_val(x.y & 0xFFFFu), bf16_val(w.y & 0xFFFFu), a);
  a = fmaf(bf16_val(x.y >> 16), bf16_val(w.y >> 16), a);
  a = fmaf(bf16_val(x.z & 0xFFFFu), bf16_val(w.z & 0xFFFFu), a);
  a = fmaf(bf16_val(x.z >> 16), bf16_val(w.z >> 16), a);
  a = fmaf(bf16_val(x.w & 0xFFFFu), bf16_val(w.w & 0xFFFFu), a);
  a = fmaf(bf16_val(x.w >> 16), bf16_val(w.w >> 16), a);
  return a;
}

__device__ __noinline__ void rnn_step(const DraftParams& p, const uint16_t* wsm, uint8_t* zs,
                                      int zbytes, int k, int d0, int sw, int lane, int stid) {
  const int r = p.r, C = 3 * r, chunks = r / 8;   // 8-entry chunks per half (r % 16 == 0)
  const int half = lane >> 4, hl = lane & 15;
  const size_t scopy = (size_t)2 * p.B * r;        // floats per state copy
  const float* s_prev = p.state + (blockIdx.x % kRnnCopies) * scopy + (size_t)((k - 1) & 1) * p.B * r;
  float* s_next = p.state + (size_t)(k & 1) * p.B * r;  // copy 0; every copy is written
  const int Bc = min(p.B, zbytes / (6 * r));       // requests per round (>= 32 for r <= 256)
  float* xs = reinterpret_cast<float*>(zs);                             // [Bc][r] s_{k-1}
  uint16_t* xe = reinterpret_cast<uint16_t*>(zs + (size_t)Bc * r * 4);   // [Bc][r] W1 rows
  for (int b0 = 0; b0 < p.B; b0 += Bc) {
    const int nb = min(Bc, p.B - b0);
    if (k > 1)
      for (int idx = stid; idx < nb * r / 4; idx += kSamplerThreads)
        cp_async16(xs + (size_t)idx * 4, s_prev + (size_t)b0 * r + (size_t)idx * 4);
    for (int idx = stid; idx < nb * chunks; idx += kSamplerThreads) {
      const int bl = idx / chunks, q = idx - bl * chunks, b = b0 + bl;
      int prev = k == 1 ? p.anchor[b] : token_of_key(__ldcg(p.keys + (size_t)(k - 2) * p.B + b));
      if (prev < 0 || prev >= p.V) {
        if (q == 0) set_device_error(p.err, DSPARK_ERR_DEVICE_CHECK);
        prev = 0;
      }
      cp_async16(xe + (size_t)bl * r + q * 8, p.W1 + (size_t)prev * r + q * 8);
    }
    cp_async_wait_all();
    named_bar_sync(kNamedBarSamplers, kSamplerThreads);
    const int n_items = p.dpc * nb;
    for (int base = 2 * sw; base < n_items; base += kRnnHalves) {
      const int it = base + half;
      const bool valid = it < n_items;
      const int e = valid ? it / nb : 0, bl = valid ? it - e * nb : 0, i = d0 + e;
      const uint16_t* wg = rnn_row(p, wsm, 0, e, d0);
      const uint16_t* wc = rnn_row(p, wsm, 1, e, d0);
      const uint16_t* wo = rnn_row(p, wsm, 2, e, d0);
      float hg = 0.f, hc = 0.f, ho = 0.f;
      if (valid) {                        // every lane of the half-warp: one address each
        const float* hpr = p.hp + ((size_t)(b0 + bl) * p.gamma + (k - 1)) * C + i;
        hg = __ldg(hpr);
        hc = __ldg(hpr + r);
        ho = __ldg(hpr + 2 * r);
      }
      float ag = 0.f, ac = 0.f, ao = 0.f;
      for (int q = hl; q < chunks; q += 16) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xe + (size_t)bl * r + q * 8);
        ag = dot8_bf16(xv, *reinterpret_cast<const uint4*>(wg + r + q * 8), ag);
        ac = dot8_bf16(xv, *reinterpret_cast<const uint4*>(wc + r + q * 8), ac);
        ao = dot8_bf16(xv, *reinterpret_cast<const uint4*>(wo + r + q * 8), ao);
        if (k > 1) {
          const float* xf = xs + (size_t)bl * r + q * 8;
          ag = dot8_f32(xf, *reinterpret_cast<const uint4*>(wg + q * 8), ag);
          ac = dot8_f32(xf, *reinterpret_cast<const uint4*>(wc + q * 8), ac);
          ao = dot8_f32(xf, *reinterpret_cast<const uint4*>(wo + q * 8), ao);
        }
      }
      ag = half_warp_sum(ag);
      ac = half_warp_sum(ac);
      ao = half_warp_sum(ao);
      if (valid) {
        // every lane has the sums; lane c of the half-warp writes copy c of s_k and of the
        // E rows (one store instruction per value), lane 0 the fp32 row kept for verification
        const int b = b0 + bl;
        const float sold = k > 1 ? xs[(size_t)bl * r + i] : 0.f;
        const float gate = 1.f / (1.f + expf(-(ag + hg)));
        const float sn = gate * sold + (1.f - gate) * tanhf(ac + hc);
        const float ev = tanhf(ao + ho);
        if (hl == 0) p.E_all[((size_t)b * p.gamma + (k - 1)) * r + i] = ev;
        if (hl < kRnnCopies) {
          const uint32_t hi = bf16_rne(ev);
          const size_t ecopy = (size_t)p.B * 2 * r;    // bf16 per E copy
          s_next[hl * scopy + (size_t)b * r + i] = sn;
          p.E_hl[hl * ecopy + (size_t)b * 2 * r + i] = (uint16_t)hi;
          p.E_hl[hl * ecopy + (size_t)b * 2 * r + r + i] = (uint16_t)bf16_rne(ev - bf16_val(hi));
        }
      }
    }
    named_bar_sync(kNamedBarSamplers, kSamplerThreads);   // the rows are read before the next round
  }
}

// Merge the G partials of request b at position kp into x, q, max and sum (one warp).
// One pass: every lane issues the loads of all its partials (G <= kDraftMaxCtas, so at
// most five per lane) and of the token key together, then merges locally and across the
// warp; a CTA that merges runs this right after its grid-barrier arrival, so it is kept
// to about one L2 round trip.
constexpr int kMergePerLane = (kDraftMaxCtas + 31) / 32;
template <bool Greedy>
__device__ __forceinline__ void finalize_row(const DraftParams& p, int b, int kp, int G, int lane) {
  const unsigned long long key = __ldcg(p.keys + (size_t)(kp - 1) * p.B + b);
  const RowState* base = p.partials + ((size_t)(kp % 3) * p.B + b) * G;
  float pm[kMergePerLane], ps[kMergePerLane], pz[kMergePerLane];
  int pi[kMergePerLane];
#pragma unroll
  for (int u = 0; u < kMergePerLane; ++u) {
    const int g = lane + 32 * u;
    pm[u] = -INFINITY; ps[u] = 0.f; pz[u] = -INFINITY; pi[u] = -1;
    if (g < G) {
      pm[u] = __ldcg(&base[g].m);
      ps[u] = __ldcg(&base[g].s);
      pz[u] = __ldcg(&base[g].z);
      pi[u] = __ldcg(&base[g].idx);
    }
  }
  const int x = token_of_key(key);
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < kMergePerLane; ++u) m = fmaxf(m, pm[u]);
  m = warp_max(m);
  float s = 0.f, zx = -INFINITY;
#pragma unroll
  for (int u = 0; u < kMergePerLane; ++u) {
    if (pm[u] != -INFINITY) s += ps[u] * expf(pm[u] - m);
    if (pi[u] == x) zx = pz[u];
  }
  s = warp_sum(s);
  zx = warp_max(zx);
  if (lane == 0) {
    const size_t o = (size_t)b * p.gamma + (kp - 1);
    p.tokens[o] = x;
    // a greedy draft proposes the point mass at x: q(x) = 1
    p.q_tok[o] = Greedy ? 1.f : expf(zx - m) / s;
    p.row_max[o] = m;
    p.row_sumexp[o] = s;
  }
}

template <int NB, bool Greedy, bool Rnn>
__global__ void __launch_bounds__(kThreads, 1) draft_fused_kernel(
    const __grid_constant__ CUtensorMap w2_map, const __grid_constant__ CUtensorMap u_map,
    const DraftParams p) {
  using S = Smem<NB, Rnn>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t w_full[S::kWStages], w_empty[S::kWStages];
  __shared__ uint64_t u_full[S::kUStages], u_empty[S::kUStages];
  __shared__ uint64_t e_full[2], e_empty[2];
  __shared__ uint64_t acc_full[S::kDepth], acc_empty[S::kDepth];
  __shared__ uint64_t z_full[S::kDepth];
  __shared__ uint64_t mma_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int t_lo = (int)((long long)cta * p.n_tiles / G);
  const int t_hi = (int)((long long)(cta + 1) * p.n_tiles / G);
  const int my_tiles = t_hi - t_lo;
  const int kc = p.kc;
  const int n_kchunks = p.r / kc;
  const int n_jobs = p.gamma * p.n_chunks;
  // tcgen05.alloc takes a power of two of at least 32 columns
  uint32_t tmem_cols = 32;
  while (tmem_cols < (uint32_t)(S::kDepth * S::kNE)) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S::kWStages; ++i) { mbar_init(&w_full[i], 1); mbar_init(&w_empty[i], 1); }
    for (int i = 0; i < S::kUStages; ++i) { mbar_init(&u_full[i], 1); mbar_init(&u_empty[i], kSamplers); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&e_full[i], 1);
      mbar_init(&e_empty[i], 1);
    }
    for (int i = 0; i < S::kDepth; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
      mbar_init(&z_full[i], 4);
    }
    mbar_init(&mma_drain, 1);
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_s, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_base_s;
  // the next kernel on the stream (launched with programmatic serialization) may be
  // scheduled as soon as SMs free up; it waits for this grid's completion itself
  pdl_launch_dependents();

  // One thread's bounded wait; a timeout aborts the CTA.  The abort flag is read only once
  // the first (sleeping) try has not seen the phase complete: a shared-memory read ahead of
  // every wait made the single-lane MMA issue loop measurably slower per tile on GB300.
  auto wait1 = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    const long long t0 = sm_cycles();
    for (;;) {
      if (*(volatile int*)&abort_s) return false;
      if (mbar_try_wait_sleep(bar, parity)) return true;
      if (sm_cycles() - t0 > p.wait_cycles) {
        set_device_error(p.err, DSPARK_ERR_TIMEOUT);
        atomicExch(&abort_s, 1);
        return false;
      }
    }
  };
  // a whole warp's bounded wait with a warp-uniform result (every lane sleeps on the
  // barrier and acquires for itself)
  auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
    const bool ok = wait1(bar, parity);
    return __all_sync(0xffffffffu, ok);
  };

  // The producer and the MMA issuer run their loops on one elected lane: a whole-warp loop
  // (every lane waiting, then a warp vote and a __syncwarp per K-chunk) measured on GB300
  // twice as slow per tile as the single-lane issue loop.
  if (warp == kProducerWarp) {
    // -------------------------------------------------------------- W2 stage producer
    if (lane == 0) {
      prefetch_tensormap(&w2_map);
      const uint64_t keep = policy_evict_last();
      const uint32_t w_bytes = 2u * (uint32_t)kc * 128u;
      uint32_t ws = 0;
      bool ok = true;
      for (int job = 0; job < n_jobs && ok; ++job) {
        for (int t = t_lo; t < t_hi && ok; ++t) {
          const int v0 = t * kGemmTileV;
          for (int i = 0; i < n_kchunks; ++i, ++ws) {
            const int s = ws % S::kWStages;
            if (!(ok = wait1(&w_empty[s], ((ws / S::kWStages) & 1) ^ 1))) break;
            uint8_t* dst = smem + S::kOffW + s * S::kWStageBytes;
            mbar_arrive_expect_tx(&w_full[s], w_bytes);
            if (p.W2p) {
              // packed: the stage image is contiguous, one 1-D bulk copy
              const uint16_t* src = p.W2p + ((size_t)t * n_kchunks + i) * (size_t)kc * 128;
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                  " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
                  "l"(reinterpret_cast<uint64_t>(src)), "r"(w_bytes), "r"(smem_u32(&w_full[s])),
                  "l"(keep)
                  : "memory");
            } else {
              tma_load_2d(dst, &w2_map, &w_full[s], v0, i * kc, keep);
              tma_load_2d(dst + kc * 128, &w2_map, &w_full[s], v0 + 64, i * kc, keep);
            }
          }
        }
      }
      // drain: every issued copy has landed before the CTA may exit (a stage whose wait
      // failed above was never issued, so only stages below ws are in flight)
      for (uint32_t i = ws > (uint32_t)S::kWStages ? ws - S::kWStages : 0; i < ws; ++i)
        mbar_wait(&w_full[i % S::kWStages], (i / S::kWStages) & 1, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp == kUProducerWarp) {
    // ----------------------------------------------------------------- U tile producer
    // U does not depend on the drafted tokens: its ring runs a ring's depth of tiles ahead
    // of the samplers, across positions, independently of the W2 ring.
    if (lane == 0) {
      prefetch_tensormap(&u_map);
      uint64_t stream_pol;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream_pol));
      uint32_t us = 0;
      bool ok = true;
      for (int job = 0; job < n_jobs && ok; ++job) {
        const int k = job / p.n_chunks + 1, c = job % p.n_chunks;
        for (int t = t_lo; t < t_hi; ++t, ++us) {
          const int su = us % S::kUStages;
          if (!(ok = wait1(&u_empty[su], ((us / S::kUStages) & 1) ^ 1))) break;
          mbar_arrive_expect_tx(&u_full[su], (uint32_t)S::kUStageBytes);
          asm volatile(
              "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
              ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(
                  smem_u32(smem + S::kOffU + su * S::kUStageBytes)),
              "l"(reinterpret_cast<uint64_t>(&u_map)), "r"(smem_u32(&u_full[su])),
              "r"(t * kGemmTileV), "r"(k - 1), "r"(c * NB), "l"(stream_pol)
              : "memory");
        }
      }
      for (uint32_t i = us > (uint32_t)S::kUStages ? us - S::kUStages : 0; i < us; ++i)
        mbar_wait(&u_full[i % S::kUStages], (i / S::kUStages) & 1, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // -------------------------------------------------------------------- MMA issuer
    // The 16-row K steps of one W2 stage are a compile-time count (1, 2 or 4): a runtime
    // trip count with guarded issues slowed the issue loop on GB300 as much as the
    // abort-flag reads did.
    // Descriptors are built once and advanced by adding (byte offset >> 4) to their start-
    // address field (bits 0-13; every operand lies below 256 KB, so the sum never carries
    // into the stride fields).  The issuing lane shares its sub-partition with sampler
    // warps, so every instruction saved here shortens the tile cadence.
    auto issue_loop = [&](auto ksteps_c) {
      constexpr int KS = decltype(ksteps_c)::value;
      // N = NB (Markov head) or 2 NB (RNN head: hi rows, then lo rows; the transposers add
      // the two accumulator halves), so one MMA per K step either way
      const uint32_t idesc = idesc_bf16_f32(128, S::kNE, 1, 0);
      const uint64_t a_base = smem_desc(smem_u32(smem + S::kOffW), (uint32_t)KS * 2048u, 1024u,
                                        kSwizzle128B);
      uint32_t ws = 0, tc = 0;
      bool ok = true;
      for (int job = 0; job < n_jobs && ok; ++job) {
        const int eb = job & 1;
        // (the E writers fenced their stores to the async proxy before arriving)
        if (!(ok = wait1(&e_full[eb], (job >> 1) & 1))) break;
        const uint64_t b_base =
            smem_desc(smem_u32(smem + S::kOffE + eb * S::kEBytes), 16u, 1024u, kSwizzle128B);
        for (int t = 0; t < my_tiles && ok; ++t, ++tc) {
          const int ab = tc % S::kDepth;
          if (!(ok = wait1(&acc_empty[ab], ((tc / S::kDepth) & 1) ^ 1))) break;
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + (uint32_t)(ab * S::kNE);
          for (int i = 0; i < n_kchunks; ++i, ++ws) {
            const int s = ws % S::kWStages;
            // TMA data: the barrier's transaction count orders it before the MMAs; no
            // tcgen05 fence here (a fence per chunk would serialise on MMA completion)
            if (!(ok = wait1(&w_full[s], (ws / S::kWStages) & 1))) break;
            const uint64_t a_s = a_base + (uint64_t)((s * S::kWStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
              const uint32_t kg = (uint32_t)(i * KS + kk);   // global 16-row K step
              // A: 16 K rows of the MN-major stage are 2048 bytes apart; B: K-block kg/4 of
              // the K-major E buffer, 32 bytes per 16-element step inside its 128-byte rows
              const uint64_t ad = a_s + (uint64_t)(kk * (2048 >> 4));
              const uint64_t bd = b_base + (uint64_t)((kg >> 2) * (uint32_t)(S::kNE * 128 / 16) + (kg & 3) * 2u);
              umma_bf16_f32(d_tmem, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(&w_empty[s]);
          }
          if (!ok) break;
          umma_commit(&acc_full[ab]);
        }
        if (ok) umma_commit(&e_empty[eb]);
      }
    };
    if (lane == 0) {
      if (kc == 64) issue_loop(std::integral_constant<int, 4>{});
      else if (kc == 32) issue_loop(std::integral_constant<int, 2>{});
      else issue_loop(std::integral_constant<int, 1>{});
      // drain: every issued MMA has completed before tensor memory is released
      umma_commit(&mma_drain);
      mbar_wait(&mma_drain, 0, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp < kFirstSampler) {
    // ----------------------------------------------- transposers: TMEM (+U) -> z rows
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int vl = q * 32 + lane;                 // vocabulary row inside the tile
    const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
    uint32_t tc = 0;
    bool ok = true;
    for (int job = 0; job < n_jobs && ok; ++job) {
      for (int t = 0; t < my_tiles && ok; ++t, ++tc) {
        const int ab = tc % S::kDepth;
        const uint32_t par = (tc / S::kDepth) & 1;
        if (!(ok = wait_warp(&acc_full[ab], par))) break;
        tc_fence_after_sync();
        // the U tile of the same tile count (the U ring has the accumulators' depth)
        if (!(ok = wait_warp(&u_full[ab], par))) break;
        float* Zs = reinterpret_cast<float*>(smem + S::kOffU + ab * S::kUStageBytes);
        if constexpr (Rnn) {
          // bias = the hi columns + the lo columns, 16 requests at a time; z = bias + U
#pragma unroll
          for (int c16 = 0; c16 < NB; c16 += 16) {
            float vh[16], vlo[16];
            tmem_ld_32x32b_x16(trow + (uint32_t)(ab * S::kNE + c16), vh);
            tmem_ld_32x32b_x16(trow + (uint32_t)(ab * S::kNE + NB + c16), vlo);
            tmem_ld_wait();
#pragma unroll
            for (int b = 0; b < 16; ++b) {
              float* zp = Zs + (c16 + b) * 128 + vl;
              *zp = (vh[b] + vlo[b]) + *zp;
            }
          }
        } else {
          float vals[NB];
#pragma unroll
          for (int c16 = 0; c16 < NB; c16 += 16)
            tmem_ld_32x32b_x16(trow + (uint32_t)(ab * NB + c16), *reinterpret_cast<float(*)[16]>(vals + c16));
          tmem_ld_wait();
#pragma unroll
          for (int b = 0; b < NB; ++b) Zs[b * 128 + vl] = vals[b] + Zs[b * 128 + vl];
        }
        tc_fence_before_sync();
        // the stage is next written by the U producer's TMA (async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&acc_empty[ab]);
          mbar_arrive(&z_full[ab]);
        }
      }
    }
  } else {
    // ----------------------------------------------------------------------- samplers
    constexpr int RPW = NB / kSamplers;           // requests per sampler warp
    const int sw = warp - kFirstSampler;
    const int stid = threadIdx.x - kFirstSampler * 32;
    uint32_t tc = 0;
    // RNN head: a recurrence CTA stages its rows of Wrec (gate, candidate and output of its
    // dpc state entries) in shared memory once, when they fit; the samplers' named barrier
    // ahead of the first recurrence step orders the copy before any use
    const uint16_t* wrec_s = nullptr;
    if constexpr (Rnn) {
      if (cta < p.n_rec && 3 * p.dpc * 4 * p.r <= S::kRecBytes) {
        uint16_t* dst = reinterpret_cast<uint16_t*>(smem + S::kOffRec);
        const int R2 = 2 * p.r, chunks = R2 / 8;   // 16-byte chunks per row
        for (int idx = stid; idx < 3 * p.dpc * chunks; idx += kSamplerThreads) {
          const int row = idx / chunks, q = idx - row * chunks;
          const int g = row / p.dpc, e = row - g * p.dpc;
          reinterpret_cast<uint4*>(dst)[idx] = __ldg(
              reinterpret_cast<const uint4*>(p.Wrec + (size_t)(g * p.r + cta * p.dpc + e) * R2) + q);
        }
        wrec_s = dst;
      }
    }
    // The first kGatherWarps sampler warps publish the E operand of job `j` (chunk c,
    // position k): E = W1[x_{k-1}] as the K-major, 128-byte-swizzled B operand (16-byte
    // chunk q of row n goes to chunk (q % 8) ^ (n % 8) of line n of K-block q / 8).  Thread
    // t takes row t % NB and every (128 / NB)-th chunk of it, all its loads in flight at
    // once.  For k > 1 they first wait for the grid barrier (one lane polls).  The other
    // sampler warps take no part: their first z tile cannot complete before E is published.
    constexpr int kGatherThreads = kGatherWarps * 32;
    constexpr int kGatherGroups = kGatherThreads / NB;
    // RNN head: at the first chunk of position k, the recurrence CTAs (cta < n_rec) first
    // wait for the grid barrier of position k - 1 (x_{k-1} known), run the recurrence for
    // their state entries with all sampler warps and count themselves in rec_count (a
    // release reduction after the samplers' named barrier); the sampler warps of every CTA
    // then wait until all n_rec have arrived for position k and load E_k as 2 NB operand
    // rows: hi = bf16(E) for request n in row n, lo = bf16(E - hi) in row NB + n, in the
    // same swizzled K-major layout.
    auto publish_E_rnn = [&](int j, int c, int k, bool wait_grid) {
      const bool rec = c == 0 && cta < p.n_rec;
      if (rec) {
        if (stid == 0 && wait_grid) {
          const unsigned int target = (unsigned int)G * (unsigned int)(k - 1) + p.grid_extra;
          const long long t0 = sm_cycles();
          while (ld_acquire_u32(p.grid_count) < target) {
            if (*(volatile int*)&abort_s || sm_cycles() - t0 > p.wait_cycles) {
              set_device_error(p.err, DSPARK_ERR_TIMEOUT);
              atomicExch(&abort_s, 1);
              break;
            }
          }
        }
        named_bar_sync(kNamedBarSamplers, kSamplerThreads);
        // called by every sampler thread whatever the abort flag says (the step's named
        // barriers need all of them; it has no other waits)
        rnn_step(p, wrec_s, smem + S::kOffZ, S::kDepth * S::kZBytes, k, cta * p.dpc, sw, lane,
                 stid);
        named_bar_sync(kNamedBarSamplers, kSamplerThreads);
        if (stid == 0)
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.rec_count) : "memory");
      }
      // every sampler warp gathers: 2 NB rows of r bf16 (hi rows, then lo rows), one row per
      // thread group, each thread's (at most four) 16-byte loads in flight together
      if (stid == 0) {
        if (c == 0) {
          const unsigned int target = (unsigned int)p.n_rec * (unsigned int)k + p.grid_extra;
          const long long t0 = sm_cycles();
          while (ld_acquire_u32(p.rec_count) < target) {
            if (*(volatile int*)&abort_s || sm_cycles() - t0 > p.wait_cycles) {
              set_device_error(p.err, DSPARK_ERR_TIMEOUT);
              atomicExch(&abort_s, 1);
              break;
            }
          }
        }
        wait1(&e_empty[j & 1], ((j >> 1) & 1) ^ 1);
      }
      named_bar_sync(kNamedBarSamplers, kSamplerThreads);
      if (!*(volatile int*)&abort_s) {
        constexpr int kRows = 2 * NB;
        constexpr int kGroups = kSamplerThreads / kRows;
        constexpr int kPerR = (32 + kGroups - 1) / kGroups;   // r / 8 <= 32 chunks per row
        uint8_t* sE = smem + S::kOffE + (j & 1) * S::kEBytes;
        const int n = stid % kRows, grp = stid / kRows;
        const int b = c * NB + (n % NB);
        const int kchunks = p.r >> 3;
        const bool ok = b < p.B;
        const uint4* src = reinterpret_cast<const uint4*>(
            p.E_hl + (size_t)(cta % kRnnCopies) * p.B * 2 * p.r +
            ((size_t)(ok ? b : 0) * 2 + (n >= NB ? 1 : 0)) * p.r);
        uint4 val[kPerR];
#pragma unroll
        for (int u = 0; u < kPerR; ++u) {
          const int q = grp + u * kGroups;
          val[u] = (ok && q < kchunks) ? __ldcg(src + q) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kPerR; ++u) {
          const int q = grp + u * kGroups;
          if (q < kchunks)
            *reinterpret_cast<uint4*>(sE + (size_t)(q >> 3) * kRows * 128 + (size_t)n * 128 +
                                      (((q & 7) ^ (n & 7)) << 4)) = val[u];
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(kNamedBarSamplers, kSamplerThreads);
      if (stid == 0) mbar_arrive(&e_full[j & 1]);
    };
    auto publish_E = [&](int j, int c, int k, bool wait_grid) {
      if constexpr (Rnn) {
        publish_E_rnn(j, c, k, wait_grid);
        return;
      }
      if (sw >= kGatherWarps) return;
      if (stid == 0) {
        if (wait_grid) {
          const unsigned int target = (unsigned int)G * (unsigned int)(k - 1) + p.grid_extra;
          const long long t0 = sm_cycles();
          while (ld_acquire_u32(p.grid_count) < target) {
            if (*(volatile int*)&abort_s || sm_cycles() - t0 > p.wait_cycles) {
              set_device_error(p.err, DSPARK_ERR_TIMEOUT);
              atomicExch(&abort_s, 1);
              break;
            }
          }
        }
        wait1(&e_empty[j & 1], ((j >> 1) & 1) ^ 1);
      }
      named_bar_sync(kNamedBarGather, kGatherThreads);
      if (!*(volatile int*)&abort_s) {
        uint8_t* sE = smem + S::kOffE + (j & 1) * S::kEBytes;
        const int n = stid % NB, grp = stid / NB;
        const int b = c * NB + n;
        const int kchunks = p.r >> 3;               // 16-byte chunks per W1 row (<= 32)
        int prev = -1;
        if (b < p.B)
          prev = (k == 1) ? p.anchor[b] : token_of_key(__ldcg(p.keys + (size_t)(k - 2) * p.B + b));
        const bool ok = b < p.B && prev >= 0 && prev < p.V;
        if (b < p.B && !ok) set_device_error(p.err, DSPARK_ERR_DEVICE_CHECK);
        const uint4* src = reinterpret_cast<const uint4*>(p.W1 + (size_t)(ok ? prev : 0) * p.r);
        constexpr int kPer = 32 / kGatherGroups > 0 ? (32 + kGatherGroups - 1) / kGatherGroups : 1;
        uint4 val[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int q = grp + i * kGatherGroups;
          val[i] = (ok && q < kchunks) ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int q = grp + i * kGatherGroups;
          if (q < kchunks)
            *reinterpret_cast<uint4*>(sE + (size_t)(q >> 3) * NB * 128 + (size_t)n * 128 +
                                      (((q & 7) ^ (n & 7)) << 4)) = val[i];
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(kNamedBarGather, kGatherThreads);
      if (stid == 0) mbar_arrive(&e_full[j & 1]);
    };
    // every sampler waits for the grid barrier (only at the end of the call)
    auto grid_wait = [&](unsigned int target) {
      if (stid == 0) {
        const long long t0 = sm_cycles();
        while (ld_acquire_u32(p.grid_count) < target) {
          if (*(volatile int*)&abort_s || sm_cycles() - t0 > p.wait_cycles) {
            set_device_error(p.err, DSPARK_ERR_TIMEOUT);
            atomicExch(&abort_s, 1);
            break;
          }
        }
      }
      named_bar_sync(kNamedBarSamplers, kSamplerThreads);
    };

    for (int job = 0; job < n_jobs; ++job) {
      const int k = job / p.n_chunks + 1, c = job % p.n_chunks;
      if (c == 0) publish_E(job, 0, k, k > 1);
      // the next chunk of the same position only needs x_{k-1}: publish it now
      if (c + 1 < p.n_chunks) publish_E(job + 1, c + 1, k, false);

      // Per-request state of this warp's rows.  Warp-uniform: the lazy reference Mr (a
      // past warp max, raised only when a logit exceeds it by more than kLazy, so that
      // exp(z - Mr) cannot overflow), the filter threshold Tf ~ exp(best - Mr) (shrunk by
      // kShrink to absorb rounding), the best exact score bsc = z* - log E*, its index and
      // logit.  Per lane: the sum of exp(z - Mr) and the max of z.
      float Mr[RPW], Tf[RPW], bsc[RPW], bz[RPW], s[RPW], mx[RPW];
      int bi[RPW];
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        Mr[i] = -INFINITY; Tf[i] = 0.f; bsc[i] = -INFINITY; bz[i] = -INFINITY; s[i] = 0.f;
        mx[i] = -INFINITY; bi[i] = -1;
      }
      for (int t = 0; t < my_tiles; ++t, ++tc) {
        const int zb = tc % S::kDepth;
        const uint32_t par = (tc / S::kDepth) & 1;
        if (!wait_warp(&z_full[zb], par)) continue;
        const float* Zs = reinterpret_cast<const float*>(smem + S::kOffU + zb * S::kUStageBytes);
        const int v = (t_lo + t) * kGemmTileV + 4 * lane;
        const bool ragged = (t_lo + t + 1) * kGemmTileV > p.V;
        // A: the logits of this lane's 4 vocabulary entries for each row
        float z[RPW][4];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          const float4 z4 = *reinterpret_cast<const float4*>(Zs + (sw * RPW + i) * 128 + 4 * lane);
          z[i][0] = z4.x; z[i][1] = z4.y; z[i][2] = z4.z; z[i][3] = z4.w;
          if (ragged) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (v + j >= p.V) z[i][j] = -INFINITY;
          }
        }
        // B: running max and the lazy reference
        bool raise = false;
        float lm[RPW];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          lm[i] = fmaxf(fmaxf(z[i][0], z[i][1]), fmaxf(z[i][2], z[i][3]));
          mx[i] = fmaxf(mx[i], lm[i]);
          raise |= lm[i] > Mr[i] + kLazy;
        }
        if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
          for (int i = 0; i < RPW; ++i) {
            const float wm = warp_max(lm[i]);
            if (wm > Mr[i] + kLazy) {
              s[i] *= (Mr[i] == -INFINITY) ? 0.f : expf(Mr[i] - wm);
              Mr[i] = wm;
              Tf[i] = bi[i] >= 0 ? expf(bsc[i] - wm) * kShrink : 0.f;
            }
          }
        }
        if constexpr (Greedy) {
          // greedy: the softmax sums, and the first index of the warp's largest logit when
          // it beats the best so far (an equal logit of a later tile has a larger index)
#pragma unroll
          for (int i = 0; i < RPW; ++i) {
            const float mL = Mr[i] * kLog2e;
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i] += ex2_approx(fmaf(z[i][j], kLog2e, -mL));
            const uint32_t kme = float_key(lm[i] + 0.f);   // +0 and -0 compare equal
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, kme);
            const float wmax = key_float(kmax);
            if (wmax > bsc[i]) {
              int jl = 3;
#pragma unroll
              for (int j = 2; j >= 0; --j)
                if (z[i][j] == lm[i]) jl = j;
              bi[i] = (int)__reduce_min_sync(0xffffffffu,
                                             kme == kmax ? (uint32_t)(v + jl) : 0xFFFFFFFFu);
              bsc[i] = wmax;
              bz[i] = wmax;
            }
          }
        } else {
          // C: the random draws (independent chains across rows)
          uint4 d[RPW];
#pragma unroll
          for (int i = 0; i < RPW; ++i)
            d[i] = philox_wide(make_uint4((uint32_t)(v >> 2), (uint32_t)k,
                                          (uint32_t)(c * NB + sw * RPW + i), 0u), p.philox);
          // D: softmax sums and the cheap candidate test exp(z - Mr) > Tf * w
          float e[RPW][4], w[RPW][4];
          unsigned cm[RPW];
#pragma unroll
          for (int i = 0; i < RPW; ++i) {
            const float mL = Mr[i] * kLog2e;
            const uint32_t dw[4] = {d[i].x, d[i].y, d[i].z, d[i].w};
            cm[i] = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              e[i][j] = ex2_approx(fmaf(z[i][j], kLog2e, -mL));
              s[i] += e[i][j];
              w[i][j] = w_of_draw(dw[j]);
              cm[i] |= (e[i][j] > Tf[i] * w[i][j] ? 1u : 0u) << j;
            }
          }
          // E: candidates.  Tighten the threshold with the best lower bound
          // e (1 - w) / w <= e / E among them, then score the survivors exactly.
#pragma unroll
          for (int i = 0; i < RPW; ++i) {
            if (__any_sync(0xffffffffu, cm[i] != 0u)) {
              float L = 0.f;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if ((cm[i] >> j) & 1u) L = fmaxf(L, e[i][j] * (1.f - w[i][j]) * rcp_approx(w[i][j]));
              const float Teff = fmaxf(Tf[i], warp_max(L) * kShrink);
              unsigned sm = 0u;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                sm |= (((cm[i] >> j) & 1u) && e[i][j] > Teff * w[i][j] ? 1u : 0u) << j;
              float sc = -INFINITY, szz = -INFINITY;
              int sv = 0x7FFFFFFF;
              // exact scores for the survivors only (about one per warp and tile), in
              // increasing j as before, so that equal scores keep the smallest index: a loop
              // over the set bits runs the logarithms once per survivor instead of under a
              // predicate for every element
              while (sm) {
                const int j = __ffs(sm) - 1;
                sm &= sm - 1u;
                const float wj = j == 0 ? w[i][0] : j == 1 ? w[i][1] : j == 2 ? w[i][2] : w[i][3];
                const float zj = j == 0 ? z[i][0] : j == 1 ? z[i][1] : j == 2 ? z[i][2] : z[i][3];
                // E accurate (log1p), its logarithm the fast one (within 3 ulp of log E)
                const float scj = zj - __logf(exp1_from_w(wj));
                if (scj > sc) { sc = scj; sv = v + j; szz = zj; }
              }
              // the warp's best (largest score, then smallest index): two integer reductions,
              // a ballot and one shuffle
              {
                const uint32_t kme = float_key(sc + 0.f);   // +0 and -0 compare equal
                const uint32_t kmax = __reduce_max_sync(0xffffffffu, kme);
                const bool top = kme == kmax;
                const uint32_t vmin = __reduce_min_sync(0xffffffffu, top ? (uint32_t)sv : 0xFFFFFFFFu);
                const int src = __ffs(__ballot_sync(0xffffffffu, top && (uint32_t)sv == vmin)) - 1;
                sc = key_float(kmax);
                sv = (int)vmin;
                szz = __shfl_sync(0xffffffffu, szz, src);
              }
              if (sv != 0x7FFFFFFF && better(sc, sv, bsc[i], bi[i])) {
                bsc[i] = sc; bi[i] = sv; bz[i] = szz;
                Tf[i] = expf(sc - Mr[i]) * kShrink;
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&u_empty[zb]);
      }
      // publish this CTA's partials of the job's requests: the warp reductions of all its
      // rows first, then the stores and atomics.  No fence here: the thread that counts
      // the CTA into the grid barrier does so with a release reduction after the
      // samplers' named barrier, which orders every sampler's stores and atomics first.
      float pm[RPW], pst[RPW];
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        pm[i] = warp_max(mx[i]);
        pst[i] = warp_sum(s[i]) * (Mr[i] == -INFINITY ? 0.f : expf(Mr[i] - pm[i]));
      }
      if (lane == 0 && !*(volatile int*)&abort_s) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          const int b = c * NB + sw * RPW + i;
          if (b >= p.B) continue;
          RowState ps;
          ps.m = pm[i];
          ps.s = pst[i];
          ps.idx = bi[i];
          ps.z = bz[i];
          ps.score = bsc[i];
          p.partials[((size_t)(k % 3) * p.B + b) * G + cta] = ps;
          if (bi[i] >= 0) {
            atomicMax(p.keys + (size_t)(k - 1) * p.B + b, argmax_key(bsc[i], bi[i]));
            // the winner is one CTA's local best: warm L2 with its W1 row for the gather
            // that follows the grid barrier
            if (k < p.gamma)
              asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                               reinterpret_cast<uint64_t>(p.W1 + (size_t)bi[i] * p.r)),
                           "r"((uint32_t)p.r * 2u)
                           : "memory");
          }
        }
      }
      if (c + 1 == p.n_chunks) {
        // this CTA is done with position k: count it in the grid barrier
        named_bar_sync(kNamedBarSamplers, kSamplerThreads);
        if (stid == 0) {
          // a release reduction: every sampler's partials and key updates (ordered before
          // this thread by the named barrier) become visible before the count does, and
          // the thread does not wait for the add to return
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.grid_count) : "memory");
        }
        // merge this CTA's share of position k-1 while the other CTAs finish position k
        // (partials rotate over three slots: slot (k-1) % 3 is next written at position
        // k+2, after the barrier this CTA has not yet passed)
        if (k > 1 && !*(volatile int*)&abort_s)
          for (int b = cta + sw * G; b < p.B; b += kSamplers * G) finalize_row<Greedy>(p, b, k - 1, G, lane);
      }
    }
    // the last position: wait for every CTA, then merge this CTA's rows
    grid_wait((unsigned int)G * (unsigned int)p.gamma + p.grid_extra);
    if (!*(volatile int*)&abort_s)
      for (int b = cta + sw * G; b < p.B; b += kSamplers * G) finalize_row<Greedy>(p, b, p.gamma, G, lane);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, tmem_cols);
}

// U [B, gamma, V] fp32 as a 3-D tensor {V, gamma, B}; a box is 128 vocabulary entries of
// one position for NB requests.  Out-of-range entries read as zero.
bool encode_u_map(CUtensorMap* map, const float* U, int B, int gamma, int V, int NB) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)gamma, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)V * 4, (cuuint64_t)gamma * V * 4};
  cuuint32_t box[3] = {128, 1, (cuuint32_t)NB};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(U), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// one CTA per SM (the cooperative grid), or 0 if the kernel does not fit an SM
template <int NB, bool Greedy, bool Rnn>
int max_grid() {
  static std::atomic<int> cache[kMaxCachedDevices];
  return per_device_grid(cache, [] {
    int per = 0;
    const size_t smem = Smem<NB, Rnn>::kBytes + 1024;
    if (cudaFuncSetAttribute(draft_fused_kernel<NB, Greedy, Rnn>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, draft_fused_kernel<NB, Greedy, Rnn>,
                                                      kThreads, smem) != cudaSuccess)
      return -1;
    return per > 0 ? 1 : 0;
  });
}

template <int NB, bool Greedy, bool Rnn>
cudaError_t launch_fused(const CUtensorMap& w2_map, const CUtensorMap& u_map, const DraftParams& p,
                         int grid, cudaStream_t stream) {
  const size_t smem = Smem<NB, Rnn>::kBytes + 1024;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, draft_fused_kernel<NB, Greedy, Rnn>, w2_map, u_map, p);
}

}  // namespace

namespace {
template <bool Greedy, bool Rnn>
int grid_for(int NB) { return NB == 16 ? max_grid<16, Greedy, Rnn>() : max_grid<32, Greedy, Rnn>(); }

template <bool Greedy, bool Rnn>
cudaError_t launch_for(int NB, const CUtensorMap& w2_map, const CUtensorMap& u_map,
                       const DraftParams& p, int grid, cudaStream_t stream) {
  return NB == 16 ? launch_fused<16, Greedy, Rnn>(w2_map, u_map, p, grid, stream)
                  : launch_fused<32, Greedy, Rnn>(w2_map, u_map, p, grid, stream);
}

cudaError_t launch_draft_common(const uint16_t* W1, const uint16_t* W2, const uint16_t* W2p,
                                const float* U, const int32_t* anchor, int B, int gamma, int V,
                                int r, uint64_t seed, int32_t* tokens, float* q_tok,
                                float* row_max, float* row_sumexp, void* region, int* err,
                                bool greedy, const RnnDraftArgs* rnn, cudaStream_t stream) {
  if (!rnn) return cudaErrorInvalidValue;
  const int NB = B <= 16 ? 16 : 32;
  const int n_tiles = cdiv(V, kGemmTileV);
  int grid = greedy ? grid_for<true, true>(NB) : grid_for<false, true>(NB);
  if (grid <= 0) return cudaErrorInvalidConfiguration;
  if (grid > n_tiles) grid = n_tiles;
  if (grid > kDraftMaxCtas) grid = kDraftMaxCtas;
  DraftParams p;
  memset(&p, 0, sizeof(p));
  p.W1 = W1;
  p.W2p = W2p;
  p.anchor = anchor;
  p.B = B; p.gamma = gamma; p.V = V; p.r = r;
  p.n_tiles = n_tiles;
  p.n_chunks = cdiv(B, NB);
  p.kc = draft_kchunk(r);   // divides r (r % 16 == 0)
  p.seed = seed;
  p.philox = philox_keys(seed);
  const size_t part_bytes = align_up((size_t)3 * B * kDraftMaxCtas * sizeof(RowState), 256);
  char* base = static_cast<char*>(region);
  p.partials = reinterpret_cast<RowState*>(base);
  p.grid_count = reinterpret_cast<unsigned int*>(base + part_bytes);
  p.keys = reinterpret_cast<unsigned long long*>(base + part_bytes + 256);
  p.tokens = tokens;
  p.q_tok = q_tok;
  p.row_max = row_max;
  p.row_sumexp = row_sumexp;
  p.err = err;
  p.wait_cycles = draft_wait_limit();
  p.grid_extra = draft_barrier_offset();
  if (rnn) {
    p.Wrec = rnn->Wrec;
    p.hp = rnn->hp;
    p.E_all = rnn->E_all;
    p.state = rnn->state;
    p.E_hl = rnn->E_hl;
    p.rec_count = p.grid_count + 32;     // same zeroed 256-byte slot, another 128-byte line
    // recurrence CTAs: the largest divisor of r that the grid holds
    int n_rec = grid < r ? grid : r;
    while (r % n_rec) --n_rec;
    p.n_rec = n_rec;
    p.dpc = r / n_rec;
  }
  cudaError_t e = cudaMemsetAsync(base + part_bytes, 0,
                                  256 + (size_t)gamma * B * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  CUtensorMap w2_map, u_map;
  memset(&w2_map, 0, sizeof(w2_map));
  if (!W2p && !encode_w2_map(&w2_map, W2, V, r, p.kc)) return cudaErrorInvalidValue;
  if (!encode_u_map(&u_map, U, B, gamma, V, NB)) return cudaErrorInvalidValue;
  return greedy ? launch_for<true, true>(NB, w2_map, u_map, p, grid, stream)
                : launch_for<false, true>(NB, w2_map, u_map, p, grid, stream);
}
}  // namespace

cudaError_t launch_draft_fused(const uint16_t* W1, const uint16_t* W2, const float* U,
                               const int32_t* anchor, int B, int gamma, int V, int r,
                               uint64_t seed, int32_t* tokens, float* q_tok, float* row_max,
                               float* row_sumexp, void* region, int* err, cudaStream_t stream) {
  return launch_draft_lanes(W1, W2, nullptr, U, anchor, B, gamma, V, r, seed, false, tokens,
                            q_tok, row_max, row_sumexp, region, err, stream);
}

cudaError_t launch_draft_fused_packed(const uint16_t* W1, const uint16_t* W2p, const float* U,
                                      const int32_t* anchor, int B, int gamma, int V, int r,
                                      uint64_t seed, int32_t* tokens, float* q_tok,
                                      float* row_max, float* row_sumexp, void* region, int* err,
                                      cudaStream_t stream) {
  return launch_draft_lanes(W1, nullptr, W2p, U, anchor, B, gamma, V, r, seed, false, tokens,
                            q_tok, row_max, row_sumexp, region, err, stream);
}

cudaError_t launch_draft_fused_greedy(const uint16_t* W1, const uint16_t* W2, const uint16_t* W2p,
                                      const float* U, const int32_t* anchor, int B, int gamma,
                                      int V, int r, int32_t* tokens, float* q_tok,
                                      float* row_max, float* row_sumexp, void* region, int* err,
                                      cudaStream_t stream) {
  return launch_draft_lanes(W1, W2p ? nullptr : W2, W2p, U, anchor, B, gamma, V, r, 0, true,
                            tokens, q_tok, row_max, row_sumexp, region, err, stream);
}

cudaError_t launch_draft_fused_rnn(const uint16_t* W1, const uint16_t* W2, const uint16_t* W2p,
                                   const float* U, const int32_t* anchor, int B, int gamma, int V,
                                   int r, uint64_t seed, bool greedy, const RnnDraftArgs& rnn,
                                   int32_t* tokens, float* q_tok, float* row_max,
                                   float* row_sumexp, void* region, int* err, cudaStream_t stream) {
  return launch_draft_common(W1, W2p ? nullptr : W2, W2p, U, anchor, B, gamma, V, r, seed, tokens,
                             q_tok, row_max, row_sumexp, region, err, greedy, &rnn, stream);
}

}  // namespace dspark
