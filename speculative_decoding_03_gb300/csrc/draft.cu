// The draft of one step (all gamma positions) in one persistent, warp-specialised kernel,
// with the Markov bias contraction laid out request-major in tensor memory.
//
// billytse.dev DSpark page, sections 3.2 and 3.3: for k = 1..gamma, in order,
//   bias = W1[x_{k-1}] W2;  z = U_k + bias;  x_k ~ softmax(z)   (x_0 = the anchor)
// for every request at once.  x_k is drawn by Gumbel-max: argmax_v z_v - log E_v with
// E_v = -log u_v (stream 0), i.e. argmax_v exp(z_v - M) / E_v for any reference M.  The
// greedy variant (section 11: the serving example drafts greedily) takes x_k = argmax_v z_v
// (ties to the smallest v) and q_k(x_k) = 1, the proposal being the point mass at x_k.
//
// Layout of the work.  The vocabulary is cut into 128-column tiles and the batch into
// chunks of NBJ requests (NBJ = 32, 64 or 128); a position's work is chunks x tiles units,
// and each CTA (one per SM, cooperative launch) owns the same contiguous run of units at
// every position: a run of tiles of one chunk, or the end of one chunk and the start of
// the next, so that large batches with small vocabularies still give every CTA many
// tiles per position.  A job is one position k and one chunk the CTA holds units of.  Per
// job and tile the tensor core computes D[m][n] = sum_i A[m][i] B[i][n] with M = 128,
// N = 128, K = r:
//   A  the E rows W1[x_{k-1}] of the chunk, in tensor memory: row m on lane m, two bf16
//      per 32-bit column.  A chunk of NBJ < 128 requests is repeated 128 / NBJ times down
//      the lanes, so that every warp quadrant (a warp reads only the 32 lanes of its
//      quadrant) holds the rows it samples;
//   B  the W2 tile, streamed through a shared-memory ring as the packed images of pack.cu
//      (MN-major, 128-byte swizzle), or as two TMA boxes per stage from W2 itself.
// A request's accumulator row is one tensor-memory lane with the vocabulary along the
// columns, so a sampler thread owns one request and a run of 16, 32 or 64 columns of every
// tile: tcgen05.ld brings the bias, the U tile comes from a TMA ring (128-byte
// swizzle, so that the threads of a warp, 32 requests, read it without bank conflicts),
// and the request's softmax sums and Gumbel race stay in the thread's registers.  Tensor
// memory holds one A buffer and three accumulators when a position is one job (up to 64
// requests), two of each for 128-request chunks.
//
// Roles (12 warps): warps 0..7 sample (warp w reads the lanes of quadrant w % 4), warp 8
// lane 0 streams W2 stages, warp 9 lane 0 streams U tiles (TMA), warp 10 scores the
// confidence head (when asked), warp 11 allocates tensor memory and its lane 0 issues the
// MMAs.  The producers do not depend on the drafted tokens and run ahead across positions.
//
// Sampler, per thread and pair of octets (16 columns): z = bias + U; running max; the
// softmax sum against a lazy per-thread reference M (raised only when a logit exceeds it by
// more than 32, so exp(z - M) cannot overflow); four Philox blocks give the 16 draws; with
// w = 1 - u (exact), w <= E = -log1p(-w) <= w / (1 - w), so exp(z - M) / w bounds an
// element's ratio exp(z - M) / E from above and exp(z - M)(1 - w) / w from below: an
// element is a candidate only if its upper bound beats exp(best - M), where best is the
// best exact score any thread of the CTA has found for the request (a 64-bit shared-memory
// atomic max, tagged with the job so that no reset is needed; for chunks of 64 or more
// requests also the best any CTA has published in the request's argmax key); a thread with
// many candidates tightens the threshold with their best lower bound, and only the
// survivors evaluate the exact score z - log E: E with log1p, log E with the fast logarithm
// (within 3 ulp, under 6e-6 absolute for every E a 23-bit draw gives: inside the 1e-5 band
// in which the draft may pick another of two near-equal scores than the fp64 reference).
//
// After its last tile of a job, every sampler thread leaves its partial (max, sum, best
// score, index, logit) in shared memory; the sampler threads merge them with a shuffle tree
// per request, publish the CTA's partial and fold the CTA's best (score, index) into a
// 64-bit atomic max key.  One grid barrier per position (a release reduction per CTA, one
// bounded poller) makes x_k known everywhere; the samplers then gather the next position's
// E rows into an A buffer with tcgen05.st.  The CTA with index b mod G
// then merges the partials of request b (from the CTAs that hold its chunk) into x_k,
// q_k(x_k), max and sum while the tensor core computes the next position's first tile.
//
// Failure handling: every wait is bounded (LParams::wait_cycles SM cycles).  A wait that
// runs out records DSPARK_ERR_TIMEOUT and sets a CTA-wide abort flag; from then on the
// sampler threads run their fixed loop counts without waiting or working (so that their
// named barriers line up), the producers and the MMA issuer stop issuing and drain what
// they issued, and the CTA releases tensor memory and exits.
#include <string.h>

#include "internal.h"
#include "schedule_block.cuh"
#include "sm100_ptx.cuh"

namespace dspark {
namespace {

using namespace sm100;

// Eight sampler warps (two per sub-partition, so that the MMA lane's sub-partition has
// issue slots to spare) that each take 2, 4 or 8 octets of a tile: warps 0..7, sampler w
// sits in quadrant w % 4; warp 8 streams W2, warp 9 streams U, warp 11 (the sub-partition
// of samplers 3 and 7) issues the MMAs; warp 10 scores the confidence head.
constexpr int kSamplers = 8;
constexpr int kWProducerWarp = 8;
constexpr int kUProducerWarp = 9;
constexpr int kConfWarp = 10;
constexpr int kMmaWarp = 11;
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kSamplerThreads = kSamplers * 32;
constexpr int kBarSamplers = 1;       // named barrier of the sampler threads
constexpr int kConfSlots = 512;       // requests per CTA whose survival it keeps
constexpr uint32_t kTmemCols = 512;   // 128-column A buffers, then 128-column accumulators
constexpr int kTileN = 128;           // vocabulary columns per tile (MMA N)
constexpr int kWStageBytes = 16384;   // one K-chunk of up to 64 rank rows of a W2 tile
constexpr int kMergeStride = 5 * 32 + 1;    // words per sampler warp in the merge area (the pad
                                            // spreads a merging warp's reads over the banks)
constexpr float kLazy = 32.f;               // reference raise margin (exp(32) fits fp32 sums)
constexpr float kShrink = 1.f - 0x1.0p-16f;  // filter slack, well above fp32 rounding

// Shared-memory plan of one NBJ (requests per job).
template <int NBJ>
struct LSmem {
  static constexpr int kCopies = 128 / NBJ;          // replicas of the chunk down the lanes
  // columns of a tile per sampler thread: 128 over the kSamplers / 4 * kCopies warps
  // that hold the same rows
  static constexpr int kCols = 4 * NBJ / kSamplers;
  static constexpr int kOct = kCols / 8;             // octets per tile per sampler thread
  static constexpr int kWStages = NBJ == 32 ? 8 : NBJ == 64 ? 6 : 4;
  static constexpr int kUStages = NBJ == 32 ? 3 : NBJ == 64 ? 3 : 2;
  static constexpr int kUStageBytes = NBJ * kTileN * 4;
  // Tensor memory: up to 64 requests make one job per position, whose E rows are gathered
  // only after the grid barrier (one A buffer; three accumulators keep the tensor core and
  // the samplers apart); 128-request chunks gather the next chunk during the current one
  // (two A buffers, two accumulators).
  static constexpr int kABufs = NBJ == 128 ? 2 : 1;
  static constexpr int kAccBufs = 4 - kABufs;
  static constexpr uint32_t kAccCol = 128u * kABufs;
  static constexpr int kOffW = 0;
  static constexpr int kOffU = kOffW + kWStages * kWStageBytes;
  static constexpr int kOffMerge = kOffU + kUStages * kUStageBytes;   // [16 warps][5][32] + pad
  static constexpr int kMergeBytes = kSamplers * kMergeStride * 4;
  static constexpr int kOffThr = kOffMerge + kMergeBytes;             // [NBJ] u64
  // 32 requests: the E rows staged in shared memory, one copy (16-byte chunk c of row i at
  // i * 512 + (c ^ (i % 8)) * 16), from which every warp stores its quadrant's copy into
  // tensor memory; larger chunks store their rows from global memory directly
  static constexpr int kOffA = (kOffThr + NBJ * 8 + 1023) / 1024 * 1024;
  static constexpr int kABytes = NBJ == 32 ? 32 * 512 : 0;
  static constexpr int kBytes = kOffA + kABytes;
};

struct LParams {
  const uint16_t* W1;
  const uint16_t* W2p;             // packed W2 tile images (null: TMA boxes from W2)
  const int32_t* anchor;
  int B, gamma, V, r;
  int n_tiles, n_chunks, kc;       // kc = rank rows per W2 stage (<= 64)
  uint64_t seed;
  PhiloxKeys philox;               // the generator's round keys for this seed
  RowState* partials;              // [3][B][G], position k in slot k % 3
  unsigned long long* keys;        // [gamma][B], zeroed before launch
  unsigned int* grid_count;        // zeroed before launch
  unsigned int* conf_count;        // (the next word) CTAs whose survivals are all written
  unsigned int* rank_count;        // (the word after) idle CTAs that ranked their items
  int32_t* tokens;
  float* q_tok;
  float* row_max;
  float* row_sumexp;
  int* err;
  long long wait_cycles;           // bound of every wait
  unsigned int grid_extra;         // added to every grid-barrier target (0; tests: unreachable)
  // the confidence head and survival, computed by the confidence warp (c_out null: not
  // computed here)
  const float* h;                  // [B][gamma][H]
  const float* w_c;                // [H + r]
  float b_c;
  int H;
  float* c_out;                    // [B][gamma]
  float* a_out;                    // [B][gamma]
  // the prefix scheduler, run after the last position (ell null: not run here): by CTA 0
  // alone when sched_keys is null, else every CTA ranks a share of the items and CTA 0
  // scans them in the order they give (sched_keys: the sorted keys, B gamma words)
  const float* sps;
  int32_t* ell;
  int32_t* B_total;
  double* theta;
  unsigned long long* sched_keys;
  // B gamma <= kThreads on a grid of more than B CTAs: the confidence warps of the CTAs
  // that hold no request rank the scheduler's items while the last position is drawn, and
  // the last CTA's scans them (sched_keys: the ranked keys)
  int sched_warp;
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta_shared_u32(unsigned int* p, unsigned int v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_cta_shared_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_volatile_shared_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.volatile.shared.u64 %0, [%1];" : "=l"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void atomic_max_shared_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("atom.shared.max.u64 _, [%0], %1;" ::"r"(smem_u32(p)), "l"(v) : "memory");
}

// Order-preserving map of a (non-NaN) float to a 32-bit unsigned key and back.
__device__ __forceinline__ uint32_t float_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

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

__device__ __forceinline__ int token_of_key(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

// The work of a position is n_chunks x n_tiles units (one chunk of NBJ requests on one
// 128-column vocabulary tile, chunk-major); CTA g owns units [g U / G, (g + 1) U / G) of
// every position: a run of tiles of one chunk, or of the end of one chunk and the start
// of the next ones.  A job is one position and one chunk that the CTA holds units of, with
// the CTA's tile range in that chunk.  (One chunk: the CTA's tiles are the same for every
// job.)
// The launch keeps U G below 2^32, so these products and quotients are 32-bit (64-bit
// division here cost the single-chunk draft 3 % in code size).
struct JobMap {
  int u_lo, u_hi, c_first, jpp, n_tiles;   // jpp: jobs per position
  __device__ __forceinline__ JobMap(int cta, int G, int n_chunks, int n_tiles_)
      : n_tiles(n_tiles_) {
    const unsigned U = (unsigned)n_chunks * (unsigned)n_tiles_;
    u_lo = (int)((unsigned)cta * U / (unsigned)G);
    u_hi = (int)((unsigned)(cta + 1) * U / (unsigned)G);
    c_first = u_lo / n_tiles_;
    jpp = (u_hi - 1) / n_tiles_ - c_first + 1;
  }
  __device__ __forceinline__ int k(int j) const { return jpp == 1 ? j + 1 : j / jpp + 1; }
  __device__ __forceinline__ int c(int j) const { return jpp == 1 ? c_first : c_first + j % jpp; }
  __device__ __forceinline__ int t_begin(int j) const {
    const int a = u_lo - c(j) * n_tiles;
    return a > 0 ? a : 0;
  }
  __device__ __forceinline__ int t_end(int j) const {
    const int e = u_hi - c(j) * n_tiles;
    return e < n_tiles ? e : n_tiles;
  }
  __device__ __forceinline__ bool last_of_position(int j) const {
    return jpp == 1 || j % jpp == jpp - 1;
  }
};
// The CTAs that hold units of chunk c (and so publish partials of its requests) are
// [first, last]: the owners of the chunk's first and last unit, unit u being owned by CTA
// ((u + 1) G - 1) / U.
__device__ __forceinline__ int2 chunk_holders(int G, int c, int n_chunks, int n_tiles) {
  if (n_chunks == 1) return make_int2(0, G - 1);
  const unsigned U = (unsigned)n_chunks * (unsigned)n_tiles, u0 = (unsigned)c * (unsigned)n_tiles;
  return make_int2((int)(((u0 + 1u) * (unsigned)G - 1u) / U),
                   (int)(((u0 + (unsigned)n_tiles) * (unsigned)G - 1u) / U));
}

// Merge the partials of request b (chunk c) at position kp from the CTAs that hold its
// chunk into x, q, max and sum (one warp; every lane issues all its loads together, so a
// merge is about one L2 round trip).
constexpr int kMergePerLane = (kDraftMaxCtas + 31) / 32;
template <bool Greedy>
__device__ __forceinline__ void finalize_row(const LParams& p, int b, int c, int kp, int G, int lane) {
  const unsigned long long key = __ldcg(p.keys + (size_t)(kp - 1) * p.B + b);
  const RowState* base = p.partials + ((size_t)(kp % 3) * p.B + b) * G;
  const int2 hold = chunk_holders(G, c, p.n_chunks, p.n_tiles);
  float pm[kMergePerLane], ps[kMergePerLane], pz[kMergePerLane];
  int pi[kMergePerLane];
#pragma unroll
  for (int u = 0; u < kMergePerLane; ++u) {
    const int g = lane + 32 * u;
    pm[u] = -INFINITY; ps[u] = 0.f; pz[u] = -INFINITY; pi[u] = -1;
    if (g >= hold.x && g <= hold.y) {
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
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f, zx = -INFINITY;
#pragma unroll
  for (int u = 0; u < kMergePerLane; ++u) {
    if (pm[u] != -INFINITY) s += ps[u] * expf(pm[u] - m);
    if (pi[u] == x) zx = pz[u];
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    zx = fmaxf(zx, __shfl_xor_sync(0xffffffffu, zx, o));
  }
  if (lane == 0) {
    const size_t o = (size_t)b * p.gamma + (kp - 1);
    p.tokens[o] = x;
    p.q_tok[o] = Greedy ? 1.f : expf(zx - m) / s;
    p.row_max[o] = m;
    p.row_sumexp[o] = s;
  }
}

// One warp's share of the scheduler's ranking (N = R gamma <= kThreads items): the keys of
// all N items in shared memory (keys), then, for each item of share w of W, the number of
// keys below it (counted over the lanes) as its rank: sched_keys[rank] = its key.
__device__ __noinline__ void warp_rank_share(const float* a, int R, int gamma, int w, int W,
                                             unsigned long long* keys,
                                             unsigned long long* sched_keys) {
  const int lane = threadIdx.x & 31;
  const int N = R * gamma;
  for (int i = lane; i < N; i += 32) {
    const int r = i / gamma, j = i - r * gamma;
    keys[i] = schedule_key(__ldcg(a + i), r, j);
  }
  __syncwarp();
  const int i0 = (int)((long long)w * N / W), i1 = (int)((long long)(w + 1) * N / W);
  for (int it = i0; it < i1; ++it) {
    const unsigned long long mine = keys[it];
    int cnt = 0;
    for (int j = lane; j < N; j += 32) cnt += keys[j] < mine ? 1 : 0;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, d);
    if (lane == 0) sched_keys[cnt] = mine;
  }
  __syncwarp();
}

// The scheduler's scan on one warp over the N = R gamma <= kThreads keys in ascending order
// (keys, shared memory): the exact sums and Theta test of schedule_block (the same first
// non-rise), lane L scanning the contiguous items [L per, (L + 1) per); cnt: R words of
// shared memory for the per-request counts.
__device__ __noinline__ void warp_scan_schedule(int R, int gamma, const float* sps, int32_t* ell,
                                                int32_t* B_total, double* theta,
                                                const unsigned long long* keys, int* cnt) {
  const int lane = threadIdx.x & 31;
  const int N = R * gamma;
  for (int r = lane; r < R; r += 32) cnt[r] = 0;
  auto A_of = [&](int n) { return 4294967296LL - (long long)(keys[n] >> 21); };
  const int per = (N + 31) / 32;
  const int c0 = min(N, lane * per), c1 = min(N, c0 + per);
  long long local = 0;
  for (int i = c0; i < c1; ++i) local += A_of(i);
  long long incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += t;
  }
  long long S = incl - local;
  int fail = N + 1;
  if (c0 < c1) {
    double th_prev = theta_at(R, S, sps[R + c0]);
    for (int i = c0; i < c1; ++i) {
      S += A_of(i);
      const double th = theta_at(R, S, sps[R + i + 1]);
      if (!(th > th_prev)) {
        fail = i + 1;
        break;
      }
      th_prev = th;
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) fail = min(fail, __shfl_xor_sync(0xffffffffu, fail, d));
  const int admitted = fail - 1;
  __syncwarp();
  for (int i = lane; i < admitted; i += 32) atomicAdd(&cnt[(int)((keys[i] >> 5) & 0xFFFFull)], 1);
  __syncwarp();
  for (int r = lane; r < R; r += 32) ell[r] = cnt[r];
  if (admitted == 0) {
    if (lane == 0) {
      *B_total = R;
      *theta = theta_at(R, 0, sps[R]) / 4294967296.0;
    }
  } else if (admitted - 1 >= c0 && admitted - 1 < c1) {
    long long Sa = incl - local;
    for (int i = c0; i < admitted; ++i) Sa += A_of(i);
    *B_total = R + admitted;
    *theta = theta_at(R, Sa, sps[R + admitted]) / 4294967296.0;
  }
}

// The scheduler's items ranked by the whole grid (up to kGridScheduleItems of them): every
// CTA builds all N keys (the scheduler's order, distinct) in shared memory and counts, for
// each item of its share [cta N / G, (cta + 1) N / G), the keys below it, the count split
// over kThreads / share threads (a share of at most kThreads items); the item's key goes
// to sched_keys[rank].  rank_s: kThreads words of shared memory.
__device__ __noinline__ void schedule_ranks(const float* a, int N, int gamma,
                                            unsigned long long* sched_keys,
                                            unsigned long long* keys, int* rank_s, int G,
                                            int cta) {
  const int tid = threadIdx.x;
  for (int i = tid; i < N; i += kThreads) {
    const int r = i / gamma, j = i - r * gamma;
    keys[i] = schedule_key(__ldcg(a + i), r, j);
  }
  rank_s[tid] = 0;
  __syncthreads();
  const int i0 = (int)((long long)cta * N / G), i1 = (int)((long long)(cta + 1) * N / G);
  const int m = i1 - i0;
  if (m > 0 && m <= kThreads) {
    const int P = kThreads / m;                   // threads per item
    const int k = tid / P, sp = tid - k * P;
    if (k < m) {
      const unsigned long long mine = keys[i0 + k];
      const int j0 = (int)((long long)sp * N / P), j1 = (int)((long long)(sp + 1) * N / P);
      int cnt = 0;
      for (int jj = j0; jj < j1; ++jj) cnt += keys[jj] < mine ? 1 : 0;
      atomicAdd(&rank_s[k], cnt);
    }
    __syncthreads();
    if (tid < m) sched_keys[rank_s[tid]] = keys[i0 + tid];
  } else if (m > kThreads) {
    // (a grid of fewer than N / kThreads CTAs: whole items per thread)
    for (int k = tid; k < m; k += kThreads) {
      const unsigned long long mine = keys[i0 + k];
      int cnt = 0;
      for (int jj = 0; jj < N; ++jj) cnt += keys[jj] < mine ? 1 : 0;
      sched_keys[cnt] = mine;
    }
  }
  __syncthreads();                                // the ranks are stored before the arrival
}

template <int NBJ, bool Greedy>
__global__ void __launch_bounds__(kThreads, 1) draft_lanes_kernel(
    const __grid_constant__ CUtensorMap w2_map, const __grid_constant__ CUtensorMap u_map,
    const LParams p) {
  using S = LSmem<NBJ>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t w_full[S::kWStages], w_empty[S::kWStages];
  __shared__ uint64_t u_full[S::kUStages], u_empty[S::kUStages];
  __shared__ uint64_t a_full[S::kABufs], a_empty[S::kABufs];
  __shared__ uint64_t acc_full[S::kAccBufs], acc_empty[S::kAccBufs];
  __shared__ uint64_t mma_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ float surv_s[kConfSlots];   // a_{k-1} of this CTA's requests
  __shared__ float hdot_s[kConfSlots];   // h_k . w_c[0:H] of the same
  __shared__ int conf_done_s;
  __shared__ unsigned long long sched_warp_keys[kThreads];   // the scheduling warp's keys
  __shared__ unsigned int grid_seen_s;   // the barrier count the samplers' poller last saw

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const JobMap jm(cta, G, p.n_chunks, p.n_tiles);
  const int kc = p.kc;
  const int n_kchunks = p.r / kc;
  const int n_jobs = p.gamma * jm.jpp;
  unsigned long long* thr = reinterpret_cast<unsigned long long*>(smem + S::kOffThr);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S::kWStages; ++i) { mbar_init(&w_full[i], 1); mbar_init(&w_empty[i], 1); }
    for (int i = 0; i < S::kUStages; ++i) {
      mbar_init(&u_full[i], 1);
      mbar_init(&u_empty[i], kSamplers);
    }
    for (int i = 0; i < S::kABufs; ++i) {
      mbar_init(&a_full[i], kSamplers);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < S::kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kSamplers);
    }
    mbar_init(&mma_drain, 1);
    abort_s = 0;
    conf_done_s = 0;
    grid_seen_s = 0u;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < NBJ; i += kThreads) thr[i] = 0ull;   // below every tagged key
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_s, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_base_s;
  pdl_launch_dependents();

  // One thread's bounded wait; a timeout aborts the CTA.  A completed phase is seen by a
  // non-blocking test; the abort flag is read only once the first (sleeping) try has not
  // seen the phase complete, so the issue loops pay nothing for it.
  auto wait1 = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_test_wait(bar, parity) || mbar_try_wait_sleep(bar, parity)) return true;
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

  if (warp == kWProducerWarp) {
    // ---------------------------------------------------------------- W2 stage producer
    if (lane == 0) {
      if (!p.W2p) prefetch_tensormap(&w2_map);
      const uint64_t keep = policy_evict_last();
      const uint32_t w_bytes = 2u * (uint32_t)kc * 128u;
      uint32_t ws = 0;
      bool ok = true;
      for (int job = 0; job < n_jobs && ok; ++job) {
        const int t_end = jm.t_end(job);
        for (int t = jm.t_begin(job); t < t_end && ok; ++t) {
          for (int i = 0; i < n_kchunks; ++i, ++ws) {
            const int s = ws % S::kWStages;
            if (!(ok = wait1(&w_empty[s], ((ws / S::kWStages) & 1) ^ 1))) break;
            uint8_t* dst = smem + S::kOffW + s * kWStageBytes;
            mbar_arrive_expect_tx(&w_full[s], w_bytes);
            if (p.W2p) {
              const uint16_t* src = p.W2p + ((size_t)t * n_kchunks + i) * (size_t)kc * 128;
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                  " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
                  "l"(reinterpret_cast<uint64_t>(src)), "r"(w_bytes), "r"(smem_u32(&w_full[s])),
                  "l"(keep)
                  : "memory");
            } else {
              tma_load_2d(dst, &w2_map, &w_full[s], t * kTileN, i * kc, keep);
              tma_load_2d(dst + kc * 128, &w2_map, &w_full[s], t * kTileN + 64, i * kc, keep);
            }
          }
        }
      }
      // every issued copy lands before the CTA may exit (a stage whose wait failed was
      // never issued, so only the stages below ws can be in flight)
      for (uint32_t i = ws > (uint32_t)S::kWStages ? ws - S::kWStages : 0; i < ws; ++i)
        mbar_wait(&w_full[i % S::kWStages], (i / S::kWStages) & 1);
    }
    __syncwarp();
  } else if (warp == kUProducerWarp) {
    // ------------------------------------------------------------------ U tile producer
    if (lane == 0) {
      prefetch_tensormap(&u_map);
      uint64_t stream_pol;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream_pol));
      uint32_t us = 0;
      bool ok = true;
      for (int job = 0; job < n_jobs && ok; ++job) {
        const int k = jm.k(job), c = jm.c(job), t_end = jm.t_end(job);
        for (int t = jm.t_begin(job); t < t_end; ++t, ++us) {
          const int su = us % S::kUStages;
          if (!(ok = wait1(&u_empty[su], ((us / S::kUStages) & 1) ^ 1))) break;
          mbar_arrive_expect_tx(&u_full[su], (uint32_t)S::kUStageBytes);
          // four boxes of 32 columns x NBJ requests (128 bytes a row: the swizzle's span)
#pragma unroll
          for (int jb = 0; jb < 4; ++jb)
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(
                    smem_u32(smem + S::kOffU + su * S::kUStageBytes + jb * NBJ * 128)),
                "l"(reinterpret_cast<uint64_t>(&u_map)), "r"(smem_u32(&u_full[su])),
                "r"(t * kTileN + 32 * jb), "r"(k - 1), "r"(c * NBJ), "l"(stream_pol)
                : "memory");
        }
      }
      for (uint32_t i = us > (uint32_t)S::kUStages ? us - S::kUStages : 0; i < us; ++i)
        mbar_wait(&u_full[i % S::kUStages], (i / S::kUStages) & 1);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // -------------------------------------------------------------------- MMA issuer
    // The K steps of one W2 stage are a compile-time count (1, 2 or 4); descriptors are
    // built once and advanced by adding (byte offset >> 4) to their start-address field.
    // The issuing lane shares its sub-partition with four busy sampler warps, so every
    // instruction of this loop costs several issue slots: a tile's MMAs are unrolled with
    // compile-time K steps per stage (KS) and stages per tile (NKC, 0: a runtime count),
    // descriptors are advanced by adds to their start-address field (every operand lies
    // below 256 KB, so the sum never carries into the stride fields), and the waits spin
    // on test_wait (one spinning lane costs the others little) for 32-request jobs, whose
    // hand-offs are short, and suspend for larger ones.
    auto spin_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (mbar_test_wait(bar, parity)) return true;
      const long long t0 = sm_cycles();
      for (;;) {
        if (NBJ >= 64 ? mbar_try_wait_sleep(bar, parity) : mbar_test_wait(bar, parity)) return true;
        if (*(volatile int*)&abort_s) return false;
        if (sm_cycles() - t0 > p.wait_cycles) {
          set_device_error(p.err, DSPARK_ERR_TIMEOUT);
          atomicExch(&abort_s, 1);
          return false;
        }
      }
    };
    auto issue_loop = [&](auto ksteps_c, auto nkc_c) {
      constexpr int KS = decltype(ksteps_c)::value;
      constexpr int NKC = decltype(nkc_c)::value;
      constexpr int WS = S::kWStages;
      const int nkc = NKC > 0 ? NKC : n_kchunks;
      const uint32_t idesc = idesc_bf16_f32(128, kTileN, 0, 1);
      const uint64_t b_base = smem_desc(smem_u32(smem + S::kOffW), (uint32_t)KS * 2048u, 1024u,
                                        kSwizzle128B);
      uint32_t ws = 0, tc = 0;
      bool ok = true;
      for (int job = 0; job < n_jobs && ok; ++job) {
        const int ab = job % S::kABufs;
        if (!(ok = wait1(&a_full[ab], (job / S::kABufs) & 1))) break;
        tc_fence_after_sync();
        const uint32_t a_t = tmem_base + (uint32_t)(128 * ab);
        const int n_t = jm.t_end(job) - jm.t_begin(job);
        for (int t = 0; t < n_t && ok; ++t, ++tc) {
          const int acc = tc % S::kAccBufs;
          if (!(ok = spin_wait(&acc_empty[acc], ((tc / S::kAccBufs) & 1) ^ 1))) break;
          tc_fence_after_sync();
          const uint32_t d_t = tmem_base + S::kAccCol + (uint32_t)(kTileN * acc);
          auto chunk = [&](int i) {
            uint32_t st = ws % WS;
            const uint32_t par = (ws / WS) & 1u;
            ++ws;
            if (!ok || !(ok = spin_wait(&w_full[st], par))) return;
            // K step g of A is columns 8g .. 8g + 7; 16 K rows of the MN-major stage are
            // 2048 bytes apart
            const uint64_t b_s = b_base + (uint64_t)(st * (kWStageBytes >> 4));
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
              umma_ts_bf16_f32(d_t, a_t + 8u * (uint32_t)(i * KS + kk),
                               b_s + (uint64_t)(kk * (2048 >> 4)), idesc,
                               (i > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&w_empty[st]);
          };
          if constexpr (NKC > 0) {
#pragma unroll
            for (int i = 0; i < NKC; ++i) chunk(i);
          } else {
            for (int i = 0; i < nkc; ++i) chunk(i);
          }
          if (!ok) break;
          umma_commit(&acc_full[acc]);
        }
        if (ok) umma_commit(&a_empty[ab]);
      }
    };
    if (lane == 0) {
      using std::integral_constant;
      if (kc == 64 && n_kchunks == 4) issue_loop(integral_constant<int, 4>{}, integral_constant<int, 4>{});
      else if (kc == 64 && n_kchunks == 2) issue_loop(integral_constant<int, 4>{}, integral_constant<int, 2>{});
      else if (kc == 64 && n_kchunks == 1) issue_loop(integral_constant<int, 4>{}, integral_constant<int, 1>{});
      else if (kc == 64) issue_loop(integral_constant<int, 4>{}, integral_constant<int, 0>{});
      else if (kc == 32) issue_loop(integral_constant<int, 2>{}, integral_constant<int, 0>{});
      else issue_loop(integral_constant<int, 1>{}, integral_constant<int, 0>{});
      // every issued MMA completes before tensor memory is released
      umma_commit(&mma_drain);
      mbar_wait(&mma_drain, 0);
    }
    __syncwarp();
  } else if (warp == kConfWarp) {
    // ---------------------------------------------------------------- confidence head
    // Position k of this CTA's requests b = cta + i G (slot i): weigao.cc DSpark-vs-MTP
    // page, "3. confidence head" (one linear layer on [h_k ; W1[x_{k-1}]], a sigmoid) and
    // billytse.dev section 5 (a_k = a_{k-1} c_k, multiplied left to right).  The h_k part
    // of the logit needs no draft: it is summed while the samplers draw position k - 1;
    // the W1[x_{k-1}] part follows once every CTA has published position k - 1.  One warp
    // per request, lanes across the features.
    if (p.c_out) {
      const int H4 = p.H >> 2;
      const float4* wv = reinterpret_cast<const float4*>(p.w_c);
      bool ok = true;
      // (a CTA holds requests cta, cta + G, ..: none when cta >= B)
      for (int k = 1; k <= p.gamma && ok && cta < p.B; ++k) {
        int i = 0;
        for (int bb = cta; bb < p.B; bb += G, ++i) {
          const float4* hv = reinterpret_cast<const float4*>(p.h + ((size_t)bb * p.gamma + (k - 1)) * p.H);
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int q0 = lane; q0 < H4; q0 += 128) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int q = q0 + 32 * j;
              if (q < H4) {
                const float4 x = __ldcs(hv + q), w = __ldg(wv + q);
                acc[j] = fmaf(x.x, w.x, acc[j]);
                acc[j] = fmaf(x.y, w.y, acc[j]);
                acc[j] = fmaf(x.z, w.z, acc[j]);
                acc[j] = fmaf(x.w, w.w, acc[j]);
              }
            }
          }
          float d = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
          for (int m = 16; m >= 1; m >>= 1) d += __shfl_xor_sync(0xffffffffu, d, m);
          if (lane == 0) hdot_s[i] = d;
        }
        if (k >= 2) {
          // x_{k-1} is final once every CTA has arrived for position k - 1, which the
          // samplers' poller publishes in shared memory (a bounded, sleeping poll: this warp
          // is off the samplers' critical path, and polling the grid counter itself would
          // add a poller per CTA on its line)
          if (lane == 0) {
            const unsigned int target = (unsigned int)G * (unsigned int)(k - 1) + p.grid_extra;
            const long long t0 = sm_cycles();
            while (ld_acquire_cta_shared_u32(&grid_seen_s) < target) {
              if (*(volatile int*)&abort_s) { ok = false; break; }
              if (sm_cycles() - t0 > p.wait_cycles) {
                set_device_error(p.err, DSPARK_ERR_TIMEOUT);
                atomicExch(&abort_s, 1);
                ok = false;
                break;
              }
              __nanosleep(256);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
        i = 0;
        for (int bb = cta; bb < p.B; bb += G, ++i) {
          int prev = (k == 1) ? p.anchor[bb] : token_of_key(__ldcg(p.keys + (size_t)(k - 2) * p.B + bb));
          if (!(prev >= 0 && prev < p.V)) {
            if (lane == 0) set_device_error(p.err, DSPARK_ERR_DEVICE_CHECK);
            prev = 0;
          }
          const uint16_t* e = p.W1 + (size_t)prev * p.r;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int q = 8 * lane; q < p.r; q += 256) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(e + q));
            const float4 w0 = __ldg(reinterpret_cast<const float4*>(p.w_c + p.H + q));
            const float4 w1 = __ldg(reinterpret_cast<const float4*>(p.w_c + p.H + q + 4));
            acc[0] = fmaf(__uint_as_float(u.x << 16), w0.x, acc[0]);
            acc[1] = fmaf(__uint_as_float(u.x & 0xFFFF0000u), w0.y, acc[1]);
            acc[2] = fmaf(__uint_as_float(u.y << 16), w0.z, acc[2]);
            acc[3] = fmaf(__uint_as_float(u.y & 0xFFFF0000u), w0.w, acc[3]);
            acc[0] = fmaf(__uint_as_float(u.z << 16), w1.x, acc[0]);
            acc[1] = fmaf(__uint_as_float(u.z & 0xFFFF0000u), w1.y, acc[1]);
            acc[2] = fmaf(__uint_as_float(u.w << 16), w1.z, acc[2]);
            acc[3] = fmaf(__uint_as_float(u.w & 0xFFFF0000u), w1.w, acc[3]);
          }
          float d = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
          for (int m = 16; m >= 1; m >>= 1) d += __shfl_xor_sync(0xffffffffu, d, m);
          if (lane == 0) {
            const float c = 1.f / (1.f + expf(-(hdot_s[i] + d + p.b_c)));
            const float a = (k == 1 ? 1.f : surv_s[i]) * c;
            surv_s[i] = a;
            const size_t o = (size_t)bb * p.gamma + (k - 1);
            p.c_out[o] = c;
            p.a_out[o] = a;
          }
        }
      }
      // c and a are ordered before the flag the samplers wait for ahead of their last
      // grid arrival (and, for the scheduling warp, before this CTA's count)
      __threadfence();
      __syncwarp();
      if (lane == 0) *(volatile int*)&conf_done_s = 1;
      if (p.sched_warp && cta < p.B && ok && lane == 0)
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.conf_count) : "memory");
      if (p.sched_warp && cta >= p.B) {
        // A CTA without requests: once every requesting CTA has written its survivals, rank
        // a share of the scheduler's items; the last CTA then scans them all
        auto wait_count = [&](const unsigned int* cnt, unsigned int target) -> bool {
          bool go = true;
          if (lane == 0) {
            const long long t0 = sm_cycles();
            while (ld_acquire_u32(cnt) < target) {
              if (*(volatile int*)&abort_s || sm_cycles() - t0 > p.wait_cycles) {
                if (!*(volatile int*)&abort_s) {
                  set_device_error(p.err, DSPARK_ERR_TIMEOUT);
                  atomicExch(&abort_s, 1);
                }
                go = false;
                break;
              }
              __nanosleep(128);
            }
          }
          __syncwarp();   // the other lanes' reads follow lane 0's acquire
          return __shfl_sync(0xffffffffu, go, 0);
        };
        const int W = G - p.B;
        if (wait_count(p.conf_count, (unsigned int)p.B)) {
          warp_rank_share(p.a_out, p.B, p.gamma, cta - p.B, W, sched_warp_keys, p.sched_keys);
          if (lane == 0)
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.rank_count) : "memory");
          if (cta == G - 1 && wait_count(p.rank_count, (unsigned int)W)) {
            const int N = p.B * p.gamma;
            for (int i = lane; i < N; i += 32) sched_warp_keys[i] = __ldcg(p.sched_keys + i);
            __syncwarp();
            warp_scan_schedule(p.B, p.gamma, p.sps, p.ell, p.B_total, p.theta, sched_warp_keys,
                               reinterpret_cast<int*>(hdot_s));
          }
        }
      }
    }
  } else if (warp < kSamplers) {
    // ----------------------------------------------------------------------- samplers
    const int sw = warp;
    const int stid = threadIdx.x;
    const int quad = warp & 3;                                  // TMEM lane quadrant
    const int ml = (32 * quad + lane) % NBJ;                    // request row in the chunk
    // column run of this warp: the warps whose quadrants hold the same rows split a tile
    // (kSamplers / 4 warps per quadrant, kCopies quadrants per row set)
    const int sidx = (sw >> 2) * S::kCopies + quad / (NBJ / 32);
    const int c0 = sidx * S::kCols;
    const uint32_t lane_base = tmem_base + ((uint32_t)(32 * quad) << 16);
    float* merge = reinterpret_cast<float*>(smem + S::kOffMerge);
    // U tile address of this thread's first column: box c0 / 32, row ml, 16-byte chunk
    // (c0 % 32) / 4 (two chunks per octet), 128-byte swizzle (chunk ^ row % 8)
    const int u_row = ml * 128;
    const int u_sw = ml & 7;

    // a whole warp's bounded wait (abort first: after an abort nothing waits)
    auto swait = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (*(volatile int*)&abort_s) return false;
      return __all_sync(0xffffffffu, wait1(bar, parity));
    };
    auto grid_wait = [&](unsigned int target) {
      if (stid == 0 && !*(volatile int*)&abort_s) {
        const long long t0 = sm_cycles();
        unsigned int seen;
        while ((seen = ld_acquire_u32(p.grid_count)) < target) {
          if (*(volatile int*)&abort_s || sm_cycles() - t0 > p.wait_cycles) {
            set_device_error(p.err, DSPARK_ERR_TIMEOUT);
            atomicExch(&abort_s, 1);
            break;
          }
        }
        // this CTA's confidence warp follows the barrier through this word
        if (seen >= target) st_release_cta_shared_u32(&grid_seen_s, seen);
      }
      named_bar_sync(kBarSamplers, kSamplerThreads);
    };
    // E rows of job j into A buffer j % kABufs: this thread's lane holds row 32 quad + lane
    // (request c NBJ + ml), this warp writes columns [jq r / 8, (jq + 1) r / 8) of it
    auto gather = [&](int j) {
      const int k = jm.k(j), c = jm.c(j);
      const int ab = j % S::kABufs;
      if constexpr (NBJ == 32) {
        // One copy of the 32 rows into the staging area (warp w loads 16-byte chunks w,
        // w + 8, ..: all in flight at once), a sampler barrier, then each warp stores its
        // quadrant's copy of its half of the columns from shared memory into the A buffer.
        // Every sampler thread reaches the barrier: an abort or a timeout skips only the
        // tensor-memory stores after it.
        const bool ready = j < S::kABufs || swait(&a_empty[ab], ((j / S::kABufs) & 1) ^ 1);
        int prev = -1;
        if (lane < p.B) {
          prev = (k == 1) ? p.anchor[lane] : token_of_key(__ldcg(p.keys + (size_t)(k - 2) * p.B + lane));
          if (prev < 0 || prev >= p.V) {
            set_device_error(p.err, DSPARK_ERR_DEVICE_CHECK);
            prev = -1;
          }
        }
        const int nch = p.r >> 3;                       // 16-byte chunks of a row
        const uint4* row = reinterpret_cast<const uint4*>(p.W1 + (size_t)(prev < 0 ? 0 : prev) * p.r);
        uint8_t* stage = smem + S::kOffA + lane * 512;
        uint4 v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
          if (sw + 8 * m < nch) v[m] = prev < 0 ? make_uint4(0u, 0u, 0u, 0u) : __ldg(row + sw + 8 * m);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          if (sw + 8 * m < nch)
            *reinterpret_cast<uint4*>(stage + (((sw + 8 * m) ^ (lane & 7)) << 4)) = v[m];
        named_bar_sync(kBarSamplers, kSamplerThreads);
        // warp-uniform: the tensor-memory stores below are whole-warp instructions
        if (!__all_sync(0xffffffffu, ready) || __any_sync(0xffffffffu, *(volatile int*)&abort_s != 0))
          return;
        tc_fence_after_sync();
        // this warp: lanes of quadrant sw % 4 (row = lane), chunks [h0, h0 + nch / 2)
        const int half = nch >> 1, h0 = (sw >> 2) * half;
        const uint32_t taddr = lane_base + (uint32_t)(128 * ab + 4 * h0);
        if ((half & 1) == 0) {
          // two chunks (8 columns) per store
          for (int q = 0; q < half; q += 2) {
            const uint4 x = *reinterpret_cast<const uint4*>(stage + (((h0 + q) ^ (lane & 7)) << 4));
            const uint4 y = *reinterpret_cast<const uint4*>(stage + (((h0 + q + 1) ^ (lane & 7)) << 4));
            const uint32_t cols[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
            tmem_st_32x32b_x8(taddr + 4u * (uint32_t)q, cols);
          }
        } else {
          for (int q = 0; q < half; ++q) {
            const uint4 x = *reinterpret_cast<const uint4*>(stage + (((h0 + q) ^ (lane & 7)) << 4));
            tmem_st_32x32b_x2(taddr + 4u * (uint32_t)q, x.x, x.y);
            tmem_st_32x32b_x2(taddr + 4u * (uint32_t)q + 2u, x.z, x.w);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[ab]);
        return;
      }
      if (j >= S::kABufs && !swait(&a_empty[ab], ((j / S::kABufs) & 1) ^ 1)) return;
      // warp-uniform: the tensor-memory stores below are whole-warp instructions
      if (__any_sync(0xffffffffu, *(volatile int*)&abort_s != 0)) return;
      tc_fence_after_sync();
      const int b = c * NBJ + ml;
      int prev = -1;
      if (b < p.B) {
        prev = (k == 1) ? p.anchor[b] : token_of_key(__ldcg(p.keys + (size_t)(k - 2) * p.B + b));
        if (prev < 0 || prev >= p.V) {
          set_device_error(p.err, DSPARK_ERR_DEVICE_CHECK);
          prev = -1;
        }
      }
      // the kSamplers / 4 warps of a quadrant split the row's r / 2 columns
      constexpr int kPerQuad = kSamplers / 4;
      const int jq = sw >> 2;
      const int ncol = (p.r >> 1) / kPerQuad;         // 32-bit columns per warp
      const uint32_t taddr = lane_base + (uint32_t)(128 * ab + jq * ncol);
      const uint16_t* src = p.W1 + (size_t)(prev < 0 ? 0 : prev) * p.r + (size_t)jq * (2 * ncol);
      if ((ncol & 7) == 0) {
        // 8 columns = 16 bf16 = two 16-byte loads per store.  One chunk of at most 32
        // requests is gathered on the critical path between positions: four stores' loads
        // in flight at a time (two round trips for r = 256; all eight would spill the
        // sampler's registers); chunks of 64 and 128 requests, whose next chunk is gathered
        // while the current one is sampled, keep two stores' loads in flight
        constexpr int kBatch = 2;
        const int n8 = ncol >> 3;                     // 1..8
#pragma unroll
        for (int h = 0; h < 8; h += kBatch) {
          uint4 v[2 * kBatch];
#pragma unroll
          for (int u = 0; u < kBatch; ++u)
            if (h + u < n8) {
              v[2 * u] = prev < 0 ? make_uint4(0u, 0u, 0u, 0u) : __ldg(reinterpret_cast<const uint4*>(src) + 2 * (h + u));
              v[2 * u + 1] = prev < 0 ? make_uint4(0u, 0u, 0u, 0u) : __ldg(reinterpret_cast<const uint4*>(src) + 2 * (h + u) + 1);
            }
#pragma unroll
          for (int u = 0; u < kBatch; ++u)
            if (h + u < n8) {
              const uint32_t cols[8] = {v[2 * u].x, v[2 * u].y, v[2 * u].z, v[2 * u].w,
                                        v[2 * u + 1].x, v[2 * u + 1].y, v[2 * u + 1].z, v[2 * u + 1].w};
              tmem_st_32x32b_x8(taddr + 8u * (h + u), cols);
            }
        }
      } else {
        // 2 columns = 4 bf16 = one 8-byte load per store
        for (int u = 0; u < (ncol >> 1); ++u) {
          const uint2 v = prev < 0 ? make_uint2(0u, 0u) : __ldg(reinterpret_cast<const uint2*>(src) + u);
          tmem_st_32x32b_x2(taddr + 2u * u, v.x, v.y);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[ab]);
    };

    uint32_t tc = 0;
    gather(0);
    for (int job = 0; job < n_jobs; ++job) {
      const int k = jm.k(job), c = jm.c(job);
      const int t_lo = jm.t_begin(job), my_tiles = jm.t_end(job) - t_lo;
      // the next chunk of the same position only needs x_{k-1}: gather it now
      if (!jm.last_of_position(job)) gather(job + 1);
      const int b = c * NBJ + ml;
      const bool valid = b < p.B;
      const unsigned long long tag = (unsigned long long)(job + 1) << 32;
      // per-thread state: lazy reference Mr, filter threshold Tf ~ exp(best_known - Mr),
      // the best exact score known for the request (this thread's or another's), the
      // thread's own best (score, index, logit), the softmax sum against Mr, the max
      float Mr = -INFINITY, Tf = 0.f, known = -INFINITY, ssum = 0.f, mx = -INFINITY;
      float bsc = -INFINITY, bz = -INFINITY;
      int bi = -1;
      // Chunks of 64 or more requests also share bounds between CTAs: the argmax key of the
      // request at this position holds the best (score, index) any CTA has published so far
      // (every value published there is an exact score of one of the request's elements,
      // so the final maximum is unchanged).  One reader per request and CTA folds it into
      // the CTA's bound a tile after loading it; a thread holding the CTA's best publishes
      // it after its second and fourth tiles.  (For 32 requests the traffic on the few key
      // lines costs more than the bound saves.)
      [[maybe_unused]] unsigned long long* kp = p.keys + (size_t)(k - 1) * p.B + (valid ? b : 0);
      [[maybe_unused]] unsigned long long gk = 0ull;
      for (int t = 0; t < my_tiles; ++t, ++tc) {
        const int acc = tc % S::kAccBufs;
        const int su = tc % S::kUStages;
        if constexpr (!Greedy && NBJ >= 64) {
          if (sidx == 0 && valid) {
            if (gk) atomic_max_shared_u64(&thr[ml], tag | (gk >> 32));
            if (t >= 1 && t + 1 < my_tiles) gk = __ldcg(kp);
          }
        }
        // both stages are held until the tile is done (the other accumulators and the U
        // ring keep the tensor core and the copies ahead)
        const bool have = swait(&acc_full[acc], (tc / S::kAccBufs) & 1) &&
                          swait(&u_full[su], (tc / S::kUStages) & 1);
        if (have) {
          tc_fence_after_sync();
          const int vt = (t_lo + t) * kTileN + c0;
          const bool ragged = (t_lo + t + 1) * kTileN > p.V;
          const uint8_t* us = smem + S::kOffU + su * S::kUStageBytes;
          if (!Greedy && valid) {
            // the best exact score any thread of the CTA has found for the request in this
            // job (keys of earlier jobs carry a smaller tag and read as nothing)
            const unsigned long long sh = ld_volatile_shared_u64(&thr[ml]);
            if (sh >= tag) {
              const float ks = key_float((uint32_t)sh);
              if (ks > known) {
                known = ks;
                if (Mr != -INFINITY) Tf = ex2_approx((known - Mr) * kLog2e) * kShrink;
              }
            }
          }
          // octets in pairs (16 columns): one tensor-memory load, four independent Philox
          // chains and one candidate mask per pair
#pragma unroll 1
          for (int o = 0; o < S::kOct; o += 2) {
            const int v = vt + 8 * o;
            const int col = c0 + 8 * o;                 // a multiple of 16
            uint32_t a16[16];
            __syncwarp();                               // a whole-warp load: every lane, converged
            tmem_ld_32x32b_sync<16>(lane_base + S::kAccCol + (uint32_t)(kTileN * acc + col), a16);
            if (!valid) continue;                       // a row beyond the batch
            // U: box col / 32, row ml, 16-byte chunks (col % 32) / 4 .. + 3, 128-byte
            // swizzle (chunk ^ row % 8)
            const uint8_t* row = us + (col >> 5) * (NBJ * 128) + u_row;
            const int ch = (col & 31) >> 2;             // 0 or 4
            float zo[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 u4 = *reinterpret_cast<const float4*>(row + (((ch + q) ^ u_sw) << 4));
              zo[4 * q + 0] = __uint_as_float(a16[4 * q + 0]) + u4.x;
              zo[4 * q + 1] = __uint_as_float(a16[4 * q + 1]) + u4.y;
              zo[4 * q + 2] = __uint_as_float(a16[4 * q + 2]) + u4.z;
              zo[4 * q + 3] = __uint_as_float(a16[4 * q + 3]) + u4.w;
            }
            if (ragged) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (v + j >= p.V) zo[j] = -INFINITY;
            }
            float lm = zo[0];
#pragma unroll
            for (int j = 1; j < 16; ++j) lm = fmaxf(lm, zo[j]);
            if (lm == -INFINITY) continue;              // wholly beyond the vocabulary
            mx = fmaxf(mx, lm);
            if (lm > Mr + kLazy) {
              ssum = (Mr == -INFINITY) ? 0.f : ssum * ex2_approx((Mr - lm) * kLog2e);
              Mr = lm;
              Tf = (known == -INFINITY) ? 0.f : ex2_approx((known - Mr) * kLog2e) * kShrink;
            }
            const float mL = Mr * kLog2e;
            if constexpr (Greedy) {
#pragma unroll
              for (int j = 0; j < 16; ++j) ssum += ex2_approx(fmaf(zo[j], kLog2e, -mL));
              if (lm > bsc) {                           // a later equal maximum has a larger v
                int jl = 15;
#pragma unroll
                for (int j = 14; j >= 0; --j)
                  if (zo[j] == lm) jl = j;
                bsc = lm; bz = lm; bi = v + jl;
              }
            } else {
              uint32_t dw[16];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 d = philox_wide(make_uint4((uint32_t)(v >> 2) + (uint32_t)q, (uint32_t)k,
                                                       (uint32_t)b, 0u), p.philox);
                dw[4 * q + 0] = d.x; dw[4 * q + 1] = d.y; dw[4 * q + 2] = d.z; dw[4 * q + 3] = d.w;
              }
              unsigned cm = 0u;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float e = ex2_approx(fmaf(zo[j], kLog2e, -mL));
                ssum += e;
                cm |= (e > Tf * w_of_draw(dw[j]) ? 1u : 0u) << j;
              }
              if (cm) {
                // candidates (rare past a job's first pair) are scored exactly in increasing
                // v (equal scores keep the smallest index).  A lane with more than two first
                // tightens its test with the best lower bound e (1 - w) / w <= e / E among
                // them and keeps the survivors.  The scoring loop runs once per set bit of
                // the lane's survivors, so a warp pays for its busiest lane only.
                unsigned sm = cm;
                if (__popc(cm) > 2) {
                  float L = 0.f;
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    if ((cm >> j) & 1u) {
                      const float e = ex2_approx(fmaf(zo[j], kLog2e, -mL)), w = w_of_draw(dw[j]);
                      L = fmaxf(L, e * (1.f - w) * rcp_approx(w));
                    }
                  const float Teff = fmaxf(Tf, L * kShrink);
                  sm = 0u;
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    if ((cm >> j) & 1u)
                      sm |= (ex2_approx(fmaf(zo[j], kLog2e, -mL)) > Teff * w_of_draw(dw[j]) ? 1u : 0u) << j;
                }
                bool improved = false;
                while (sm) {
                  const int j = __ffs(sm) - 1;
                  sm &= sm - 1u;
                  // element j's logit and draw: a select tree on the bits of j (depth 4)
                  float zj;
                  uint32_t dj;
                  {
                    float z8[8];
                    uint32_t d8[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                      z8[q] = (j & 1) ? zo[2 * q + 1] : zo[2 * q];
                      d8[q] = (j & 1) ? dw[2 * q + 1] : dw[2 * q];
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                      z8[q] = (j & 2) ? z8[2 * q + 1] : z8[2 * q];
                      d8[q] = (j & 2) ? d8[2 * q + 1] : d8[2 * q];
                    }
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                      z8[q] = (j & 4) ? z8[2 * q + 1] : z8[2 * q];
                      d8[q] = (j & 4) ? d8[2 * q + 1] : d8[2 * q];
                    }
                    zj = (j & 8) ? z8[1] : z8[0];
                    dj = (j & 8) ? d8[1] : d8[0];
                  }
                  // E accurate (log1p), its logarithm the fast one: within 3 ulp of log E,
                  // under 6e-6 for every E a 23-bit draw gives, 1.5e-6 for E in [0.01, 16]
                  const float scj = zj - __logf(exp1_from_w(w_of_draw(dj)));
                  if (scj > bsc) { bsc = scj; bi = v + j; bz = zj; improved = true; }
                }
                if (improved) {
                  if (bsc > known) {
                    known = bsc;
                    Tf = ex2_approx((known - Mr) * kLog2e) * kShrink;
                  }
                  atomic_max_shared_u64(&thr[ml], tag | (unsigned long long)float_key(bsc));
                }
              }
            }
          }
        }
        if constexpr (!Greedy && NBJ >= 64) {
          if (valid && (t == 1 || t == 3) && t + 2 < my_tiles && bi >= 0 && bsc >= known)
            atomicMax(kp, argmax_key(bsc, bi));
        }
        if (have) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&acc_empty[acc]);
            mbar_arrive(&u_empty[su]);
          }
        }
      }
      // ---- this thread's partial, then a shuffle tree per request of the chunk: every
      // request has E = kSamplerThreads / NBJ partials (one per sampler warp holding its
      // rows), and sampler thread t merges entry t % E of request t / E with its E - 1
      // neighbours
      {
        const float st = (Mr == -INFINITY || mx == -INFINITY) ? 0.f : ssum * ex2_approx((Mr - mx) * kLog2e);
        float* mw = merge + sw * kMergeStride + lane;
        mw[0] = mx;
        mw[32] = st;
        mw[64] = bsc;
        mw[96] = bz;
        mw[128] = __int_as_float(bi);
      }
      named_bar_sync(kBarSamplers, kSamplerThreads);
      {
        constexpr int E = kSamplerThreads / NBJ;       // 8, 4 or 2 consecutive lanes
        const int mrow = stid / E, e = stid % E;
        const int src = (mrow >> 5) + (NBJ / 32) * e;  // the e-th warp holding row mrow
        const float* mr = merge + src * kMergeStride + (mrow & 31);
        float m = mr[0], s = mr[32], sc = mr[64], zz = mr[96];
        int ix = __float_as_int(mr[128]);
#pragma unroll
        for (int o = E / 2; o >= 1; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
          const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
          const float sc2 = __shfl_xor_sync(0xffffffffu, sc, o);
          const float z2 = __shfl_xor_sync(0xffffffffu, zz, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, ix, o);
          const float mm = fmaxf(m, m2);
          if (mm != -INFINITY)
            s = (m == -INFINITY ? 0.f : s * ex2_approx((m - mm) * kLog2e)) +
                (m2 == -INFINITY ? 0.f : s2 * ex2_approx((m2 - mm) * kLog2e));
          m = mm;
          if (better(sc2, i2, sc, ix)) { sc = sc2; ix = i2; zz = z2; }
        }
        const int bm = c * NBJ + mrow;
        if (e == 0 && bm < p.B && !*(volatile int*)&abort_s) {
          RowState ps;
          ps.m = m; ps.s = s; ps.score = sc; ps.z = zz; ps.idx = ix;
          p.partials[((size_t)(k % 3) * p.B + bm) * G + cta] = ps;
          if (ix >= 0) {
            atomicMax(p.keys + (size_t)(k - 1) * p.B + bm, argmax_key(sc, ix));
            // one CTA's local best: warm L2 with its W1 row for the gather after the barrier
            if (k < p.gamma)
              asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                               reinterpret_cast<uint64_t>(p.W1 + (size_t)ix * p.r)),
                           "r"((uint32_t)p.r * 2u)
                           : "memory");
          }
        }
      }
      // the partials and keys are ordered before the grid arrival by this barrier; the
      // merge area is free again after it
      named_bar_sync(kBarSamplers, kSamplerThreads);
      if (jm.last_of_position(job)) {
        if (stid == 0 && !*(volatile int*)&abort_s) {
          // the last arrival also carries this CTA's survivals: wait for the confidence warp
          if (k == p.gamma && p.c_out) {
            const long long t0 = sm_cycles();
            while (!*(volatile int*)&conf_done_s) {
              if (*(volatile int*)&abort_s || sm_cycles() - t0 > p.wait_cycles) {
                set_device_error(p.err, DSPARK_ERR_TIMEOUT);
                atomicExch(&abort_s, 1);
                break;
              }
            }
            __threadfence();
          }
          if (!*(volatile int*)&abort_s)
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.grid_count) : "memory");
        }
        if (job + 1 < n_jobs) {
          grid_wait((unsigned int)G * (unsigned int)k + p.grid_extra);
          gather(job + 1);
          // every CTA has published position k: merge this CTA's share of it while the
          // tensor core computes the next position's first tile (slot k % 3 is next
          // written at position k + 3)
          if (!*(volatile int*)&abort_s) {
            for (int bb = cta + sw * G; bb < p.B; bb += kSamplers * G)
              finalize_row<Greedy>(p, bb, bb / NBJ, k, G, lane);
          }
        }
      }
    }
    // the last position: wait for every CTA, then merge this CTA's rows
    grid_wait((unsigned int)G * (unsigned int)p.gamma + p.grid_extra);
    if (!*(volatile int*)&abort_s)
      for (int bb = cta + sw * G; bb < p.B; bb += kSamplers * G)
        finalize_row<Greedy>(p, bb, bb / NBJ, p.gamma, G, lane);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, kTmemCols);
  // The prefix scheduler over every request's survivals once the last position is done:
  // every CTA wrote its survivals before its last grid arrival, which the samplers' final
  // wait acquired and the barrier above passed on to every thread.  The W2 and U rings
  // (their copies and MMAs drained) hold the keys.
  if (p.ell && !p.sched_warp && !*(volatile int*)&abort_s) {
    const int N = p.B * p.gamma;
    int Npad = 2;
    while (Npad < N) Npad <<= 1;
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem + S::kOffW);
    const size_t key_bytes = (size_t)(S::kOffMerge - S::kOffW);
    if (!p.sched_keys) {
      if (cta == 0)
        schedule_block<false>(p.a_out, p.B, p.gamma, Npad, p.sps, nullptr, nullptr, p.ell,
                              p.B_total, p.theta, keys, key_bytes);
    } else {
      schedule_ranks(p.a_out, N, p.gamma, p.sched_keys, keys,
                     reinterpret_cast<int*>(smem + S::kOffMerge), G, cta);
      // count in once more; CTA 0 waits for every share, then scans in that order
      if (threadIdx.x == 0 && !*(volatile int*)&abort_s)
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.grid_count) : "memory");
      if (cta == 0) {
        if (threadIdx.x == 0) {
          const unsigned int target = (unsigned int)G * (unsigned int)(p.gamma + 1) + p.grid_extra;
          const long long t0 = sm_cycles();
          while (ld_acquire_u32(p.grid_count) < target) {
            if (*(volatile int*)&abort_s || sm_cycles() - t0 > p.wait_cycles) {
              set_device_error(p.err, DSPARK_ERR_TIMEOUT);
              atomicExch(&abort_s, 1);
              break;
            }
          }
        }
        __syncthreads();
        if (!*(volatile int*)&abort_s) {
          for (int i = threadIdx.x; i < N; i += kThreads) keys[i] = __ldcg(p.sched_keys + i);
          __syncthreads();
          schedule_block<false>(p.a_out, p.B, p.gamma, Npad, p.sps, nullptr, nullptr, p.ell,
                                p.B_total, p.theta, keys, key_bytes, /*presorted=*/true);
        }
      }
    }
  }
}

// U [B, gamma, V] fp32 as a 3-D tensor {V, gamma, B}; a box is 32 vocabulary entries (128
// bytes, the 128-byte swizzle's span) of one position for NBJ requests.  Entries out of
// range read as zero.
bool encode_u_map_sw(CUtensorMap* map, const float* U, int B, int gamma, int V, int NBJ) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)gamma, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)V * 4, (cuuint64_t)gamma * V * 4};
  cuuint32_t box[3] = {32, 1, (cuuint32_t)NBJ};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(U), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NBJ, bool Greedy>
int lanes_grid() {
  static std::atomic<int> cache[kMaxCachedDevices];
  return per_device_grid(cache, [] {
    int per = 0;
    const size_t smem = LSmem<NBJ>::kBytes + 1024;
    if (cudaFuncSetAttribute(draft_lanes_kernel<NBJ, Greedy>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, draft_lanes_kernel<NBJ, Greedy>,
                                                      kThreads, smem) != cudaSuccess)
      return -1;
    return per > 0 ? 1 : 0;
  });
}

template <int NBJ, bool Greedy>
cudaError_t launch_lanes(const CUtensorMap& w2_map, const CUtensorMap& u_map, const LParams& p,
                         int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = LSmem<NBJ>::kBytes + 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, draft_lanes_kernel<NBJ, Greedy>, w2_map, u_map, p);
}

template <bool Greedy>
int grid_of(int NBJ) {
  return NBJ == 32 ? lanes_grid<32, Greedy>() : NBJ == 64 ? lanes_grid<64, Greedy>()
                                                          : lanes_grid<128, Greedy>();
}
template <bool Greedy>
cudaError_t launch_of(int NBJ, const CUtensorMap& w2_map, const CUtensorMap& u_map,
                      const LParams& p, int grid, cudaStream_t stream) {
  return NBJ == 32 ? launch_lanes<32, Greedy>(w2_map, u_map, p, grid, stream)
       : NBJ == 64 ? launch_lanes<64, Greedy>(w2_map, u_map, p, grid, stream)
                   : launch_lanes<128, Greedy>(w2_map, u_map, p, grid, stream);
}

// bound of the draft kernel's waits and the grid-barrier offset used by the next launches
// (dspark_testing_set_wait_limit); 0 / 0 is the production setting
std::atomic<long long> g_wait_cycles{0};
std::atomic<unsigned int> g_grid_extra{0};

}  // namespace

void set_draft_wait_limit(long long cycles, unsigned int grid_extra) {
  g_wait_cycles.store(cycles);
  g_grid_extra.store(grid_extra);
}

long long draft_wait_limit() {
  const long long wc = g_wait_cycles.load();
  return wc > 0 ? wc : kWaitCycles;
}
unsigned int draft_barrier_offset() { return g_grid_extra.load(); }

size_t draft_region_bytes(int B, int gamma) {
  return align_up((size_t)3 * B * kDraftMaxCtas * sizeof(RowState), 256) + 256 +
         align_up((size_t)gamma * B * sizeof(unsigned long long), 256);
}

int draft_kchunk(int r) { return (r % 64 == 0) ? 64 : (r % 32 == 0) ? 32 : 16; }

int draft_fused_schedule_limit() { return kGridScheduleItems; }

cudaError_t launch_draft_lanes(const uint16_t* W1, const uint16_t* W2, const uint16_t* W2p,
                               const float* U, const int32_t* anchor, int B, int gamma, int V,
                               int r, uint64_t seed, bool greedy, int32_t* tokens, float* q_tok,
                               float* row_max, float* row_sumexp, void* region, int* err,
                               cudaStream_t stream, const DraftStepArgs* step) {
  const int NBJ = B <= 32 ? 32 : B <= 64 ? 64 : 128;
  const int n_tiles = cdiv(V, kTileN);
  int grid = greedy ? grid_of<true>(NBJ) : grid_of<false>(NBJ);
  if (grid <= 0) return cudaErrorInvalidConfiguration;
  if (grid > n_tiles) grid = n_tiles;
  if (grid > kDraftMaxCtas) grid = kDraftMaxCtas;
  LParams p;
  memset(&p, 0, sizeof(p));
  p.W1 = W1;
  p.W2p = W2p;
  p.anchor = anchor;
  p.B = B; p.gamma = gamma; p.V = V; p.r = r;
  p.n_tiles = n_tiles;
  p.n_chunks = cdiv(B, NBJ);
  // the kernel's unit arithmetic is 32-bit: (chunks x tiles) x CTAs < 2^32
  if ((unsigned long long)p.n_chunks * (unsigned long long)n_tiles * (unsigned long long)grid >=
      (1ull << 32))
    return cudaErrorNotSupported;
  p.kc = draft_kchunk(r);
  p.seed = seed;
  p.philox = philox_keys(seed);
  const size_t part_bytes = align_up((size_t)3 * B * kDraftMaxCtas * sizeof(RowState), 256);
  char* base = static_cast<char*>(region);
  p.partials = reinterpret_cast<RowState*>(base);
  p.grid_count = reinterpret_cast<unsigned int*>(base + part_bytes);
  p.conf_count = p.grid_count + 1;
  p.rank_count = p.grid_count + 2;
  p.keys = reinterpret_cast<unsigned long long*>(base + part_bytes + 256);
  p.tokens = tokens;
  p.q_tok = q_tok;
  p.row_max = row_max;
  p.row_sumexp = row_sumexp;
  p.err = err;
  const long long wc = g_wait_cycles.load();
  p.wait_cycles = wc > 0 ? wc : kWaitCycles;
  p.grid_extra = g_grid_extra.load();
  if (step) {
    // survivals are kept for kConfSlots requests of every CTA
    if ((long long)B > (long long)kConfSlots * grid) return cudaErrorNotSupported;
    p.h = step->h; p.w_c = step->w_c; p.b_c = step->b_c; p.H = step->H;
    p.c_out = step->c; p.a_out = step->a;
    if (step->ell && (long long)B * gamma <= kThreads) {
      p.sps = step->sps; p.ell = step->ell; p.B_total = step->B_total; p.theta = step->theta;
      p.sched_warp = grid > B && step->sched_keys ? 1 : 0;
      p.sched_keys = step->sched_keys;
    } else if (step->ell && step->sched_keys && (long long)B * gamma <= kGridScheduleItems) {
      p.sps = step->sps; p.ell = step->ell; p.B_total = step->B_total; p.theta = step->theta;
      p.sched_keys = step->sched_keys;
    }
  }
  cudaError_t e = cudaMemsetAsync(base + part_bytes, 0,
                                  256 + (size_t)gamma * B * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  CUtensorMap w2_map, u_map;
  memset(&w2_map, 0, sizeof(w2_map));
  if (!W2p && !encode_w2_map(&w2_map, W2, V, r, p.kc)) return cudaErrorInvalidValue;
  if (!encode_u_map_sw(&u_map, U, B, gamma, V, NBJ)) return cudaErrorInvalidValue;
  return greedy ? launch_of<true>(NBJ, w2_map, u_map, p, grid, stream)
                : launch_of<false>(NBJ, w2_map, u_map, p, grid, stream);
}

}  // namespace dspark
