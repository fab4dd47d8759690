// Host-side plan of the DSpark calls: launch splits and the workspace layout, plus the
// launchers each translation unit provides.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/dspark.h"
#include "common.cuh"

namespace dspark {

constexpr int kSampleThreads = 256;      // threads of the row-sampling kernels
constexpr int kTargetCtas = 608;         // CTAs a row-sampling launch aims for (4 per SM)
constexpr int kMaxScheduleItems = 16384; // R * gamma handled by the one-CTA scheduler
constexpr int kGemmTileV = 128;          // vocabulary rows per tensor-core tile (MMA M)
constexpr int kDraftMaxCtas = 160;       // upper bound of the persistent draft grid
// scheduler items (B gamma) the step's first launch ranks itself (more: a scheduler kernel)
constexpr int kGridScheduleItems = 4096;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

// Split of a V-long row into `splits` segments of `seg` elements (seg % 4 == 0).
struct RowSplit {
  int splits, seg;
};
inline RowSplit row_split(int rows, int V) {
  int want = cdiv(kTargetCtas, rows > 0 ? rows : 1);
  int most = cdiv(V, 4 * kSampleThreads);    // at least one float4 per thread per segment
  if (want > most) want = most;
  if (want > 64) want = 64;
  if (want < 1) want = 1;
  RowSplit s;
  s.seg = (int)align_up((size_t)cdiv(V, want), 4);
  s.splits = cdiv(V, s.seg);
  return s;
}

// Fixed segments of the verify kernels: every thread of a 256-thread CTA issues all its
// 128-bit loads of a segment at once (16 per thread for the target statistics, 4 per
// input row for the final sample, which loads three rows).
constexpr int kStatsVec = 16;
constexpr int kStatsSeg = 4 * kSampleThreads * kStatsVec;   // 16384 logits
constexpr int kVerVec = 4;
constexpr int kVerSeg = 4 * kSampleThreads * kVerVec;       // 4096 logits
inline RowSplit fixed_split(int V, int seg) {
  RowSplit s;
  s.seg = seg;
  s.splits = cdiv(V, seg);
  return s;
}

size_t draft_region_bytes(int B, int gamma);

// copies of the RNN head's state and E rows kept in the workspace (see draft_fused.cu)
constexpr int kRnnStateCopies = 2;

struct Plan {
  int B, gamma, V, r, H;
  RowSplit stats, ver;
  // byte offsets into the workspace
  size_t off_err, off_draft, off_bias, off_part, off_mode,
      off_pos, off_prev, off_slot, off_nres, off_fallback, off_rec, off_sched, off_cand_n,
      off_cand, off_rnn_state, total;
};

inline Plan make_plan(int B, int gamma, int V, int r, int H) {
  Plan p;
  p.B = B; p.gamma = gamma; p.V = V; p.r = r; p.H = H;
  p.stats = fixed_split(V, kStatsSeg);
  p.ver = fixed_split(V, kVerSeg);
  size_t o = 0;
  p.off_err = o; o += 256;
  p.off_draft = o; o = align_up(o + draft_region_bytes(B, gamma), 256);
  p.off_bias = o; o = align_up(o + (size_t)B * V * sizeof(float), 256);
  const size_t parts = (size_t)B * gamma * p.stats.splits;
  p.off_part = o; o = align_up(o + parts * sizeof(RowState), 256);
  p.off_mode = o; o = align_up(o + (size_t)B * sizeof(int32_t), 256);
  p.off_pos = o; o = align_up(o + (size_t)B * sizeof(int32_t), 256);
  p.off_prev = o; o = align_up(o + (size_t)B * sizeof(int32_t), 256);   // by residual slot
  p.off_slot = o; o = align_up(o + (size_t)B * sizeof(int32_t), 256);   // slot of request b
  p.off_nres = o; o += 256;                                              // residual count
  p.off_fallback = o; o = align_up(o + (size_t)B * sizeof(int32_t), 256);
  p.off_rec = o; o = align_up(o + (size_t)B * 32, 256);                 // final-draw records
  // the first launch's scheduler keys in ranked order (batches of 385 .. 4096 items)
  p.off_sched = o;
  if ((long long)B * gamma <= kGridScheduleItems) o = align_up(o + (size_t)B * gamma * 8, 256);
  // the final draw's candidates: a count and up to 64 entries of 16 bytes per segment
  p.off_cand_n = o; o = align_up(o + (size_t)B * p.ver.splits * sizeof(int), 256);
  p.off_cand = o; o = align_up(o + (size_t)B * p.ver.splits * 64 * 16, 256);
  // RNN head: state [2][B][r] fp32, then the current position's rows [B][2][r] bf16
  // RNN head: kRnnStateCopies copies of the state [2][B][r] fp32 and of the E rows [B][2][r] bf16
  p.off_rnn_state = o;
  o = align_up(o + (size_t)kRnnStateCopies * ((size_t)2 * B * r * sizeof(float) + (size_t)2 * B * r * 2), 256);
  p.total = o;
  return p;
}

// Per-device launch setup.  A kernel's dynamic shared-memory attribute and the number of
// its CTAs an SM holds belong to a device, so `setup` (which sets the attribute on the
// current device and returns the CTAs per SM, or a negative value on failure) runs once
// per device; the SM count times its result is cached per device (failures are not).
// Returns 0 when the device cannot be queried or setup fails.
constexpr int kMaxCachedDevices = 64;
template <typename F>
inline int per_device_grid(std::atomic<int> (&cache)[kMaxCachedDevices], F&& setup) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxCachedDevices) return 0;
  const int v = cache[dev].load(std::memory_order_acquire);
  if (v != 0) return v - 1;            // stored plus one: zero means "not set up yet"
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  const int per = setup();
  if (per < 0) return 0;
  cache[dev].store(sms * per + 1, std::memory_order_release);
  return sms * per;
}

template <typename T>
inline T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// Launch with programmatic stream serialization (see pdl_wait in common.cuh): the kernel
// must call pdl_wait() before it reads earlier kernels' outputs or exits.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- tensor maps ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();
// W2 [r, V] bf16 as {V, r} with boxes of 64 columns x box_rows rows, 128-byte swizzle
bool encode_w2_map(CUtensorMap* map, const uint16_t* W2, int V, int r, int box_rows);

// ---- launchers (return cudaError_t of the launch) ----
// bias[b][v] = sum_i W1[prev_b][i] * W2[i][v] for b < rows, v < V (rows with prev_b == -1
// are 0); rows = B, or min(B, *n_rows) when n_rows (a device value the previous kernel on
// the stream writes) is not null.  W2p: the packed tile images of pack.cu in place of W2.
cudaError_t launch_bias_gemm(const uint16_t* W2, const uint16_t* W2p, const uint16_t* W1,
                             const int32_t* prev, int prev_stride, int B, const int* n_rows, int V,
                             int r, float* out, int* err, cudaStream_t stream);
// bias[b][v] = sum_i Ef[prev_b][i] * W2[i][v] with fp32 rows Ef [table_rows][r] taken as two
// bf16 terms each (rows with prev_b == -1 are 0); rows as above
cudaError_t launch_bias_gemm_rows(const uint16_t* W2, const uint16_t* W2p, const float* Ef,
                                  int table_rows, const int32_t* prev, int B, const int* n_rows,
                                  int V, int r, float* out, int* err, cudaStream_t stream);

// the whole draft (all gamma positions) in one cooperative launch of the request-major
// kernel of draft.cu (W2p: packed tile images, else W2 by TMA; greedy: x = argmax z);
// `region` holds draft_region_bytes(B, gamma) of workspace
// with `step` (may be null) the same launch also computes the confidence head and the
// survivals at every position boundary, and, when B * gamma <= draft_fused_schedule_limit(),
// runs the prefix scheduler after the last position (up to 384 items in CTA 0, more with
// the grid ranking the items into step->sched_keys)
struct DraftStepArgs {
  const float* h;      // [B][gamma][H]
  const float* w_c;    // [H + r]
  float b_c;
  int H;
  float* c;            // [B][gamma]
  float* a;            // [B][gamma]
  const float* sps;    // the scheduler (ell null: not run in the draft)
  int32_t* ell;
  int32_t* B_total;
  double* theta;
  unsigned long long* sched_keys;   // [B gamma] scratch when B gamma > 384 (the grid ranks)
};
int draft_fused_schedule_limit();
cudaError_t launch_draft_lanes(const uint16_t* W1, const uint16_t* W2, const uint16_t* W2p,
                               const float* U, const int32_t* anchor, int B, int gamma, int V,
                               int r, uint64_t seed, bool greedy, int32_t* tokens, float* q_tok,
                               float* row_max, float* row_sumexp, void* region, int* err,
                               cudaStream_t stream, const DraftStepArgs* step = nullptr);
// bound (SM cycles, 0: the default of about 2 s) of that kernel's waits and an offset added
// to its grid-barrier targets, for the launches that follow (tests of the timeout path)
void set_draft_wait_limit(long long cycles, unsigned int grid_extra);
// the current setting of that hook: the bound of every wait (0: the production bound) and
// the offset added to every grid-barrier target
long long draft_wait_limit();
unsigned int draft_barrier_offset();

// the same entry points under their ABI names (see draft_fused.cu)
cudaError_t launch_draft_fused(const uint16_t* W1, const uint16_t* W2, const float* U,
                               const int32_t* anchor, int B, int gamma, int V, int r,
                               uint64_t seed, int32_t* tokens, float* q_tok, float* row_max,
                               float* row_sumexp, void* region, int* err, cudaStream_t stream);

// the same with W2 given as packed tile images (see pack.cu)
cudaError_t launch_draft_fused_packed(const uint16_t* W1, const uint16_t* W2p, const float* U,
                                      const int32_t* anchor, int B, int gamma, int V, int r,
                                      uint64_t seed, int32_t* tokens, float* q_tok,
                                      float* row_max, float* row_sumexp, void* region, int* err,
                                      cudaStream_t stream);
// the greedy draft (x_k = argmax z_k, q_tok = 1) with W2 or, when W2p is not null, the
// packed tile images
cudaError_t launch_draft_fused_greedy(const uint16_t* W1, const uint16_t* W2, const uint16_t* W2p,
                                      const float* U, const int32_t* anchor, int B, int gamma,
                                      int V, int r, int32_t* tokens, float* q_tok,
                                      float* row_max, float* row_sumexp, void* region, int* err,
                                      cudaStream_t stream);
// the draft with the RNN head (see draft_fused.cu and rnn.cu): Wrec [3r][2r] (rnn_pack),
// hp [B][gamma][3r] (rnn_project), E_all [B][gamma][r] written, state
// [kRnnStateCopies][2][B][r] and E_hl [kRnnStateCopies][B][2][r] bf16 scratch
struct RnnDraftArgs {
  const uint16_t* Wrec;
  const float* hp;
  float* E_all;
  float* state;
  uint16_t* E_hl;
};
cudaError_t launch_draft_fused_rnn(const uint16_t* W1, const uint16_t* W2, const uint16_t* W2p,
                                   const float* U, const int32_t* anchor, int B, int gamma, int V,
                                   int r, uint64_t seed, bool greedy, const RnnDraftArgs& rnn,
                                   int32_t* tokens, float* q_tok, float* row_max,
                                   float* row_sumexp, void* region, int* err, cudaStream_t stream);
cudaError_t launch_rnn_pack(const uint16_t* W_rnn, int r, uint16_t* Wrec, cudaStream_t stream);
cudaError_t launch_rnn_project(const float* h, const uint16_t* W_rnn, const float* b_rnn, int M,
                               int H, int r, float* hp, cudaStream_t stream);
// rank rows per W2 stage of the draft kernel (and per packed K-chunk image)
int draft_kchunk(int r);
// the ABI status of a draft launch: cudaErrorNotSupported (a shape beyond the draft
// kernel's limits) is DSPARK_ERR_UNSUPPORTED, any other failure DSPARK_ERR_CUDA
inline dspark_status draft_status(cudaError_t e) {
  return e == cudaSuccess ? DSPARK_OK
       : e == cudaErrorNotSupported ? DSPARK_ERR_UNSUPPORTED : DSPARK_ERR_CUDA;
}

cudaError_t launch_confidence(const float* h, const int32_t* anchor, const int32_t* tokens,
                              const uint16_t* W1, const float* w_c, float b_c, int B, int gamma,
                              int H, int r, int V, float* c, float* a, int* err,
                              cudaStream_t stream);

// K_in / K_out: the two-step capacity (both may be null; see schedule.cu)
// confidence + survival and then, in the grid's last CTA, the prefix scheduler over all of
// them; `done` is a workspace counter that is zero between calls
cudaError_t launch_confidence_schedule(const float* h, const int32_t* anchor,
                                       const int32_t* tokens, const uint16_t* W1,
                                       const float* w_c, float b_c, int B, int gamma, int H,
                                       int r, int V, const float* sps, float* c, float* a,
                                       int32_t* ell, int32_t* B_total, double* theta,
                                       unsigned int* done, int* err, cudaStream_t stream);

cudaError_t launch_schedule(const float* a, int R, int gamma, const float* sps,
                            const int32_t* K_in, int32_t* K_out, int32_t* ell, int32_t* B_total,
                            double* theta, int* err, cudaStream_t stream);

cudaError_t launch_schedule_threshold(const float* a, int R, int gamma, float threshold,
                                      int32_t* ell, int32_t* B_total, cudaStream_t stream);

// T[b, j] for j <= ell[b] from T_src (memory the device reads, host memory included) into T
cudaError_t launch_copy_target_rows(const float* T_src, float* T, const int32_t* ell, int B,
                                    int gamma, int V, int* err, cudaStream_t stream);

// E_all (null for the Markov head): the RNN head's output rows [B][gamma][r] of the draft
cudaError_t launch_verify(const Plan& p, const float* T, const float* U, const uint16_t* W1,
                          const uint16_t* W2, const uint16_t* W2p, const float* E_all,
                          const int32_t* anchor,
                          const int32_t* tokens, const float* q_tok, const float* row_max,
                          const float* row_sumexp, const int32_t* ell, uint64_t seed,
                          int32_t* accept_len, int32_t* out_tokens, int32_t* n_out, void* ws,
                          cudaStream_t stream);

}  // namespace dspark
