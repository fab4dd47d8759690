// Markov transition bias on the tensor cores.
//
// billytse.dev DSpark page, section 3.3: the first-order Markov head's bias for every
// request is B(x_{k-1}, .) = W1[x_{k-1}] W2, rank r.  For a whole batch this is the
// contraction  bias^T [V, B] = W2^T [V, r] x E^T [r, B]  with E[b] = W1[prev_b].
//
// A persistent, warp-specialised kernel (one or two CTAs per SM, each owning a contiguous
// run of 128-row vocabulary tiles) computes bias^T tile by tile:
//   producer warp   streams the W2^T tiles as K-chunks of up to 64 rank rows (two TMA boxes
//                   of 64 vocabulary columns, 128-byte swizzle, or one bulk copy of the
//                   packed tile image) through a 4-stage ring;
//   MMA warp        one lane issues tcgen05.mma (M = 128 vocabulary rows, N = NB requests,
//                   K = 16 per instruction, bf16 in, fp32 accumulators in tensor memory)
//                   into one of four accumulators;
//   4 epilogue warps gather E = W1[prev_b] for each chunk of NB requests into the K-major
//                   B operand, and read the accumulators back (lane = vocabulary row) into
//                   coalesced 128-byte stores of bias[b][v].
// The producer starts on W2 (an input) before the previous kernel on the stream has
// finished; the epilogue warps wait for it before reading prev.
//
// Compact mode (verification): the row count is a device value written by the previous
// kernel (the number of rejected requests), read by the epilogue after that kernel has
// finished and published to the producer and the MMA issuer through an mbarrier; the first
// pass over W2 is streamed before the count is known, later passes only when needed.  A
// pass covers NB <= 256 rows (one tensor-core N per vocabulary tile; 256 only when the
// whole batch fits one pass).
//
// Split mode (the RNN head's verification): E[b] = Ef[prev_b], fp32 rows of a table of
// table_rows rows; each row enters the contraction as two bf16 images, hi = bf16(E) and
// lo = bf16(E - hi), and every K step issues one MMA per image on the same W2 rows, so
// the bias keeps fp32-level accuracy (|E - hi - lo| <= 2^-18 |E|).
#include "internal.h"
#include "sm100_ptx.cuh"

#include <string.h>

#include <type_traits>

namespace dspark {
namespace {

using namespace sm100;

__device__ __forceinline__ void named_bar_sync_n(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

constexpr int kBiasStages = 4;                // W2 K-chunk ring (16 KB each at 64 rows)
constexpr int kBiasDepth = 4;                 // accumulators in tensor memory
constexpr int kBiasKChunkMax = 64;
constexpr int kBiasNamedBar = 1;              // the epilogue warps' barrier

template <int NB, bool Split>
struct BiasSmem {
  static constexpr int kStageBytes = 2 * kBiasKChunkMax * 128;
  static constexpr int kOffW = 0;
  static constexpr int kOffE = kOffW + kBiasStages * kStageBytes;
  static constexpr int kEHalf = NB * 256 * 2;    // NB rows x r <= 256, one image
  static constexpr int kEBytes = (Split ? 2 : 1) * kEHalf;
  // 256-row passes: one E buffer and two accumulators (512 tensor-memory columns)
  static constexpr int kEBufs = NB == 256 ? 1 : 2;
  static constexpr int kDepth = NB == 256 ? 2 : kBiasDepth;
  static constexpr int kBytes = kOffE + kEBufs * kEBytes;
  // warps: producer, MMA, then the epilogue warps, one per tensor-memory lane quarter and
  // column half of a pass of 128 or 256 rows (eight: such a pass's fp32 results per tile
  // and its operand gather take two warps per quarter), one per quarter otherwise
  static constexpr int kEpiWarps = NB >= 128 ? 8 : 4;
  static constexpr int kThreads = (2 + kEpiWarps) * 32;
  static constexpr int kEpiThreads = kEpiWarps * 32;
};

__device__ __forceinline__ uint32_t bf16_bits_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

template <int NB, bool Split>
__global__ void __launch_bounds__(BiasSmem<NB, Split>::kThreads) bias_gemm_kernel(
    const __grid_constant__ CUtensorMap w2_map, const uint16_t* __restrict__ W2p,
    const uint16_t* __restrict__ W1, const float* __restrict__ Ef, int table_rows,
    const int32_t* __restrict__ prev, int prev_stride, int B, const int* __restrict__ n_rows,
    int V, int r, int kc, int n_tiles, float* __restrict__ out, int* err) {
  using S = BiasSmem<NB, Split>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t w_full[kBiasStages], w_empty[kBiasStages];
  __shared__ uint64_t e_full[S::kEBufs], e_empty[S::kEBufs];
  __shared__ uint64_t acc_full[S::kDepth], acc_empty[S::kDepth];
  __shared__ uint64_t mma_drain;
  __shared__ uint64_t count_ready;   // the epilogue has published the pass count
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int rows_s, jobs_s;
  __shared__ int pv_s[NB];           // the current pass's predecessor rows
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int t_lo = (int)((long long)cta * n_tiles / G);
  const int t_hi = (int)((long long)(cta + 1) * n_tiles / G);
  const int my_tiles = t_hi - t_lo;
  const int n_kchunks = r / kc;
  uint32_t tmem_cols = 32;
  while (tmem_cols < (uint32_t)(S::kDepth * NB)) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kBiasStages; ++i) { mbar_init(&w_full[i], 1); mbar_init(&w_empty[i], 1); }
    for (int i = 0; i < S::kEBufs; ++i) { mbar_init(&e_full[i], 1); mbar_init(&e_empty[i], 1); }
    for (int i = 0; i < S::kDepth; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], S::kEpiWarps);
    }
    mbar_init(&mma_drain, 1);
    mbar_init(&count_ready, 1);
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_base_s;

  // bounded wait; a timeout records the error and aborts the CTA
  auto wait1 = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    const long long t0 = sm_cycles();
    for (;;) {
      if (*(volatile int*)&abort_s) return false;
      if (mbar_try_wait_sleep(bar, parity)) return true;
      if (sm_cycles() - t0 > kWaitCycles) {
        set_device_error(err, DSPARK_ERR_TIMEOUT);
        atomicExch(&abort_s, 1);
        return false;
      }
    }
  };

  // the number of passes over W2: known to the epilogue after the previous kernel; the
  // first pass needs no count (it runs in every case), the others wait for it
  auto passes_after_first = [&]() -> int {
    if (!wait1(&count_ready, 0)) return 0;
    return *(volatile int*)&jobs_s;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      if (!W2p) prefetch_tensormap(&w2_map);
      const uint64_t keep = policy_evict_last();
      const uint32_t w_bytes = 2u * (uint32_t)kc * 128u;
      uint32_t ws = 0;
      bool ok = true;
      int n_jobs = 0x7FFFFFFF;                    // decided before the second pass
      for (int job = 0; job < n_jobs && ok; ++job) {
        if (job == 1 && (n_jobs = passes_after_first()) <= 1) break;
        for (int t = t_lo; t < t_hi && ok; ++t) {
          for (int i = 0; i < n_kchunks; ++i, ++ws) {
            const int s = ws % kBiasStages;
            if (!(ok = wait1(&w_empty[s], ((ws / kBiasStages) & 1) ^ 1))) break;
            uint8_t* dst = smem + S::kOffW + s * S::kStageBytes;
            mbar_arrive_expect_tx(&w_full[s], w_bytes);
            if (W2p) {
              // packed: the stage image is contiguous, one 1-D bulk copy
              const uint16_t* src = W2p + ((size_t)t * n_kchunks + i) * (size_t)kc * 128;
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                  " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
                  "l"(reinterpret_cast<uint64_t>(src)), "r"(w_bytes), "r"(smem_u32(&w_full[s])),
                  "l"(keep)
                  : "memory");
            } else {
              tma_load_2d(dst, &w2_map, &w_full[s], t * kGemmTileV, i * kc, keep);
              tma_load_2d(dst + kc * 128, &w2_map, &w_full[s], t * kGemmTileV + 64, i * kc, keep);
            }
          }
        }
      }
      // drain: every issued copy has landed before the CTA may exit
      for (uint32_t i = ws > (uint32_t)kBiasStages ? ws - kBiasStages : 0; i < ws; ++i)
        mbar_wait(&w_full[i % kBiasStages], (i / kBiasStages) & 1, 2000000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------------- MMA issuer
    auto issue_loop = [&](auto ksteps_c) {
      constexpr int KS = decltype(ksteps_c)::value;
      const uint32_t idesc = idesc_bf16_f32(128, NB, 1, 0);
      const uint64_t a_base = smem_desc(smem_u32(smem + S::kOffW), (uint32_t)KS * 2048u, 1024u,
                                        kSwizzle128B);
      uint32_t ws = 0, tc = 0;
      bool ok = true;
      int n_jobs = 0x7FFFFFFF;
      for (int job = 0; job < n_jobs && ok; ++job) {
        if (job == 1 && (n_jobs = passes_after_first()) <= 1) break;
        const int eb = job % S::kEBufs;
        if (!(ok = wait1(&e_full[eb], (job / S::kEBufs) & 1))) break;
        const uint64_t b_base =
            smem_desc(smem_u32(smem + S::kOffE + eb * S::kEBytes), 16u, 1024u, kSwizzle128B);
        for (int t = 0; t < my_tiles && ok; ++t, ++tc) {
          const int ab = tc % S::kDepth;
          if (!(ok = wait1(&acc_empty[ab], ((tc / S::kDepth) & 1) ^ 1))) break;
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + (uint32_t)(ab * NB);
          for (int i = 0; i < n_kchunks; ++i, ++ws) {
            const int s = ws % kBiasStages;
            if (!(ok = wait1(&w_full[s], (ws / kBiasStages) & 1))) break;
            const uint64_t a_s = a_base + (uint64_t)((s * S::kStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
              const uint32_t kg = (uint32_t)(i * KS + kk);
              const uint64_t ad = a_s + (uint64_t)(kk * (2048 >> 4));
              const uint64_t bd = b_base + (uint64_t)((kg >> 2) * (uint32_t)(NB * 128 / 16) + (kg & 3) * 2u);
              umma_bf16_f32(d_tmem, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
              if constexpr (Split) umma_bf16_f32(d_tmem, ad, bd + (uint64_t)(S::kEHalf >> 4), idesc, 1u);
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
      umma_commit(&mma_drain);
      mbar_wait(&mma_drain, 0, 2000000000ull);
    }
    __syncwarp();
  } else {
    // --------------------------------------------- epilogue: E gather, TMEM -> bias rows
    pdl_wait();                 // prev (and the row count) may come from the previous kernel
    pdl_launch_dependents();
    constexpr int kEpiT = S::kEpiThreads;
    const int et = threadIdx.x - 64;              // 0 .. kEpiT - 1
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int half = (warp - 2) >> 2;             // column half (eight epilogue warps)
    const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
    const int kchunks = r >> 3;                   // 16-byte chunks per W1 row
    if (et == 0) {
      int rows = B;
      if (n_rows) {
        rows = *n_rows;
        rows = rows < 0 ? 0 : rows > B ? B : rows;
      }
      rows_s = rows;
      jobs_s = rows > NB ? (rows + NB - 1) / NB : 1;
      mbar_arrive(&count_ready);                  // release: rows_s and jobs_s first
    }
    named_bar_sync_n(kBiasNamedBar, kEpiT);
    const int rows = *(volatile int*)&rows_s;
    const int n_jobs = *(volatile int*)&jobs_s;
    uint32_t tc = 0;
    for (int job = 0; job < n_jobs; ++job) {
      const int b0 = job * NB;
      const int eb = job % S::kEBufs;
      // E = W1[prev_b] as the K-major, 128-byte-swizzled B operand: 16-byte chunk c of row n
      // goes to chunk (c % 8) ^ (n % 8) of line n of K-block c / 8
      if (et == 0) wait1(&e_empty[eb], ((job / S::kEBufs) & 1) ^ 1);
      named_bar_sync_n(kBiasNamedBar, kEpiT);
      uint8_t* sE = smem + S::kOffE + eb * S::kEBytes;
      // the pass's predecessor rows, once (checked here), then the operand rows; a 256-row
      // pass keeps four 16-byte loads in flight per thread (measured: one is best at 128)
      for (int n = et; n < NB; n += kEpiT) {
        const int b = b0 + n;
        int pv = -1;
        if (b < rows) {
          pv = prev[(size_t)b * prev_stride];
          if (pv < -1 || pv >= table_rows) {
            set_device_error(err, DSPARK_ERR_DEVICE_CHECK);
            pv = -1;
          }
        }
        pv_s[n] = pv;
      }
      named_bar_sync_n(kBiasNamedBar, kEpiT);
      if (!*(volatile int*)&abort_s) {
        constexpr int kBatch = NB == 256 ? 4 : 1;
        for (int idx0 = et; idx0 < NB * kchunks; idx0 += kEpiT * kBatch) {
          uint4 val[kBatch], lo[kBatch];
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const int idx = idx0 + kEpiT * u;
            val[u] = make_uint4(0u, 0u, 0u, 0u);
            lo[u] = val[u];
            if (idx < NB * kchunks) {
              const int n = idx / kchunks, c = idx - n * kchunks;
              const int pv = pv_s[n];
              if (pv >= 0) {
                if constexpr (Split) {
                  const float4* src = reinterpret_cast<const float4*>(Ef + (size_t)pv * r) + 2 * c;
                  const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
                  const float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                  uint32_t hb[8], lb[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    hb[e] = bf16_bits_rne(x[e]);
                    lb[e] = bf16_bits_rne(x[e] - __uint_as_float(hb[e] << 16));
                  }
                  val[u] = make_uint4(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16), hb[4] | (hb[5] << 16),
                                      hb[6] | (hb[7] << 16));
                  lo[u] = make_uint4(lb[0] | (lb[1] << 16), lb[2] | (lb[3] << 16), lb[4] | (lb[5] << 16),
                                     lb[6] | (lb[7] << 16));
                } else {
                  val[u] = __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)pv * r) + c);
                }
              }
            }
          }
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const int idx = idx0 + kEpiT * u;
            if (idx < NB * kchunks) {
              const int n = idx / kchunks, c = idx - n * kchunks;
              const size_t off = (size_t)(c >> 3) * NB * 128 + (size_t)n * 128 + (((c & 7) ^ (n & 7)) << 4);
              *reinterpret_cast<uint4*>(sE + off) = val[u];
              if constexpr (Split) *reinterpret_cast<uint4*>(sE + S::kEHalf + off) = lo[u];
            }
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync_n(kBiasNamedBar, kEpiT);
      if (et == 0) mbar_arrive(&e_full[eb]);
      for (int t = 0; t < my_tiles; ++t, ++tc) {
        const int ab = tc % S::kDepth;
        const bool ok = wait1(&acc_full[ab], (tc / S::kDepth) & 1);
        if (!__all_sync(0xffffffffu, ok)) continue;
        tc_fence_after_sync();
        const int v = (t_lo + t) * kGemmTileV + q * 32 + lane;
        // this warp's columns (rows b) 16 at a time (in a pass of 128 or more rows the next 16
        // load from tensor memory while the current ones are stored); the accumulator is
        // released after the last
        constexpr int kCols = NB / (S::kEpiWarps / 4);
        const int c_beg = half * kCols;
        const int c_end = min(c_beg + kCols, rows - b0);
        const uint32_t tacc = trow + (uint32_t)(ab * NB);
        auto store16 = [&](const uint32_t (&vals)[16], int c) {
          if (v < V) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (b0 + c + j < rows) out[(size_t)(b0 + c + j) * V + v] = __uint_as_float(vals[j]);
          }
        };
        if constexpr (NB < 128) {
          // (one column run per quarter: 16 columns at a time, each load waited for)
#pragma unroll 1
          for (int c = 0; c < NB && b0 + c < rows; c += 16) {
            uint32_t vals[16];
            tmem_ld_32x32b_sync<16>(tacc + (uint32_t)c, vals);
            if (v < V) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (b0 + c + j < rows) out[(size_t)(b0 + c + j) * V + v] = __uint_as_float(vals[j]);
            }
          }
        } else if (c_beg < c_end) {
          uint32_t va[16], vb[16];
          tmem_ld_32x32b_x16_async(tacc + (uint32_t)c_beg, va);
          tmem_ld_wait();
#pragma unroll 1
          for (int c = c_beg; c < c_end; c += 32) {
            const bool more = c + 16 < c_end, more2 = c + 32 < c_end;
            if (more) tmem_ld_32x32b_x16_async(tacc + (uint32_t)(c + 16), vb);
            store16(va, c);
            if (more) {
              tmem_ld_wait();
              if (more2) tmem_ld_32x32b_x16_async(tacc + (uint32_t)(c + 32), va);
              store16(vb, c + 16);
              if (more2) tmem_ld_wait();
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem_base, tmem_cols);
}

template <int NB, bool Split>
int bias_grid(int n_tiles) {
  static std::atomic<int> cache[kMaxCachedDevices];
  const int g = per_device_grid(cache, [] {
    int per = 0;
    const size_t smem = BiasSmem<NB, Split>::kBytes + 1024;
    if (cudaFuncSetAttribute(bias_gemm_kernel<NB, Split>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, bias_gemm_kernel<NB, Split>,
                                                      BiasSmem<NB, Split>::kThreads,
                                                      smem) != cudaSuccess)
      return -1;
    return per;
  });
  return g < n_tiles ? g : n_tiles;
}

}  // namespace

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// W2 [r, V] bf16 row-major as a 2-D tensor {V, r}; a box is 64 vocabulary columns (128 B,
// the 128-byte swizzle span) by box_rows rank rows.  Out-of-range columns read as zero.
bool encode_w2_map(CUtensorMap* map, const uint16_t* W2, int V, int r, int box_rows) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)V, (cuuint64_t)r};
  cuuint64_t strides[1] = {(cuuint64_t)V * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(W2), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS;
}

namespace {
template <int NB, bool Split>
cudaError_t launch_bias_nb(const CUtensorMap& w2_map, const uint16_t* W2p, const uint16_t* W1,
                           const float* Ef, int table_rows, const int32_t* prev, int prev_stride,
                           int B, const int* n_rows, int V, int r, int kc, int n_tiles, float* out,
                           int* err, cudaStream_t stream) {
  const int grid = bias_grid<NB, Split>(n_tiles);
  if (grid <= 0) return cudaErrorInvalidConfiguration;
  return launch_pdl(bias_gemm_kernel<NB, Split>, dim3(grid), dim3(BiasSmem<NB, Split>::kThreads),
                    (size_t)BiasSmem<NB, Split>::kBytes + 1024, stream, w2_map, W2p, W1, Ef,
                    table_rows, prev, prev_stride, B, n_rows, V, r, kc, n_tiles, out, err);
}

template <bool Split>
cudaError_t launch_bias_common(const uint16_t* W2, const uint16_t* W2p, const uint16_t* W1,
                               const float* Ef, int table_rows, const int32_t* prev,
                               int prev_stride, int B, const int* n_rows, int V, int r, float* out,
                               int* err, cudaStream_t stream) {
  const int kc = draft_kchunk(r);
  CUtensorMap w2_map;
  memset(&w2_map, 0, sizeof(w2_map));
  if (!W2p && !encode_w2_map(&w2_map, W2, V, r, kc)) return cudaErrorInvalidValue;
  const int n_tiles = cdiv(V, kGemmTileV);
  // rows per pass: the smallest tensor-core N that holds the batch (the split mode's two
  // operand images fit 64 rows)
  if (B <= 16)
    return launch_bias_nb<16, Split>(w2_map, W2p, W1, Ef, table_rows, prev, prev_stride, B, n_rows,
                                     V, r, kc, n_tiles, out, err, stream);
  if (B <= 32)
    return launch_bias_nb<32, Split>(w2_map, W2p, W1, Ef, table_rows, prev, prev_stride, B, n_rows,
                                     V, r, kc, n_tiles, out, err, stream);
  if (B <= 64 || Split)
    return launch_bias_nb<64, Split>(w2_map, W2p, W1, Ef, table_rows, prev, prev_stride, B, n_rows,
                                     V, r, kc, n_tiles, out, err, stream);
  // up to 256 rows: one pass over W2 with N = 256 (two accumulators); a larger batch takes
  // passes of 128 rows, whose four accumulators keep the stores of one tile under the
  // contraction of the next (faster when the bias is store-bound)
  if (B > 128 && B <= 256)
    return launch_bias_nb<256, false>(w2_map, W2p, W1, Ef, table_rows, prev, prev_stride, B, n_rows,
                                      V, r, kc, n_tiles, out, err, stream);
  return launch_bias_nb<128, false>(w2_map, W2p, W1, Ef, table_rows, prev, prev_stride, B, n_rows,
                                    V, r, kc, n_tiles, out, err, stream);
}
}  // namespace

cudaError_t launch_bias_gemm(const uint16_t* W2, const uint16_t* W2p, const uint16_t* W1,
                             const int32_t* prev, int prev_stride, int B, const int* n_rows, int V,
                             int r, float* out, int* err, cudaStream_t stream) {
  return launch_bias_common<false>(W2, W2p, W1, nullptr, V, prev, prev_stride, B, n_rows, V, r, out,
                                   err, stream);
}

cudaError_t launch_bias_gemm_rows(const uint16_t* W2, const uint16_t* W2p, const float* Ef,
                                  int table_rows, const int32_t* prev, int B, const int* n_rows,
                                  int V, int r, float* out, int* err, cudaStream_t stream) {
  return launch_bias_common<true>(W2, W2p, nullptr, Ef, table_rows, prev, 1, B, n_rows, V, r, out,
                                  err, stream);
}

}  // namespace dspark
