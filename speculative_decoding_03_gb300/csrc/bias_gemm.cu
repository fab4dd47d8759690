// Markov transition bias on the tensor cores.
//
// billytse.dev DSpark page, section 3.3: the first-order Markov head's bias for every
// request is B(x_{k-1}, .) = W1[x_{k-1}] W2, rank r.  For a whole batch this is the
// contraction  bias^T [V, B] = W2^T [V, r] x E^T [r, B]  with E[b] = W1[prev_b].
//
// One CTA computes a 128-row vocabulary tile for one batch chunk of NB requests:
//   A = W2^T tile (M = 128 vocabulary rows, K = r), MN-major in shared memory, brought in
//       by two TMA tile loads of 64 columns x r rows with the 128-byte swizzle;
//   B = E^T (N = NB requests, K = r), K-major, gathered from W1 rows by the CTA's threads
//       and written in the same 128-byte-swizzled layout;
//   D = fp32 accumulators in tensor memory (128 lanes x NB columns), issued by one thread
//       as r / 16 tcgen05.mma instructions (kind::f16, bf16 inputs);
// then the four warps read D back (lane = vocabulary row) and store bias[b][v] with
// coalesced 128-byte rows.
#include "internal.h"
#include "sm100_ptx.cuh"

namespace dspark {
namespace {

using namespace sm100;

__global__ void __launch_bounds__(128) bias_gemm_kernel(const __grid_constant__ CUtensorMap w2_map,
                                                        const uint16_t* __restrict__ W1,
                                                        const int32_t* __restrict__ prev,
                                                        int prev_stride, int B, int V, int r,
                                                        int NB, uint32_t tmem_cols,
                                                        float* __restrict__ out, int* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_base_s;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;                          // two 64-row blocks of r x 128 bytes
  uint8_t* sB = sA + 2 * (size_t)r * 128;      // ceil(r/64) K-blocks of NB x 128 bytes

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int v0 = blockIdx.x * kGemmTileV;
  const int b0 = blockIdx.y * NB;

  if (tid == 0) {
    prefetch_tensormap(&w2_map);
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_base_s;

  if (tid == 0) {
    const uint64_t pol = policy_evict_last();
    mbar_arrive_expect_tx(&bar_tma, 2u * (uint32_t)r * 128u);
    tma_load_2d(sA, &w2_map, &bar_tma, v0, 0, pol);
    tma_load_2d(sA + (size_t)r * 128, &w2_map, &bar_tma, v0 + 64, 0, pol);
  }
  // the W2 tile is an input; the request tokens (prev) may come from the previous kernel
  pdl_wait();
  pdl_launch_dependents();

  // Gather E = W1[prev_b] (rows b0 .. b0+NB-1) as the K-major B operand: row n is 128-byte
  // lines of 64 bf16 per K-block, 16-byte chunk c of row n stored at chunk c ^ (n % 8).
  const int kchunks = r >> 3;  // 16-byte chunks per W1 row
  for (int idx = tid; idx < NB * kchunks; idx += blockDim.x) {
    const int n = idx / kchunks, c = idx - n * kchunks;
    const int b = b0 + n;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (b < B) {
      const int p = prev[(size_t)b * prev_stride];
      if (p >= 0 && p < V) {
        val = __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)p * r) + c);
      } else if (p != -1) {
        set_device_error(err, DSPARK_ERR_DEVICE_CHECK);
      }
    }
    const int kb = c >> 3, cc = c & 7;
    *reinterpret_cast<uint4*>(sB + (size_t)kb * NB * 128 + (size_t)n * 128 + ((cc ^ (n & 7)) << 4)) =
        val;
  }
  fence_proxy_async_smem();
  __syncthreads();

  if (tid == 0) {
    if (mbar_wait(&bar_tma, 0)) {
      tc_fence_after_sync();
      const uint32_t idesc = idesc_bf16_f32(128, NB, /*A MN-major*/ 1, /*B K-major*/ 0);
      const uint32_t a0 = smem_u32(sA), b0s = smem_u32(sB);
      for (int kk = 0; kk < (r >> 4); ++kk) {
        // A: 16 K-rows = two 8-row groups (SBO = 1024 B); the second 64-row block at LBO
        const uint64_t ad = smem_desc(a0 + (uint32_t)kk * 2048u, (uint32_t)r * 128u, 1024u,
                                      kSwizzle128B);
        // B: K-block kk/4, 32-byte step inside the 128-byte swizzle atom; 8-row groups 1 KB
        const uint64_t bd = smem_desc(b0s + (uint32_t)(kk >> 2) * (uint32_t)NB * 128u +
                                          (uint32_t)(kk & 3) * 32u,
                                      16u, 1024u, kSwizzle128B);
        umma_bf16_f32(tmem_base, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
    } else {
      set_device_error(err, DSPARK_ERR_TIMEOUT);
    }
    umma_commit(&bar_mma);
  }

  // Epilogue: warp w reads TMEM lanes 32w..32w+31 (vocabulary rows v0 + 32w + lane).
  const bool ok = mbar_wait(&bar_mma, 0);
  if (!ok && lane == 0) set_device_error(err, DSPARK_ERR_TIMEOUT);
  tc_fence_after_sync();
  const int v = v0 + warp * 32 + lane;
  const uint32_t trow = tmem_base + ((uint32_t)(warp * 32) << 16);
  for (int c0 = 0; c0 < NB; c0 += 16) {
    float vals[16];
    tmem_ld_32x32b_x16(trow + (uint32_t)c0, vals);
    tmem_ld_wait();
    if (ok && v < V) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int b = b0 + c0 + j;
        if (b < B) out[(size_t)b * V + v] = vals[j];
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_base, tmem_cols);
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

cudaError_t launch_bias_gemm(const CUtensorMap* w2_map, const uint16_t* W1, const int32_t* prev,
                             int prev_stride, int B, int V, int r, float* out, int* err,
                             cudaStream_t stream) {
  const int NB = gemm_chunk(B);
  uint32_t cols = 32;
  while ((int)cols < NB) cols <<= 1;
  const size_t smem = gemm_smem_bytes(r, NB);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(bias_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(cdiv(V, kGemmTileV), cdiv(B, NB));
  return launch_pdl(bias_gemm_kernel, grid, dim3(128), smem, stream, *w2_map, W1, prev, prev_stride,
                    B, V, r, NB, cols, out, err);
}

}  // namespace dspark
