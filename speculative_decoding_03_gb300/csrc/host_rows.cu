// The target rows a verification reads, fetched from host memory.
//
// billytse.dev DSpark page, section 1: the target scores the scheduled prefix, so
// verification reads T[b, j] for the verified positions j < l_b and the row the final
// token is drawn from, T[b, l_b] at the latest (the bonus row when everything is
// accepted); rows beyond l_b are never read.  When a step's target logits arrive in host
// memory, copying only those rows over the host link (the step's bottleneck: it moves
// about 0.2 TB/s, HBM 30 times that) instead of the whole [B][gamma + 1][V] block saves
// the unread rows' bytes.  Which rows are needed is known only on the device (the
// scheduler's l), so the copy is a kernel that reads the source through the device's
// mapping of host memory: one item is a 32 KB segment of a row, every thread keeps eight
// 16-byte loads in flight, and items of rows beyond l_b return at once.
#include "internal.h"

namespace dspark {
namespace {

constexpr int kRowCopyThreads = 256;
constexpr int kRowCopyVec = 8;                                   // 16-byte loads in flight
constexpr int kRowSeg4 = kRowCopyThreads * kRowCopyVec;          // float4 per item (32 KB)

__global__ void __launch_bounds__(kRowCopyThreads) copy_target_rows_kernel(
    const float4* __restrict__ src, float4* __restrict__ dst, const int32_t* __restrict__ ell,
    int B, int gamma, int V4, int n_seg, int* err) {
  pdl_wait();                   // l comes from the scheduler
  pdl_launch_dependents();
  const long long n_items = (long long)B * (gamma + 1) * n_seg;
  for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const long long row = item / n_seg;
    const int seg = (int)(item - row * n_seg);
    const int b = (int)(row / (gamma + 1)), j = (int)(row - (long long)b * (gamma + 1));
    int L = ell[b];
    if (L < 0 || L > gamma) {
      if (threadIdx.x == 0 && j == 0 && seg == 0) set_device_error(err, DSPARK_ERR_DEVICE_CHECK);
      L = L < 0 ? 0 : gamma;
    }
    if (j > L) continue;
    const long long base = row * V4 + (long long)seg * kRowSeg4;
    const int n4 = V4 - seg * kRowSeg4 < kRowSeg4 ? V4 - seg * kRowSeg4 : kRowSeg4;
    float4 v[kRowCopyVec];
#pragma unroll
    for (int u = 0; u < kRowCopyVec; ++u) {
      const int q = threadIdx.x + u * kRowCopyThreads;
      if (q < n4) v[u] = __ldcs(src + base + q);
    }
#pragma unroll
    for (int u = 0; u < kRowCopyVec; ++u) {
      const int q = threadIdx.x + u * kRowCopyThreads;
      if (q < n4) dst[base + q] = v[u];
    }
  }
}

}  // namespace

cudaError_t launch_copy_target_rows(const float* T_src, float* T, const int32_t* ell, int B,
                                    int gamma, int V, int* err, cudaStream_t stream) {
  const int V4 = V / 4;
  const int n_seg = cdiv(V4, kRowSeg4);
  int sms = 0, dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long n_items = (long long)B * (gamma + 1) * n_seg;
  const long long want = 4LL * sms;
  const int grid = (int)(n_items < want ? n_items : want);
  return launch_pdl(copy_target_rows_kernel, dim3(grid), dim3(kRowCopyThreads), 0, stream,
                    reinterpret_cast<const float4*>(T_src), reinterpret_cast<float4*>(T), ell, B,
                    gamma, V4, n_seg, err);
}

}  // namespace dspark
