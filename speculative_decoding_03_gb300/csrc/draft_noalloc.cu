// dspark_draft_noalloc: the draft of one step without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they draft: a serving
// loop whose memory is fully reserved by its own pool, a plugin inside a host framework
// that hands out only the input and output buffers, or code that runs where a
// cudaMalloc would synchronise the device or fail.  For them the draft kernel's scratch
// (per-CTA partial results, the grid-barrier counter and the argmax keys) lives in a
// fixed array inside this library instead of a workspace.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes (about 2.5 MB); the
// CUDA runtime creates it on every GPU that loads the library and keeps it until the
// process exits.  It serves batches of at most kNoAllocMaxB requests and kNoAllocMaxGamma
// positions.  Host code cannot use the array's name as a device address, so the first
// call on each device looks up its address with cudaGetSymbolAddress (that device
// current) and caches it; make that first call before any stream capture.
//
// Every call shares the one array, so calls whose kernels overlap on the GPU (several
// streams, several host threads) race and must be serialised by the caller.  The counter
// and keys that must start at zero are cleared by each call on its stream; the rest is
// overwritten before it is read.  Device-side checks (an anchor id out of range, a wait
// that ran out) are recorded in the array but not reported by this entry point; use
// dspark_draft with a workspace to read them.
#include <mutex>

#include "internal.h"

namespace dspark {
namespace {

constexpr int kNoAllocMaxB = 256;
constexpr int kNoAllocMaxGamma = 32;
// status word (256 B) + the draft region for the largest batch served
constexpr size_t kNoAllocScratchBytes =
    256 + ((3ull * kNoAllocMaxB * kDraftMaxCtas * sizeof(RowState) + 255) / 256) * 256 + 256 +
    ((8ull * kNoAllocMaxB * kNoAllocMaxGamma + 255) / 256) * 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned_ptr(const void* p, uintptr_t a) {
  return p && (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" dspark_status dspark_draft_noalloc(const float* U, const uint16_t* W1,
                                              const uint16_t* W2, const int32_t* anchor, int B,
                                              int gamma, int V, int r, uint64_t seed,
                                              int32_t* tokens, float* q_tok, float* row_max,
                                              float* row_sumexp, cudaStream_t stream) {
  if (B < 1 || gamma < 1 || V < 8 || r < 1) return DSPARK_ERR_INVALID_ARG;
  if (B > kNoAllocMaxB || gamma > kNoAllocMaxGamma) return DSPARK_ERR_UNSUPPORTED;
  if (V % 8 != 0 || r % 16 != 0 || r > 256 || r < 16) return DSPARK_ERR_UNSUPPORTED;
  if (!aligned_ptr(U, 16) || !aligned_ptr(W1, 16) || !aligned_ptr(W2, 16) ||
      !aligned_ptr(anchor, 4) || !aligned_ptr(tokens, 4) || !aligned_ptr(q_tok, 4) ||
      !aligned_ptr(row_max, 4) || !aligned_ptr(row_sumexp, 4))
    return DSPARK_ERR_INVALID_ARG;
  if (256 + draft_region_bytes(B, gamma) > kNoAllocScratchBytes) return DSPARK_ERR_UNSUPPORTED;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return DSPARK_ERR_CUDA;
  char* scratch = static_cast<char*>(base);
  int* err = reinterpret_cast<int*>(scratch);
  if (cudaMemsetAsync(err, 0, sizeof(int), stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  return draft_status(launch_draft_fused(W1, W2, U, anchor, B, gamma, V, r, seed, tokens, q_tok,
                                         row_max, row_sumexp, scratch + 256, err, stream));
}
