// Packed Markov-head weights: W2 [r, V] rearranged once into the exact shared-memory
// images the draft kernel's tensor-core operand uses, so that the draft streams each
// 16 KB operand chunk with one contiguous bulk copy.
//
// Why: the draft kernel reads, for every 128-row vocabulary tile and every position, the
// W2^T tile (MN-major, 128-byte swizzle).  Read straight from W2 [r, V] a tile is r rows of
// 2 x 128 bytes, 2V bytes apart, spread over all of W2; the packed copy makes every tile one
// contiguous block (n_kchunks x 2 x kc x 128 bytes).
//
// Layout of W2p (16-byte units), for tile t, K-chunk i (kc rank rows each), half h (the
// vocabulary rows t*128 + 64h .. +63), rank row kl inside the chunk, physical 16-byte slot s:
//   W2p[t][i][h][kl][s] = W2[i*kc + kl][t*128 + 64h + 8c .. +7],  c = s ^ (kl % 8)
// (the 128-byte swizzle: logical 16-byte chunk c of a 128-byte line kl sits in slot
// c ^ (kl mod 8)); vocabulary rows >= V are zero.
#include "internal.h"

namespace dspark {
namespace {

__global__ void pack_w2_kernel(const uint16_t* __restrict__ W2, int V, int r, int kc,
                               int n_tiles, uint4* __restrict__ W2p) {
  const int n_kchunks = r / kc;
  const size_t total = (size_t)n_tiles * r * 2 * 8;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int slot = (int)(idx & 7);
    size_t rest = idx >> 3;
    const int kl = (int)(rest % kc);
    rest /= kc;
    const int h = (int)(rest & 1);
    rest >>= 1;
    const int i = (int)(rest % n_kchunks);
    const int t = (int)(rest / n_kchunks);
    const int c = slot ^ (kl & 7);
    const int k = i * kc + kl;
    const int v = t * 128 + h * 64 + c * 8;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (v < V) val = __ldg(reinterpret_cast<const uint4*>(W2 + (size_t)k * V + v));
    W2p[idx] = val;
  }
}

bool aligned_ptr(const void* p, uintptr_t a) {
  return p && (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

dspark_status check_wshape(int V, int r) {
  if (V < 8 || r < 1) return DSPARK_ERR_INVALID_ARG;
  if (V % 8 != 0 || r % 16 != 0 || r > 256 || r < 16) return DSPARK_ERR_UNSUPPORTED;
  return DSPARK_OK;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" {

size_t dspark_packed_w2_bytes(int V, int r) {
  if (check_wshape(V, r) != DSPARK_OK) return 0;
  return (size_t)cdiv(V, kGemmTileV) * kGemmTileV * (size_t)r * sizeof(uint16_t);
}

dspark_status dspark_pack_w2(const uint16_t* W2, int V, int r, uint16_t* W2p, size_t W2p_bytes,
                             cudaStream_t stream) {
  dspark_status st = check_wshape(V, r);
  if (st != DSPARK_OK) return st;
  if (!aligned_ptr(W2, 16) || !aligned_ptr(W2p, 16)) return DSPARK_ERR_INVALID_ARG;
  if (W2p_bytes < dspark_packed_w2_bytes(V, r)) return DSPARK_ERR_INVALID_ARG;
  const int n_tiles = cdiv(V, kGemmTileV);
  pack_w2_kernel<<<1216, 256, 0, stream>>>(W2, V, r, draft_kchunk(r), n_tiles,
                                           reinterpret_cast<uint4*>(W2p));
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

dspark_status dspark_draft_packed(const float* U, const uint16_t* W1, const uint16_t* W2p,
                                  const int32_t* anchor, int B, int gamma, int V, int r,
                                  uint64_t seed, int32_t* tokens, float* q_tok, float* row_max,
                                  float* row_sumexp, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
  if (B < 1 || gamma < 1) return DSPARK_ERR_INVALID_ARG;
  if (B >= 65536 || gamma > 32 || (long long)B * (gamma + 1) >= (1LL << 21))
    return DSPARK_ERR_UNSUPPORTED;
  dspark_status st = check_wshape(V, r);
  if (st != DSPARK_OK) return st;
  if (!aligned_ptr(U, 16) || !aligned_ptr(W1, 16) || !aligned_ptr(W2p, 16) ||
      !aligned_ptr(anchor, 4) || !aligned_ptr(tokens, 4) || !aligned_ptr(q_tok, 4) ||
      !aligned_ptr(row_max, 4) || !aligned_ptr(row_sumexp, 4))
    return DSPARK_ERR_INVALID_ARG;
  const Plan p = make_plan(B, gamma, V, r, 0);
  if (!aligned_ptr(workspace, 256) || workspace_bytes < p.total) return DSPARK_ERR_INVALID_ARG;
  return draft_status(launch_draft_fused_packed(W1, W2p, U, anchor, B, gamma, V, r, seed, tokens,
                                                q_tok, row_max, row_sumexp,
                                                ws_at<char>(workspace, p.off_draft),
                                                ws_at<int>(workspace, p.off_err), stream));
}

}  // extern "C"
