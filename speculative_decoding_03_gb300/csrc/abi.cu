// extern "C" entry points of libdspark: host-side argument validation, workspace carving
// and the launch sequence of each call.  See include/dspark.h for the contract.
#include <stdint.h>

#include "internal.h"

using namespace dspark;

namespace {

bool aligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

dspark_status check_shape(int B, int gamma, int V, int r, int H) {
  if (B < 1 || gamma < 1 || V < 8 || r < 1 || H < 0) return DSPARK_ERR_INVALID_ARG;
  if (B >= 65536 || gamma > 32) return DSPARK_ERR_UNSUPPORTED;
  if ((long long)B * (gamma + 1) >= (1LL << 21)) return DSPARK_ERR_UNSUPPORTED;
  if (V % 8 != 0 || r % 16 != 0 || r > 256 || r < 16 || H % 4 != 0) return DSPARK_ERR_UNSUPPORTED;
  return DSPARK_OK;
}

dspark_status check_ws(void* ws, size_t bytes, const Plan& p) {
  if (!aligned(ws, 256)) return DSPARK_ERR_INVALID_ARG;
  if (bytes < p.total) return DSPARK_ERR_INVALID_ARG;
  return DSPARK_OK;
}

}  // namespace

extern "C" {

const char* dspark_status_string(dspark_status s) {
  switch (s) {
    case DSPARK_OK: return "DSPARK_OK";
    case DSPARK_ERR_INVALID_ARG: return "DSPARK_ERR_INVALID_ARG";
    case DSPARK_ERR_UNSUPPORTED: return "DSPARK_ERR_UNSUPPORTED";
    case DSPARK_ERR_CUDA: return "DSPARK_ERR_CUDA";
    case DSPARK_ERR_TIMEOUT: return "DSPARK_ERR_TIMEOUT";
    case DSPARK_ERR_DEVICE_CHECK: return "DSPARK_ERR_DEVICE_CHECK";
  }
  return "DSPARK_ERR_UNKNOWN";
}

size_t dspark_workspace_bytes(int B, int gamma, int V, int r, int H) {
  if (check_shape(B, gamma, V, r, H) != DSPARK_OK) return 0;
  return make_plan(B, gamma, V, r, H).total;
}

dspark_status dspark_markov_bias(const uint16_t* W1, const uint16_t* W2, const int32_t* prev,
                                 int prev_stride, int B, int V, int r, float* out, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  if (B < 1 || prev_stride < 1) return DSPARK_ERR_INVALID_ARG;
  dspark_status st = check_shape(B, 1, V, r, 0);
  if (st != DSPARK_OK) return st;
  if (!aligned(W1, 16) || !aligned(W2, 16) || !aligned(prev, 4) || !aligned(out, 4))
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || workspace_bytes < 256) return DSPARK_ERR_INVALID_ARG;
  if (launch_bias_gemm(W2, nullptr, W1, prev, prev_stride, B, nullptr, V, r, out,
                       ws_at<int>(workspace, 0), stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_draft(const float* U, const uint16_t* W1, const uint16_t* W2,
                           const int32_t* anchor, int B, int gamma, int V, int r, uint64_t seed,
                           int32_t* tokens, float* q_tok, float* row_max, float* row_sumexp,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  dspark_status st = check_shape(B, gamma, V, r, 0);
  if (st != DSPARK_OK) return st;
  if (!aligned(U, 16) || !aligned(W1, 16) || !aligned(W2, 16) || !aligned(anchor, 4) ||
      !aligned(tokens, 4) || !aligned(q_tok, 4) || !aligned(row_max, 4) || !aligned(row_sumexp, 4))
    return DSPARK_ERR_INVALID_ARG;
  const Plan p = make_plan(B, gamma, V, r, 0);
  if ((st = check_ws(workspace, workspace_bytes, p)) != DSPARK_OK) return st;

  return draft_status(launch_draft_fused(W1, W2, U, anchor, B, gamma, V, r, seed, tokens, q_tok,
                                         row_max, row_sumexp, ws_at<char>(workspace, p.off_draft),
                                         ws_at<int>(workspace, p.off_err), stream));
}

dspark_status dspark_confidence(const float* h, const int32_t* anchor, const int32_t* tokens,
                                const uint16_t* W1, const float* w_c, float b_c, int B, int gamma,
                                int H, int r, int V, float* c, float* a, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  dspark_status st = check_shape(B, gamma, V, r, H);
  if (st != DSPARK_OK) return st;
  if (!aligned(h, 16) || !aligned(w_c, 16) || !aligned(W1, 16) || !aligned(anchor, 4) ||
      !aligned(tokens, 4) || !aligned(c, 4) || !aligned(a, 4))
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || workspace_bytes < 256) return DSPARK_ERR_INVALID_ARG;
  int* err = ws_at<int>(workspace, 0);
  if (launch_confidence(h, anchor, tokens, W1, w_c, b_c, B, gamma, H, r, V, c, a, err, stream) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_confidence_schedule(const float* h, const int32_t* anchor,
                                         const int32_t* tokens, const uint16_t* W1,
                                         const float* w_c, float b_c, int B, int gamma, int H,
                                         int r, int V, const float* sps, int sps_len, float* c,
                                         float* a, int32_t* ell, int32_t* B_total,
                                         double* theta, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream) {
  dspark_status st = check_shape(B, gamma, V, r, H);
  if (st != DSPARK_OK) return st;
  if ((long long)B * gamma > kMaxScheduleItems) return DSPARK_ERR_UNSUPPORTED;
  if ((long long)sps_len < (long long)B * (gamma + 1) + 1) return DSPARK_ERR_INVALID_ARG;
  if (!aligned(h, 16) || !aligned(w_c, 16) || !aligned(W1, 16) || !aligned(anchor, 4) ||
      !aligned(tokens, 4) || !aligned(c, 4) || !aligned(a, 4) || !aligned(sps, 4) ||
      !aligned(ell, 4) || !aligned(B_total, 4) || !aligned(theta, 8))
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || workspace_bytes < 256) return DSPARK_ERR_INVALID_ARG;
  int* err = ws_at<int>(workspace, 0);
  // the CTA counter shares the status word's 256-byte slot (byte 128; zero between calls)
  unsigned int* done = ws_at<unsigned int>(workspace, 128);
  if (launch_confidence_schedule(h, anchor, tokens, W1, w_c, b_c, B, gamma, H, r, V, sps, c, a,
                                 ell, B_total, theta, done, err, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_draft_confidence_schedule(
    const float* U, const uint16_t* W1, const uint16_t* W2p, const int32_t* anchor, const float* h,
    const float* w_c, float b_c, const float* sps, int sps_len, int B, int gamma, int V, int r, int H,
    uint64_t seed, int32_t* tokens, float* q_tok, float* row_max, float* row_sumexp, float* c,
    float* a, int32_t* ell, int32_t* B_total, double* theta, void* workspace,
    size_t workspace_bytes, cudaStream_t stream) {
  dspark_status st = check_shape(B, gamma, V, r, H);
  if (st != DSPARK_OK) return st;
  if ((long long)B * gamma > kMaxScheduleItems) return DSPARK_ERR_UNSUPPORTED;
  if ((long long)sps_len < (long long)B * (gamma + 1) + 1) return DSPARK_ERR_INVALID_ARG;
  if (!aligned(U, 16) || !aligned(W1, 16) || !aligned(W2p, 16) || !aligned(anchor, 4) ||
      !aligned(h, 16) || !aligned(w_c, 16) || !aligned(sps, 4) || !aligned(tokens, 4) ||
      !aligned(q_tok, 4) || !aligned(row_max, 4) || !aligned(row_sumexp, 4) || !aligned(c, 4) ||
      !aligned(a, 4) || !aligned(ell, 4) || !aligned(B_total, 4) || !aligned(theta, 8))
    return DSPARK_ERR_INVALID_ARG;
  const Plan p = make_plan(B, gamma, V, r, H);
  if ((st = check_ws(workspace, workspace_bytes, p)) != DSPARK_OK) return st;
  DraftStepArgs step;
  step.h = h; step.w_c = w_c; step.b_c = b_c; step.H = H; step.c = c; step.a = a;
  step.sps = sps; step.ell = ell; step.B_total = B_total; step.theta = theta;
  step.sched_keys = ws_at<unsigned long long>(workspace, p.off_sched);
  int* err = ws_at<int>(workspace, p.off_err);
  const cudaError_t e = launch_draft_lanes(W1, nullptr, W2p, U, anchor, B, gamma, V, r, seed,
                                           false, tokens, q_tok, row_max, row_sumexp,
                                           ws_at<char>(workspace, p.off_draft), err, stream, &step);
  if (e == cudaErrorNotSupported) return DSPARK_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  // batches beyond the draft's in-kernel scheduler: the scheduler kernel follows
  if ((long long)B * gamma > draft_fused_schedule_limit() &&
      launch_schedule(a, B, gamma, sps, nullptr, nullptr, ell, B_total, theta, err, stream) !=
          cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_schedule(const float* a, int R, int gamma, const float* sps, int sps_len,
                              int32_t* ell, int32_t* B_total, double* theta, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  if (R < 1 || gamma < 1) return DSPARK_ERR_INVALID_ARG;
  if (R >= 65536 || gamma > 32 || (long long)R * gamma > kMaxScheduleItems ||
      (long long)R * (gamma + 1) >= (1LL << 21))
    return DSPARK_ERR_UNSUPPORTED;
  if ((long long)sps_len < (long long)R * (gamma + 1) + 1) return DSPARK_ERR_INVALID_ARG;
  if (!aligned(a, 4) || !aligned(sps, 4) || !aligned(ell, 4) || !aligned(B_total, 4) ||
      !aligned(theta, 8))
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || workspace_bytes < 256) return DSPARK_ERR_INVALID_ARG;
  int* err = ws_at<int>(workspace, 0);
  if (launch_schedule(a, R, gamma, sps, nullptr, nullptr, ell, B_total, theta, err, stream) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_schedule_async(const float* a, int R, int gamma, const float* sps,
                                    int sps_len, const int32_t* K_in, int32_t* K_out,
                                    int32_t* ell, int32_t* B_total, double* theta,
                                    void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
  if (R < 1 || gamma < 1) return DSPARK_ERR_INVALID_ARG;
  if (R >= 65536 || gamma > 32 || (long long)R * gamma > kMaxScheduleItems ||
      (long long)R * (gamma + 1) >= (1LL << 21))
    return DSPARK_ERR_UNSUPPORTED;
  if ((long long)sps_len < (long long)R * (gamma + 1) + 1) return DSPARK_ERR_INVALID_ARG;
  if (!aligned(a, 4) || !aligned(sps, 4) || !aligned(ell, 4) || !aligned(B_total, 4) ||
      !aligned(theta, 8) || (K_in && !aligned(K_in, 4)) || (K_out && !aligned(K_out, 4)))
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || workspace_bytes < 256) return DSPARK_ERR_INVALID_ARG;
  int* err = ws_at<int>(workspace, 0);
  if (launch_schedule(a, R, gamma, sps, K_in, K_out, ell, B_total, theta, err, stream) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_schedule_threshold(const float* a, int R, int gamma, float threshold,
                                        int32_t* ell, int32_t* B_total, cudaStream_t stream) {
  if (R < 1 || gamma < 1) return DSPARK_ERR_INVALID_ARG;
  if (R >= 65536 || gamma > 32) return DSPARK_ERR_UNSUPPORTED;
  if (threshold != threshold) return DSPARK_ERR_INVALID_ARG;     // NaN
  if (!aligned(a, 4) || !aligned(ell, 4) || !aligned(B_total, 4)) return DSPARK_ERR_INVALID_ARG;
  if (launch_schedule_threshold(a, R, gamma, threshold, ell, B_total, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_draft_greedy(const float* U, const uint16_t* W1, const uint16_t* W2,
                                  const uint16_t* W2p, const int32_t* anchor, int B, int gamma,
                                  int V, int r, int32_t* tokens, float* q_tok, float* row_max,
                                  float* row_sumexp, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
  if ((W2 == nullptr) == (W2p == nullptr)) return DSPARK_ERR_INVALID_ARG;
  dspark_status st = check_shape(B, gamma, V, r, 0);
  if (st != DSPARK_OK) return st;
  if (!aligned(U, 16) || !aligned(W1, 16) || !aligned(W2 ? W2 : W2p, 16) || !aligned(anchor, 4) ||
      !aligned(tokens, 4) || !aligned(q_tok, 4) || !aligned(row_max, 4) || !aligned(row_sumexp, 4))
    return DSPARK_ERR_INVALID_ARG;
  const Plan p = make_plan(B, gamma, V, r, 0);
  if ((st = check_ws(workspace, workspace_bytes, p)) != DSPARK_OK) return st;
  return draft_status(launch_draft_fused_greedy(W1, W2, W2p, U, anchor, B, gamma, V, r, tokens,
                                                q_tok, row_max, row_sumexp,
                                                ws_at<char>(workspace, p.off_draft),
                                                ws_at<int>(workspace, p.off_err), stream));
}

dspark_status dspark_verify_greedy(const float* T, const int32_t* tokens, const int32_t* ell,
                                   int B, int gamma, int V, uint64_t seed, int32_t* accept_len,
                                   int32_t* out_tokens, int32_t* n_out, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
  // the workspace layout does not depend on r or H: any supported r gives the same plan
  dspark_status st = check_shape(B, gamma, V, 16, 0);
  if (st != DSPARK_OK) return st;
  if (!aligned(T, 16) || !aligned(tokens, 4) || !aligned(ell, 4) || !aligned(accept_len, 4) ||
      !aligned(out_tokens, 4) || !aligned(n_out, 4))
    return DSPARK_ERR_INVALID_ARG;
  const Plan p = make_plan(B, gamma, V, 16, 0);
  if ((st = check_ws(workspace, workspace_bytes, p)) != DSPARK_OK) return st;
  if (launch_verify(p, T, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, tokens, nullptr,
                    nullptr, nullptr, ell, seed, accept_len, out_tokens, n_out, workspace, stream) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

}  // extern "C"

namespace {

// dspark_verify and dspark_verify_packed: W2 xor W2p (the packed tile images) is given
dspark_status verify_common(const float* T, const float* U, const uint16_t* W1, const uint16_t* W2,
                            const uint16_t* W2p, const int32_t* anchor, const int32_t* tokens,
                            const float* q_tok, const float* row_max, const float* row_sumexp,
                            const int32_t* ell, int B, int gamma, int V, int r, uint64_t seed,
                            int32_t* accept_len, int32_t* out_tokens, int32_t* n_out,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  dspark_status st = check_shape(B, gamma, V, r, 0);
  if (st != DSPARK_OK) return st;
  if (!aligned(T, 16) || !aligned(U, 16) || !aligned(W1, 16) || !aligned(W2 ? W2 : W2p, 16) ||
      !aligned(anchor, 4) || !aligned(tokens, 4) || !aligned(q_tok, 4) || !aligned(row_max, 4) ||
      !aligned(row_sumexp, 4) || !aligned(ell, 4) || !aligned(accept_len, 4) ||
      !aligned(out_tokens, 4) || !aligned(n_out, 4))
    return DSPARK_ERR_INVALID_ARG;
  const Plan p = make_plan(B, gamma, V, r, 0);
  if ((st = check_ws(workspace, workspace_bytes, p)) != DSPARK_OK) return st;
  if (launch_verify(p, T, U, W1, W2, W2p, nullptr, anchor, tokens, q_tok, row_max, row_sumexp, ell,
                    seed, accept_len, out_tokens, n_out, workspace, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

}  // namespace

extern "C" {

dspark_status dspark_verify(const float* T, const float* U, const uint16_t* W1, const uint16_t* W2,
                            const int32_t* anchor, const int32_t* tokens, const float* q_tok,
                            const float* row_max, const float* row_sumexp, const int32_t* ell,
                            int B, int gamma, int V, int r, uint64_t seed, int32_t* accept_len,
                            int32_t* out_tokens, int32_t* n_out, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
  if (!W2) return DSPARK_ERR_INVALID_ARG;
  return verify_common(T, U, W1, W2, nullptr, anchor, tokens, q_tok, row_max, row_sumexp, ell, B,
                       gamma, V, r, seed, accept_len, out_tokens, n_out, workspace,
                       workspace_bytes, stream);
}

dspark_status dspark_verify_packed(const float* T, const float* U, const uint16_t* W1,
                                   const uint16_t* W2p, const int32_t* anchor,
                                   const int32_t* tokens, const float* q_tok,
                                   const float* row_max, const float* row_sumexp,
                                   const int32_t* ell, int B, int gamma, int V, int r,
                                   uint64_t seed, int32_t* accept_len, int32_t* out_tokens,
                                   int32_t* n_out, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
  if (!W2p) return DSPARK_ERR_INVALID_ARG;
  return verify_common(T, U, W1, nullptr, W2p, anchor, tokens, q_tok, row_max, row_sumexp, ell, B,
                       gamma, V, r, seed, accept_len, out_tokens, n_out, workspace,
                       workspace_bytes, stream);
}

size_t dspark_rnn_packed_bytes(int r) {
  if (r < 16 || r > 256 || r % 16 != 0) return 0;
  return (size_t)3 * r * 2 * r * sizeof(uint16_t);
}

dspark_status dspark_rnn_pack(const uint16_t* W_rnn, int r, uint16_t* Wrec, size_t Wrec_bytes,
                              cudaStream_t stream) {
  const size_t need = dspark_rnn_packed_bytes(r);
  if (need == 0) return DSPARK_ERR_UNSUPPORTED;
  if (!aligned(W_rnn, 16) || !aligned(Wrec, 16) || Wrec_bytes < need) return DSPARK_ERR_INVALID_ARG;
  if (launch_rnn_pack(W_rnn, r, Wrec, stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_rnn_project(const float* h, const uint16_t* W_rnn, const float* b_rnn,
                                 int B, int gamma, int H, int r, float* hp, cudaStream_t stream) {
  if (B < 1 || gamma < 1 || H < 1) return DSPARK_ERR_INVALID_ARG;
  if (r < 16 || r > 256 || r % 16 != 0 || H % 4 != 0 || gamma > 32 || B >= 65536)
    return DSPARK_ERR_UNSUPPORTED;
  if (!aligned(h, 16) || !aligned(W_rnn, 16) || !aligned(b_rnn, 16) || !aligned(hp, 16))
    return DSPARK_ERR_INVALID_ARG;
  if (launch_rnn_project(h, W_rnn, b_rnn, B * gamma, H, r, hp, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_draft_rnn(const float* U, const uint16_t* W1, const uint16_t* W2,
                               const uint16_t* W2p, const uint16_t* Wrec, const float* hp,
                               const int32_t* anchor, int B, int gamma, int V, int r,
                               uint64_t seed, int greedy, int32_t* tokens, float* q_tok,
                               float* row_max, float* row_sumexp, float* E, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  if ((W2 == nullptr) == (W2p == nullptr)) return DSPARK_ERR_INVALID_ARG;
  dspark_status st = check_shape(B, gamma, V, r, 0);
  if (st != DSPARK_OK) return st;
  if (!aligned(U, 16) || !aligned(W1, 16) || !aligned(W2 ? W2 : W2p, 16) || !aligned(Wrec, 16) ||
      !aligned(hp, 16) || !aligned(E, 16) || !aligned(anchor, 4) || !aligned(tokens, 4) ||
      !aligned(q_tok, 4) || !aligned(row_max, 4) || !aligned(row_sumexp, 4))
    return DSPARK_ERR_INVALID_ARG;
  const Plan p = make_plan(B, gamma, V, r, 0);
  if ((st = check_ws(workspace, workspace_bytes, p)) != DSPARK_OK) return st;
  RnnDraftArgs rnn;
  rnn.Wrec = Wrec;
  rnn.hp = hp;
  rnn.E_all = E;
  rnn.state = ws_at<float>(workspace, p.off_rnn_state);
  rnn.E_hl = reinterpret_cast<uint16_t*>(rnn.state + (size_t)kRnnStateCopies * 2 * B * r);
  if (launch_draft_fused_rnn(W1, W2, W2p, U, anchor, B, gamma, V, r, seed, greedy != 0, rnn, tokens,
                             q_tok, row_max, row_sumexp, ws_at<char>(workspace, p.off_draft),
                             ws_at<int>(workspace, p.off_err), stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_verify_rnn(const float* T, const float* U, const float* E, const uint16_t* W2,
                                const uint16_t* W2p, const int32_t* tokens, const float* q_tok,
                                const float* row_max, const float* row_sumexp, const int32_t* ell,
                                int B, int gamma, int V, int r, uint64_t seed,
                                int32_t* accept_len, int32_t* out_tokens, int32_t* n_out,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if ((W2 == nullptr) == (W2p == nullptr)) return DSPARK_ERR_INVALID_ARG;
  dspark_status st = check_shape(B, gamma, V, r, 0);
  if (st != DSPARK_OK) return st;
  if (!aligned(T, 16) || !aligned(U, 16) || !aligned(E, 16) || !aligned(W2 ? W2 : W2p, 16) ||
      !aligned(tokens, 4) || !aligned(q_tok, 4) || !aligned(row_max, 4) ||
      !aligned(row_sumexp, 4) || !aligned(ell, 4) || !aligned(accept_len, 4) ||
      !aligned(out_tokens, 4) || !aligned(n_out, 4))
    return DSPARK_ERR_INVALID_ARG;
  const Plan p = make_plan(B, gamma, V, r, 0);
  if ((st = check_ws(workspace, workspace_bytes, p)) != DSPARK_OK) return st;
  if (launch_verify(p, T, U, nullptr, W2, W2p, E, nullptr, tokens, q_tok, row_max, row_sumexp, ell,
                    seed, accept_len, out_tokens, n_out, workspace, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

dspark_status dspark_last_device_status(void* workspace, cudaStream_t stream) {
  if (!aligned(workspace, 256)) return DSPARK_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (code != 0) {
    if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return DSPARK_ERR_CUDA;
    return (dspark_status)code;
  }
  return DSPARK_OK;
}

void dspark_testing_set_wait_limit(long long wait_cycles, int unreachable_barrier) {
  set_draft_wait_limit(wait_cycles > 0 ? wait_cycles : 0, unreachable_barrier ? (1u << 30) : 0u);
}

dspark_status dspark_copy_target_rows(const float* T_src, float* T, const int32_t* ell, int B,
                                      int gamma, int V, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream) {
  dspark_status st = check_shape(B, gamma, V, 16, 0);
  if (st != DSPARK_OK) return st;
  if (!aligned(T_src, 16) || !aligned(T, 16) || !aligned(ell, 4) || !aligned(workspace, 256) ||
      workspace_bytes < 256)
    return DSPARK_ERR_INVALID_ARG;
  // the source must be memory the device reads: device or managed memory, host memory
  // pinned or registered with CUDA, or pageable host memory where the device reads it
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, T_src) != cudaSuccess) {
    cudaGetLastError();
    return DSPARK_ERR_INVALID_ARG;
  }
  if (attr.type == cudaMemoryTypeUnregistered) {
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess ||
        !pageable)
      return DSPARK_ERR_INVALID_ARG;
  }
  if (launch_copy_target_rows(T_src, T, ell, B, gamma, V, ws_at<int>(workspace, 0), stream) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

}  // extern "C"
