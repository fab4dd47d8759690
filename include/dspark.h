/*
 * dspark.h -- C ABI of the DSpark per-step hot path on one GPU (sm_103a).
 *
 * One speculative step of DSpark ("DSpark: Confidence-Scheduled Speculative Decoding with
 * Semi-Autoregressive Generation") is four calls, run in this order on one stream:
 *
 *   dspark_draft       semi-autoregressive block drafting with the low-rank Markov head
 *   dspark_confidence  confidence head c_k and survival a_j = prod_{i<=j} c_i
 *   dspark_schedule    hardware-aware prefix scheduler choosing l_r per request
 *   dspark_verify      lossless rejection-sampling verification with correction / bonus
 *
 * The backbone forward (base logits U, hidden states h) and the target forward (target
 * logits T) are not part of this library; their outputs are inputs here.
 *
 * Conventions shared by every call
 *   - All array pointers are DEVICE pointers, owned by the caller, row-major and
 *     contiguous, 16-byte aligned.  The library allocates no memory: scratch space comes
 *     from the caller's workspace (size from dspark_workspace_bytes; 256-byte aligned,
 *     zero-filled before its first use: its first 256 bytes hold the device status
 *     word).  One workspace may serve all calls of a step as long as they run in order
 *     on one stream; calls that overlap on the GPU must not share a workspace.
 *   - bf16 weights are passed as their uint16_t bit patterns.
 *   - Every call is asynchronous on `stream` and may be captured in a CUDA graph.
 *   - Requests b are 0-based, draft positions k are 1-based (k = 1..gamma).
 *   - Random numbers: Philox4x32 with 7 rounds (Salmon et al., SC'11; 7 is the fewest
 *     rounds that paper reports passing TestU01 BigCrush) keyed by `seed` (low word,
 *     high word); the 32-bit draw for vocabulary index v of (request b, position k,
 *     stream s) is word v % 4 of the block with counter (v / 4, k, b, s);
 *     U01(x) = ((x >> 9) + 1/2) * 2^-23.  Streams: 0 draft Gumbel, 1 acceptance uniform
 *     (v = 0), 2 residual Gumbel, 3 bonus Gumbel.  Gumbel g = -log(-log U01).
 *   - Shape limits: 1 <= B < 65536, 1 <= gamma <= 32, B * (gamma + 1) < 2^21,
 *     8 <= V < 2^31 with V % 8 == 0, 16 <= r <= 256 with r % 16 == 0, H % 4 == 0; the
 *     draft calls also need ceil(B / 128) * ceil(V / 128) < 26843545 (2^32 / 160).
 *
 * Errors
 *   - Every call validates its arguments on the host before launching anything and
 *     returns DSPARK_ERR_INVALID_ARG (null pointer, misaligned pointer, bad shape,
 *     workspace too small, table too short) or DSPARK_ERR_UNSUPPORTED (shape outside the
 *     limits above).  Nothing is launched in that case.
 *   - A failed launch returns DSPARK_ERR_CUDA.
 *   - Kernels never trap.  A device-side check (a token id out of range, a bounded wait
 *     that ran out) writes a code into the workspace's status word and skips the access;
 *     dspark_last_device_status() reads and clears it.
 */
#ifndef DSPARK_H_
#define DSPARK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __CUDA_RUNTIME_H__
typedef struct CUstream_st* cudaStream_t;
#endif

typedef enum {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = 1,
  DSPARK_ERR_UNSUPPORTED = 2,
  DSPARK_ERR_CUDA = 3,
  DSPARK_ERR_TIMEOUT = 4,
  DSPARK_ERR_DEVICE_CHECK = 5
} dspark_status;

/* Human-readable name of a status code (static string). */
const char* dspark_status_string(dspark_status s);

/* Workspace bytes needed by every call on shapes (B, gamma, V, r, H); 0 on bad shapes. */
size_t dspark_workspace_bytes(int B, int gamma, int V, int r, int H);

/*
 * Markov transition bias for a batch of predecessors.  billytse.dev DSpark page, section
 * 3.3: the first-order Markov head adds B(x_{k-1}, .) = W1[x_{k-1}] W2 (rank r) to the
 * base logits.  Computed on the tensor cores with fp32 accumulation:
 *   out[b, v] = sum_i W1[prev[b * prev_stride], i] * W2[i, v]   (0 <= b < B, 0 <= v < V)
 * A predecessor of -1 gives a zero row; any other id outside [0, V) gives a zero row and
 * records DSPARK_ERR_DEVICE_CHECK.
 *
 *   W1 [V, r] bf16, W2 [r, V] bf16, prev [B * prev_stride] int32  ->  out [B, V] fp32
 */
dspark_status dspark_markov_bias(const uint16_t* W1, const uint16_t* W2, const int32_t* prev,
                                 int prev_stride, int B, int V, int r, float* out,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Semi-autoregressive draft.  billytse.dev DSpark page, section 3.2 (block distribution
 * p_k(v | x_<k) = softmax(U_k(v) + B_k(x_<k, v))) and section 3.3 (first-order Markov
 * head B(x_{k-1}, .) = W1[x_{k-1}] W2 with rank r; the left-to-right loop prev = anchor;
 * bias = W1[prev] @ W2; probs = softmax(base_logits[k] + bias); token = sample(probs);
 * prev = token).  Sampling is Gumbel-max: x_k = argmax_v (z_v + g_v), ties to the
 * smallest v, with g from stream 0.
 *
 *   U        [B, gamma, V] fp32   base logits U_k
 *   W1       [V, r] bf16          previous-token embedding of the Markov head
 *   W2       [r, V] bf16          projection back to vocabulary logits
 *   anchor   [B] int32            last committed token of each request (0 <= id < V)
 * outputs
 *   tokens     [B, gamma] int32   x_k
 *   q_tok      [B, gamma] fp32    q_k(x_k) = softmax(z_k)(x_k)
 *   row_max    [B, gamma] fp32    max_v z_k(v)
 *   row_sumexp [B, gamma] fp32    sum_v exp(z_k(v) - row_max)
 */
dspark_status dspark_draft(const float* U, const uint16_t* W1, const uint16_t* W2,
                           const int32_t* anchor, int B, int gamma, int V, int r,
                           uint64_t seed, int32_t* tokens, float* q_tok, float* row_max,
                           float* row_sumexp, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * Packed Markov-head projection.  The draft kernel's tensor-core operand is the W2^T
 * vocabulary tile; read from W2 [r, V] a tile is r short rows spread over all of W2.
 * dspark_pack_w2 rearranges W2 once (at weight-load time) into contiguous per-tile
 * images of exactly that operand, and dspark_draft_packed streams them with one bulk
 * copy per 16 KB chunk.  Results are identical to dspark_draft.
 *
 *   dspark_packed_w2_bytes(V, r): bytes of the packed copy (ceil(V/128)*128 * r * 2);
 *   0 on unsupported shapes.
 *   dspark_pack_w2: W2 [r, V] bf16 -> W2p (caller-owned, W2p_bytes >= the size above,
 *   16-byte aligned).  Layout, in 16-byte units, for tile t, rank chunk i of kc rows
 *   (kc = 64 if r % 64 == 0, else 32 if r % 32 == 0, else 16), half h, rank row kl,
 *   slot s:  W2p[t][i][h][kl][s] = W2[i*kc + kl][t*128 + 64h + 8(s ^ (kl % 8)) .. +7],
 *   zero beyond V.
 *   dspark_draft_packed: dspark_draft with W2p in place of W2 (same arguments,
 *   workspace and outputs otherwise).
 */
size_t dspark_packed_w2_bytes(int V, int r);
dspark_status dspark_pack_w2(const uint16_t* W2, int V, int r, uint16_t* W2p, size_t W2p_bytes,
                             cudaStream_t stream);
dspark_status dspark_draft_packed(const float* U, const uint16_t* W1, const uint16_t* W2p,
                                  const int32_t* anchor, int B, int gamma, int V, int r,
                                  uint64_t seed, int32_t* tokens, float* q_tok, float* row_max,
                                  float* row_sumexp, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/*
 * Confidence head and survival.  weigao.cc DSpark-vs-MTP page, "3. confidence head"
 * (c_k = P(position k survives | positions < k accepted), one linear layer on
 * [output_hidden_k ; markov_embedding(prev_token)]) and billytse.dev DSpark page,
 * section 5 (a_j = prod_{i<=j} c_i).  The Markov embedding is the W1 row of prev
 * (prev = anchor for k = 1, tokens[b, k-1] after that):
 *   c[b,k] = 1 / (1 + exp(-(sum_j w_c[j] h[b,k,j] + sum_i w_c[H+i] W1[prev,i] + b_c)))
 *   a[b,k] = c[b,1] * ... * c[b,k]   (multiplied left to right)
 *
 *   h [B, gamma, H] fp32, anchor [B], tokens [B, gamma], W1 [V, r] bf16,
 *   w_c [H + r] fp32, b_c  ->  c [B, gamma] fp32, a [B, gamma] fp32
 */
dspark_status dspark_confidence(const float* h, const int32_t* anchor, const int32_t* tokens,
                                const uint16_t* W1, const float* w_c, float b_c, int B,
                                int gamma, int H, int r, int V, float* c, float* a,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Hardware-aware prefix scheduler.  billytse.dev DSpark page, section 6 (B = sum_r
 * (1 + l_r); tau = sum_r (1 + sum_{j<=l_r} a_{r,j}); maximise Theta = tau * SPS(B) by
 * adding positions in descending expected return and stopping as soon as Theta would
 * fall) and section 7 (early stopping keeps the rule non-anticipating).
 *
 * Items (r, j) are ranked by (A desc, r asc, j asc) with A = floor(clamp(a, 0, 1) * 2^32
 * + 1/2) (NaN counts as 0); sums are exact integers; Theta_n = double(R 2^32 + S_n) *
 * double(sps[R + n]) and item n is admitted while Theta_n > Theta_{n-1}.  l_r is the
 * number of admitted positions of request r (a prefix when a is non-increasing in j).
 *
 *   a   [R, gamma] fp32 survival; sps [sps_len] fp32 steps/s indexed by token-batch size,
 *       sps_len >= R * (gamma + 1) + 1
 *   ->  ell [R] int32, B_total [1] int32 (= R + admitted), theta [1] fp64 (= tau SPS(B))
 * R * gamma must not exceed 16384.
 */
dspark_status dspark_schedule(const float* a, int R, int gamma, const float* sps, int sps_len,
                              int32_t* ell, int32_t* B_total, double* theta, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * dspark_confidence followed by dspark_schedule in one launch: the confidence kernel's
 * last CTA to finish runs the prefix scheduler over all survivals (the CTAs count
 * themselves in a counter kept in the workspace's first 256 bytes, which the call leaves at
 * zero).  Arguments, outputs, limits and results are those of the two calls (R = B, and
 * B * gamma must not exceed 16384).
 */
dspark_status dspark_confidence_schedule(const float* h, const int32_t* anchor,
                                         const int32_t* tokens, const uint16_t* W1,
                                         const float* w_c, float b_c, int B, int gamma, int H,
                                         int r, int V, const float* sps, int sps_len, float* c,
                                         float* a, int32_t* ell, int32_t* B_total,
                                         double* theta, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream);

/*
 * Lossless verification.  billytse.dev DSpark page, section 1 (accept x_k with
 * probability min(1, p_k(x_k) / q_k(x_k)), keep the longest accepted prefix, fix the
 * first rejected position with a token from the residual) and xhh.club DSpark page
 * (Q&A on the acceptance rule: the residual is norm(max(0, p - q)), so that
 * min(q, p) + (p - min(p, q)) = p).  The target distribution is p_k = softmax(T[b, k]).
 *
 * For each request b and k = 1..ell[b]: u = U01(stream 1 draw at v = 0); accept iff
 * u < p_k(x_k) / q_tok[b,k].  At the first reject j: y = argmax over {v: P_j(v) > Q_j(v)}
 * of log(P_j(v) - Q_j(v)) + g_v (stream 2) with Q_j = softmax(U[b,j] + W1[prev_j] W2)
 * rebuilt from row_max / row_sumexp; if that set is empty, y = argmax T[b,j,v] + g_v
 * (stream 2).  If all ell[b] positions are accepted, y is the target's bonus token
 * argmax T[b, ell+1, v] + g_v (stream 3).
 *
 *   T [B, gamma+1, V] fp32 target logits (row gamma+1 is the bonus row), U, W1, W2,
 *   anchor, tokens, q_tok, row_max, row_sumexp as produced by dspark_draft, ell [B].
 *   ->  accept_len [B] int32, out_tokens [B, gamma+1] int32 (accepted prefix, then the
 *       correction or bonus token, then -1), n_out [B] int32 (= accept_len + 1)
 */
dspark_status dspark_verify(const float* T, const float* U, const uint16_t* W1,
                            const uint16_t* W2, const int32_t* anchor, const int32_t* tokens,
                            const float* q_tok, const float* row_max, const float* row_sumexp,
                            const int32_t* ell, int B, int gamma, int V, int r, uint64_t seed,
                            int32_t* accept_len, int32_t* out_tokens, int32_t* n_out,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * dspark_verify with the packed tile images of dspark_pack_w2 (W2p) in place of W2: the
 * residual rows' bias contraction streams W2p, which a preceding dspark_draft_packed call
 * has just brought into L2.  Same arguments, workspace, outputs and results otherwise;
 * W2p is caller-owned, 16-byte aligned, of dspark_packed_w2_bytes(V, r) bytes.
 */
dspark_status dspark_verify_packed(const float* T, const float* U, const uint16_t* W1,
                                   const uint16_t* W2p, const int32_t* anchor,
                                   const int32_t* tokens, const float* q_tok,
                                   const float* row_max, const float* row_sumexp,
                                   const int32_t* ell, int B, int gamma, int V, int r,
                                   uint64_t seed, int32_t* accept_len, int32_t* out_tokens,
                                   int32_t* n_out, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream);

/*
 * The draft of dspark_draft for callers that cannot allocate device memory when they
 * draft (a serving loop whose device memory is all reserved by its own pool, a plugin
 * that is handed only its input and output buffers, code where a cudaMalloc would
 * synchronise or fail).  The paper has no counterpart: this is a packaging of the same
 * kernel.  Same arguments, outputs and results as dspark_draft, without the workspace:
 * the kernel's scratch lives in a fixed array inside the library, about 2.5 MB, which
 * every GPU that loads the library holds until the process exits.
 *   - Limits: B <= 256 and gamma <= 32 (otherwise DSPARK_ERR_UNSUPPORTED), plus the
 *     shape limits above.
 *   - The first call on each device looks up the array's device address (with that
 *     device current); make that first call before any stream capture.
 *   - All calls share the array: calls whose kernels overlap on the GPU (other streams,
 *     other host threads) race; serialise them.  Each call clears what must start at
 *     zero on its stream.
 *   - Device-side checks are not reported by this entry point (there is no workspace
 *     status word); use dspark_draft to diagnose them.
 *   - It allocates nothing: no cudaMalloc, no cudaFree.
 */
dspark_status dspark_draft_noalloc(const float* U, const uint16_t* W1, const uint16_t* W2,
                                   const int32_t* anchor, int B, int gamma, int V, int r,
                                   uint64_t seed, int32_t* tokens, float* q_tok, float* row_max,
                                   float* row_sumexp, cudaStream_t stream);

/*
 * Greedy draft.  billytse.dev DSpark page, section 11: the serving example selects the
 * greedy draft sampling method.  The loop of dspark_draft with x_k = argmax_v z_k(v) (ties
 * to the smallest v) in place of the random draw; no random numbers are used.  The
 * proposal is the point mass at x_k, so q_tok = 1; row_max and row_sumexp are the softmax
 * statistics of z_k as in dspark_draft.
 *
 *   Exactly one of W2 ([r, V] bf16) and W2p (the packed copy of dspark_pack_w2) is
 *   non-NULL; otherwise the arguments, workspace and outputs are those of dspark_draft.
 *   Verify its tokens with dspark_verify_greedy.
 */
dspark_status dspark_draft_greedy(const float* U, const uint16_t* W1, const uint16_t* W2,
                                  const uint16_t* W2p, const int32_t* anchor, int B, int gamma,
                                  int V, int r, int32_t* tokens, float* q_tok, float* row_max,
                                  float* row_sumexp, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/*
 * Lossless verification of a greedy draft.  The rule of dspark_verify with the greedy
 * proposal Q_k = point mass at x_k: accept iff u < p_k(x_k) (u from stream 1 as before);
 * at the first reject j the residual max(0, P_j - Q_j) is P_j without x_j, so
 * y = argmax over v != x_j of T[b,j,v] + g_v (stream 2); the bonus token is as in
 * dspark_verify.  U, W1, W2 and the draft's row statistics are not needed.
 *
 *   T [B, gamma+1, V] fp32, tokens [B, gamma] int32 (from dspark_draft_greedy or any
 *   deterministic proposer), ell [B] int32  ->  accept_len, out_tokens, n_out as in
 *   dspark_verify.  The workspace is one of dspark_workspace_bytes(B, gamma, V, r, H)
 *   bytes for any r and H.
 */
dspark_status dspark_verify_greedy(const float* T, const int32_t* tokens, const int32_t* ell,
                                   int B, int gamma, int V, uint64_t seed, int32_t* accept_len,
                                   int32_t* out_tokens, int32_t* n_out, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream);

/*
 * Asynchronous two-step capacity scheduler.  weigao.cc DSpark-vs-MTP page, "4. hardware-
 * aware prefix scheduler" (the production scheduler fixes the next step's capacity from
 * the predictions of two steps earlier, so that CUDA-graph replay and zero-overhead
 * scheduling know the batch ahead, while the current candidates are still ranked by
 * their latest cumulative confidence) and billytse.dev DSpark page, section 7 (the old
 * information decides only how large the top-K is, never whether a given token is
 * admitted).
 *
 * With K = *K_in (clamped to R * gamma) the first K items in the order of
 * dspark_schedule are admitted: ell [R] counts each request's items among them, B_total =
 * R + K, theta = (R + S_K) * SPS(R + K) with the fixed-point sum of dspark_schedule.
 * *K_out receives n*, this step's own early-stop count (dspark_schedule's B_total - R),
 * the capacity for the step after next.  K_in == NULL or *K_in < 0 admits n* itself, so
 * the call then equals dspark_schedule.  K_in and K_out are device int32 words; they may
 * be the same word (the input is read before the output is written), and K_out may be
 * NULL.  A two-slot ring, slot t % 2 for step t, starting at -1, gives the pipeline.
 * Arguments, limits and workspace otherwise as dspark_schedule.
 */
dspark_status dspark_schedule_async(const float* a, int R, int gamma, const float* sps,
                                    int sps_len, const int32_t* K_in, int32_t* K_out,
                                    int32_t* ell, int32_t* B_total, double* theta,
                                    void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream);

/*
 * Fixed confidence-threshold truncation.  billytse.dev DSpark page, section 8 (the
 * confidence-threshold sweep under fixed-length verification) and the xhh.club DSpark page
 * (a fixed threshold on the survival probability cannot follow the load: the baseline the
 * adaptive scheduler improves on).  ell[r] = the number of leading positions j = 1, 2, ...
 * with a[r, j] > threshold (strict; the scan stops at the first failure), B_total =
 * sum_r (1 + ell[r]).  threshold < 0 verifies every position (fixed-length verification).
 *
 *   a [R, gamma] fp32, 1 <= gamma <= 32, 1 <= R < 65536  ->  ell [R] int32, B_total [1] int32
 */
dspark_status dspark_schedule_threshold(const float* a, int R, int gamma, float threshold,
                                        int32_t* ell, int32_t* B_total, cudaStream_t stream);

/*
 * RNN head.  weigao.cc DSpark-vs-MTP page, "2. Markov head and RNN head": the head keeps a
 * recurrent state inside the draft block; each step concatenates the previous state, the
 * previous token's embedding and the position's hidden state, one linear layer splits the
 * result into gate, candidate and output, state_k = gate * state_{k-1} + (1 - gate) *
 * candidate, and the bias is W2 tanh(output) (billytse.dev section 3.3: the head that lets
 * every position remember the whole block prefix).  Readings: the state has r entries;
 * the token embedding is the W1 row; gate = sigmoid, candidate = tanh of their blocks;
 * state_0 = 0; the layer is W_rnn [2r + H, 3r] bf16 + b_rnn [3r] fp32, rows [0, r) for the
 * state, [r, 2r) for W1[prev], [2r, 2r + H) for h_k, column blocks gate | candidate |
 * output; the head computes in fp32, and its output rows E_k = tanh(output) enter the
 * tensor-core contraction as two bf16 terms (hi + lo, |E - hi - lo| <= 2^-18 |E|).
 *
 *   dspark_rnn_packed_bytes(r): bytes of the transposed recurrent rows (3r * 2r * 2); 0 on
 *   an unsupported r.
 *   dspark_rnn_pack: Wrec[c][j] = W_rnn[j][c] for c < 3r, j < 2r (caller-owned, 16-byte
 *   aligned; once per weights).
 *   dspark_rnn_project: hp[b, k, c] = b_rnn[c] + sum_j h[b, k, j] W_rnn[2r + j][c] for every
 *   (b, k) -- the part of the layer that does not depend on drafted tokens.  h [B, gamma, H]
 *   fp32 (H % 4 == 0), hp [B, gamma, 3r] fp32; all 16-byte aligned.  Computed on the tensor
 *   cores with fp32 accuracy (h as three exact bf16 terms).  The call has no status word: if
 *   one of its bounded device waits runs out, the affected 128 x 128 tiles of hp are NaN.
 *   dspark_draft_rnn: dspark_draft (greedy == 0) or dspark_draft_greedy (greedy != 0) with
 *   the RNN head's bias in place of the Markov bias: exactly one of W2 and W2p non-NULL,
 *   Wrec from dspark_rnn_pack, hp from dspark_rnn_project.  Also writes E [B, gamma, r]
 *   fp32, the output rows tanh(output) (16-byte aligned), which dspark_verify_rnn needs.
 *   dspark_verify_rnn: dspark_verify for a Gumbel-sampled RNN draft: the residual's
 *   proposal is Q_j = softmax(U[b, j] + E[b, j] W2); W1 and the anchors are not needed.
 *   (A greedy RNN draft is verified with dspark_verify_greedy.)
 */
size_t dspark_rnn_packed_bytes(int r);
dspark_status dspark_rnn_pack(const uint16_t* W_rnn, int r, uint16_t* Wrec, size_t Wrec_bytes,
                              cudaStream_t stream);
dspark_status dspark_rnn_project(const float* h, const uint16_t* W_rnn, const float* b_rnn,
                                 int B, int gamma, int H, int r, float* hp, cudaStream_t stream);
dspark_status dspark_draft_rnn(const float* U, const uint16_t* W1, const uint16_t* W2,
                               const uint16_t* W2p, const uint16_t* Wrec, const float* hp,
                               const int32_t* anchor, int B, int gamma, int V, int r,
                               uint64_t seed, int greedy, int32_t* tokens, float* q_tok,
                               float* row_max, float* row_sumexp, float* E, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);
dspark_status dspark_verify_rnn(const float* T, const float* U, const float* E, const uint16_t* W2,
                                const uint16_t* W2p, const int32_t* tokens, const float* q_tok,
                                const float* row_max, const float* row_sumexp, const int32_t* ell,
                                int B, int gamma, int V, int r, uint64_t seed,
                                int32_t* accept_len, int32_t* out_tokens, int32_t* n_out,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Reads and clears the device status word kept in `workspace` after synchronising
 * `stream`.  Returns DSPARK_OK, or the first device-side failure recorded since the last
 * read (DSPARK_ERR_DEVICE_CHECK, DSPARK_ERR_TIMEOUT), or DSPARK_ERR_CUDA.
 */
dspark_status dspark_last_device_status(void* workspace, cudaStream_t stream);

/*
 * One launch for the first three calls of a step: dspark_draft_packed, then
 * dspark_confidence_schedule on the drafted tokens.  The draft kernel computes the
 * confidence head and survival of position k (weigao.cc DSpark-vs-MTP page, "3.
 * confidence head"; billytse.dev DSpark page, section 5) in a warp of its own, the h_k part
 * while position k - 1 is drawn and the rest once x_{k-1} is known; after the last position
 * it runs the prefix scheduler (billytse.dev sections 6 and 7): when B * gamma <= 384, in
 * the confidence warps of the CTAs that hold no request while the last position is drawn
 * (else in one CTA after it), with every CTA ranking a share of the items when
 * B * gamma <= 4096;
 * larger batches get the scheduler kernel as a second launch.  Outputs and their meaning are those of the three
 * calls (tokens, q_tok, row_max, row_sumexp; c, a; ell, B_total, theta); the draft's
 * outputs are identical to dspark_draft_packed's, c and a agree with dspark_confidence's to
 * fp32 rounding (another summation order), and ell, B_total, theta are the scheduler's
 * on this a.  W2p is the packed W2 of dspark_pack_w2; h, w_c, b_c, sps as in
 * dspark_confidence_schedule.  The workspace is one of dspark_workspace_bytes(B, gamma, V,
 * r, H).  Requires B * gamma <= 16384; DSPARK_ERR_UNSUPPORTED also when the vocabulary is
 * so small that the draft grid keeps no survival slot for some request (B > 512 x the
 * draft grid, the smaller of the number of 128-column vocabulary tiles and the number of
 * CTAs the device holds at once).
 */
dspark_status dspark_draft_confidence_schedule(
    const float* U, const uint16_t* W1, const uint16_t* W2p, const int32_t* anchor, const float* h,
    const float* w_c, float b_c, const float* sps, int sps_len, int B, int gamma, int V, int r, int H,
    uint64_t seed, int32_t* tokens, float* q_tok, float* row_max, float* row_sumexp, float* c,
    float* a, int32_t* ell, int32_t* B_total, double* theta, void* workspace,
    size_t workspace_bytes, cudaStream_t stream);

/*
 * Testing hook for the failure path of the draft (no passage of the pages: the bounded
 * waits are this library's own failure detection).  Every wait inside the draft kernels of
 * dspark_draft, dspark_draft_packed, dspark_draft_greedy, dspark_draft_noalloc,
 * dspark_draft_confidence_schedule and dspark_draft_rnn is bounded, by default to about 2 s
 * of SM clock; a wait that runs out records DSPARK_ERR_TIMEOUT in the status word and the
 * kernel drains its copies and MMAs, frees its tensor memory and returns.  This call
 * changes, for the draft launches that follow in the process, the bound to `wait_cycles`
 * SM cycles (<= 0: the default) and, when `unreachable_barrier` is non-zero, adds an offset
 * to the kernels' barrier targets (the grid barrier, and the RNN head's recurrence count)
 * so that the first barrier cannot complete and a wait must run out.  (0, 0) restores the
 * production setting.  Not for use while draft launches are in flight or being captured.
 */
void dspark_testing_set_wait_limit(long long wait_cycles, int unreachable_barrier);

/*
 * The rows of the target logits that a verification reads under the schedule ell, copied
 * from T_src into T (both [B][gamma + 1][V] fp32, 16-byte aligned): T[b, j] for
 * 0 <= j <= ell[b], the verified positions' rows and the row the final token is drawn
 * from (billytse.dev DSpark page, section 1: the target scores the scheduled prefix; the
 * later rows are never read).  T_src may be host memory that the device reads directly
 * (pinned or registered with CUDA, or pageable memory on systems whose GPU reads it): a
 * kernel fetches the rows over the host link, so a step whose target logits arrive in host
 * memory moves only the rows it verifies; device memory works too.  The other rows of T
 * are left as they are.  ell (device, B entries) is the scheduler's output; an entry
 * outside [0, gamma] is clamped and reported as DSPARK_ERR_DEVICE_CHECK through the status
 * word of `workspace` (any workspace of this library; only its status word is used, so 256
 * bytes suffice).  DSPARK_ERR_INVALID_ARG when T_src is host memory the device cannot read.
 */
dspark_status dspark_copy_target_rows(const float* T_src, float* T, const int32_t* ell, int B,
                                      int gamma, int V, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H_ */
