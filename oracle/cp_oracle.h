/*
 * cp_oracle.h -- CPU oracle for the CodePredictor speculative round.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C
 * restatement of what the method computes, used to check the CUDA library.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header or table with the CUDA path.
 *
 * Sources (page title, section):
 *  - "CodePredictor Speculative Decoding" (TensorRT-Edge-LLM docs),
 *    sections "Why the draft is free", "How a round works", "Options".
 *  - "Speculative Decoding, Beyond Text", sections 02 (exact greedy and
 *    stochastic algorithms, the sum-min = 1 - TV identity), 03 (one round),
 *    07 (KV transaction / logit shift).
 *  - "RVQ Position Aware Speculative Decoding for On Device TTS", section 1
 *    Figure 1 (inner step k consumes c_{k-1}, emits c_k) and 2.1 (one
 *    embedding table and one LM head per codebook position).
 *  - "Awesome-ML-SYS-Tutorial" (Fast AR / MTP sections): the two-position
 *    prefix [hidden, code-0 embedding], per-frame KV rebuilt each frame.
 *  - "RVQ Position Aware Speculative Decoding for On Device TTS", section 2.2
 *    (position-aware offsets) and Figure 3: the draft at lookahead t reads
 *    head_{k+t} on h_k + b_t; the target head never sees an offset.
 *
 * Precision: the forward pass runs in float64 on weights given as float32
 * (bf16 and fp32 storage values are exact in float32); logits are rounded
 * to float32.  The softmax of the logit processing is float64 (exp and
 * sum) with one rounding of each probability to float32; the categorical
 * draw and the acceptance test are float32 with the exact orders documented
 * at each function.
 *
 * Parity pins: every function here is checked in tests/ against something
 * other than itself (published Philox known-answer vectors, brute-force
 * sorting, a torch float64 restatement with library attention/RMSNorm,
 * no-cache recomputation, exact greedy AR equality, statistical equality of
 * the speculative and autoregressive output laws, the sum-min identity).
 * The absolute acceptance rate on synthetic random weights has no pin
 * ("parity unpinned"): the pages' 1.70 / 2.47 tokens per step need trained
 * checkpoints and real audio.
 */
#ifndef CP_ORACLE_H
#define CP_ORACLE_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_DRAFT = 0, ORC_ACCEPT = 1, ORC_TARGET = 2, ORC_INPUT = 3, ORC_TREE_ACCEPT = 4 /* + child index */ };

typedef struct {
  int H, L, nq, nkv, d, F, V, G;
  double theta, eps;
  /* all float32, row-major; layer tensors stacked over layers */
  const float *embed;      /* [G-1][V][H]  table j is E_j (input for position j+1) */
  const float *head;       /* [G-1][V][H]  index j-1 is head_j                     */
  const float *final_norm; /* [H]          */
  const float *attn_norm;  /* [L][H]       */
  const float *wq;         /* [L][nq*d][H] */
  const float *wk;         /* [L][nkv*d][H]*/
  const float *wv;         /* [L][nkv*d][H]*/
  const float *wo;         /* [L][H][nq*d] */
  const float *ffn_norm;   /* [L][H]       */
  const float *w_gate;     /* [L][F][H]    */
  const float *w_up;       /* [L][F][H]    */
  const float *w_down;     /* [L][H][F]    */
  /* Position-aware draft offsets b_1..b_K ([K][H], float32), shared by every
   * starting depth.  K = 0 (or NULL): the heads are reused as they are. */
  int K;
  const float *draft_offset;
} orc_model;

typedef struct {
  int64_t frames, passes, rounds, committed, bonus, rejections;
  int64_t drafted_by_offset[9];  /* index t = 1..8 */
  int64_t accepted_by_offset[9];
} orc_stats;

typedef struct {
  int32_t frame, stream, s, n_d, m, n_acc, s_new, pad;
  int32_t drafts[8];
  double min_margin;
} orc_round_rec;

/* Philox4x32-10 block function (Salmon, Moraes, Dror, Shaw, SC'11). */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* u = (word0 >> 8) * 2^-24 of Philox(counter = (stream, frame, depth, purpose),
 * key = (seed mod 2^32, seed >> 32)). */
float orc_uniform(uint64_t seed, uint32_t stream, uint32_t frame, uint32_t depth, uint32_t purpose);
void orc_uniform_fill(uint64_t seed, int n, const uint32_t* ctr4 /*[n][4]*/, float* out);

/* Logit processing: T == 0 -> one-hot argmax (lowest index on ties); else
 * z = fl32(logit / T), keep exactly min(k, V) entries by (z desc, index asc),
 * e_i = exp(z_i - zmax) and S = sum of the kept e_i in float64,
 * p_i = fl32(e_i / S).  margin (optional) = decision gap in logit units. */
void orc_process(const float* logits, int V, int top_k, float T, float* probs, double* margin);
/* Categorical draw: candidates = {i : w_i > 0} ascending; S_j sequential
 * float32 prefix sums; t = fl32(u * S_last); first j with S_j > t, else the
 * last candidate.  Returns -1 if no candidate.  margin = relative distance
 * of t to the nearest adjacent boundary. */
int orc_sample(const float* w, int V, float u, double* margin);
/* Left-to-right exact speculative acceptance over n_d drafts with explicit
 * uniforms.  q: [n_d][V], p: [m][V] with m in {n_d, n_d + 1}; p row t-1
 * scores draft t.  Accept draft t iff u_acc[t-1] < fl32(p_t(y)/q_t(y)); on
 * the first rejection emit a draw from norm(max(0, p_t - q_t)) with
 * u_tgt[t-1] (from p_t if that residual is all zero) and stop; if all are
 * accepted and m > n_d emit the bonus drawn from p row n_d with u_tgt[n_d].
 * Returns the number of accepted drafts. */
int orc_accept_chain(int V, int n_d, int m, const float* q, const int* drafts, const float* p,
                     const float* u_acc, const float* u_tgt, int* emitted, int* n_emitted,
                     double* margin);
/* Acceptance microbenchmark: R independent rounds of N-1 drafts and N
 * target rows.  mode 0: inputs are logits (processed with top_k / T);
 * mode 1: inputs are already-processed float32 probabilities.  Philox
 * counter (stream = r, frame = 0, depth = t, purpose).  tokens: [R][N],
 * -1 padded; n_acc: [R]; drafts (optional) [R][N-1]; margins optional [R]. */
void orc_accept_batch(int R, int N, int V, int top_k, float T, uint64_t seed, int mode,
                      const float* target, const float* draft, int* tokens, int* n_acc,
                      int* drafts, double* margins);

size_t orc_kv_doubles(const orc_model* M);
/* One causal block pass: rows at the given positions are appended to the
 * KV cache (float64 [L][2][G][nkv][d]) and each row attends to cache
 * positions 0..pos.  out: final-RMSNorm'ed hidden per row [n][H]. */
void orc_forward(const orc_model* M, double* kv, int n, const double* in_rows, const int* positions,
                 double* out_normed);
/* logits of head_j (1 <= j <= G-1) on a normed hidden, float64 and float32. */
void orc_head_logits(const orc_model* M, int j, const double* hn, double* out64, float* out32);
/* Draft logits at lookahead t >= 1 from the normed hidden hn of depth s
 * (j = s + t): head_j on hn + b_t when t <= K, head_j on hn otherwise. */
void orc_draft_logits(const orc_model* M, int j, int t, const double* hn, float* out32);
/* Teacher-forced logits over positions 0..P-1 of one frame (rows x,
 * E_0(c_0), ..., E_{P-2}(c_{P-2})): logits [P-1][V] for head_j at position
 * j; draft (optional) [P-1][n_draft][V]: the draft logits of lookahead t
 * at position j (orc_draft_logits with head_{j+t}; zero where j+t > G-1). */
void orc_teacher_logits(const orc_model* M, const float* x, const int* codes, int P, int n_draft,
                        float* logits, float* draft);
/* Decode frames.  N = 0: autoregressive loop; N in 2..8: speculative rounds.
 * top_k / temp per stream [B].  x [F][B][H], c0 [F][B], codes out [F][B][G]
 * (codes[...][0] = c0).  Returns 0, or -1 on bad arguments. */
int orc_decode_frames(const orc_model* M, int N, const int* top_k, const float* temp, uint64_t seed,
                      int B, int F, int first_frame, const float* x, const int* c0, int* codes,
                      orc_stats* st, orc_round_rec* log, int log_cap, int* n_log);
/* Adaptive window ("Speculative Decoding, Beyond Text", runtime policies;
 * "CodePredictor Speculative Decoding", "Options": acceptance flattens past
 * a few drafts): each stream picks its window for the next frame from its
 * acceptance by offset so far in the call (orc_policy_window).  pct = 0
 * turns the policy off (every frame uses N).  The window depends only on
 * earlier frames, so each frame keeps the autoregressive law. */
int orc_policy_window(int N, int pct, int min_reached, const int64_t* reach /*[9]*/, const int64_t* acc /*[9]*/);
int orc_decode_frames_policy(const orc_model* M, int N, const int* top_k, const float* temp, uint64_t seed,
                             int B, int F, int first_frame, const float* x, const int* c0, int* codes,
                             orc_stats* st, orc_round_rec* log, int log_cap, int* n_log, int pct,
                             int min_reached);

/* Sparse draft tree ("RVQ Position Aware Speculative Decoding for On Device
 * TTS", section 2.2, Figure 2): n nodes (at most 62), parents first; node i
 * has parent[i] (-1: a child of the committed code) and rank[i], the rank of
 * its token among the draft logits of its depth (value descending, index
 * ascending); siblings appear in ascending rank.  Nodes deeper than the
 * codes left in a frame are dropped. */
typedef struct {
  int n;
  const int *parent;
  const int *rank;
} orc_tree;
/* Decode frames with tree rounds (acceptance walk described at the
 * definition).  Log records: n_d = kept nodes, m = rows verified, n_acc =
 * accepted depth, drafts = the accepted path.  drafted_by_offset stays zero;
 * accepted_by_offset counts accepted nodes by depth. */
int orc_decode_frames_tree(const orc_model* M, const orc_tree* T, const int* top_k, const float* temp,
                           uint64_t seed, int B, int F, int first_frame, const float* x, const int* c0, int* codes,
                           orc_stats* st, orc_round_rec* log, int log_cap, int* n_log);

#ifdef __cplusplus
}
#endif
#endif
