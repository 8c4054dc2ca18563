/*
 * cp_spec.h -- C ABI of the GB300 CodePredictor speculative-decoding library.
 *
 * The library runs the inner RVQ loop of a Qwen3-TTS / Qwen3-Omni style
 * CodePredictor: per audio frame, given the talker hidden x and the first
 * code c_0, it emits the residual codes c_1..c_{G-1}, either one decoder pass
 * per code (autoregressive, verify_window = 0) or by speculative rounds
 * ("CodePredictor Speculative Decoding", section "How a round works"):
 *   1. draft: lm_head_{s+1..s+N-1} applied to the current hidden h_s
 *      (section "Why the draft is free"), top-k / temperature sampling;
 *   2. verify: one causal decoder pass over the committed code and the
 *      N-1 drafts against the per-stream KV cache;
 *   3. accept: exact speculative sampling, min(1, p/q), residual
 *      norm(max(0, p - q)) at the first rejection, bonus code when every
 *      draft is accepted ("Speculative Decoding, Beyond Text", section 02);
 *      greedy (temperature 0) is exact argmax equality;
 *   4. reconcile: the KV cache keeps positions 0..s' (s' = last committed
 *      depth); rejected entries stay in memory but are never read (section 07).
 * Two options change only the drafts, so the committed codes keep the
 * autoregressive law: position-aware draft offsets (the draft of lookahead t
 * reads head_{s+t} on h_s + b_t; "RVQ Position Aware Speculative Decoding for
 * On Device TTS", section 2.2) and an adaptive window per stream chosen from
 * its acceptance by offset ("Speculative Decoding, Beyond Text", runtime
 * policies).
 *
 * Sequence layout of one frame: position 0 holds x, position j >= 1 holds
 * the embedding E_{j-1}(c_{j-1}); the decoder output at position j, through
 * the final RMSNorm and head_j, gives the law p_j of c_j ("RVQ Position Aware
 * Speculative Decoding for On Device TTS", Figure 1 and section 2.1).
 *
 * Conventions for every entry point:
 *  - Pointers named d_* are DEVICE pointers, h_* are HOST pointers.  The
 *    caller owns all device memory (weights, workspace, inputs, outputs) and
 *    must keep it alive while work it was passed to is in flight.  The
 *    library never allocates device memory.  A context (cp_spec_ctx) is host
 *    memory owned by the library until cp_spec_destroy.
 *  - Every device pointer must be 16-byte aligned; otherwise the call
 *    returns CP_SPEC_E_INVALID.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls enqueue work on it and return without synchronising,
 *    except where stated.  Argument errors are returned synchronously and
 *    enqueue nothing.  Device-side errors (bad code index, a weight tile
 *    copy that did not land in time) are recorded in a device status word and reported by
 *    cp_spec_status_word() or by the next call on the same context.
 *  - Randomness is Philox4x32-10 (Salmon et al., SC'11) with counter
 *    (stream id, frame index, depth, purpose) and key = (seed mod 2^32,
 *    seed >> 32); purpose DRAFT = 0, ACCEPT = 1, TARGET = 2.  u = (word0 >> 8)
 *    * 2^-24.  Results are therefore reproducible bit for bit and
 *    independent of batching or of how streams are split across calls.
 *  - No entry point ever traps, asserts or spins without a bound on the GPU.
 */
#ifndef CP_SPEC_H
#define CP_SPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CP_SPEC_MAX_LAYERS 64
#define CP_SPEC_MAX_WINDOW 8
#define CP_SPEC_MAX_CODE_GROUPS 64
#define CP_SPEC_MAX_VOCAB 8192
/* Size of the library-owned scratch of cp_spec_decode_frames_static (8 MiB). */
#define CP_SPEC_STATIC_SCRATCH_BYTES (8u << 20)

typedef enum {
  CP_SPEC_OK = 0,
  CP_SPEC_W_AR_FALLBACK = 1,       /* warning: speculation disabled, runs the AR loop */
  CP_SPEC_E_INVALID = -1,          /* bad argument (range, null, alignment)           */
  CP_SPEC_E_UNSUPPORTED = -2,      /* shape outside what the kernels implement        */
  CP_SPEC_E_CUDA = -3,             /* a CUDA runtime call failed                      */
  CP_SPEC_E_WORKSPACE = -4,        /* workspace smaller than cp_spec_workspace_bytes  */
  CP_SPEC_E_DEVICE_TIMEOUT = -5,   /* a bounded device-side wait gave up              */
  CP_SPEC_E_STATE = -6,            /* call out of order (e.g. round before begin)     */
  CP_SPEC_E_DEVICE = -7            /* device-side check failed (e.g. code out of range) */
} cp_spec_status;

/* Decoder shape.  dtype: 0 = float32 weights, 1 = bfloat16 weights.
 * Norm gains are always float32.  Requirements: hidden % 8 == 0,
 * ffn % 8 == 0, n_q_heads * head_dim % 8 == 0, head_dim even and <= 256,
 * n_q_heads % n_kv_heads == 0, 1 <= n_layers <= 64,
 * 2 <= num_code_groups <= 64, 2 <= vocab <= 8192. */
typedef struct {
  int32_t hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab, num_code_groups;
  int32_t dtype;
  float rope_theta; /* rotary base, rotate-half pairing (i, i + head_dim/2) */
  float rms_eps;    /* RMSNorm epsilon                                       */
} cp_spec_model;

/* Device pointers to the weights (borrowed, read-only, row-major).
 * embed:   [G-1][V][H]   table j (0-based) embeds c_j as the input of position j+1.
 * lm_head: [G-1][V][H]   index j-1 is head_j (scores c_j).
 * Per layer l: wq [nq*d][H], wk [nkv*d][H], wv [nkv*d][H], wo [H][nq*d],
 * w_gate [F][H], w_up [F][H], w_down [H][F]; attn_norm, ffn_norm [H] fp32.
 * final_norm [H] fp32.  The blocks are pre-norm: h += Wo attn(RMSNorm(h));
 * h += Wdown (silu(Wgate b) * Wup b) with b = RMSNorm(h).
 * draft_offset: [K][H] fp32 position-aware draft offsets b_1..b_K, K =
 * config.draft_offsets (NULL when K = 0).  The draft of lookahead t reads
 * head_{s+t} on h_s + b_t for t <= K, and h_s alone beyond K, where h_s is
 * the final-normed hidden the target head_s reads; the target heads never see
 * an offset, so the committed codes keep the autoregressive law ("RVQ
 * Position Aware Speculative Decoding for On Device TTS", section 2.2 and
 * Figure 3).  The library reads b once, in cp_spec_init (and in every
 * cp_spec_decode_frames_static call), and keeps the products head_j . b_t
 * in the workspace: later changes to the values behind the pointer are not
 * seen by an existing context. */
typedef struct {
  const void* embed;
  const void* lm_head;
  const float* final_norm;
  const float* attn_norm[CP_SPEC_MAX_LAYERS];
  const void* wq[CP_SPEC_MAX_LAYERS];
  const void* wk[CP_SPEC_MAX_LAYERS];
  const void* wv[CP_SPEC_MAX_LAYERS];
  const void* wo[CP_SPEC_MAX_LAYERS];
  const float* ffn_norm[CP_SPEC_MAX_LAYERS];
  const void* w_gate[CP_SPEC_MAX_LAYERS];
  const void* w_up[CP_SPEC_MAX_LAYERS];
  const void* w_down[CP_SPEC_MAX_LAYERS];
  const float* draft_offset;
} cp_spec_weights;

/* verify_window: 0 = autoregressive loop; 2..8 = one committed depth plus
 * N-1 drafted depths ("CodePredictor Speculative Decoding", "Options": 1 is
 * rejected because it leaves no draft slot).  top_k: 1..vocab, the default
 * for every stream and the maximum any stream may use.  temperature: 0 =
 * greedy, else in [1e-3, 100].  max_streams: streams the workspace is sized
 * for (>= 1).  draft_offsets: K, the number of position-aware draft offset
 * vectors in weights.draft_offset, 0..7 (0 = the heads are reused without
 * offsets); offsets beyond verify_window - 1 are never read.
 * adapt_accept_pct, adapt_min_reached: the adaptive window ("Speculative
 * Decoding, Beyond Text", runtime policies).  0 = off: every round drafts
 * min(verify_window - 1, codes left).  With pct in 1..100, each stream picks
 * the window of its next frame from its acceptance by offset earlier in the
 * same cp_spec_decode_frames call: offsets t = 1, 2, ... are kept while each
 * has fewer than adapt_min_reached (>= 1) drafts reached by the left-to-right
 * test, or accepted at least pct percent of them (100 * accepted >= pct *
 * reached); the window is 1 + the kept leading offsets.  Window 1 runs the
 * frame without drafts, one row per pass.  The choice depends only on
 * earlier frames, so the committed codes keep the autoregressive law.  Each
 * call (and each cp_spec_begin_frame) starts with no history, i.e. with the
 * full window. */
typedef struct {
  int32_t verify_window;
  int32_t top_k;
  float temperature;
  uint64_t seed;
  int32_t max_streams;
  int32_t draft_offsets;
  int32_t adapt_accept_pct;
  int32_t adapt_min_reached;
} cp_spec_config;

/* Counters accumulated since init (or the last cp_spec_reset_stats).
 * committed = codes c_1..c_{G-1} emitted; passes = decoder passes (frame
 * prefills + rounds, or AR steps); accepted/drafted_by_offset[t] = drafts at
 * offset t (1..8) accepted / reached by the left-to-right test (every draft
 * up to and including the first rejection; "report acceptance by offset",
 * "Speculative Decoding, Beyond Text", section 06).  weight_bytes and
 * kv_bytes count the algorithmic HBM bytes of all decoder passes (every
 * layer matrix once per pass, each distinct lm_head applied in the pass
 * once, the KV positions each pass reads). */
typedef struct {
  int64_t frames, passes, rounds, committed, bonus, rejections;
  int64_t drafted_by_offset[9];
  int64_t accepted_by_offset[9];
  int64_t weight_bytes, kv_bytes, heads_applied;
  /* Pass kernels executed on the device (5 per layer + lm_heads, top-k and
   * accept, per pass; counted by the accept kernel). */
  int64_t kernel_launches;
  int64_t reserved[7];
} cp_spec_stats;

typedef struct cp_spec_ctx cp_spec_ctx;

/* Bytes of device workspace cp_spec_init needs for this model/config
 * (KV cache, activations, logits, sampling lists, per-stream state).
 * Returns 0 if the arguments are invalid. */
size_t cp_spec_workspace_bytes(const cp_spec_model* model, const cp_spec_config* config);

/* Validate, carve the caller's workspace (d_workspace, >= the size above),
 * initialise device state on the current device (synchronously) and return a
 * context in *out.  Returns CP_SPEC_W_AR_FALLBACK (and a usable context in AR
 * mode) when verify_window >= 2 but num_code_groups < 3, i.e. there is no
 * draft slot after the first code ("CodePredictor Speculative Decoding",
 * "Limitations": automatic fallback).  vocab above CP_SPEC_MAX_VOCAB returns
 * CP_SPEC_E_UNSUPPORTED: there is no second backend and no CPU fallback. */
cp_spec_status cp_spec_init(const cp_spec_model* model, const cp_spec_weights* weights,
                            const cp_spec_config* config, void* d_workspace, size_t workspace_bytes,
                            cp_spec_ctx** out);

/* Sparse draft tree ("RVQ Position Aware Speculative Decoding for On Device
 * TTS", section 2.2 "tree attention / sparse tree attention", Figure 2).
 * HOST arrays of n entries (1 <= n <= 62), nodes listed parents first:
 * parent[i] is -1 for a child of the committed code, else an earlier node;
 * rank[i] is the rank of the node's token among the draft logits of its
 * depth (value descending, index ascending; 0 = the largest), below
 * min(top_k rounded up to a multiple of 4, vocab).  Siblings come in
 * ascending rank without repeats; depth at most CP_SPEC_MAX_WINDOW - 1.
 * The arrays are read during the call only. */
typedef struct {
  int32_t n;
  const int32_t* parent;
  const int32_t* rank;
} cp_spec_tree;

/* Workspace bytes of a tree context (0 if the arguments are invalid). */
size_t cp_spec_workspace_bytes_tree(const cp_spec_model* model, const cp_spec_config* config,
                                    const cp_spec_tree* tree);

/* cp_spec_init for tree rounds instead of chain rounds: every round drafts
 * the tree's nodes (node i carries the rank[i]-th draft logit of head_{s+d}
 * on h_s, d its depth; nodes deeper than the codes left are dropped),
 * verifies the committed code and every node short of the frame end in one
 * pass (each node attends to the prefix and to its own ancestors), and walks
 * the tree from the committed code: the children of a node are tested in
 * rank order as point-mass drafts against the node's target law (accept
 * child c iff u < p'(c), p' the remaining mass renormalised; Philox purpose
 * 4 + the child's index among those tested), and one code is drawn from what
 * remains when none is accepted (purpose TARGET).  Every committed code keeps
 * the autoregressive law; under temperature 0 the codes equal greedy
 * autoregressive decoding.  config->verify_window, adapt_accept_pct and
 * adapt_min_reached are ignored (the tree fixes the drafts); draft_offsets
 * applies to depths 1..K.  The accepted path's K/V rows are copied from the
 * nodes' slots to their positions: the one place a round moves cache data.
 * Decode with cp_spec_decode_frames / cp_spec_begin_frame + cp_spec_round as
 * for chain contexts.  Errors as cp_spec_init, plus CP_SPEC_E_INVALID for a
 * malformed tree or fewer than 3 code groups. */
cp_spec_status cp_spec_init_tree(const cp_spec_model* model, const cp_spec_weights* weights,
                                 const cp_spec_config* config, const cp_spec_tree* tree, void* d_workspace,
                                 size_t workspace_bytes, cp_spec_ctx** out);

/* Per-stream sampling overrides, HOST arrays of n entries (n <= max_streams):
 * top_k in 1..config.top_k, temperature 0 (greedy) or in [1e-3, 100].
 * Synchronous (small host-to-device copy). */
cp_spec_status cp_spec_set_stream_sampling(cp_spec_ctx* ctx, int32_t n, const int32_t* h_top_k,
                                           const float* h_temperature);

/* Decode n_frames frames for streams 0..n_streams-1 (n_streams <= max_streams).
 * d_x: [n_frames][n_streams][H] float32 talker hiddens; d_c0: [n_frames][n_streams]
 * int32 first codes; d_codes (out): [n_frames][n_streams][G] int32, with
 * d_codes[f][b][0] = c_0.  Frame f uses Philox frame index first_frame + f.
 * One launch of the context's call graph on `stream` (a setup kernel, then
 * a device-controlled loop of decoder passes, 5 L + 3 kernels each, until
 * every stream has finished its frames; the graph is built and instantiated
 * on the first call, in host memory); streams advance through their frames
 * independently.  Asynchronous. */
cp_spec_status cp_spec_decode_frames(cp_spec_ctx* ctx, int32_t n_streams, int32_t n_frames,
                                     int32_t first_frame, const float* d_x, const int32_t* d_c0,
                                     int32_t* d_codes, void* stream);

/* Step-wise API.  cp_spec_begin_frame stages one frame for every stream
 * (d_x [n_streams][H], d_c0 [n_streams], both read by later rounds and kept
 * alive by the caller until the frame completes).  Each cp_spec_round runs
 * one decoder pass for every unfinished stream: the first is the frame
 * prefill (rows x, E_0(c_0); commits c_1), later ones are speculative
 * rounds (or AR steps).  d_codes [n_streams][G] receives codes as they are
 * committed; d_committed [n_streams] (optional) receives s+1, the number of
 * codes of the frame known so far (G when the frame is complete).
 * Asynchronous. */
cp_spec_status cp_spec_begin_frame(cp_spec_ctx* ctx, int32_t n_streams, const float* d_x,
                                   const int32_t* d_c0, int32_t frame_idx, void* stream);
cp_spec_status cp_spec_round(cp_spec_ctx* ctx, int32_t* d_codes, int32_t* d_committed, void* stream);

/* Teacher-forced logits, for checking the decoder numerics: rows x,
 * E_0(c_0), ..., E_{P-2}(c_{P-2}) at positions 0..P-1 (2 <= P <= G) for each
 * stream, run through the same verify-pass kernels in chunks of at most
 * max(verify_window, 2) rows.  d_codes [n_streams][P-1]; d_logits (out)
 * [n_streams][P-1][V] = head_j at position j; d_draft_logits (optional, out,
 * speculative configs only) [n_streams][P-1][N-1][V] = head_{j+t} at
 * position j (zero where j+t > G-1).  Asynchronous. */
cp_spec_status cp_spec_teacher_logits(cp_spec_ctx* ctx, int32_t n_streams, int32_t P, const float* d_x,
                                      const int32_t* d_codes, float* d_logits, float* d_draft_logits,
                                      void* stream);

/* Acceptance kernels alone (no model): R independent rounds of N-1 drafts
 * verified against N target rows (2 <= N <= 8, 2 <= V <= 8192).
 * mode 0: d_target [R][N][V] and d_draft [R][N-1][V] are float32 logits,
 *         processed with top_k / temperature as in the full path;
 * mode 1: they are already-processed float32 probabilities (each row's
 *         non-zero entries are its support; top_k/temperature ignored,
 *         temperature 0 not allowed).
 * Draft t (1..N-1) is drawn from draft row t-1 with Philox (r, 0, t, DRAFT),
 * accepted with (r, 0, t, ACCEPT); residual / bonus draws use (r, 0, t,
 * TARGET).  Outputs: d_tokens [R][N] committed codes, -1 padded;
 * d_n_accepted [R]; d_drafts [R][N-1] (optional).  Asynchronous; needs no
 * context and no workspace. */
cp_spec_status cp_spec_accept_batch(int32_t R, int32_t N, int32_t V, int32_t top_k, float temperature,
                                    uint64_t seed, int32_t mode, const float* d_target,
                                    const float* d_draft, int32_t* d_tokens, int32_t* d_n_accepted,
                                    int32_t* d_drafts, void* stream);

/* Decode without any allocation: cp_spec_decode_frames for a one-off job,
 * with no context and no caller workspace.  The pages describe no such call;
 * it exists for callers that cannot allocate device memory when they decode:
 * a runtime with no device allocator of its own, a host whose memory pool is
 * frozen after start-up, or one that must keep its device footprint fixed.
 * The KV cache, activations, sampling lists and stream state live instead in
 * a library-owned array of CP_SPEC_STATIC_SCRATCH_BYTES in the module's
 * global memory, reserved by the CUDA runtime when the library's module is
 * loaded (one copy per device).
 *
 * Arguments are those of cp_spec_init plus cp_spec_decode_frames (same
 * layouts; streams 0..n_streams-1, n_streams <= config->max_streams).  The
 * workspace it needs is cp_spec_workspace_bytes(model, config); above
 * CP_SPEC_STATIC_SCRATCH_BYTES the call returns CP_SPEC_E_WORKSPACE and
 * enqueues nothing (lower max_streams).  d_status (optional, device, one
 * int32, 4-byte aligned; the other device pointers need 16 bytes) receives
 * the device status word after the decode: CP_SPEC_OK,
 * CP_SPEC_E_DEVICE_TIMEOUT or CP_SPEC_E_DEVICE.
 *
 * Every call clears the scratch, resets it to the state cp_spec_init leaves
 * (on `stream`, before the decode) and decodes: results equal those of a
 * fresh context with the same config, bit for bit.  Per-stream sampling
 * overrides and counters are not available.  Asynchronous; returns
 * CP_SPEC_W_AR_FALLBACK under the same condition as cp_spec_init.
 *
 * The first call on each device looks up the scratch address
 * (cudaGetSymbolAddress, which may load the module) and caches it; make that
 * first call before any stream capture begins.  The decode runs as a call
 * graph (host objects, no device allocation by the library) that is cached
 * per device and rebuilt, after a device synchronisation, when the model,
 * weights or configuration change.  All calls on one device share
 * the one scratch array: calls whose work overlaps in time (different
 * streams, or threads without ordering) race on it and give wrong results.
 * Order them on one stream.  Launches count in the context-free counter of
 * cp_spec_launch_count(NULL). */
cp_spec_status cp_spec_decode_frames_static(const cp_spec_model* model, const cp_spec_weights* weights,
                                            const cp_spec_config* config, int32_t n_streams, int32_t n_frames,
                                            int32_t first_frame, const float* d_x, const int32_t* d_c0,
                                            int32_t* d_codes, int32_t* d_status, void* stream);

/* Synchronise `stream` and return the device status word of the context:
 * CP_SPEC_OK, CP_SPEC_E_DEVICE_TIMEOUT or CP_SPEC_E_DEVICE.  Clears it. */
cp_spec_status cp_spec_status_word(cp_spec_ctx* ctx, void* stream);

/* Synchronise `stream` and copy the counters to *h_stats. */
cp_spec_status cp_spec_read_stats(cp_spec_ctx* ctx, cp_spec_stats* h_stats, void* stream);
cp_spec_status cp_spec_reset_stats(cp_spec_ctx* ctx, void* stream);

/* Diagnostic hook for tests (the pages have no counterpart).
 * wait_limit_ns (1e4 .. 6e10; default 2e9) bounds every device-side wait of
 * the context's kernels (a weight or input copy that has not landed): after
 * it the kernel records CP_SPEC_E_DEVICE_TIMEOUT in the status word, waits
 * (with the same bound) for its own copies still in flight and returns; the
 * pass loop then stops.  flags (0 .. 3):
 *   bit 0 (1): one wait of the first decoder kernel of every pass (CTA 0)
 *     never completes, so that wait always runs out;
 *   bit 1 (2): after each decision the accept kernel writes NaN into every
 *     KV slot of the stream that the next pass must not read (positions past
 *     the committed depth, the tree nodes' slots, and at a frame's end the
 *     whole cache), so a pass that read a stale slot would show NaN
 *     ("Speculative Decoding, Beyond Text", section 07: the logical length
 *     and the valid-position mask).
 * 0 restores normal operation.  Nothing traps or spins without a bound.
 * Synchronises the device if the context's call graph exists (it is rebuilt
 * on the next call). */
cp_spec_status cp_spec_test_hooks(cp_spec_ctx* ctx, uint64_t wait_limit_ns, int32_t flags);

/* Number of launches the library has enqueued on this context: kernels
 * launched directly, plus one per launch of the context's call graph (whose
 * pass kernels are counted on the device: cp_spec_stats.kernel_launches).
 * cp_spec_accept_batch and cp_spec_decode_frames_static count in a
 * process-wide counter, ctx = NULL. */
int64_t cp_spec_launch_count(const cp_spec_ctx* ctx);

/* Last error message of the context (or of the last context-free call when
 * ctx is NULL).  Never NULL. */
const char* cp_spec_last_error(const cp_spec_ctx* ctx);

/* Release the host context.  Does not touch the caller's device memory. */
void cp_spec_destroy(cp_spec_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* CP_SPEC_H */
