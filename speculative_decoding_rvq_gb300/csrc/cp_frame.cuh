// cp_frame.cuh -- parameter block and workspace layout of the pass kernels
// (shared by the kernels and the host-side C ABI).
//
// One decoder pass (the verify forward of every active stream's rows, the
// lm_heads, top-k and acceptance) is a chain of 5 L + 3 kernels; consecutive
// kernels overlap through programmatic dependent launch and the chain runs
// inside a CUDA graph whose while loop repeats passes until every stream is
// done.  Kernels exchange data through the plain fp32 buffers below; the
// kernel boundary orders every write before every read of the next kernel.
#pragma once
#include <stdint.h>

#include "../../include/cp_spec.h"

namespace cpk {

enum StreamPhase : int { kPhasePrefill = 0, kPhaseAR = 1, kPhaseSpec = 2, kPhaseTeacher = 3, kPhaseDone = 4 };
enum RunMode : int { kModeDecode = 0, kModeTeacher = 1 };

constexpr int kThreads = 256;               // threads of every pass kernel
constexpr int kWarps = kThreads / 32;
constexpr int kSlotBytes = 48 * 1024;       // GEMV weight tile (two slots per CTA)
constexpr int kRB = 4;                      // weight rows per GEMV batch
constexpr int kMaxTileRows = 192;           // rows of one weight tile (bounds the partial-sum buffer)
constexpr int kMaxHeadsPerPass = 64;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // bounded device waits give up after 2 s
// Small-batch tensor-core GEMV path (contexts with at most kMvMaxRows row slots).
constexpr int kMvMaxRows = 8;        // pass rows: two column groups of four
constexpr int kMvRowPad = 0;         // bytes after each weight row in shared memory (none: rows copied in runs)
constexpr int kMvPhaseBlocks = 4;    // M-blocks of one phase (partial sums held at once)
constexpr int kMvMaxBlocks = 96;     // M-blocks of one CTA
constexpr int kMvMaxPhases = 48;

// GEMV kinds, in pass order within a layer; kHeads closes a pass.
enum GemvKind : int { kQKV = 0, kO = 1, kGU = 2, kDown = 3, kHeads = 4 };

// Per-stream device state (one warp owns it in the accept kernel).
struct StreamState {
  int phase;      // StreamPhase of the pass that is in flight
  int frame;      // frame index within the current launch sequence
  int frame_abs;  // Philox frame index
  int s;          // committed depth (codes c_0..c_s known)
  int m;          // rows in the pass in flight
  int pos0;       // position of row 0 of the pass
  int n_d;        // drafts verified by the pass in flight
  int w;          // verify window of the current frame (the adaptive policy; N when it is off)
  int drafts[8];
  int codes[CP_SPEC_MAX_CODE_GROUPS];
  int reach[8];   // drafts at offsets 1..8 the left-to-right test reached in this call
  int acc[8];     // ... and accepted (the adaptive policy's counters)
};

struct StreamStats {
  long long frames, passes, rounds, committed, bonus, rejections;
  long long drafted[9], accepted[9];
};

// Persistent control words.
struct Control {
  long long weight_bytes, kv_bytes, heads_applied, passes;
  long long phase_ns[8];             // reserved (zero)
  long long kernels;                 // pass kernels executed
  int active;                        // streams with frames left
  int status;                        // device status word (cp_spec_status values)
  int done;                          // CTAs of the current setup/accept kernel that finished (last-CTA election)
  int pass;                          // passes of the current call
  int pad[4];
};
constexpr int kControlCounters = 13;  // long longs reset by cp_spec_reset_stats, from weight_bytes

// The rows of the pass in flight, compacted, and the lm_heads it applies.
struct Plan {
  int nrows;
  int nheads;
  int heads[kMaxHeadsPerPass];
};

// What changes from call to call (in device memory, written before launch).
struct CallArgs {
  int mode;        // RunMode
  int B;           // streams
  int n_frames;
  int first_frame;
  int max_passes;  // 0 = until every stream finished
  int P;           // teacher positions
  int pass_cap;    // passes after which the loop stops with a device error
  int pad;
  const float* x;        // [n_frames][B][H]
  const int* c0;         // [n_frames][B]
  int* codes_out;        // [n_frames][B][G]
  int* committed_out;    // [B] or null
  const int* t_codes;    // [B][P-1]
  float* t_logits;       // [B][P-1][V]
  float* t_draft;        // [B][P-1][ND][V] or null
};

// Tensor map of a weight matrix for the tcgen05 tiles: layer l's wq, wk, wv,
// wo, w_gate, w_up, w_down at 7 l + 0..6, the lm_heads (as one matrix of
// (G - 1) V rows) at 7 L.
enum : int { kMapQ = 0, kMapK = 1, kMapV = 2, kMapO = 3, kMapGate = 4, kMapUp = 5, kMapDown = 6 };
constexpr int kT5M = 128;  // weight rows per tile (the MMA's M)
__host__ __device__ inline int t5_map_index(int L, int l, int which) { return which < 0 ? 7 * L : 7 * l + which; }

// Sparse draft tree of a context ("RVQ Position Aware Speculative Decoding
// for On Device TTS", section 2.2, Figure 2): node i has parent[i] (-1: a
// child of the committed code, else an earlier node) and rank[i], the rank
// of its token among its depth's draft logits (value descending, index
// ascending); siblings come in ascending rank.  Derived on the host: dep[i]
// (1 for a child of the committed code), anc[i] (bit j set for every
// ancestor j of i and for i itself), need[t] (1 + the largest rank at depth
// t) and dmax (the deepest node).
constexpr int kTreeMaxNodes = 62;
struct TreeTab {
  int n, dmax;
  int parent[64];
  int rank[64];
  int dep[64];
  unsigned long long anc[64];
  int need[CP_SPEC_MAX_WINDOW + 1];
};

struct FrameParams {
  // model
  int H, L, nq, nkv, d, F, V, G, dtype;
  float eps;
  int N;    // verify window (0 = autoregressive)
  int NS;   // row slots per stream = max(N, 2)
  int ND;   // draft logit slots per row = max(N - 1, 0)
  int KC;   // list capacity = min(max top_k, V) rounded up to a multiple of 4
  int Bmax; // stream capacity of the workspace (row slots = Bmax * NS)
  int kernels_per_pass;
  int tc;   // bf16 GEMVs on the tensor-core path (contexts with many rows per pass)
  int KO;   // lookaheads with a position-aware draft offset = min(K, ND)
  int adapt_pct;  // adaptive window: keep an offset at >= this acceptance percentage (0 = off)
  int adapt_min;  // ... or while it has fewer reached drafts than this
  int mv;         // bf16 GEMVs on the small-batch tensor-core path (at most kMvMaxRows row slots)
  int mv_slots[5];  // small-batch path: weight-row slots of shared memory per GEMV kind
  int t5;           // bf16 GEMVs as tcgen05 tiles (contexts with many rows per pass)
  int t5_rb[5];     // ... pass rows per CTA tile, per GEMV kind (16, 32 or 64)
  int t5_stages[5]; // ... stages of the weight / input ring, per GEMV kind
  const unsigned char* tmaps;  // ... TMA tensor maps of the weight matrices, 128 bytes each (t5_map_index)
  int test_stall;   // test hook: one bounded wait of the first GEMV of a pass never completes
  int test_poison;  // test hook: the accept kernel writes NaN into the KV slots the next pass must not read
  int tree_n;       // sparse-tree rounds: nodes of the tree (0 = chain rounds)
  int GS;           // KV slots per stream and layer: G canonical positions, then tree_n node slots
  unsigned long long wait_ns;         // limit of every bounded device-side wait
  unsigned long long seed;
  unsigned long long cond;            // graph conditional handle of the pass loop (0 = none)
  long long layer_bytes, head_bytes;  // algorithmic bytes per layer / per lm_head
  const void* embed;
  const void* head;
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
  const float* draft_offset;  // [K][H] b_1..b_K (read by the offset table kernel only)
  // workspace (row slot r = b * NS + k)
  float* h;        // [Bmax*NS][H]     residual stream
  float* qbuf;     // [Bmax*NS][nq*d]  queries after RoPE
  float* abuf;     // [Bmax*NS][nq*d]  attention outputs
  float* fbuf;     // [Bmax*NS][F]     SwiGLU activations
  float* kv;       // [Bmax][L][2][G][nkv][d]
  float* logits;   // [Bmax*NS][1+ND][V]
  float* otab;     // [G-1][KO][V]     head_j . b_t, added to the lookahead-t draft logits
  int* lidx;       // [Bmax*NS][1+ND][KC]
  float* lprob;    // [Bmax*NS][1+ND][KC]
  int* lcount;     // [Bmax*NS][1+ND]
  int* qidx;       // [Bmax][max(ND,1)][KC]
  float* qprob;    // [Bmax][max(ND,1)][KC]
  int* qcount;     // [Bmax][max(ND,1)]
  int* row_pos;    // [Bmax*NS] position, -1 = inactive
  int* row_code;   // [Bmax*NS] code whose embedding is the row input (frame index at position 0)
  int* prow;       // [Bmax*NS] the pass's active row slots, ascending
  int* ppos;       // [Bmax*NS] their positions
  int* pcode;      // [Bmax*NS] their input codes
  int* row_slot;   // [Bmax*NS] KV slot of the row (its position, or G + node index for a tree node)
  int* pslot;      // [Bmax*NS] the pass's rows' KV slots
  int* ttok;       // [Bmax][64] tree rounds: the token of each node of the stream's current tree
  const TreeTab* tree;  // tree rounds: the tree (device copy)
  Plan* plan;
  StreamState* st; // [Bmax]
  StreamStats* sstats;  // [Bmax]
  float2* rope;    // [G][d/2] (cos, sin)
  int* top_k;      // [Bmax]
  float* temp;     // [Bmax]
  Control* ctl;
  CallArgs* call;
};

// Staged probability lists of one stream in the accept kernel: the target
// lists of NSr row slots, NDr saved draft lists q_t, and the NDr draft
// slots of each row (the next pass's candidates).  Chain rounds: NSr = NS =
// max(N, 2), NDr = max(NS - 1, 1).  Tree rounds: NSr = 2 (the walk's
// current list, and the frame prefill's rows), NDr = max(depth, 1).
inline __host__ __device__ int accept_rows(int NS, int tree_n) { return tree_n > 0 ? 2 : NS; }
inline __host__ __device__ int accept_drafts(int NS, int ND, int tree_n) {
  return tree_n > 0 ? (ND > 1 ? ND : 1) : (NS > 2 ? NS - 1 : 1);
}
inline __host__ __device__ int accept_lists(int NSr, int NDr) { return NSr + NDr + NSr * NDr; }

// Per-warp shared scratch of the accept kernel: the stream state, the staged
// lists (index and probability arrays of capacity KC), one list of residual
// weights, 32 uniforms and the list lengths.
inline __host__ __device__ size_t accept_scratch_bytes(int NSr, int NDr, int KC) {
  const size_t n = (size_t)accept_lists(NSr, NDr);
  return (sizeof(StreamState) + n * KC * 8 + (size_t)KC * 4 + 32 * 4 + n * 4 + 15) / 16 * 16;
}

// Workspace carve-up, computed identically by the host for sizing.
struct Layout {
  size_t h, qbuf, abuf, fbuf, kv, logits, otab, lidx, lprob, lcount, qidx, qprob, qcount, row_pos, row_code, prow, ppos,
      pcode, row_slot, pslot, ttok, tree, tmaps, plan, st, sstats, rope, top_k, temp, ctl, call, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// NS row slots per stream, ND draft slots per row, GS KV slots per stream
// and layer (chain rounds: NS = max(N, 2), ND = max(N - 1, 0), GS = G).
inline Layout make_layout(int H, int L, int nq, int nkv, int d, int F, int V, int G, int NS, int ND, int GS, int KC,
                          int Bmax, int KO) {
  const int NDq = ND > 0 ? ND : 1;
  const size_t rows = (size_t)Bmax * NS;
  Layout o{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + bytes, 256); return at; };
  o.h = take(4 * rows * H);
  o.qbuf = take(4 * rows * nq * d);
  o.abuf = take(4 * rows * nq * d);
  o.fbuf = take(4 * rows * F);
  o.kv = take(4 * (size_t)Bmax * L * 2 * GS * nkv * d);
  o.logits = take(4 * rows * (1 + ND) * V);
  o.otab = take(4 * (size_t)(G - 1) * KO * V);
  o.lidx = take(sizeof(int) * rows * (1 + ND) * KC);
  o.lprob = take(sizeof(float) * rows * (1 + ND) * KC);
  o.lcount = take(sizeof(int) * rows * (1 + ND));
  o.qidx = take(sizeof(int) * (size_t)Bmax * NDq * KC);
  o.qprob = take(sizeof(float) * (size_t)Bmax * NDq * KC);
  o.qcount = take(sizeof(int) * (size_t)Bmax * NDq);
  o.row_pos = take(sizeof(int) * rows);
  o.row_code = take(sizeof(int) * rows);
  o.prow = take(sizeof(int) * rows);
  o.ppos = take(sizeof(int) * rows);
  o.pcode = take(sizeof(int) * rows);
  o.row_slot = take(sizeof(int) * rows);
  o.pslot = take(sizeof(int) * rows);
  o.ttok = take(sizeof(int) * (size_t)Bmax * 64);
  o.tree = take(sizeof(TreeTab));
  o.tmaps = take((size_t)(7 * L + 1) * 128);  // tensor maps of the weight matrices (tcgen05 tiles)
  o.plan = take(sizeof(Plan));
  o.st = take(sizeof(StreamState) * (size_t)Bmax);
  o.sstats = take(sizeof(StreamStats) * (size_t)Bmax);
  o.rope = take(sizeof(float) * 2 * (size_t)G * (d / 2));
  o.top_k = take(sizeof(int) * (size_t)Bmax);
  o.temp = take(sizeof(float) * (size_t)Bmax);
  o.ctl = take(sizeof(Control));
  o.call = take(sizeof(CallArgs));
  o.total = off;
  return o;
}

}  // namespace cpk
