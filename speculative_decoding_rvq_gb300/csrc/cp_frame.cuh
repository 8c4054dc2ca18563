// cp_frame.cuh -- parameter block and workspace layout of the persistent
// frame kernel (shared by the kernel and the host-side C ABI).
#pragma once
#include <stdint.h>

#include "../../include/cp_spec.h"

namespace cpk {

enum StreamPhase : int { kPhasePrefill = 0, kPhaseAR = 1, kPhaseSpec = 2, kPhaseTeacher = 3, kPhaseDone = 4 };
enum RunMode : int { kModeDecode = 0, kModeTeacher = 1 };

// A CTA is kWarps consumer warps (all compute, sampling and acceptance) plus
// one producer warp that only streams weight tiles into shared memory.  Eight
// warps in all keep two warps per SM sub-partition, so a thread may hold up
// to 255 registers (nine would cap it at 168 and force spills).
constexpr int kWarps = 7;
constexpr int kConsumers = kWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxSlots = 8;        // weight-stream ring depth
constexpr int kMaxTiles = 40;       // tiles of one GEMV kind per CTA
constexpr int kKPart = 512;         // input elements per lane group of a GEMV task (16 per lane)
constexpr int kMaxTileRows = 64;    // weight rows per tile
constexpr int kRB = 4;              // weight rows per GEMV task (a batch)
constexpr int kRedPerTask = kRB * 4;  // partial sums a task writes (batch row x input row)

// GEMV kinds, in weight-stream order within a layer; kHeads closes a pass.
enum GemvKind : int { kQKV = 0, kO = 1, kGU = 2, kDown = 3, kHeads = 4 };

// Per-stream device state (one warp owns it in the accept phase).
struct StreamState {
  int phase;      // StreamPhase of the pass that is in flight
  int frame;      // frame index within the current launch sequence
  int frame_abs;  // Philox frame index
  int s;          // committed depth (codes c_0..c_s known)
  int m;          // rows in the pass in flight
  int pos0;       // position of row 0 of the pass
  int n_d;        // drafts verified by the pass in flight
  int pad;
  int drafts[8];
  int codes[CP_SPEC_MAX_CODE_GROUPS];
};

struct StreamStats {
  long long frames, passes, rounds, committed, bonus, rejections;
  long long drafted[9], accepted[9];
};

// Persistent control words (survive across launches, except `bar`).
struct Control {
  unsigned long long bar;            // grid barrier counter, zeroed before each launch
  unsigned long long head_mask[2];   // lm_heads needed by the next pass (double-buffered by pass parity)
  long long weight_bytes, kv_bytes, heads_applied, passes;
  long long phase_ns[8];             // ns per phase kind as seen by CTA 0
  int active;                        // streams with frames left
  int pass_global;                   // passes run since init: parity of head_mask, exchange flags
  int status;                        // device status word (cp_spec_status values)
  int pad;
  int dbg_pass, dbg_phase, dbg_active, dbg_gen;  // progress record of CTA 0 (diagnostics)
};

// An exchange element: a float32 value in the low word and the flag of the
// pass that wrote it in the high word, stored with one 64-bit access so a
// reader that sees the flag sees the value.
typedef unsigned long long xel;

struct FrameParams {
  // model
  int H, L, nq, nkv, d, F, V, G, dtype;
  float eps;
  int N;    // verify window (0 = autoregressive)
  int NS;   // row slots per stream = max(N, 2)
  int ND;   // draft logit slots per row = max(N - 1, 0)
  int KC;   // list capacity = min(max top_k, V) rounded up to a multiple of 4
  // plan (host-computed)
  int Bmax;          // stream capacity of the workspace (row slots = Bmax * NS)
  int nslots;        // weight-stream ring depth
  int slot_bytes;    // bytes per ring slot
  int accept_warps;  // warps per CTA that own streams in the accept phase
  int off_ring, off_uni, off_red, off_hown, off_rope;  // dynamic shared memory carve-up (bytes; rope -1 = global)
  int uni_floats;    // phase scratch capacity (staged activations, top-k, acceptance)
  int red_floats;    // GEMV partial sums of one phase (floats)
  int hown_cap;      // owned residual values per active row in shared memory
  unsigned long long seed;
  unsigned long long timeout_ns;
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
  // workspace: exchange buffers (xel) written once per pass, indexed by row slot
  xel* hpub;       // [L][2][Bmax*NS][H]  residual after O (0) and after down (1)
  xel* qpub;       // [L][Bmax*NS][nq*d]  query rows after RoPE
  xel* opub;       // [L][Bmax*NS][nq*d]  attention outputs
  xel* apub;       // [L][Bmax*NS][F]     SwiGLU activations
  xel* kv;         // [Bmax][L][2][G][nkv][d]
  xel* logits;     // [Bmax*NS][1+ND][V]
  int* lidx;       // [Bmax*NS][1+ND][KC]
  float* lprob;    // [Bmax*NS][1+ND][KC]
  unsigned long long* lflag;  // [Bmax*NS][1+ND]: count | flag << 32 (release store)
  int* qidx;       // [Bmax][max(ND,1)][KC]
  float* qprob;    // [Bmax][max(ND,1)][KC]
  int* qcount;     // [Bmax][max(ND,1)]
  int* row_pos;    // [Bmax*NS] position, -1 = inactive
  int* row_code;   // [Bmax*NS] code whose embedding is the row input (frame index at position 0)
  StreamState* st; // [Bmax]
  StreamStats* sstats;  // [Bmax]
  float2* rope;    // [G][d/2] (cos, sin)
  int* top_k;      // [Bmax]
  float* temp;     // [Bmax]
  Control* ctl;
  // this launch
  int mode;        // RunMode
  int B;           // streams
  int n_frames;
  int first_frame;
  int max_passes;  // 0 = until every stream finished
  int do_setup;    // stage the first frame / teacher chunk before the first pass
  const float* x;  // [n_frames][B][H]
  const int* c0;   // [n_frames][B]
  int* codes_out;  // [n_frames][B][G]
  int* committed_out;  // [B] or null
  int P;                 // teacher positions
  const int* t_codes;    // [B][P-1]
  float* t_logits;       // [B][P-1][V]
  float* t_draft;        // [B][P-1][ND][V] or null
};

// Per-warp shared scratch of the accept phase: the stream state plus 2*NS
// staged probability lists (index and probability arrays of capacity KC)
// and their lengths.
inline __host__ __device__ size_t accept_scratch_bytes(int NS, int KC) {
  return (sizeof(StreamState) + (size_t)2 * NS * KC * 8 + (size_t)2 * NS * 4 + 15) / 16 * 16;
}

// Workspace carve-up, computed identically by the host for sizing.
struct Layout {
  size_t hpub, qpub, opub, apub, kv, logits, lidx, lprob, lflag, qidx, qprob, qcount, row_pos, row_code, st,
      sstats, rope, top_k, temp, ctl, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline Layout make_layout(int H, int L, int nq, int nkv, int d, int F, int V, int G, int N, int KC, int Bmax) {
  const int NS = N > 2 ? N : 2, ND = N > 1 ? N - 1 : 0, NDq = ND > 0 ? ND : 1;
  const size_t rows = (size_t)Bmax * NS;
  const size_t X = sizeof(xel);
  Layout o{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + bytes, 256); return at; };
  o.hpub = take(X * L * 2 * rows * H);
  o.qpub = take(X * L * rows * nq * d);
  o.opub = take(X * L * rows * nq * d);
  o.apub = take(X * L * rows * F);
  o.kv = take(X * (size_t)Bmax * L * 2 * G * nkv * d);
  o.logits = take(X * rows * (1 + ND) * V);
  o.lidx = take(sizeof(int) * rows * (1 + ND) * KC);
  o.lprob = take(sizeof(float) * rows * (1 + ND) * KC);
  o.lflag = take(8 * rows * (1 + ND));
  o.qidx = take(sizeof(int) * (size_t)Bmax * NDq * KC);
  o.qprob = take(sizeof(float) * (size_t)Bmax * NDq * KC);
  o.qcount = take(sizeof(int) * (size_t)Bmax * NDq);
  o.row_pos = take(sizeof(int) * rows);
  o.row_code = take(sizeof(int) * rows);
  o.st = take(sizeof(StreamState) * (size_t)Bmax);
  o.sstats = take(sizeof(StreamStats) * (size_t)Bmax);
  o.rope = take(sizeof(float) * 2 * (size_t)G * (d / 2));
  o.top_k = take(sizeof(int) * (size_t)Bmax);
  o.temp = take(sizeof(float) * (size_t)Bmax);
  o.ctl = take(sizeof(Control));
  o.total = off;
  return o;
}

}  // namespace cpk
