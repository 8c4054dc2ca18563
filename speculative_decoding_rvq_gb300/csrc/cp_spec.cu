// cp_spec.cu -- host side of the C ABI declared in include/cp_spec.h.
//
// Validates arguments, carves the caller's workspace, fills the launch
// parameter block and enqueues the kernels.  Never allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/cp_spec.h"
#include "cp_frame.cuh"

namespace cpk_host {
cudaError_t configure_kernels(const cpk::FrameParams& P, int accept_warps);
cudaError_t enqueue_setup(const cpk::FrameParams& P, int accept_warps, cudaStream_t s);
cudaError_t enqueue_pass(const cpk::FrameParams& P, int sms, int accept_warps, cudaStream_t s);
cudaError_t build_call_graph(cpk::FrameParams P, int sms, int accept_warps, cudaStream_t cs, cudaGraphExec_t* out);
size_t accept_smem(const cpk::FrameParams& P, int warps);
cudaError_t launch_init_tables(float2* rope, int G, int d, double theta, int* top_k, float* temp, int Bmax, int k,
                               float T, cudaStream_t stream);
cudaError_t launch_offset_table(const cpk::FrameParams& P, cudaStream_t stream);
bool plan_mv(cpk::FrameParams& P, int sms);
bool plan_t5(cpk::FrameParams& P, int sms);
cudaError_t launch_accept_batch(int R, int N, int V, int k, float T, unsigned long long seed, int mode,
                                const float* tgt, const float* drf, int* tokens, int* nacc, int* drafts,
                                cudaStream_t stream);
}  // namespace cpk_host

struct cp_spec_ctx {
  cp_spec_model model;
  cp_spec_weights weights;
  cp_spec_config config;
  int N;  // effective window (0 after an AR fallback)
  int device, sms, accept_warps;
  cpk::Layout lay;
  unsigned char* ws;
  cpk::FrameParams base;
  long long launches;
  std::string err;
  // the call graph (setup + pass loop), built on the first whole-call decode
  cudaGraphExec_t graph;
  cudaStream_t capture;
  // step-wise API
  bool staged, need_setup;
  int staged_B, staged_frame;
  const float* staged_x;
  const int* staged_c0;
};

namespace {

std::string g_err = "";
std::atomic<long long> g_free_launches{0};

cp_spec_status fail(cp_spec_ctx* c, cp_spec_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) c->err = buf; else g_err = buf;
  return s;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

cp_spec_status check_cuda(cp_spec_ctx* c, cudaError_t e, const char* what) {
  if (e == cudaSuccess) return CP_SPEC_OK;
  return fail(c, CP_SPEC_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int window_of(const cp_spec_config* cfg) { return cfg->verify_window; }

cp_spec_status validate(const cp_spec_model* m, const cp_spec_config* cfg, cp_spec_ctx* c) {
  if (!m || !cfg) return fail(c, CP_SPEC_E_INVALID, "null model or config");
  if (m->dtype != 0 && m->dtype != 1) return fail(c, CP_SPEC_E_INVALID, "dtype must be 0 (fp32) or 1 (bf16)");
  if (m->hidden <= 0 || m->hidden % 16) return fail(c, CP_SPEC_E_UNSUPPORTED, "hidden must be a positive multiple of 16");
  if (m->ffn <= 0 || m->ffn % 16) return fail(c, CP_SPEC_E_UNSUPPORTED, "ffn must be a positive multiple of 16");
  if (m->head_dim <= 0 || m->head_dim % 8 || m->head_dim > 256)
    return fail(c, CP_SPEC_E_UNSUPPORTED, "head_dim must be a multiple of 8 in [8, 256]");
  if (m->n_q_heads <= 0 || m->n_kv_heads <= 0 || m->n_q_heads % m->n_kv_heads)
    return fail(c, CP_SPEC_E_UNSUPPORTED, "n_q_heads must be a positive multiple of n_kv_heads");
  if ((m->n_q_heads * m->head_dim) % 16)
    return fail(c, CP_SPEC_E_UNSUPPORTED, "n_q_heads*head_dim must be a multiple of 16");
  if (m->n_layers < 1 || m->n_layers > CP_SPEC_MAX_LAYERS) return fail(c, CP_SPEC_E_UNSUPPORTED, "n_layers must be in [1, 64]");
  if (m->num_code_groups < 2 || m->num_code_groups > CP_SPEC_MAX_CODE_GROUPS)
    return fail(c, CP_SPEC_E_INVALID, "num_code_groups must be in [2, 64]");
  if (m->vocab < 2 || m->vocab % 2) return fail(c, CP_SPEC_E_UNSUPPORTED, "vocab must be even and >= 2");
  if (m->vocab > CP_SPEC_MAX_VOCAB)
    return fail(c, CP_SPEC_E_UNSUPPORTED, "vocab %d above the small-vocabulary bound %d", m->vocab, CP_SPEC_MAX_VOCAB);
  if (!(m->rope_theta > 0.0f) || !(m->rms_eps >= 0.0f)) return fail(c, CP_SPEC_E_INVALID, "bad rope_theta or rms_eps");
  const int N = window_of(cfg);
  if (!(N == 0 || (N >= 2 && N <= CP_SPEC_MAX_WINDOW)))
    return fail(c, CP_SPEC_E_INVALID, "verify_window must be 0 or in [2, 8] (1 leaves no draft slot)");
  if (cfg->top_k < 1 || cfg->top_k > m->vocab) return fail(c, CP_SPEC_E_INVALID, "top_k must be in [1, vocab]");
  const float T = cfg->temperature;
  if (!(T == 0.0f || (T >= 1e-3f && T <= 100.0f))) return fail(c, CP_SPEC_E_INVALID, "temperature must be 0 or in [1e-3, 100]");
  if (cfg->max_streams < 1) return fail(c, CP_SPEC_E_INVALID, "max_streams must be >= 1");
  if (cfg->draft_offsets < 0 || cfg->draft_offsets > CP_SPEC_MAX_WINDOW - 1)
    return fail(c, CP_SPEC_E_INVALID, "draft_offsets must be in [0, %d]", CP_SPEC_MAX_WINDOW - 1);
  if (cfg->adapt_accept_pct < 0 || cfg->adapt_accept_pct > 100 ||
      (cfg->adapt_accept_pct > 0 && cfg->adapt_min_reached < 1))
    return fail(c, CP_SPEC_E_INVALID, "adapt_accept_pct must be in [0, 100], with adapt_min_reached >= 1 when set");
  return CP_SPEC_OK;
}

int effective_window(const cp_spec_model* m, const cp_spec_config* cfg) {
  const int N = window_of(cfg);
  if (N >= 2 && m->num_code_groups < 3) return 0;  // no draft slot after c_1: AR fallback
  return N;
}

// List capacity: min(top_k, V) rounded up to a multiple of 4 so every list
// row is 16-byte aligned for cp.async staging.
int list_capacity(const cp_spec_model* m, const cp_spec_config* cfg) {
  const int k = cfg->top_k < m->vocab ? cfg->top_k : m->vocab;
  return (k + 3) / 4 * 4;
}

// Lookaheads that carry a position-aware draft offset: offsets beyond the
// drafted depths (N - 1) are never read.
int offset_lookaheads(const cp_spec_config* cfg, int N) {
  const int ND = N > 1 ? N - 1 : 0;
  return cfg->draft_offsets < ND ? cfg->draft_offsets : ND;
}

// Row slots per stream, draft slots per row and KV slots per stream and
// layer: chain rounds NS = max(N, 2), ND = max(N - 1, 0), GS = G; tree
// rounds NS = 1 + nodes (the root row, then one per node), ND = the tree's
// depth, GS = G + nodes.
struct Slots {
  int NS, ND, GS;
};
Slots slots_for(const cp_spec_model* m, int N, const cpk::TreeTab* tree) {
  if (tree) return Slots{1 + tree->n, tree->dmax, m->num_code_groups + tree->n};
  return Slots{N > 2 ? N : 2, N > 1 ? N - 1 : 0, m->num_code_groups};
}

cpk::Layout layout_for(const cp_spec_model* m, const cp_spec_config* cfg, int N, const cpk::TreeTab* tree = nullptr) {
  const int KC = list_capacity(m, cfg);
  const Slots sl = slots_for(m, N, tree);
  return cpk::make_layout(m->hidden, m->n_layers, m->n_q_heads, m->n_kv_heads, m->head_dim, m->ffn, m->vocab,
                          m->num_code_groups, sl.NS, sl.ND, sl.GS, KC, cfg->max_streams, offset_lookaheads(cfg, N));
}

// Checks a sparse tree ("RVQ Position Aware Speculative Decoding for On
// Device TTS", section 2.2, Figure 2) and derives its table: 1..62 nodes,
// parents first, siblings in ascending rank without repeats, depth at most
// CP_SPEC_MAX_WINDOW - 1, and every rank below the list capacity (a draft
// slot's list holds the candidates up to the largest rank of its depth).
cp_spec_status build_tree(const cp_spec_model* m, const cp_spec_config* cfg, const cp_spec_tree* t, cpk::TreeTab* out) {
  if (!t) return fail(nullptr, CP_SPEC_E_INVALID, "tree is null");
  if (t->n < 1 || t->n > cpk::kTreeMaxNodes || !t->parent || !t->rank)
    return fail(nullptr, CP_SPEC_E_INVALID, "tree needs 1..%d nodes with parent and rank arrays", cpk::kTreeMaxNodes);
  cpk::TreeTab T;
  memset(&T, 0, sizeof T);
  T.n = t->n;
  const int KC = list_capacity(m, cfg);
  for (int i = 0; i < t->n; ++i) {
    const int par = t->parent[i], rk = t->rank[i];
    if (par < -1 || par >= i) return fail(nullptr, CP_SPEC_E_INVALID, "tree node %d: parent must be -1 or an earlier node", i);
    if (rk < 0 || rk >= KC || rk >= m->vocab)
      return fail(nullptr, CP_SPEC_E_INVALID, "tree node %d: rank %d outside [0, %d)", i, rk, std::min(KC, m->vocab));
    for (int j = 0; j < i; ++j)
      if (t->parent[j] == par && t->rank[j] >= rk)
        return fail(nullptr, CP_SPEC_E_INVALID, "tree node %d: siblings must come in ascending rank", i);
    T.parent[i] = par;
    T.rank[i] = rk;
    T.dep[i] = par < 0 ? 1 : T.dep[par] + 1;
    T.anc[i] = (par < 0 ? 0ull : T.anc[par]) | (1ull << i);
    if (T.dep[i] > CP_SPEC_MAX_WINDOW - 1)
      return fail(nullptr, CP_SPEC_E_INVALID, "tree node %d: depth above %d", i, CP_SPEC_MAX_WINDOW - 1);
    T.dmax = std::max(T.dmax, T.dep[i]);
    T.need[T.dep[i]] = std::max(T.need[T.dep[i]], rk + 1);
  }
  *out = T;
  return CP_SPEC_OK;
}

template <typename T>
T* at(unsigned char* base, size_t off) { return reinterpret_cast<T*>(base + off); }

cp_spec_status check_weights(const cp_spec_model* model, const cp_spec_config* config, const cp_spec_weights* weights) {
  if (!weights) return fail(nullptr, CP_SPEC_E_INVALID, "weights is null");
  if (config->draft_offsets > 0 && (!weights->draft_offset || !aligned16(weights->draft_offset)))
    return fail(nullptr, CP_SPEC_E_INVALID, "draft_offsets > 0 needs a 16-byte aligned draft_offset pointer");
  const void* ptrs[] = {weights->embed, weights->lm_head, weights->final_norm};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return fail(nullptr, CP_SPEC_E_INVALID, "embed/lm_head/final_norm null or not 16-byte aligned");
  for (int l = 0; l < model->n_layers; ++l) {
    const void* lp[] = {weights->attn_norm[l], weights->wq[l], weights->wk[l], weights->wv[l], weights->wo[l],
                        weights->ffn_norm[l], weights->w_gate[l], weights->w_up[l], weights->w_down[l]};
    for (const void* p : lp)
      if (!p || !aligned16(p)) return fail(nullptr, CP_SPEC_E_INVALID, "layer %d weight null or not 16-byte aligned", l);
  }
  return CP_SPEC_OK;
}

// Shape limits of the pass kernels (checked before anything is launched).
constexpr size_t kSmemPerSm = 227 * 1024;
constexpr int kMaxChunksPerRow = 3 * cpk::kThreads;  // a GEMV thread owns at most 3 chunks of a row
constexpr int kRedFloatsHost = 1536;                 // the GEMV kernel's partial-sum buffer (floats)
constexpr int kRedQHost = 8;                         // its input-row stride
constexpr int kTcMinRows = 32;                       // rows per pass (max_streams x row slots) that select the tensor path

cp_spec_status check_shapes(const cp_spec_model* m, int N, int KC) {
  const size_t eb = m->dtype == 1 ? 2 : 4;
  const int H = m->hidden, F = m->ffn, QD = m->n_q_heads * m->head_dim;
  const size_t unit = std::max(std::max((size_t)2 * H, (size_t)QD), (size_t)F) * eb;
  if (unit > (size_t)cpk::kSlotBytes)
    return fail(nullptr, CP_SPEC_E_UNSUPPORTED, "a weight row pair of %zu bytes exceeds the %d-byte tile", unit, cpk::kSlotBytes);
  const size_t maxk = (size_t)std::max(std::max(H, QD), F) * eb / 16;
  if (maxk > (size_t)kMaxChunksPerRow)
    return fail(nullptr, CP_SPEC_E_UNSUPPORTED, "GEMV width %zu bytes above %d", maxk * 16, kMaxChunksPerRow * 16);
  if (m->num_code_groups > 64 ||
      ((size_t)2 * m->num_code_groups * m->head_dim + (size_t)(m->n_q_heads / m->n_kv_heads) * m->head_dim + 4 * 64) * 4 >
          kSmemPerSm)
    return fail(nullptr, CP_SPEC_E_UNSUPPORTED, "attention scratch too large");
  // partial sums of one GEMV tile: rows x 8 input rows x warps per row group
  // (the kernel's tile and row-group geometry, restated)
  const int Ks[4] = {H, QD, F, H};
  const int rpus[4] = {2, 1, 1, 1};
  for (int i = 0; i < 4; ++i) {
    const int nch = (int)((size_t)Ks[i] * eb / 16);
    const int TPG = std::min(cpk::kThreads, (nch + 31) / 32 * 32);
    const int WPG = TPG / 32;
    const int rows = std::max(1, std::min((int)(cpk::kSlotBytes / ((size_t)rpus[i] * nch * 16)), cpk::kMaxTileRows / rpus[i])) * rpus[i];
    if ((size_t)rows * kRedQHost * WPG > (size_t)kRedFloatsHost / 2)  // two tiles' sums at once
      return fail(nullptr, CP_SPEC_E_UNSUPPORTED, "GEMV partial-sum buffer too small for width %d", Ks[i]);
  }
  (void)N;
  (void)KC;
  return CP_SPEC_OK;
}

// Device facts of one configuration.
struct DevicePlan {
  int dev, sms, KC, accept_warps;
};

// Queries the current device and checks that the configuration fits the
// pass kernels (shared memory of the top-k and accept kernels).
cp_spec_status plan_device(const cp_spec_model* model, const cp_spec_config* config, int N, DevicePlan* dp,
                           const cpk::TreeTab* tree = nullptr) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return check_cuda(nullptr, e, "device query");
  const int KC = list_capacity(model, config);
  cp_spec_status v = check_shapes(model, N, KC);
  if (v != CP_SPEC_OK) return v;
  const Slots sl = slots_for(model, N, tree);
  const int tn = tree ? tree->n : 0;
  const size_t per_warp =
      cpk::accept_scratch_bytes(cpk::accept_rows(sl.NS, tn), cpk::accept_drafts(sl.NS, sl.ND, tn), KC);
  const int aw = (int)std::min<size_t>(cpk::kWarps, kSmemPerSm / per_warp);
  if (aw < 1)
    return fail(nullptr, CP_SPEC_E_UNSUPPORTED, "top_k %d too large for verify window %d (accept lists exceed shared memory)",
                config->top_k, config->verify_window);
  const size_t topk_b = ((size_t)model->vocab * 4 + 15) / 16 * 16 + (size_t)cpk::kWarps * 1024 + ((size_t)KC * 4 + 15) / 16 * 16 + 256;
  if (topk_b > kSmemPerSm) return fail(nullptr, CP_SPEC_E_UNSUPPORTED, "vocabulary too large for the top-k kernel");
  *dp = DevicePlan{dev, sms, KC, aw};
  return CP_SPEC_OK;
}

// Fills the launch-invariant parameters: model shape, weight pointers and
// the carve-up of the workspace at `ws`.
void fill_params(const cp_spec_model* model, const cp_spec_weights* weights, const cp_spec_config* config, int N,
                 const DevicePlan& dp, const cpk::Layout& lay, unsigned char* ws, cpk::FrameParams* out,
                 const cpk::TreeTab* tree = nullptr) {
  cpk::FrameParams& P = *out;
  memset(&P, 0, sizeof P);
  const int L = model->n_layers;
  const Slots sl = slots_for(model, N, tree);
  const int NS = sl.NS;
  P.H = model->hidden; P.L = L; P.nq = model->n_q_heads; P.nkv = model->n_kv_heads; P.d = model->head_dim;
  P.F = model->ffn; P.V = model->vocab; P.G = model->num_code_groups; P.dtype = model->dtype;
  P.eps = model->rms_eps;
  P.N = N; P.NS = NS; P.ND = sl.ND; P.KC = dp.KC;
  P.tree_n = tree ? tree->n : 0;
  P.GS = sl.GS;
  P.Bmax = config->max_streams;
  P.kernels_per_pass = 5 * L + 3;
  P.KO = offset_lookaheads(config, N);
  P.adapt_pct = tree ? 0 : config->adapt_accept_pct;  // the tree fixes the drafts of every round
  P.adapt_min = config->adapt_min_reached;
  // bf16 contexts with many rows per pass run the GEMVs on tensor cores
  // (every GEMV width a multiple of 32); the choice depends on the context,
  // not on the pass, so a stream's results do not depend on its batch-mates
  P.tc = (model->dtype == 1 && config->max_streams * NS >= kTcMinRows && model->hidden % 32 == 0 &&
          model->ffn % 32 == 0 && (model->n_q_heads * model->head_dim) % 32 == 0) ? 1 : 0;
  P.mv = 0;
  P.t5 = 0;
  if (!P.tc) cpk_host::plan_mv(P, dp.sms);  // bf16 contexts with at most 8 row slots
  else cpk_host::plan_t5(P, dp.sms);        // tcgen05 tiles where the shape fits them
  P.wait_ns = cpk::kDefaultWaitNs;
  P.test_stall = 0;
  P.test_poison = 0;
  P.seed = config->seed;
  P.cond = 0;
  const long long eb = model->dtype == 1 ? 2 : 4;
  const long long H = model->hidden, qd = (long long)model->n_q_heads * model->head_dim,
                  kvd = (long long)model->n_kv_heads * model->head_dim, F = model->ffn;
  P.layer_bytes = (qd * H + 2 * kvd * H + H * qd + 3 * F * H) * eb + 2 * H * 4;
  P.head_bytes = (long long)model->vocab * H * eb;
  P.embed = weights->embed; P.head = weights->lm_head; P.final_norm = weights->final_norm;
  for (int l = 0; l < L; ++l) {
    P.attn_norm[l] = weights->attn_norm[l]; P.wq[l] = weights->wq[l]; P.wk[l] = weights->wk[l];
    P.wv[l] = weights->wv[l]; P.wo[l] = weights->wo[l]; P.ffn_norm[l] = weights->ffn_norm[l];
    P.w_gate[l] = weights->w_gate[l]; P.w_up[l] = weights->w_up[l]; P.w_down[l] = weights->w_down[l];
  }
  P.draft_offset = P.KO > 0 ? weights->draft_offset : nullptr;
  P.h = at<float>(ws, lay.h); P.qbuf = at<float>(ws, lay.qbuf); P.abuf = at<float>(ws, lay.abuf);
  P.fbuf = at<float>(ws, lay.fbuf); P.kv = at<float>(ws, lay.kv); P.logits = at<float>(ws, lay.logits);
  P.otab = at<float>(ws, lay.otab);
  P.lidx = at<int>(ws, lay.lidx); P.lprob = at<float>(ws, lay.lprob); P.lcount = at<int>(ws, lay.lcount);
  P.qidx = at<int>(ws, lay.qidx); P.qprob = at<float>(ws, lay.qprob); P.qcount = at<int>(ws, lay.qcount);
  P.row_pos = at<int>(ws, lay.row_pos); P.row_code = at<int>(ws, lay.row_code);
  P.prow = at<int>(ws, lay.prow); P.ppos = at<int>(ws, lay.ppos); P.pcode = at<int>(ws, lay.pcode);
  P.row_slot = at<int>(ws, lay.row_slot); P.pslot = at<int>(ws, lay.pslot); P.ttok = at<int>(ws, lay.ttok);
  P.tree = at<cpk::TreeTab>(ws, lay.tree);
  P.tmaps = at<unsigned char>(ws, lay.tmaps);
  P.plan = at<cpk::Plan>(ws, lay.plan);
  P.st = at<cpk::StreamState>(ws, lay.st); P.sstats = at<cpk::StreamStats>(ws, lay.sstats); P.rope = at<float2>(ws, lay.rope);
  P.top_k = at<int>(ws, lay.top_k); P.temp = at<float>(ws, lay.temp); P.ctl = at<cpk::Control>(ws, lay.ctl);
  P.call = at<cpk::CallArgs>(ws, lay.call);
}

// TMA tensor maps of the weight matrices for the tcgen05 tiles: bf16, 2D
// (K contiguous, then rows), boxes of 64 K elements (128 bytes, the
// 128-byte swizzle span) by the rows one copy of a tile's slab covers (d/2 for
// the RoPE halves of Wq / Wk / Wv, 64 for gate and up, 128 otherwise).
// cuTensorMapEncodeTiled comes from the driver through the runtime's entry
// point query.  Returns false (and leaves the tiles off) if the driver does
// not provide it or a map is rejected.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool build_tmaps(const cpk::FrameParams& P, std::vector<CUtensorMap>* out) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  out->assign((size_t)7 * P.L + 1, CUtensorMap{});
  auto one = [&](int idx, const void* base, long long rows, long long K, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1u, 1u};
    return enc(&(*out)[idx], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const int half = P.d / 2, QD = P.nq * P.d, KD = P.nkv * P.d;
  bool ok = true;
  for (int l = 0; l < P.L && ok; ++l) {
    ok = one(cpk::t5_map_index(P.L, l, cpk::kMapQ), P.wq[l], QD, P.H, half) &&
         one(cpk::t5_map_index(P.L, l, cpk::kMapK), P.wk[l], KD, P.H, half) &&
         one(cpk::t5_map_index(P.L, l, cpk::kMapV), P.wv[l], KD, P.H, half) &&
         one(cpk::t5_map_index(P.L, l, cpk::kMapO), P.wo[l], P.H, QD, cpk::kT5M) &&
         one(cpk::t5_map_index(P.L, l, cpk::kMapGate), P.w_gate[l], P.F, P.H, cpk::kT5M / 2) &&
         one(cpk::t5_map_index(P.L, l, cpk::kMapUp), P.w_up[l], P.F, P.H, cpk::kT5M / 2) &&
         one(cpk::t5_map_index(P.L, l, cpk::kMapDown), P.w_down[l], P.H, P.F, cpk::kT5M);
  }
  if (ok) ok = one(cpk::t5_map_index(P.L, 0, -1), P.head, (long long)(P.G - 1) * P.V, P.H, cpk::kT5M);
  return ok;
}

// Pass cap of a call: every pass commits at least one code of every
// unfinished stream, so a decode needs at most n_frames * (G - 1) passes and
// a teacher run ceil(P / NS); anything beyond that is a logic error,
// reported, not looped.
int pass_cap_of(const cpk::FrameParams& P, const cpk::CallArgs& ca) {
  if (ca.max_passes > 0) return ca.max_passes;
  if (ca.mode == cpk::kModeTeacher) return (ca.P + P.NS - 1) / P.NS + 1;
  return ca.n_frames * (P.G - 1) + 1;
}

// Copies the call arguments to the device (ordered on `s`).
cp_spec_status put_call(cp_spec_ctx* c, const cpk::FrameParams& P, cpk::CallArgs ca, cudaStream_t s) {
  ca.pass_cap = pass_cap_of(P, ca);
  cudaError_t e = cudaMemcpyAsync(P.call, &ca, sizeof ca, cudaMemcpyHostToDevice, s);
  return check_cuda(c, e, "call arguments copy");
}

// A whole call through the context's graph (built on first use).
cp_spec_status run_call(cp_spec_ctx* c, const cpk::CallArgs& ca, cudaStream_t s) {
  if (!c->graph) {
    cudaError_t e = cudaSuccess;
    if (!c->capture) e = cudaStreamCreateWithFlags(&c->capture, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cpk_host::build_call_graph(c->base, c->sms, c->accept_warps, c->capture, &c->graph);
    if (e != cudaSuccess) { c->graph = nullptr; return check_cuda(c, e, "call graph"); }
  }
  cp_spec_status v = put_call(c, c->base, ca, s);
  if (v != CP_SPEC_OK) return v;
  cudaError_t e = cudaGraphLaunch(c->graph, s);
  if (e != cudaSuccess) return check_cuda(c, e, "graph launch");
  c->launches += 1;
  return CP_SPEC_OK;
}

// Scratch of cp_spec_decode_frames_static: a fixed array in this module's
// global memory, reserved by the CUDA runtime when the module is loaded on a
// device (one copy per device), so the call itself reserves nothing.
__device__ __align__(256) unsigned char g_static_scratch[CP_SPEC_STATIC_SCRATCH_BYTES];

constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mu;
unsigned char* g_static_addr[kMaxStaticDevices] = {};

// Address of g_static_scratch on device `dev` (the current device), looked up
// on the first call for that device and cached.
cp_spec_status static_scratch(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxStaticDevices)
    return fail(nullptr, CP_SPEC_E_UNSUPPORTED, "device ordinal %d above %d", dev, kMaxStaticDevices - 1);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return check_cuda(nullptr, e, "cudaGetSymbolAddress(static scratch)");
    if (!p || !aligned16(p)) return fail(nullptr, CP_SPEC_E_CUDA, "static scratch address not 16-byte aligned");
    g_static_addr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_static_addr[dev];
  return CP_SPEC_OK;
}

// The call graph of cp_spec_decode_frames_static, cached per device for the
// last parameter block it was built for (rebuilt, after a device
// synchronisation, when the model, weights or configuration change).
struct StaticGraph {
  bool valid;
  cpk::FrameParams P;
  cudaGraphExec_t exec;
  cudaStream_t capture;
};
StaticGraph g_static_graph[kMaxStaticDevices];

cp_spec_status static_graph(const DevicePlan& dp, const cpk::FrameParams& P, cudaGraphExec_t* out) {
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticGraph& sg = g_static_graph[dp.dev];
  if (sg.valid && memcmp(&sg.P, &P, sizeof P) == 0) { *out = sg.exec; return CP_SPEC_OK; }
  cudaError_t e = cudaSuccess;
  if (sg.valid) {
    e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaGraphExecDestroy(sg.exec);
    sg.valid = false;
    if (e != cudaSuccess) return check_cuda(nullptr, e, "static graph rebuild");
  }
  if (!sg.capture) e = cudaStreamCreateWithFlags(&sg.capture, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cpk_host::configure_kernels(P, dp.accept_warps);
  if (e == cudaSuccess) e = cpk_host::build_call_graph(P, dp.sms, dp.accept_warps, sg.capture, &sg.exec);
  if (e != cudaSuccess) return check_cuda(nullptr, e, "static call graph");
  sg.P = P;
  sg.valid = true;
  *out = sg.exec;
  return CP_SPEC_OK;
}

}  // namespace

extern "C" {

size_t cp_spec_workspace_bytes(const cp_spec_model* model, const cp_spec_config* config) {
  if (validate(model, config, nullptr) != CP_SPEC_OK) return 0;
  return layout_for(model, config, effective_window(model, config)).total;
}

}  // extern "C"

namespace {

// cp_spec_init, with a sparse tree (tree != null) or chain rounds.
cp_spec_status init_impl(const cp_spec_model* model, const cp_spec_weights* weights, const cp_spec_config* config,
                         const cp_spec_tree* tree_in, void* d_workspace, size_t workspace_bytes, cp_spec_ctx** out) {
  if (!out) return fail(nullptr, CP_SPEC_E_INVALID, "out is null");
  *out = nullptr;
  cp_spec_status v = validate(model, config, nullptr);
  if (v != CP_SPEC_OK) return v;
  v = check_weights(model, config, weights);
  if (v != CP_SPEC_OK) return v;
  if (!d_workspace || !aligned16(d_workspace)) return fail(nullptr, CP_SPEC_E_INVALID, "workspace null or not 16-byte aligned");
  cpk::TreeTab tab;
  const cpk::TreeTab* tree = nullptr;
  if (tree_in) {
    v = build_tree(model, config, tree_in, &tab);
    if (v != CP_SPEC_OK) return v;
    if (model->num_code_groups < 3) return fail(nullptr, CP_SPEC_E_INVALID, "tree rounds need at least 3 code groups");
    tree = &tab;
  }
  const int N = tree ? tree->dmax + 1 : effective_window(model, config);
  const cpk::Layout lay = layout_for(model, config, N, tree);
  if (workspace_bytes < lay.total)
    return fail(nullptr, CP_SPEC_E_WORKSPACE, "workspace %zu bytes < required %zu", workspace_bytes, lay.total);
  DevicePlan dp;
  v = plan_device(model, config, N, &dp, tree);
  if (v != CP_SPEC_OK) return v;

  cp_spec_ctx* c = new (std::nothrow) cp_spec_ctx();
  if (!c) return fail(nullptr, CP_SPEC_E_INVALID, "host allocation failed");
  c->model = *model;
  c->weights = *weights;
  c->config = *config;
  c->N = N;
  c->device = dp.dev;
  c->sms = dp.sms;
  c->accept_warps = dp.accept_warps;
  c->lay = lay;
  c->ws = static_cast<unsigned char*>(d_workspace);
  c->launches = 0;
  c->graph = nullptr;
  c->capture = nullptr;
  c->staged = c->need_setup = false;

  cpk::FrameParams& P = c->base;
  fill_params(model, weights, config, N, dp, lay, c->ws, &P, tree);
  std::vector<CUtensorMap> maps;
  if (P.t5 && !build_tmaps(P, &maps)) P.t5 = 0;  // no tensor maps: the tiles stay off

  cudaError_t e = cpk_host::configure_kernels(P, dp.accept_warps);
  if (e == cudaSuccess) e = cudaMemset(c->ws, 0, lay.total);
  if (e == cudaSuccess && tree) e = cudaMemcpy((void*)P.tree, tree, sizeof *tree, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && P.t5)
    e = cudaMemcpy((void*)P.tmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemset(P.row_pos, 0xFF, sizeof(int) * (size_t)config->max_streams * P.NS);
  if (e == cudaSuccess)
    e = cpk_host::launch_init_tables(P.rope, P.G, P.d, (double)model->rope_theta, P.top_k, P.temp, config->max_streams,
                                     config->top_k, config->temperature, 0);
  if (e == cudaSuccess && P.KO > 0) e = cpk_host::launch_offset_table(P, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cp_spec_status s = check_cuda(nullptr, e, "workspace initialisation");
    delete c;
    return s;
  }
  c->launches += P.KO > 0 ? 2 : 1;
  *out = c;
  if (!tree && N != window_of(config)) {
    c->err = "speculation disabled: fewer than 3 code groups leave no draft slot; running the autoregressive loop";
    return CP_SPEC_W_AR_FALLBACK;
  }
  return CP_SPEC_OK;
}

}  // namespace

extern "C" {

cp_spec_status cp_spec_init(const cp_spec_model* model, const cp_spec_weights* weights, const cp_spec_config* config,
                            void* d_workspace, size_t workspace_bytes, cp_spec_ctx** out) {
  return init_impl(model, weights, config, nullptr, d_workspace, workspace_bytes, out);
}

size_t cp_spec_workspace_bytes_tree(const cp_spec_model* model, const cp_spec_config* config, const cp_spec_tree* tree) {
  if (validate(model, config, nullptr) != CP_SPEC_OK) return 0;
  cpk::TreeTab tab;
  if (build_tree(model, config, tree, &tab) != CP_SPEC_OK) return 0;
  return layout_for(model, config, tab.dmax + 1, &tab).total;
}

cp_spec_status cp_spec_init_tree(const cp_spec_model* model, const cp_spec_weights* weights,
                                 const cp_spec_config* config, const cp_spec_tree* tree, void* d_workspace,
                                 size_t workspace_bytes, cp_spec_ctx** out) {
  if (!tree) return fail(nullptr, CP_SPEC_E_INVALID, "tree is null");
  return init_impl(model, weights, config, tree, d_workspace, workspace_bytes, out);
}

cp_spec_status cp_spec_set_stream_sampling(cp_spec_ctx* c, int32_t n, const int32_t* h_top_k, const float* h_temp) {
  if (!c) return fail(nullptr, CP_SPEC_E_INVALID, "null context");
  if (n < 1 || n > c->config.max_streams || !h_top_k || !h_temp)
    return fail(c, CP_SPEC_E_INVALID, "n must be in [1, max_streams] with non-null arrays");
  for (int i = 0; i < n; ++i) {
    if (h_top_k[i] < 1 || h_top_k[i] > c->config.top_k)
      return fail(c, CP_SPEC_E_INVALID, "stream %d: top_k out of [1, %d]", i, c->config.top_k);
    const float T = h_temp[i];
    if (!(T == 0.0f || (T >= 1e-3f && T <= 100.0f))) return fail(c, CP_SPEC_E_INVALID, "stream %d: bad temperature", i);
  }
  cudaError_t e = cudaMemcpy(c->base.top_k, h_top_k, sizeof(int) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(c->base.temp, h_temp, sizeof(float) * n, cudaMemcpyHostToDevice);
  return check_cuda(c, e, "set_stream_sampling copy");
}

cp_spec_status cp_spec_decode_frames(cp_spec_ctx* c, int32_t n_streams, int32_t n_frames, int32_t first_frame,
                                     const float* d_x, const int32_t* d_c0, int32_t* d_codes, void* stream) {
  if (!c) return fail(nullptr, CP_SPEC_E_INVALID, "null context");
  if (n_streams < 1 || n_streams > c->config.max_streams) return fail(c, CP_SPEC_E_INVALID, "n_streams out of [1, max_streams]");
  if (n_frames < 0 || first_frame < 0) return fail(c, CP_SPEC_E_INVALID, "negative n_frames or first_frame");
  if (n_frames == 0) return CP_SPEC_OK;
  if (!d_x || !d_c0 || !d_codes || !aligned16(d_x) || !aligned16(d_c0) || !aligned16(d_codes))
    return fail(c, CP_SPEC_E_INVALID, "x/c0/codes null or not 16-byte aligned");
  cpk::CallArgs ca{};
  ca.mode = cpk::kModeDecode;
  ca.B = n_streams; ca.n_frames = n_frames; ca.first_frame = first_frame;
  ca.max_passes = 0;
  ca.x = d_x; ca.c0 = d_c0; ca.codes_out = d_codes; ca.committed_out = nullptr;
  c->staged = false;
  return run_call(c, ca, static_cast<cudaStream_t>(stream));
}

cp_spec_status cp_spec_begin_frame(cp_spec_ctx* c, int32_t n_streams, const float* d_x, const int32_t* d_c0,
                                   int32_t frame_idx, void* stream) {
  (void)stream;
  if (!c) return fail(nullptr, CP_SPEC_E_INVALID, "null context");
  if (n_streams < 1 || n_streams > c->config.max_streams) return fail(c, CP_SPEC_E_INVALID, "n_streams out of [1, max_streams]");
  if (frame_idx < 0) return fail(c, CP_SPEC_E_INVALID, "negative frame index");
  if (!d_x || !d_c0 || !aligned16(d_x) || !aligned16(d_c0)) return fail(c, CP_SPEC_E_INVALID, "x/c0 null or misaligned");
  c->staged = true;
  c->need_setup = true;
  c->staged_B = n_streams;
  c->staged_frame = frame_idx;
  c->staged_x = d_x;
  c->staged_c0 = d_c0;
  return CP_SPEC_OK;
}

cp_spec_status cp_spec_round(cp_spec_ctx* c, int32_t* d_codes, int32_t* d_committed, void* stream) {
  if (!c) return fail(nullptr, CP_SPEC_E_INVALID, "null context");
  if (!c->staged) return fail(c, CP_SPEC_E_STATE, "cp_spec_round before cp_spec_begin_frame");
  if (!d_codes || !aligned16(d_codes) || (d_committed && !aligned16(d_committed)))
    return fail(c, CP_SPEC_E_INVALID, "codes null or misaligned");
  cpk::CallArgs ca{};
  ca.mode = cpk::kModeDecode;
  ca.B = c->staged_B; ca.n_frames = 1; ca.first_frame = c->staged_frame;
  ca.max_passes = 1;
  ca.x = c->staged_x; ca.c0 = c->staged_c0; ca.codes_out = d_codes; ca.committed_out = d_committed;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cp_spec_status v = put_call(c, c->base, ca, s);
  if (v != CP_SPEC_OK) return v;
  cudaError_t e = cudaSuccess;
  if (c->need_setup) {
    e = cpk_host::enqueue_setup(c->base, c->accept_warps, s);
    if (e != cudaSuccess) return check_cuda(c, e, "setup launch");
    c->launches += 1;
    c->need_setup = false;
  }
  e = cpk_host::enqueue_pass(c->base, c->sms, c->accept_warps, s);
  if (e != cudaSuccess) return check_cuda(c, e, "pass launch");
  c->launches += c->base.kernels_per_pass;
  return CP_SPEC_OK;
}

cp_spec_status cp_spec_teacher_logits(cp_spec_ctx* c, int32_t n_streams, int32_t P_, const float* d_x,
                                      const int32_t* d_codes, float* d_logits, float* d_draft_logits, void* stream) {
  if (!c) return fail(nullptr, CP_SPEC_E_INVALID, "null context");
  if (n_streams < 1 || n_streams > c->config.max_streams) return fail(c, CP_SPEC_E_INVALID, "n_streams out of [1, max_streams]");
  if (P_ < 2 || P_ > c->model.num_code_groups) return fail(c, CP_SPEC_E_INVALID, "P must be in [2, num_code_groups]");
  if (!d_x || !d_codes || !d_logits || !aligned16(d_x) || !aligned16(d_codes) || !aligned16(d_logits))
    return fail(c, CP_SPEC_E_INVALID, "x/codes/logits null or misaligned");
  if (d_draft_logits && (c->N < 2 || !aligned16(d_draft_logits)))
    return fail(c, CP_SPEC_E_INVALID, "draft logits need a speculative window and 16-byte alignment");
  cpk::CallArgs ca{};
  ca.mode = cpk::kModeTeacher;
  ca.B = n_streams; ca.n_frames = 1; ca.first_frame = 0;
  ca.max_passes = 0;
  ca.x = d_x; ca.c0 = nullptr; ca.codes_out = nullptr; ca.committed_out = nullptr;
  ca.P = P_; ca.t_codes = d_codes; ca.t_logits = d_logits; ca.t_draft = d_draft_logits;
  c->staged = false;
  return run_call(c, ca, static_cast<cudaStream_t>(stream));
}

cp_spec_status cp_spec_accept_batch(int32_t R, int32_t N, int32_t V, int32_t top_k, float temperature, uint64_t seed,
                                    int32_t mode, const float* d_target, const float* d_draft, int32_t* d_tokens,
                                    int32_t* d_n_accepted, int32_t* d_drafts, void* stream) {
  if (R < 0) return fail(nullptr, CP_SPEC_E_INVALID, "R must be >= 0");
  if (N < 2 || N > CP_SPEC_MAX_WINDOW) return fail(nullptr, CP_SPEC_E_INVALID, "N must be in [2, 8]");
  if (V < 2 || V > CP_SPEC_MAX_VOCAB) return fail(nullptr, CP_SPEC_E_UNSUPPORTED, "V must be in [2, %d]", CP_SPEC_MAX_VOCAB);
  if (mode != 0 && mode != 1) return fail(nullptr, CP_SPEC_E_INVALID, "mode must be 0 (logits) or 1 (probabilities)");
  if (mode == 0) {
    if (top_k < 1 || top_k > V) return fail(nullptr, CP_SPEC_E_INVALID, "top_k must be in [1, V]");
    if (!(temperature == 0.0f || (temperature >= 1e-3f && temperature <= 100.0f)))
      return fail(nullptr, CP_SPEC_E_INVALID, "temperature must be 0 or in [1e-3, 100]");
  } else {
    top_k = 1;  // lists unused in probability mode
    temperature = 1.0f;
  }
  if (R == 0) return CP_SPEC_OK;
  if (!d_target || !d_draft || !d_tokens || !d_n_accepted || !aligned16(d_target) || !aligned16(d_draft) ||
      !aligned16(d_tokens) || !aligned16(d_n_accepted) || (d_drafts && !aligned16(d_drafts)))
    return fail(nullptr, CP_SPEC_E_INVALID, "null or misaligned pointer");
  cudaError_t e = cpk_host::launch_accept_batch(R, N, V, top_k, temperature, seed, mode, d_target, d_draft, d_tokens,
                                                d_n_accepted, d_drafts, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return check_cuda(nullptr, e, "accept kernel launch");
  g_free_launches.fetch_add(1);
  return CP_SPEC_OK;
}

cp_spec_status cp_spec_decode_frames_static(const cp_spec_model* model, const cp_spec_weights* weights,
                                            const cp_spec_config* config, int32_t n_streams, int32_t n_frames,
                                            int32_t first_frame, const float* d_x, const int32_t* d_c0,
                                            int32_t* d_codes, int32_t* d_status, void* stream) {
  cp_spec_status v = validate(model, config, nullptr);
  if (v != CP_SPEC_OK) return v;
  v = check_weights(model, config, weights);
  if (v != CP_SPEC_OK) return v;
  if (n_streams < 1 || n_streams > config->max_streams)
    return fail(nullptr, CP_SPEC_E_INVALID, "n_streams out of [1, max_streams]");
  if (n_frames < 0 || first_frame < 0) return fail(nullptr, CP_SPEC_E_INVALID, "negative n_frames or first_frame");
  const int N = effective_window(model, config);
  const cpk::Layout lay = layout_for(model, config, N);
  if (lay.total > (size_t)CP_SPEC_STATIC_SCRATCH_BYTES)
    return fail(nullptr, CP_SPEC_E_WORKSPACE, "needs %zu bytes of scratch, above the static maximum %zu (lower max_streams)",
                lay.total, (size_t)CP_SPEC_STATIC_SCRATCH_BYTES);
  if (n_frames == 0) return CP_SPEC_OK;
  if (!d_x || !d_c0 || !d_codes || !aligned16(d_x) || !aligned16(d_c0) || !aligned16(d_codes) ||
      (d_status && ((uintptr_t)d_status & 3u) != 0))
    return fail(nullptr, CP_SPEC_E_INVALID, "x/c0/codes null or not 16-byte aligned, or d_status not 4-byte aligned");
  DevicePlan dp;
  v = plan_device(model, config, N, &dp);
  if (v != CP_SPEC_OK) return v;
  unsigned char* ws = nullptr;
  v = static_scratch(dp.dev, &ws);
  if (v != CP_SPEC_OK) return v;

  cpk::FrameParams P;
  fill_params(model, weights, config, N, dp, lay, ws, &P);
  std::vector<CUtensorMap> maps;
  if (P.t5 && !build_tmaps(P, &maps)) P.t5 = 0;
  cpk::CallArgs ca{};
  ca.mode = cpk::kModeDecode;
  ca.B = n_streams; ca.n_frames = n_frames; ca.first_frame = first_frame;
  ca.max_passes = 0;
  ca.x = d_x; ca.c0 = d_c0; ca.codes_out = d_codes; ca.committed_out = nullptr;

  // Same starting state as a fresh cp_spec_init, enqueued on the caller's stream.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, lay.total, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(P.row_pos, 0xFF, sizeof(int) * (size_t)config->max_streams * P.NS, s);
  // the maps are staged from pageable host memory: the copy has read them when it returns
  if (e == cudaSuccess && P.t5)
    e = cudaMemcpyAsync((void*)P.tmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cpk_host::launch_init_tables(P.rope, P.G, P.d, (double)model->rope_theta, P.top_k, P.temp, config->max_streams,
                                     config->top_k, config->temperature, s);
  if (e == cudaSuccess && P.KO > 0) e = cpk_host::launch_offset_table(P, s);
  if (e != cudaSuccess) return check_cuda(nullptr, e, "static scratch initialisation");
  v = put_call(nullptr, P, ca, s);
  if (v != CP_SPEC_OK) return v;
  cudaGraphExec_t g = nullptr;
  v = static_graph(dp, P, &g);
  if (v != CP_SPEC_OK) return v;
  e = cudaGraphLaunch(g, s);
  if (e != cudaSuccess) return check_cuda(nullptr, e, "graph launch");
  if (d_status) {
    e = cudaMemcpyAsync(d_status, &P.ctl->status, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return check_cuda(nullptr, e, "status copy");
  }
  g_free_launches.fetch_add(P.KO > 0 ? 4 : 3);
  if (N != window_of(config)) {
    fail(nullptr, CP_SPEC_W_AR_FALLBACK,
         "speculation disabled: fewer than 3 code groups leave no draft slot; running the autoregressive loop");
    return CP_SPEC_W_AR_FALLBACK;
  }
  return CP_SPEC_OK;
}

cp_spec_status cp_spec_status_word(cp_spec_ctx* c, void* stream) {
  if (!c) return fail(nullptr, CP_SPEC_E_INVALID, "null context");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return check_cuda(c, e, "stream synchronize");
  cpk::Control* ctl = c->base.ctl;
  int st = 0;
  e = cudaMemcpy(&st, &ctl->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && st != 0) e = cudaMemset(&ctl->status, 0, sizeof(int));
  if (e != cudaSuccess) return check_cuda(c, e, "status word read");
  if (st == CP_SPEC_E_DEVICE_TIMEOUT) return fail(c, CP_SPEC_E_DEVICE_TIMEOUT, "a weight tile copy did not land in time");
  if (st != 0) return fail(c, CP_SPEC_E_DEVICE, "device-side check failed (code out of range)");
  return CP_SPEC_OK;
}

cp_spec_status cp_spec_read_stats(cp_spec_ctx* c, cp_spec_stats* out, void* stream) {
  if (!c || !out) return fail(c, CP_SPEC_E_INVALID, "null argument");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return check_cuda(c, e, "stream synchronize");
  const int B = c->config.max_streams;
  cpk::StreamStats* hs = new (std::nothrow) cpk::StreamStats[B];
  if (!hs) return fail(c, CP_SPEC_E_INVALID, "host allocation failed");
  cpk::Control ctl;
  e = cudaMemcpy(hs, c->base.sstats, sizeof(cpk::StreamStats) * B, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&ctl, c->base.ctl, sizeof ctl, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) { delete[] hs; return check_cuda(c, e, "stats copy"); }
  memset(out, 0, sizeof *out);
  for (int b = 0; b < B; ++b) {
    out->frames += hs[b].frames; out->rounds += hs[b].rounds; out->committed += hs[b].committed;
    out->bonus += hs[b].bonus; out->rejections += hs[b].rejections;
    for (int t = 0; t < 9; ++t) { out->drafted_by_offset[t] += hs[b].drafted[t]; out->accepted_by_offset[t] += hs[b].accepted[t]; }
  }
  out->passes = ctl.passes;
  out->weight_bytes = ctl.weight_bytes;
  out->kv_bytes = ctl.kv_bytes;
  out->heads_applied = ctl.heads_applied;
  out->kernel_launches = ctl.kernels;
  delete[] hs;
  return CP_SPEC_OK;
}

cp_spec_status cp_spec_reset_stats(cp_spec_ctx* c, void* stream) {
  if (!c) return fail(nullptr, CP_SPEC_E_INVALID, "null context");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(c->base.sstats, 0, sizeof(cpk::StreamStats) * c->config.max_streams, s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(&c->base.ctl->weight_bytes, 0, cpk::kControlCounters * sizeof(long long), s);
  return check_cuda(c, e, "reset stats");
}

cp_spec_status cp_spec_test_hooks(cp_spec_ctx* c, uint64_t wait_limit_ns, int32_t flags) {
  if (!c) return fail(nullptr, CP_SPEC_E_INVALID, "null context");
  if (wait_limit_ns < 10000ull || wait_limit_ns > 60ull * 1000000000ull)
    return fail(c, CP_SPEC_E_INVALID, "wait_limit_ns must be in [1e4, 6e10]");
  if (flags < 0 || flags > 3) return fail(c, CP_SPEC_E_INVALID, "flags must be in [0, 3]");
  // the parameter block is part of the call graph: drop the graph (rebuilt on the next call)
  if (c->graph) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaGraphExecDestroy(c->graph);
    c->graph = nullptr;
    if (e != cudaSuccess) return check_cuda(c, e, "graph release");
  }
  c->base.wait_ns = wait_limit_ns;
  c->base.test_stall = flags & 1;
  c->base.test_poison = (flags >> 1) & 1;
  return CP_SPEC_OK;
}

int64_t cp_spec_launch_count(const cp_spec_ctx* c) {
  return c ? c->launches : g_free_launches.load();
}

const char* cp_spec_last_error(const cp_spec_ctx* c) { return c ? c->err.c_str() : g_err.c_str(); }

void cp_spec_destroy(cp_spec_ctx* c) {
  if (!c) return;
  if (c->graph) cudaGraphExecDestroy(c->graph);
  if (c->capture) cudaStreamDestroy(c->capture);
  delete c;
}

}  // extern "C"
