/*
 * cp_oracle.c -- CPU oracle for the CodePredictor speculative round.
 *
 * TEST INFRASTRUCTURE ONLY (see cp_oracle.h).  Plain loops, no blocking, no
 * fusion, no reordering beyond what each definition states, so that a reader
 * can check it against the pages by eye.  Build with -ffp-contract=off so the
 * float32 sampling arithmetic is the same on every host.
 */
#include "cp_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ Philox */
/* Philox4x32-10, from its published definition (Salmon et al., "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64
 * multiplications with the Weyl-sequence key schedule. */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { k0 += PHILOX_W0; k1 += PHILOX_W1; }
    uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)x0;
    uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)x2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t y0 = hi1 ^ x1 ^ k0;
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x3 ^ k1;
    uint32_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

float orc_uniform(uint64_t seed, uint32_t stream, uint32_t frame, uint32_t depth, uint32_t purpose) {
  uint32_t c[4] = {stream, frame, depth, purpose};
  uint32_t k[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t o[4];
  orc_philox4x32_10(c, k, o);
  return (float)(o[0] >> 8) * (1.0f / 16777216.0f);
}

void orc_uniform_fill(uint64_t seed, int n, const uint32_t* ctr4, float* out) {
  for (int i = 0; i < n; ++i)
    out[i] = orc_uniform(seed, ctr4[4 * i], ctr4[4 * i + 1], ctr4[4 * i + 2], ctr4[4 * i + 3]);
}

/* ------------------------------------------------------- logit processing */
typedef struct { float z; int idx; } zi_t;

static int cmp_desc(const void* a, const void* b) {
  const zi_t* x = (const zi_t*)a;
  const zi_t* y = (const zi_t*)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

/* Top-k / temperature processing ("Speculative Decoding, Beyond Text",
 * section 02: q_i and p_i are the draft and target laws after temperature,
 * top-k and the other processors; only temperature and top-k are used here).
 * z_i = fl32(logit_i / T); keep exactly min(k, V) entries ordered by
 * (z desc, index asc); then the softmax over the kept set in float64:
 * e_i = exp(z_i - z_max), S = sum of e_i (ascending index order),
 * p_i = e_i / S, each p_i rounded once to float32.  The pages fix no
 * precision for this step; float64 with one final rounding is the plain
 * definition.  T = 0 is argmax with the lowest index on ties.  `margin`
 * (optional) is the decision gap that a change of rounding would have to
 * cross: the logit gap at the top-k boundary (or to the runner-up for
 * greedy). */
void orc_process(const float* logits, int V, int top_k, float T, float* probs, double* margin) {
  if (V <= 0) return;
  for (int i = 0; i < V; ++i) probs[i] = 0.0f;
  if (T == 0.0f) {
    int best = 0;
    for (int i = 1; i < V; ++i)
      if (logits[i] > logits[best]) best = i;
    if (margin) {
      double gap = INFINITY;
      for (int i = 0; i < V; ++i)
        if (i != best) {
          double g = (double)logits[best] - (double)logits[i];
          if (g < gap) gap = g;
        }
      *margin = gap;
    }
    probs[best] = 1.0f;
    return;
  }
  zi_t* zs = (zi_t*)malloc(sizeof(zi_t) * (size_t)V);
  unsigned char* keep = (unsigned char*)calloc((size_t)V, 1);
  for (int i = 0; i < V; ++i) {
    zs[i].z = logits[i] / T;
    zs[i].idx = i;
  }
  qsort(zs, (size_t)V, sizeof(zi_t), cmp_desc);
  int kk = top_k < V ? top_k : V;
  for (int r = 0; r < kk; ++r) keep[zs[r].idx] = 1;
  const double zmax = (double)zs[0].z;
  double S = 0.0;
  for (int i = 0; i < V; ++i)
    if (keep[i]) S += exp((double)(logits[i] / T) - zmax);
  for (int i = 0; i < V; ++i)
    if (keep[i]) probs[i] = (float)(exp((double)(logits[i] / T) - zmax) / S);
  if (margin) *margin = (kk < V) ? ((double)zs[kk - 1].z - (double)zs[kk].z) * (double)T : INFINITY;
  free(zs);
  free(keep);
}

/* ------------------------------------------------------- categorical draw */
int orc_sample(const float* w, int V, float u, double* margin) {
  float S = 0.0f;
  int last = -1;
  for (int i = 0; i < V; ++i)
    if (w[i] > 0.0f) { S = S + w[i]; last = i; }
  if (last < 0) { if (margin) *margin = 0.0; return -1; }
  float t = u * S;
  float acc = 0.0f, prev = 0.0f;
  int pick = last;
  float lo = 0.0f, hi = S;
  for (int i = 0; i < V; ++i) {
    if (!(w[i] > 0.0f)) continue;
    prev = acc;
    acc = acc + w[i];
    if (acc > t) { pick = i; lo = prev; hi = acc; break; }
  }
  if (margin) {
    double a = (double)t - (double)lo, b = (double)hi - (double)t;
    double m = a < b ? a : b;
    *margin = (S > 0.0f) ? m / (double)S : 0.0;
  }
  return pick;
}

/* ------------------------------------------------------------- acceptance */
/* "How a round works", step 3 (CodePredictor Speculative Decoding) and
 * "Exact stochastic decoding" (Speculative Decoding, Beyond Text, 02). */
int orc_accept_chain(int V, int n_d, int m, const float* q, const int* drafts, const float* p,
                     const float* u_acc, const float* u_tgt, int* emitted, int* n_emitted,
                     double* margin) {
  double mg = INFINITY, m2;
  if (n_d < 0 || m < n_d || m > n_d + 1 || V <= 0) return -1; /* p must score every draft */
  float* res = (float*)malloc(sizeof(float) * (size_t)V);
  int n_acc = n_d;
  int done = 0;
  for (int t = 1; t <= n_d && !done; ++t) {
    const float* qt = q + (size_t)(t - 1) * V;
    const float* pt = p + (size_t)(t - 1) * V;
    int y = drafts[t - 1];
    float ratio = pt[y] / qt[y];
    double gap = fabs((double)u_acc[t - 1] - (double)ratio);
    if (gap < mg) mg = gap;
    if (u_acc[t - 1] < ratio) {
      emitted[t - 1] = y;
      continue;
    }
    for (int i = 0; i < V; ++i) {
      float dlt = pt[i] - qt[i];
      res[i] = dlt > 0.0f ? dlt : 0.0f;
    }
    int c = orc_sample(res, V, u_tgt[t - 1], &m2);
    if (c < 0) c = orc_sample(pt, V, u_tgt[t - 1], &m2);
    if (m2 < mg) mg = m2;
    emitted[t - 1] = c;
    *n_emitted = t;
    n_acc = t - 1;
    done = 1;
  }
  if (!done) {
    if (m > n_d) {
      int c = orc_sample(p + (size_t)n_d * V, V, u_tgt[n_d], &m2);
      if (m2 < mg) mg = m2;
      emitted[n_d] = c;
      *n_emitted = n_d + 1;
    } else {
      *n_emitted = n_d;
    }
  }
  free(res);
  if (margin) *margin = mg;
  return n_acc;
}

void orc_accept_batch(int R, int N, int V, int top_k, float T, uint64_t seed, int mode,
                      const float* target, const float* draft, int* tokens, int* n_acc,
                      int* drafts_out, double* margins) {
  int nd = N - 1;
  float* q = (float*)malloc(sizeof(float) * (size_t)(nd > 0 ? nd : 1) * V);
  float* p = (float*)malloc(sizeof(float) * (size_t)N * V);
  int dr[8], em[9];
  float ua[8], ut[9];
  for (int r = 0; r < R; ++r) {
    double mg = INFINITY, m1;
    for (int t = 1; t <= nd; ++t) {
      const float* src = draft + ((size_t)r * nd + (t - 1)) * V;
      if (mode == 0) {
        orc_process(src, V, top_k, T, q + (size_t)(t - 1) * V, &m1);
        if (m1 < mg) mg = m1;
      } else {
        memcpy(q + (size_t)(t - 1) * V, src, sizeof(float) * (size_t)V);
      }
      dr[t - 1] = orc_sample(q + (size_t)(t - 1) * V, V, orc_uniform(seed, (uint32_t)r, 0, (uint32_t)t, ORC_DRAFT), &m1);
      if (m1 < mg) mg = m1;
      ua[t - 1] = orc_uniform(seed, (uint32_t)r, 0, (uint32_t)t, ORC_ACCEPT);
    }
    for (int t = 1; t <= N; ++t) {
      const float* src = target + ((size_t)r * N + (t - 1)) * V;
      if (mode == 0) {
        orc_process(src, V, top_k, T, p + (size_t)(t - 1) * V, &m1);
        if (m1 < mg) mg = m1;
      } else {
        memcpy(p + (size_t)(t - 1) * V, src, sizeof(float) * (size_t)V);
      }
      ut[t - 1] = orc_uniform(seed, (uint32_t)r, 0, (uint32_t)t, ORC_TARGET);
    }
    int ne = 0;
    int na = orc_accept_chain(V, nd, N, q, dr, p, ua, ut, em, &ne, &m1);
    if (m1 < mg) mg = m1;
    for (int t = 0; t < N; ++t) tokens[(size_t)r * N + t] = t < ne ? em[t] : -1;
    n_acc[r] = na;
    if (drafts_out)
      for (int t = 0; t < nd; ++t) drafts_out[(size_t)r * nd + t] = dr[t];
    if (margins) margins[r] = mg;
  }
  free(q);
  free(p);
}

/* ---------------------------------------------------------------- forward */
size_t orc_kv_doubles(const orc_model* M) {
  return (size_t)M->L * 2 * M->G * M->nkv * M->d;
}

static double* kv_at(const orc_model* M, double* kv, int layer, int which, int pos, int kvh) {
  return kv + ((((size_t)layer * 2 + which) * M->G + pos) * M->nkv + kvh) * M->d;
}

/* RMSNorm: h / sqrt(mean(h^2) + eps) * gain. */
static void rmsnorm(const double* h, const float* g, int H, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < H; ++i) ss += h[i] * h[i];
  double inv = 1.0 / sqrt(ss / (double)H + eps);
  for (int i = 0; i < H; ++i) out[i] = h[i] * inv * (double)g[i];
}

/* y = W x, W [rows][cols] float32 row-major. */
static void matvec(const float* W, int rows, int cols, const double* x, double* y) {
  for (int r = 0; r < rows; ++r) {
    double acc = 0.0;
    const float* w = W + (size_t)r * cols;
    for (int c = 0; c < cols; ++c) acc += (double)w[c] * x[c];
    y[r] = acc;
  }
}

/* Rotary embedding, rotate-half pairing (i, i + d/2), frequency theta^(-2i/d). */
static void rope(double* v, int d, int pos, double theta) {
  int h = d / 2;
  for (int i = 0; i < h; ++i) {
    double freq = pow(theta, -2.0 * (double)i / (double)d);
    double ang = (double)pos * freq;
    double c = cos(ang), s = sin(ang);
    double x1 = v[i], x2 = v[i + h];
    v[i] = x1 * c - x2 * s;
    v[i + h] = x2 * c + x1 * s;
  }
}

static double silu(double x) { return x / (1.0 + exp(-x)); }

void orc_forward(const orc_model* M, double* kv, int n, const double* in_rows, const int* positions,
                 double* out_normed) {
  const int H = M->H, d = M->d, nq = M->nq, nkv = M->nkv, F = M->F;
  const int qd = nq * d, kvd = nkv * d, grp = nq / nkv;
  double* h = (double*)malloc(sizeof(double) * (size_t)n * H);
  double* a = (double*)malloc(sizeof(double) * (size_t)H);
  double* q = (double*)malloc(sizeof(double) * (size_t)n * qd);
  double* k = (double*)malloc(sizeof(double) * (size_t)kvd);
  double* v = (double*)malloc(sizeof(double) * (size_t)kvd);
  double* o = (double*)malloc(sizeof(double) * (size_t)n * qd);
  double* t = (double*)malloc(sizeof(double) * (size_t)H);
  double* g = (double*)malloc(sizeof(double) * (size_t)F);
  double* u = (double*)malloc(sizeof(double) * (size_t)F);
  double* sc = (double*)malloc(sizeof(double) * (size_t)M->G);
  memcpy(h, in_rows, sizeof(double) * (size_t)n * H);
  const double scale = 1.0 / sqrt((double)d);

  for (int l = 0; l < M->L; ++l) {
    const float* wq = M->wq + (size_t)l * qd * H;
    const float* wk = M->wk + (size_t)l * kvd * H;
    const float* wv = M->wv + (size_t)l * kvd * H;
    const float* wo = M->wo + (size_t)l * H * qd;
    const float* wg = M->w_gate + (size_t)l * F * H;
    const float* wu = M->w_up + (size_t)l * F * H;
    const float* wd = M->w_down + (size_t)l * H * F;
    /* attention block: norm, projections, rotary, append to the cache */
    for (int r = 0; r < n; ++r) {
      rmsnorm(h + (size_t)r * H, M->attn_norm + (size_t)l * H, H, M->eps, a);
      matvec(wq, qd, H, a, q + (size_t)r * qd);
      matvec(wk, kvd, H, a, k);
      matvec(wv, kvd, H, a, v);
      for (int hq = 0; hq < nq; ++hq) rope(q + (size_t)r * qd + (size_t)hq * d, d, positions[r], M->theta);
      for (int hk = 0; hk < nkv; ++hk) {
        rope(k + (size_t)hk * d, d, positions[r], M->theta);
        memcpy(kv_at(M, kv, l, 0, positions[r], hk), k + (size_t)hk * d, sizeof(double) * (size_t)d);
        memcpy(kv_at(M, kv, l, 1, positions[r], hk), v + (size_t)hk * d, sizeof(double) * (size_t)d);
      }
    }
    /* causal attention: row at position p reads cache positions 0..p */
    for (int r = 0; r < n; ++r) {
      int pos = positions[r];
      for (int hq = 0; hq < nq; ++hq) {
        int hk = hq / grp;
        const double* qv = q + (size_t)r * qd + (size_t)hq * d;
        double mx = -INFINITY;
        for (int j = 0; j <= pos; ++j) {
          const double* kj = kv_at(M, kv, l, 0, j, hk);
          double s = 0.0;
          for (int e = 0; e < d; ++e) s += qv[e] * kj[e];
          sc[j] = s * scale;
          if (sc[j] > mx) mx = sc[j];
        }
        double den = 0.0;
        for (int j = 0; j <= pos; ++j) { sc[j] = exp(sc[j] - mx); den += sc[j]; }
        double* ov = o + (size_t)r * qd + (size_t)hq * d;
        for (int e = 0; e < d; ++e) ov[e] = 0.0;
        for (int j = 0; j <= pos; ++j) {
          const double* vj = kv_at(M, kv, l, 1, j, hk);
          double w = sc[j] / den;
          for (int e = 0; e < d; ++e) ov[e] += w * vj[e];
        }
      }
    }
    for (int r = 0; r < n; ++r) {
      matvec(wo, H, qd, o + (size_t)r * qd, t);
      for (int i = 0; i < H; ++i) h[(size_t)r * H + i] += t[i];
    }
    /* SwiGLU feed-forward block */
    for (int r = 0; r < n; ++r) {
      rmsnorm(h + (size_t)r * H, M->ffn_norm + (size_t)l * H, H, M->eps, a);
      matvec(wg, F, H, a, g);
      matvec(wu, F, H, a, u);
      for (int i = 0; i < F; ++i) g[i] = silu(g[i]) * u[i];
      matvec(wd, H, F, g, t);
      for (int i = 0; i < H; ++i) h[(size_t)r * H + i] += t[i];
    }
  }
  for (int r = 0; r < n; ++r) rmsnorm(h + (size_t)r * H, M->final_norm, H, M->eps, out_normed + (size_t)r * H);
  free(h); free(a); free(q); free(k); free(v); free(o); free(t); free(g); free(u); free(sc);
}

void orc_head_logits(const orc_model* M, int j, const double* hn, double* out64, float* out32) {
  const float* W = M->head + (size_t)(j - 1) * M->V * M->H;
  for (int v = 0; v < M->V; ++v) {
    double acc = 0.0;
    const float* w = W + (size_t)v * M->H;
    for (int c = 0; c < M->H; ++c) acc += (double)w[c] * hn[c];
    if (out64) out64[v] = acc;
    if (out32) out32[v] = (float)acc;
  }
}

/* "RVQ Position Aware Speculative Decoding for On Device TTS", section 2.2:
 * the drafter adds the offset of its lookahead distance to the hidden state
 * the heads read (the final-normed output), then applies the later head. */
void orc_draft_logits(const orc_model* M, int j, int t, const double* hn, float* out32) {
  if (t > M->K || !M->draft_offset) {
    orc_head_logits(M, j, hn, NULL, out32);
    return;
  }
  double* shifted = (double*)malloc(sizeof(double) * (size_t)M->H);
  const float* b = M->draft_offset + (size_t)(t - 1) * M->H;
  for (int i = 0; i < M->H; ++i) shifted[i] = hn[i] + (double)b[i];
  orc_head_logits(M, j, shifted, NULL, out32);
  free(shifted);
}

/* Input row of position pos: x at position 0, E_{pos-1}(code) otherwise. */
static void input_row(const orc_model* M, const float* x, int pos, int code, double* row) {
  if (pos == 0) {
    for (int i = 0; i < M->H; ++i) row[i] = (double)x[i];
  } else {
    const float* e = M->embed + ((size_t)(pos - 1) * M->V + code) * M->H;
    for (int i = 0; i < M->H; ++i) row[i] = (double)e[i];
  }
}

void orc_teacher_logits(const orc_model* M, const float* x, const int* codes, int P, int n_draft,
                        float* logits, float* draft) {
  const int H = M->H, V = M->V;
  double* kv = (double*)calloc(orc_kv_doubles(M), sizeof(double));
  double* rows = (double*)malloc(sizeof(double) * (size_t)P * H);
  double* hn = (double*)malloc(sizeof(double) * (size_t)P * H);
  int* pos = (int*)malloc(sizeof(int) * (size_t)P);
  for (int j = 0; j < P; ++j) {
    pos[j] = j;
    input_row(M, x, j, j > 0 ? codes[j - 1] : 0, rows + (size_t)j * H);
  }
  orc_forward(M, kv, P, rows, pos, hn);
  for (int j = 1; j < P; ++j) {
    orc_head_logits(M, j, hn + (size_t)j * H, NULL, logits + (size_t)(j - 1) * V);
    if (draft) {
      for (int t = 1; t <= n_draft; ++t) {
        float* dst = draft + ((size_t)(j - 1) * n_draft + (t - 1)) * V;
        if (j + t <= M->G - 1) orc_draft_logits(M, j + t, t, hn + (size_t)j * H, dst);
        else for (int v = 0; v < V; ++v) dst[v] = 0.0f;
      }
    }
  }
  free(kv); free(rows); free(hn); free(pos);
}

/* ------------------------------------------------------------ frame loop */
static void log_round(orc_round_rec* log, int log_cap, int* n_log, int frame, int stream, int s,
                      int n_d, int m, int n_acc, int s_new, const int* drafts, double mg) {
  if (!log || !n_log || *n_log >= log_cap) { if (n_log) ++*n_log; return; }
  orc_round_rec* r = &log[*n_log];
  memset(r, 0, sizeof(*r));
  r->frame = frame; r->stream = stream; r->s = s; r->n_d = n_d; r->m = m;
  r->n_acc = n_acc; r->s_new = s_new; r->min_margin = mg;
  for (int t = 0; t < n_d && t < 8; ++t) r->drafts[t] = drafts[t];
  ++*n_log;
}

/* One frame of one stream.  Sequence layout: position 0 holds the talker
 * hidden x, position j >= 1 holds E_{j-1}(c_{j-1}); the output at position
 * j is h_j and p_j = proc(head_j . h_j) is the law of c_j. */
static void decode_one_frame(const orc_model* M, int N, int w, int top_k, float T, uint64_t seed, int stream,
                             int frame, const float* x, int c0, int* codes, orc_stats* st,
                             orc_round_rec* log, int log_cap, int* n_log, int64_t* reach, int64_t* acc) {
  const int H = M->H, V = M->V, G = M->G;
  double* kv = (double*)calloc(orc_kv_doubles(M), sizeof(double));
  double* rows = (double*)malloc(sizeof(double) * 9 * H);
  double* hn = (double*)malloc(sizeof(double) * 9 * H);
  double* hs = (double*)malloc(sizeof(double) * H);
  float* lg = (float*)malloc(sizeof(float) * V);
  float* q = (float*)malloc(sizeof(float) * 8 * V);
  float* p = (float*)malloc(sizeof(float) * 9 * V);
  int pos[9], dr[8], em[9];
  float ua[8], ut[9];
  double mg, m1;

  codes[0] = c0;
  /* Frame prefill: rows [x, E_0(c_0)] at positions 0, 1; c_1 ~ p_1. */
  input_row(M, x, 0, 0, rows);
  input_row(M, x, 1, c0, rows + H);
  pos[0] = 0; pos[1] = 1;
  orc_forward(M, kv, 2, rows, pos, hn);
  int committed_len = 2; /* KV positions 0..1 are final */
  st->passes++;
  orc_head_logits(M, 1, hn + H, NULL, lg);
  orc_process(lg, V, top_k, T, p, &mg);
  codes[1] = orc_sample(p, V, orc_uniform(seed, (uint32_t)stream, (uint32_t)frame, 1, ORC_TARGET), &m1);
  if (m1 < mg) mg = m1;
  log_round(log, log_cap, n_log, frame, stream, 0, 0, 1, 0, 1, dr, mg);
  int s = 1;
  memcpy(hs, hn + H, sizeof(double) * H);

  if (N == 0) {
    /* Autoregressive baseline: one single-row pass per code. */
    for (int j = 2; j <= G - 1; ++j) {
      input_row(M, x, j, codes[j - 1], rows);
      pos[0] = j;
      orc_forward(M, kv, 1, rows, pos, hn);
      committed_len = j + 1;
      st->passes++;
      orc_head_logits(M, j, hn, NULL, lg);
      orc_process(lg, V, top_k, T, p, &mg);
      codes[j] = orc_sample(p, V, orc_uniform(seed, (uint32_t)stream, (uint32_t)frame, (uint32_t)j, ORC_TARGET), &m1);
      if (m1 < mg) mg = m1;
      log_round(log, log_cap, n_log, frame, stream, j - 1, 0, 1, 0, j, dr, mg);
    }
  } else {
    while (s < G - 1) {
      const int R = G - 1 - s;
      const int n_d = (w - 1) < R ? (w - 1) : R; /* the frame's window w <= N */
      mg = INFINITY;
      /* Draft: head_{s+t} applied to the current hidden h_s (plus the
       * offset b_t where one is given). */
      for (int t = 1; t <= n_d; ++t) {
        orc_draft_logits(M, s + t, t, hs, lg);
        orc_process(lg, V, top_k, T, q + (size_t)(t - 1) * V, &m1);
        if (m1 < mg) mg = m1;
        dr[t - 1] = orc_sample(q + (size_t)(t - 1) * V, V,
                               orc_uniform(seed, (uint32_t)stream, (uint32_t)frame, (uint32_t)(s + t), ORC_DRAFT), &m1);
        if (m1 < mg) mg = m1;
        st->drafted_by_offset[t]++;
      }
      /* Verify: one causal pass over the committed code and the drafts. */
      const int m = (n_d + 1) < R ? (n_d + 1) : R;
      if (committed_len != s + 1) { /* transaction invariant: L = s + 1 */
        break;
      }
      for (int i = 0; i < m; ++i) {
        int code = (i == 0) ? codes[s] : dr[i - 1];
        pos[i] = s + 1 + i;
        input_row(M, x, s + 1 + i, code, rows + (size_t)i * H);
      }
      orc_forward(M, kv, m, rows, pos, hn);
      st->passes++;
      for (int i = 0; i < m; ++i) {
        orc_head_logits(M, s + 1 + i, hn + (size_t)i * H, NULL, lg);
        orc_process(lg, V, top_k, T, p + (size_t)i * V, &m1);
        if (m1 < mg) mg = m1;
      }
      /* Accept left to right. */
      for (int t = 1; t <= n_d; ++t) {
        ua[t - 1] = orc_uniform(seed, (uint32_t)stream, (uint32_t)frame, (uint32_t)(s + t), ORC_ACCEPT);
        ut[t - 1] = orc_uniform(seed, (uint32_t)stream, (uint32_t)frame, (uint32_t)(s + t), ORC_TARGET);
      }
      ut[n_d] = orc_uniform(seed, (uint32_t)stream, (uint32_t)frame, (uint32_t)(s + n_d + 1), ORC_TARGET);
      int ne = 0;
      int na = orc_accept_chain(V, n_d, m, q, dr, p, ua, ut, em, &ne, &m1);
      if (m1 < mg) mg = m1;
      for (int t = 1; t <= na; ++t) st->accepted_by_offset[t]++;
      /* the window policy's counters: drafts the left-to-right test reached
       * (up to and including the first rejection) and accepted, by offset */
      for (int t = 1; t <= n_d && t <= na + 1; ++t) reach[t]++;
      for (int t = 1; t <= na; ++t) acc[t]++;
      if (ne > na && na < n_d) st->rejections++;
      if (ne > n_d) st->bonus++;
      for (int i = 0; i < ne; ++i) codes[s + 1 + i] = em[i];
      const int s_new = s + ne;
      /* Reconcile: keep KV positions 0..s_new, i.e. L' = s_new + 1.  Stale
       * entries above are overwritten before any later row can read them. */
      committed_len = s_new + 1;
      memcpy(hs, hn + (size_t)(s_new - s - 1) * H, sizeof(double) * H);
      st->rounds++;
      log_round(log, log_cap, n_log, frame, stream, s, n_d, m, na, s_new, dr, mg);
      s = s_new;
    }
  }
  st->committed += G - 1;
  st->frames++;
  free(kv); free(rows); free(hn); free(hs); free(lg); free(q); free(p);
}

/* Window of a stream's next frame under the acceptance policy: offsets
 * t = 1, 2, ... are kept while each either has fewer than min_reached
 * reached drafts or accepted at least pct percent of them (integer test
 * 100 * acc >= pct * reach); the window is 1 + the kept leading offsets, at
 * most N.  Window 1 runs the frame's rounds without drafts (one row per
 * pass, each code drawn from the target as in the AR loop). */
int orc_policy_window(int N, int pct, int min_reached, const int64_t* reach, const int64_t* acc) {
  if (N < 2 || pct <= 0) return N;
  int w = 1;
  for (int t = 1; t <= N - 1; ++t) {
    const int keep = reach[t] < min_reached || 100 * acc[t] >= (int64_t)pct * reach[t];
    if (!keep) break;
    w = t + 1;
  }
  return w;
}

int orc_decode_frames_policy(const orc_model* M, int N, const int* top_k, const float* temp, uint64_t seed,
                             int B, int F, int first_frame, const float* x, const int* c0, int* codes,
                             orc_stats* st, orc_round_rec* log, int log_cap, int* n_log, int pct,
                             int min_reached) {
  if (!M || !codes || !x || !c0 || !st) return -1;
  if (!(N == 0 || (N >= 2 && N <= 8))) return -1;
  if (M->G < 2 || M->nq % M->nkv != 0 || M->d % 2 != 0) return -1;
  if (M->K < 0 || (M->K > 0 && !M->draft_offset)) return -1;
  if (pct < 0 || pct > 100 || (pct > 0 && min_reached < 1)) return -1;
  if (n_log) *n_log = 0;
  /* per-stream policy counters, from the start of the call */
  int64_t* reach = (int64_t*)calloc((size_t)(B > 0 ? B : 1) * 9, sizeof(int64_t));
  int64_t* acc = (int64_t*)calloc((size_t)(B > 0 ? B : 1) * 9, sizeof(int64_t));
  for (int f = 0; f < F; ++f)
    for (int b = 0; b < B; ++b) {
      const int w = orc_policy_window(N, pct, min_reached, reach + (size_t)b * 9, acc + (size_t)b * 9);
      decode_one_frame(M, N, w, top_k[b], temp[b], seed, b, first_frame + f,
                       x + ((size_t)f * B + b) * M->H, c0[(size_t)f * B + b],
                       codes + ((size_t)f * B + b) * M->G, st, log, log_cap, n_log,
                       reach + (size_t)b * 9, acc + (size_t)b * 9);
    }
  free(reach);
  free(acc);
  return 0;
}

int orc_decode_frames(const orc_model* M, int N, const int* top_k, const float* temp, uint64_t seed,
                      int B, int F, int first_frame, const float* x, const int* c0, int* codes,
                      orc_stats* st, orc_round_rec* log, int log_cap, int* n_log) {
  return orc_decode_frames_policy(M, N, top_k, temp, seed, B, F, first_frame, x, c0, codes, st, log, log_cap,
                                  n_log, 0, 1);
}

/* ------------------------------------------------------------ sparse tree */
/* Tree rounds ("RVQ Position Aware Speculative Decoding for On Device TTS",
 * section 2.2, tree attention and sparse tree attention, Figure 2).  The
 * drafts of depth t all come from head_{s+t} on h_s (+ b_t), so a node is
 * named by its depth and the rank of its token among that depth's draft
 * logits (value descending, index ascending); the tree is a set of such rank
 * paths, given parents first.  Every node is verified in one pass attending
 * to the committed prefix and its own ancestors; here each node's output is
 * computed by a plain causal pass over the prefix cache plus its path, which
 * is that definition written out.  Acceptance walks down from the committed
 * code: at a node with target law p, the children are tested in rank order
 * as drafts with point-mass draft laws (accept child c iff u < p'(c), p' the
 * residual renormalised over what is left, else remove c), and when none is
 * accepted, or the node has no child, one code is drawn from what is left
 * (a correction, or the bonus).  Each draw is then distributed as p, so the
 * committed codes keep the autoregressive law. */

static int tree_depth(const orc_tree* T, int i) {
  int d = 0;
  for (int j = i; j >= 0; j = T->parent[j]) ++d;
  return d;
}

/* Final-normed output of the last row of [c_s, path...] at positions
 * s+1..s+1+len on a copy of the prefix cache. */
static void path_output(const orc_model* M, const double* kv0, double* kvw, const float* x, int s, int c_s,
                        const int* path, int len, double* rows, double* outs, double* last) {
  const size_t nkv = orc_kv_doubles(M);
  memcpy(kvw, kv0, sizeof(double) * nkv);
  int pos[64];
  input_row(M, x, s + 1, c_s, rows);
  pos[0] = s + 1;
  for (int i = 0; i < len; ++i) {
    input_row(M, x, s + 2 + i, path[i], rows + (size_t)(i + 1) * M->H);
    pos[i + 1] = s + 2 + i;
  }
  orc_forward(M, kvw, len + 1, rows, pos, outs);
  memcpy(last, outs + (size_t)len * M->H, sizeof(double) * M->H);
}

static void decode_one_frame_tree(const orc_model* M, const orc_tree* T, int top_k, float Tmp, uint64_t seed,
                                  int stream, int frame, const float* x, int c0, int* codes, orc_stats* st,
                                  orc_round_rec* log, int log_cap, int* n_log) {
  const int H = M->H, V = M->V, G = M->G, n = T->n;
  const size_t nkv = orc_kv_doubles(M);
  double* kv = (double*)calloc(nkv, sizeof(double));
  double* kvw = (double*)malloc(sizeof(double) * nkv);
  double* rows = (double*)malloc(sizeof(double) * 64 * H);
  double* outs = (double*)malloc(sizeof(double) * 64 * H);
  double* hs = (double*)malloc(sizeof(double) * H);
  double* hn = (double*)malloc(sizeof(double) * H);
  float* lg = (float*)malloc(sizeof(float) * V);
  float* pn = (float*)malloc(sizeof(float) * (size_t)(n + 1) * V); /* law at the root (0) and node i (i + 1) */
  float* work = (float*)malloc(sizeof(float) * V);
  int* order = (int*)malloc(sizeof(int) * V);
  int* tok = (int*)malloc(sizeof(int) * (n > 0 ? n : 1));
  int* dep = (int*)malloc(sizeof(int) * (n > 0 ? n : 1));
  int* keep = (int*)malloc(sizeof(int) * (n > 0 ? n : 1));
  int pos[2], path[64], dr[8] = {0};
  double mg, m1;

  /* frame prefill, as in the chain rounds */
  codes[0] = c0;
  input_row(M, x, 0, 0, rows);
  input_row(M, x, 1, c0, rows + H);
  pos[0] = 0; pos[1] = 1;
  orc_forward(M, kv, 2, rows, pos, outs);
  st->passes++;
  orc_head_logits(M, 1, outs + H, NULL, lg);
  orc_process(lg, V, top_k, Tmp, work, &mg);
  codes[1] = orc_sample(work, V, orc_uniform(seed, (uint32_t)stream, (uint32_t)frame, 1, ORC_TARGET), &m1);
  if (m1 < mg) mg = m1;
  log_round(log, log_cap, n_log, frame, stream, 0, 0, 1, 0, 1, dr, mg);
  memcpy(hs, outs + H, sizeof(double) * H);
  int s = 1;
  while (s < G - 1) {
    const int R = G - 1 - s;
    mg = INFINITY;
    int nkeep = 0, dmax = 0;
    for (int i = 0; i < n; ++i) {
      dep[i] = tree_depth(T, i);
      keep[i] = dep[i] <= R && T->rank[i] < V && (T->parent[i] < 0 || keep[T->parent[i]]);
      if (keep[i]) { ++nkeep; if (dep[i] > dmax) dmax = dep[i]; }
    }
    /* candidate tokens: rank r of depth t's draft logits (selection by
     * value descending, index ascending) */
    for (int t = 1; t <= dmax; ++t) {
      orc_draft_logits(M, s + t, t, hs, lg);
      int need = 0;
      for (int i = 0; i < n; ++i)
        if (keep[i] && dep[i] == t && T->rank[i] + 1 > need) need = T->rank[i] + 1;
      for (int r = 0; r < need && r < V; ++r) {
        int best = -1;
        for (int v = 0; v < V; ++v) {
          int used = 0;
          for (int q = 0; q < r; ++q) used |= order[q] == v;
          if (used) continue;
          if (best < 0 || lg[v] > lg[best]) best = v;
        }
        order[r] = best;
      }
      /* near-ties between consecutive ranks may order differently in float32 */
      for (int r = 0; r + 1 < need && r + 1 < V; ++r) {
        const double g = (double)lg[order[r]] - (double)lg[order[r + 1]];
        if (g < mg) mg = g;
      }
      for (int i = 0; i < n; ++i)
        if (keep[i] && dep[i] == t) tok[i] = order[T->rank[i]];
    }
    /* verify: the law at the root (p_{s+1}) and at every kept node short of depth R */
    path_output(M, kv, kvw, x, s, codes[s], path, 0, rows, outs, hn);
    orc_head_logits(M, s + 1, hn, NULL, lg);
    orc_process(lg, V, top_k, Tmp, pn, &m1);
    if (m1 < mg) mg = m1;
    for (int i = 0; i < n; ++i) {
      if (!keep[i] || dep[i] >= R) continue;
      int len = dep[i];
      for (int j = i, k = len - 1; j >= 0; j = T->parent[j], --k) path[k] = tok[j];
      path_output(M, kv, kvw, x, s, codes[s], path, len, rows, outs, hn);
      orc_head_logits(M, s + len + 1, hn, NULL, lg);
      orc_process(lg, V, top_k, Tmp, pn + (size_t)(i + 1) * V, &m1);
      if (m1 < mg) mg = m1;
    }
    st->passes++;
    /* walk down from the committed code */
    int cur = -1, d = 0, acc_n = 0;
    while (s + d < G - 1) {
      const float* p = pn + (size_t)(cur + 1) * V;
      memcpy(work, p, sizeof(float) * V);
      int taken = -1, ci = 0;
      for (int i = 0; i < n && taken < 0; ++i) {
        if (!keep[i] || T->parent[i] != cur) continue;
        float S = 0.0f;
        for (int v = 0; v < V; ++v) S = S + work[v];
        const float r = S > 0.0f ? work[tok[i]] / S : 0.0f;
        const float u = orc_uniform(seed, (uint32_t)stream, (uint32_t)frame, (uint32_t)(s + d + 1),
                                    (uint32_t)(ORC_TREE_ACCEPT + ci));
        const double g = fabs((double)u - (double)r);
        if (g < mg) mg = g;
        if (u < r) taken = i;
        else work[tok[i]] = 0.0f;
        ++ci;
      }
      if (taken >= 0) {
        codes[s + d + 1] = tok[taken];
        cur = taken;
        ++d;
        ++acc_n;
        st->accepted_by_offset[d < 9 ? d : 8]++;
        continue;
      }
      const float u = orc_uniform(seed, (uint32_t)stream, (uint32_t)frame, (uint32_t)(s + d + 1), ORC_TARGET);
      int y = orc_sample(work, V, u, &m1);
      if (y < 0) y = orc_sample(p, V, u, &m1);
      if (m1 < mg) mg = m1;
      codes[s + d + 1] = y;
      ++d;
      if (ci > 0) st->rejections++; else st->bonus++;
      break;
    }
    const int s_new = s + d;
    /* reconcile: the cache keeps positions 0..s_new (the committed code and
     * the accepted path); the new hidden is the output at position s_new */
    if (s_new < G - 1) {
      for (int k = 0; k < d - 1; ++k) path[k] = codes[s + 1 + k];
      path_output(M, kv, kvw, x, s, codes[s], path, d - 1, rows, outs, hs);
      memcpy(kv, kvw, sizeof(double) * nkv);
    }
    st->rounds++;
    for (int k = 0; k < 8; ++k) dr[k] = k < acc_n ? codes[s + 1 + k] : -1;
    log_round(log, log_cap, n_log, frame, stream, s, nkeep, nkeep + 1, acc_n, s_new, dr, mg);
    s = s_new;
  }
  st->committed += G - 1;
  st->frames++;
  free(kv); free(kvw); free(rows); free(outs); free(hs); free(hn); free(lg); free(pn); free(work);
  free(order); free(tok); free(dep); free(keep);
}

int orc_decode_frames_tree(const orc_model* M, const orc_tree* T, const int* top_k, const float* temp,
                           uint64_t seed, int B, int F, int first_frame, const float* x, const int* c0, int* codes,
                           orc_stats* st, orc_round_rec* log, int log_cap, int* n_log) {
  if (!M || !T || !codes || !x || !c0 || !st) return -1;
  if (M->G < 2 || M->nq % M->nkv != 0 || M->d % 2 != 0) return -1;
  if (M->K < 0 || (M->K > 0 && !M->draft_offset)) return -1;
  if (T->n < 0 || T->n > 62 || (T->n > 0 && (!T->parent || !T->rank))) return -1;
  for (int i = 0; i < T->n; ++i) {
    if (T->parent[i] < -1 || T->parent[i] >= i || T->rank[i] < 0) return -1; /* parents first */
    for (int j = 0; j < i; ++j) /* siblings in ascending rank, no repeats */
      if (T->parent[j] == T->parent[i] && T->rank[j] >= T->rank[i]) return -1;
  }
  if (n_log) *n_log = 0;
  for (int f = 0; f < F; ++f)
    for (int b = 0; b < B; ++b)
      decode_one_frame_tree(M, T, top_k[b], temp[b], seed, b, first_frame + f, x + ((size_t)f * B + b) * M->H,
                            c0[(size_t)f * B + b], codes + ((size_t)f * B + b) * M->G, st, log, log_cap, n_log);
  return 0;
}
