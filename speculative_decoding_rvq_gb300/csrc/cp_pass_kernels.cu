// cp_pass_kernels.cu -- the kernels of one decoder pass and their launches.
//
// A pass ("CodePredictor Speculative Decoding", "How a round works") is, for
// every active stream, one causal CodePredictor forward over its rows (the
// committed position plus the drafted ones) against the stream's KV cache,
// the lm_heads of those rows (the target heads and, on the row at the
// committed depth, the draft heads head_{s+1..s+N-1}: "Why the draft is
// free"), top-k / temperature processing of every logit row, and the exact
// acceptance that commits codes and stages the next pass.  It runs as
//
//   per layer: QKV GEMV (RMSNorm, RoPE, KV append) -> attention -> O GEMV
//              (residual) -> gate/up GEMV (RMSNorm, SwiGLU) -> down GEMV
//              (residual)
//   then:      lm_head GEMV (final RMSNorm) -> top-k -> accept
//
// one kernel each.  Every kernel after the first is launched as a
// programmatic dependent and lets its own successor start as soon as it
// begins (griddepcontrol.launch_dependents): a kernel's CTAs start while its
// predecessor still runs, issue the bulk copies of their weight tiles and
// copy what the pass plan, the call arguments, the RoPE table and the norm
// gains hold, and only then wait (griddepcontrol.wait) for the
// predecessor's results.  Nothing read before the wait is written inside
// the pass: the plan and the call arguments are written before the pass's
// first kernel starts, and that kernel is a full dependent of earlier work.
//
// Numerics: bf16 (or fp32) weights, fp32 activations, KV cache and
// accumulation.  Every reduction has a fixed order that depends only on the
// model shape (per thread in element order, a butterfly over the warp, warps
// in index order), never on which rows share the pass, so greedy speculative
// decoding reproduces greedy autoregressive decoding exactly.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "cp_common.cuh"
#include "cp_frame.cuh"
#include "cp_sampling.cuh"

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

namespace cpk {

// ------------------------------------------------------------ weight types
// One 16-byte chunk of a weight row in shared memory: loaded raw, then
// converted to float2 pairs.
template <typename WT> struct WTraits;
template <> struct WTraits<float> {
  static constexpr int EB = 4;   // bytes per element
  static constexpr int EPC = 4;  // elements per 16-byte chunk
  typedef float4 Raw;
  __device__ __forceinline__ static Raw ld_raw(const unsigned char* p) { return *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ static void cvt(const Raw& v, float2 (&w)[2]) {
    w[0] = make_float2(v.x, v.y);
    w[1] = make_float2(v.z, v.w);
  }
  __device__ __forceinline__ static float load1(const void* base, size_t i) {
    return __ldg(static_cast<const float*>(base) + i);
  }
};
template <> struct WTraits<__nv_bfloat16> {
  static constexpr int EB = 2;
  static constexpr int EPC = 8;
  typedef uint4 Raw;
  __device__ __forceinline__ static Raw ld_raw(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ static void cvt(const Raw& v, float2 (&w)[4]) {
    w[0] = bf16x2_to_f2(v.x);
    w[1] = bf16x2_to_f2(v.y);
    w[2] = bf16x2_to_f2(v.z);
    w[3] = bf16x2_to_f2(v.w);
  }
  __device__ __forceinline__ static float load1(const void* base, size_t i) {
    const unsigned short u = __ldg(static_cast<const unsigned short*>(base) + i);
    return __uint_as_float((uint32_t)u << 16);
  }
};

// -------------------------------------------------- programmatic launches
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------ GEMV shapes
// Output units of a GEMV kind: QKV = RoPE pair (e, e + d/2) of a head;
// O, down = output row; gate/up = feature (gate row + up row);
// lm_heads = (head of the pass, vocabulary row).
__host__ __device__ __forceinline__ int rows_per_unit(int kind) { return (kind == kQKV || kind == kGU) ? 2 : 1; }

__device__ __forceinline__ int gemv_K(const FrameParams& P, int kind) {
  return kind == kO ? P.nq * P.d : (kind == kDown ? P.F : P.H);
}

__device__ __forceinline__ int gemv_units(const FrameParams& P, int kind, int nheads) {
  switch (kind) {
    case kQKV: return (P.nq + 2 * P.nkv) * (P.d / 2);
    case kO: case kDown: return P.H;
    case kGU: return P.F;
    default: return nheads * P.V;
  }
}

struct Tile {
  int u0, n;  // first output unit and unit count
};
constexpr int kMaxTiles = 96;
constexpr int kRedQ = 8;               // input rows per group at most (partial-sum row stride)
constexpr int kRedFloats = 1536;       // GEMV partial sums of two tiles: rows x kRedQ x warps per row group, per tile
constexpr int kRopeSmemBytes = 8192;   // RoPE table copied to shared memory up to this size

// The two (or one) contiguous byte runs of a tile in global memory: QKV
// rows e and e + d/2 of one head; gate and up rows; else one run.
struct TileRuns {
  const unsigned char* src0;
  const unsigned char* src1;
  uint32_t bytes;  // per run
};

template <typename WT>
__device__ __forceinline__ TileRuns tile_runs(const FrameParams& P, int kind, int l, const int* heads, Tile t) {
  constexpr int EB = WTraits<WT>::EB;
  TileRuns r;
  r.src1 = nullptr;
  switch (kind) {
    case kQKV: {
      const int half = P.d / 2, hh = t.u0 / half, e = t.u0 - hh * half;
      const size_t rb = (size_t)P.H * EB;
      const unsigned char* base;
      if (hh < P.nq) base = static_cast<const unsigned char*>(P.wq[l]) + (size_t)hh * P.d * rb;
      else if (hh < P.nq + P.nkv) base = static_cast<const unsigned char*>(P.wk[l]) + (size_t)(hh - P.nq) * P.d * rb;
      else base = static_cast<const unsigned char*>(P.wv[l]) + (size_t)(hh - P.nq - P.nkv) * P.d * rb;
      r.src0 = base + (size_t)e * rb;
      r.src1 = base + (size_t)(e + half) * rb;
      r.bytes = (uint32_t)(t.n * rb);
      break;
    }
    case kO: {
      const size_t rb = (size_t)P.nq * P.d * EB;
      r.src0 = static_cast<const unsigned char*>(P.wo[l]) + (size_t)t.u0 * rb;
      r.bytes = (uint32_t)(t.n * rb);
      break;
    }
    case kGU: {
      const size_t rb = (size_t)P.H * EB;
      r.src0 = static_cast<const unsigned char*>(P.w_gate[l]) + (size_t)t.u0 * rb;
      r.src1 = static_cast<const unsigned char*>(P.w_up[l]) + (size_t)t.u0 * rb;
      r.bytes = (uint32_t)(t.n * rb);
      break;
    }
    case kDown: {
      const size_t rb = (size_t)P.F * EB;
      r.src0 = static_cast<const unsigned char*>(P.w_down[l]) + (size_t)t.u0 * rb;
      r.bytes = (uint32_t)(t.n * rb);
      break;
    }
    default: {
      const size_t rb = (size_t)P.H * EB;
      const int hi = t.u0 / P.V, v = t.u0 - hi * P.V;
      r.src0 = static_cast<const unsigned char*>(P.head) + ((size_t)(heads[hi] - 1) * P.V + v) * rb;
      r.bytes = (uint32_t)(t.n * rb);
    }
  }
  return r;
}

// Tiles of share c of g, units [U*c/g, U*(c+1)/g) of a kind: at most `upt`
// units each, none crossing a head boundary (QKV, lm_heads).
__device__ int make_tiles(int U, int upt, int period, int c, int g, Tile* out) {
  const int u0 = (int)(((long long)U * c) / g), u1 = (int)(((long long)U * (c + 1)) / g);
  int n = 0;
  for (int u = u0; u < u1;) {
    int e = min(u1, u + upt);
    if (period > 0) e = min(e, (u / period + 1) * period);
    if (n >= kMaxTiles) return -1;
    out[n++] = Tile{u, e - u};
    u = e;
  }
  return n;
}

// ------------------------------------------------------------ GEMV kernels
// Butterfly reduce-scatter of NV values over the warp (offsets 16, 8, 4, 2, 1):
// lane l ends with value l >> (5 - log2 NV) summed over all 32 lanes.  The
// pairing of lanes is the same for every value and every NV, so a value's
// rounding does not depend on its index or on how many values travel.
template <int N, int S>
__device__ __forceinline__ void rs_step(float* v, int lane) {
  if constexpr (N >= 2) {
    constexpr int h = N / 2;
    const bool up = (lane & S) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? v[i] : v[i + h];
      const float keep = up ? v[i + h] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, S);
    }
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], S);
  }
}

template <int NV>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV]) {
  const int lane = threadIdx.x & 31;
  rs_step<NV, 16>(v, lane);
  rs_step<(NV >= 2 ? NV / 2 : 1), 8>(v, lane);
  rs_step<(NV >= 4 ? NV / 4 : 1), 4>(v, lane);
  rs_step<(NV >= 8 ? NV / 8 : 1), 2>(v, lane);
  rs_step<(NV >= 16 ? NV / 16 : 1), 1>(v, lane);
  return v[0];
}

// Where a GEMV input row comes from: an fp32 row, or (first layer, positions
// >= 1) a row of the code embedding in the weight type.
struct ActRow {
  const float* f;
  const void* w;
};

// How the CTA's threads cover a weight row of nch 16-byte chunks: row groups
// of TPG threads (a multiple of 32), thread tl of a group owning chunks
// tl, tl + TPG, ... (CPT of them); group g takes tile rows g, g + RG, ...
struct RowGeom {
  int nch, TPG, RG, CPT;
};

__device__ __forceinline__ RowGeom row_geom(int nch) {
  RowGeom g;
  g.nch = nch;
  g.TPG = min(kThreads, (nch + 31) / 32 * 32);
  g.RG = kThreads / g.TPG;
  g.CPT = (nch + g.TPG - 1) / g.TPG;
  return g;
}

// Raw input element values k0 .. k0 + EPC - 1 of row `src` (as float2 pairs).
template <typename WT>
__device__ __forceinline__ void load_act(const ActRow& src, int k0, float2 (&out)[WTraits<WT>::EPC / 2]) {
  constexpr int EPC = WTraits<WT>::EPC, PPC = EPC / 2;
  if (src.f != nullptr) {
#pragma unroll
    for (int i = 0; i < EPC; i += 4) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(src.f + k0 + i));
      out[i / 2] = make_float2(x.x, x.y);
      out[i / 2 + 1] = make_float2(x.z, x.w);
    }
  } else {
    WTraits<WT>::cvt(__ldg(reinterpret_cast<const typename WTraits<WT>::Raw*>(
                         static_cast<const unsigned char*>(src.w) + (size_t)k0 * WTraits<WT>::EB)),
                     out);
  }
  (void)PPC;
}

// The pass rows as a GEMV CTA sees them: the plan's arrays, copied to
// shared memory before the dependency wait (the plan is written before the
// pass's first kernel starts).
struct PassRows {
  const int* prow;
  const int* ppos;
  const int* pcode;
};

// Input row i of the pass (compacted index) for a GEMV kind.
template <typename WT>
__device__ __forceinline__ ActRow act_row(const FrameParams& P, const CallArgs& ca, const PassRows& pr, int kind, int l,
                                          int i) {
  const int r = pr.prow[i];
  ActRow a{nullptr, nullptr};
  switch (kind) {
    case kQKV:
      if (l == 0) {
        const int pos = pr.ppos[i], code = pr.pcode[i], b = r / P.NS;
        if (pos == 0)
          a.f = ca.mode == kModeTeacher ? ca.x + (size_t)b * P.H : ca.x + ((size_t)code * ca.B + b) * P.H;
        else
          a.w = static_cast<const WT*>(P.embed) + ((size_t)(pos - 1) * P.V + code) * P.H;
      } else {
        a.f = P.h + (size_t)r * P.H;
      }
      break;
    case kO: a.f = P.abuf + (size_t)r * P.nq * P.d; break;
    case kGU: a.f = P.h + (size_t)r * P.H; break;
    case kDown: a.f = P.fbuf + (size_t)r * P.F; break;
    default: a.f = P.h + (size_t)r * P.H;
  }
  return a;
}

// Outputs of one unit for pass row gi: RoPE + q / KV append (QKV), residual
// update (O, down), SwiGLU (gate/up), logits (lm_heads).
template <int KIND>
__device__ __forceinline__ void gemv_out(const FrameParams& P, int l, const int* heads, const PassRows& pr,
                                         const float2* rope, int u, int gi, float y0, float y1, float hold) {
  const int r = pr.prow[gi], pos = pr.ppos[gi];
  if (KIND == kQKV) {
    const int half = P.d / 2, hh = u / half, e = u - hh * half;
    const int b = r / P.NS;
    if (hh < P.nq + P.nkv) {
      const float2 cs2 = rope[(size_t)pos * half + e];
      const float r0 = y0 * cs2.x - y1 * cs2.y;
      const float r1 = y1 * cs2.x + y0 * cs2.y;
      if (hh < P.nq) {
        float* qd = P.qbuf + (size_t)r * P.nq * P.d + (size_t)hh * P.d;
        qd[e] = r0;
        qd[e + half] = r1;
      } else {
        const int slot = P.tree_n ? __ldcg(P.pslot + gi) : pos;  // KV slot (a tree node's own slot)
        float* kd = P.kv + (((((size_t)b * P.L + l) * 2 + 0) * P.GS + slot) * P.nkv + (hh - P.nq)) * P.d;
        kd[e] = r0;
        kd[e + half] = r1;
      }
    } else {
      const int slot = P.tree_n ? __ldcg(P.pslot + gi) : pos;
      float* vd = P.kv + (((((size_t)b * P.L + l) * 2 + 1) * P.GS + slot) * P.nkv + (hh - P.nq - P.nkv)) * P.d;
      vd[e] = y0;
      vd[e + half] = y1;
    }
  } else if (KIND == kO || KIND == kDown) {
    P.h[(size_t)r * P.H + u] = hold + y0;
  } else if (KIND == kGU) {
    P.fbuf[(size_t)r * P.F + u] = y0 / (1.0f + expf(-y0)) * y1;
  } else {
    const int hi = u / P.V, v = u - hi * P.V;
    const int slot = heads[hi] - pos;
    // a lookahead-t draft with a position-aware offset reads head_j on
    // h + b_t = head_j . h + head_j . b_t (the second term from the table)
    if (slot >= 1 && slot <= P.KO) y0 += __ldg(&P.otab[((size_t)(heads[hi] - 1) * P.KO + slot - 1) * P.V + v]);
    if (pos >= 1 && slot >= 0 && slot <= P.ND) P.logits[((size_t)r * (1 + P.ND) + slot) * P.V + v] = y0;
  }
}

// Shared state of a GEMV CTA.
struct GemvShared {
  uint64_t full[2];           // tile landed in slot 0 / 1
  Tile tiles[kMaxTiles];
  int ntiles;
  int heads[kMaxHeadsPerPass];
  int issued;                 // tiles whose copies were issued
  int blk0, blk1;             // tensor path: the CTA's blocks of 16 pass rows
  int wcnt[kWarps];           // tensor path, lm_heads: rows found per warp (compaction)
  ActRow src[kRedQ];
  float ss[kWarps][kRedQ];    // RMSNorm partial sums of squares per warp
};

// Issue the bulk copies of tile t into slot t & 1 (thread 0).
template <typename WT, int KIND>
__device__ __forceinline__ void gemv_issue(const FrameParams& P, int l, GemvShared& sh, unsigned char* slots, int t) {
  const int slot = t & 1;
  const TileRuns r = tile_runs<WT>(P, KIND, l, sh.heads, sh.tiles[t]);
  unsigned char* dst = slots + (size_t)slot * kSlotBytes;
  const uint64_t pol = l2_evict_first_policy();
  // test hook: the first tile of the pass's first GEMV in CTA 0 expects 16
  // bytes that no copy delivers, so its bounded wait runs out
  const uint32_t stall = (P.test_stall && KIND == kQKV && l == 0 && t == 0 && blockIdx.x == 0) ? 16u : 0u;
  mbar_arrive_expect_tx(&sh.full[slot], (r.src1 ? 2 * r.bytes : r.bytes) + stall);
  bulk_copy_g2s(dst, r.src0, r.bytes, &sh.full[slot], pol);
  if (r.src1) bulk_copy_g2s(dst + r.bytes, r.src1, r.bytes, &sh.full[slot], pol);
  sh.issued = t + 1;
}


// One input group (rows q0 .. q0 + NQ - 1, rows past nqv repeat row nqv - 1
// and are discarded) against tiles [ta, tb).  A thread loads its chunks of
// the group's inputs once; for the normed kinds the sum of squares of each
// row is taken over row group 0 (per thread over its chunks in order, the
// warp butterfly, the warps in order) and the values are scaled by
// inv * gain.  Per tile: all threads wait for the slot, form their partial
// sums (per (row, input row) a lane accumulates its chunks in order, even and
// odd elements in the two halves of an f32x2 accumulator; the warp's
// reduce-scatter adds the lanes), then the epilogue adds the warps of a row
// group in order and writes the outputs.  With `issue_next`, thread 0 refills
// a slot with tile t + 2 once every thread is past tile t.
template <typename WT, int KIND, int CPT, int NQ>
__device__ __forceinline__ bool gemv_run(const FrameParams& P, const CallArgs& ca, int l, const RowGeom& G,
                                         GemvShared& sh, const PassRows& pr, const float2* rope, unsigned char* slots,
                                         float* red, int q0, int nqv, int ta, int tb, bool issue_next,
                                         const float* gain) {
  using Raw = typename WTraits<WT>::Raw;
  constexpr int EPC = WTraits<WT>::EPC, PPC = EPC / 2;
  constexpr int EB = WTraits<WT>::EB;
  constexpr int KRB = NQ >= 8 ? 2 : kRB;  // weight rows per batch (fewer with 8 input rows, for registers)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = tid / G.TPG;
  const bool active = g < G.RG;  // whole warps: TPG is a multiple of 32
  const int tl = tid - g * G.TPG, wg = tl >> 5, WPG = G.TPG >> 5;
  const int K = G.nch * 16 / EB;
  const int rpu = rows_per_unit(KIND);
  const size_t row_bytes = (size_t)G.nch * 16;
  if (tid < 32 * nqv && lane == 0) sh.src[warp] = act_row<WT>(P, ca, pr, KIND, l, q0 + warp);
  __syncthreads();
  float2 av[CPT][NQ][PPC];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = tl + j * G.TPG;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (active && c < G.nch) {
        load_act<WT>(sh.src[min(q, nqv - 1)], c * EPC, av[j][q]);
      } else {
#pragma unroll
        for (int p = 0; p < PPC; ++p) av[j][q][p] = make_float2(0.f, 0.f);
      }
    }
  }
  if (gain != nullptr) {
    float ss[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      ss[q] = 0.0f;
#pragma unroll
      for (int j = 0; j < CPT; ++j)
#pragma unroll
        for (int p = 0; p < PPC; ++p) {
          ss[q] = fmaf(av[j][q][p].x, av[j][q][p].x, ss[q]);
          ss[q] = fmaf(av[j][q][p].y, av[j][q][p].y, ss[q]);
        }
      ss[q] = warp_sum(ss[q]);
    }
    if (g == 0 && lane == 0)
#pragma unroll
      for (int q = 0; q < NQ; ++q) sh.ss[wg][q] = ss[q];
    __syncthreads();
    float inv[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      float t = 0.0f;
      for (int w = 0; w < WPG; ++w) t += sh.ss[w][q];
      inv[q] = 1.0f / sqrtf(t / (float)K + P.eps);
    }
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = tl + j * G.TPG;
      if (!active || c >= G.nch) continue;
#pragma unroll
      for (int i = 0; i < EPC; i += 4) {
        const float4 gg = *reinterpret_cast<const float4*>(gain + c * EPC + i);  // shared memory
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float2& a0 = av[j][q][i / 2];
          float2& a1 = av[j][q][i / 2 + 1];
          a0.x = a0.x * inv[q] * gg.x;
          a0.y = a0.y * inv[q] * gg.y;
          a1.x = a1.x * inv[q] * gg.z;
          a1.y = a1.y * inv[q] * gg.w;
        }
      }
    }
  }
  bool ok = true;
  // tiles in pairs (one per slot): both computed, then one epilogue
  for (int t0 = ta; t0 < tb; t0 += 2) {
    const int nt = min(2, tb - t0);
    Tile tiles[2];
    tiles[0] = sh.tiles[t0];
    tiles[1] = nt > 1 ? sh.tiles[t0 + 1] : Tile{0, 0};
    const int n_items0 = tiles[0].n * nqv, n_items = n_items0 + tiles[1].n * nqv;
    // residual values the epilogue adds to (O, down), fetched before the tile is computed
    constexpr int kHold = 2;
    float hold[kHold] = {0.0f, 0.0f};
    if (KIND == kO || KIND == kDown) {
#pragma unroll
      for (int m = 0; m < kHold; ++m) {
        const int it = tid + m * kThreads;
        if (it < n_items) {
          const int k = it < n_items0 ? 0 : 1, jt = it - k * n_items0;
          const int i = jt / nqv, q = jt - i * nqv;
          hold[m] = __ldcg(P.h + (size_t)pr.prow[q0 + q] * P.H + tiles[k].u0 + i);
        }
      }
    }
    for (int k = 0; k < nt; ++k) {
      const int t = t0 + k, slot = t & 1;
      const int R = tiles[k].n * rpu;
      float* rk = red + k * (kRedFloats / 2);
      if (!mbar_wait_bounded(&sh.full[slot], (uint32_t)(t >> 1) & 1u, &P.ctl->status, P.wait_ns)) ok = false;
      if (!active || !ok) continue;
      const unsigned char* tp = slots + (size_t)slot * kSlotBytes;
      const int nrow = (R - g + G.RG - 1) / G.RG;  // rows g, g + RG, ... of the tile
      for (int i0 = 0; i0 < nrow; i0 += KRB) {
        int rw[KRB];
#pragma unroll
        for (int w = 0; w < KRB; ++w) rw[w] = g + G.RG * min(i0 + w, nrow - 1);
        float2 acc[KRB][NQ];
#pragma unroll
        for (int w = 0; w < KRB; ++w)
#pragma unroll
          for (int q = 0; q < NQ; ++q) acc[w][q] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int c = tl + j * G.TPG;
          if (c >= G.nch) continue;
          Raw raw[KRB];
#pragma unroll
          for (int w = 0; w < KRB; ++w) raw[w] = WTraits<WT>::ld_raw(tp + (size_t)rw[w] * row_bytes + (size_t)c * 16);
#pragma unroll
          for (int w = 0; w < KRB; ++w) {
            float2 wv[PPC];
            WTraits<WT>::cvt(raw[w], wv);
#pragma unroll
            for (int q = 0; q < NQ; ++q)
#pragma unroll
              for (int p = 0; p < PPC; ++p) acc[w][q] = ffma2(wv[p], av[j][q][p], acc[w][q]);
          }
        }
        float v[KRB * NQ];
#pragma unroll
        for (int w = 0; w < KRB; ++w)
#pragma unroll
          for (int q = 0; q < NQ; ++q) v[w * NQ + q] = acc[w][q].x + acc[w][q].y;
        const float sum = reduce_scatter<KRB * NQ>(v);
        constexpr int NV = KRB * NQ;
        constexpr int shift = NV >= 32 ? 0 : (NV >= 16 ? 1 : (NV >= 8 ? 2 : (NV >= 4 ? 3 : 4)));
        if ((lane & ((1 << shift) - 1)) == 0) {
          const int vi = lane >> shift, w = vi / NQ, q = vi % NQ;
          if (i0 + w < nrow) rk[((size_t)rw[w] * kRedQ + q) * WPG + wg] = sum;
        }
      }
    }
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (!ok) return false;
    for (int it = tid, m = 0; it < n_items; it += kThreads, ++m) {
      const int k = it < n_items0 ? 0 : 1, jt = it - k * n_items0;
      const int i = jt / nqv, q = jt - i * nqv;
      const Tile tile = tiles[k];
      const float* rk = red + k * (kRedFloats / 2);
      float ys[2] = {0.0f, 0.0f};
      for (int h = 0; h < rpu; ++h) {
        const float* rr = rk + ((size_t)(i + h * tile.n) * kRedQ + q) * WPG;
        float s = 0.0f;
        for (int w = 0; w < WPG; ++w) s += rr[w];
        ys[h] = s;
      }
      float ho = 0.0f;
      if (KIND == kO || KIND == kDown) {
#pragma unroll
        for (int mm = 0; mm < kHold; ++mm) if (mm == m) ho = hold[mm];
        if (m >= kHold) ho = __ldcg(P.h + (size_t)pr.prow[q0 + q] * P.H + tile.u0 + i);
      }
      gemv_out<KIND>(P, l, sh.heads, pr, rope, tile.u0 + i, q0 + q, ys[0], ys[1], ho);
    }
    __syncthreads();  // red reuse; the slots are free
    if (issue_next && tid == 0)
      for (int k = 0; k < nt; ++k)
        if (t0 + k + 2 < sh.ntiles) gemv_issue<WT, KIND>(P, l, sh, slots, t0 + k + 2);
  }
  return true;
}


// --------------------------------------------------- tensor-core GEMV path
// For contexts with many rows per pass (many streams), the bf16 GEMVs are
// small GEMMs: mma.sync m16n8k16 (bf16 x bf16 -> f32) with the weight tile
// in shared memory as the column-major B operand and the input rows as A.
// The fp32 inputs are split into bf16 hi + lo parts (two MMAs per step), so
// an input keeps 16 mantissa bits.  Within each 32-element block of K a
// fixed permutation gives every lane 16 contiguous bytes of a weight row and
// two float4 of an input row per two k-steps (the same permutation on A and
// B, so the dot product is unchanged).  Every output element is one warp's
// MMA chain over K in order: its value does not depend on the other rows
// of the pass.

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (x0, x1) -> bf16x2 hi and bf16x2 lo with x ~ hi + lo (low half = x0).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 o = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&o);
}

// Eight input values k0 .. k0 + 7 of a row (fp32 row or bf16 embedding row).
__device__ __forceinline__ void load_act8(const ActRow& a, int k0, float (&v)[8]) {
  if (a.f != nullptr) {
    const float4 x0 = __ldcg(reinterpret_cast<const float4*>(a.f + k0));
    const float4 x1 = __ldcg(reinterpret_cast<const float4*>(a.f + k0 + 4));
    v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w; v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
  } else {
    float2 w[4];
    WTraits<__nv_bfloat16>::cvt(__ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.w) + k0)), w);
#pragma unroll
    for (int p = 0; p < 4; ++p) { v[2 * p] = w[p].x; v[2 * p + 1] = w[p].y; }
  }
}

constexpr int kTcMaxN = 4;  // n-tiles of 8 weight rows per tile (tiles hold at most 32 rows on this path)
constexpr int kTcPipe = 1;  // K blocks of 32 whose inputs are loaded ahead
// per-warp output blocks (16 rows x the columns of two tiles) and 16 row descriptors
constexpr int kTcYCols = 2 * kTcMaxN * 8;
constexpr int kTcYFloats = kWarps * 16 * kTcYCols + kWarps * 16 * (int)(sizeof(ActRow) / sizeof(float));

// A pair of resident tiles (R0 and R1 weight rows, K inputs; R1 = 0 when
// there is one) against pass rows [m0, m0 + 16) by one warp: one MMA chain
// over K per 8-row n-tile, the inputs loaded and split once for both tiles;
// then the outputs of the tiles' units for those rows.  src: the warp's 16
// input rows (rows past nrows repeat the last).  Normed kinds (gain set):
// RMSNorm(x) . w = inv(x) * sum_k (x_k g_k) w_k, so the MMAs take x * g and
// the row's sum of squares is accumulated in the same pass over K (per lane
// in element order, then over the 4 lanes of a row in a fixed order); the
// scale inv = 1 / sqrt(mean(x^2) + eps) multiplies the accumulators.
template <int KIND, int NTT>
__device__ __noinline__ void tc_block(const FrameParams& P, int l, const int* heads, const PassRows& pr,
                                         const float2* rope, const unsigned char* tp0, const unsigned char* tp1,
                                         Tile tl0, Tile tl1, int nt0, int K, const ActRow* src,
                                         const float* gain, int m0, int nrows, const int* rl, float* y) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int rpu = rows_per_unit(KIND);
  const int R0 = tl0.n * rpu, R1 = tl1.n * rpu;
  const size_t row_bytes = (size_t)K * 2;
  float c[NTT][4];
#pragma unroll
  for (int j = 0; j < NTT; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.0f;
  const ActRow ra = src[g], rb = src[g + 8];
  float ssa = 0.0f, ssb = 0.0f;
  // weight row of n-tile j for this lane, as a byte offset from tp0 (the
  // second slot follows the first)
  uint32_t wr[NTT];
#pragma unroll
  for (int j = 0; j < NTT; ++j)
    wr[j] = (uint32_t)(j < nt0 ? (size_t)min(8 * j + g, R0 - 1) * row_bytes
                               : (size_t)(tp1 - tp0) + (size_t)min(8 * (j - nt0) + g, R1 - 1) * row_bytes) +
            (uint32_t)t * 16;
  // K in blocks of 32; the inputs of kTcPipe blocks are loaded before any of
  // them is used, so that many L2 reads are in flight per warp
  for (int kb0 = 0; kb0 < K; kb0 += 32 * kTcPipe) {
    float pa[kTcPipe][8], pb[kTcPipe][8];
#pragma unroll
    for (int u = 0; u < kTcPipe; ++u) {
      const int kb = kb0 + 32 * u;
      if (kb < K) {
        load_act8(ra, kb + 8 * t, pa[u]);
        load_act8(rb, kb + 8 * t, pb[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kTcPipe; ++u) {
      const int kb = kb0 + 32 * u;
      if (kb >= K) break;
      const int k0 = kb + 8 * t;
      float (&va)[8] = pa[u];
      float (&vb)[8] = pb[u];
      if (gain != nullptr) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float gk = gain[k0 + e];
          ssa = fmaf(va[e], va[e], ssa);
          ssb = fmaf(vb[e], vb[e], ssb);
          va[e] *= gk;
          vb[e] *= gk;
        }
      }
      uint32_t ah[2][4], al[2][4];
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        split_bf16x2(va[4 * s + 0], va[4 * s + 1], ah[s][0], al[s][0]);
        split_bf16x2(vb[4 * s + 0], vb[4 * s + 1], ah[s][1], al[s][1]);
        split_bf16x2(va[4 * s + 2], va[4 * s + 3], ah[s][2], al[s][2]);
        split_bf16x2(vb[4 * s + 2], vb[4 * s + 3], ah[s][3], al[s][3]);
      }
#pragma unroll
      for (int j = 0; j < NTT; ++j) {
        const uint4 w = *reinterpret_cast<const uint4*>(tp0 + wr[j] + (size_t)kb * 2);
        mma_bf16_16816(c[j], ah[0][0], ah[0][1], ah[0][2], ah[0][3], w.x, w.y);
        mma_bf16_16816(c[j], al[0][0], al[0][1], al[0][2], al[0][3], w.x, w.y);
        mma_bf16_16816(c[j], ah[1][0], ah[1][1], ah[1][2], ah[1][3], w.z, w.w);
        mma_bf16_16816(c[j], al[1][0], al[1][1], al[1][2], al[1][3], w.z, w.w);
      }
    }
  }
  if (gain != nullptr) {
    ssa += __shfl_xor_sync(0xffffffffu, ssa, 1);
    ssb += __shfl_xor_sync(0xffffffffu, ssb, 1);
    ssa += __shfl_xor_sync(0xffffffffu, ssa, 2);
    ssb += __shfl_xor_sync(0xffffffffu, ssb, 2);
    const float ia = 1.0f / sqrtf(ssa / (float)K + P.eps), ib = 1.0f / sqrtf(ssb / (float)K + P.eps);
#pragma unroll
    for (int j = 0; j < NTT; ++j) {
      c[j][0] *= ia;
      c[j][1] *= ia;
      c[j][2] *= ib;
      c[j][3] *= ib;
    }
  }
  // C fragment: c[j][0..1] = row g, cols 8j + 2t, +1; c[j][2..3] = row g + 8
  constexpr int W = NTT * 8;
#pragma unroll
  for (int j = 0; j < NTT; ++j) {
    y[g * W + 8 * j + 2 * t] = c[j][0];
    y[g * W + 8 * j + 2 * t + 1] = c[j][1];
    y[(g + 8) * W + 8 * j + 2 * t] = c[j][2];
    y[(g + 8) * W + 8 * j + 2 * t + 1] = c[j][3];
  }
  __syncwarp();
  const int rows = min(16, nrows - m0);
  for (int k = 0; k < 2; ++k) {
    const Tile tl = k == 0 ? tl0 : tl1;
    const int col0 = k == 0 ? 0 : 8 * nt0;
    for (int it = lane; it < tl.n * rows; it += 32) {
      const int i = it / rows, q = it - i * rows;
      const float y0 = y[q * W + col0 + i], y1 = rpu == 2 ? y[q * W + col0 + i + tl.n] : 0.0f;
      const int gi = rl != nullptr ? rl[m0 + q] : m0 + q;
      float ho = 0.0f;
      if (KIND == kO || KIND == kDown) ho = __ldcg(P.h + (size_t)pr.prow[gi] * P.H + tl.u0 + i);
      gemv_out<KIND>(P, l, heads, pr, rope, tl.u0 + i, gi, y0, y1, ho);
    }
  }
  __syncwarp();
}

// The pass rows (compacted indices, ascending) whose logit slots read head
// h0 or h1: the rows the lm_head epilogue keeps an output of.  Every thread
// of the CTA takes part.
__device__ int heads_rows(const FrameParams& P, const PassRows& pr, int nrows, int h0, int h1, int* out, int* wcnt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int total = 0;
  for (int base = 0; base < nrows; base += kThreads) {
    const int i = base + threadIdx.x;
    bool need = false;
    if (i < nrows) {
      const int pos = pr.ppos[i], s0 = h0 - pos, s1 = h1 - pos;
      need = pos >= 1 && ((s0 >= 0 && s0 <= P.ND) || (s1 >= 0 && s1 <= P.ND));
    }
    const unsigned bal = __ballot_sync(0xffffffffu, need);
    if (lane == 0) wcnt[warp] = __popc(bal);
    __syncthreads();
    int off = total, sum = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) off += wcnt[w];
      sum += wcnt[w];
    }
    if (need) out[off + __popc(bal & ((1u << lane) - 1u))] = i;
    total += sum;
    __syncthreads();
  }
  return total;
}

// The tensor-core GEMV of one kind for the CTA's blocks of 16 pass rows
// [blk0, blk1) (bf16 weights): tiles in resident pairs (both slots); per
// pair, warp w takes blocks blk0 + w, blk0 + w + kWarps, ..., so each block's
// inputs are read and split once per pair.
template <int KIND>
__device__ __forceinline__ bool gemv_tc(const FrameParams& P, const CallArgs& ca, int l, GemvShared& sh,
                                        const PassRows& pr, const float2* rope, unsigned char* slots, float* ybuf,
                                        int* s_rl, int nrows, const float* gain) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = gemv_K(P, KIND);
  const int rpu = rows_per_unit(KIND);
  float* y = ybuf + (size_t)warp * 16 * kTcYCols;
  ActRow* src = reinterpret_cast<ActRow*>(ybuf + (size_t)kWarps * 16 * kTcYCols) + warp * 16;  // 16 row descriptors per warp
  bool ok = true;
  for (int t0 = 0; t0 < sh.ntiles; t0 += 2) {
    const bool two = t0 + 1 < sh.ntiles;
    const Tile tl0 = sh.tiles[t0], tl1 = two ? sh.tiles[t0 + 1] : Tile{0, 0};
    // lm_heads: only the rows whose logit slots read the pair's heads (each
    // row reads 1 + N-1 of the pass's heads); other kinds: every row
    int nr = nrows;
    const int* rl = nullptr;
    if (KIND == kHeads) {
      nr = heads_rows(P, pr, nrows, sh.heads[tl0.u0 / P.V], sh.heads[(two ? tl1.u0 : tl0.u0) / P.V], s_rl, sh.wcnt);
      rl = s_rl;
    }
    const int nblk = min((nr + 15) / 16, sh.blk1);
    if (!mbar_wait_bounded(&sh.full[0], (uint32_t)(t0 >> 1) & 1u, &P.ctl->status, P.wait_ns)) ok = false;
    if (two && !mbar_wait_bounded(&sh.full[1], (uint32_t)(t0 >> 1) & 1u, &P.ctl->status, P.wait_ns)) ok = false;
    if (ok) {
      const int nt0 = (tl0.n * rpu + 7) / 8, ntt = nt0 + (tl1.n * rpu + 7) / 8;
      for (int mb = sh.blk0 + warp; mb < nblk; mb += kWarps) {
        const int m0 = mb * 16;
        if (lane < 16) {
          const int q = min(m0 + lane, nr - 1);
          src[lane] = act_row<__nv_bfloat16>(P, ca, pr, KIND, l, rl != nullptr ? rl[q] : q);
        }
        __syncwarp();
#define CP_TC(N_) \
  tc_block<KIND, N_>(P, l, sh.heads, pr, rope, slots, slots + kSlotBytes, tl0, tl1, nt0, K, src, gain, m0, nr, rl, y)
        switch (ntt) {
          case 1: CP_TC(1); break;
          case 2: CP_TC(2); break;
          case 3: CP_TC(3); break;
          case 4: CP_TC(4); break;
          case 5: CP_TC(5); break;
          case 6: CP_TC(6); break;
          case 7: CP_TC(7); break;
          default: CP_TC(8); break;
        }
#undef CP_TC
      }
    }
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (!ok) return false;
    if (threadIdx.x == 0) {
      if (t0 + 2 < sh.ntiles) gemv_issue<__nv_bfloat16, KIND>(P, l, sh, slots, t0 + 2);
      if (t0 + 3 < sh.ntiles) gemv_issue<__nv_bfloat16, KIND>(P, l, sh, slots, t0 + 3);
    }
  }
  return true;
}

template <typename WT, int KIND>
__device__ __forceinline__ bool gemv_tc_any(const FrameParams& P, const CallArgs& ca, int l, GemvShared& sh,
                                            const PassRows& pr, const float2* rope, unsigned char* slots, float* ybuf,
                                            int* s_rl, int nrows, const float* gain) {
  if constexpr (WTraits<WT>::EB == 2) return gemv_tc<KIND>(P, ca, l, sh, pr, rope, slots, ybuf, s_rl, nrows, gain);
  return false;  // fp32 weights never take the tensor path
}

// Input rows per group for a geometry: 8 when a thread owns one chunk of a
// row, 4 with two and 2 with three (registers).
__device__ __forceinline__ int group_rows(const RowGeom& G) { return G.CPT >= 3 ? 2 : (G.CPT == 2 ? 4 : 8); }

template <typename WT, int KIND>
__device__ __forceinline__ bool gemv_dispatch(const FrameParams& P, const CallArgs& ca, int l, const RowGeom& G,
                                              GemvShared& sh, const PassRows& pr, const float2* rope,
                                              unsigned char* slots, float* red, int q0, int nqv, int ta, int tb,
                                              bool issue_next, const float* gain) {
#define CP_RUN(C_, Q_) \
  gemv_run<WT, KIND, C_, Q_>(P, ca, l, G, sh, pr, rope, slots, red, q0, nqv, ta, tb, issue_next, gain)
  if (G.CPT == 1) {
    if (nqv >= 5) return CP_RUN(1, 8);
    if (nqv >= 3) return CP_RUN(1, 4);
    if (nqv == 2) return CP_RUN(1, 2);
    return CP_RUN(1, 1);
  }
  if (G.CPT == 2) {
    if (nqv >= 3) return CP_RUN(2, 4);
    if (nqv == 2) return CP_RUN(2, 2);
    return CP_RUN(2, 1);
  }
  if (nqv >= 2) return CP_RUN(3, 2);
  return CP_RUN(3, 1);
#undef CP_RUN
}

// One GEMV kind of one layer for every row of the pass.  The CTA's share of
// output units is cut into tiles of at most kSlotBytes; tiles stream through
// two shared-memory slots by TMA bulk copies, the first two issued before the
// dependency wait.  With one input group (up to 4 rows) or at most two
// tiles, each group's inputs are loaded once and every tile streams through
// them; otherwise tile by tile, group by group.
template <typename WT, int KIND, bool TC>
__global__ void __launch_bounds__(kThreads, TC ? 1 : 2) gemv_kernel(const __grid_constant__ FrameParams P, int l) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  __shared__ GemvShared sh;
  __shared__ CallArgs s_ca;
  __shared__ int s_nrows;
  constexpr int EB = WTraits<WT>::EB;
  const int K = gemv_K(P, KIND);
  const RowGeom G = row_geom(K * EB / 16);
  const int rpu = rows_per_unit(KIND);
  const size_t row_bytes = (size_t)G.nch * 16;
  int upt = max(1, min((int)(kSlotBytes / (rpu * row_bytes)), kMaxTileRows / rpu));
  if (TC) upt = max(1, min(upt, kTcMaxN * 8 / rpu));  // tensor path: at most 32 rows per tile
  const int rows_cap = P.Bmax * P.NS;
  unsigned char* slots = smem;
  float* red = reinterpret_cast<float*>(smem + 2 * (size_t)kSlotBytes);
  int* s_rows = reinterpret_cast<int*>(red + kRedFloats);
  PassRows pr{s_rows, s_rows + rows_cap, s_rows + 2 * rows_cap};
  const size_t rope_n = (size_t)P.G * (P.d / 2);
  const bool rope_in_smem = KIND == kQKV && rope_n * sizeof(float2) <= (size_t)kRopeSmemBytes;
  float2* s_rope = reinterpret_cast<float2*>(s_rows + (3 * rows_cap + 3) / 4 * 4);  // 16-byte aligned
  // RMSNorm gain (a weight) in shared memory after the RoPE table; then, on
  // the tensor path, the per-warp output blocks and row descriptors and the
  // rows' RMSNorm scales
  float* s_gain = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(s_rope) + kRopeSmemBytes);
  float* s_tcy = s_gain + (P.H + 3) / 4 * 4;
  int* s_rl = reinterpret_cast<int*>(s_tcy + kTcYFloats);  // tensor path, lm_heads: row list
  const float* gain_g = KIND == kQKV ? P.attn_norm[l] : (KIND == kGU ? P.ffn_norm[l] : (KIND == kHeads ? P.final_norm : nullptr));
  // Before the dependency wait: everything that does not come from the
  // previous kernels of the pass (weight tiles, call arguments, the pass
  // plan, the RoPE table, the norm gain).
  if (threadIdx.x == 0) {
    int nheads = 0;
    if (KIND == kHeads) {
      nheads = min(__ldcg(&P.plan->nheads), kMaxHeadsPerPass);
      for (int i = 0; i < nheads; ++i) sh.heads[i] = __ldcg(&P.plan->heads[i]);
    }
    s_nrows = min(__ldcg(&P.plan->nrows), rows_cap);
    const int period = KIND == kQKV ? P.d / 2 : (KIND == kHeads ? P.V : 0);
    const int U = gemv_units(P, KIND, nheads);
    // Share of the output units.  On the tensor path, when there are fewer
    // tile pairs than CTAs, the CTAs also split the pass's blocks of 16 rows
    // S ways (S CTAs per unit share), so that each CTA reads and splits 1/S
    // of the input rows; an output element is still one warp's MMA chain.
    int c = blockIdx.x, g = gridDim.x;
    sh.blk0 = 0;
    sh.blk1 = 1 << 30;
    if (TC && KIND != kHeads) {
      const int nblk = (s_nrows + 15) / 16;
      const int pairs = max(1, ((U + upt - 1) / upt + 1) / 2);
      const int S = max(1, min(g / pairs, nblk));
      const int NG = g / S;
      if (c < NG * S) {
        const int rs = c / NG;
        sh.blk0 = (nblk * rs) / S;
        sh.blk1 = (nblk * (rs + 1)) / S;
        c -= rs * NG;
        g = NG;
      } else {
        c = -1;  // spare CTA: no share
      }
    }
    int n = c < 0 ? 0 : make_tiles(U, upt, period, c, g, sh.tiles);
    if (n < 0) { raise_status(&P.ctl->status, kStatusDevice); n = 0; }
    sh.ntiles = n;
    sh.issued = 0;
    mbar_init(&sh.full[0], 1);
    mbar_init(&sh.full[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int t = 0; t < min(n, 2); ++t) gemv_issue<WT, KIND>(P, l, sh, slots, t);
    s_ca = *P.call;
  }
  __syncthreads();
  const int nrows = s_nrows;
  for (int i = threadIdx.x; i < nrows; i += kThreads) {
    s_rows[i] = __ldcg(P.prow + i);
    s_rows[rows_cap + i] = __ldcg(P.ppos + i);
    s_rows[2 * rows_cap + i] = __ldcg(P.pcode + i);
  }
  if (rope_in_smem)
    for (size_t i = threadIdx.x; i < rope_n; i += kThreads) s_rope[i] = __ldg(P.rope + i);
  if (gain_g != nullptr)
    for (int i = threadIdx.x; i < K / 4; i += kThreads)
      reinterpret_cast<float4*>(s_gain)[i] = __ldg(reinterpret_cast<const float4*>(gain_g) + i);
  __syncthreads();
  pdl_wait();
  const CallArgs& ca = s_ca;
  const float2* rope = rope_in_smem ? s_rope : P.rope;
  const int ntiles = sh.ntiles;
  const float* gain = gain_g != nullptr ? s_gain : nullptr;
  if (KIND == kQKV && l == 0) {
    // the residual stream starts as the input rows: this CTA's slice of H
    const int c0 = (int)(((long long)P.H * blockIdx.x) / gridDim.x), c1 = (int)(((long long)P.H * (blockIdx.x + 1)) / gridDim.x);
    const int w = c1 - c0;
    for (int it = threadIdx.x; it < nrows * w; it += kThreads) {
      const int i = it / w, k = c0 + (it - i * w);
      const ActRow a = act_row<WT>(P, ca, pr, KIND, l, i);
      P.h[(size_t)pr.prow[i] * P.H + k] = a.f ? __ldcg(a.f + k) : WTraits<WT>::load1(a.w, (size_t)k);
    }
  }
  const int NQG = group_rows(G);
  const int ngroups = (nrows + NQG - 1) / NQG;
  bool ok = true;
  if constexpr (TC) {
    if (nrows > 0) ok = gemv_tc_any<WT, KIND>(P, ca, l, sh, pr, rope, slots, s_tcy, s_rl, nrows, gain);
  } else if (ngroups <= 1 || ntiles <= 2) {
    for (int gq = 0; gq < ngroups && ok; ++gq)
      ok = gemv_dispatch<WT, KIND>(P, ca, l, G, sh, pr, rope, slots, red, gq * NQG, min(NQG, nrows - gq * NQG), 0,
                                   ntiles, gq == ngroups - 1, gain);
  } else {
    for (int t = 0; t < ntiles && ok; ++t)
      for (int gq = 0; gq < ngroups && ok; ++gq)
        ok = gemv_dispatch<WT, KIND>(P, ca, l, G, sh, pr, rope, slots, red, gq * NQG, min(NQG, nrows - gq * NQG), t,
                                     t + 1, gq == ngroups - 1, gain);
  }
  if ((!ok || ngroups == 0) && threadIdx.x == 0) {
    // no copy may land after the CTA exits: wait (bounded) for the ones in flight
    for (int t = max(0, sh.issued - 2); t < sh.issued; ++t)
      mbar_wait_bounded(&sh.full[t & 1], (uint32_t)(t >> 1) & 1u, &P.ctl->status, P.wait_ns);
  }
}

// ------------------------------------------- small-batch tensor-core GEMV
// Contexts with bf16 weights and at most kMvMaxRows row slots (one stream at
// any verify window: the batch-1 path).  A GEMV there is a product of
// (output units) x (pass rows <= 8) x K whose cost is reading the weights
// once; after its dependency wait a kernel is limited by the latency of its
// arithmetic, so the weights are the M operand of mma.sync m16n8k16
// (bf16 x bf16 -> fp32) and the pass rows the N operand.  Each fp32 input x
// is split into bf16 hi = rn(x) and lo = rn(x - hi) (16 mantissa bits
// together); pass row r of a group of four takes column 2r (hi) and 2r + 1
// (lo), so one MMA covers four rows and the lane that holds C[u][2r] also
// holds C[u][2r + 1].
//
// A CTA owns a contiguous range of output units, cut into M-blocks of 16
// weight rows: 16 units, or 8 units x (first, second) row of a RoPE pair or
// a gate/up pair, so that both rows of a pair end in the same lane.  The
// TMA unit copies the weight rows into shared memory with one 1-D bulk copy
// per contiguous run of rows (a head of QKV or of the lm_heads, else the
// whole tile; first rows and second rows of pairs apart), because a copy
// costs about as much to issue as a few kilobytes take to land.  Inside
// each 32-element block of K a fixed permutation gives lane t the physical
// elements 8t..8t+7 on both operands, so a lane reads one 16-byte chunk of
// each of its two weight rows and two float4 of its input row per two MMAs.
// The input rows are bulk-copied into shared memory once per CTA.  The warps
// split K; within its slice a warp converts each input block once and runs
// it against every M-block of the phase.  The warps' partial sums meet in
// shared memory and the epilogue adds them in warp order.  Reduction orders
// depend on the model shape and the grid only, never on which rows share a
// pass.
//
// Tiles larger than the CTA's weight region stream in phases through two
// banks (phase p in bank p & 1); the first two phases are issued before the
// dependency wait, phase p + 2 once phase p is consumed.  Each kernel also
// prefetches into L2 the weight rows that the same CTA index of the GEMV two
// kernels ahead will copy, so HBM keeps streaming through the dependency
// waits of the chain.

struct MvBlock {
  int s0, s1;  // slot of A row 0 and of A row 8 (pair kinds: the second rows)
  int n, n2;   // valid A rows among 0..7 (n) and 8..15 (n2), counted from 0 and from 8
  int u;       // first unit
  int pad[3];
};

struct MvShared {
  uint64_t wbar[2];  // weight rows of the phase in bank 0 / 1
  uint64_t ibar;     // input rows
  int nblk, nphase, nrows, nheads, nbank, issued;
  int plan_w[2];     // plan words nrows, nheads as loaded
  int ph[kMvMaxPhases + 1];  // first block of each phase
  int heads[kMaxHeadsPerPass];
  int rbf[kMvMaxRows];       // input row held as bf16 (a code embedding of layer 0)
  float inv[kMvMaxRows];     // RMSNorm scale per pass row
  CallArgs ca;
  MvBlock blk[kMvMaxBlocks];
};

// Global address of weight row h (0, or 1 = the second row of a pair) of
// output unit u of a GEMV kind (bf16 weights).
__device__ __forceinline__ const unsigned char* mv_row_src(const FrameParams& P, int kind, int l, const int* heads,
                                                            int u, int h) {
  switch (kind) {
    case kQKV: {
      const int half = P.d / 2, hh = u / half, e = u - hh * half;
      const size_t rb = (size_t)P.H * 2;
      const unsigned char* base;
      if (hh < P.nq) base = static_cast<const unsigned char*>(P.wq[l]) + (size_t)hh * P.d * rb;
      else if (hh < P.nq + P.nkv) base = static_cast<const unsigned char*>(P.wk[l]) + (size_t)(hh - P.nq) * P.d * rb;
      else base = static_cast<const unsigned char*>(P.wv[l]) + (size_t)(hh - P.nq - P.nkv) * P.d * rb;
      return base + (size_t)(e + h * half) * rb;
    }
    case kO: return static_cast<const unsigned char*>(P.wo[l]) + (size_t)u * P.nq * P.d * 2;
    case kGU: return static_cast<const unsigned char*>(h ? P.w_up[l] : P.w_gate[l]) + (size_t)u * P.H * 2;
    case kDown: return static_cast<const unsigned char*>(P.w_down[l]) + (size_t)u * P.F * 2;
    default: {
      const int hi = u / P.V, v = u - hi * P.V;
      return static_cast<const unsigned char*>(P.head) + ((size_t)(heads[hi] - 1) * P.V + v) * P.H * 2;
    }
  }
}

__device__ __forceinline__ int mv_period(const FrameParams& P, int kind) {
  return kind == kQKV ? P.d / 2 : (kind == kHeads ? P.V : 0);
}

// Units [ua, ub) of CTA c of g for U units (U * g < 2^31: at most 64 heads of
// 8192 rows on a few hundred CTAs).
__device__ __forceinline__ void mv_range(int U, int c, int g, int* ua, int* ub) {
  *ua = (int)(((unsigned)U * (unsigned)c) / (unsigned)g);
  *ub = (int)(((unsigned)U * (unsigned)(c + 1)) / (unsigned)g);
}

// L2 prefetch of the weight rows CTA blockIdx.x of GEMV (kind, l) copies:
// one bulk prefetch per contiguous run.  Warp-wide.
__device__ void mv_prefetch_l2(const FrameParams& P, int kind, int l, const int* heads, int nheads) {
  const int lane = threadIdx.x & 31;
  const int U = gemv_units(P, kind, nheads);
  const int period = mv_period(P, kind);
  int ua, ub;
  mv_range(U, blockIdx.x, gridDim.x, &ua, &ub);
  const int rpu = rows_per_unit(kind);
  const uint32_t rowb = (uint32_t)gemv_K(P, kind) * 2u;
  int j = 0;
  for (int u = ua; u < ub;) {
    const int e = period > 0 ? min(ub, (u / period + 1) * period) : ub;
    for (int h = 0; h < rpu; ++h, ++j)
      if ((j & 31) == lane) prefetch_l2(mv_row_src(P, kind, l, heads, u, h), (uint32_t)(e - u) * rowb);
    u = e;
  }
}

// This CTA's units cut into M-blocks and phases (one thread): one phase
// when the whole tile fits the S row slots in at most kMvPhaseBlocks blocks,
// else phases alternating between two banks of S/2 slots.
__device__ void mv_build(const FrameParams& P, MvShared& sh, int S, int nheads, int kind) {
  const bool kPair = kind == kQKV || kind == kGU;
  const int rpu = kPair ? 2 : 1;
  const int U = gemv_units(P, kind, nheads);
  const int period = mv_period(P, kind);
  int ua, ub;
  mv_range(U, blockIdx.x, gridDim.x, &ua, &ub);
  int nb = 0, np = 0, nbank = 1;
  bool bad = false;
  for (int attempt = 0; attempt < 2; ++attempt) {
    nbank = attempt + 1;
    const int cap = nbank == 1 ? S : S / 2;  // row slots of a bank
    const int upb = max(1, min(kPair ? 8 : 16, cap / rpu));
    int used = 0, inph = 0;
    nb = 0;
    np = 0;
    bad = false;
    sh.ph[0] = 0;
    for (int u = ua; u < ub;) {
      int e = min(ub, u + upb);
      if (period > 0) e = min(e, (u / period + 1) * period);
      const int n = e - u, rows = n * rpu;
      if (used + rows > cap || inph == kMvPhaseBlocks) {
        if (nbank == 1 || np + 2 > kMvMaxPhases) { bad = true; break; }
        sh.ph[++np] = nb;
        used = 0;
        inph = 0;
      }
      if (nb >= kMvMaxBlocks) { bad = true; break; }
      MvBlock B;
      B.s0 = (nbank == 2 ? (np & 1) * cap : 0) + used / rpu;  // pair kinds: second rows placed below
      B.s1 = kPair ? 0 : B.s0 + 8;
      B.n = kPair ? n : min(n, 8);
      B.n2 = kPair ? n : max(0, n - 8);
      B.u = u;
      sh.blk[nb++] = B;
      used += rows;
      ++inph;
      u = e;
    }
    if (!bad) break;
  }
  // pair kinds: the first rows of a phase's units fill its slots in unit
  // order, the second rows follow them (so each contiguous run of units is
  // two bulk copies)
  if (kPair && !bad) {
    for (int p = 0; p <= np; ++p) {
      const int b0 = p == 0 ? 0 : sh.ph[p], b1 = p < np ? sh.ph[p + 1] : nb;
      int units = 0;
      for (int b = b0; b < b1; ++b) units += sh.blk[b].n;
      for (int b = b0; b < b1; ++b) sh.blk[b].s1 = sh.blk[b].s0 + units;
    }
  }
  if (bad) { raise_status(&P.ctl->status, kStatusDevice); nb = 0; }
  sh.ph[nb > 0 ? np + 1 : 0] = nb;
  sh.nphase = nb > 0 ? np + 1 : 0;
  sh.nblk = nb;
  sh.nbank = nbank;
}

// Issue the bulk copies of the weight rows of phase p into its bank.  Warp-wide.
__device__ void mv_issue_phase(const FrameParams& P, int l, MvShared& sh, unsigned char* wreg, int RS, int p, int kind) {
  const int rpu = (kind == kQKV || kind == kGU) ? 2 : 1;
  const int lane = threadIdx.x & 31;
  const int b0 = sh.ph[p], b1 = sh.ph[p + 1];
  const uint32_t rowb = (uint32_t)gemv_K(P, kind) * 2u;
  uint64_t* bar = &sh.wbar[p & 1];
  if (lane == 0) {
    uint32_t rows = 0;  // pair kinds: n units of two rows; otherwise n + n2 units of one row
    for (int b = b0; b < b1; ++b) rows += rpu == 2 ? 2u * (uint32_t)sh.blk[b].n : (uint32_t)(sh.blk[b].n + sh.blk[b].n2);
    mbar_arrive_expect_tx(bar, rows * rowb);
  }
  __syncwarp();
  const uint64_t pol = l2_evict_first_policy();
  // runs of blocks whose units are consecutive rows in global memory (one
  // head of QKV or of the lm_heads; the whole tile otherwise) and
  // consecutive slots: one bulk copy per run and row half, one lane each
  const int period = mv_period(P, kind);
  int j = 0;
  for (int b = b0; b < b1;) {
    int e = b + 1, nu = rpu == 2 ? sh.blk[b].n : sh.blk[b].n + sh.blk[b].n2;
    while (e < b1 && (period == 0 || sh.blk[e].u / period == sh.blk[b].u / period)) {
      nu += rpu == 2 ? sh.blk[e].n : sh.blk[e].n + sh.blk[e].n2;
      ++e;
    }
    for (int h = 0; h < rpu; ++h, ++j)
      if ((j & 31) == lane)
        bulk_copy_g2s(wreg + (size_t)(h ? sh.blk[b].s1 : sh.blk[b].s0) * RS,
                      mv_row_src(P, kind, l, sh.heads, sh.blk[b].u, h), rowb * (uint32_t)nu, bar, pol);
    b = e;
  }
  __syncwarp();
}

// bf16x2 of (x0, x1): the hi parts rn(x), or the lo parts rn(x - rn(x)).
__device__ __forceinline__ uint32_t mv_part(float x0, float x1, bool lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 o = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  const uint32_t hu = *reinterpret_cast<const uint32_t*>(&h), ou = *reinterpret_cast<const uint32_t*>(&o);
  return lo ? ou : hu;
}

// The MMAs of the blocks [b0, b1) of one phase (at most kMvPhaseBlocks):
// warp w takes K elements [w K/8, (w+1) K/8); per 32-element step it forms
// its B fragments once (input x gain, split hi or lo; NG groups of four pass
// rows) and runs them against every block.  The warp leaves its partial
// sums (hi + lo added) in
// red[(block - b0)][w][A row][pass row] and, with `do_ss`, the sums of
// squares of its K slice per pass row in s_ss.  Every order here depends on
// the tile (model shape and grid), not on the pass rows.
template <int NG>
__device__ __forceinline__ void mv_compute(const MvShared& sh, const unsigned char* wreg, int RS, const float* in,
                                           const float* gain, float* red, float* s_ss, int K, int RW, int b0, int b1,
                                           bool do_ss) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int KW = K / kWarps, k0 = warp * KW;
  const int nrows = sh.nrows;
  const bool lo = (g & 1) != 0;
  const int nbp = b1 - b0;
  uint32_t pa[kMvPhaseBlocks], pb[kMvPhaseBlocks];  // shared-memory addresses of this lane's A chunks
  bool va[kMvPhaseBlocks], vb[kMvPhaseBlocks];
  const uint32_t wbase = smem_u32(wreg);
#pragma unroll
  for (int j = 0; j < kMvPhaseBlocks; ++j) {
    const MvBlock B = sh.blk[b0 + min(j, nbp - 1)];
    va[j] = j < nbp && g < B.n;
    vb[j] = j < nbp && g < B.n2;
    pa[j] = wbase + (uint32_t)((B.s0 + g) * RS + t * 16 + k0 * 2);
    pb[j] = wbase + (uint32_t)((B.s1 + g) * RS + t * 16 + k0 * 2);
  }
  const float* rowp[NG];
  bool rv[NG], r16[NG];
#pragma unroll
  for (int q = 0; q < NG; ++q) {
    const int r = 4 * q + (g >> 1);
    rv[q] = r < nrows;
    r16[q] = rv[q] && sh.rbf[r] != 0;
    rowp[q] = in + (size_t)(rv[q] ? r : 0) * K;
  }
  float acc[kMvPhaseBlocks][NG][4];
  float ssq[NG];
#pragma unroll
  for (int j = 0; j < kMvPhaseBlocks; ++j)
#pragma unroll
    for (int q = 0; q < NG; ++q) acc[j][q][0] = acc[j][q][1] = acc[j][q][2] = acc[j][q][3] = 0.0f;
#pragma unroll
  for (int q = 0; q < NG; ++q) ssq[q] = 0.0f;
#pragma unroll 2
  for (int kk = 0; kk < KW; kk += 32) {
    const int k = k0 + kk + 8 * t;
    float gv[8];
    if (gain != nullptr) {
      const float4 g0 = *reinterpret_cast<const float4*>(gain + k);
      const float4 g1 = *reinterpret_cast<const float4*>(gain + k + 4);
      gv[0] = g0.x; gv[1] = g0.y; gv[2] = g0.z; gv[3] = g0.w; gv[4] = g1.x; gv[5] = g1.y; gv[6] = g1.z; gv[7] = g1.w;
    }
    uint32_t bp[NG][4];
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      float x[8];
      if (!rv[q]) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.0f;
      } else if (r16[q]) {
        const uint4 w = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(rowp[q]) + k);
        const float2 a = bf16x2_to_f2(w.x), b = bf16x2_to_f2(w.y), c = bf16x2_to_f2(w.z), d = bf16x2_to_f2(w.w);
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y; x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
      } else {
        const float4 a = *reinterpret_cast<const float4*>(rowp[q] + k), b = *reinterpret_cast<const float4*>(rowp[q] + k + 4);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      }
      if (do_ss && !lo) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ssq[q] = fmaf(x[e], x[e], ssq[q]);
      }
      if (gain != nullptr) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= gv[e];
      }
      bp[q][0] = mv_part(x[0], x[1], lo);
      bp[q][1] = mv_part(x[2], x[3], lo);
      bp[q][2] = mv_part(x[4], x[5], lo);
      bp[q][3] = mv_part(x[6], x[7], lo);
    }
#pragma unroll
    for (int j = 0; j < kMvPhaseBlocks; ++j) {
      if (j >= nbp) break;
      uint4 A0 = make_uint4(0u, 0u, 0u, 0u), A1 = make_uint4(0u, 0u, 0u, 0u);
      if (va[j]) asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(A0.x), "=r"(A0.y), "=r"(A0.z), "=r"(A0.w) : "r"(pa[j] + kk * 2));
      if (vb[j]) asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(A1.x), "=r"(A1.y), "=r"(A1.z), "=r"(A1.w) : "r"(pb[j] + kk * 2));
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        mma_bf16_16816(acc[j][q], A0.x, A1.x, A0.y, A1.y, bp[q][0], bp[q][1]);
        mma_bf16_16816(acc[j][q], A0.z, A1.z, A0.w, A1.w, bp[q][2], bp[q][3]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kMvPhaseBlocks; ++j) {
    if (j >= nbp) break;
    float* rb = red + (size_t)(j * kWarps + warp) * 16 * RW;
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      rb[g * RW + 4 * q + t] = acc[j][q][0] + acc[j][q][1];
      rb[(g + 8) * RW + 4 * q + t] = acc[j][q][2] + acc[j][q][3];
    }
  }
  if (do_ss) {
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      float v = ssq[q];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if (t == 0 && !lo) s_ss[warp * kMvMaxRows + 4 * q + (g >> 1)] = v;
    }
  }
}

// Shared-memory carve-up of the small-batch GEMV kernel (the host sizes the
// launch with the same arithmetic).
struct MvSmem {
  size_t w, in, gain, red, ss, rows, rope, total;
};
__host__ __device__ inline MvSmem mv_smem_layout(int kind, int S, int K, int rows_cap, int G, int d) {
  MvSmem o;
  size_t off = 0;
  const size_t RS = (size_t)K * 2 + kMvRowPad;
  o.w = off; off += (size_t)S * RS;
  o.in = off; off += (size_t)rows_cap * K * 4;
  o.gain = off; off += (kind == kQKV || kind == kGU || kind == kHeads) ? (size_t)K * 4 : 0;
  const int RW = 4 * ((rows_cap + 3) / 4);
  o.red = off; off += (size_t)kMvPhaseBlocks * kWarps * 16 * RW * 4;
  o.ss = off; off += (size_t)kWarps * kMvMaxRows * 4;
  o.rows = off; off += (size_t)((3 * rows_cap + 3) / 4 * 4) * 4;
  o.rope = off; off += kind == kQKV && (size_t)G * (d / 2) * 8 <= (size_t)kRopeSmemBytes ? (size_t)kRopeSmemBytes : 0;
  o.total = off;
  return o;
}

// Kind two GEMVs ahead in the pass (QKV, O, GU, down per layer, then the
// lm_heads), wrapping to the next pass.
__device__ __forceinline__ void mv_ahead(const FrameParams& P, int kind, int l, int* kind2, int* l2) {
  switch (kind) {
    case kQKV: *kind2 = kGU; *l2 = l; break;
    case kO: *kind2 = kDown; *l2 = l; break;
    case kGU: if (l + 1 < P.L) { *kind2 = kQKV; *l2 = l + 1; } else { *kind2 = kHeads; *l2 = 0; } break;
    case kDown: if (l + 1 < P.L) { *kind2 = kO; *l2 = l + 1; } else { *kind2 = kQKV; *l2 = 0; } break;
    default: *kind2 = kO; *l2 = 0;
  }
}

// One GEMV of the pass (lk = 8 * layer + kind; the kind is also the template
// argument, so each kind compiles to straight-line code of its own).
template <int KIND>
__global__ void __launch_bounds__(kThreads, 2) mv_kernel(const __grid_constant__ FrameParams P, int lk) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  __shared__ MvShared sh;
  const int l = lk >> 3;
  constexpr bool kPair = KIND == kQKV || KIND == kGU;
  constexpr bool kNormed = KIND == kQKV || KIND == kGU || KIND == kHeads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = gemv_K(P, KIND);
  const int RS = K * 2 + kMvRowPad;
  const int S = P.mv_slots[KIND];
  const int rows_cap = P.Bmax * P.NS;
  const MvSmem L = mv_smem_layout(KIND, S, K, rows_cap, P.G, P.d);
  unsigned char* wreg = smem + L.w;
  float* in = reinterpret_cast<float*>(smem + L.in);
  float* s_gain = reinterpret_cast<float*>(smem + L.gain);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* s_ss = reinterpret_cast<float*>(smem + L.ss);
  int* s_rows = reinterpret_cast<int*>(smem + L.rows);
  float2* s_rope = reinterpret_cast<float2*>(smem + L.rope);
  const int RW = 4 * ((rows_cap + 3) / 4);
  PassRows pr{s_rows, s_rows + rows_cap, s_rows + 2 * rows_cap};
  const size_t rope_n = (size_t)P.G * (P.d / 2);
  const bool rope_in_smem = KIND == kQKV && rope_n * sizeof(float2) <= (size_t)kRopeSmemBytes;
  const float* gain_g = KIND == kQKV ? P.attn_norm[l] : (KIND == kGU ? P.ffn_norm[l] : (KIND == kHeads ? P.final_norm : nullptr));
  const bool inputs_early = KIND == kQKV && l == 0;  // call inputs and embeddings: not written inside the pass
  const bool need_heads = KIND == kHeads || (KIND == kGU && l == P.L - 1);

  // ---------------- before the dependency wait: what no kernel of the pass writes
  // (1) the weight tile: its shape depends on the model and the grid only
  //     (the lm_heads also on the pass's heads, loaded first)
  if (KIND != kHeads && warp == 0) {
    if (lane == 0) {
      mbar_init(&sh.wbar[0], 1);
      mbar_init(&sh.wbar[1], 1);
      mbar_init(&sh.ibar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      mv_build(P, sh, S, 0, KIND);
    }
    __syncwarp();
    for (int p = 0; p < min(sh.nphase, sh.nbank); ++p) mv_issue_phase(P, l, sh, wreg, RS, p, KIND);
    if (lane == 0) sh.issued = min(sh.nphase, sh.nbank);
  }
  // (2) every thread: the plan words, pass rows, call arguments, RoPE table
  //     and norm gain, all loads in flight at once
  if (tid < 2) sh.plan_w[tid] = __ldcg(tid == 0 ? &P.plan->nrows : &P.plan->nheads);
  if (need_heads && tid >= 32 && tid < 32 + kMaxHeadsPerPass) sh.heads[tid - 32] = __ldcg(&P.plan->heads[tid - 32]);
  if (tid >= 96 && tid < 96 + 3 * rows_cap) {
    const int a = (tid - 96) / rows_cap, i = (tid - 96) - a * rows_cap;
    s_rows[a * rows_cap + i] = __ldcg((a == 0 ? P.prow : (a == 1 ? P.ppos : P.pcode)) + i);
  }
  if (tid >= 128 && tid < 128 + (int)(sizeof(CallArgs) / 4))
    reinterpret_cast<int*>(&sh.ca)[tid - 128] = __ldcg(reinterpret_cast<const int*>(P.call) + (tid - 128));
  // RoPE table and norm gain: asynchronous 16-byte copies, all in flight at once
  if (rope_in_smem)
    for (int i = tid; i < (int)(rope_n / 2); i += kThreads) cp_async16(s_rope + 2 * i, P.rope + 2 * i);
  if (gain_g != nullptr)
    for (int i = tid; i < K / 4; i += kThreads) cp_async16(s_gain + 4 * i, gain_g + 4 * i);
  cp_async_wait_all();
  __syncthreads();
  const int nrows = min(sh.plan_w[0], rows_cap);
  if (warp == 0) {
    if (lane == 0) {
      sh.nrows = nrows;
      sh.nheads = need_heads ? min(sh.plan_w[1], kMaxHeadsPerPass) : 0;
      for (int r = 0; r < kMvMaxRows; ++r) sh.rbf[r] = (inputs_early && r < nrows && pr.ppos[r] > 0) ? 1 : 0;
      if (KIND == kHeads) {
        mbar_init(&sh.wbar[0], 1);
        mbar_init(&sh.wbar[1], 1);
        mbar_init(&sh.ibar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mv_build(P, sh, S, sh.nheads, KIND);
      }
    }
    __syncwarp();
    if (KIND == kHeads) {
      for (int p = 0; p < min(sh.nphase, sh.nbank); ++p) mv_issue_phase(P, l, sh, wreg, RS, p, KIND);
      if (lane == 0) sh.issued = min(sh.nphase, sh.nbank);
    }
    // input rows of layer 0 (x and code embeddings), one bulk copy each
    if (inputs_early) {
      if (lane == 0) {
        uint32_t bytes = 0;
        for (int r = 0; r < nrows; ++r) bytes += (uint32_t)K * (sh.rbf[r] ? 2u : 4u);
        if (P.test_stall && blockIdx.x == 0) bytes += 16u;  // test hook: never completes
        mbar_arrive_expect_tx(&sh.ibar, bytes);
      }
      __syncwarp();
      if (lane < nrows) {
        const ActRow a = act_row<__nv_bfloat16>(P, sh.ca, pr, KIND, l, lane);
        const void* src = a.f != nullptr ? static_cast<const void*>(a.f) : a.w;
        bulk_copy_g2s_plain(in + (size_t)lane * K, src, (uint32_t)K * (sh.rbf[lane] ? 2u : 4u), &sh.ibar);
      }
    }
    // L2 prefetch for the GEMV two kernels ahead
    int k2, l2;
    mv_ahead(P, KIND, l, &k2, &l2);
    mv_prefetch_l2(P, k2, l2, sh.heads, k2 == kHeads ? sh.nheads : 0);
  }
  pdl_wait();
  // input rows written by the previous kernels of the pass: 16-byte
  // asynchronous copies by every thread, all in flight at once
  if (!inputs_early) {
    const int k4 = K / 4;
    for (int idx = tid; idx < nrows * k4; idx += kThreads) {
      const int r = idx / k4, c = idx - r * k4;
      cp_async16(in + (size_t)r * K + 4 * c, act_row<__nv_bfloat16>(P, sh.ca, pr, KIND, l, r).f + 4 * c);
    }
    cp_async_wait_all();
  }
  __syncthreads();  // sh.nrows, sh.rbf, the tile of the lm_heads, the input rows
  const float2* rope = rope_in_smem ? s_rope : P.rope;
  const float* gain = kNormed ? s_gain : nullptr;
  // residual values the first phase's epilogue adds to (O, down), fetched now
  float hold[2] = {0.0f, 0.0f};
  if ((KIND == kO || KIND == kDown) && sh.nphase > 0 && nrows > 0) {
    int it = tid;
#pragma unroll
    for (int m = 0; m < 2; ++m, it += kThreads) {
      int rem = it;
      for (int b = sh.ph[0]; b < sh.ph[1]; ++b) {
        const int nu = sh.blk[b].n + sh.blk[b].n2, cnt = nu * nrows;
        if (rem < cnt) {
          const int i = rem / nrows, r = rem - i * nrows;
          hold[m] = __ldcg(P.h + (size_t)pr.prow[r] * P.H + sh.blk[b].u + i);
          break;
        }
        rem -= cnt;
      }
    }
  }
  bool ok = !inputs_early || mbar_wait_bounded(&sh.ibar, 0, &P.ctl->status, P.wait_ns);
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  int waited = 0;  // phases whose barrier has completed
  if (ok && KIND == kQKV && l == 0) {
    // the residual stream starts as the input rows: this CTA's slice of H
    const int c0 = (int)(((long long)P.H * blockIdx.x) / gridDim.x), c1 = (int)(((long long)P.H * (blockIdx.x + 1)) / gridDim.x);
    const int w = c1 - c0;
    for (int it = tid; it < nrows * w; it += kThreads) {
      const int i = it / w, k = c0 + (it - i * w);
      const float v = sh.rbf[i] ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(in + (size_t)i * K)[k])
                                : in[(size_t)i * K + k];
      P.h[(size_t)pr.prow[i] * P.H + k] = v;
    }
  }
  for (int p = 0; p < sh.nphase && ok; ++p) {
    if (!mbar_wait_bounded(&sh.wbar[p & 1], (uint32_t)(p >> 1) & 1u, &P.ctl->status, P.wait_ns)) ok = false;
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (!ok) break;
    waited = p + 1;
    const int b0 = sh.ph[p], b1 = sh.ph[p + 1];
    if (nrows > 4) mv_compute<2>(sh, wreg, RS, in, gain, red, s_ss, K, RW, b0, b1, kNormed && p == 0);
    else mv_compute<1>(sh, wreg, RS, in, gain, red, s_ss, K, RW, b0, b1, kNormed && p == 0);
    __syncthreads();
    if (kNormed && p == 0) {
      if (tid < nrows) {
        float ts = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) ts += s_ss[w * kMvMaxRows + tid];
        sh.inv[tid] = rsqrtf(ts / (float)K + P.eps);
      }
      __syncthreads();
    }
    // epilogue: per (unit, pass row), the warps' partial sums in warp order
    int it = tid;
    for (int m = 0;; ++m, it += kThreads) {
      int rem = it, b = b0;
      for (; b < b1; ++b) {
        const int nu = kPair ? sh.blk[b].n : sh.blk[b].n + sh.blk[b].n2, cnt = nu * nrows;
        if (rem < cnt) break;
        rem -= cnt;
      }
      if (b >= b1) break;
      const MvBlock B = sh.blk[b];
      const int i = rem / nrows, r = rem - i * nrows;
      const float* rbase = red + (size_t)(b - b0) * kWarps * 16 * RW;
      float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        y0 += rbase[((size_t)w * 16 + i) * RW + r];
        if (kPair) y1 += rbase[((size_t)w * 16 + i + 8) * RW + r];
      }
      if (kNormed) {
        y0 *= sh.inv[r];
        y1 *= sh.inv[r];
      }
      float ho = 0.0f;
      if (KIND == kO || KIND == kDown) {
        if (p == 0 && m < 2) ho = m == 0 ? hold[0] : hold[1];
        else ho = __ldcg(P.h + (size_t)pr.prow[r] * P.H + B.u + i);
      }
      gemv_out<KIND>(P, l, sh.heads, pr, rope, B.u + i, r, y0, y1, ho);
    }
    __syncthreads();  // the partial sums and this phase's bank are free
    if (warp == 0 && sh.nbank == 2 && p + 2 < sh.nphase) {
      mv_issue_phase(P, l, sh, wreg, RS, p + 2, KIND);
      if (lane == 0) sh.issued = p + 3;
    }
  }
  if (!ok && tid == 0) {
    // no copy may land after the CTA exits: wait (bounded) for every one in flight
    for (int q = waited; q < sh.issued; ++q)
      mbar_wait_bounded(&sh.wbar[q & 1], (uint32_t)(q >> 1) & 1u, &P.ctl->status, P.wait_ns);
    if (inputs_early) mbar_wait_bounded(&sh.ibar, 0, &P.ctl->status, P.wait_ns);
  }
}

#include "cp_t5.cuh"

// ------------------------------------------------------------- attention
// Causal GQA attention of one pass row over its keys in the stream's KV
// cache (this pass's rows were appended by the QKV kernel), one CTA per
// (pass row, KV group).  The keys of a chain row at position pos are the
// canonical positions 0..pos.  A tree node's row ("RVQ Position Aware
// Speculative Decoding for On Device TTS", section 2.2, sparse tree
// attention) sees the canonical positions 0..base (the committed prefix and
// the round's root row, base = pos - depth) and then the slots of its
// ancestors and of itself, in node order, which along one path is position
// order.  The row's plan entry is read before the dependency wait; after it
// the group's K and V rows of the keys and the group's queries are staged in
// shared memory by one round of asynchronous 16-byte copies.  Then one warp
// per query head: lane j scores key j (and j + 32), the dot product over the
// head dimensions taken in 4-element chunks starting at the lane's own chunk
// (so the lanes of a quarter warp read distinct banks), a fixed order per
// key; the weights exp(s_j - max) / den with den the warp's butterfly sum;
// then each output pair sums the weighted value rows in key order.  Every
// order depends on the keys and the head shape only, never on the other rows
// of the pass.
constexpr int kAttnThreads = 128;
__global__ void __launch_bounds__(kAttnThreads) attention_kernel(const __grid_constant__ FrameParams P, int l) {
  extern __shared__ __align__(16) float asmem[];
  pdl_launch_dependents();
  const int i = blockIdx.x / P.nkv, g = blockIdx.x - i * P.nkv;
  const int nrows = __ldcg(&P.plan->nrows);  // written before the pass starts
  if (i >= nrows) return;
  const int r = __ldcg(P.prow + i), b = r / P.NS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = kAttnThreads / 32;
  const int d = P.d, grp = P.nq / P.nkv, d4 = d / 4, lines = d / 2;
  // keys: canonical 0..base, then (tree node rows) the ancestor-or-self slots
  int base = __ldcg(P.ppos + i);
  unsigned long long anc = 0;
  if (P.tree_n) {
    const int slot = __ldcg(P.pslot + i);
    if (slot >= P.G) {
      const int node = slot - P.G;
      base -= __ldg(&P.tree->dep[node]);
      anc = __ldg(&P.tree->anc[node]);
    }
  }
  const int np = base + 1 + __popcll(anc);
  const int pos = np - 1;                  // index of the last key (the row itself)
  float* ks = asmem;                       // [np][d]
  float* vs = ks + (size_t)P.G * d;        // [np][d]
  float* qs = vs + (size_t)P.G * d;        // [grp][d]
  float* ws = qs + (size_t)grp * d;        // [nw][64] softmax weights
  const size_t pstride = (size_t)P.nkv * d;
  const float* kb = P.kv + ((((size_t)b * P.L + l) * 2 + 0) * P.GS) * pstride + (size_t)g * d;
  const float* vb = kb + (size_t)P.GS * pstride;
  const float* qb = P.qbuf + (size_t)r * P.nq * d + (size_t)g * grp * d;
  pdl_wait();
  for (int idx = tid; idx < np * d4; idx += kAttnThreads) {
    const int j = idx / d4, c = idx - j * d4;
    // key j's KV slot: j itself up to base, then the (j - base - 1)-th set bit of anc
    int sj = j;
    if (j > base) {
      unsigned long long m = anc;
      for (int q = j - base - 1; q > 0; --q) m &= m - 1;
      sj = P.G + __ffsll((long long)m) - 1;
    }
    cp_async16(ks + (size_t)j * d + 4 * c, kb + (size_t)sj * pstride + 4 * c);
    cp_async16(vs + (size_t)j * d + 4 * c, vb + (size_t)sj * pstride + 4 * c);
  }
  for (int idx = tid; idx < grp * d4; idx += kAttnThreads) cp_async16(qs + 4 * idx, qb + 4 * idx);
  cp_async_wait_all();
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)d);
  float* w = ws + warp * CP_SPEC_MAX_CODE_GROUPS;
  for (int hh = warp; hh < grp; hh += nw) {
    const float* q = qs + (size_t)hh * d;
    float sj[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int j = lane + 32 * h2;
      if (j > pos) continue;
      const float* kj = ks + (size_t)j * d;
      const int c0 = lane % d4;
      float acc = 0.0f;
      for (int cc = 0; cc < d4; ++cc) {
        const int c = c0 + cc < d4 ? c0 + cc : c0 + cc - d4;
        const float4 kv4 = *reinterpret_cast<const float4*>(kj + 4 * c);
        const float4 q4 = *reinterpret_cast<const float4*>(q + 4 * c);
        acc = fmaf(q4.x, kv4.x, acc);
        acc = fmaf(q4.y, kv4.y, acc);
        acc = fmaf(q4.z, kv4.z, acc);
        acc = fmaf(q4.w, kv4.w, acc);
      }
      sj[h2] = acc * scale;
    }
    const float mx = warp_max(fmaxf(sj[0], sj[1]));
    const float e0 = lane <= pos ? expf(sj[0] - mx) : 0.0f;
    const float e1 = lane + 32 <= pos ? expf(sj[1] - mx) : 0.0f;
    const float den = warp_sum(e0 + e1);
    if (lane <= pos) w[lane] = e0 / den;
    if (lane + 32 <= pos) w[lane + 32] = e1 / den;
    __syncwarp();
    float2 o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) o[u] = make_float2(0.f, 0.f);
    for (int j = 0; j <= pos; ++j) {
      const float wj = w[j];
      const float2* vj = reinterpret_cast<const float2*>(vs + (size_t)j * d);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int ln = lane + 32 * u;
        if (ln >= lines) continue;
        const float2 v = vj[ln];
        o[u].x = fmaf(wj, v.x, o[u].x);
        o[u].y = fmaf(wj, v.y, o[u].y);
      }
    }
    float2* dst = reinterpret_cast<float2*>(P.abuf + (size_t)r * P.nq * d + (size_t)(g * grp + hh) * d);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int ln = lane + 32 * u;
      if (ln < lines) dst[ln] = o[u];
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ top-k
// One vocabulary row (in shared memory as floats in `keys` on entry)
// processed by the CTA, with the semantics of the oracle's processing:
// z = fl32(logit/T), exactly min(k, V) entries kept by (z desc, index asc),
// e = cp_expf(z - zmax), S = float32 sum of e in ascending index order,
// p = fl32(e / S); T = 0 is argmax (lowest index).  Thread t owns indices
// [t*E, t*E + E).  The k-th key is found by an MSB-first 8-bit radix select
// over warp-private histograms (shared-memory atomic increments); one scan
// of packed (greater, equal) counts places every kept entry in index order.  Scratch: hw [kWarps][256], ebuf [min(k, V)],
// sx [64].  Returns the length.
__device__ __noinline__ int block_topk(int V, int k, float T, uint32_t* keys, uint32_t* hw, float* ebuf, int* sx,
                                       int* out_idx, float* out_prob) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = reinterpret_cast<const float*>(keys);
  const int E = (V + kThreads - 1) / kThreads;
  const int i0 = tid * E, i1 = min(V, i0 + E);
  if (T == 0.0f) {
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = i0; i < i1; ++i)
      if (row[i] > best) { best = row[i]; bi = i; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    float* sbest = reinterpret_cast<float*>(sx);
    int* sbi = sx + 16;
    if (lane == 0) { sbest[warp] = best; sbi[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
      float bb = sbest[0];
      int ix = sbi[0];
      for (int w = 1; w < kWarps; ++w)
        if (sbest[w] > bb || (sbest[w] == bb && sbi[w] < ix)) { bb = sbest[w]; ix = sbi[w]; }
      out_idx[0] = ix;
      out_prob[0] = 1.0f;
    }
    __syncthreads();
    return 1;
  }
  // keys (in place) and the maximum key
  uint32_t kmax = 0;
  for (int i = i0; i < i1; ++i) {
    float z = __fdiv_rn(row[i], T);
    if (z == 0.0f) z = 0.0f;
    const uint32_t key = float_key(z);
    keys[i] = key;
    kmax = max(kmax, key);
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) sx[warp] = (int)kmax;
  __syncthreads();
  kmax = 0;
  for (int w = 0; w < kWarps; ++w) kmax = max(kmax, (uint32_t)sx[w]);
  const int kk = k < V ? k : V;
  uint32_t prefix = 0, mask = 0;
  int need = kk;
  bool eq_all = (kk == V);
  uint32_t* my = hw + warp * 256;
  for (int shift = 24; shift >= 0 && !eq_all; shift -= 8) {
    // warp-private histogram (shared-memory atomics; integer counts, so the
    // result does not depend on their order)
#pragma unroll
    for (int j = 0; j < 8; ++j) my[lane * 8 + j] = 0;
    __syncwarp();
    for (int e = 0; e < E; ++e) {
      const int i = i0 + e;
      if (i < i1) {
        const uint32_t key = keys[i];
        if ((key & mask) == prefix) atomicAdd(&my[(key >> shift) & 255u], 1u);
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255-8l .. 248-8l (descending), summed over the warps
      uint32_t cnt[8], chunk = 0;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int bb = 255 - 8 * lane - m;
        uint32_t c = 0;
        for (int w = 0; w < kWarps; ++w) c += hw[w * 256 + bb];
        cnt[m] = c;
        chunk += c;
      }
      uint32_t incl = chunk;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - chunk;
      if (excl < (uint32_t)need && (uint32_t)need <= incl) {
        uint32_t acc = excl;
        for (int m = 0; m < 8; ++m) {
          if (acc + cnt[m] >= (uint32_t)need) { sx[32] = 255 - 8 * lane - m; sx[33] = (int)acc; sx[34] = (int)cnt[m]; break; }
          acc += cnt[m];
        }
      }
    }
    __syncthreads();
    const uint32_t bin = (uint32_t)sx[32], above = (uint32_t)sx[33], cbin = (uint32_t)sx[34];
    need -= (int)above;
    prefix |= bin << shift;
    mask |= 0xFFu << shift;
    if ((int)cbin == need) eq_all = true;
  }
  // one scan of packed counts (greater | equal << 16), index order
  int n_gt = 0, n_eq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t km = keys[i] & mask;
    n_gt += km > prefix;
    n_eq += km == prefix;
  }
  const int packed = n_gt | (n_eq << 16);
  int incl = packed;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sx[40 + warp] = incl;
  __syncthreads();
  int before = incl - packed;
  for (int w = 0; w < warp; ++w) before += sx[40 + w];
  int gb = before & 0xFFFF, eb = before >> 16;
  const float zmax = key_float(kmax);
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = keys[i];
    const uint32_t km = key & mask;
    int pos = -1;
    if (km > prefix) { pos = gb + min(eb, need); ++gb; }
    else if (km == prefix) { if (eq_all || eb < need) pos = gb + eb; ++eb; }
    if (pos >= 0) { out_idx[pos] = i; ebuf[pos] = cp_expf(__fsub_rn(key_float(key), zmax)); }
  }
  __syncthreads();
  if (tid == 0) {
    float S = 0.0f;
    for (int p = 0; p < kk; ++p) S = __fadd_rn(S, ebuf[p]);
    reinterpret_cast<float*>(sx)[48] = S;
  }
  __syncthreads();
  const float S = reinterpret_cast<float*>(sx)[48];
  for (int p = tid; p < kk; p += kThreads) out_prob[p] = __fdiv_rn(ebuf[p], S);
  __syncthreads();
  return kk;
}

// Top-k / temperature / softmax of one (pass row, logit slot) per CTA (slot
// t of the row at position pos holds head pos + t; slots past the last code
// group are unused).  Decode mode only.
__global__ void __launch_bounds__(kThreads, 2) topk_kernel(const __grid_constant__ FrameParams P) {
  extern __shared__ __align__(16) unsigned char tsmem[];
  pdl_launch_dependents();
  pdl_wait();
  if (P.call->mode != kModeDecode) return;
  const int slots = 1 + P.ND;
  const int nrows = __ldcg(&P.plan->nrows);
  const int i = blockIdx.x / slots, t = blockIdx.x - i * slots;
  if (i >= nrows) return;
  const int pos = __ldcg(P.ppos + i);
  if (pos < 1 || pos + t > P.G - 1) return;
  const int r = __ldcg(P.prow + i), b = r / P.NS;
  const size_t keys_bytes = ((size_t)P.V * 4 + 15) / 16 * 16;
  uint32_t* keys = reinterpret_cast<uint32_t*>(tsmem);
  uint32_t* hw = reinterpret_cast<uint32_t*>(tsmem + keys_bytes);
  float* ebuf = reinterpret_cast<float*>(tsmem + keys_bytes + kWarps * 1024);
  int* sx = reinterpret_cast<int*>(tsmem + keys_bytes + kWarps * 1024 + ((size_t)P.KC * 4 + 15) / 16 * 16);
  const size_t li = (size_t)r * slots + t;
  const float* src = P.logits + li * P.V;
  if ((P.V & 3) == 0) {
    for (int v = threadIdx.x; v < P.V / 4; v += kThreads)
      reinterpret_cast<float4*>(keys)[v] = __ldcg(reinterpret_cast<const float4*>(src) + v);
  } else {
    for (int v = threadIdx.x; v < P.V; v += kThreads) reinterpret_cast<float*>(keys)[v] = __ldcg(src + v);
  }
  __syncthreads();
  // tree rounds: a draft slot keeps the need[t] largest raw logits (candidate
  // ranks do not depend on the temperature; T = 1 leaves z = logit exactly)
  const bool rank_slot = P.tree_n > 0 && t > 0;
  const int kk = rank_slot ? __ldg(&P.tree->need[t]) : __ldg(P.top_k + b);
  const float TT = rank_slot ? 1.0f : __ldg(P.temp + b);
  const int n = block_topk(P.V, kk, TT, keys, hw, ebuf, sx, P.lidx + li * P.KC, P.lprob + li * P.KC);
  if (threadIdx.x == 0) P.lcount[li] = n;
}

// ------------------------------------------------------ per-stream logic
// One warp owns one stream in the setup and accept kernels.
__device__ __forceinline__ int valid_code(const FrameParams& P, int c) {
  if (c < 0 || c >= P.V) { raise_status(&P.ctl->status, kStatusDevice); return 0; }
  return c;
}

// When the setup or accept kernel runs as a single CTA, the rows it records
// are mirrored in shared memory so that its plan is built without a round
// trip through L2.
constexpr int kMirrorRows = 64;
__shared__ int g_mirror_on;
__shared__ int g_mpos[kMirrorRows];
__shared__ int g_mcode[kMirrorRows];
__shared__ int g_mslot[kMirrorRows];

__device__ __forceinline__ void mirror_init(const FrameParams& P, const CallArgs& ca) {
  if (threadIdx.x == 0) g_mirror_on = (gridDim.x == 1 && ca.B * P.NS <= kMirrorRows) ? 1 : 0;
  for (int i = threadIdx.x; i < kMirrorRows; i += blockDim.x) { g_mpos[i] = -1; g_mcode[i] = 0; g_mslot[i] = 0; }
  __syncthreads();
}

// Record the rows of stream b's next pass (state already updated in S):
// positions pos0.. and the code whose embedding each row carries (the frame
// index for the x row at position 0).  Warp-wide.
template <typename WT>
__device__ __noinline__ void set_pass_rows(const FrameParams& P, int b, const StreamState& S, const int* codes_in) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  for (int k = lane; k < P.NS; k += 32) {  // rows at consecutive positions from pos0, KV slot = position
    const int on = k < S.m;
    P.row_pos[b * P.NS + k] = on ? S.pos0 + k : -1;
    P.row_code[b * P.NS + k] = on ? codes_in[k] : 0;
    P.row_slot[b * P.NS + k] = on ? S.pos0 + k : 0;
    if (g_mirror_on) {
      g_mpos[b * P.NS + k] = on ? S.pos0 + k : -1;
      g_mcode[b * P.NS + k] = on ? codes_in[k] : 0;
      g_mslot[b * P.NS + k] = on ? S.pos0 + k : 0;
    }
  }
  if (lane == 0) {
    const long long kvb = (long long)(S.pos0 + S.m) * P.L * 2 * P.nkv * P.d * (long long)sizeof(float);
    atomicAdd((unsigned long long*)&P.ctl->kv_bytes, (unsigned long long)kvb);
    atomicAdd((unsigned long long*)&P.ctl->weight_bytes, (unsigned long long)((long long)S.m * P.H * sizeof(WT)));
  }
  __syncwarp();
}

__device__ __forceinline__ void retire_stream(const FrameParams& P, int b, StreamState& S) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane == 0) {
    S.phase = kPhaseDone;
    S.m = 0;
    for (int i = 0; i < P.NS; ++i) P.row_pos[b * P.NS + i] = -1;
    if (g_mirror_on)
      for (int i = 0; i < P.NS; ++i) g_mpos[b * P.NS + i] = -1;
    atomicSub(&P.ctl->active, 1);
  }
  __syncwarp();
}

// Frame start: rows [x, E_0(c_0)] at positions 0, 1.  Scalar state fields
// are written by lane 0 only; every all-lane read of them follows a __syncwarp().
// Verify window of a stream's next frame ("Speculative Decoding, Beyond
// Text", runtime policies: size the window from measured acceptance by
// offset, stop drafting when it collapses): offsets t = 1, 2, ... are kept
// while each has fewer than adapt_min reached drafts in this call or
// accepted at least adapt_pct percent of them; the window is 1 + the kept
// leading offsets.  Window 1 runs rounds without drafts (one row per pass,
// each code drawn from the target).  It depends only on earlier frames, so
// every frame keeps the autoregressive law.
__device__ __forceinline__ int frame_window(const FrameParams& P, const StreamState& S) {
  if (P.N < 2 || P.adapt_pct <= 0) return P.N;
  int w = 1;
  for (int t = 1; t <= P.N - 1; ++t) {
    const int r = S.reach[t - 1], a = S.acc[t - 1];
    const bool keep = r < P.adapt_min || 100ll * a >= (long long)P.adapt_pct * r;
    if (!keep) break;
    w = t + 1;
  }
  return w;
}

template <typename WT>
__device__ __noinline__ void setup_frame(const FrameParams& P, const CallArgs& ca, int b, StreamState& S, int frame) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane == 0) {
    const int c0 = valid_code(P, __ldg(ca.c0 + (size_t)frame * ca.B + b));
    S.frame = frame;
    S.frame_abs = ca.first_frame + frame;
    S.codes[0] = c0;
    S.s = 0;
    S.phase = kPhasePrefill;
    S.pos0 = 0;
    S.m = 2;
    S.n_d = 0;
    S.w = frame_window(P, S);
    ca.codes_out[((size_t)frame * ca.B + b) * P.G] = c0;
    if (ca.committed_out) ca.committed_out[b] = 1;
  }
  __syncwarp();
  const int codes_in[2] = {frame, S.codes[0]};
  set_pass_rows<WT>(P, b, S, codes_in);
}

template <typename WT>
__device__ __noinline__ void setup_teacher_chunk(const FrameParams& P, const CallArgs& ca, int b, StreamState& S) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  const int pos0 = S.pos0;
  const int m = min(P.NS, ca.P - pos0);
  __syncwarp();
  if (lane == 0) { S.m = m; S.phase = kPhaseTeacher; }
  __syncwarp();
  int codes_in[CP_SPEC_MAX_WINDOW];
  for (int i = 0; i < m; ++i) {
    const int pos = pos0 + i;
    codes_in[i] = pos > 0 ? valid_code(P, __ldg(ca.t_codes + (size_t)b * (ca.P - 1) + pos - 1)) : 0;
  }
  set_pass_rows<WT>(P, b, S, codes_in);
}

__device__ __forceinline__ void load_state(const FrameParams& P, int b, StreamState& S) {
  const int lane = threadIdx.x & 31;
  const int* src = reinterpret_cast<const int*>(P.st + b);
  int* dst = reinterpret_cast<int*>(&S);
  for (int i = lane; i < (int)(sizeof(StreamState) / 4); i += 32) dst[i] = __ldcg(src + i);
  __syncwarp();
}

__device__ __forceinline__ void store_state(const FrameParams& P, int b, const StreamState& S) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  int* dst = reinterpret_cast<int*>(P.st + b);
  const int* src = reinterpret_cast<const int*>(&S);
  for (int i = lane; i < (int)(sizeof(StreamState) / 4); i += 32) dst[i] = src[i];
  __syncwarp();
}

// Counter increment that does not wait for the old value (a reduction in
// L2): the accept path never reads its counters back.
__device__ __forceinline__ void bump(long long& c, long long v = 1) {
  atomicAdd(reinterpret_cast<unsigned long long*>(&c), (unsigned long long)v);
}

// Per-warp view of the accept scratch (see accept_scratch_bytes).  List
// slots: target list of row i of the stream at i (i < NS), saved draft list
// q_t at NS + t - 1, draft slot t of row i at NS + NDr + i * NDr + t - 1.
struct AcceptScratch {
  StreamState* S;
  int* idx;    // [lists][KC]
  float* prob; // [lists][KC]
  int* cnt;    // [lists]
  float* r;    // [KC] residual weights
  float* u;    // [32] Philox uniforms of the decision
  int NS, NDr;
  __device__ __forceinline__ int tslot(int i) const { return i; }
  __device__ __forceinline__ int qslot(int t) const { return NS + t - 1; }
  __device__ __forceinline__ int dslot(int i, int t) const { return NS + NDr + i * NDr + t - 1; }
};

__device__ __forceinline__ AcceptScratch accept_scratch(const FrameParams& P, unsigned char* base_all) {
  const int warp = threadIdx.x >> 5;
  const int NSr = accept_rows(P.NS, P.tree_n), NDr = accept_drafts(P.NS, P.ND, P.tree_n);
  const int n = accept_lists(NSr, NDr);
  unsigned char* base = base_all + (size_t)warp * accept_scratch_bytes(NSr, NDr, P.KC);
  AcceptScratch a;
  a.S = reinterpret_cast<StreamState*>(base);
  a.idx = reinterpret_cast<int*>(base + sizeof(StreamState));
  a.prob = reinterpret_cast<float*>(a.idx + (size_t)n * P.KC);
  a.r = a.prob + (size_t)n * P.KC;
  a.u = a.r + P.KC;
  a.cnt = reinterpret_cast<int*>(a.u + 32);
  a.NS = NSr;
  a.NDr = NDr;
  return a;
}

__device__ __forceinline__ void stage_list_async(const FrameParams& P, AcceptScratch& A, int slot, const int* gidx,
                                                 const float* gprob) {
  warp_copy_async(A.idx + (size_t)slot * P.KC, gidx, P.KC * 4);
  warp_copy_async(A.prob + (size_t)slot * P.KC, gprob, P.KC * 4);
}

// Categorical draw from a shared-memory list (idx, w) of n entries (arrays
// 16-byte aligned, capacity a multiple of 4), one thread, with the semantics
// of list_sample: sequential float32 prefix sums over entries with w > 0 in
// index order, t = fl32(u * S), the first entry whose prefix exceeds t, else
// the last candidate; -1 when no entry is positive.  Loads are issued four at
// a time ahead of the dependent sums.
__device__ __forceinline__ int list_sample_s(const int* idx, const float* w, int n, float u) {
  float S = 0.0f;
  int last = -1;
  for (int j = 0; j < n; j += 4) {
    const float4 p4 = *reinterpret_cast<const float4*>(w + j);
    const int4 i4 = *reinterpret_cast<const int4*>(idx + j);
    const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
    const int iv[4] = {i4.x, i4.y, i4.z, i4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (j + e < n && pv[e] > 0.0f) { S = __fadd_rn(S, pv[e]); last = iv[e]; }
  }
  if (last < 0) return -1;
  const float t = __fmul_rn(u, S);
  float acc = 0.0f;
  for (int j = 0; j < n; j += 4) {
    const float4 p4 = *reinterpret_cast<const float4*>(w + j);
    const int4 i4 = *reinterpret_cast<const int4*>(idx + j);
    const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
    const int iv[4] = {i4.x, i4.y, i4.z, i4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (j + e < n && pv[e] > 0.0f) {
        acc = __fadd_rn(acc, pv[e]);
        if (acc > t) return iv[e];
      }
  }
  return last;
}

// Residual weights max(0, p - q) on the entries of the p list (index order),
// the lanes in parallel: outside the p list p = 0, so max(0, -q) = 0 adds
// nothing to the draw.  Warp-wide; r has the p list's capacity.
__device__ __forceinline__ void residual_weights(const int* pi, const float* pp, int np, const int* qi,
                                                 const float* qp, int nq, float* r) {
  const int lane = threadIdx.x & 31;
  for (int j = lane; j < np; j += 32) {
    const float d = __fsub_rn(pp[j], list_lookup(qi, qp, nq, pi[j]));
    r[j] = d > 0.0f ? d : 0.0f;
  }
  __syncwarp();
}

// After codes up to depth s_new are committed: finish the frame or set up
// the next pass (the drafts are drawn from this pass's draft slots on row
// hrow).  Warp-wide; lane 0 owns the scalar state.
template <typename WT>
__device__ __noinline__ void after_commit(const FrameParams& P, const CallArgs& ca, int b, AcceptScratch& A,
                                          int s_new, int hrow) {
  StreamState& S = *A.S;
  const int lane = threadIdx.x & 31;
  StreamStats* ss = P.sstats + b;
  __syncwarp();
  const int frame = S.frame;
  __syncwarp();
  if (s_new >= P.G - 1) {
    if (lane == 0) { bump(ss->frames); bump(ss->committed, P.G - 1); }
    const int nf = frame + 1;
    if (nf < ca.n_frames) setup_frame<WT>(P, ca, b, S, nf);
    else retire_stream(P, b, S);
    return;
  }
  if (P.N == 0) {
    if (lane == 0) { S.s = s_new; S.phase = kPhaseAR; S.pos0 = s_new + 1; S.m = 1; S.n_d = 0; }
    __syncwarp();
    const int code = S.codes[s_new];
    set_pass_rows<WT>(P, b, S, &code);
    return;
  }
  const int R = P.G - 1 - s_new;
  const int n_d = min(S.w - 1, R);  // the frame's window (N unless the adaptive policy narrowed it)
  // The draft distributions q_t = proc(head_{s+t} . h_s), t = 1..n_d, are
  // this pass's speculative draft slots on the row at position s_new
  // (already staged with the target lists): draw the drafts (uniforms one
  // per lane) and keep the lists for the next pass.
  const int ih = hrow - b * P.NS;  // the row's index within the stream
  if (lane < n_d) {
    // draft t = lane + 1, one lane each
    const float u = philox_uniform(P.seed, (uint32_t)b, (uint32_t)S.frame_abs, (uint32_t)(s_new + 1 + lane), kDraft);
    const int ds = A.dslot(ih, lane + 1);
    S.drafts[lane] = valid_code(P, list_sample_s(A.idx + (size_t)ds * P.KC, A.prob + (size_t)ds * P.KC, A.cnt[ds], u));
  }
  __syncwarp();
  if (lane == 0) {
    S.s = s_new;
    S.n_d = n_d;
    S.m = min(n_d + 1, R);
    S.pos0 = s_new + 1;
    S.phase = kPhaseSpec;
  }
  // save q_1..q_{n_d} (16-byte stores) for the next pass's acceptance
  const int kc4 = P.KC >> 2;
  for (int i = lane; i < n_d * kc4; i += 32) {
    const int t = i / kc4, c = i - t * kc4;
    const size_t qi = ((size_t)b * P.ND + t) * P.KC;
    const int ds = A.dslot(ih, t + 1);
    reinterpret_cast<int4*>(P.qidx + qi)[c] = reinterpret_cast<const int4*>(A.idx + (size_t)ds * P.KC)[c];
    reinterpret_cast<float4*>(P.qprob + qi)[c] = reinterpret_cast<const float4*>(A.prob + (size_t)ds * P.KC)[c];
  }
  if (lane < n_d) P.qcount[(size_t)b * P.ND + lane] = A.cnt[A.dslot(ih, lane + 1)];
  __syncwarp();
  int codes_in[CP_SPEC_MAX_WINDOW];
  const int m = S.m;
  codes_in[0] = S.codes[s_new];
  for (int i = 1; i < m; ++i) codes_in[i] = S.drafts[i - 1];
  set_pass_rows<WT>(P, b, S, codes_in);
}

// Teacher-forced run: copy this chunk's target (and draft) logits out.
__device__ void teacher_copy(const FrameParams& P, const CallArgs& ca, int b, const StreamState& S) {
  const int lane = threadIdx.x & 31;
  const int slots = 1 + P.ND;
  for (int i = 0; i < S.m; ++i) {
    const int row = b * P.NS + i, pos = S.pos0 + i;
    if (pos < 1) continue;
    for (int t = 0; t <= (ca.t_draft ? P.ND : 0); ++t) {
      const bool ok = pos + t <= P.G - 1;
      float* dst = t == 0 ? ca.t_logits + ((size_t)b * (ca.P - 1) + pos - 1) * P.V
                          : ca.t_draft + (((size_t)b * (ca.P - 1) + pos - 1) * P.ND + (t - 1)) * P.V;
      const float* src = P.logits + ((size_t)row * slots + t) * P.V;
      for (int v = 2 * lane; v < P.V; v += 64)
        *reinterpret_cast<float2*>(dst + v) = ok ? __ldcg(reinterpret_cast<const float2*>(src + v)) : make_float2(0.f, 0.f);
    }
  }
}

// What the acceptance of stream b reads that no kernel of the pass writes:
// the stream state and, for a speculative round, the draft lists q_t saved
// by the previous pass (staged asynchronously).  Before the dependency wait.
__device__ void accept_prefetch(const FrameParams& P, int b, AcceptScratch& A) {
  StreamState& S = *A.S;
  const int lane = threadIdx.x & 31;
  load_state(P, b, S);
  if (S.phase != kPhaseSpec) return;
  const int n_d = S.n_d;
  for (int t = 1; t <= n_d; ++t) {
    const size_t qi = ((size_t)b * P.ND + t - 1) * P.KC;
    stage_list_async(P, A, A.qslot(t), P.qidx + qi, P.qprob + qi);
  }
  if (lane < n_d) A.cnt[A.qslot(lane + 1)] = __ldcg(P.qcount + (size_t)b * P.ND + lane);
  __syncwarp();
}

// Test hook: NaN into every KV slot of stream b from `from` on (all layers,
// K and V) -- the slots the next pass must write before any row reads them.
// Warp-wide.
__device__ void poison_kv(const FrameParams& P, int b, int from) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (from < 0) from = 0;
  const int per = P.nkv * P.d / 4;        // float4 per slot
  const int n = (P.GS - from) * per;      // per (layer, K/V)
  const float4 nan4 = make_float4(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000),
                                  __int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
  for (int lk = 0; lk < 2 * P.L; ++lk) {
    float4* base = reinterpret_cast<float4*>(P.kv + (((size_t)b * P.L * 2 + lk) * P.GS + from) * P.nkv * P.d);
    for (int q = lane; q < n; q += 32) base[q] = nan4;
  }
  __syncwarp();
}

template <typename WT>
__device__ void accept_stream_tree(const FrameParams& P, const CallArgs& ca, int b, AcceptScratch& A);

// The acceptance decision of stream b for the pass that just ran ("Speculative
// Decoding, Beyond Text", section 02; "CodePredictor Speculative Decoding",
// "How a round works" step 3), then the next pass's rows.  Warp-wide, after
// accept_prefetch and the dependency wait: the target lists are staged in
// one round trip, the uniforms of the decision are drawn one per lane
// meanwhile, and lane 0 runs the left-to-right chain.
template <typename WT>
__device__ void accept_stream(const FrameParams& P, const CallArgs& ca, int b, AcceptScratch& A) {
  StreamState& S = *A.S;
  const int lane = threadIdx.x & 31;
  if (S.phase == kPhaseDone) return;
  const int slots = 1 + P.ND;
  StreamStats* ss = P.sstats + b;
  if (S.phase == kPhaseTeacher) {
    teacher_copy(P, ca, b, S);
    __syncwarp();
    const int next = S.pos0 + S.m;
    __syncwarp();
    if (lane == 0) S.pos0 = next;
    __syncwarp();
    if (next >= ca.P) retire_stream(P, b, S);
    else setup_teacher_chunk<WT>(P, ca, b, S);
    store_state(P, b, S);
    return;
  }
  if (P.tree_n) {
    accept_stream_tree<WT>(P, ca, b, A);
    return;
  }
  // Stage the lists this decision reads (the saved draft lists q_t of a
  // speculative round were staged by accept_prefetch).
  const bool spec = S.phase == kPhaseSpec;
  const int row0 = b * P.NS + (S.phase == kPhasePrefill ? 1 : 0);
  const int s = S.s, n_d = S.n_d, m = S.m;
  const uint32_t fr = (uint32_t)S.frame_abs;
  // the target lists (slot 0) of the rows the decision reads and, when the
  // next pass drafts, the draft slots of every row the commit can stop at
  const int ndn = P.N >= 2 ? P.ND : 0;  // draft slots per row
  const int r_lo = spec ? 0 : row0 - b * P.NS, r_hi = spec ? m : r_lo + 1;
  for (int i = r_lo; i < r_hi; ++i) {
    const size_t li = (size_t)(b * P.NS + i) * slots;
    stage_list_async(P, A, A.tslot(spec ? i : 0), P.lidx + li * P.KC, P.lprob + li * P.KC);
    for (int t = 1; t <= ndn; ++t)
      stage_list_async(P, A, A.dslot(i, t), P.lidx + (li + t) * P.KC, P.lprob + (li + t) * P.KC);
  }
  for (int k = lane; k < (r_hi - r_lo) * (1 + ndn); k += 32) {
    const int i = r_lo + k / (1 + ndn), t = k - (k / (1 + ndn)) * (1 + ndn);
    const int c = __ldcg(P.lcount + (size_t)(b * P.NS + i) * slots + t);
    A.cnt[t == 0 ? A.tslot(spec ? i : 0) : A.dslot(i, t)] = c;
  }
  // uniforms, one per lane, while the lists land: lane t-1 (t = 1..8) the
  // ACCEPT draw at depth s + t; lane 8 + t - 1 (t = 1..9) the TARGET draw at
  // depth s + t (residual at a rejection at t, or the bonus at n_d + 1)
  if (lane < 8 && lane < n_d) A.u[lane] = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + 1 + lane), kAccept);
  if (lane >= 8 && lane < 17 && lane - 8 <= n_d)
    A.u[lane] = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + 1 + lane - 8), kTarget);
  cp_async_wait_all();
  __syncwarp();
  const int* Li = A.idx;
  const float* Lp = A.prob;
  const int KC = P.KC;
  int s_new = 0, hrow = 0, rej = 0;  // rej = 1 + offset of the rejected draft (0: none)
  if (spec) {
    // exact left-to-right acceptance: draft t+1 is accepted iff
    // u_ACCEPT < fl32(p(y) / q(y)); lane t forms that test for draft t+1 and
    // the first failing draft is the rejection (later ones are not reached)
    bool fail = false;
    if (lane < n_d) {
      const int y = S.drafts[lane];
      const int qs = A.qslot(lane + 1), ps = A.tslot(lane);  // scratch slots of q_{t} and p_{s+t}
      const float qy = list_lookup(Li + (size_t)qs * KC, Lp + (size_t)qs * KC, A.cnt[qs], y);
      const float py = list_lookup(Li + (size_t)ps * KC, Lp + (size_t)ps * KC, A.cnt[ps], y);
      fail = !(A.u[lane] < __fdiv_rn(py, qy));
    }
    const unsigned fails = __ballot_sync(0xffffffffu, fail);
    rej = fails ? __ffs(fails) : 0;
    const int reached = rej ? rej : n_d;  // drafts tested
    const int acc = rej ? rej - 1 : n_d;  // drafts accepted
    if (lane < reached) { bump(ss->drafted[lane + 1]); S.reach[lane] += 1; }
    if (lane < acc) { bump(ss->accepted[lane + 1]); S.acc[lane] += 1; S.codes[s + 1 + lane] = S.drafts[lane]; }
    __syncwarp();
  }
  if (lane == 0) {
    if (!spec) {
      const int j = s + 1;  // the pass scored c_j
      const int c = valid_code(P, list_sample_s(Li, Lp, A.cnt[0], A.u[8]));
      S.codes[j] = c;
      ca.codes_out[((size_t)S.frame * ca.B + b) * P.G + j] = c;
      s_new = j;
      hrow = row0;
      bump(ss->passes);
    } else {
      if (rej == 0) {
        if (m > n_d) {
          S.codes[s + n_d + 1] =
              valid_code(P, list_sample_s(Li + (size_t)A.tslot(n_d) * KC, Lp + (size_t)A.tslot(n_d) * KC,
                                          A.cnt[A.tslot(n_d)], A.u[8 + n_d]));
          bump(ss->bonus);
          s_new = s + n_d + 1;
        } else {
          s_new = s + n_d;
        }
      }
      bump(ss->rounds);
      bump(ss->passes);
    }
  }
  rej = __shfl_sync(0xffffffffu, rej, 0);
  if (rej > 0) {
    // draw from norm(max(0, p - q)) at the rejected offset (from p if the
    // residual is zero everywhere)
    const int ps = A.tslot(rej - 1), qs = A.qslot(rej);
    residual_weights(Li + (size_t)ps * KC, Lp + (size_t)ps * KC, A.cnt[ps], Li + (size_t)qs * KC,
                     Lp + (size_t)qs * KC, A.cnt[qs], A.r);
    if (lane == 0) {
      const float ut = A.u[8 + rej - 1];
      int c = list_sample_s(Li + (size_t)ps * KC, A.r, A.cnt[ps], ut);
      if (c < 0) c = list_sample_s(Li + (size_t)ps * KC, Lp + (size_t)ps * KC, A.cnt[ps], ut);
      S.codes[s + rej] = valid_code(P, c);
      bump(ss->rejections);
      s_new = s + rej;
    }
  }
  if (lane == 0) {
    if (spec) {
      for (int j = s + 1; j <= s_new; ++j) ca.codes_out[((size_t)S.frame * ca.B + b) * P.G + j] = S.codes[j];
      hrow = b * P.NS + (s_new - s - 1);
    }
    if (ca.committed_out) ca.committed_out[b] = s_new + 1;
  }
  s_new = __shfl_sync(0xffffffffu, s_new, 0);
  hrow = __shfl_sync(0xffffffffu, hrow, 0);
  __syncwarp();
  if (P.test_poison) poison_kv(P, b, s_new >= P.G - 1 ? 0 : s_new + 1);
  after_commit<WT>(P, ca, b, A, s_new, hrow);
  store_state(P, b, S);
}

// ------------------------------------------------------- sparse-tree rounds
// "RVQ Position Aware Speculative Decoding for On Device TTS", section 2.2
// and Figure 2.  The drafts of depth t are the ranked candidates of
// head_{s+t} on h_s: node i carries the rank[i]-th largest draft logit of its
// depth (value descending, index ascending).  One pass verifies the round's
// root row (position s + 1, the committed code c_s) and a row per kept node
// short of the frame end (position s + 1 + depth, its own KV slot G + i,
// attending to the prefix and its ancestors).  The walk then starts at the
// root: at a node with target law p, its children are tested in rank order
// as point-mass drafts (accept child c iff u < p'(c) with p' the remaining
// mass renormalised, else remove c); a node without an accepted child
// draws one code from what remains (a correction, or the bonus), so every
// committed code keeps the autoregressive law.

// Nodes of the tree kept at codes-left R: depth <= R, rank < V, parent kept
// (bit i).
__device__ __forceinline__ unsigned long long tree_keep(const FrameParams& P, int R) {
  unsigned long long keep = 0;
  for (int i = 0; i < P.tree_n; ++i) {
    const int par = __ldg(&P.tree->parent[i]);
    if (__ldg(&P.tree->dep[i]) <= R && __ldg(&P.tree->rank[i]) < P.V && (par < 0 || ((keep >> par) & 1ull)))
      keep |= 1ull << i;
  }
  return keep;
}

// After codes up to depth s_new are committed in a tree context: finish the
// frame, or set up the next round's tree from the draft slots of row hrow
// (whose output is h_{s_new}).  Warp-wide; lane 0 owns the scalar state.
template <typename WT>
__device__ __noinline__ void after_commit_tree(const FrameParams& P, const CallArgs& ca, int b, AcceptScratch& A,
                                               int s_new, int hrow) {
  StreamState& S = *A.S;
  const int lane = threadIdx.x & 31;
  StreamStats* ss = P.sstats + b;
  __syncwarp();
  const int frame = S.frame;
  __syncwarp();
  if (s_new >= P.G - 1) {
    if (lane == 0) { bump(ss->frames); bump(ss->committed, P.G - 1); }
    const int nf = frame + 1;
    if (nf < ca.n_frames) setup_frame<WT>(P, ca, b, S, nf);
    else retire_stream(P, b, S);
    return;
  }
  const int R = P.G - 1 - s_new;
  const unsigned long long keep = tree_keep(P, R);
  const int slots = 1 + P.ND;
  int* tok = P.ttok + (size_t)b * 64;
  // candidates of depth t: the draft slot's list holds the need[t] largest
  // logits in index order; rank them by (logit descending, index ascending)
  if (lane == 0) {
    for (int t = 1; t <= P.tree->dmax && t <= R; ++t) {
      const size_t li = (size_t)hrow * slots + t;
      const int n = min(P.lcount[li], 64);
      int ord[64];
      float val[64];
      for (int j = 0; j < n; ++j) {
        const int v = P.lidx[li * P.KC + j];
        const float x = P.logits[li * P.V + v];
        int at = j;  // insertion: after every entry with a larger logit, or an equal one (lower index)
        while (at > 0 && val[at - 1] < x) { val[at] = val[at - 1]; ord[at] = ord[at - 1]; --at; }
        val[at] = x;
        ord[at] = v;
      }
      for (int i = 0; i < P.tree_n; ++i)
        if (((keep >> i) & 1ull) && __ldg(&P.tree->dep[i]) == t) {
          const int rk = __ldg(&P.tree->rank[i]);
          tok[i] = valid_code(P, rk < n ? ord[rk] : -1);
        }
    }
  }
  __syncwarp();
  // the next pass's rows: the root (position s_new + 1, code c_{s_new}) in
  // row slot 0, kept node i short of the frame end in row slot i + 1
  long long kvpos = 0;
  int m = 0;
  for (int k = lane; k < P.NS; k += 32) {
    int pos = -1, code = 0, slot = 0;
    if (k == 0) {
      pos = s_new + 1; code = S.codes[s_new]; slot = pos;
    } else {
      const int i = k - 1, dep = __ldcg(&P.tree->dep[i]);
      if (i < P.tree_n && ((keep >> i) & 1ull) && dep < R) {
        pos = s_new + 1 + dep; code = __ldcg(tok + i); slot = P.G + i;
      }
    }
    P.row_pos[b * P.NS + k] = pos;
    P.row_code[b * P.NS + k] = code;
    P.row_slot[b * P.NS + k] = slot;
    if (g_mirror_on) { g_mpos[b * P.NS + k] = pos; g_mcode[b * P.NS + k] = code; g_mslot[b * P.NS + k] = slot; }
    if (pos >= 0) { ++m; kvpos += s_new + 2 + (k == 0 ? 0 : __ldcg(&P.tree->dep[k - 1])); }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m += __shfl_xor_sync(0xffffffffu, m, o);
    kvpos += __shfl_xor_sync(0xffffffffu, kvpos, o);
  }
  if (lane == 0) {
    S.s = s_new;
    S.n_d = 0;
    S.m = m;
    S.pos0 = s_new + 1;
    S.phase = kPhaseSpec;
    atomicAdd((unsigned long long*)&P.ctl->kv_bytes,
              (unsigned long long)(kvpos * P.L * 2 * P.nkv * P.d * (long long)sizeof(float)));
    atomicAdd((unsigned long long*)&P.ctl->weight_bytes, (unsigned long long)((long long)m * P.H * sizeof(WT)));
  }
  __syncwarp();
}

// The tree round's decision for stream b (or the frame prefill's commit of
// c_1), the accepted path's K/V copied to its canonical positions, then the
// next round.  Warp-wide; lane 0 walks the tree.
template <typename WT>
__device__ void accept_stream_tree(const FrameParams& P, const CallArgs& ca, int b, AcceptScratch& A) {
  StreamState& S = *A.S;
  const int lane = threadIdx.x & 31;
  StreamStats* ss = P.sstats + b;
  const int slots = 1 + P.ND, KC = P.KC;
  const int s = S.s;
  const uint32_t fr = (uint32_t)S.frame_abs;
  int s_new = 0, hrow = 0, acc_n = 0;
  if (lane == 0) {
    if (S.phase == kPhasePrefill) {
      // the prefill scored c_1 on the row of E_0(c_0)
      const size_t li = (size_t)(b * P.NS + 1) * slots;
      const float u = philox_uniform(P.seed, (uint32_t)b, fr, 1u, kTarget);
      const int c = valid_code(P, list_sample(P.lidx + li * KC, P.lprob + li * KC, P.lcount[li], u));
      S.codes[1] = c;
      ca.codes_out[((size_t)S.frame * ca.B + b) * P.G + 1] = c;
      s_new = 1;
      hrow = b * P.NS + 1;
      bump(ss->passes);
    } else {
      const int R = P.G - 1 - s;
      const unsigned long long keep = tree_keep(P, R);
      const int* tok = P.ttok + (size_t)b * 64;
      float* work = A.r;  // the current node's remaining mass, aligned with its list
      int cur = -1, d = 0;
      while (s + d < P.G - 1) {
        const size_t li = (size_t)(b * P.NS + cur + 1) * slots;  // the row of node cur (root: row 0)
        const int* pidx = P.lidx + li * KC;
        const float* pp = P.lprob + li * KC;
        const int pn = P.lcount[li];
        for (int j = 0; j < pn; ++j) work[j] = pp[j];
        int taken = -1, ci = 0;
        for (int i = 0; i < P.tree_n && taken < 0; ++i) {
          if (!((keep >> i) & 1ull) || __ldg(&P.tree->parent[i]) != cur) continue;
          float Sm = 0.0f;
          for (int j = 0; j < pn; ++j) Sm = __fadd_rn(Sm, work[j]);
          const int y = tok[i];
          int at = -1;
          for (int j = 0; j < pn; ++j)
            if (pidx[j] == y) { at = j; break; }
          const float rr = Sm > 0.0f ? __fdiv_rn(at >= 0 ? work[at] : 0.0f, Sm) : 0.0f;
          const float u = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + d + 1), kTreeAccept + (uint32_t)ci);
          if (u < rr) taken = i;
          else if (at >= 0) work[at] = 0.0f;
          ++ci;
        }
        if (taken >= 0) {
          S.codes[s + d + 1] = tok[taken];
          S.drafts[d < 8 ? d : 7] = taken;  // the accepted path (node per depth)
          cur = taken;
          ++d;
          ++acc_n;
          bump(ss->accepted[d < 9 ? d : 8]);
          continue;
        }
        const float u = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + d + 1), kTarget);
        int y = list_sample(pidx, work, pn, u);
        if (y < 0) y = list_sample(pidx, pp, pn, u);
        S.codes[s + d + 1] = valid_code(P, y);
        ++d;
        if (ci > 0) bump(ss->rejections);
        else bump(ss->bonus);
        break;
      }
      s_new = s + d;
      hrow = b * P.NS + cur + 1;
      for (int j = s + 1; j <= s_new; ++j) ca.codes_out[((size_t)S.frame * ca.B + b) * P.G + j] = S.codes[j];
      bump(ss->rounds);
      bump(ss->passes);
    }
    if (ca.committed_out) ca.committed_out[b] = s_new + 1;
  }
  s_new = __shfl_sync(0xffffffffu, s_new, 0);
  hrow = __shfl_sync(0xffffffffu, hrow, 0);
  acc_n = __shfl_sync(0xffffffffu, acc_n, 0);
  __syncwarp();
  // the accepted nodes' K/V (tree slots) to canonical positions s + 2 .. s + 1 + acc_n,
  // which the next round's rows read as their prefix
  if (s_new < P.G - 1 && acc_n > 0) {
    const int d4 = P.nkv * P.d / 4;  // float4 per slot
    const int per = 2 * P.L * d4;
    for (int q = lane; q < acc_n * per; q += 32) {
      const int j = q / per, rem = q - j * per;
      const int lk = rem / d4, c = rem - lk * d4;  // lk = 2 layer + (0: K, 1: V)
      const size_t base = ((size_t)b * P.L * 2 + lk) * P.GS;
      const float4* src = reinterpret_cast<const float4*>(P.kv + (base + P.G + S.drafts[j]) * P.nkv * P.d) + c;
      float4* dst = reinterpret_cast<float4*>(P.kv + (base + s + 2 + j) * P.nkv * P.d) + c;
      *dst = __ldcg(src);
    }
  }
  __syncwarp();
  if (P.test_poison) poison_kv(P, b, s_new >= P.G - 1 ? 0 : s_new + 1);
  after_commit_tree<WT>(P, ca, b, A, s_new, hrow);
  store_state(P, b, S);
}

// The rows of the next pass, compacted, and the lm_heads it needs (head_j
// for j in [pos, pos + ND] of every row at pos >= 1).  One warp.
__device__ int build_plan(const FrameParams& P, const CallArgs& ca) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  int n = 0;
  const int total = ca.B * P.NS;
  unsigned long long mask = 0;
  for (int j0 = 0; j0 < total; j0 += 32) {
    const int r = j0 + lane;
    const int pos = r < total ? (g_mirror_on ? g_mpos[r] : __ldcg(P.row_pos + r)) : -1;
    const bool on = pos >= 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, on);
    if (on) {
      const int at = n + __popc(bal & lt);
      P.prow[at] = r;
      P.ppos[at] = pos;
      P.pcode[at] = g_mirror_on ? g_mcode[r] : __ldcg(P.row_code + r);
      P.pslot[at] = g_mirror_on ? g_mslot[r] : __ldcg(P.row_slot + r);
      if (pos >= 1)
        for (int t = 0; t <= P.ND && pos + t <= P.G - 1; ++t) mask |= 1ull << (pos + t);
    }
    n += __popc(bal);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mask |= __shfl_xor_sync(0xffffffffu, mask, o);
  if (lane == 0) {
    int nh = 0;
    for (int hd = 1; hd < P.G && hd < 64; ++hd)
      if ((mask >> hd) & 1ull) P.plan->heads[nh++] = hd;
    P.plan->nheads = nh;
    P.plan->nrows = n;
    if (n > 0) {
      atomicAdd(reinterpret_cast<unsigned long long*>(&P.ctl->weight_bytes),
                (unsigned long long)((long long)P.L * P.layer_bytes + (long long)nh * P.head_bytes));
      atomicAdd(reinterpret_cast<unsigned long long*>(&P.ctl->heads_applied), (unsigned long long)nh);
    }
  }
  __syncwarp();
  return n;
}

// Last-CTA election: true in the CTA that finishes last; its threads then
// see every other CTA's writes (each CTA fences before counting itself).
__device__ __forceinline__ bool last_cta(Control* ctl) {
  __shared__ int s_last;
  if (gridDim.x == 1) {  // the block's own writes are visible to it after the barrier
    __syncthreads();
    return true;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&ctl->done, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (s_last) __threadfence();
  return s_last != 0;
}

// Sets the pass loop's condition (inside a graph): continue while streams
// are active and the pass cap is not reached.
__device__ __forceinline__ void set_loop(const FrameParams& P, bool go) {
  if (P.cond != 0) cudaGraphSetConditional((cudaGraphConditionalHandle)P.cond, go ? 1u : 0u);
}

// Stream setup of a call: frame 0 (decode) or the first teacher chunk; then
// the first pass's plan.
template <typename WT>
__global__ void __launch_bounds__(kThreads, 2) setup_kernel(const __grid_constant__ FrameParams P) {
  extern __shared__ __align__(16) unsigned char ssmem[];
  const CallArgs ca = *P.call;
  const int warp = threadIdx.x >> 5;
  if (blockIdx.x == 0 && threadIdx.x == 0) { P.ctl->active = ca.B; P.ctl->pass = 0; }
  mirror_init(P, ca);
  const int b = blockIdx.x * (blockDim.x >> 5) + warp;
  if (b < ca.B) {
    AcceptScratch A = accept_scratch(P, ssmem);
    StreamState& S = *A.S;
    for (int i = threadIdx.x & 31; i < (int)(sizeof(StreamState) / 4); i += 32) reinterpret_cast<int*>(&S)[i] = 0;
    __syncwarp();
    if (ca.mode == kModeTeacher) {
      if ((threadIdx.x & 31) == 0) { S.frame_abs = ca.first_frame; S.pos0 = 0; }
      setup_teacher_chunk<WT>(P, ca, b, S);
    } else {
      setup_frame<WT>(P, ca, b, S, 0);
    }
    store_state(P, b, S);
  }
  if (!last_cta(P.ctl)) return;
  int nrows = 0;
  if (warp == 0) nrows = build_plan(P, ca);
  if (threadIdx.x == 0) {
    if (gridDim.x > 1) P.ctl->done = 0;
    set_loop(P, nrows > 0);
  }
}

// Acceptance of every stream (warp per stream), then the next pass's plan
// and the loop condition.
template <typename WT>
__global__ void __launch_bounds__(kThreads, 2) accept_kernel(const __grid_constant__ FrameParams P) {
  extern __shared__ __align__(16) unsigned char ssmem[];
  const CallArgs ca = *P.call;
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.x * (blockDim.x >> 5) + warp;
  // loop bookkeeping words, fetched early (CTA 0 is not necessarily the last)
  int pass0 = 0, status0 = 0;
  if (threadIdx.x == 0) { pass0 = __ldcg(&P.ctl->pass); status0 = __ldcg(&P.ctl->status); }
  mirror_init(P, ca);
  AcceptScratch A = accept_scratch(P, ssmem);
  if (b < ca.B) accept_prefetch(P, b, A);
  pdl_wait();
  if (b < ca.B) accept_stream<WT>(P, ca, b, A);
  if (!last_cta(P.ctl)) return;
  int nrows = 0;
  if (warp == 0) nrows = build_plan(P, ca);
  if (threadIdx.x == 0) {
    Control* ctl = P.ctl;
    if (gridDim.x > 1) { ctl->done = 0; pass0 = __ldcg(&ctl->pass); status0 = __ldcg(&ctl->status); }
    atomicAdd(reinterpret_cast<unsigned long long*>(&ctl->passes), 1ull);
    atomicAdd(reinterpret_cast<unsigned long long*>(&ctl->kernels), (unsigned long long)P.kernels_per_pass);
    const int pass = pass0 + 1;
    ctl->pass = pass;
    // every unfinished stream has rows in the next pass
    const bool more = nrows > 0;
    const bool capped = pass >= ca.pass_cap;
    if (more && capped && ca.max_passes == 0) raise_status(&ctl->status, kStatusDevice);
    set_loop(P, more && !capped && status0 == 0);
  }
}

// ------------------------------------------------------------- init kernel
__global__ void init_tables_kernel(float2* rope, int G, int d, double theta, int* top_k, float* temp, int Bmax, int k,
                                   float T) {
  const int half = d / 2;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < G * half; i += gridDim.x * blockDim.x) {
    const int pos = i / half, e = i % half;
    const double inv = pow(theta, -2.0 * e / (double)d);
    const double ang = (double)pos * inv;
    rope[i] = make_float2((float)cos(ang), (float)sin(ang));
  }
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < Bmax; b += gridDim.x * blockDim.x) {
    top_k[b] = k;
    temp[b] = T;
  }
}

// Position-aware draft offsets ("RVQ Position Aware Speculative Decoding for
// On Device TTS", section 2.2): the draft of lookahead t applies head_j to
// h + b_t.  The product is linear, so head_j . b_t is formed once per
// context: otab[j-1][t-1][v] = sum_k head_j[v][k] b_t[k], one warp per
// (head, vocabulary row), fp32 accumulation in a fixed order.
template <typename WT>
__global__ void __launch_bounds__(256) offset_table_kernel(const void* head, const float* b, float* otab, int G,
                                                            int V, int H, int KO) {
  constexpr int kMaxKO = CP_SPEC_MAX_WINDOW - 1;
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long w = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; w < (long long)(G - 1) * V;
       w += nwarps) {
    const size_t row = (size_t)w * H;  // head j = w / V + 1, vocabulary row v = w % V
    float acc[kMaxKO];
#pragma unroll
    for (int t = 0; t < kMaxKO; ++t) acc[t] = 0.0f;
    for (int k = lane; k < H; k += 32) {
      const float x = WTraits<WT>::load1(head, row + k);
#pragma unroll
      for (int t = 0; t < kMaxKO; ++t)
        if (t < KO) acc[t] = fmaf(x, __ldg(&b[(size_t)t * H + k]), acc[t]);
    }
#pragma unroll
    for (int t = 0; t < kMaxKO; ++t) {
      float a = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      acc[t] = a;
    }
    if (lane == 0) {
      const int hj = (int)(w / V), v = (int)(w % V);
      for (int t = 0; t < KO; ++t) otab[((size_t)hj * KO + t) * V + v] = acc[t];
    }
  }
}

}  // namespace cpk

// ------------------------------------------------------------ host side
namespace cpk_host {

using cpk::FrameParams;

template <typename WT>
struct KernelSet {
  template <bool TC>
  static const void* gemv_t(int kind) {
    switch (kind) {
      case cpk::kQKV: return (const void*)cpk::gemv_kernel<WT, cpk::kQKV, TC>;
      case cpk::kO: return (const void*)cpk::gemv_kernel<WT, cpk::kO, TC>;
      case cpk::kGU: return (const void*)cpk::gemv_kernel<WT, cpk::kGU, TC>;
      case cpk::kDown: return (const void*)cpk::gemv_kernel<WT, cpk::kDown, TC>;
      default: return (const void*)cpk::gemv_kernel<WT, cpk::kHeads, TC>;
    }
  }
  static const void* gemv(int kind, bool tc) { return tc ? gemv_t<true>(kind) : gemv_t<false>(kind); }
  static const void* setup() { return (const void*)cpk::setup_kernel<WT>; }
  static const void* accept() { return (const void*)cpk::accept_kernel<WT>; }
};

const void* mv_fn(int kind) {
  switch (kind) {
    case cpk::kQKV: return (const void*)cpk::mv_kernel<cpk::kQKV>;
    case cpk::kO: return (const void*)cpk::mv_kernel<cpk::kO>;
    case cpk::kGU: return (const void*)cpk::mv_kernel<cpk::kGU>;
    case cpk::kDown: return (const void*)cpk::mv_kernel<cpk::kDown>;
    default: return (const void*)cpk::mv_kernel<cpk::kHeads>;
  }
}

const void* t5_fn(int kind) {
  switch (kind) {
    case cpk::kQKV: return (const void*)cpk::t5_kernel<cpk::kQKV>;
    case cpk::kO: return (const void*)cpk::t5_kernel<cpk::kO>;
    case cpk::kGU: return (const void*)cpk::t5_kernel<cpk::kGU>;
    case cpk::kDown: return (const void*)cpk::t5_kernel<cpk::kDown>;
    default: return (const void*)cpk::t5_kernel<cpk::kHeads>;
  }
}

// The GEMV kernel of a kind for a parameter block: the small-batch tensor
// path (bf16, few rows), the tcgen05 tiles (bf16, many rows), the mma.sync
// tensor path (bf16, many rows, shapes the tiles do not take), or CUDA cores.
const void* gemv_fn(const FrameParams& P, int kind) {
  if (P.dtype == 1 && P.t5) return t5_fn(kind);
  if (P.dtype == 1 && P.mv) return mv_fn(kind);
  return P.dtype == 1 ? KernelSet<__nv_bfloat16>::gemv(kind, P.tc != 0) : KernelSet<float>::gemv(kind, false);
}
const void* setup_fn(int dtype) { return dtype == 1 ? KernelSet<__nv_bfloat16>::setup() : KernelSet<float>::setup(); }
const void* accept_fn(int dtype) { return dtype == 1 ? KernelSet<__nv_bfloat16>::accept() : KernelSet<float>::accept(); }

static int gemv_K_host(const FrameParams& P, int kind) {
  return kind == cpk::kO ? P.nq * P.d : (kind == cpk::kDown ? P.F : P.H);
}

// Dynamic shared memory of each kernel for a parameter block.
size_t gemv_smem(const FrameParams& P, int kind) {
  if (P.dtype == 1 && P.t5)
    return cpk::t5_smem_layout(kind, P.t5_rb[kind], P.t5_stages[kind], gemv_K_host(P, kind), P.Bmax * P.NS, P.G, P.d).total;
  if (P.dtype == 1 && P.mv)
    return cpk::mv_smem_layout(kind, P.mv_slots[kind], gemv_K_host(P, kind), P.Bmax * P.NS, P.G, P.d).total;
  // two weight slots, the partial sums of one tile, the pass rows (3
  // arrays), then (QKV) the RoPE table and (normed kinds) the gain.  Sized
  // per kind so that consecutive kernels' CTAs fit on one SM together.
  size_t b = 2 * (size_t)cpk::kSlotBytes + cpk::kRedFloats * sizeof(float) +
             ((3 * (size_t)P.Bmax * P.NS + 3) / 4 * 4) * sizeof(int);
  if (P.tc)  // every region, then the tensor path's output blocks and row descriptors, and a row list
    return b + cpk::kRopeSmemBytes + (size_t)(P.H + 3) / 4 * 4 * sizeof(float) + cpk::kTcYFloats * sizeof(float) +
           (size_t)P.Bmax * P.NS * sizeof(int);
  if (kind == cpk::kQKV || kind == cpk::kGU || kind == cpk::kHeads) b += cpk::kRopeSmemBytes + (size_t)P.H * sizeof(float);
  return b;
}
size_t attention_smem(const FrameParams& P) {
  return ((size_t)2 * P.G * P.d + (size_t)(P.nq / P.nkv) * P.d + (size_t)(cpk::kAttnThreads / 32) * CP_SPEC_MAX_CODE_GROUPS) *
         sizeof(float);
}
size_t topk_smem(const FrameParams& P) {
  return ((size_t)P.V * 4 + 15) / 16 * 16 + (size_t)cpk::kWarps * 1024 + ((size_t)P.KC * 4 + 15) / 16 * 16 + 256;
}
size_t accept_smem(const FrameParams& P, int warps) {
  return (size_t)warps * cpk::accept_scratch_bytes(cpk::accept_rows(P.NS, P.tree_n),
                                                   cpk::accept_drafts(P.NS, P.ND, P.tree_n), P.KC);
}

// Small-batch tensor path: the weight-row slots of each GEMV kind, or false
// when the shape does not fit it (then the context keeps the other paths).
// Every layer kind's per-CTA tile must fit the weight budget and is held
// whole (one phase, every row copied before the dependency wait); the
// lm_heads tile may be larger and streams through two banks.
constexpr size_t kMvWeightBudget = 100 * 1024;   // weight region of one CTA
constexpr size_t kMvSmemLimit = 220 * 1024;      // dynamic shared memory of one CTA
bool plan_mv(FrameParams& P, int sms) {
  const int rows_cap = P.Bmax * P.NS;
  if (P.dtype != 1 || rows_cap > cpk::kMvMaxRows || sms < 1) return false;
  const int Ks[3] = {P.H, P.nq * P.d, P.F};
  for (int K : Ks)
    if (K % (32 * cpk::kWarps) != 0) return false;  // each warp's K slice: whole 32-element blocks
  for (int kind = cpk::kQKV; kind <= cpk::kHeads; ++kind) {
    const int K = gemv_K_host(P, kind);
    const size_t RS = (size_t)K * 2 + cpk::kMvRowPad;
    const int rpu = (kind == cpk::kQKV || kind == cpk::kGU) ? 2 : 1;
    long long U;
    switch (kind) {
      case cpk::kQKV: U = (long long)(P.nq + 2 * P.nkv) * (P.d / 2); break;
      case cpk::kO: case cpk::kDown: U = P.H; break;
      case cpk::kGU: U = P.F; break;
      default: U = (long long)std::min(P.G - 1, cpk::kMaxHeadsPerPass) * P.V;
    }
    const long long need = (U + sms - 1) / sms * rpu;  // rows of the largest tile
    long long S = std::min<long long>(need, (long long)(kMvWeightBudget / RS));
    // a layer GEMV whose tile does not fit one phase would serialise its
    // banks' copies on every pass: such shapes keep the CUDA-core kernel
    if (S < need && kind != cpk::kHeads) return false;
    if (S < need) S = std::max<long long>(S / 2 * 2, 4);
    while (S >= 4 && cpk::mv_smem_layout(kind, (int)S, K, rows_cap, P.G, P.d).total > kMvSmemLimit) S -= 2;
    if (S < 4 || (S < need && S / 2 < rpu)) return false;
    P.mv_slots[kind] = (int)S;
  }
  P.mv = 1;
  return true;
}

// Units of a GEMV kind with the most lm_heads a pass can apply.
static long long gemv_units_max(const FrameParams& P, int kind) {
  switch (kind) {
    case cpk::kQKV: return (long long)(P.nq + 2 * P.nkv) * (P.d / 2);
    case cpk::kO: case cpk::kDown: return P.H;
    case cpk::kGU: return P.F;
    default: return (long long)std::min(P.G - 1, cpk::kMaxHeadsPerPass) * P.V;
  }
}

// tcgen05 tiles: pass rows per tile and ring stages of each GEMV kind, or
// false when the shape does not fit them (every GEMV width a multiple of the
// 64-element slab; a tile of the lm_heads inside one head).  The rows per
// tile (64, 32 or 16) minimise waves of one CTA per SM x the work of a tile
// (a fixed part per slab plus the conversion of its rows) for a full pass;
// the ring takes as many stages as fit the shared-memory budget.
constexpr size_t kT5SmemBudget = 200 * 1024;
bool plan_t5(FrameParams& P, int sms) {
  const int rows_cap = P.Bmax * P.NS;
  // (a tile's RoPE halves are whole boxes of d/2 rows: d/2 divides 64)
  if (P.dtype != 1 || sms < 1 || P.H % 64 != 0 || (P.nq * P.d) % 64 != 0 || P.F % 64 != 0 || P.V % cpk::kT5M != 0 ||
      P.d % 2 != 0 || P.d / 2 > 64 || 64 % (P.d / 2) != 0)
    return false;
  for (int kind = cpk::kQKV; kind <= cpk::kHeads; ++kind) {
    const int K = gemv_K_host(P, kind);
    const long long mtiles = cpk::t5_mtiles(kind, (int)gemv_units_max(P, kind));
    int RB = 16;
    long long best = -1;
    for (int rb : {64, 32, 16}) {
      const long long waves = (mtiles * ((rows_cap + rb - 1) / rb) + sms - 1) / sms;
      const long long cost = waves * (32 + rb);
      if (best < 0 || cost < best) { best = cost; RB = rb; }
    }
    int st = cpk::kT5MaxStages;
    while (st > 3 && cpk::t5_smem_layout(kind, RB, st, K, rows_cap, P.G, P.d).total > kT5SmemBudget) --st;
    if (cpk::t5_smem_layout(kind, RB, st, K, rows_cap, P.G, P.d).total > kT5SmemBudget || mtiles > 65535) return false;
    P.t5_rb[kind] = RB;
    P.t5_stages[kind] = st;
  }
  P.t5 = 1;
  return true;
}

static dim3 t5_grid(const FrameParams& P, int kind) {
  const int rows_cap = P.Bmax * P.NS, RB = P.t5_rb[kind];
  return dim3((rows_cap + RB - 1) / RB, cpk::t5_mtiles(kind, (int)gemv_units_max(P, kind)));
}

// Raise (never lower) a kernel's dynamic shared-memory limit on the current
// device.  Contexts and the allocation-free path share the kernels; a limit
// set for a smaller configuration must not shrink it under a graph that an
// earlier, larger configuration instantiated.
static std::mutex g_attr_mu;
static std::map<std::pair<int, const void*>, size_t> g_smem_high;
static cudaError_t raise_smem_limit(const void* fn, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  size_t& high = g_smem_high[std::make_pair(dev, fn)];
  if (bytes <= high) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) high = bytes;
  return e;
}

// Raise the dynamic shared-memory limit of every pass kernel of a dtype.
cudaError_t configure_kernels(const FrameParams& P, int accept_warps) {
  cudaError_t e = cudaSuccess;
  // every pass kernel asks for the largest shared-memory carve-out, so the
  // SM configuration never changes between consecutive kernels and a
  // dependent's CTA can start beside its predecessor's
  for (int k = cpk::kQKV; k <= cpk::kHeads && e == cudaSuccess; ++k) {
    e = raise_smem_limit(gemv_fn(P, k), gemv_smem(P, k));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemv_fn(P, k), cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  }
  const void* others[] = {(const void*)cpk::attention_kernel, (const void*)cpk::topk_kernel, setup_fn(P.dtype),
                          accept_fn(P.dtype)};
  for (const void* f : others)
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) e = raise_smem_limit((const void*)cpk::attention_kernel, attention_smem(P));
  if (e == cudaSuccess) e = raise_smem_limit((const void*)cpk::topk_kernel, topk_smem(P));
  if (e == cudaSuccess) e = raise_smem_limit(setup_fn(P.dtype), accept_smem(P, accept_warps));
  if (e == cudaSuccess) e = raise_smem_limit(accept_fn(P.dtype), accept_smem(P, accept_warps));
  return e;
}

static cudaError_t launch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// Stream setup of a call (not a programmatic dependent: it follows every
// earlier piece of work on the stream).
cudaError_t enqueue_setup(const FrameParams& P, int accept_warps, cudaStream_t s) {
  void* args[] = {const_cast<FrameParams*>(&P)};
  const int grid = (P.Bmax + accept_warps - 1) / accept_warps;
  return launch(setup_fn(P.dtype), dim3(grid), dim3(32 * accept_warps), accept_smem(P, accept_warps), s, false, args);
}

// One pass: 5 L + 3 kernels; the first is a full dependent of earlier work,
// the others programmatic dependents of their predecessor.
cudaError_t enqueue_pass(const FrameParams& P, int sms, int accept_warps, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  bool first = true;
  int l = 0, arg = 0;
  void* gargs[] = {const_cast<FrameParams*>(&P), &arg};
  void* pargs[] = {const_cast<FrameParams*>(&P)};
  const int rows = P.Bmax * P.NS;
  // a GEMV of one kind: the small-batch kernel takes 8 * layer + kind
  auto gemv = [&](int kind, bool pdl) {
    if (P.t5) {
      arg = l;
      return launch(gemv_fn(P, kind), t5_grid(P, kind), dim3(cpk::kT5Threads), gemv_smem(P, kind), s, pdl, gargs);
    }
    arg = P.mv ? 8 * l + kind : l;
    return launch(gemv_fn(P, kind), dim3(sms), dim3(cpk::kThreads), gemv_smem(P, kind), s, pdl, gargs);
  };
  for (l = 0; l < P.L && e == cudaSuccess; ++l) {
    e = gemv(cpk::kQKV, !first);
    first = false;
    if (e == cudaSuccess) {
      arg = l;
      e = launch((const void*)cpk::attention_kernel, dim3(rows * P.nkv), dim3(cpk::kAttnThreads), attention_smem(P), s, true,
                 gargs);
    }
    if (e == cudaSuccess) e = gemv(cpk::kO, true);
    if (e == cudaSuccess) e = gemv(cpk::kGU, true);
    if (e == cudaSuccess) e = gemv(cpk::kDown, true);
  }
  l = 0;
  if (e == cudaSuccess) e = gemv(cpk::kHeads, true);
  if (e == cudaSuccess)
    e = launch((const void*)cpk::topk_kernel, dim3(rows * (1 + P.ND)), dim3(cpk::kThreads), topk_smem(P), s, true, pargs);
  if (e == cudaSuccess) {
    const int grid = (P.Bmax + accept_warps - 1) / accept_warps;
    e = launch(accept_fn(P.dtype), dim3(grid), dim3(32 * accept_warps), accept_smem(P, accept_warps), s, true, pargs);
  }
  return e;
}

// The graph of a whole call: the setup kernel, then a while loop whose body
// is one pass; the accept kernel of each pass sets the loop condition.
// `P.cond` is filled in here.  `cs` is a non-default stream used for capture.
cudaError_t build_call_graph(FrameParams P, int sms, int accept_warps, cudaStream_t cs, cudaGraphExec_t* out) {
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaGraphCreate(&g, 0);
  if (e != cudaSuccess) return e;
  cudaGraphConditionalHandle h;
  e = cudaGraphConditionalHandleCreate(&h, g, 1, cudaGraphCondAssignDefault);
  P.cond = (unsigned long long)h;
  cudaGraphNode_t setup_node = nullptr, loop_node = nullptr;
  if (e == cudaSuccess) {
    cudaKernelNodeParams kp = {};
    void* args[] = {&P};
    kp.func = const_cast<void*>(setup_fn(P.dtype));
    kp.gridDim = dim3((P.Bmax + accept_warps - 1) / accept_warps);
    kp.blockDim = dim3(32 * accept_warps);
    kp.sharedMemBytes = (unsigned)accept_smem(P, accept_warps);
    kp.kernelParams = args;
    e = cudaGraphAddKernelNode(&setup_node, g, nullptr, 0, &kp);
  }
  cudaGraphNodeParams cp = {};
  if (e == cudaSuccess) {
    cp.type = cudaGraphNodeTypeConditional;
    cp.conditional.handle = h;
    cp.conditional.type = cudaGraphCondTypeWhile;
    cp.conditional.size = 1;
    e = cudaGraphAddNode(&loop_node, g, &setup_node, nullptr, 1, &cp);
  }
  if (e == cudaSuccess) {
    cudaGraph_t body = cp.conditional.phGraph_out[0];
    e = cudaStreamBeginCaptureToGraph(cs, body, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      const cudaError_t e1 = enqueue_pass(P, sms, accept_warps, cs);
      const cudaError_t e2 = cudaStreamEndCapture(cs, &body);
      e = e1 != cudaSuccess ? e1 : e2;
    }
  }
  if (e == cudaSuccess) e = cudaGraphInstantiate(out, g, 0);
  cudaGraphDestroy(g);
  return e;
}

cudaError_t launch_init_tables(float2* rope, int G, int d, double theta, int* top_k, float* temp, int Bmax, int k,
                               float T, cudaStream_t stream) {
  cpk::init_tables_kernel<<<8, 256, 0, stream>>>(rope, G, d, theta, top_k, temp, Bmax, k, T);
  return cudaGetLastError();
}

cudaError_t launch_offset_table(const FrameParams& P, cudaStream_t stream) {
  if (P.KO <= 0) return cudaSuccess;
  if (P.KO > CP_SPEC_MAX_WINDOW - 1 || !P.draft_offset) return cudaErrorInvalidValue;
  const long long warps = (long long)(P.G - 1) * P.V;
  const int blocks = (int)((warps + 7) / 8 < 65535 ? (warps + 7) / 8 : 65535);
  if (P.dtype == 1)
    cpk::offset_table_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(P.head, P.draft_offset, P.otab, P.G, P.V, P.H, P.KO);
  else
    cpk::offset_table_kernel<float><<<blocks, 256, 0, stream>>>(P.head, P.draft_offset, P.otab, P.G, P.V, P.H, P.KO);
  return cudaGetLastError();
}

}  // namespace cpk_host
