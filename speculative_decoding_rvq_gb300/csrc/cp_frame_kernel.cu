// cp_frame_kernel.cu -- the persistent CodePredictor frame kernel.
//
// One cooperative launch (one CTA per SM) runs decoder passes until every
// stream has finished its frames.  A pass is, for all streams at once:
//
//   per layer: [QKV + RoPE + KV append] | [attention over the stream's KV]
//              | [O + residual] | [RMSNorm + gate/up + SwiGLU] | [down + residual]
//   [final RMSNorm + lm_heads]  target head_j on the row at position j, and,
//                               speculatively, head_{j+1..j+N-1} on the same
//                               row: the free drafts of the next round
//                               ("CodePredictor Speculative Decoding", "Why
//                               the draft is free")
//   [top-k / temperature / softmax]   one warp per (row, head) vocabulary row
//   [accept / commit / reconcile]     one warp per stream: exact speculative
//                               sampling ("How a round works" step 3), codes
//                               committed, draft codes for the next round
//                               sampled, next rows staged, KV length = s'+1
//
// Phases are separated by bounded grid barriers.  The GEMV phases are
// HBM-bound at small batch: each CTA streams a contiguous share of the
// weight rows with 128-bit non-allocating loads and, before waiting at a
// barrier, issues bulk L2 prefetches for its share of the next two weight
// phases so the weight stream does not stop at phase boundaries.  Every
// (row, feature) dot product is computed by one warp in a fixed order, so a
// row's result does not depend on which other rows share the pass (greedy
// speculative decoding reproduces greedy autoregressive decoding exactly).
#include <cuda_bf16.h>
#include <stdio.h>

#include "cp_common.cuh"
#include "cp_frame.cuh"
#include "cp_sampling.cuh"

namespace cpk {

// ------------------------------------------------------------ weight types
template <typename WT> struct WTraits;
template <> struct WTraits<float> {
  static constexpr int EPC = 4;  // elements per 16-byte chunk
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static float load1(const float* p) { return __ldg(p); }
};
template <> struct WTraits<__nv_bfloat16> {
  static constexpr int EPC = 8;
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    float2 a = bf16x2_to_f2(u.x), b = bf16x2_to_f2(u.y), c = bf16x2_to_f2(u.z), d = bf16x2_to_f2(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  __device__ __forceinline__ static float load1(const __nv_bfloat16* p) {
    const unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(((uint32_t)u) << 16);
  }
};

enum GemvKind : int { kQKV = 0, kO = 1, kGU = 2, kDown = 3, kHeads = 4 };

struct CtaShared {
  int nrows;
  int nheads;
  int heads[CP_SPEC_MAX_CODE_GROUPS];
};

// Pair p of a GEMV phase -> the two weight rows it reads.
template <typename WT>
__device__ __forceinline__ void pair_rows(const FrameParams& P, int kind, int l, int p, const CtaShared& cs,
                                          const WT*& w0, const WT*& w1) {
  const int H = P.H, d = P.d, half = P.d / 2;
  switch (kind) {
    case kQKV: {
      const int hh = p / half, e = p % half;
      const WT* base;
      int hr;
      if (hh < P.nq) { base = (const WT*)P.wq[l]; hr = hh; }
      else if (hh < P.nq + P.nkv) { base = (const WT*)P.wk[l]; hr = hh - P.nq; }
      else { base = (const WT*)P.wv[l]; hr = hh - P.nq - P.nkv; }
      w0 = base + ((size_t)hr * d + e) * H;
      w1 = base + ((size_t)hr * d + e + half) * H;
      break;
    }
    case kO: {
      const WT* base = (const WT*)P.wo[l];
      const int K = P.nq * d;
      w0 = base + (size_t)(2 * p) * K;
      w1 = w0 + K;
      break;
    }
    case kGU:
      w0 = (const WT*)P.w_gate[l] + (size_t)p * H;
      w1 = (const WT*)P.w_up[l] + (size_t)p * H;
      break;
    case kDown: {
      const WT* base = (const WT*)P.w_down[l];
      w0 = base + (size_t)(2 * p) * P.F;
      w1 = w0 + P.F;
      break;
    }
    default: {  // heads: pair p covers vocab entries (2p, 2p+1) of the (p*2/V)-th needed head
      const int f = 2 * p;
      const int hd = cs.heads[f / P.V];
      w0 = (const WT*)P.head + ((size_t)(hd - 1) * P.V + (f % P.V)) * H;
      w1 = w0 + H;
    }
  }
}

__device__ __forceinline__ int gemv_pairs(const FrameParams& P, int kind, const CtaShared& cs) {
  switch (kind) {
    case kQKV: return (P.nq + 2 * P.nkv) * (P.d / 2);
    case kO: return P.H / 2;
    case kGU: return P.F;
    case kDown: return P.H / 2;
    default: return cs.nheads * (P.V / 2);
  }
}

__device__ __forceinline__ int gemv_K(const FrameParams& P, int kind) {
  return kind == kO ? P.nq * P.d : (kind == kDown ? P.F : P.H);
}

__device__ __forceinline__ void cta_pair_range(int np, int& p0, int& p1) {
  p0 = (int)(((long long)np * blockIdx.x) / gridDim.x);
  p1 = (int)(((long long)np * (blockIdx.x + 1)) / gridDim.x);
}

// Issue bulk L2 prefetches for this CTA's share of a weight phase.
template <typename WT>
__device__ __noinline__ void prefetch_phase(const FrameParams& P, int kind, int l, const CtaShared& cs) {
  if (threadIdx.x != 0) return;
  const int np = gemv_pairs(P, kind, cs);
  int p0, p1;
  cta_pair_range(np, p0, p1);
  const size_t rb = (size_t)gemv_K(P, kind) * sizeof(WT);
  for (int which = 0; which < 2; ++which) {
    const char* start = nullptr;
    size_t len = 0;
    for (int p = p0; p < p1; ++p) {
      const WT *w0, *w1;
      pair_rows<WT>(P, kind, l, p, cs, w0, w1);
      const char* r = (const char*)(which ? w1 : w0);
      if (kind == kO || kind == kDown || kind == kHeads) {  // both rows adjacent: one range
        if (which) break;
        const char* r0 = (const char*)w0;
        if (start && r0 == start + len) { len += 2 * rb; continue; }
        if (start) prefetch_l2(start, (uint32_t)len);
        start = r0; len = 2 * rb;
        continue;
      }
      if (start && r == start + len) { len += rb; continue; }
      if (start) prefetch_l2(start, (uint32_t)len);
      start = r; len = rb;
    }
    if (start) prefetch_l2(start, (uint32_t)len);
  }
}

// Stage activation rows into shared memory (optionally RMS-normalised).
// bf16 weights use a split layout: element k of a row goes to half
// (k & 7) >> 2, slot 4*(k >> 3) + (k & 3), so a lane's 8-element chunk is
// two conflict-free float4 reads.
template <typename WT>
__device__ void stage_rows(const FrameParams& P, const float* src, int ld, int K, const float* gain,
                           const int* rows, int nr, float* xs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < nr; r += kWarps) {
    const float* s = src + (size_t)rows[r] * ld;
    float inv = 1.0f;
    if (gain) {
      float ss = 0.0f;
      for (int k = lane * 4; k < K; k += 128) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(s + k));
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
      ss = warp_sum(ss);
      inv = 1.0f / sqrtf(ss / (float)K + P.eps);
    }
    float* dst = xs + (size_t)r * K;
    for (int k = lane * 4; k < K; k += 128) {
      float4 v = __ldcg(reinterpret_cast<const float4*>(s + k));
      if (gain) {
        const float4 g = __ldg(reinterpret_cast<const float4*>(gain + k));
        v.x = v.x * inv * g.x; v.y = v.y * inv * g.y; v.z = v.z * inv * g.z; v.w = v.w * inv * g.w;
      }
      if (WTraits<WT>::EPC == 8) {
        const int c = k >> 3, hf = (k & 7) >> 2;
        *reinterpret_cast<float4*>(dst + hf * (K / 2) + 4 * c) = v;
      } else {
        *reinterpret_cast<float4*>(dst + k) = v;
      }
    }
  }
}

// Partial dot products of two weight rows with nr staged rows over chunks
// [cb, ce) (16-byte chunks), lanes striding by 32 chunks.
template <typename WT, int RB>
__device__ __forceinline__ void gemv_pair_partial(const WT* __restrict__ w0, const WT* __restrict__ w1,
                                                  const float* xs, int K, int nr, int cb, int ce,
                                                  float (&a0)[RB], float (&a1)[RB]) {
  constexpr int EPC = WTraits<WT>::EPC;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < RB; ++r) { a0[r] = 0.0f; a1[r] = 0.0f; }
  constexpr int U = 4;
  for (int c0 = cb + lane; c0 < ce; c0 += 32 * U) {
    uint4 u0[U], u1[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int c = c0 + 32 * j;
      if (c < ce) { u0[j] = ldg_stream(w0 + (size_t)c * EPC); u1[j] = ldg_stream(w1 + (size_t)c * EPC); }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int c = c0 + 32 * j;
      if (c >= ce) break;
      float f0[EPC], f1[EPC];
      WTraits<WT>::unpack(u0[j], f0);
      WTraits<WT>::unpack(u1[j], f1);
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        if (r >= nr) break;
        const float* xr = xs + (size_t)r * K;
        if (EPC == 8) {
          const float4 x0 = *reinterpret_cast<const float4*>(xr + 4 * c);
          const float4 x1 = *reinterpret_cast<const float4*>(xr + K / 2 + 4 * c);
          float s0 = a0[r], s1 = a1[r];
          s0 = fmaf(f0[0], x0.x, s0); s0 = fmaf(f0[1], x0.y, s0); s0 = fmaf(f0[2], x0.z, s0); s0 = fmaf(f0[3], x0.w, s0);
          s0 = fmaf(f0[4], x1.x, s0); s0 = fmaf(f0[5], x1.y, s0); s0 = fmaf(f0[6], x1.z, s0); s0 = fmaf(f0[7], x1.w, s0);
          s1 = fmaf(f1[0], x0.x, s1); s1 = fmaf(f1[1], x0.y, s1); s1 = fmaf(f1[2], x0.z, s1); s1 = fmaf(f1[3], x0.w, s1);
          s1 = fmaf(f1[4], x1.x, s1); s1 = fmaf(f1[5], x1.y, s1); s1 = fmaf(f1[6], x1.z, s1); s1 = fmaf(f1[7], x1.w, s1);
          a0[r] = s0; a1[r] = s1;
        } else {
          const float4 x0 = *reinterpret_cast<const float4*>(xr + 4 * c);
          float s0 = a0[r], s1 = a1[r];
          s0 = fmaf(f0[0], x0.x, s0); s0 = fmaf(f0[1], x0.y, s0); s0 = fmaf(f0[2], x0.z, s0); s0 = fmaf(f0[3], x0.w, s0);
          s1 = fmaf(f1[0], x0.x, s1); s1 = fmaf(f1[1], x0.y, s1); s1 = fmaf(f1[2], x0.z, s1); s1 = fmaf(f1[3], x0.w, s1);
          a0[r] = s0; a1[r] = s1;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RB; ++r) { a0[r] = warp_sum(a0[r]); a1[r] = warp_sum(a1[r]); }
}

// Epilogue of one (pair, row): writes the phase's outputs.
template <typename WT>
__device__ __forceinline__ void gemv_epilogue(const FrameParams& P, int kind, int l, int p, int row, float y0,
                                              float y1, const CtaShared& cs) {
  switch (kind) {
    case kQKV: {
      const int half = P.d / 2, hh = p / half, e = p % half;
      const int pos = __ldcg(P.row_pos + row);
      const int b = row / P.NS;
      if (hh < P.nq + P.nkv) {
        const float2 cs2 = P.rope[(size_t)pos * half + e];
        const float r0 = y0 * cs2.x - y1 * cs2.y;
        const float r1 = y1 * cs2.x + y0 * cs2.y;
        if (hh < P.nq) {
          float* q = P.qbuf + (size_t)row * P.nq * P.d + (size_t)hh * P.d;
          q[e] = r0; q[e + half] = r1;
        } else {
          float* k = P.kv + (((((size_t)b * P.L + l) * 2 + 0) * P.G + pos) * P.nkv + (hh - P.nq)) * P.d;
          k[e] = r0; k[e + half] = r1;
        }
      } else {
        float* v = P.kv + (((((size_t)b * P.L + l) * 2 + 1) * P.G + pos) * P.nkv + (hh - P.nq - P.nkv)) * P.d;
        v[e] = y0; v[e + half] = y1;
      }
      break;
    }
    case kO:
    case kDown: {
      float* h = P.h + (size_t)row * P.H + 2 * p;
      const float2 old = __ldcg(reinterpret_cast<const float2*>(h));
      *reinterpret_cast<float2*>(h) = make_float2(old.x + y0, old.y + y1);
      break;
    }
    case kGU: {
      const float silu = y0 / (1.0f + expf(-y0));
      P.act[(size_t)row * P.F + p] = silu * y1;
      break;
    }
    default: {
      const int f = 2 * p, hd = cs.heads[f / P.V], v = f % P.V;
      const int pos = __ldcg(P.row_pos + row);
      const int slot = hd - pos;
      if (pos >= 1 && slot >= 0 && slot <= P.ND) {
        float* dst = P.logits + ((size_t)row * (1 + P.ND) + slot) * P.V + v;
        *reinterpret_cast<float2*>(dst) = make_float2(y0, y1);
      }
    }
  }
}

template <typename WT, int RB>
__device__ __noinline__ void gemv_phase(const FrameParams& P, int kind, int l, const CtaShared& cs, const int* rows,
                           float* uni) {
  const int K = gemv_K(P, kind);
  const int np = gemv_pairs(P, kind, cs);
  int p0, p1;
  cta_pair_range(np, p0, p1);
  const int npc = p1 - p0;
  if (npc <= 0 || cs.nrows <= 0) return;
  const float* src;
  int ld;
  const float* gain;
  switch (kind) {
    case kQKV: src = P.h; ld = P.H; gain = P.attn_norm[l]; break;
    case kO: src = P.obuf; ld = P.nq * P.d; gain = nullptr; break;
    case kGU: src = P.h; ld = P.H; gain = P.ffn_norm[l]; break;
    case kDown: src = P.act; ld = P.F; gain = nullptr; break;
    default: src = P.h; ld = P.H; gain = P.final_norm;
  }
  constexpr int EPC = WTraits<WT>::EPC;
  const int nch = K / EPC;
  // K-split factor: a fixed function of the shapes, never of the row count
  int KS = 1;
  while (KS < 8 && npc * KS * 2 <= kWarps && nch / (KS * 2) >= 32) KS *= 2;
  const int gpr = kWarps / KS;  // groups (pairs) per round
  float* xs = uni;
  float* red = uni + (size_t)RB * K;  // [kWarps][2][RB]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int cb = 0; cb < cs.nrows; cb += RB) {
    const int nr = min(RB, cs.nrows - cb);
    __syncthreads();
    stage_rows<WT>(P, src, ld, K, gain, rows + cb, nr, xs);
    __syncthreads();
    for (int g0 = 0; g0 < npc; g0 += gpr) {
      const int g = g0 + warp / KS, ks = warp % KS;
      float a0[RB], a1[RB];
      if (g < npc) {
        const WT *w0, *w1;
        pair_rows<WT>(P, kind, l, p0 + g, cs, w0, w1);
        const int cb_ = (int)(((long long)nch * ks) / KS), ce_ = (int)(((long long)nch * (ks + 1)) / KS);
        gemv_pair_partial<WT, RB>(w0, w1, xs, K, nr, cb_, ce_, a0, a1);
      }
      if (KS == 1) {
        if (g < npc) {
#pragma unroll
          for (int r = 0; r < RB; ++r)
            if (r < nr && lane == r) gemv_epilogue<WT>(P, kind, l, p0 + g, rows[cb + r], a0[r], a1[r], cs);
        }
      } else {
        if (g < npc) {
#pragma unroll
          for (int r = 0; r < RB; ++r)
            if (lane == r) { red[(warp * 2 + 0) * RB + r] = a0[r]; red[(warp * 2 + 1) * RB + r] = a1[r]; }
        }
        __syncthreads();
        if (g < npc && ks == 0 && lane < nr) {
          float y0 = 0.0f, y1 = 0.0f;
          for (int j = 0; j < KS; ++j) {
            y0 += red[((warp + j) * 2 + 0) * RB + lane];
            y1 += red[((warp + j) * 2 + 1) * RB + lane];
          }
          gemv_epilogue<WT>(P, kind, l, p0 + g, rows[cb + lane], y0, y1, cs);
        }
        __syncthreads();
      }
    }
  }
}

template <typename WT>
__device__ void gemv_dispatch(const FrameParams& P, int kind, int l, const CtaShared& cs, const int* rows,
                              float* uni) {
  switch (P.RB) {
    case 8: gemv_phase<WT, 8>(P, kind, l, cs, rows, uni); break;
    case 4: gemv_phase<WT, 4>(P, kind, l, cs, rows, uni); break;
    case 2: gemv_phase<WT, 2>(P, kind, l, cs, rows, uni); break;
    default: gemv_phase<WT, 1>(P, kind, l, cs, rows, uni); break;
  }
}

// Causal GQA attention of every (row, query head) over positions 0..pos.
__device__ __noinline__ void attention_phase(const FrameParams& P, int l, const CtaShared& cs, const int* rows, float* uni) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sq = uni + (size_t)warp * (256 + 64);
  float* sw = sq + 256;
  const int items = cs.nrows * P.nq;
  const int grp = P.nq / P.nkv, d = P.d;
  const float scale = 1.0f / sqrtf((float)d);
  for (int it = blockIdx.x * kWarps + warp; it < items; it += gridDim.x * kWarps) {
    const int r = rows[it / P.nq], hq = it % P.nq, g = hq / grp;
    const int b = r / P.NS;
    const int pos = __ldcg(P.row_pos + r);
    const float* qv = P.qbuf + (size_t)r * P.nq * d + (size_t)hq * d;
    for (int e = lane * 4; e < d; e += 128)
      *reinterpret_cast<float4*>(sq + e) = __ldcg(reinterpret_cast<const float4*>(qv + e));
    __syncwarp();
    const float* kb = P.kv + ((((size_t)b * P.L + l) * 2 + 0) * P.G) * P.nkv * d + (size_t)g * d;
    const float* vb = P.kv + ((((size_t)b * P.L + l) * 2 + 1) * P.G) * P.nkv * d + (size_t)g * d;
    float sc[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = lane + 32 * jj;
      if (j <= pos) {
        const float* kj = kb + (size_t)j * P.nkv * d;
        float s = 0.0f;
        for (int e = 0; e < d; e += 4) {
          const float4 kk = __ldcg(reinterpret_cast<const float4*>(kj + e));
          const float4 qq = *reinterpret_cast<const float4*>(sq + e);
          s = fmaf(qq.x, kk.x, s); s = fmaf(qq.y, kk.y, s); s = fmaf(qq.z, kk.z, s); s = fmaf(qq.w, kk.w, s);
        }
        sc[jj] = s * scale;
      }
    }
    const float mx = warp_max(fmaxf(sc[0], sc[1]));
    float ex[2];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) ex[jj] = (lane + 32 * jj <= pos) ? expf(sc[jj] - mx) : 0.0f;
    const float den = warp_sum(ex[0] + ex[1]);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
      if (lane + 32 * jj <= pos) sw[lane + 32 * jj] = ex[jj] / den;
    __syncwarp();
    float* ov = P.obuf + (size_t)r * P.nq * d + (size_t)hq * d;
    for (int e = lane * 4; e < d; e += 128) {
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j <= pos; ++j) {
        const float w = sw[j];
        const float4 vv = __ldcg(reinterpret_cast<const float4*>(vb + (size_t)j * P.nkv * d + e));
        o.x = fmaf(w, vv.x, o.x); o.y = fmaf(w, vv.y, o.y); o.z = fmaf(w, vv.z, o.z); o.w = fmaf(w, vv.w, o.w);
      }
      *reinterpret_cast<float4*>(ov + e) = o;
    }
    __syncwarp();
  }
}

// Top-k / temperature / softmax of every (row, slot) vocabulary row.
__device__ __noinline__ void proc_phase(const FrameParams& P, const CtaShared& cs, const int* rows, float* uni) {
  const int warp = threadIdx.x >> 5;
  if (warp >= P.proc_warps) return;
  const size_t per_warp = (size_t)P.V * 4 + 1024 + (size_t)P.KC * 8;
  unsigned char* base = reinterpret_cast<unsigned char*>(uni) + (size_t)warp * ((per_warp + 15) / 16 * 16);
  double* ebuf = reinterpret_cast<double*>(base);
  uint32_t* hist = reinterpret_cast<uint32_t*>(base + (size_t)P.KC * 8);
  uint32_t* keys = hist + 256;
  const int slots = 1 + P.ND;
  const int items = cs.nrows * slots;
  for (int it = blockIdx.x + gridDim.x * warp; it < items; it += gridDim.x * P.proc_warps) {
    const int r = rows[it / slots], t = it % slots;
    const int pos = __ldcg(P.row_pos + r);
    if (pos < 1 || pos + t > P.G - 1) continue;
    const int b = r / P.NS;
    const int k = P.top_k[b];
    const float T = P.temp[b];
    const size_t li = (size_t)r * slots + t;
    const int n = warp_process_row(P.logits + li * P.V, P.V, k, T, keys, hist, ebuf, P.lidx + li * P.KC,
                                   P.lprob + li * P.KC);
    if ((threadIdx.x & 31) == 0) P.lcount[li] = n;
  }
}

// ------------------------------------------------------ per-stream logic
struct WarpScratch {
  StreamState s;
};

template <typename WT>
__device__ void stage_input_row(const FrameParams& P, int row, int pos, int code, const float* x) {
  const int lane = threadIdx.x & 31;
  float* dst = P.h + (size_t)row * P.H;
  if (pos == 0) {
    for (int k = lane * 4; k < P.H; k += 128)
      *reinterpret_cast<float4*>(dst + k) = __ldg(reinterpret_cast<const float4*>(x + k));
  } else {
    const WT* e = (const WT*)P.embed + ((size_t)(pos - 1) * P.V + code) * P.H;
    for (int k = lane; k < P.H; k += 32) dst[k] = WTraits<WT>::load1(e + k);
  }
}

// Mark the lm_heads the rows at positions pos0..pos0+m-1 need in the next pass.
__device__ __forceinline__ void mark_heads(const FrameParams& P, int pos0, int m, int parity_next) {
  unsigned long long bits = 0;
  for (int i = 0; i < m; ++i) {
    const int pos = pos0 + i;
    if (pos < 1) continue;
    for (int t = 0; t <= P.ND && pos + t <= P.G - 1; ++t) bits |= 1ull << (pos + t);
  }
  if (bits) atomicOr(&P.ctl->head_mask[parity_next], bits);
}

// Stage the rows of the next pass for stream b (state already updated in S).
template <typename WT>
__device__ void stage_pass_rows(const FrameParams& P, int b, StreamState& S, const int* codes_in,
                                const float* x, int parity_next) {
  const int lane = threadIdx.x & 31;
  for (int i = 0; i < P.NS; ++i) {
    const int row = b * P.NS + i;
    if (i < S.m) {
      const int pos = S.pos0 + i;
      int code = 0;
      if (pos > 0) code = codes_in[i];
      if (lane == 0) P.row_pos[row] = pos;
      stage_input_row<WT>(P, row, pos, code, x);
    } else if (lane == 0) {
      P.row_pos[row] = -1;
    }
  }
  if (lane == 0) {
    mark_heads(P, S.pos0, S.m, parity_next);
    const long long kvb = (long long)(S.pos0 + S.m) * P.L * 2 * P.nkv * P.d * (long long)sizeof(float);
    atomicAdd((unsigned long long*)&P.ctl->kv_bytes, (unsigned long long)kvb);
    atomicAdd((unsigned long long*)&P.ctl->weight_bytes, (unsigned long long)((long long)S.m * P.H * sizeof(WT)));
  }
  __syncwarp();
}

__device__ __forceinline__ int valid_code(const FrameParams& P, int c) {
  if (c < 0 || c >= P.V) { raise_status(&P.ctl->status, kStatusDevice); return 0; }
  return c;
}

// Frame start: rows [x, E_0(c_0)] at positions 0, 1.
// Scalar state fields are written by lane 0 only; every all-lane read of them
// follows a __syncwarp().
template <typename WT>
__device__ void setup_frame(const FrameParams& P, int b, StreamState& S, int frame, int parity_next) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane == 0) {
    const int c0 = valid_code(P, __ldg(P.c0 + (size_t)frame * P.B + b));
    S.frame = frame;
    S.frame_abs = P.first_frame + frame;
    S.codes[0] = c0;
    S.s = 0;
    S.phase = kPhasePrefill;
    S.pos0 = 0;
    S.m = 2;
    S.n_d = 0;
    P.codes_out[((size_t)frame * P.B + b) * P.G] = c0;
    if (P.committed_out) P.committed_out[b] = 1;
  }
  __syncwarp();
  int codes_in[2] = {0, S.codes[0]};
  stage_pass_rows<WT>(P, b, S, codes_in, P.x + ((size_t)frame * P.B + b) * P.H, parity_next);
}

template <typename WT>
__device__ void setup_teacher_chunk(const FrameParams& P, int b, StreamState& S, int parity_next) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  const int pos0 = S.pos0;
  const int m = min(P.NS, P.P - pos0);
  __syncwarp();
  if (lane == 0) { S.m = m; S.phase = kPhaseTeacher; }
  __syncwarp();
  int codes_in[CP_SPEC_MAX_WINDOW];
  for (int i = 0; i < m; ++i) {
    const int pos = pos0 + i;
    codes_in[i] = pos > 0 ? valid_code(P, __ldg(P.t_codes + (size_t)b * (P.P - 1) + pos - 1)) : 0;
  }
  stage_pass_rows<WT>(P, b, S, codes_in, P.x + (size_t)b * P.H, parity_next);
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

// After codes up to depth s_new are committed: finish the frame or stage the next pass.
template <typename WT>
__device__ void after_commit(const FrameParams& P, int b, StreamState& S, int s_new, int hrow, int parity_next) {
  const int lane = threadIdx.x & 31;
  StreamStats* ss = P.sstats + b;
  __syncwarp();
  const int frame = S.frame;
  __syncwarp();
  if (s_new >= P.G - 1) {
    if (lane == 0) { ss->frames += 1; ss->committed += P.G - 1; }
    const int nf = frame + 1;
    if (nf < P.n_frames) {
      setup_frame<WT>(P, b, S, nf, parity_next);
    } else {
      if (lane == 0) {
        S.phase = kPhaseDone;
        S.m = 0;
        for (int i = 0; i < P.NS; ++i) P.row_pos[b * P.NS + i] = -1;
        atomicSub(&P.ctl->active, 1);
      }
      __syncwarp();
    }
    return;
  }
  if (P.N == 0) {
    if (lane == 0) { S.s = s_new; S.phase = kPhaseAR; S.pos0 = s_new + 1; S.m = 1; S.n_d = 0; }
    __syncwarp();
    int code = S.codes[s_new];
    stage_pass_rows<WT>(P, b, S, &code, nullptr, parity_next);
    return;
  }
  const int R = P.G - 1 - s_new;
  const int n_d = min(P.N - 1, R);
  const int slots = 1 + P.ND;
  // save the draft distributions q_t = proc(head_{s+t} . h_s): they are the
  // rows of this pass's speculative draft slots on the row at position s_new
  for (int t = 1; t <= n_d; ++t) {
    const size_t li = (size_t)hrow * slots + t;
    const int n = __ldcg(P.lcount + li);
    const size_t qi = ((size_t)b * P.ND + (t - 1)) * P.KC;
    for (int j = lane; j < n; j += 32) {
      P.qidx[qi + j] = __ldcg(P.lidx + li * P.KC + j);
      P.qprob[qi + j] = __ldcg(P.lprob + li * P.KC + j);
    }
    if (lane == 0) P.qcount[(size_t)b * P.ND + (t - 1)] = n;
  }
  __syncwarp();
  if (lane == 0) {
    for (int t = 1; t <= n_d; ++t) {
      const size_t qi = ((size_t)b * P.ND + (t - 1)) * P.KC;
      const int n = P.qcount[(size_t)b * P.ND + (t - 1)];
      const float u = philox_uniform(P.seed, (uint32_t)b, (uint32_t)S.frame_abs, (uint32_t)(s_new + t), kDraft);
      S.drafts[t - 1] = valid_code(P, list_sample(P.qidx + qi, P.qprob + qi, n, u));
    }
    S.s = s_new;
    S.n_d = n_d;
    S.m = min(n_d + 1, R);
    S.pos0 = s_new + 1;
    S.phase = kPhaseSpec;
  }
  __syncwarp();
  int codes_in[CP_SPEC_MAX_WINDOW];
  const int m = S.m;
  codes_in[0] = S.codes[s_new];
  for (int i = 1; i < m; ++i) codes_in[i] = S.drafts[i - 1];
  stage_pass_rows<WT>(P, b, S, codes_in, nullptr, parity_next);
}

template <typename WT>
__device__ void accept_stream(const FrameParams& P, int b, StreamState& S, int parity_next) {
  const int lane = threadIdx.x & 31;
  load_state(P, b, S);
  if (S.phase == kPhaseDone) return;
  const int slots = 1 + P.ND;
  StreamStats* ss = P.sstats + b;
  if (S.phase == kPhaseTeacher) {
    for (int i = 0; i < S.m; ++i) {
      const int row = b * P.NS + i, pos = S.pos0 + i;
      if (pos < 1) continue;
      const float* lg = P.logits + (size_t)row * slots * P.V;
      float* dst = P.t_logits + ((size_t)b * (P.P - 1) + pos - 1) * P.V;
      for (int v = lane; v < P.V; v += 32) dst[v] = __ldcg(lg + v);
      if (P.t_draft) {
        for (int t = 1; t <= P.ND; ++t) {
          float* dd = P.t_draft + (((size_t)b * (P.P - 1) + pos - 1) * P.ND + (t - 1)) * P.V;
          const bool ok = pos + t <= P.G - 1;
          for (int v = lane; v < P.V; v += 32) dd[v] = ok ? __ldcg(lg + (size_t)t * P.V + v) : 0.0f;
        }
      }
    }
    __syncwarp();
    const int next = S.pos0 + S.m;
    __syncwarp();
    if (lane == 0) S.pos0 = next;
    __syncwarp();
    if (next >= P.P) {
      if (lane == 0) {
        S.phase = kPhaseDone;
        S.m = 0;
        for (int i = 0; i < P.NS; ++i) P.row_pos[b * P.NS + i] = -1;
        atomicSub(&P.ctl->active, 1);
      }
      __syncwarp();
    } else {
      setup_teacher_chunk<WT>(P, b, S, parity_next);
    }
    store_state(P, b, S);
    return;
  }
  int s_new = 0, hrow = 0;
  if (lane == 0) {
    const uint32_t fr = (uint32_t)S.frame_abs;
    const int s = S.s;
    if (S.phase == kPhasePrefill || S.phase == kPhaseAR) {
      const int j = s + 1;  // the pass scored c_j
      const int row = b * P.NS + (S.phase == kPhasePrefill ? 1 : 0);
      const size_t li = (size_t)row * slots;
      const float u = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)j, kTarget);
      const int c = valid_code(P, list_sample<LdCG>(P.lidx + li * P.KC, P.lprob + li * P.KC, __ldcg(P.lcount + li), u));
      S.codes[j] = c;
      P.codes_out[((size_t)S.frame * P.B + b) * P.G + j] = c;
      s_new = j;
      hrow = row;
      ss->passes += 1;
    } else {  // speculative round: exact left-to-right acceptance
      const int n_d = S.n_d, m = S.m;
      int t = 1;
      bool rejected = false;
      for (; t <= n_d; ++t) {
        const int y = S.drafts[t - 1];
        const size_t qi = ((size_t)b * P.ND + (t - 1)) * P.KC;
        const int nq = P.qcount[(size_t)b * P.ND + (t - 1)];
        const size_t li = (size_t)(b * P.NS + t - 1) * slots;
        const int np = __ldcg(P.lcount + li);
        const int* pi = P.lidx + li * P.KC;
        const float* pp = P.lprob + li * P.KC;
        const float qy = list_lookup(P.qidx + qi, P.qprob + qi, nq, y);
        const float py = list_lookup<LdCG>(pi, pp, np, y);
        const float ratio = __fdiv_rn(py, qy);
        ss->drafted[t] += 1;
        const float ua = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + t), kAccept);
        if (ua < ratio) {
          S.codes[s + t] = y;
          ss->accepted[t] += 1;
          continue;
        }
        const float ut = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + t), kTarget);
        int c = residual_sample<LdCG>(pi, pp, np, P.qidx + qi, P.qprob + qi, nq, ut);
        if (c < 0) c = list_sample<LdCG>(pi, pp, np, ut);
        S.codes[s + t] = valid_code(P, c);
        rejected = true;
        break;
      }
      if (rejected) {
        s_new = s + t;
        ss->rejections += 1;
      } else if (m > n_d) {
        const size_t li = (size_t)(b * P.NS + n_d) * slots;
        const float ut = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + n_d + 1), kTarget);
        S.codes[s + n_d + 1] =
            valid_code(P, list_sample<LdCG>(P.lidx + li * P.KC, P.lprob + li * P.KC, __ldcg(P.lcount + li), ut));
        ss->bonus += 1;
        s_new = s + n_d + 1;
      } else {
        s_new = s + n_d;
      }
      for (int j = s + 1; j <= s_new; ++j) P.codes_out[((size_t)S.frame * P.B + b) * P.G + j] = S.codes[j];
      hrow = b * P.NS + (s_new - s - 1);
      ss->rounds += 1;
      ss->passes += 1;
    }
    if (P.committed_out) P.committed_out[b] = s_new + 1;
  }
  s_new = __shfl_sync(0xffffffffu, s_new, 0);
  hrow = __shfl_sync(0xffffffffu, hrow, 0);
  __syncwarp();
  after_commit<WT>(P, b, S, s_new, hrow, parity_next);
  store_state(P, b, S);
}

template <typename WT>
__device__ __noinline__ void accept_phase(const FrameParams& P, int parity_next, float* uni, bool setup) {
  const int warp = threadIdx.x >> 5;
  StreamState& S = reinterpret_cast<WarpScratch*>(uni)[warp].s;
  for (int b = blockIdx.x + gridDim.x * warp; b < P.B; b += gridDim.x * kWarps) {
    if (setup) {
      if (P.mode == kModeTeacher) {
        for (int i = threadIdx.x & 31; i < (int)(sizeof(StreamState) / 4); i += 32) reinterpret_cast<int*>(&S)[i] = 0;
        __syncwarp();
        if ((threadIdx.x & 31) == 0) { S.frame_abs = P.first_frame; S.pos0 = 0; }
        setup_teacher_chunk<WT>(P, b, S, parity_next);
      } else {
        for (int i = threadIdx.x & 31; i < (int)(sizeof(StreamState) / 4); i += 32) reinterpret_cast<int*>(&S)[i] = 0;
        __syncwarp();
        setup_frame<WT>(P, b, S, 0, parity_next);
      }
      store_state(P, b, S);
    } else {
      accept_stream<WT>(P, b, S, parity_next);
    }
  }
}

// Active rows of the pass and the lm_heads it needs, identical in every CTA.
__device__ __noinline__ void build_pass_lists(const FrameParams& P, int parity, CtaShared& cs, int* rows) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const unsigned lt = (1u << lane) - 1u;
    int n = 0;
    const int total = P.B * P.NS;
    for (int j0 = 0; j0 < total; j0 += 32) {
      const int r = j0 + lane;
      const bool on = r < total && __ldcg(P.row_pos + r) >= 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, on);
      if (on) rows[n + __popc(bal & lt)] = r;
      n += __popc(bal);
    }
    if (lane == 0) {
      cs.nrows = n;
      const unsigned long long mask = __ldcg(&P.ctl->head_mask[parity]);
      int nh = 0;
      for (int hd = 1; hd < P.G && hd < 64; ++hd)
        if ((mask >> hd) & 1ull) cs.heads[nh++] = hd;
      cs.nheads = nh;
    }
  }
  __syncthreads();
}

template <typename WT>
__device__ void prefetch_weight_phase(const FrameParams& P, int w, CtaShared& cs) {
  const int per_pass = 4 * P.L + 1;
  const int idx = w % per_pass;
  if (idx == 4 * P.L) {
    prefetch_phase<WT>(P, kHeads, 0, cs);
  } else {
    const int l = idx / 4, kind = idx % 4;  // kQKV, kO, kGU, kDown
    prefetch_phase<WT>(P, kind, l, cs);
  }
}

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) frame_kernel(const __grid_constant__ FrameParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // dynamic shared memory: [active row list, B*NS ints][phase union region]
  int* rows = reinterpret_cast<int*>(smem_raw);
  const size_t rows_bytes = ((size_t)P.B * P.NS * 4 + 15) / 16 * 16;
  float* uni = reinterpret_cast<float*>(smem_raw + rows_bytes);
  __shared__ CtaShared cs;
  Control* ctl = P.ctl;
  unsigned long long gen = 0;
  const int pass_base = __ldcg(&ctl->pass_global);
  int pass = 0;
  if (P.do_setup) {
    if (blockIdx.x == 0 && threadIdx.x == 0) ctl->active = P.B;
    accept_phase<WT>(P, pass_base & 1, uni, true);
    if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) return;
  }
  // Every pass commits at least one code of every unfinished stream, so a
  // decode needs at most n_frames * (G - 1) passes and a teacher run
  // ceil(P / NS); anything beyond that is a logic error, reported, not looped.
  const int pass_cap = P.max_passes > 0 ? P.max_passes
                       : (P.mode == kModeTeacher ? (P.P + P.NS - 1) / P.NS + 1 : P.n_frames * (P.G - 1) + 1);
  const int per_pass = 4 * P.L + 1;  // weight phases per pass: 4 per layer + lm_heads
  int wcur = 0;                      // next weight phase of this launch to prefetch
  // Prefetch every weight phase up to index `upto` (two phases of lookahead).
  // A heads phase is only reached by the cursor inside its own pass, when the
  // pass's head list is known.
  auto advance = [&](int upto) {
    for (; wcur <= upto; ++wcur) prefetch_weight_phase<WT>(P, wcur, cs);
  };
  for (;;) {
    if (*(volatile int*)&ctl->active <= 0) break;
    if (pass >= pass_cap) {
      if (P.max_passes == 0 && blockIdx.x == 0 && threadIdx.x == 0) raise_status(&ctl->status, kStatusDevice);
      break;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      ctl->dbg_pass = pass;
      ctl->dbg_active = *(volatile int*)&ctl->active;
      ctl->dbg_gen = (int)gen;
    }
    const int parity = (pass_base + pass) & 1;
    build_pass_lists(P, parity, cs, rows);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      ctl->head_mask[parity ^ 1] = 0ull;
      ctl->passes += 1;
      ctl->weight_bytes += (long long)P.L * P.layer_bytes + (long long)cs.nheads * P.head_bytes;
      ctl->heads_applied += cs.nheads;
    }
    const int wbase = pass * per_pass;
    for (int l = 0; l < P.L; ++l) {
      advance(wbase + 4 * l + 2);
      gemv_dispatch<WT>(P, kQKV, l, cs, rows, uni);
      if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) return;
      attention_phase(P, l, cs, rows, uni);
      if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) return;
      advance(wbase + 4 * l + 3);
      gemv_dispatch<WT>(P, kO, l, cs, rows, uni);
      if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) return;
      advance(wbase + 4 * l + 4);
      gemv_dispatch<WT>(P, kGU, l, cs, rows, uni);
      if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) return;
      advance(wbase + 4 * l + 5);
      gemv_dispatch<WT>(P, kDown, l, cs, rows, uni);
      if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) return;
    }
    advance(wbase + 4 * P.L + 2);
    gemv_dispatch<WT>(P, kHeads, 0, cs, rows, uni);
    if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) return;
    if (P.mode == kModeDecode) {
      proc_phase(P, cs, rows, uni);
      if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) return;
    }
    accept_phase<WT>(P, parity ^ 1, uni, false);
    if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) return;
    ++pass;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) ctl->pass_global = pass_base + pass;
}

template __global__ void frame_kernel<float>(const __grid_constant__ FrameParams P);
template __global__ void frame_kernel<__nv_bfloat16>(const __grid_constant__ FrameParams P);

// ------------------------------------------------------------- init kernels
__global__ void init_tables_kernel(float2* rope, int G, int d, double theta, int* top_k, float* temp, int Bmax,
                                   int k, float T) {
  const int half = d / 2;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < G * half; i += gridDim.x * blockDim.x) {
    const int pos = i / half, e = i % half;
    const double freq = pow(theta, -2.0 * (double)e / (double)d);
    const double ang = (double)pos * freq;
    rope[i] = make_float2((float)cos(ang), (float)sin(ang));
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < Bmax; i += gridDim.x * blockDim.x) {
    top_k[i] = k;
    temp[i] = T;
  }
}

}  // namespace cpk

// Host-side launch helpers (used by cp_spec.cu).
namespace cpk_host {

cudaError_t launch_frame_kernel(const cpk::FrameParams& P, int grid, size_t smem, cudaStream_t stream) {
  void* args[] = {const_cast<cpk::FrameParams*>(&P)};
  const void* fn = (P.dtype == 1) ? (const void*)cpk::frame_kernel<__nv_bfloat16> : (const void*)cpk::frame_kernel<float>;
  return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(cpk::kThreads), args, smem, stream);
}

cudaError_t frame_kernel_config(int dtype, size_t smem, int* max_blocks_per_sm) {
  const void* fn = (dtype == 1) ? (const void*)cpk::frame_kernel<__nv_bfloat16> : (const void*)cpk::frame_kernel<float>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_blocks_per_sm, fn, cpk::kThreads, smem);
}

cudaError_t launch_init_tables(float2* rope, int G, int d, double theta, int* top_k, float* temp, int Bmax, int k,
                               float T, cudaStream_t stream) {
  cpk::init_tables_kernel<<<32, 256, 0, stream>>>(rope, G, d, theta, top_k, temp, Bmax, k, T);
  return cudaGetLastError();
}

}  // namespace cpk_host
