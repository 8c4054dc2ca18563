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
  const int* rpos;  // positions of the active rows (shared memory, parallel to the row list)
  int kind, layer;  // GEMV phase to run (read at run time so the code is not cloned per phase)
  // weight stream (thread 0 produces; every thread tracks `consumed` itself)
  uint64_t wbar[2];     // one mbarrier per shared-memory slot
  int issued;           // tiles issued since kernel start
  int cur_w, cur_t;     // next tile to issue: launch-relative weight phase, tile within it
  int pass;             // pass being run (launch-relative)
  int wok;              // verdict of the last slot wait
  // per-kind tile geometry of this CTA (QKV, O, gate/up, down, lm_heads):
  // pair range [tp0, tp1), pairs per tile, tiles; computed once (lm_heads once per pass)
  int tp0[5], tp1[5], tppt[5], tnt[5];
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
  // np * gridDim.x stays far below 2^32 for every supported shape
  p0 = (int)(((unsigned)np * blockIdx.x) / gridDim.x);
  p1 = (int)(((unsigned)np * (blockIdx.x + 1)) / gridDim.x);
}

// ------------------------------------------------------- weight stream
// Each CTA streams its share of every weight phase into a ring of two
// shared-memory slots with 1-D TMA bulk copies; a slot is refilled with the
// next tile of the sequence (phases of this pass, then the next pass) as soon
// as it is consumed, so weights arrive while earlier phases and barriers run.
// A tile is a run of whole pairs.  Layouts in a slot: "split" (QKV, gate/up):
// first-row block then second-row block; "adjacent" (O, down, lm_heads): the
// two rows of a pair are neighbours, as in global memory.

template <typename WT>
__device__ __forceinline__ int pair_row_bytes(const FrameParams& P, int kind) {
  return gemv_K(P, kind) * (int)sizeof(WT);
}

template <typename WT>
__device__ __forceinline__ int pairs_per_tile_calc(const FrameParams& P, int kind) {
  return max(1, P.slot_bytes / (2 * pair_row_bytes<WT>(P, kind)));
}

// Fill the tile table entry of `kind` (thread 0).
template <typename WT>
__device__ __noinline__ void tile_table_fill(const FrameParams& P, CtaShared& cs, int kind) {
  int p0, p1;
  cta_pair_range(gemv_pairs(P, kind, cs), p0, p1);
  const int ppt = pairs_per_tile_calc<WT>(P, kind);
  cs.tp0[kind] = p0;
  cs.tp1[kind] = p1;
  cs.tppt[kind] = ppt;
  cs.tnt[kind] = p1 > p0 ? (p1 - p0 + ppt - 1) / ppt : 0;
}

__device__ __forceinline__ int pairs_per_tile(const CtaShared& cs, int kind) { return cs.tppt[kind]; }
__device__ __forceinline__ int phase_tiles(const CtaShared& cs, int kind) { return cs.tnt[kind]; }
__device__ __forceinline__ void tile_pairs(const CtaShared& cs, int kind, int t, int& pa, int& pb) {
  pa = cs.tp0[kind] + t * cs.tppt[kind];
  pb = min(cs.tp1[kind], pa + cs.tppt[kind]);
}

__device__ __forceinline__ void weight_phase_of(const FrameParams& P, int w, int& kind, int& l) {
  const int idx = w % (4 * P.L + 1);
  if (idx == 4 * P.L) { kind = kHeads; l = 0; }
  else { kind = idx % 4; l = idx / 4; }
}

__device__ __forceinline__ unsigned char* slot_base(const FrameParams& P, unsigned char* slots, int slot) {
  return slots + (size_t)slot * P.slot_bytes;
}

// Thread 0: issue the bulk copies of tile (kind, l, t) into `slot`.
template <typename WT>
__device__ __noinline__ void issue_tile(const FrameParams& P, CtaShared& cs, unsigned char* slots, int slot, int kind,
                                        int l, int t) {
  int pa, pb;
  tile_pairs(cs, kind, t, pa, pb);
  const int n = pb - pa;
  const size_t K = (size_t)gemv_K(P, kind);
  const uint32_t rb = (uint32_t)(K * sizeof(WT));
  unsigned char* dst = slot_base(P, slots, slot);
  uint64_t* bar = &cs.wbar[slot];
  mbar_arrive_expect_tx(bar, 2u * rb * (uint32_t)n);
  switch (kind) {
    case kQKV: {  // pair (head hh, e): rows hh*d + e (first block) and hh*d + e + d/2 (second block)
      const int half = P.d / 2;
      for (int hh = pa / half; hh * half < pb; ++hh) {
        const int e0 = max(pa - hh * half, 0), e1 = min(pb - hh * half, half);
        const WT* base;
        int hr;
        if (hh < P.nq) { base = (const WT*)P.wq[l]; hr = hh; }
        else if (hh < P.nq + P.nkv) { base = (const WT*)P.wk[l]; hr = hh - P.nq; }
        else { base = (const WT*)P.wv[l]; hr = hh - P.nq - P.nkv; }
        const int off = hh * half + e0 - pa;
        bulk_copy_g2s(dst + (size_t)off * rb, base + ((size_t)hr * P.d + e0) * K, (uint32_t)(e1 - e0) * rb, bar);
        bulk_copy_g2s(dst + (size_t)(n + off) * rb, base + ((size_t)hr * P.d + e0 + half) * K,
                      (uint32_t)(e1 - e0) * rb, bar);
      }
      break;
    }
    case kGU:
      bulk_copy_g2s(dst, (const WT*)P.w_gate[l] + (size_t)pa * K, (uint32_t)n * rb, bar);
      bulk_copy_g2s(dst + (size_t)n * rb, (const WT*)P.w_up[l] + (size_t)pa * K, (uint32_t)n * rb, bar);
      break;
    case kO:
      bulk_copy_g2s(dst, (const WT*)P.wo[l] + (size_t)(2 * pa) * K, 2u * (uint32_t)n * rb, bar);
      break;
    case kDown:
      bulk_copy_g2s(dst, (const WT*)P.w_down[l] + (size_t)(2 * pa) * K, 2u * (uint32_t)n * rb, bar);
      break;
    default: {  // lm_heads: features 2pa .. 2pb of the needed-head list, one copy per head
      const int f0 = 2 * pa, f1 = 2 * pb;
      for (int hi = f0 / P.V; hi * P.V < f1; ++hi) {
        const int v0 = max(f0 - hi * P.V, 0), v1 = min(f1 - hi * P.V, P.V);
        bulk_copy_g2s(dst + (size_t)(hi * P.V + v0 - f0) * rb,
                      (const WT*)P.head + ((size_t)(cs.heads[hi] - 1) * P.V + v0) * K, (uint32_t)(v1 - v0) * rb, bar);
      }
    }
  }
}

// Thread 0: keep both slots filled.  `consumed` tiles have been released.
// The lm_head tiles of a later pass are never issued early (their heads are
// only known once that pass starts).
template <typename WT>
__device__ __noinline__ void refill_slots(const FrameParams& P, CtaShared& cs, unsigned char* slots, int consumed) {
  if (threadIdx.x != 0) return;
  const int per_pass = 4 * P.L + 1;
  int guard = 0;
  while (cs.issued - consumed < 2 && guard++ < 2 * per_pass + 4) {
    int kind, l;
    weight_phase_of(P, cs.cur_w, kind, l);
    if (kind == kHeads && cs.cur_w / per_pass != cs.pass) break;
    const int nt = phase_tiles(cs, kind);
    if (cs.cur_t >= nt) { cs.cur_w += 1; cs.cur_t = 0; continue; }
    issue_tile<WT>(P, cs, slots, cs.issued & 1, kind, l, cs.cur_t);
    cs.issued += 1;
    cs.cur_t += 1;
  }
}

// Stage activation rows into shared memory (optionally RMS-normalised) in
// one round trip: every thread issues 16-byte cp.async copies, then each
// warp normalises its rows in place.  bf16 weights use a split layout:
// element k of a row goes to half (k & 7) >> 2, slot 4*(k >> 3) + (k & 3),
// so a lane's 8-element weight chunk meets two conflict-free float4 reads.
// Must be called by the whole CTA.
template <typename WT>
__device__ void stage_rows(const FrameParams& P, const float* src, int ld, int K, const float* gain,
                           const int* rows, int nr, float* xs, uint64_t* wbar = nullptr, uint32_t wpar = 0,
                           int* wok = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool split = WTraits<WT>::EPC == 8;
  const int n4 = K >> 2;
  for (int i = threadIdx.x; i < nr * n4; i += kThreads) {
    const int r = i / n4, k = (i - r * n4) << 2;
    float* dst = xs + (size_t)r * K + (split ? ((k & 7) >> 2) * (K >> 1) + 4 * (k >> 3) : k);
    cp_async16(dst, src + (size_t)rows[r] * ld + k);
  }
  // optionally, thread 0 waits (bounded) for a weight tile while the copies fly;
  // the barrier below publishes its verdict
  if (wbar && threadIdx.x == 0) *wok = mbar_wait_bounded(wbar, wpar, &P.ctl->status, P.timeout_ns) ? 1 : 0;
  cp_async_wait_all();
  __syncthreads();
  if (gain) {
    for (int r = warp; r < nr; r += kWarps) {
      float* x = xs + (size_t)r * K;
      float ss = 0.0f;
      for (int i = lane * 4; i < K; i += 128) {
        const float4 v = *reinterpret_cast<const float4*>(x + i);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
      ss = warp_sum(ss);
      const float inv = 1.0f / sqrtf(ss / (float)K + P.eps);
      for (int i = lane * 4; i < K; i += 128) {
        // smem slot i holds element k of the row
        const int k = split ? (8 * ((i % (K >> 1)) >> 2) + 4 * (i / (K >> 1))) : i;
        const float4 g = __ldg(reinterpret_cast<const float4*>(gain + k));
        float4 v = *reinterpret_cast<const float4*>(x + i);
        v.x = v.x * inv * g.x; v.y = v.y * inv * g.y; v.z = v.z * inv * g.z; v.w = v.w * inv * g.w;
        *reinterpret_cast<float4*>(x + i) = v;
      }
    }
    __syncthreads();
  }
}

// A GEMV task is (pair, K-slice): one warp, at most kU 16-byte chunks of
// each of the pair's two weight rows per lane (lane owns chunks cb + lane +
// 32 j), held in registers as floats.
constexpr int kU = 4;

template <typename WT>
struct PairChunks {
  float w0[kU][WTraits<WT>::EPC], w1[kU][WTraits<WT>::EPC];
};

// Load this lane's chunks of a pair's two rows from a shared-memory tile.
template <typename WT>
__device__ __forceinline__ void gemv_load_task(const WT* r0, const WT* r1, int cb, int ce, uint4 (&u0)[kU],
                                               uint4 (&u1)[kU]) {
  constexpr int EPC = WTraits<WT>::EPC;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < kU; ++j) {
    const int c = cb + lane + 32 * j;
    u0[j] = make_uint4(0, 0, 0, 0);
    u1[j] = u0[j];
    if (c < ce) {
      u0[j] = *reinterpret_cast<const uint4*>(r0 + (size_t)c * EPC);
      u1[j] = *reinterpret_cast<const uint4*>(r1 + (size_t)c * EPC);
    }
  }
}

// Dot products of the task's chunks with staged rows 0..nr-1, four rows at
// a time with two partial sums per output (16 independent FMA chains per
// lane), reduced over the warp; lane 0 stores the two sums of row r at
// red[r] and red[RBS + r].  The accumulation order is fixed: per lane, even
// chunks and odd chunks separately, each in (chunk, element) order, then
// even + odd, then a butterfly over the lanes.
template <typename WT>
__device__ __noinline__ void gemv_task_rows(const uint4 (&u0)[kU], const uint4 (&u1)[kU], int cb, int ce,
                                            const float* xs, int K, int nr, float* red, int RBS) {
  constexpr int EPC = WTraits<WT>::EPC;
  const int lane = threadIdx.x & 31;
  float f0[kU][EPC], f1[kU][EPC];
#pragma unroll
  for (int j = 0; j < kU; ++j) { WTraits<WT>::unpack(u0[j], f0[j]); WTraits<WT>::unpack(u1[j], f1[j]); }
#pragma unroll 1
  for (int r0 = 0; r0 < nr; r0 += 4) {
    float a[4][2][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) { a[q][0][0] = a[q][0][1] = a[q][1][0] = a[q][1][1] = 0.0f; }
    const float* xr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) xr[q] = xs + (size_t)min(r0 + q, nr - 1) * K;
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int c = cb + lane + 32 * j;
      if (c < ce) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float x[EPC];
          const float4 x0 = *reinterpret_cast<const float4*>(xr[q] + 4 * c);
          x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
          if (EPC == 8) {
            const float4 x1 = *reinterpret_cast<const float4*>(xr[q] + K / 2 + 4 * c);
            x[EPC - 4] = x1.x; x[EPC - 3] = x1.y; x[EPC - 2] = x1.z; x[EPC - 1] = x1.w;
          }
#pragma unroll
          for (int e = 0; e < EPC; ++e) {
            a[q][0][j & 1] = fmaf(f0[j][e], x[e], a[q][0][j & 1]);
            a[q][1][j & 1] = fmaf(f1[j][e], x[e], a[q][1][j & 1]);
          }
        }
      }
    }
    float v[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) { v[2 * q] = a[q][0][0] + a[q][0][1]; v[2 * q + 1] = a[q][1][0] + a[q][1][1]; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    }
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (r0 + q < nr) { red[r0 + q] = v[2 * q]; red[RBS + r0 + q] = v[2 * q + 1]; }
    }
  }
}

// Epilogue of one (pair, row): writes the phase's outputs.  `pos` is the
// row's position; `rope` the staged (cos, sin) row of that position (QKV).
template <typename WT>
__device__ __noinline__ void gemv_epilogue(const FrameParams& P, int kind, int l, int p, int row, int pos,
                                              const float2* rope, float y0, float y1, const CtaShared& cs) {
  switch (kind) {
    case kQKV: {
      const int half = P.d / 2, hh = p / half, e = p % half;
      const int b = row / P.NS;
      if (hh < P.nq + P.nkv) {
        const float2 cs2 = rope[e];
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
      const int slot = hd - pos;
      if (pos >= 1 && slot >= 0 && slot <= P.ND) {
        float* dst = P.logits + ((size_t)row * (1 + P.ND) + slot) * P.V + v;
        *reinterpret_cast<float2*>(dst) = make_float2(y0, y1);
      }
    }
  }
}

// K-split of a GEMV phase: a fixed function of the shapes (never of the row
// count), so each (row, feature) is reduced in the same order in every pass.
__device__ __forceinline__ int gemv_ksplit(int nch, int npc) {
  int KS = 1;
  while (KS < kWarps && nch > KS * 32 * kU) KS *= 2;                     // <= kU chunks per lane
  while (KS < kWarps && npc * KS * 2 <= kWarps && nch / (KS * 2) >= 32) KS *= 2;  // fill the warps
  return KS;
}

// One GEMV phase over the tiles of this CTA's pair range.  Returns the
// number of weight tiles it consumed (the caller's running count).
template <typename WT>
__device__ __noinline__ int gemv_phase(const FrameParams& P, CtaShared& cs, const int* rows, float* uni,
                                       unsigned char* slots, int consumed) {
  const int kind = cs.kind, l = cs.layer;
  const int K = gemv_K(P, kind);
  const int nt = phase_tiles(cs, kind);
  if (nt == 0) return consumed;
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
  const bool split = (kind == kQKV || kind == kGU);
  const int KS = gemv_ksplit(nch, pairs_per_tile(cs, kind));
  const int ppr = kWarps / KS;  // pairs per round
  const int RB = P.RB;
  float* xs = uni;
  float* red = uni + (size_t)RB * K;  // [2 rounds][kWarps][2][RB]
  float2* srope = reinterpret_cast<float2*>(red + (size_t)2 * kWarps * 2 * RB);  // [RB][d/2]
  const int half = P.d / 2;
  const int warp = threadIdx.x >> 5;
  const int ks = warp % KS;
  const int cb = (int)(((long long)nch * ks) / KS), ce = (int)(((long long)nch * (ks + 1)) / KS);
  const int nchunks = (cs.nrows + RB - 1) / RB;
  int staged = -1;
  for (int t = 0; t < nt; ++t) {
    int pa, pb;
    tile_pairs(cs, kind, t, pa, pb);
    const int npt = pb - pa;
    const int slot = consumed & 1;
    const uint32_t par = (uint32_t)((consumed >> 1) & 1);
    const WT* tile = reinterpret_cast<const WT*>(slot_base(P, slots, slot));
    for (int ch = 0; ch < nchunks; ++ch) {
      const int rb0 = ch * RB, nr = min(RB, cs.nrows - rb0);
      if (staged != ch) {
        __syncthreads();  // the previous chunk is done with xs / srope / red
        if (kind == kQKV)
          for (int i = threadIdx.x; i < nr * (half / 2); i += kThreads) {
            const int r = i / (half / 2), c = i - r * (half / 2);
            cp_async16(srope + (size_t)r * half + 2 * c, P.rope + (size_t)cs.rpos[rb0 + r] * half + 2 * c);
          }
        // thread 0 also waits (bounded) for this tile; stage_rows' barriers publish the verdict
        stage_rows<WT>(P, src, ld, K, gain, rows + rb0, nr, xs, ch == 0 ? &cs.wbar[slot] : nullptr, par, &cs.wok);
        staged = ch;
      } else if (ch == 0) {
        if (threadIdx.x == 0) cs.wok = mbar_wait_bounded(&cs.wbar[slot], par, &P.ctl->status, P.timeout_ns) ? 1 : 0;
        __syncthreads();
      }
      if (ch == 0) {
        if (!cs.wok) return -1;
        while (!mbar_try_wait(&cs.wbar[slot], par)) {  // completed: every thread acquires the TMA writes
        }
      }
      const int rounds = (npt + ppr - 1) / ppr;
      for (int rd = 0; rd < rounds; ++rd) {
        float* rbuf = red + (size_t)(rd & 1) * kWarps * 2 * RB;
        const int g = rd * ppr + warp / KS;  // pair within the tile
        if (g < npt) {
          const WT *r0, *r1;
          if (split) { r0 = tile + (size_t)g * K; r1 = tile + (size_t)(npt + g) * K; }
          else { r0 = tile + (size_t)(2 * g) * K; r1 = r0 + K; }
          uint4 u0[kU], u1[kU];
          gemv_load_task<WT>(r0, r1, cb, ce, u0, u1);
          gemv_task_rows<WT>(u0, u1, cb, ce, xs, K, nr, rbuf + (size_t)warp * 2 * RB, RB);
        }
        __syncthreads();  // rbuf complete; the other buffer is free for the next round
        // finish: sum the K-split partials in order, then the epilogue
        for (int i = threadIdx.x; i < ppr * nr; i += kThreads) {
          const int gi = i / nr, r = i - gi * nr;
          const int gg = rd * ppr + gi;
          if (gg >= npt) continue;
          float y0 = 0.0f, y1 = 0.0f;
          for (int j = 0; j < KS; ++j) {
            y0 += rbuf[((gi * KS + j) * 2 + 0) * RB + r];
            y1 += rbuf[((gi * KS + j) * 2 + 1) * RB + r];
          }
          gemv_epilogue<WT>(P, kind, l, pa + gg, rows[rb0 + r], cs.rpos[rb0 + r], srope + (size_t)r * half, y0, y1, cs);
        }
      }
      __syncthreads();  // tile rows and xs no longer read
    }
    // the slot is free: refill it with the next tile of the sequence
    ++consumed;
    refill_slots<WT>(P, cs, slots, consumed);
  }
  return consumed;
}

template <typename WT>
__device__ int gemv_dispatch(const FrameParams& P, int kind, int l, CtaShared& cs, const int* rows, float* uni,
                             unsigned char* slots, int consumed) {
  if (threadIdx.x == 0) { cs.kind = kind; cs.layer = l; }
  __syncthreads();
  return gemv_phase<WT>(P, cs, rows, uni, slots, consumed);
}

// Causal GQA attention of every (row, query head) over positions 0..pos,
// one warp per item.  The query and 16-position blocks of keys and values
// are staged into warp-private shared memory with cp.async (one memory round
// trip per block); lane j scores position j of a block, lanes then split the
// head dimension for the weighted sum.  Orders are fixed for every row.
__device__ __noinline__ void attention_phase(const FrameParams& P, int l, const CtaShared& cs, const int* rows,
                                             float* uni) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= P.attn_warps) return;
  const int d = P.d, grp = P.nq / P.nkv;
  float* sq = uni + (size_t)warp * (33 * d + 64);  // [d] query, [16][d] keys, [16][d] values, [64] scores
  float* sk = sq + d;
  float* sv = sk + 16 * d;
  float* sw = sv + 16 * d;
  const float scale = 1.0f / sqrtf((float)d);
  const size_t pos_stride = (size_t)P.nkv * d;
  const int items = cs.nrows * P.nq;
  for (int it = blockIdx.x * P.attn_warps + warp; it < items; it += gridDim.x * P.attn_warps) {
    const int r = rows[it / P.nq], hq = it % P.nq, g = hq / grp;
    const int b = r / P.NS;
    const int pos = cs.rpos[it / P.nq];
    const float* kb = P.kv + ((((size_t)b * P.L + l) * 2 + 0) * P.G) * pos_stride + (size_t)g * d;
    const float* vb = P.kv + ((((size_t)b * P.L + l) * 2 + 1) * P.G) * pos_stride + (size_t)g * d;
    warp_copy_async(sq, P.qbuf + (size_t)r * P.nq * d + (size_t)hq * d, d * 4);
    float mx = -INFINITY;
    for (int j0 = 0; j0 <= pos; j0 += 16) {
      const int nb = min(16, pos + 1 - j0);
      for (int jj = 0; jj < nb; ++jj) warp_copy_async(sk + jj * d, kb + (size_t)(j0 + jj) * pos_stride, d * 4);
      if (j0 == 0)
        for (int jj = 0; jj < nb; ++jj) warp_copy_async(sv + jj * d, vb + (size_t)jj * pos_stride, d * 4);
      cp_async_wait_all();
      __syncwarp();
      if (lane < nb) {
        const float* kr = sk + lane * d;
        float sdot = 0.0f;
#pragma unroll 4
        for (int e = 0; e < d; e += 4) {
          const float4 kk = *reinterpret_cast<const float4*>(kr + e);
          const float4 qq = *reinterpret_cast<const float4*>(sq + e);
          sdot = fmaf(qq.x, kk.x, sdot); sdot = fmaf(qq.y, kk.y, sdot);
          sdot = fmaf(qq.z, kk.z, sdot); sdot = fmaf(qq.w, kk.w, sdot);
        }
        sw[j0 + lane] = sdot * scale;
      }
      __syncwarp();
    }
    for (int j = 0; j <= pos; ++j) mx = fmaxf(mx, sw[j]);
    float den = 0.0f;
    for (int j = 0; j <= pos; ++j) den += expf(sw[j] - mx);  // same order in every lane
    float4 o[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int j0 = 0; j0 <= pos; j0 += 16) {
      const int nb = min(16, pos + 1 - j0);
      if (j0 > 0) {
        __syncwarp();
        for (int jj = 0; jj < nb; ++jj) warp_copy_async(sv + jj * d, vb + (size_t)(j0 + jj) * pos_stride, d * 4);
        cp_async_wait_all();
        __syncwarp();
      }
      for (int jj = 0; jj < nb; ++jj) {
        const float w = expf(sw[j0 + jj] - mx) / den;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int e = 4 * (lane + 32 * c);
          if (e < d) {
            const float4 vv = *reinterpret_cast<const float4*>(sv + jj * d + e);
            o[c].x = fmaf(w, vv.x, o[c].x); o[c].y = fmaf(w, vv.y, o[c].y);
            o[c].z = fmaf(w, vv.z, o[c].z); o[c].w = fmaf(w, vv.w, o[c].w);
          }
        }
      }
    }
    float* ov = P.obuf + (size_t)r * P.nq * d + (size_t)hq * d;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int e = 4 * (lane + 32 * c);
      if (e < d) *reinterpret_cast<float4*>(ov + e) = o[c];
    }
    __syncwarp();
  }
}

// Exclusive block-wide prefix sum of one int per thread (all threads call).
__device__ __forceinline__ int block_exclusive_scan(int v, int* sscan, int& total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sscan[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int w = 0; w < kWarps; ++w) { const int t = sscan[w]; sscan[w] = acc; acc += t; }
    sscan[kWarps] = acc;
  }
  __syncthreads();
  total = sscan[kWarps];
  const int r = sscan[warp] + incl - v;
  __syncthreads();
  return r;
}

// One vocabulary row processed by the whole CTA: the same semantics as
// warp_process_row (z = fl32(logit/T), exact top-k by (z desc, index asc)
// with an MSB-first radix select, float64 softmax summed in index order).
// Thread t owns indices [t*E, t*E + E) so the compaction is in index order.
// Returns the list length.
__device__ __noinline__ int block_process_row(const float* __restrict__ logits, int V, int k, float T,
                                              uint32_t* keys, int* sscan, double* ebuf, int* out_idx,
                                              float* out_prob) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_sel[4];
  __shared__ double s_sum;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* row = reinterpret_cast<float*>(keys);
  // stage the row (16-byte async copies when aligned)
  int done = 0;
  if ((((uintptr_t)logits) & 15u) == 0) {
    done = V & ~3;
    for (int i = tid * 4; i < done; i += kThreads * 4) cp_async16(row + i, logits + i);
  }
  for (int i = done + tid; i < V; i += kThreads) row[i] = __ldcg(logits + i);
  cp_async_wait_all();
  __syncthreads();
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
    float* sbest = reinterpret_cast<float*>(sscan + kWarps + 1);
    int* sbi = sscan + 2 * (kWarps + 1);
    if (lane == 0) { sbest[warp] = best; sbi[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
      float b = sbest[0];
      int ix = sbi[0];
      for (int w = 1; w < kWarps; ++w)
        if (sbest[w] > b || (sbest[w] == b && sbi[w] < ix)) { b = sbest[w]; ix = sbi[w]; }
      out_idx[0] = ix;
      out_prob[0] = 1.0f;
    }
    __syncthreads();
    return 1;
  }
  uint32_t kmax = 0;
  for (int i = i0; i < i1; ++i) {
    float z = __fdiv_rn(row[i], T);
    if (z == 0.0f) z = 0.0f;
    const uint32_t key = float_key(z);
    keys[i] = key;
    kmax = max(kmax, key);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  if (lane == 0) sscan[warp] = (int)kmax;
  __syncthreads();
  if (tid == 0) {
    uint32_t m = 0;
    for (int w = 0; w < kWarps; ++w) m = max(m, (uint32_t)sscan[w]);
    s_sel[3] = m;
  }
  __syncthreads();
  kmax = s_sel[3];
  const int kk = k < V ? k : V;
  uint32_t prefix = 0, mask = 0;
  int need = kk;
  bool eq_all = (kk == V);
  for (int shift = 24; shift >= 0 && !eq_all; shift -= 8) {
    hist[tid & 255] = 0;
    __syncthreads();
    for (int i = i0; i < i1; ++i) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t cnt[8];
      uint32_t chunk = 0;
#pragma unroll
      for (int m = 0; m < 8; ++m) { cnt[m] = hist[255 - 8 * lane - m]; chunk += cnt[m]; }
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
          if (acc + cnt[m] >= (uint32_t)need) { s_sel[0] = 255 - 8 * lane - m; s_sel[1] = acc; s_sel[2] = cnt[m]; break; }
          acc += cnt[m];
        }
      }
    }
    __syncthreads();
    const uint32_t bin = s_sel[0], above = s_sel[1], cbin = s_sel[2];
    need -= (int)above;
    prefix |= bin << shift;
    mask |= 0xFFu << shift;
    if ((int)cbin == need) eq_all = true;
    __syncthreads();
  }
  // rank among keys equal to the threshold (index order), then compaction
  int n_eq = 0;
  for (int i = i0; i < i1; ++i) n_eq += ((keys[i] & mask) == prefix);
  int tot;
  int eq_before = block_exclusive_scan(n_eq, sscan, tot);
  int n_sel = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t km = keys[i] & mask;
    if (km > prefix) ++n_sel;
    else if (km == prefix) { if (eq_all || eq_before < need) ++n_sel; ++eq_before; }
  }
  int sel_before = block_exclusive_scan(n_sel, sscan, tot);
  eq_before = block_exclusive_scan(n_eq, sscan, tot);
  const double zmax = (double)key_float(kmax);
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = keys[i];
    const uint32_t km = key & mask;
    bool sel = km > prefix;
    if (km == prefix) { sel = eq_all || eq_before < need; ++eq_before; }
    if (sel) {
      out_idx[sel_before] = i;
      ebuf[sel_before] = exp((double)key_float(key) - zmax);
      ++sel_before;
    }
  }
  __syncthreads();
  if (tid == 0) {
    double S = 0.0;
    for (int p = 0; p < kk; ++p) S = __dadd_rn(S, ebuf[p]);
    s_sum = S;
  }
  __syncthreads();
  const double S = s_sum;
  for (int p = tid; p < kk; p += kThreads) out_prob[p] = __double2float_rn(__ddiv_rn(ebuf[p], S));
  __syncthreads();
  return kk;
}

// Top-k / temperature / softmax of every (row, slot) vocabulary row, one CTA
// per row.
__device__ __noinline__ void proc_phase(const FrameParams& P, const CtaShared& cs, const int* rows, float* uni) {
  const size_t keys_bytes = ((size_t)P.V * 4 + 15) / 16 * 16;
  uint32_t* keys = reinterpret_cast<uint32_t*>(uni);
  int* sscan = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(uni) + keys_bytes);  // 3*(kWarps+1) ints
  double* ebuf = reinterpret_cast<double*>(reinterpret_cast<unsigned char*>(uni) + keys_bytes + 128);
  const int slots = 1 + P.ND;
  const int items = cs.nrows * slots;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int r = rows[it / slots], t = it % slots;
    const int pos = cs.rpos[it / slots];
    if (pos < 1 || pos + t > P.G - 1) continue;
    const int b = r / P.NS;
    const size_t li = (size_t)r * slots + t;
    const int n = block_process_row(P.logits + li * P.V, P.V, P.top_k[b], P.temp[b], keys, sscan, ebuf,
                                    P.lidx + li * P.KC, P.lprob + li * P.KC);
    if (threadIdx.x == 0) P.lcount[li] = n;
  }
}

// ------------------------------------------------------ per-stream logic
// Write the input rows of the next pass into the residual buffer: x at
// position 0, E_{pos-1}(code) otherwise, as float32.  All m rows are gathered
// together with 16-byte loads, 8 in flight per lane.
template <typename WT>
__device__ __noinline__ void stage_input_rows(const FrameParams& P, int b, int pos0, int m, const int* codes_in, const float* x) {
  const int lane = threadIdx.x & 31;
  constexpr int EPC = WTraits<WT>::EPC;
  const int cpr = P.H / EPC;  // 16-byte chunks per embedding row
  const int total = m * cpr;
  for (int c0 = lane; c0 < total; c0 += 32 * 8) {
    uint4 u[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = c0 + 32 * j;
      if (c < total) {
        const int i = c / cpr, k = (c - i * cpr) * EPC, pos = pos0 + i;
        const void* src;
        if (pos == 0) src = x + k;  // EPC floats of x: for bf16 two float4 loads below
        else src = (const WT*)P.embed + ((size_t)(pos - 1) * P.V + codes_in[i]) * P.H + k;
        u[j] = (pos == 0) ? make_uint4(0, 0, 0, 0) : ldg_stream(src);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = c0 + 32 * j;
      if (c >= total) break;
      const int i = c / cpr, k = (c - i * cpr) * EPC, pos = pos0 + i;
      float* dst = P.h + (size_t)(b * P.NS + i) * P.H + k;
      if (pos == 0) {
#pragma unroll
        for (int q = 0; q < EPC; q += 4)
          *reinterpret_cast<float4*>(dst + q) = __ldg(reinterpret_cast<const float4*>(x + k + q));
      } else {
        float f[EPC];
        WTraits<WT>::unpack(u[j], f);
#pragma unroll
        for (int q = 0; q < EPC; q += 4) *reinterpret_cast<float4*>(dst + q) = make_float4(f[q], f[q + 1], f[q + 2], f[q + 3]);
      }
    }
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
__device__ __noinline__ void stage_pass_rows(const FrameParams& P, int b, StreamState& S, const int* codes_in,
                                const float* x, int parity_next) {
  const int lane = threadIdx.x & 31;
  if (lane < P.NS) P.row_pos[b * P.NS + lane] = lane < S.m ? S.pos0 + lane : -1;
  stage_input_rows<WT>(P, b, S.pos0, S.m, codes_in, x);
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
__device__ __noinline__ void setup_frame(const FrameParams& P, int b, StreamState& S, int frame, int parity_next) {
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
__device__ __noinline__ void setup_teacher_chunk(const FrameParams& P, int b, StreamState& S, int parity_next) {
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

// Per-warp view of the accept scratch (see accept_scratch_bytes).
struct AcceptScratch {
  StreamState* S;
  int* idx;    // [2*NS][KC]
  float* prob; // [2*NS][KC]
  int* cnt;    // [2*NS]
};

__device__ __forceinline__ AcceptScratch accept_scratch(const FrameParams& P, float* uni) {
  const int warp = threadIdx.x >> 5;
  unsigned char* base = reinterpret_cast<unsigned char*>(uni) + (size_t)warp * accept_scratch_bytes(P.NS, P.KC);
  AcceptScratch a;
  a.S = reinterpret_cast<StreamState*>(base);
  a.idx = reinterpret_cast<int*>(base + sizeof(StreamState));
  a.prob = reinterpret_cast<float*>(a.idx + (size_t)2 * P.NS * P.KC);
  a.cnt = reinterpret_cast<int*>(a.prob + (size_t)2 * P.NS * P.KC);
  return a;
}

// Issue the async copy of one global list (capacity KC) into scratch slot `slot`.
__device__ __forceinline__ void stage_list_async(const FrameParams& P, AcceptScratch& A, int slot, const int* gidx,
                                                 const float* gprob) {
  warp_copy_async(A.idx + (size_t)slot * P.KC, gidx, P.KC * 4);
  warp_copy_async(A.prob + (size_t)slot * P.KC, gprob, P.KC * 4);
}

// After codes up to depth s_new are committed: finish the frame or stage the next pass.
template <typename WT>
__device__ __noinline__ void after_commit(const FrameParams& P, int b, AcceptScratch& A, int s_new, int hrow, int parity_next) {
  StreamState& S = *A.S;
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
  // The draft distributions q_t = proc(head_{s+t} . h_s), t = 1..n_d, are
  // this pass's speculative draft slots on the row at position s_new: stage
  // them, sample the drafts, and keep them for the next pass's acceptance.
  int cnt = 0;
  if (lane < n_d) cnt = __ldcg(P.lcount + (size_t)hrow * slots + 1 + lane);
  for (int t = 1; t <= n_d; ++t) {
    const size_t li = (size_t)hrow * slots + t;
    stage_list_async(P, A, t - 1, P.lidx + li * P.KC, P.lprob + li * P.KC);
  }
  if (lane < n_d) A.cnt[lane] = cnt;
  cp_async_wait_all();
  __syncwarp();
  if (lane == 0) {
    for (int t = 1; t <= n_d; ++t) {
      const float u = philox_uniform(P.seed, (uint32_t)b, (uint32_t)S.frame_abs, (uint32_t)(s_new + t), kDraft);
      S.drafts[t - 1] = valid_code(P, list_sample(A.idx + (size_t)(t - 1) * P.KC, A.prob + (size_t)(t - 1) * P.KC,
                                                  A.cnt[t - 1], u));
    }
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
    reinterpret_cast<int4*>(P.qidx + qi)[c] = reinterpret_cast<const int4*>(A.idx + (size_t)t * P.KC)[c];
    reinterpret_cast<float4*>(P.qprob + qi)[c] = reinterpret_cast<const float4*>(A.prob + (size_t)t * P.KC)[c];
  }
  if (lane < n_d) P.qcount[(size_t)b * P.ND + lane] = A.cnt[lane];
  __syncwarp();
  int codes_in[CP_SPEC_MAX_WINDOW];
  const int m = S.m;
  codes_in[0] = S.codes[s_new];
  for (int i = 1; i < m; ++i) codes_in[i] = S.drafts[i - 1];
  stage_pass_rows<WT>(P, b, S, codes_in, nullptr, parity_next);
}

template <typename WT>
__device__ void accept_stream(const FrameParams& P, int b, AcceptScratch& A, int parity_next) {
  StreamState& S = *A.S;
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
  // Stage the lists this decision reads: the target rows' slot-0 lists
  // (p_{s+1..s+m}) and, for a speculative round, the saved draft lists q_t.
  const bool spec = S.phase == kPhaseSpec;
  const int nl = spec ? S.m + S.n_d : 1;
  const int row0 = b * P.NS + (S.phase == kPhasePrefill ? 1 : 0);
  int cnt = 0;
  if (spec) {
    if (lane < S.m) cnt = __ldcg(P.lcount + (size_t)(b * P.NS + lane) * slots);
    else if (lane < nl) cnt = __ldcg(P.qcount + (size_t)b * P.ND + (lane - S.m));
    for (int i = 0; i < S.m; ++i) {
      const size_t li = (size_t)(b * P.NS + i) * slots;
      stage_list_async(P, A, i, P.lidx + li * P.KC, P.lprob + li * P.KC);
    }
    for (int t = 0; t < S.n_d; ++t) {
      const size_t qi = ((size_t)b * P.ND + t) * P.KC;
      stage_list_async(P, A, S.m + t, P.qidx + qi, P.qprob + qi);
    }
  } else {
    if (lane == 0) cnt = __ldcg(P.lcount + (size_t)row0 * slots);
    stage_list_async(P, A, 0, P.lidx + (size_t)row0 * slots * P.KC, P.lprob + (size_t)row0 * slots * P.KC);
  }
  if (lane < nl) A.cnt[lane] = cnt;
  cp_async_wait_all();
  __syncwarp();
  const int* Li = A.idx;
  const float* Lp = A.prob;
  const int KC = P.KC;
  int s_new = 0, hrow = 0;
  if (lane == 0) {
    const uint32_t fr = (uint32_t)S.frame_abs;
    const int s = S.s;
    if (!spec) {
      const int j = s + 1;  // the pass scored c_j
      const float u = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)j, kTarget);
      const int c = valid_code(P, list_sample(Li, Lp, A.cnt[0], u));
      S.codes[j] = c;
      P.codes_out[((size_t)S.frame * P.B + b) * P.G + j] = c;
      s_new = j;
      hrow = row0;
      ss->passes += 1;
    } else {  // speculative round: exact left-to-right acceptance
      const int n_d = S.n_d, m = S.m;
      int t = 1;
      bool rejected = false;
      for (; t <= n_d; ++t) {
        const int y = S.drafts[t - 1];
        const int qs = m + t - 1, ps = t - 1;  // scratch slots of q_t and p_{s+t}
        const float qy = list_lookup(Li + (size_t)qs * KC, Lp + (size_t)qs * KC, A.cnt[qs], y);
        const float py = list_lookup(Li + (size_t)ps * KC, Lp + (size_t)ps * KC, A.cnt[ps], y);
        const float ratio = __fdiv_rn(py, qy);
        ss->drafted[t] += 1;
        const float ua = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + t), kAccept);
        if (ua < ratio) {
          S.codes[s + t] = y;
          ss->accepted[t] += 1;
          continue;
        }
        const float ut = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + t), kTarget);
        int c = residual_sample(Li + (size_t)ps * KC, Lp + (size_t)ps * KC, A.cnt[ps], Li + (size_t)qs * KC,
                                Lp + (size_t)qs * KC, A.cnt[qs], ut);
        if (c < 0) c = list_sample(Li + (size_t)ps * KC, Lp + (size_t)ps * KC, A.cnt[ps], ut);
        S.codes[s + t] = valid_code(P, c);
        rejected = true;
        break;
      }
      if (rejected) {
        s_new = s + t;
        ss->rejections += 1;
      } else if (m > n_d) {
        const float ut = philox_uniform(P.seed, (uint32_t)b, fr, (uint32_t)(s + n_d + 1), kTarget);
        S.codes[s + n_d + 1] =
            valid_code(P, list_sample(Li + (size_t)n_d * KC, Lp + (size_t)n_d * KC, A.cnt[n_d], ut));
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
  after_commit<WT>(P, b, A, s_new, hrow, parity_next);
  store_state(P, b, S);
}

template <typename WT>
__device__ __noinline__ void accept_phase(const FrameParams& P, int parity_next, float* uni, bool setup) {
  const int warp = threadIdx.x >> 5;
  if (warp >= P.accept_warps) return;
  AcceptScratch A = accept_scratch(P, uni);
  StreamState& S = *A.S;
  for (int b = blockIdx.x + gridDim.x * warp; b < P.B; b += gridDim.x * P.accept_warps) {
    if (setup) {
      for (int i = threadIdx.x & 31; i < (int)(sizeof(StreamState) / 4); i += 32) reinterpret_cast<int*>(&S)[i] = 0;
      __syncwarp();
      if (P.mode == kModeTeacher) {
        if ((threadIdx.x & 31) == 0) { S.frame_abs = P.first_frame; S.pos0 = 0; }
        setup_teacher_chunk<WT>(P, b, S, parity_next);
      } else {
        setup_frame<WT>(P, b, S, 0, parity_next);
      }
      store_state(P, b, S);
    } else {
      accept_stream<WT>(P, b, A, parity_next);
    }
  }
}

// Active rows of the pass, their positions and the lm_heads the pass needs,
// identical in every CTA (rows[] and rpos[] live in shared memory).
__device__ __noinline__ void build_pass_lists(const FrameParams& P, int parity, CtaShared& cs, int* rows, int* rpos) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const unsigned lt = (1u << lane) - 1u;
    int n = 0;
    const int total = P.B * P.NS;
    const unsigned long long mask = __ldcg(&P.ctl->head_mask[parity]);
    for (int j0 = 0; j0 < total; j0 += 32) {
      const int r = j0 + lane;
      const int pos = r < total ? __ldcg(P.row_pos + r) : -1;
      const bool on = pos >= 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, on);
      if (on) { rows[n + __popc(bal & lt)] = r; rpos[n + __popc(bal & lt)] = pos; }
      n += __popc(bal);
    }
    if (lane == 0) {
      cs.nrows = n;
      cs.rpos = rpos;
      int nh = 0;
      for (int hd = 1; hd < P.G && hd < 64; ++hd)
        if ((mask >> hd) & 1ull) cs.heads[nh++] = hd;
      cs.nheads = nh;
    }
  }
  __syncthreads();
}

// Grid barrier that also charges the elapsed critical-path time since the
// previous barrier exit to phase `kind` (measured by CTA 0, %globaltimer,
// accumulated in registers and flushed when the kernel ends).
struct PhaseClock {
  uint64_t last;
  long long ns[8];
};

__device__ __forceinline__ bool phase_barrier(Control* ctl, unsigned long long& gen, uint64_t timeout_ns, int kind,
                                              PhaseClock& clk) {
  if (!grid_barrier(&ctl->bar, &ctl->status, gen, timeout_ns)) return false;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const uint64_t now = globaltimer_ns();
    clk.ns[kind] += (long long)(now - clk.last);
    clk.last = now;
  }
  return true;
}

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) frame_kernel(const __grid_constant__ FrameParams Pg) {
  // The parameter block is copied to shared memory once: every phase reads
  // its fields through a reference, and a generic reference into the
  // parameter buffer would become an L2 round trip after each grid barrier
  // (the barrier's acquire invalidates L1).
  __shared__ __align__(16) FrameParams sP;
  {
    const int4* src = reinterpret_cast<const int4*>(&Pg);
    int4* dst = reinterpret_cast<int4*>(&sP);
    for (int i = threadIdx.x; i < (int)(sizeof(FrameParams) / 16); i += kThreads) dst[i] = src[i];
    if (threadIdx.x == 0)
      for (size_t i = sizeof(FrameParams) / 16 * 16; i < sizeof(FrameParams); ++i)
        reinterpret_cast<char*>(&sP)[i] = reinterpret_cast<const char*>(&Pg)[i];
    __syncthreads();
  }
  const FrameParams& P = sP;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // dynamic shared memory: [active rows, their positions][2 weight slots][phase union region]
  int* rows = reinterpret_cast<int*>(smem_raw);
  int* rpos = rows + (size_t)P.B * P.NS;
  const size_t rows_bytes = ((size_t)P.B * P.NS * 8 + 127) / 128 * 128;
  unsigned char* slots = smem_raw + rows_bytes;
  float* uni = reinterpret_cast<float*>(slots + 2 * (size_t)P.slot_bytes);
  __shared__ CtaShared cs;
  Control* ctl = P.ctl;
  unsigned long long gen = 0;
  PhaseClock clk = {};    // CTA 0: per-phase critical-path time
  long long n_pass = 0, w_bytes = 0, n_heads = 0;
  const int pass_base = __ldcg(&ctl->pass_global);
  int pass = 0, consumed = 0;
  if (threadIdx.x == 0) {
    mbar_init(&cs.wbar[0], 1);
    mbar_init(&cs.wbar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    cs.issued = 0; cs.cur_w = 0; cs.cur_t = 0; cs.pass = -1; cs.nheads = 0;
    for (int kind = kQKV; kind <= kDown; ++kind) tile_table_fill<WT>(P, cs, kind);
    tile_table_fill<WT>(P, cs, kHeads);  // no heads until the first pass
  }
  __syncthreads();
  refill_slots<WT>(P, cs, slots, consumed);  // layer-0 weights stream during the setup
  if (P.do_setup) {
    if (blockIdx.x == 0 && threadIdx.x == 0) ctl->active = P.B;
    accept_phase<WT>(P, pass_base & 1, uni, true);
    if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns)) goto drain;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) clk.last = globaltimer_ns();
  {
    // Every pass commits at least one code of every unfinished stream, so a
    // decode needs at most n_frames * (G - 1) passes and a teacher run
    // ceil(P / NS); anything beyond that is a logic error, reported, not looped.
    const int pass_cap = P.max_passes > 0 ? P.max_passes
                         : (P.mode == kModeTeacher ? (P.P + P.NS - 1) / P.NS + 1 : P.n_frames * (P.G - 1) + 1);
    for (;;) {
      if (*(volatile int*)&ctl->active <= 0) break;
      if (pass >= pass_cap) {
        if (P.max_passes == 0 && blockIdx.x == 0 && threadIdx.x == 0) raise_status(&ctl->status, kStatusDevice);
        break;
      }
      const int parity = (pass_base + pass) & 1;
      build_pass_lists(P, parity, cs, rows, rpos);
      if (threadIdx.x == 0) {
        tile_table_fill<WT>(P, cs, kHeads);
        cs.pass = pass;
      }
      refill_slots<WT>(P, cs, slots, consumed);
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        ctl->head_mask[parity ^ 1] = 0ull;
        n_pass += 1;
        w_bytes += (long long)P.L * P.layer_bytes + (long long)cs.nheads * P.head_bytes;
        n_heads += cs.nheads;
      }
      for (int l = 0; l < P.L; ++l) {
        consumed = gemv_dispatch<WT>(P, kQKV, l, cs, rows, uni, slots, consumed);
        if (consumed < 0 || !phase_barrier(ctl, gen, P.timeout_ns, 0, clk)) goto drain;
        attention_phase(P, l, cs, rows, uni);
        if (!phase_barrier(ctl, gen, P.timeout_ns, 1, clk)) goto drain;
        consumed = gemv_dispatch<WT>(P, kO, l, cs, rows, uni, slots, consumed);
        if (consumed < 0 || !phase_barrier(ctl, gen, P.timeout_ns, 2, clk)) goto drain;
        consumed = gemv_dispatch<WT>(P, kGU, l, cs, rows, uni, slots, consumed);
        if (consumed < 0 || !phase_barrier(ctl, gen, P.timeout_ns, 3, clk)) goto drain;
        consumed = gemv_dispatch<WT>(P, kDown, l, cs, rows, uni, slots, consumed);
        if (consumed < 0 || !phase_barrier(ctl, gen, P.timeout_ns, 4, clk)) goto drain;
      }
      consumed = gemv_dispatch<WT>(P, kHeads, 0, cs, rows, uni, slots, consumed);
      if (consumed < 0 || !phase_barrier(ctl, gen, P.timeout_ns, 5, clk)) goto drain;
      if (P.mode == kModeDecode) {
        proc_phase(P, cs, rows, uni);
        if (!phase_barrier(ctl, gen, P.timeout_ns, 6, clk)) goto drain;
      }
      accept_phase<WT>(P, parity ^ 1, uni, false);
      if (!phase_barrier(ctl, gen, P.timeout_ns, 7, clk)) goto drain;
      ++pass;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    ctl->pass_global = pass_base + pass;
    ctl->passes += n_pass;
    ctl->weight_bytes += w_bytes;
    ctl->heads_applied += n_heads;
    for (int i = 0; i < 8; ++i) ctl->phase_ns[i] += clk.ns[i];
    ctl->dbg_pass = pass;
    ctl->dbg_gen = (int)gen;
  }
drain:
  // never leave with a bulk copy in flight into this CTA's shared memory
  __syncthreads();
  if (threadIdx.x == 0 && consumed >= 0) {
    for (int i = consumed; i < cs.issued; ++i)
      if (!mbar_wait_bounded(&cs.wbar[i & 1], (uint32_t)((i >> 1) & 1), &ctl->status, P.timeout_ns)) break;
  }
  __syncthreads();
}

template __global__ void frame_kernel<float>(const __grid_constant__ FrameParams Pg);
template __global__ void frame_kernel<__nv_bfloat16>(const __grid_constant__ FrameParams Pg);

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
