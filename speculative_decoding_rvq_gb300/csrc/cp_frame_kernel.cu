// cp_frame_kernel.cu -- the persistent CodePredictor frame kernel.
//
// One cooperative launch (one CTA per SM) runs decoder passes until every
// stream has finished its frames.  A pass is, for all streams at once:
//
//   per layer: [QKV + RoPE + KV append] -> [attention over the stream's KV]
//              -> [O + residual] -> [RMSNorm + gate/up + SwiGLU] -> [down + residual]
//   [final RMSNorm + lm_heads]  target head_j on the row at position j, and,
//                               speculatively, head_{j+1..j+N-1} on the same
//                               row: the free drafts of the next round
//                               ("CodePredictor Speculative Decoding", "Why
//                               the draft is free")
//   [top-k / temperature / softmax]   one CTA per (row, head) vocabulary row
//   [accept / commit / reconcile]     one warp per stream: exact speculative
//                               sampling ("How a round works" step 3), codes
//                               committed, draft codes for the next round
//                               sampled, KV length = s'+1
//
// Weight stream.  A CTA is 8 consumer warps and one producer warp.  The
// producer walks the CTA's fixed share of every weight matrix of the pass in
// consumption order and copies it, tile by tile, into a ring of shared-memory
// slots with 1-D TMA bulk copies (mbarrier completion).  Weights do not
// depend on activations, so the producer runs ahead of the consumers across
// phase boundaries, bounded only by the ring; the lm_heads of a pass are
// issued once the pass's head list is known.
//
// Phase hand-off.  Phase outputs go to exchange buffers of 64-bit elements
// {value, pass flag} written with one 64-bit store; a consumer reads its
// whole input vector and re-reads the elements whose flag is not yet the
// current pass's (no grid barrier, one L2 round trip once the data is
// there).  Buffers are per layer, so an element is written once per pass.
// One grid barrier per pass (after acceptance) orders the stream state, the
// KV cache of committed positions and the row lists of the next pass.
//
// GEMV.  Each CTA owns contiguous output units of every matrix.  A tile's
// rows are split into tasks of kRB weight rows x 512 input elements x up to
// 4 input rows; a lane holds 16 input elements of 4 rows in registers and
// accumulates kRB x 4 float2 partial sums with packed FMAs; a fixed butterfly
// reduce-scatter over the warp and a sum over the 512-element parts in
// index order give every (row, output) the same reduction order whatever
// rows share the pass, the tile or the CTA, so greedy speculative decoding
// reproduces greedy autoregressive decoding exactly.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "cp_common.cuh"
#include "cp_frame.cuh"
#include "cp_sampling.cuh"

namespace cpk {

// ------------------------------------------------------------ weight types
// One 16-byte chunk of a weight row in shared memory, as float2 pairs.
template <typename WT> struct WTraits;
template <> struct WTraits<float> {
  static constexpr int EB = 4;   // bytes per element
  static constexpr int EPC = 4;  // elements per 16-byte chunk
  static constexpr int JW = 4;   // 16-byte chunks per lane per task
  __device__ __forceinline__ static void load_chunk(const unsigned char* p, float2 (&w)[2]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
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
  static constexpr int JW = 2;
  __device__ __forceinline__ static void load_chunk(const unsigned char* p, float2 (&w)[4]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
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

// Shared-memory slot (in float4 units) of input element k in the staged
// activation rows: the float4s a lane reads for its chunks of a task are
// contiguous across the warp (conflict-free 16-byte loads).
template <typename WT>
__device__ __forceinline__ int act_f4(int k) {
  if (WTraits<WT>::EPC == 4) return k >> 2;
  const int c = k >> 3;
  return ((c >> 5) << 6) + (((k >> 2) & 1) << 5) + (c & 31);
}

// ------------------------------------------------------------------ sync
// Named barrier 1 over the consumer warps (the producer warp never joins).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// consumer_sync that also returns the OR of `v` over the consumer threads:
// keeps a failure verdict uniform before any later barrier.
__device__ __forceinline__ bool consumer_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kConsumers)
      : "memory");
  return r != 0;
}

// Grid-wide barrier of the consumer warps of every CTA (cooperative launch;
// `counter` is zeroed before the launch; generation g completes at g * grid).
// Bounded by timeout_ns of %globaltimer, by an iteration count and by the
// status word: on failure the status is set and false is returned.
__device__ __forceinline__ bool grid_barrier(unsigned long long* counter, int* status, unsigned long long& gen,
                                             uint64_t timeout_ns, int* s_ok) {
  consumer_sync();
  ++gen;
  if (threadIdx.x == 0) {
    bool ok = true;
    const unsigned long long target = gen * (unsigned long long)gridDim.x;
    __threadfence();
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(counter) : "memory");
    const uint64_t t0 = globaltimer_ns();
    uint32_t spins = 0;
    while (ld_acquire_u64(counter) < target) {
      ++spins;
      if ((spins & 63u) == 0) {
        const uint64_t now = globaltimer_ns();
        if (now - t0 > timeout_ns || spins > (1u << 30)) { raise_status(status, kStatusTimeout); ok = false; break; }
        if (ld_relaxed_i32(status) != 0) { ok = false; break; }
      }
      if (spins > 2048u) __nanosleep(128);
    }
    *s_ok = ok ? 1 : 0;
  }
  consumer_sync();
  return *s_ok != 0;
}

// Bounded poll helper: call every iteration; returns false once the
// deadline passed or another CTA raised the status word.
struct Deadline {
  uint64_t t0;
  uint32_t it;
  __device__ __forceinline__ void start() { t0 = 0; it = 0; }
  __device__ __forceinline__ bool ok(const FrameParams& P) {
    ++it;
    if ((it & 31u) != 0) return true;
    const uint64_t now = globaltimer_ns();
    if (t0 == 0) t0 = now;
    if (now - t0 > P.timeout_ns || it > (1u << 30)) { raise_status(&P.ctl->status, kStatusTimeout); return false; }
    if (ld_relaxed_i32(&P.ctl->status) != 0) return false;
    if (it > 256u) __nanosleep(64);
    return true;
  }
};

// ------------------------------------------------------------ tile plans
struct Tile {
  int u0, n;  // first output unit and unit count
};

// Output units of a GEMV kind: QKV = RoPE pair (e, e + d/2) of a head;
// O, down = output row; gate/up = feature (gate row + up row);
// lm_heads = (head of the pass, vocabulary row).
__device__ __forceinline__ int rows_per_unit(int kind) { return (kind == kQKV || kind == kGU) ? 2 : 1; }

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

// Tiles of this CTA's share [U*c/grid, U*(c+1)/grid) of `kind`, none wider
// than a slot or kMaxTileRows rows, none crossing a head boundary (QKV, lm_heads).
template <typename WT>
__device__ int make_tiles(const FrameParams& P, int kind, int nheads, Tile* out) {
  const int U = gemv_units(P, kind, nheads);
  const int c = blockIdx.x, g = gridDim.x;
  const int u0 = (int)(((long long)U * c) / g), u1 = (int)(((long long)U * (c + 1)) / g);
  const int rpu = rows_per_unit(kind);
  const int ub = rpu * gemv_K(P, kind) * WTraits<WT>::EB;
  int upt = P.slot_bytes / ub;
  upt = min(upt, kMaxTileRows / rpu);
  const int period = kind == kQKV ? P.d / 2 : (kind == kHeads ? P.V : 0);
  int n = 0;
  for (int u = u0; u < u1;) {
    int e = min(u1, u + upt);
    if (period > 0) e = min(e, (u / period + 1) * period);
    if (n >= kMaxTiles) { raise_status(&P.ctl->status, kStatusDevice); break; }
    out[n++] = Tile{u, e - u};
    u = e;
  }
  return n;
}

// The two (or one) contiguous byte runs of a tile in global memory.
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

// CTA-wide shared state.
struct CtaShared {
  uint64_t full[kMaxSlots];   // tile landed (TMA transaction count)
  uint64_t empty[kMaxSlots];  // tile released by all consumer warps
  Tile tab[4][kMaxTiles];     // static GEMV kinds of every layer
  int ntab[4];
  Tile htab[2][kMaxTiles];    // lm_head tiles of a pass (by pass parity)
  int nhtab[2];
  int hheads[2][64];          // the pass's heads (by pass parity), for the producer
  volatile int heads_ready;   // pass index whose head tiles are published
  volatile int stop;          // consumers are leaving: the producer stops issuing
  int tile_done[kMaxSlots];   // tasks finished per ring slot (the last one runs the epilogue)
  int nrows;                  // active rows of the pass
  int nheads;
  int heads[64];
  int own0, own1;             // owned residual rows [own0, own1) (O and down outputs)
  int s_ok;
  long long clk_ns[8];        // CTA 0: time per phase kind
  uint64_t clk_last;
  long long n_pass, w_bytes, n_heads;  // CTA 0: counters flushed at exit
  float srms[kWarps][16];     // RMSNorm partial sums per warp and staged row
  float sinv[16];
};

// ------------------------------------------------------------- producer
// Lane 0 of the producer warp.  Streams the tiles of every pass in the
// consumers' order until they raise `stop`; then waits for the copies in
// flight so no bulk copy lands after the CTA exits.
template <typename WT>
__device__ __noinline__ void producer_loop(const FrameParams& P, CtaShared& cs, unsigned char* ring) {
  uint32_t n = 0;  // tiles issued
  const uint64_t pol = l2_evict_first_policy();
  for (int pass = 0;; ++pass) {
    for (int l = 0; l < P.L; ++l) {
      for (int kind = kQKV; kind <= kDown; ++kind) {
        for (int t = 0; t < cs.ntab[kind]; ++t) {
          const uint32_t slot = n % (uint32_t)P.nslots, use = n / (uint32_t)P.nslots;
          if (use > 0) {
            while (!mbar_try_wait_hint(&cs.empty[slot], (use - 1) & 1u, 20000u)) {
              if (cs.stop) goto drain;
            }
          }
          if (cs.stop) goto drain;
          const TileRuns r = tile_runs<WT>(P, kind, l, nullptr, cs.tab[kind][t]);
          unsigned char* dst = ring + (size_t)slot * P.slot_bytes;
          mbar_arrive_expect_tx(&cs.full[slot], r.src1 ? 2 * r.bytes : r.bytes);
          bulk_copy_g2s(dst, r.src0, r.bytes, &cs.full[slot], pol);
          if (r.src1) bulk_copy_g2s(dst + r.bytes, r.src1, r.bytes, &cs.full[slot], pol);
          ++n;
        }
      }
    }
    // lm_heads of this pass: wait until the consumers published the head list
    while (cs.heads_ready < pass) {
      if (cs.stop) goto drain;
      __nanosleep(32);
    }
    __threadfence_block();
    {
      const int par = pass & 1;
      for (int t = 0; t < cs.nhtab[par]; ++t) {
        const uint32_t slot = n % (uint32_t)P.nslots, use = n / (uint32_t)P.nslots;
        if (use > 0) {
          while (!mbar_try_wait_hint(&cs.empty[slot], (use - 1) & 1u, 20000u)) {
            if (cs.stop) goto drain;
          }
        }
        if (cs.stop) goto drain;
        const TileRuns r = tile_runs<WT>(P, kHeads, 0, cs.hheads[par], cs.htab[par][t]);
        mbar_arrive_expect_tx(&cs.full[slot], r.bytes);
        bulk_copy_g2s(ring + (size_t)slot * P.slot_bytes, r.src0, r.bytes, &cs.full[slot], pol);
        ++n;
      }
    }
  }
drain:
  // the last min(n, nslots) tiles may still be in flight
  for (uint32_t i = n > (uint32_t)P.nslots ? n - P.nslots : 0; i < n; ++i) {
    const uint32_t slot = i % (uint32_t)P.nslots;
    if (!mbar_wait_bounded(&cs.full[slot], (i / (uint32_t)P.nslots) & 1u, &P.ctl->status, P.timeout_ns)) break;
  }
}

// --------------------------------------------------------- pass context
// What every consumer phase of a pass needs (shared-memory lists and views).
// It lives in shared memory: every field but `fail` is written with the same
// value by all consumer threads after a barrier; `fail` only ever goes from 0
// to 1, so no thread can overwrite another's failure.
struct PassCtx {
  const int* rows;   // active row slots (b * NS + k), ascending
  const int* rpos;   // their positions
  const int* rcode;  // their input code (frame index at position 0)
  int nr;            // active rows
  uint32_t flag;     // exchange flag of this pass
  float* uni;        // phase scratch (staged activations, top-k, acceptance, attention)
  float* red;        // GEMV partial sums of a phase (P.red_floats)
  const float2* rope;  // RoPE (cos, sin) table [G][d/2] (shared memory when it fits)
  float* hown;       // owned residual values [row][own1 - own0]
  unsigned char* ring;
  uint32_t tile_seq; // tiles consumed so far by this CTA
  volatile int fail;
};

__device__ __forceinline__ void mark_fail(PassCtx& X) { X.fail = 1; }

// Barrier over the consumer warps that also agrees on failure (v or any
// earlier mark_fail by any thread).
__device__ __forceinline__ bool agree_fail(PassCtx& X, bool v = false) {
  const bool r = consumer_sync_or(v || X.fail != 0);
  if (r) X.fail = 1;
  return r;
}

// Input element k of pass row i (x at position 0, else E_{pos-1}(code)).
template <typename WT>
__device__ __forceinline__ const void* input_row(const FrameParams& P, const PassCtx& X, int i, bool& is_x) {
  const int r = X.rows[i], pos = X.rpos[i], code = X.rcode[i];
  const int b = r / P.NS;
  if (pos == 0) {
    is_x = true;
    return P.mode == kModeTeacher ? P.x + (size_t)b * P.H : P.x + ((size_t)code * P.B + b) * P.H;
  }
  is_x = false;
  return static_cast<const WT*>(P.embed) + ((size_t)(pos - 1) * P.V + code) * P.H;
}

// Row stride (floats) of staged activations of width K.
template <typename WT>
__device__ __forceinline__ int act_stride(int K) {
  return WTraits<WT>::EPC == 8 ? (K + 255) / 256 * 256 : K;
}

// Stage rows [g0, g0 + ng) of a GEMV input (width K) into shared memory in
// act_f4 layout: from exchange buffer `xs` (row slot stride K, polled until
// every element carries this pass's flag) or, when xs is null, from the
// pass input rows; with `hown` the raw input values of the CTA's owned
// residual rows are also copied there (first layer).  With `gain`, rows are
// RMS-normalised: the sum of squares is taken in a fixed order (per thread
// in element order, a butterfly over the warp, the warps in index order),
// then x * (1/sqrt(ss/K + eps)) * gain.  Called by all consumer threads.
template <typename WT>
__device__ __noinline__ void stage_act(const FrameParams& P, CtaShared& cs, PassCtx& X, const xel* xs, int K,
                                       const float* gain, int g0, int ng, float* act, float* hown) {
  constexpr int kPollBatch = 8;
  constexpr int kGainPairs = 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int KS = act_stride<WT>(K);
  const int npair = K >> 1;
  // gains of this thread's pairs, fetched before the inputs arrive
  float2 gpre[kGainPairs];
  if (gain != nullptr) {
#pragma unroll
    for (int j = 0; j < kGainPairs; ++j) {
      const int i = tid + kConsumers * j;
      gpre[j] = i < npair ? __ldg(reinterpret_cast<const float2*>(gain) + i) : make_float2(0.f, 0.f);
    }
  }
  consumer_sync();  // earlier readers of `act` are done
  if (xs == nullptr) {
    for (int q = 0; q < ng; ++q) {
      bool is_x;
      const void* src = input_row<WT>(P, X, g0 + q, is_x);
      float* dst = act + (size_t)q * KS;
      for (int i = tid; i < npair; i += kConsumers) {
        float2 v;
        if (is_x) {
          v = __ldg(reinterpret_cast<const float2*>(src) + i);
        } else if (WTraits<WT>::EB == 2) {
          v = bf16x2_to_f2(__ldg(reinterpret_cast<const uint32_t*>(src) + i));
        } else {
          v = __ldg(reinterpret_cast<const float2*>(src) + i);
        }
        const int k = 2 * i;
        *reinterpret_cast<float2*>(dst + 4 * act_f4<WT>(k) + (k & 3)) = v;
      }
    }
  } else if (!X.fail) {
    // poll: every thread owns pairs i = tid + kConsumers * j of every row; a
    // pending bit per (row, j), at most 32 at a time
    const int ppt = (npair + kConsumers - 1) / kConsumers;
    const int rpb = max(1, 32 / ppt);  // rows per poll batch
    const int* const xrows = X.rows;
    const uint32_t flag = X.flag;
    bool failed = false;
    for (int qb = 0; qb < ng && !failed; qb += rpb) {
      const int nq = min(rpb, ng - qb);
      uint32_t pend = 0;
      for (int q = 0; q < nq; ++q)
        for (int j = 0; j < ppt; ++j)
          if (tid + kConsumers * j < npair) pend |= 1u << (q * ppt + j);
      Deadline dl;
      dl.start();
      while (pend) {
        uint32_t left = pend;
        while (left) {
          // up to kPollBatch loads in flight before any flag is checked
          int bit[kPollBatch];
          unsigned long long va[kPollBatch], vb[kPollBatch];
#pragma unroll
          for (int u = 0; u < kPollBatch; ++u) {
            bit[u] = -1;
            if (left) {
              bit[u] = __ffs(left) - 1;
              left &= left - 1;
              const int q = bit[u] / ppt, j = bit[u] - q * ppt;
              xel_load2(xs + (size_t)xrows[g0 + qb + q] * K + 2 * (tid + kConsumers * j), va[u], vb[u]);
            }
          }
#pragma unroll
          for (int u = 0; u < kPollBatch; ++u) {
            if (bit[u] >= 0 && xel_flag(va[u]) == flag && xel_flag(vb[u]) == flag) {
              const int q = bit[u] / ppt, j = bit[u] - q * ppt;
              const int k = 2 * (tid + kConsumers * j);
              *reinterpret_cast<float2*>(act + (size_t)(qb + q) * KS + 4 * act_f4<WT>(k) + (k & 3)) =
                  make_float2(xel_value(va[u]), xel_value(vb[u]));
              pend &= ~(1u << bit[u]);
            }
          }
        }
        if (pend && !dl.ok(P)) { failed = true; break; }
      }
    }
    if (failed) mark_fail(X);
  }
  agree_fail(X);
  if (hown != nullptr) {
    const int nown = cs.own1 - cs.own0;
    for (int idx = tid; idx < ng * nown; idx += kConsumers) {
      const int q = idx / nown, n = cs.own0 + (idx - q * nown);
      hown[(size_t)(g0 + q) * P.hown_cap + (n - cs.own0)] = act[(size_t)q * KS + 4 * act_f4<WT>(n) + (n & 3)];
    }
  }
  if (gain != nullptr) {
    // per-thread sums of squares over its own pairs, in element order
    for (int q0 = 0; q0 < ng; q0 += 16) {
      const int nq = min(16, ng - q0);
      for (int q = 0; q < nq; ++q) {
        const float* row = act + (size_t)(q0 + q) * KS;
        float ss = 0.0f;
        for (int i = tid; i < npair; i += kConsumers) {
          const int k = 2 * i;
          const float2 v = *reinterpret_cast<const float2*>(row + 4 * act_f4<WT>(k) + (k & 3));
          ss = fmaf(v.x, v.x, ss);
          ss = fmaf(v.y, v.y, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) cs.srms[warp][q] = ss;
      }
      consumer_sync();
      if (tid < nq) {
        float ss = 0.0f;
        for (int w = 0; w < kWarps; ++w) ss += cs.srms[w][tid];
        cs.sinv[tid] = 1.0f / sqrtf(ss / (float)K + P.eps);
      }
      consumer_sync();
      for (int q = 0; q < nq; ++q) {
        float* row = act + (size_t)(q0 + q) * KS;
        const float inv = cs.sinv[q];
#pragma unroll
        for (int j = 0; j < kGainPairs; ++j) {
          const int i = tid + kConsumers * j;
          if (i < npair) {
            const int k = 2 * i;
            float2* pv = reinterpret_cast<float2*>(row + 4 * act_f4<WT>(k) + (k & 3));
            float2 v = *pv;
            v.x = v.x * inv * gpre[j].x;
            v.y = v.y * inv * gpre[j].y;
            *pv = v;
          }
        }
        for (int i = tid + kConsumers * kGainPairs; i < npair; i += kConsumers) {
          const int k = 2 * i;
          float2* pv = reinterpret_cast<float2*>(row + 4 * act_f4<WT>(k) + (k & 3));
          const float2 g = __ldg(reinterpret_cast<const float2*>(gain) + i);
          float2 v = *pv;
          v.x = v.x * inv * g.x;
          v.y = v.y * inv * g.y;
          *pv = v;
        }
      }
      consumer_sync();  // cs.srms / cs.sinv reuse
    }
  }
}

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

// One GEMV task: weight rows [kRB*b, kRB*b + kRB) of a tile (rows of nch
// 16-byte chunks) times input rows q0..q0+NQ-1 over input part kp.  Rows past
// the tile's end and input rows past nqv are read (in bounds: the row index
// is clamped, the ring is followed by scratch) and their sums discarded, so
// the loads carry no branches.  CHECK guards chunks past the row end when the
// width is not a multiple of the input part.  The lane's chunks are taken one
// at a time (input rows of the chunk in registers, then the weight rows),
// accumulating each (weight row, input row) in a fixed order.  Writes
// kRedPerTask partial sums (index w * 4 + q) to `out`.
template <typename WT, int NQ, bool CHECK>
__device__ __forceinline__ void gemv_task(const unsigned char* tile, int nch, int b, int kp, const float* act, int KS,
                                          int q0, int nqv, float* out) {
  constexpr int JW = WTraits<WT>::JW;
  constexpr int PPC = WTraits<WT>::EPC / 2;  // float2 pairs per chunk
  const int lane = threadIdx.x & 31;
  const size_t row_bytes = (size_t)nch * 16;
  const unsigned char* wrow = tile + (size_t)(kRB * b) * row_bytes;
  const float4* arow[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) arow[q] = reinterpret_cast<const float4*>(act + (size_t)(q0 + min(q, nqv - 1)) * KS);
  float2 acc[kRB][NQ];
#pragma unroll
  for (int w = 0; w < kRB; ++w)
#pragma unroll
    for (int q = 0; q < NQ; ++q) acc[w][q] = make_float2(0.f, 0.f);
#pragma unroll 1
  for (int j = 0; j < JW; ++j) {
    const int c = kp * 32 * JW + 32 * j + lane;
    if (CHECK && c >= nch) continue;
    float2 a[NQ][PPC];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (PPC == 4) {
        const float4 lo = arow[q][(kp * JW + j) * 64 + lane], hi = arow[q][(kp * JW + j) * 64 + 32 + lane];
        a[q][0] = make_float2(lo.x, lo.y);
        a[q][1] = make_float2(lo.z, lo.w);
        a[q][PPC - 2] = make_float2(hi.x, hi.y);
        a[q][PPC - 1] = make_float2(hi.z, hi.w);
      } else {
        const float4 v = arow[q][c];
        a[q][0] = make_float2(v.x, v.y);
        a[q][PPC - 1] = make_float2(v.z, v.w);
      }
    }
#pragma unroll
    for (int w = 0; w < kRB; ++w) {
      float2 wv[PPC];
      WTraits<WT>::load_chunk(wrow + (size_t)w * row_bytes + (size_t)c * 16, wv);
#pragma unroll
      for (int q = 0; q < NQ; ++q)
#pragma unroll
        for (int p = 0; p < PPC; ++p) acc[w][q] = ffma2(wv[p], a[q][p], acc[w][q]);
    }
  }
  float v[kRB * NQ];
#pragma unroll
  for (int w = 0; w < kRB; ++w)
#pragma unroll
    for (int q = 0; q < NQ; ++q) v[w * NQ + q] = acc[w][q].x + acc[w][q].y;
  const float sum = reduce_scatter<kRB * NQ>(v);
  constexpr int NV = kRB * NQ;
  constexpr int shift = NV >= 32 ? 0 : (NV >= 16 ? 1 : (NV >= 8 ? 2 : (NV >= 4 ? 3 : 4)));
  if ((lane & ((1 << shift) - 1)) == 0) {
    const int vi = lane >> shift;
    out[(vi / NQ) * 4 + (vi % NQ)] = sum;
  }
}

// ------------------------------------------------------------ GEMV phase
__device__ __forceinline__ size_t row_slots(const FrameParams& P) { return (size_t)P.Bmax * P.NS; }

// Units per tile of a kind (the same rule as make_tiles) and the partial-sum
// floats one tile needs.
template <typename WT>
__device__ __forceinline__ int units_per_tile(const FrameParams& P, int kind) {
  const int rpu = rows_per_unit(kind);
  return min(P.slot_bytes / (rpu * gemv_K(P, kind) * WTraits<WT>::EB), kMaxTileRows / rpu);
}

// Outputs of one unit for staged row gi: RoPE + q / KV append (QKV),
// residual update and publication (O, down), SwiGLU (gate/up), logits (lm_heads).
template <typename WT>
__device__ __forceinline__ void gemv_out(const FrameParams& P, const CtaShared& cs, const PassCtx& X, int kind, int l,
                                         int u, int gi, float y0, float y1) {
  const size_t RS = row_slots(P);
  const int r = X.rows[gi], pos = X.rpos[gi];
  switch (kind) {
    case kQKV: {
      const int half = P.d / 2, hh = u / half, e = u - hh * half;
      const int b = r / P.NS;
      if (hh < P.nq + P.nkv) {
        const float2 cs2 = X.rope[(size_t)pos * half + e];
        const float r0 = y0 * cs2.x - y1 * cs2.y;
        const float r1 = y1 * cs2.x + y0 * cs2.y;
        if (hh < P.nq) {
          xel* qd = P.qpub + ((size_t)l * RS + r) * P.nq * P.d + (size_t)hh * P.d;
          xel_store(qd + e, r0, X.flag);
          xel_store(qd + e + half, r1, X.flag);
        } else {
          xel* kd = P.kv + (((((size_t)b * P.L + l) * 2 + 0) * P.G + pos) * P.nkv + (hh - P.nq)) * P.d;
          xel_store(kd + e, r0, X.flag);
          xel_store(kd + e + half, r1, X.flag);
        }
      } else {
        xel* vd = P.kv + (((((size_t)b * P.L + l) * 2 + 1) * P.G + pos) * P.nkv + (hh - P.nq - P.nkv)) * P.d;
        xel_store(vd + e, y0, X.flag);
        xel_store(vd + e + half, y1, X.flag);
      }
      break;
    }
    case kO:
    case kDown: {
      float* hv = X.hown + (size_t)gi * P.hown_cap + (u - cs.own0);
      const float nv = *hv + y0;
      *hv = nv;
      xel_store(P.hpub + (((size_t)l * 2 + (kind == kDown ? 1 : 0)) * RS + r) * P.H + u, nv, X.flag);
      break;
    }
    case kGU: {
      const float a = y0 / (1.0f + expf(-y0)) * y1;
      xel_store(P.apub + ((size_t)l * RS + r) * P.F + u, a, X.flag);
      break;
    }
    default: {
      const int hi = u / P.V, v = u - hi * P.V;
      const int slot = cs.heads[hi] - pos;
      if (pos >= 1 && slot >= 0 && slot <= P.ND)
        xel_store(P.logits + ((size_t)r * (1 + P.ND) + slot) * P.V + v, y0, X.flag);
    }
  }
}

// Epilogue of tiles [0, ntiles), all consumer threads: the final sum of every
// (weight row, staged row) over the input parts in index order, then the
// outputs.  `red` holds `tstride` floats per tile.
template <typename WT>
__device__ __forceinline__ void gemv_epilogue(const FrameParams& P, const CtaShared& cs, const PassCtx& X, int kind, int l,
                                           const Tile* tiles, int ntiles, int KP, int QG, const float* red,
                                           int tstride, int g0, int ng) {
  const int rpu = rows_per_unit(kind);
  for (int t = 0; t < ntiles; ++t) {
    const Tile tl = tiles[t];
    const float* rt = red + (size_t)t * tstride;
    for (int it = threadIdx.x; it < tl.n * ng; it += kConsumers) {
      const int i = it / ng, q = it - i * ng;
      float ys[2] = {0.0f, 0.0f};
      for (int h = 0; h < rpu; ++h) {
        const int row = i + h * tl.n;
        const float* base = rt + ((size_t)(row / kRB) * KP * QG + (q >> 2)) * kRedPerTask + (row % kRB) * 4 + (q & 3);
        float sum = 0.0f;
        for (int kp = 0; kp < KP; ++kp) sum += base[(size_t)kp * QG * kRedPerTask];
        ys[h] = sum;
      }
      gemv_out<WT>(P, cs, X, kind, l, tl.u0 + i, g0 + q, ys[0], ys[1]);
    }
  }
}

// Wait (all lanes of the warp) until the tile in `slot` has landed.
__device__ __forceinline__ bool wait_tile(const FrameParams& P, CtaShared& cs, uint32_t seq) {
  const uint32_t slot = seq % (uint32_t)P.nslots, par = (seq / (uint32_t)P.nslots) & 1u;
  Deadline dl;
  dl.start();
  while (!mbar_try_wait_hint(&cs.full[slot], par, 4000u))
    if (!dl.ok(P)) return false;
  return true;
}

__device__ __forceinline__ void release_tile(const FrameParams& P, CtaShared& cs, uint32_t seq) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&cs.empty[seq % (uint32_t)P.nslots]);
}

template <typename WT>
__device__ __forceinline__ void run_task(const unsigned char* tile, int nch, bool check, int b, int kp,
                                         const float* act, int KS, int q0, int nqv, float* out) {
  if (check) {
    if (nqv >= 3) gemv_task<WT, 4, true>(tile, nch, b, kp, act, KS, q0, nqv, out);
    else if (nqv == 2) gemv_task<WT, 2, true>(tile, nch, b, kp, act, KS, q0, nqv, out);
    else gemv_task<WT, 1, true>(tile, nch, b, kp, act, KS, q0, nqv, out);
  } else {
    if (nqv >= 3) gemv_task<WT, 4, false>(tile, nch, b, kp, act, KS, q0, nqv, out);
    else if (nqv == 2) gemv_task<WT, 2, false>(tile, nch, b, kp, act, KS, q0, nqv, out);
    else gemv_task<WT, 1, false>(tile, nch, b, kp, act, KS, q0, nqv, out);
  }
}

// The tasks of tiles [0, ntiles) of a phase for staged rows [0, ng): warp w
// takes tasks w, w + kWarps, ... in tile order, waits for a tile before its first
// task on it and releases every tile once past it.
template <typename WT>
__device__ __noinline__ void gemv_tasks(const FrameParams& P, CtaShared& cs, PassCtx& X, int rpu, int nch,
                                           bool check, int KP, int QG, const Tile* tiles, int ntiles, uint32_t seq0,
                                           const float* act, int KS, int ng, float* red, int tstride, bool release) {
  const int warp = threadIdx.x >> 5;
  int t = 0, base = 0, waited = -1;
  auto ntask = [&](int tt) { return ((tiles[tt].n * rpu + kRB - 1) / kRB) * KP * QG; };
  for (int tau = warp;; tau += kWarps) {
    while (t < ntiles && tau >= base + ntask(t)) {
      if (release) {
        if (waited != t && !X.fail && !wait_tile(P, cs, seq0 + t)) mark_fail(X);
        release_tile(P, cs, seq0 + t);
      }
      base += ntask(t);
      ++t;
    }
    if (t >= ntiles) break;
    const uint32_t seq = seq0 + t;
    if (waited != t) {
      if (!X.fail && !wait_tile(P, cs, seq)) mark_fail(X);
      waited = t;
    }
    const int loc = tau - base;
    const int qg = loc % QG, kp = (loc / QG) % KP, b = loc / (QG * KP);
    if (!X.fail)
      run_task<WT>(X.ring + (size_t)(seq % (uint32_t)P.nslots) * P.slot_bytes, nch, check, b, kp, act, KS, 4 * qg,
                   min(4, ng - 4 * qg), red + (size_t)t * tstride + ((size_t)(b * KP + kp) * QG + qg) * kRedPerTask);
  }
  if (release) {
    for (; t < ntiles; ++t) {
      if (waited != t && !X.fail && !wait_tile(P, cs, seq0 + t)) mark_fail(X);
      release_tile(P, cs, seq0 + t);
    }
  }
}

// One GEMV kind of one layer over this CTA's tiles (consumer warps).
template <typename WT>
__device__ __forceinline__ bool gemv_phase(const FrameParams& P, CtaShared& cs, PassCtx& X, int kind, int l,
                                        const Tile* tiles, int ntiles) {
  constexpr int EB = WTraits<WT>::EB;
  const int K = gemv_K(P, kind);
  const int nch = K * EB / 16;
  const int KP = (K + kKPart - 1) / kKPart;
  const bool check = (K % kKPart) != 0;
  const int KS = act_stride<WT>(K);
  const int rpu = rows_per_unit(kind);
  const size_t RS = row_slots(P);
  const xel* xs = nullptr;
  const float* gain = nullptr;
  switch (kind) {
    case kQKV: xs = l == 0 ? nullptr : P.hpub + ((size_t)(l - 1) * 2 + 1) * RS * P.H; gain = P.attn_norm[l]; break;
    case kO: xs = P.opub + (size_t)l * RS * P.nq * P.d; break;
    case kGU: xs = P.hpub + ((size_t)l * 2) * RS * P.H; gain = P.ffn_norm[l]; break;
    case kDown: xs = P.apub + (size_t)l * RS * P.F; break;
    default: xs = P.hpub + ((size_t)(P.L - 1) * 2 + 1) * RS * P.H; gain = P.final_norm;
  }
  float* act = X.uni;
  const int cap = max(1, min(16, P.uni_floats / KS));
  const uint32_t seq0 = X.tile_seq;
  const int NBt = (units_per_tile<WT>(P, kind) * rpu + kRB - 1) / kRB;
  if (X.nr <= cap) {
    const int QG = (X.nr + 3) >> 2;
    const int tstride = NBt * KP * QG * kRedPerTask;
    // waves of up to nslots - 2 tiles: the next wave streams in while this one computes
    const int W = max(1, P.nslots - 2);
    if (min(ntiles, W) * tstride > P.red_floats) { raise_status(&P.ctl->status, kStatusDevice); mark_fail(X); }
    stage_act<WT>(P, cs, X, xs, K, gain, 0, X.nr, act, (kind == kQKV && l == 0) ? X.hown : nullptr);
    for (int w0 = 0; w0 < ntiles; w0 += W) {
      const int nw = min(W, ntiles - w0);
      if (w0 > 0) consumer_sync();  // the previous wave's epilogue has read the partial sums
      gemv_tasks<WT>(P, cs, X, rpu, nch, check, KP, QG, tiles + w0, nw, seq0 + w0, act, KS, X.nr, X.red, tstride,
                     true);
      if (!agree_fail(X))  // every partial sum of the wave is written
        gemv_epilogue<WT>(P, cs, X, kind, l, tiles + w0, nw, KP, QG, X.red, tstride, 0, X.nr);
    }
  } else {
    // more rows than fit: tile by tile, row group by row group (re-staging)
    for (int t = 0; t < ntiles; ++t) {
      for (int g0 = 0; g0 < X.nr; g0 += cap) {
        const int ng = min(cap, X.nr - g0);
        const int QG = (ng + 3) >> 2;
        const int tstride = NBt * KP * QG * kRedPerTask;
        stage_act<WT>(P, cs, X, xs, K, gain, g0, ng, act, (kind == kQKV && l == 0) ? X.hown : nullptr);
        gemv_tasks<WT>(P, cs, X, rpu, nch, check, KP, QG, tiles + t, 1, seq0 + t, act, KS, ng, X.red, tstride,
                       g0 + ng >= X.nr);
        if (!agree_fail(X)) gemv_epilogue<WT>(P, cs, X, kind, l, tiles + t, 1, KP, QG, X.red, tstride, g0, ng);
      }
    }
  }
  X.tile_seq = seq0 + ntiles;
  return !agree_fail(X);  // the verdict every thread acts on
}

// ------------------------------------------------------------- attention
// Causal GQA attention of every (row, query head) over positions 0..pos, one
// CTA per item: warp w scores positions w, w + kWarps, ... (the dot product split
// over lanes, reduced by a butterfly) and parks their value rows in shared
// memory; then every thread forms the softmax over all positions in index
// order and each output pair is summed over positions in index order.
// Entries of positions written by this pass are polled for the pass flag;
// older positions were ordered by the previous pass's grid barrier.
__device__ __noinline__ bool attention_phase(const FrameParams& P, CtaShared& cs, PassCtx& X, int l) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = P.d, grp = P.nq / P.nkv;
  const int lines = d / 2;
  float* sc = X.uni;       // [64] scores
  float* vs = X.uni + 64;  // [G][d] value rows
  const float scale = 1.0f / sqrtf((float)d);
  const size_t RS = row_slots(P);
  const size_t pstride = (size_t)P.nkv * d;
  const int items = X.nr * P.nq;
  const uint32_t flag = X.flag;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int i = it / P.nq, hq = it - i * P.nq;
    const int r = X.rows[i], pos = X.rpos[i], b = r / P.NS, g = hq / grp;
    const int pos_new = pos - (r - b * P.NS);
    const xel* qsrc = P.qpub + ((size_t)l * RS + r) * P.nq * d + (size_t)hq * d;
    const xel* kb = P.kv + ((((size_t)b * P.L + l) * 2 + 0) * P.G) * pstride + (size_t)g * d;
    const xel* vb = P.kv + ((((size_t)b * P.L + l) * 2 + 1) * P.G) * pstride + (size_t)g * d;
    bool ok = !X.fail;
    for (int m0 = 0; warp + kWarps * m0 <= pos && ok; m0 += 2) {
      // the query and two positions' keys and values, loads issued together
      Deadline dl;
      dl.start();
      for (bool done = false; ok && !done;) {
        unsigned long long qa[4], qc[4], ka[2][4], kc[2][4], va[2][4], vc[2][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ln = lane + 32 * u;
          if (ln < lines) {
            xel_load2(qsrc + 2 * ln, qa[u], qc[u]);
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
              const int j = warp + kWarps * (m0 + mm);
              if (j <= pos) {
                xel_load2(kb + (size_t)j * pstride + 2 * ln, ka[mm][u], kc[mm][u]);
                xel_load2(vb + (size_t)j * pstride + 2 * ln, va[mm][u], vc[mm][u]);
              }
            }
          }
        }
        done = true;
        float part[2] = {0.0f, 0.0f};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ln = lane + 32 * u;
          if (ln >= lines) continue;
          if (xel_flag(qa[u]) != flag || xel_flag(qc[u]) != flag) done = false;
#pragma unroll
          for (int mm = 0; mm < 2; ++mm) {
            const int j = warp + kWarps * (m0 + mm);
            if (j > pos) continue;
            if (j >= pos_new && (xel_flag(ka[mm][u]) != flag || xel_flag(kc[mm][u]) != flag ||
                                 xel_flag(va[mm][u]) != flag || xel_flag(vc[mm][u]) != flag))
              done = false;
            part[mm] = fmaf(xel_value(qa[u]), xel_value(ka[mm][u]), part[mm]);
            part[mm] = fmaf(xel_value(qc[u]), xel_value(kc[mm][u]), part[mm]);
            *reinterpret_cast<float2*>(vs + (size_t)j * d + 2 * ln) = make_float2(xel_value(va[mm][u]), xel_value(vc[mm][u]));
          }
        }
        done = __all_sync(0xffffffffu, done);
        if (!done) {
          if (!dl.ok(P)) ok = false;
          continue;
        }
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
          const int j = warp + kWarps * (m0 + mm);
          const float sdot = warp_sum(part[mm]) * scale;
          if (lane == 0 && j <= pos) sc[j] = sdot;
        }
      }
    }
    agree_fail(X, !ok);
    if (!X.fail && tid < lines) {
      float mx = -INFINITY;
      for (int j = 0; j <= pos; ++j) mx = fmaxf(mx, sc[j]);
      float den = 0.0f;
      for (int j = 0; j <= pos; ++j) den += expf(sc[j] - mx);
      float2 o = make_float2(0.f, 0.f);
      for (int j = 0; j <= pos; ++j) {
        const float w = expf(sc[j] - mx) / den;
        const float2 v = *reinterpret_cast<const float2*>(vs + (size_t)j * d + 2 * tid);
        o.x = fmaf(w, v.x, o.x);
        o.y = fmaf(w, v.y, o.y);
      }
      xel* od = P.opub + ((size_t)l * RS + r) * P.nq * d + (size_t)hq * d + 2 * tid;
      xel_store(od, o.x, flag);
      xel_store(od + 1, o.y, flag);
    }
    consumer_sync();
  }
  return !agree_fail(X);
}

// ------------------------------------------------------------------ top-k
// One vocabulary row (in shared memory as floats in `keys` on entry)
// processed by the consumer warps, with the semantics of the oracle's
// processing: z = fl32(logit/T), exactly min(k, V) entries kept by
// (z desc, index asc), e = cp_expf(z - zmax), S = float32 sum of e in
// ascending index order, p = fl32(e / S); T = 0 is argmax (lowest index).
// Thread t owns indices [t*E, t*E + E).  The k-th key is found by an
// MSB-first 8-bit radix select over warp-private histograms (increments
// aggregated per bin across the warp, no atomics); one scan of packed
// (greater, equal) counts places every kept entry in index order.
// Scratch: hw [kWarps][256], ebuf [min(k, V)], sx [64].  Returns the length.
__device__ __noinline__ int block_topk(int V, int k, float T, uint32_t* keys, uint32_t* hw, float* ebuf, int* sx,
                                       int* out_idx, float* out_prob) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = reinterpret_cast<const float*>(keys);
  const int E = (V + kConsumers - 1) / kConsumers;
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
    consumer_sync();
    if (tid == 0) {
      float b = sbest[0];
      int ix = sbi[0];
      for (int w = 1; w < kWarps; ++w)
        if (sbest[w] > b || (sbest[w] == b && sbi[w] < ix)) { b = sbest[w]; ix = sbi[w]; }
      out_idx[0] = ix;
      out_prob[0] = 1.0f;
    }
    consumer_sync();
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
  consumer_sync();
  kmax = 0;
  for (int w = 0; w < kWarps; ++w) kmax = max(kmax, (uint32_t)sx[w]);
  const int kk = k < V ? k : V;
  uint32_t prefix = 0, mask = 0;
  int need = kk;
  bool eq_all = (kk == V);
  uint32_t* my = hw + warp * 256;
  for (int shift = 24; shift >= 0 && !eq_all; shift -= 8) {
    // warp-private histogram, aggregated increments (no atomics: one leader per bin per step)
#pragma unroll
    for (int j = 0; j < 8; ++j) my[lane * 8 + j] = 0;
    __syncwarp();
    for (int e = 0; e < E; ++e) {
      const int i = i0 + e;
      const uint32_t key = i < i1 ? keys[i] : 0u;
      const bool hit = i < i1 && (key & mask) == prefix;
      const uint32_t bin = (key >> shift) & 255u;
      const unsigned grp = __match_any_sync(0xffffffffu, hit ? bin : 0xFFFFFFFFu);
      if (hit && lane == __ffs(grp) - 1) my[bin] += (uint32_t)__popc(grp);
      __syncwarp();
    }
    consumer_sync();
    if (warp == 0) {
      // lane l holds bins 255-8l .. 248-8l (descending), summed over the warps
      uint32_t cnt[8], chunk = 0;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int b = 255 - 8 * lane - m;
        uint32_t c = 0;
        for (int w = 0; w < kWarps; ++w) c += hw[w * 256 + b];
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
    consumer_sync();
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
  consumer_sync();
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
  consumer_sync();
  if (tid == 0) {
    float S = 0.0f;
    for (int p = 0; p < kk; ++p) S = __fadd_rn(S, ebuf[p]);
    reinterpret_cast<float*>(sx)[48] = S;
  }
  consumer_sync();
  const float S = reinterpret_cast<float*>(sx)[48];
  for (int p = tid; p < kk; p += kConsumers) out_prob[p] = __fdiv_rn(ebuf[p], S);
  consumer_sync();
  return kk;
}

// Poll one exchange row of n values (n even) into shared memory.
__device__ bool poll_row(const FrameParams& P, const xel* src, int n, uint32_t flag, float* dst) {
  const int tid = threadIdx.x;
  const int lines = n >> 1;
  const int lpt = (lines + kConsumers - 1) / kConsumers;
  for (int c0 = 0; c0 < lpt; c0 += 8) {
    uint32_t pend = 0;
    for (int u = 0; u < 8 && c0 + u < lpt; ++u)
      if (tid + kConsumers * (c0 + u) < lines) pend |= 1u << u;
    Deadline dl;
    dl.start();
    while (pend) {
      unsigned long long a[8], b[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (pend & (1u << u)) xel_load2(src + 2 * (tid + kConsumers * (c0 + u)), a[u], b[u]);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if ((pend & (1u << u)) && xel_flag(a[u]) == flag && xel_flag(b[u]) == flag) {
          *reinterpret_cast<float2*>(dst + 2 * (tid + kConsumers * (c0 + u))) = make_float2(xel_value(a[u]), xel_value(b[u]));
          pend &= ~(1u << u);
        }
      if (pend && !dl.ok(P)) return false;
    }
  }
  return true;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Top-k / temperature / softmax of every (row, slot) vocabulary row, one CTA
// per row; the list is published with a release store of (count, flag).
__device__ __noinline__ bool topk_phase(const FrameParams& P, CtaShared& cs, PassCtx& X) {
  const size_t keys_bytes = ((size_t)P.V * 4 + 15) / 16 * 16;
  unsigned char* base = reinterpret_cast<unsigned char*>(X.uni);
  uint32_t* keys = reinterpret_cast<uint32_t*>(base);
  uint32_t* hw = reinterpret_cast<uint32_t*>(base + keys_bytes);
  float* ebuf = reinterpret_cast<float*>(base + keys_bytes + kWarps * 1024);
  int* sx = reinterpret_cast<int*>(base + keys_bytes + kWarps * 1024 + ((size_t)P.KC * 4 + 15) / 16 * 16);
  const int slots = 1 + P.ND;
  const int items = X.nr * slots;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int i = it / slots, t = it - i * slots;
    const int pos = X.rpos[i];
    if (pos < 1 || pos + t > P.G - 1) continue;
    const int r = X.rows[i], b = r / P.NS;
    const size_t li = (size_t)r * slots + t;
    consumer_sync();  // keys / scratch reuse
    if (!X.fail && !poll_row(P, P.logits + li * P.V, P.V, X.flag, reinterpret_cast<float*>(keys))) mark_fail(X);
    if (agree_fail(X)) continue;
    const int n = block_topk(P.V, P.top_k[b], P.temp[b], keys, hw, ebuf, sx, P.lidx + li * P.KC, P.lprob + li * P.KC);
    if (threadIdx.x == 0) {
      __threadfence();
      st_release_u64(P.lflag + li, (unsigned long long)(uint32_t)n | ((unsigned long long)X.flag << 32));
    }
  }
  return !agree_fail(X);
}

// ------------------------------------------------------ per-stream logic
__device__ __forceinline__ int valid_code(const FrameParams& P, int c) {
  if (c < 0 || c >= P.V) { raise_status(&P.ctl->status, kStatusDevice); return 0; }
  return c;
}

// Record the rows of stream b's next pass (state already updated in S):
// positions pos0.. and the code whose embedding each row carries (the frame
// index for the x row at position 0).  Warp-wide.
template <typename WT>
__device__ __noinline__ void set_pass_rows(const FrameParams& P, int b, const StreamState& S, const int* codes_in,
                                           int parity_next) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane < P.NS) {
    const int on = lane < S.m;
    P.row_pos[b * P.NS + lane] = on ? S.pos0 + lane : -1;
    P.row_code[b * P.NS + lane] = on ? codes_in[lane] : 0;
  }
  (void)parity_next;
  if (lane == 0) {
    const long long kvb = (long long)(S.pos0 + S.m) * P.L * 2 * P.nkv * P.d * (long long)sizeof(float);
    atomicAdd((unsigned long long*)&P.ctl->kv_bytes, (unsigned long long)kvb);
    atomicAdd((unsigned long long*)&P.ctl->weight_bytes, (unsigned long long)((long long)S.m * P.H * sizeof(WT)));
  }
  __syncwarp();
}

// Frame start: rows [x, E_0(c_0)] at positions 0, 1.  Scalar state fields
// are written by lane 0 only; every all-lane read of them follows a __syncwarp().
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
  const int codes_in[2] = {frame, S.codes[0]};
  set_pass_rows<WT>(P, b, S, codes_in, parity_next);
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
  set_pass_rows<WT>(P, b, S, codes_in, parity_next);
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

__device__ __forceinline__ void stage_list_async(const FrameParams& P, AcceptScratch& A, int slot, const int* gidx,
                                                 const float* gprob) {
  warp_copy_async(A.idx + (size_t)slot * P.KC, gidx, P.KC * 4);
  warp_copy_async(A.prob + (size_t)slot * P.KC, gprob, P.KC * 4);
}

// Lane `lane` < n waits (acquire) for the published list li[lane] of this
// pass and returns its length; the warp agrees on success.
__device__ __forceinline__ bool wait_lists(const FrameParams& P, uint32_t flag, size_t li, bool mine, int& cnt) {
  bool ok = true;
  cnt = 0;
  if (mine) {
    Deadline dl;
    dl.start();
    for (;;) {
      const unsigned long long w = ld_acquire_u64(P.lflag + li);
      if ((uint32_t)(w >> 32) == flag) { cnt = (int)(uint32_t)w; break; }
      if (!dl.ok(P)) { ok = false; break; }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// After codes up to depth s_new are committed: finish the frame or set up the next pass.
template <typename WT>
__device__ __noinline__ bool after_commit(const FrameParams& P, uint32_t flag, int b, AcceptScratch& A, int s_new,
                                          int hrow, int parity_next) {
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
    return true;
  }
  if (P.N == 0) {
    if (lane == 0) { S.s = s_new; S.phase = kPhaseAR; S.pos0 = s_new + 1; S.m = 1; S.n_d = 0; }
    __syncwarp();
    const int code = S.codes[s_new];
    set_pass_rows<WT>(P, b, S, &code, parity_next);
    return true;
  }
  const int R = P.G - 1 - s_new;
  const int n_d = min(P.N - 1, R);
  const int slots = 1 + P.ND;
  // The draft distributions q_t = proc(head_{s+t} . h_s), t = 1..n_d, are
  // this pass's speculative draft slots on the row at position s_new: stage
  // them, sample the drafts, and keep them for the next pass's acceptance.
  int cnt = 0;
  if (!wait_lists(P, flag, (size_t)hrow * slots + 1 + lane, lane < n_d, cnt)) return false;
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
  set_pass_rows<WT>(P, b, S, codes_in, parity_next);
  return true;
}

// Teacher-forced run: copy this chunk's target (and draft) logits out.
__device__ bool teacher_copy(const FrameParams& P, uint32_t flag, int b, const StreamState& S) {
  const int lane = threadIdx.x & 31;
  const int slots = 1 + P.ND;
  for (int i = 0; i < S.m; ++i) {
    const int row = b * P.NS + i, pos = S.pos0 + i;
    if (pos < 1) continue;
    for (int t = 0; t <= (P.t_draft ? P.ND : 0); ++t) {
      const bool ok = pos + t <= P.G - 1;
      float* dst = t == 0 ? P.t_logits + ((size_t)b * (P.P - 1) + pos - 1) * P.V
                          : P.t_draft + (((size_t)b * (P.P - 1) + pos - 1) * P.ND + (t - 1)) * P.V;
      const xel* src = P.logits + ((size_t)row * slots + t) * P.V;
      for (int v = 2 * lane; v < P.V; v += 64) {
        float2 o = make_float2(0.f, 0.f);
        if (ok) {
          Deadline dl;
          dl.start();
          for (;;) {
            unsigned long long a, c;
            xel_load2(src + v, a, c);
            if (xel_flag(a) == flag && xel_flag(c) == flag) { o = make_float2(xel_value(a), xel_value(c)); break; }
            if (!dl.ok(P)) return false;
          }
        }
        *reinterpret_cast<float2*>(dst + v) = o;
      }
    }
  }
  return true;
}

template <typename WT>
__device__ bool accept_stream(const FrameParams& P, uint32_t flag, int b, AcceptScratch& A, int parity_next) {
  StreamState& S = *A.S;
  const int lane = threadIdx.x & 31;
  load_state(P, b, S);
  if (S.phase == kPhaseDone) return true;
  const int slots = 1 + P.ND;
  StreamStats* ss = P.sstats + b;
  if (S.phase == kPhaseTeacher) {
    if (!__all_sync(0xffffffffu, teacher_copy(P, flag, b, S))) return false;
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
    return true;
  }
  // Stage the lists this decision reads: the target rows' slot-0 lists
  // (p_{s+1..s+m}) and, for a speculative round, the saved draft lists q_t.
  const bool spec = S.phase == kPhaseSpec;
  const int nl = spec ? S.m + S.n_d : 1;
  const int row0 = b * P.NS + (S.phase == kPhasePrefill ? 1 : 0);
  int cnt = 0;
  if (spec) {
    if (!wait_lists(P, flag, (size_t)(b * P.NS + lane) * slots, lane < S.m, cnt)) return false;
    if (lane >= S.m && lane < nl) cnt = __ldcg(P.qcount + (size_t)b * P.ND + (lane - S.m));
    for (int i = 0; i < S.m; ++i) {
      const size_t li = (size_t)(b * P.NS + i) * slots;
      stage_list_async(P, A, i, P.lidx + li * P.KC, P.lprob + li * P.KC);
    }
    for (int t = 0; t < S.n_d; ++t) {
      const size_t qi = ((size_t)b * P.ND + t) * P.KC;
      stage_list_async(P, A, S.m + t, P.qidx + qi, P.qprob + qi);
    }
  } else {
    if (!wait_lists(P, flag, (size_t)row0 * slots, lane == 0, cnt)) return false;
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
  if (!after_commit<WT>(P, flag, b, A, s_new, hrow, parity_next)) return false;
  store_state(P, b, S);
  return true;
}

// Streams are owned by warps of CTAs from the end of the grid (the top-k
// items start at CTA 0).  Returns false (uniformly over the consumers) on a
// failed wait.
template <typename WT>
__device__ __noinline__ bool accept_phase(const FrameParams& P, PassCtx& X, int parity_next, bool setup) {
  const int warp = threadIdx.x >> 5;
  bool ok = !X.fail;
  if (warp < P.accept_warps && ok) {
    AcceptScratch A = accept_scratch(P, X.uni);
    StreamState& S = *A.S;
    const int cta = gridDim.x - 1 - blockIdx.x;
    for (int b = cta + gridDim.x * warp; b < P.B && ok; b += gridDim.x * P.accept_warps) {
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
        ok = accept_stream<WT>(P, X.flag, b, A, parity_next);
      }
    }
  }
  return !agree_fail(X, !ok);
}

// Active rows of the pass, their positions, input codes and the lm_heads the
// pass needs, identical in every CTA; publishes the lm_head tiles to the producer.
template <typename WT>
__device__ __noinline__ void build_pass_lists(const FrameParams& P, int pass, CtaShared& cs, int* rows, int* rpos,
                                              int* rcode) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const unsigned lt = (1u << lane) - 1u;
    int n = 0;
    const int total = P.B * P.NS;
    unsigned long long mask = 0;  // lm_heads: head_j for j in [pos, pos + ND] of every row at pos >= 1
    for (int j0 = 0; j0 < total; j0 += 32) {
      const int r = j0 + lane;
      const int pos = r < total ? __ldcg(P.row_pos + r) : -1;
      const bool on = pos >= 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, on);
      if (on) {
        const int at = n + __popc(bal & lt);
        rows[at] = r;
        rpos[at] = pos;
        rcode[at] = __ldcg(P.row_code + r);
        if (pos >= 1)
          for (int t = 0; t <= P.ND && pos + t <= P.G - 1; ++t) mask |= 1ull << (pos + t);
      }
      n += __popc(bal);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mask |= __shfl_xor_sync(0xffffffffu, mask, o);
    if (lane == 0) {
      cs.nrows = n;
      int nh = 0;
      for (int hd = 1; hd < P.G && hd < 64; ++hd)
        if ((mask >> hd) & 1ull) cs.heads[nh++] = hd;
      cs.nheads = nh;
      const int par = pass & 1;
      for (int i = 0; i < nh; ++i) cs.hheads[par][i] = cs.heads[i];
      cs.nhtab[par] = make_tiles<WT>(P, kHeads, nh, cs.htab[par]);
      __threadfence_block();
      cs.heads_ready = pass;
    }
  }
  consumer_sync();
}

// Per-phase time as seen by CTA 0 (thread 0), accumulated in shared memory.
__device__ __forceinline__ void clk_tick(CtaShared& cs, int kind) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const uint64_t now = globaltimer_ns();
    cs.clk_ns[kind] += (long long)(now - cs.clk_last);
    cs.clk_last = now;
  }
}

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) frame_kernel(const __grid_constant__ FrameParams Pg) {
  // The parameter block is copied to shared memory once: phases read it
  // through a reference, which must not become a generic load from the
  // parameter space on every use.
  __shared__ __align__(16) FrameParams sP;
  {
    const int4* src = reinterpret_cast<const int4*>(&Pg);
    int4* dst = reinterpret_cast<int4*>(&sP);
    for (int i = threadIdx.x; i < (int)(sizeof(FrameParams) / 16); i += kThreads) dst[i] = src[i];
    if (threadIdx.x == 0)
      for (size_t i = sizeof(FrameParams) / 16 * 16; i < sizeof(FrameParams); ++i)
        reinterpret_cast<char*>(&sP)[i] = reinterpret_cast<const char*>(&Pg)[i];
  }
  const FrameParams& P = sP;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ CtaShared cs;
  __syncthreads();
  const int rows_cap = P.Bmax * P.NS;
  int* rows = reinterpret_cast<int*>(smem_raw);
  int* rpos = rows + rows_cap;
  int* rcode = rpos + rows_cap;
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.nslots; ++s) {
      mbar_init(&cs.full[s], 1);
      mbar_init(&cs.empty[s], kWarps);
      cs.tile_done[s] = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    cs.heads_ready = -1;
    cs.stop = 0;
    for (int kind = kQKV; kind <= kDown; ++kind) cs.ntab[kind] = make_tiles<WT>(P, kind, 0, cs.tab[kind]);
    cs.own0 = (int)(((long long)P.H * blockIdx.x) / gridDim.x);
    cs.own1 = (int)(((long long)P.H * (blockIdx.x + 1)) / gridDim.x);
  }
  __syncthreads();
  unsigned char* ring = smem_raw + P.off_ring;
  if (threadIdx.x >= kConsumers) {
    if (threadIdx.x == kConsumers) producer_loop<WT>(P, cs, ring);
    return;
  }
  Control* ctl = P.ctl;
  __shared__ PassCtx Xs;
  PassCtx& X = Xs;
  X.rows = rows;
  X.rpos = rpos;
  X.rcode = rcode;
  X.nr = 0;
  X.uni = reinterpret_cast<float*>(smem_raw + P.off_uni);
  X.red = reinterpret_cast<float*>(smem_raw + P.off_red);
  X.hown = reinterpret_cast<float*>(smem_raw + P.off_hown);
  X.ring = ring;
  X.rope = P.rope;
  if (P.off_rope >= 0) {
    float2* sr = reinterpret_cast<float2*>(smem_raw + P.off_rope);
    for (int i = threadIdx.x; i < P.G * (P.d / 2); i += kConsumers) sr[i] = P.rope[i];
    X.rope = sr;
    consumer_sync();
  }
  X.tile_seq = 0;
  X.fail = 0;
  consumer_sync();
  unsigned long long gen = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) cs.clk_ns[i] = 0;
    cs.n_pass = cs.w_bytes = cs.n_heads = 0;
  }
  const int pass_base = __ldcg(&ctl->pass_global);
  int pass = 0;
  X.flag = (uint32_t)pass_base + 1u;
  if (P.do_setup) {
    if (blockIdx.x == 0 && threadIdx.x == 0) ctl->active = P.B;
    if (!accept_phase<WT>(P, X, (pass_base + 1) & 1, true) ||
        !grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns, &cs.s_ok)) { mark_fail(X); goto done; }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) cs.clk_last = globaltimer_ns();
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
      X.flag = (uint32_t)(pass_base + pass) + 1u;
      build_pass_lists<WT>(P, pass, cs, rows, rpos, rcode);
      X.nr = cs.nrows;
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        cs.n_pass += 1;
        cs.w_bytes += (long long)P.L * P.layer_bytes + (long long)cs.nheads * P.head_bytes;
        cs.n_heads += cs.nheads;
        ctl->dbg_pass = pass;
      }
      // one call site per phase type: per layer QKV, attention, O, gate/up,
      // down; then the lm_heads
      for (int step = 0; step <= 5 * P.L; ++step) {
        const int l = step / 5, sub = step - 5 * l;
        bool ok;
        if (step < 5 * P.L && sub == 1) {
          ok = attention_phase(P, cs, X, l);
        } else {
          const int kind = step == 5 * P.L ? (int)kHeads : (sub == 0 ? (int)kQKV : sub - 1);
          const Tile* tiles = kind == kHeads ? cs.htab[pass & 1] : cs.tab[kind];
          const int nt = kind == kHeads ? cs.nhtab[pass & 1] : cs.ntab[kind];
          ok = gemv_phase<WT>(P, cs, X, kind, kind == kHeads ? 0 : l, tiles, nt);
        }
        if (!ok) goto done;
        clk_tick(cs, step == 5 * P.L ? 5 : sub);
      }
      if (P.mode == kModeDecode) {
        if (!topk_phase(P, cs, X)) goto done;
        clk_tick(cs, 6);
      }
      if (!accept_phase<WT>(P, X, (pass_base + pass + 1) & 1, false)) goto done;
      ++pass;
      if (!grid_barrier(&ctl->bar, &ctl->status, gen, P.timeout_ns, &cs.s_ok)) { mark_fail(X); goto done; }
      clk_tick(cs, 7);
    }
  }
done:
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // exchange flags must never repeat: after a failure skip past any pass a
    // faster CTA may have started
    ctl->pass_global = pass_base + pass + (X.fail ? 2 : 0);
    ctl->passes += cs.n_pass;
    ctl->weight_bytes += cs.w_bytes;
    ctl->heads_applied += cs.n_heads;
    for (int i = 0; i < 8; ++i) ctl->phase_ns[i] += cs.clk_ns[i];
    ctl->dbg_gen = (int)gen;
  }
  consumer_sync();
  if (threadIdx.x == 0) cs.stop = 1;
}

template __global__ void frame_kernel<float>(const __grid_constant__ FrameParams Pg);
template __global__ void frame_kernel<__nv_bfloat16>(const __grid_constant__ FrameParams Pg);

// ------------------------------------------------------------- init kernels
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

}  // namespace cpk

// Host-side launch helpers (used by cp_spec.cu).
namespace cpk_host {

cudaError_t launch_frame_kernel(const cpk::FrameParams& P, int grid, size_t smem, cudaStream_t stream) {
  void* args[] = {const_cast<cpk::FrameParams*>(&P)};
  const void* fn = P.dtype == 1 ? (const void*)cpk::frame_kernel<__nv_bfloat16> : (const void*)cpk::frame_kernel<float>;
  return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(cpk::kThreads), args, smem, stream);
}

cudaError_t frame_kernel_config(int dtype, size_t smem, int* max_blocks_per_sm) {
  const void* fn = dtype == 1 ? (const void*)cpk::frame_kernel<__nv_bfloat16> : (const void*)cpk::frame_kernel<float>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_blocks_per_sm, fn, cpk::kThreads, smem);
}

cudaError_t launch_init_tables(float2* rope, int G, int d, double theta, int* top_k, float* temp, int Bmax, int k,
                               float T, cudaStream_t stream) {
  cpk::init_tables_kernel<<<8, 256, 0, stream>>>(rope, G, d, theta, top_k, temp, Bmax, k, T);
  return cudaGetLastError();
}

}  // namespace cpk_host
